/*
 * attn.h -- C ABI of the GB300 (sm_103a) scaled dot-product attention library.
 *
 * The library computes multi-head scaled dot-product attention forward,
 *
 *     out = softmax(Q K^T * scale + M) V        independently per (batch, head),
 *
 * where M is 0 for an allowed (query, key) pair and -inf for a forbidden one,
 * applied before the softmax.  The definition is the one shared by the pages
 * "Attention from First Principles" (section 1, "In one line"; section 4,
 * "Tiny example"), "Self-Attention" ("Scaled Dot-Product Attention", "Causal
 * Masking") and "Attention from Scratch" (kube-dojo), Parts 2 and 3.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.   Tensors are dense, row-major (B, H, S, D) arrays with D fastest:
 *           element (b, h, s, d) lives at ((b*H + h)*S + s)*D + d.  This is
 *           the head-split layout of "Attention from scratch"
 *           (open-llm-engineering), split_heads.  Decode tensors q and out are
 *           (B, H, D), i.e. (B, H, 1, D).
 * Memory.   Every tensor pointer is DEVICE memory owned by the caller, aligned
 *           to 16 bytes (a pointer to an empty tensor may be NULL).  The
 *           library never frees or retains it.  kv_len, when
 *           not NULL, is a DEVICE array of B int32 values; it is read by the
 *           kernels (no host synchronisation), and each value is clamped to
 *           [0, Skv].
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 *           Calls are asynchronous: they enqueue work and return.  Argument
 *           errors are detected on the host before anything is enqueued.
 *           Kernels are launched with programmatic stream serialisation
 *           (programmatic dependent launch): one may be placed while the
 *           previous kernel in the stream finishes, but it reads no input
 *           and writes nothing before that kernel has completed, so stream
 *           order holds as for an ordinary launch.
 * dtype.    ATTN_BF16: bfloat16 inputs and output, fp32 accumulation and
 *           softmax statistics, output rounded to nearest even.
 *           ATTN_F32: float32 everywhere (no TF32).  Output dtype = input dtype.
 * Masking.  causal: key j is visible from query i iff j <= i + (Skv - Sq)
 *           (the last query is aligned with the last key; for Sq == Skv this
 *           is the lower-triangular mask of the pages).  kv_len: keys
 *           j >= kv_len[b] are masked (right padding, "Attention from Scratch"
 *           (kube-dojo), Part 3 padding mask).  A query row that sees no key
 *           outputs exact zeros (the pages raise an error for such a row; an
 *           error cannot be raised per row from a batched kernel).
 * Errors.   Every entry point returns ATTN_OK (0) or a negative code; on error
 *           attn_last_error() (per calling thread) describes it.  Nothing is
 *           printed and nothing aborts.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stdint.h>

#if defined(_WIN32)
#define ATTN_API
#else
#define ATTN_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
#define ATTN_F32 0
#define ATTN_BF16 1

/* Status codes. */
#define ATTN_OK 0
#define ATTN_EINVAL (-1)       /* bad argument: NULL pointer, bad size, misalignment, ... */
#define ATTN_EUNSUPPORTED (-2) /* valid request this library does not implement (never a silent fallback) */
#define ATTN_ECUDA (-3)        /* a CUDA runtime or driver call failed; see attn_last_error() */
#define ATTN_ENOMEM (-4)       /* workspace allocation failed */
#define ATTN_ETIMEOUT (-5)     /* a device-side wait hit its iteration limit (reported by attn_device_status) */
#define ATTN_ECONFLICT (-6)    /* two bf16 prefill launches shared one work counter (reported by attn_device_status) */

/*
 * attn_fwd -- prefill attention for a batch of multi-head sequences.
 *
 * Defines: "Attention from First Principles", section 5 "The full
 * multi-head computation" (scores, scale by 1/sqrt(d_head), causal mask,
 * softmax over keys, weights @ V), with the key-padding mask of "Attention
 * from Scratch" (kube-dojo), Part 3, combined by logical AND.
 *
 *   q    (B, H, Sq,  D)  query rows
 *   k    (B, H, Skv, D)  key rows
 *   v    (B, H, Skv, D)  value rows
 *   out  (B, H, Sq,  D)  written; must not overlap q, k or v
 *   scale   multiplier of Q K^T; must be finite and >= 0 (1/sqrt(D) is the
 *           pages' choice, "Why divide by the square root of the head
 *           dimension?")
 *   causal  0 or 1; causal with Sq > Skv is rejected (ATTN_EINVAL)
 *   kv_len  NULL, or device int32[B]: per-sequence valid length; keys
 *           j >= kv_len[b] are masked.  With Sq == Skv the call is
 *           self-attention over a right-padded batch and query rows
 *           i >= kv_len[b] output zeros too.  With Sq != Skv only non-causal
 *           calls take kv_len (cross-attention with a padded source,
 *           "Attention from Scratch" (kube-dojo), Part 7: the padding mask
 *           spans the source length); for a causal chunk of queries against a
 *           cache use attn_fwd_chunked.
 *   dtype   ATTN_BF16: D must be 64 or 128.  ATTN_F32: D must be 64 or 128.
 *
 * Sizes: B, H >= 1; Sq, Skv >= 0 (an empty call returns ATTN_OK and does
 * nothing); D as above; B*H*max(Sq,Skv)*D must fit in 2^31 rows of D.
 *
 * Concurrency (bf16).  The kernel hands out its work through a counter in a
 * fixed table of the library (no allocation, no clearing launch).  Direct
 * calls take the table's first 64 counters in turn, so at most 64 bf16
 * prefill calls (attn_fwd, attn_fwd_gqa, attn_fwd_chunked, attn_fwd_host's
 * chunks) may be in flight on one device at once.  A call made while its
 * stream is being captured into a CUDA graph gets a counter of its own from
 * 1024 further ones, which every replay of that graph node uses; so one
 * graph must not be replayed on two streams at the same time, and at most
 * 1024 captured prefill calls should be alive.  A launch that finds its
 * counter in use by another launch records that in the device status word:
 * attn_device_status() then returns ATTN_ECONFLICT, and the outputs of both
 * launches are undefined.  A conflict can leave the shared counter
 * unbalanced, and so can a launch that gave up on a device-side wait
 * (ATTN_ETIMEOUT), so that later launches on it report ATTN_ECONFLICT too:
 * once no call is in flight on the device, attn_release() clears every
 * counter.
 */
ATTN_API int attn_fwd(const void *q, const void *k, const void *v, void *out, int B, int H,
                      int Sq, int Skv, int D, float scale, int causal, const int32_t *kv_len,
                      int dtype, void *stream);

/*
 * attn_fwd_gqa -- attn_fwd with grouped-query (or multi-query) attention.
 *
 * Defines: "Attention from First Principles", section 5 "The full
 * multi-head computation" and "MHA, GQA, MQA -- the KV cache lever"; "Scaled
 * dot-product attention with masking", "Grouped-query attention (GQA)": the
 * keys and values have H_kv heads, H_kv divides H, and query head h attends
 * with key/value head h / (H / H_kv) -- the head that repeating K and V
 * H / H_kv times along the head axis (repeat_interleave) puts at position h.
 * Nothing is repeated in memory.  H_kv == H is attn_fwd; H_kv == 1 is
 * multi-query attention.
 *
 *   q    (B, H,    Sq,  D)
 *   k    (B, H_kv, Skv, D)
 *   v    (B, H_kv, Skv, D)
 *   out  (B, H,    Sq,  D)  written; must not overlap q, k or v
 *
 * Every other argument, rule and error is as in attn_fwd; H_kv < 1 or H not
 * a multiple of H_kv returns ATTN_EINVAL.
 */
ATTN_API int attn_fwd_gqa(const void *q, const void *k, const void *v, void *out, int B, int H,
                          int H_kv, int Sq, int Skv, int D, float scale, int causal,
                          const int32_t *kv_len, int dtype, void *stream);

/*
 * attn_fwd_host -- attn_fwd_gqa with q, k, v, out and kv_len in HOST memory:
 * the same attention ("Attention from First Principles", section 5 "The full
 * multi-head computation"), with the copies to and from the GPU done by the
 * library and overlapped with the computation.
 *
 * The batch is cut into chunks of whole key/value-head groups (whole
 * sequences, or runs of key/value heads of one sequence), each a contiguous
 * run of (b, h) slices; chunk c is copied in while chunk c - 1 is computed
 * and chunk c - 2 is copied out, on the library's own copy streams.  Each
 * chunk is computed exactly as attn_fwd_gqa computes those slices, so the
 * result equals attn_fwd_gqa's bit for bit.
 *
 *   q, k, v, out  host pointers, layouts and sizes as in attn_fwd_gqa.  Page-
 *                 locked (pinned) memory lets the copies run asynchronously at
 *                 full speed; pageable memory works but is staged.  out must
 *                 not overlap the inputs.
 *   kv_len        NULL or HOST int32[B], meaning as in attn_fwd_gqa.
 *   stream        the work starts after work already queued on `stream`, which
 *                 resumes after the last copy out.
 *
 * Synchronous: returns when out holds the result (or on error).  D must be 64
 * or 128 (ATTN_EUNSUPPORTED otherwise).  The library keeps device copies of
 * q, k, v, out (grown on demand, freed by attn_release), so concurrent calls
 * on one device run one after the other.  Other errors as in attn_fwd_gqa;
 * ATTN_ENOMEM if the device copies cannot be allocated.
 */
ATTN_API int attn_fwd_host(const void *q, const void *k, const void *v, void *out, int B, int H,
                           int H_kv, int Sq, int Skv, int D, float scale, int causal,
                           const int32_t *kv_len, int dtype, void *stream);

/*
 * attn_fwd_chunked -- prefill of a chunk of new queries against a KV cache,
 * with the log-sum-exp of every row.
 *
 * Defines: the cache append before causal attention of "Scaled
 * dot-product attention with masking" ("The full multi-head computation":
 * past keys and values are concatenated with the new ones), with positions
 * kept absolute ("Attention from scratch" (open-llm-engineering), "KV cache
 * position drift").  Sequence b holds L_b = cache_len[b] valid cache
 * positions, the last Sq of which are the chunk's own keys and values
 * (appended by the caller); query i sits at position L_b - Sq + i and sees
 * keys j <= L_b - Sq + i.  A query whose position is negative (L_b < Sq)
 * sees no key: its row is zero.  Grouped-query heads as in attn_fwd_gqa.
 *
 *   q          (B, H,    Sq,  D)  the chunk's queries
 *   kcache     (B, H_kv, Skv, D)  cache capacity Skv >= Sq
 *   vcache     (B, H_kv, Skv, D)
 *   out        (B, H,    Sq,  D)  written; must not overlap the inputs
 *   lse        NULL, or device float (B, H, Sq), written: log(sum_j
 *              exp(scale * q_i . k_j)) over the visible keys (natural log,
 *              fp32), -inf for a row that sees none.  Not on the pages: it is
 *              what lets a caller merge attention over split key sets exactly,
 *              out = sum_c exp(lse_c - LSE) out_c with LSE = log sum_c exp(lse_c).
 *   cache_len  NULL (every L_b = Skv) or device int32[B], clamped to [0, Skv].
 *
 * dtype, D, scale, sizes and errors as in attn_fwd; Sq > Skv returns
 * ATTN_EINVAL.  With cache_len NULL and no lse this is attn_fwd_gqa with
 * causal = 1.
 */
ATTN_API int attn_fwd_chunked(const void *q, const void *kcache, const void *vcache, void *out,
                              float *lse, int B, int H, int H_kv, int Sq, int Skv, int D, float scale,
                              const int32_t *cache_len, int dtype, void *stream);

/*
 * attn_fwd_debug -- the general attention of "Attention from Scratch"
 * (kube-dojo), Part 2, for inspection: T_q != T_k, value depth d_v != d_k,
 * and the attention weights returned with the output (Part 4 "Attention
 * Maps").  One warp per query row in fp32; not a fast path.
 *
 *   q        (B, H,    Sq,  Dk)     dtype ATTN_F32 or ATTN_BF16
 *   k        (B, H_kv, Skv, Dk)
 *   v        (B, H_kv, Skv, Dv)
 *   out      (B, H,    Sq,  Dv)     written, in the input dtype
 *   weights  NULL or device float (B, H, Sq, Skv), written: the softmax
 *            weights of each row, exactly 0 for a masked key, all 0 for a
 *            row that sees no key (and for a padded query row)
 *
 * Dk, Dv in [1, 256]; Skv <= 16384 (ATTN_EUNSUPPORTED above); tensors
 * aligned to their element size.  scale, causal, kv_len, H_kv and the mask
 * rules are those of attn_fwd / attn_fwd_gqa.
 */
ATTN_API int attn_fwd_debug(const void *q, const void *k, const void *v, void *out, float *weights,
                            int B, int H, int H_kv, int Sq, int Skv, int Dk, int Dv, float scale,
                            int causal, const int32_t *kv_len, int dtype, void *stream);

/*
 * attn_decode -- one new query per (batch, head) against a KV cache.
 *
 * Defines: "Attention from First Principles", section 6 "Under the hood"
 * (decode is a matrix-vector product against the whole cache) and "Scaled
 * dot-product attention with masking", "Adding the causal mask" (with
 * seq_q = 1 the query attends to every cached position, no mask).  The
 * scale is 1/sqrt(D).
 *
 *   q       (B, H, D)        the new queries
 *   kcache  (B, H, Skv, D)   cached keys, padded to Skv
 *   vcache  (B, H, Skv, D)   cached values, padded to Skv
 *   out     (B, H, D)        written
 *   kv_len  NULL (every sequence uses all Skv positions) or device int32[B];
 *           keys j >= kv_len[b] are ignored, kv_len[b] == 0 gives zeros.
 *   dtype   ATTN_BF16 or ATTN_F32 (fp32 everywhere, on the CUDA cores); D
 *           must be 64 or 128.  All pointers 16-byte aligned.
 *
 * The kernel splits each sequence's keys into chunks processed in parallel
 * and merges the partial softmax results; the partials live in a workspace
 * the library allocates on first use (and grows when a call needs more),
 * which attn_release() frees.  The workspace is shared by all calls on a
 * device: calls that overlap in time on different streams of one device race.
 *
 * CUDA graphs: a captured call keeps the workspace's address.  Growing the
 * workspace never frees the old buffer (it is kept until attn_release), so
 * a graph captured before a larger call stays valid.  A call made during a
 * capture cannot allocate: if it needs a larger workspace than the device
 * has, it returns ATTN_EINVAL without enqueuing anything, so make one
 * ordinary call of the largest size before capturing.  Destroy every graph
 * that holds a decode call before attn_release().
 */
ATTN_API int attn_decode(const void *q, const void *kcache, const void *vcache, void *out, int B,
                         int H, int Skv, int D, const int32_t *kv_len, int dtype, void *stream);

/*
 * attn_decode_gqa -- attn_decode with grouped-query (or multi-query) attention.
 *
 * Defines: as attn_decode, with the head grouping of attn_fwd_gqa: the cache
 * has H_kv heads, H_kv divides H, and query head h attends with cached head
 * h / (H / H_kv).  One read of a cached head serves all H / H_kv query heads
 * of its group, which is why grouping raises decode's arithmetic intensity to
 * about H / H_kv flops per byte ("Attention from First Principles", section 6
 * "Under the hood").
 *
 *   q       (B, H, D)
 *   kcache  (B, H_kv, Skv, D)
 *   vcache  (B, H_kv, Skv, D)
 *   out     (B, H, D)   written
 *
 * Every other argument, rule, error and the workspace behaviour are as in
 * attn_decode; H_kv < 1 or H not a multiple of H_kv returns ATTN_EINVAL.
 * H_kv == H runs attn_decode's kernels.  In bf16, groups of G = H / H_kv >= 4
 * heads (up to 128) run on the tensor cores, the group's queries forming the
 * rows of one tile; smaller groups and fp32 run on the CUDA cores.
 */
ATTN_API int attn_decode_gqa(const void *q, const void *kcache, const void *vcache, void *out, int B,
                             int H, int H_kv, int Skv, int D, const int32_t *kv_len, int dtype,
                             void *stream);

/*
 * attn_decode_noalloc -- attn_decode that never allocates device memory.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * must not allocate device memory while they run.  attn_decode allocates its
 * scratch (the per-chunk partial results) with cudaMalloc on first use and
 * whenever a call needs more; that fails or misbehaves for callers that have
 * reserved all device memory up front for their own pool (an inference server
 * sizing its KV cache to the whole GPU), and cudaMalloc / cudaFree can
 * synchronise the device, which a latency-bound decode loop cannot afford.
 * This variant runs the same kernels with the scratch in a fixed array inside
 * the library instead, so it calls no allocation routine at all.
 *
 * Arguments, layouts, dtype support and results are those of attn_decode.
 * Limit: B*H*attn_decode_splits(B,H,Skv,D)*(D + 2)*4 bytes must not exceed
 * 32 MiB (33554432); larger requests return ATTN_EINVAL with a message saying
 * how much they need (B64 H32 Skv8192 D128 needs about 17 MB).
 *
 * The array is part of the library image: every GPU that loads the library's
 * decode code holds these 32 MiB until the process exits.  The first call on
 * each device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current) and caches it; make that first call before any stream
 * capture on the device.  All calls on a device share the one array and its
 * contents persist between calls (nothing in it needs to start at zero: each
 * call writes every partial it reads), so calls that overlap on the GPU (on
 * different streams, or from different threads) race and must be serialised
 * by the caller.
 */
ATTN_API int attn_decode_noalloc(const void *q, const void *kcache, const void *vcache, void *out, int B,
                                 int H, int Skv, int D, const int32_t *kv_len, int dtype, void *stream);

/*
 * attn_decode_splits -- number of KV chunks attn_decode uses per (batch,
 * head) for these sizes (for benchmarks and tests); negative on bad sizes.
 */
ATTN_API int attn_decode_splits(int B, int H, int Skv, int D);

/*
 * attn_device_status -- synchronise `stream`, then report and clear the
 * device-side status word.  Returns ATTN_OK, ATTN_ETIMEOUT when a kernel gave
 * up on a device-side wait (its output is then undefined), ATTN_ECONFLICT
 * when two bf16 prefill launches in flight shared one work counter (see
 * attn_fwd, "Concurrency"; both outputs are undefined), or ATTN_ECUDA when
 * the synchronisation itself failed.
 */
ATTN_API int attn_device_status(void *stream);

/*
 * attn_selftest_wait_timeout -- diagnostic: enqueue a one-warp kernel whose
 * only device-side wait can never complete, with a limit of `limit_cycles` SM
 * clock cycles (0 .. 2e9).  The wait gives up, the kernel records the timeout
 * in the device status word and exits, so the next attn_device_status(stream)
 * returns ATTN_ETIMEOUT (and clears the word).  Used to check, on a real
 * device and without any fault or hang, the path every kernel's bounded waits
 * take when a logic error would otherwise deadlock.  There is no counterpart
 * on the pages.
 */
ATTN_API int attn_selftest_wait_timeout(long long limit_cycles, void *stream);

/* Description of the last error on the calling thread ("" if none). */
ATTN_API const char *attn_last_error(void);

/* Free library-owned device memory on the current device: the decode
 * workspace (with every smaller buffer it replaced) and attn_fwd_host's
 * device copies; and clear the bf16 prefill work counters (the recovery after
 * ATTN_ECONFLICT).  Not while any call of the library is running on the
 * device, and not while a CUDA graph that holds a library call may still be
 * replayed. */
ATTN_API void attn_release(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
