// Internal interface between the C-ABI shim (api.cu) and the kernel files.
// Arguments arrive here already validated by the shim.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Launch with programmatic stream serialisation: the kernel may be placed
// while the previous kernel in the stream finishes, and waits for it
// (griddepcontrol.wait) before it reads its inputs or writes anything, so
// back-to-back launches do not pay the full launch gap.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct FwdArgs {
    const void *q, *k, *v;  // (B, H, Sq|Skv, D), device
    void *out;              // (B, H, Sq, D), device
    const int32_t *kv_len;  // device int32[B] or nullptr
    int B, H, Sq, Skv, D;
    float scale;            // multiplier of Q K^T
    int causal;
    int *status;            // device status word
    cudaStream_t stream;
    int n_sm;               // streaming multiprocessors on the device
    int H_kv;               // key/value heads (divides H); query head h reads head h / (H / H_kv)
    // Chunk-against-cache mode (attn_fwd_chunked): kv_len[b] is the cached
    // length L_b, query i sits at position L_b - Sq + i (causal), and no query
    // row is treated as padding.
    int chunked;
    float *lse;             // (B, H, Sq) natural-log log-sum-exp of each row, or nullptr
};

struct DecodeArgs {
    const void *q;          // (B, H, D) bf16 (fp32 for launch_decode_f32)
    const void *k, *v;      // (B, H_kv, Skv, D), same dtype
    void *out;              // (B, H, D), same dtype
    const int32_t *kv_len;  // device int32[B] or nullptr
    int B, H, Skv, D;
    float scale;
    int chunk;              // keys per split (multiple of 64, <= kDecodeMaxChunk)
    int n_split;            // ceil(Skv / chunk), >= 1
    float *part_o;          // B*H*n_split*D fp32 partial outputs
    float *part_ml;         // B*H*n_split*2 fp32 (running max in log2 units, sum)
    int *status;
    cudaStream_t stream;
    int H_kv;               // cached heads (divides H); query head h reads head h / (H / H_kv)
};

constexpr int kDecodeMaxChunk = 1024;
constexpr int kDecodeGqaMaxChunk = 512;

// Debug attention (attn_fwd_debug): any d_k, d_v <= 256, optional weights.
struct DebugArgs {
    const void *q, *k, *v;  // (B, H, Sq, Dk), (B, H_kv, Skv, Dk), (B, H_kv, Skv, Dv)
    void *out;              // (B, H, Sq, Dv), input dtype
    float *weights;         // (B, H, Sq, Skv) fp32 or nullptr
    const int32_t *kv_len;  // device int32[B] or nullptr
    int B, H, H_kv, Sq, Skv, Dk, Dv;
    float scale;
    int causal;
    int dtype_bf16;
    cudaStream_t stream;
};
cudaError_t launch_debug_attention(const DebugArgs &a);

// fp32 SIMT prefill (D in {64, 128}).
cudaError_t launch_prefill_f32(const FwdArgs &a);

// bf16 tcgen05 prefill (D in {64, 128}); tq/tk/tv are 3-D tensor maps over
// (D, S, B*H) with 64 x 128 x 1 boxes and 128-byte swizzle.
cudaError_t launch_prefill_tc(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv);

// Clears every work counter of the bf16 prefill kernels on the current device
// (synchronous; no prefill launch may be in flight).
cudaError_t reset_prefill_counters();

// bf16 split-KV decode: partial kernel then combine kernel.
cudaError_t launch_decode(const DecodeArgs &a);

// The combine kernel alone (per query head: merge the chunk partials).
cudaError_t launch_decode_combine(const DecodeArgs &a);

// Grouped-query decode (H_kv < H): partial kernel per (b, h_kv, head subgroup,
// chunk), then the combine kernel.  a.chunk must not exceed
// kDecodeGqaMaxChunk (the kernel's score buffer holds that many keys).
cudaError_t launch_decode_gqa(const DecodeArgs &a);
int decode_gqa_heads_per_cta(int G);

// fp32 decode (any grouping H_kv | H): q, caches and out are fp32; partial
// kernel per (b, h, chunk <= kDecodeMaxChunk keys) on the CUDA cores, then an
// fp32-output combine.
cudaError_t launch_decode_f32(const DecodeArgs &a);

// Grouped-query / multi-query decode on the tensor cores (G = H / H_kv query
// heads per cached head, kDecodeTcMinGroup <= G <= 128; below that the CUDA-core
// kernels are as fast or faster): the G queries are the
// rows of one 128-row tile.  tq views q as (D, B*H) with 64 x 128 boxes; tk, tv
// view the caches as (D, Skv, B*H_kv) with 64 x 64 x 1 boxes (128-byte swizzle).
// a.chunk (a multiple of 64 keys, from decode_tc_chunk) and a.n_split as for
// the other decode kernels; the partials are merged by the decode combine.
#ifndef ATTN_DTC_MIN_GROUP
#define ATTN_DTC_MIN_GROUP 4
#endif
constexpr int kDecodeTcMinGroup = ATTN_DTC_MIN_GROUP;
int decode_tc_chunk(int B, int H_kv, int Skv, int n_sm);
cudaError_t launch_decode_tc(const DecodeArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv);

// Size of the library-static decode scratch used by attn_decode_noalloc.
constexpr size_t kDecodeNoAllocScratchBytes = 32u << 20;

// Decode with its partials in the library-static scratch (no allocation).
// The caller has checked that the partials fit in kDecodeNoAllocScratchBytes.
cudaError_t launch_decode_noalloc(DecodeArgs a, bool f32);

// One-warp kernel whose only wait can never complete: exercises the bounded
// wait and the status word (attn_selftest_wait_timeout).
cudaError_t launch_wait_timeout_probe(long long limit, int *status, cudaStream_t stream);

// Writes zeros over n bytes (multiple of 16, 16-byte aligned) -- degenerate
// calls whose every row sees no key.
cudaError_t launch_zero_fill(void *out, size_t n_bytes, cudaStream_t stream);

}  // namespace attn
