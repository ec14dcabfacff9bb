// C-ABI shim: argument validation, kernel dispatch, TMA descriptor encoding,
// decode workspace and the device status word.  The contract of every entry
// point is documented in include/attn.h.
#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"

#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

namespace attn {
namespace {

constexpr int kMaxDevices = 64;

thread_local char g_last_error[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(ATTN_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte ranges [a, a + na) and [b, b + nb) overlap?
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// ------------------------------------------------------------ device status word

__device__ int g_status_word;

std::mutex g_mutex;
int *g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];

int current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (*dev < 0 || *dev >= kMaxDevices) return fail(ATTN_EUNSUPPORTED, "device ordinal %d out of range", *dev);
    return ATTN_OK;
}

int status_word(int **out) {
    int dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    *out = g_status_ptr[dev];
    return ATTN_OK;
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_num_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

// ------------------------------------------------------------ TMA descriptors

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;

int get_encode(EncodeTiledFn *fn) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
            return fail(ATTN_ECUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode = reinterpret_cast<EncodeTiledFn>(p);
    }
    *fn = g_encode;
    return ATTN_OK;
}

// (D, S, B*H) bf16 view of a (B, H, S, D) tensor; boxes of 64 x box_rows x 1
// with 128-byte swizzle, out-of-range rows read as zero.
int make_map(CUtensorMap *map, const void *base, int D, int S, long long BH, int box_rows = 128) {
    EncodeTiledFn encode;
    int rc = get_encode(&encode);
    if (rc) return rc;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(S) * D * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ECUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return ATTN_OK;
}

// (D, rows) bf16 view of a row-major (rows, D) tensor; boxes of 64 x 128 with
// 128-byte swizzle, rows past the end read as zero.
int make_map_rows(CUtensorMap *map, const void *base, int D, long long rows) {
    EncodeTiledFn encode;
    int rc = get_encode(&encode);
    if (rc) return rc;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ECUDA, "cuTensorMapEncodeTiled (2-D) failed (%d)", static_cast<int>(r));
    return ATTN_OK;
}

// ------------------------------------------------------------ decode workspace

// The decode partials.  A buffer the workspace outgrows is kept on the
// retired list, not freed: a CUDA graph captured earlier may still write to
// it on every replay.  attn_release frees them all.
constexpr int kMaxRetired = 64;
struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
    void *retired[kMaxRetired] = {};
    int n_retired = 0;
};
Workspace g_ws[kMaxDevices];

int workspace(size_t bytes, cudaStream_t stream, void **out) {
    int dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(g_mutex);
    Workspace &w = g_ws[dev];
    if (w.bytes < bytes) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(stream, &cap);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
        if (cap != cudaStreamCaptureStatusNone)
            return fail(ATTN_EINVAL,
                        "attn_decode: a captured call needs %zu bytes of workspace but the device has %zu; "
                        "make one ordinary call of this size before capturing",
                        bytes, w.bytes);
        if (w.ptr && w.n_retired == kMaxRetired)
            return fail(ATTN_ENOMEM, "attn_decode: the workspace grew %d times; call attn_release", kMaxRetired);
        // grow at least geometrically, so retired buffers add up to less than the live one
        const size_t want = bytes > 2 * w.bytes ? bytes : 2 * w.bytes;
        void *p = nullptr;
        e = cudaMalloc(&p, want);
        if (e != cudaSuccess)
            return fail(ATTN_ENOMEM, "decode workspace of %zu bytes: %s", want, cudaGetErrorString(e));
        if (w.ptr) w.retired[w.n_retired++] = w.ptr;
        w.ptr = p;
        w.bytes = want;
    }
    *out = w.ptr;
    return ATTN_OK;
}

// ------------------------------------------------------------ host-buffer prefill

// Chunks per call (about) and the smallest chunk worth a copy of its own.
#ifndef ATTN_HOST_CHUNKS
#define ATTN_HOST_CHUNKS 8
#endif
constexpr int kHostChunks = ATTN_HOST_CHUNKS;
constexpr size_t kHostMinChunkBytes = 8u << 20;
constexpr int kHostEvents = 16;  // event pairs in flight; older chunks are waited for

// Per device: device copies of Q, K, V, O and kv_len (grown on demand), the
// two copy streams and the events that order them with the caller's stream.
struct HostExec {
    std::mutex mutex;
    void *buf = nullptr;
    size_t bytes = 0;
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev[2 * kHostEvents] = {};
    cudaEvent_t ev_start = nullptr, ev_end = nullptr;

    int ensure(size_t need) {
        if (!ready) {
            cudaError_t e = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking);
            if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking);
            for (int i = 0; i < 2 * kHostEvents && e == cudaSuccess; ++i)
                e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_end, cudaEventDisableTiming);
            if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_host: streams and events");
            ready = true;
        }
        if (bytes < need) {
            if (buf) cudaFree(buf);  // synchronises the device: no call still uses it
            buf = nullptr;
            bytes = 0;
            cudaError_t e = cudaMalloc(&buf, need);
            if (e != cudaSuccess) {
                buf = nullptr;
                return fail(ATTN_ENOMEM, "attn_fwd_host: %zu bytes of device buffers: %s", need, cudaGetErrorString(e));
            }
            bytes = need;
        }
        return ATTN_OK;
    }
    void release() {
        std::lock_guard<std::mutex> lock(mutex);
        if (buf) cudaFree(buf);
        buf = nullptr;
        bytes = 0;
    }
};
HostExec g_host[kMaxDevices];

// Grouped-query decode: CTAs are (b, h_kv, head subgroup, chunk); the chunk
// is at most kDecodeGqaMaxChunk keys (the kernel's score buffer).
int decode_chunk_gqa(int B, int H, int H_kv, int Skv) {
    const int G = H / H_kv;
    const int gt = decode_gqa_heads_per_cta(G);
    const long long units = static_cast<long long>(B) * H_kv * ((G + gt - 1) / gt);
    const long long want = 6LL * num_sms();
    int chunk = kDecodeGqaMaxChunk;
    while (chunk > 64 && units * ((Skv + chunk - 1) / chunk) < want) chunk /= 2;
    return chunk;
}

int decode_chunk(int B, int H, int Skv) {
    // Aim for at least ~6 CTAs per SM; shorter chunks only when the batch is small.
    const long long want = 6LL * num_sms();
    int chunk = 512;
    while (chunk > 64 && static_cast<long long>(B) * H * ((Skv + chunk - 1) / chunk) < want) chunk /= 2;
    return chunk;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

ATTN_API const char *attn_last_error(void) { return g_last_error; }

ATTN_API int attn_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int Sq,
                      int Skv, int D, float scale, int causal, const int32_t *kv_len, int dtype,
                      void *stream) {
    return attn_fwd_gqa(q, k, v, out, B, H, H, Sq, Skv, D, scale, causal, kv_len, dtype, stream);
}

// Shared by attn_fwd_gqa (chunked = 0, no lse) and attn_fwd_chunked (causal,
// kv_len = cache lengths, chunked = 1, optional lse).
static int fwd_impl(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                    int H_kv, int Sq, int Skv, int D, float scale, int causal, const int32_t *kv_len,
                    int chunked, int dtype, void *stream) {
    g_last_error[0] = '\0';
    if (B < 1 || H < 1 || Sq < 0 || Skv < 0)
        return fail(ATTN_EINVAL, "attn_fwd: need B >= 1, H >= 1, Sq >= 0, Skv >= 0 (got %d, %d, %d, %d)", B, H, Sq, Skv);
    if (H_kv < 1 || H % H_kv != 0)
        return fail(ATTN_EINVAL, "attn_fwd: H_kv must divide H (got H = %d, H_kv = %d)", H, H_kv);
    if ((Sq > 0 && (!q || !out)) || (Skv > 0 && (!k || !v)))
        return fail(ATTN_EINVAL, "attn_fwd: q and out (Sq > 0), k and v (Skv > 0) must not be NULL");
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return fail(ATTN_EINVAL, "attn_fwd: unknown dtype %d", dtype);
    if (D <= 0) return fail(ATTN_EINVAL, "attn_fwd: D must be positive (got %d)", D);
    if (D != 64 && D != 128) return fail(ATTN_EUNSUPPORTED, "attn_fwd: D = %d not supported (64 or 128)", D);
    if (!(scale >= 0.f) || isinf(scale)) return fail(ATTN_EINVAL, "attn_fwd: scale must be finite and >= 0");
    if (causal != 0 && causal != 1) return fail(ATTN_EINVAL, "attn_fwd: causal must be 0 or 1");
    if (causal && Sq > Skv) return fail(ATTN_EINVAL, "attn_fwd: causal needs Sq <= Skv (got %d > %d)", Sq, Skv);
    if (kv_len && !chunked && causal && Sq != Skv)
        return fail(ATTN_EINVAL, "attn_fwd: causal kv_len needs Sq == Skv (a chunk against a cache is attn_fwd_chunked)");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(ATTN_EINVAL, "attn_fwd: lse must be 4-byte aligned");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(ATTN_EINVAL, "attn_fwd: q, k, v and out must be 16-byte aligned");
    if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u))
        return fail(ATTN_EINVAL, "attn_fwd: kv_len must be 4-byte aligned");
    const long long bh = static_cast<long long>(B) * H;
    const long long rows = bh * (Sq > Skv ? Sq : Skv);
    if (rows >= (1LL << 31) || bh > 65535LL * 65535LL)
        return fail(ATTN_EINVAL, "attn_fwd: B*H*S = %lld rows is too large", rows);
    const size_t esz = dtype == ATTN_BF16 ? 2 : 4;
    const long long bh_kv = static_cast<long long>(B) * H_kv;
    const size_t q_bytes = static_cast<size_t>(bh) * Sq * D * esz;
    const size_t kv_bytes = static_cast<size_t>(bh_kv) * Skv * D * esz;
    if (overlaps(out, q_bytes, q, q_bytes) || overlaps(out, q_bytes, k, kv_bytes) ||
        overlaps(out, q_bytes, v, kv_bytes))
        return fail(ATTN_EINVAL, "attn_fwd: out overlaps an input");
    const size_t lse_bytes = static_cast<size_t>(bh) * Sq * sizeof(float);
    if (lse && (overlaps(lse, lse_bytes, q, q_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
                overlaps(lse, lse_bytes, v, kv_bytes) || overlaps(lse, lse_bytes, out, q_bytes)))
        return fail(ATTN_EINVAL, "attn_fwd: lse overlaps another tensor");
    if (Sq == 0) return ATTN_OK;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Skv == 0) {  // no row sees a key
        cudaError_t e = launch_zero_fill(out, q_bytes, st);
        return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_fwd zero fill");
    }
    int *status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    FwdArgs a{q, k, v, out, kv_len, B, H, Sq, Skv, D, scale, causal, status, st, num_sms(), H_kv,
              chunked, lse};
    cudaError_t e;
    if (dtype == ATTN_F32) {
        if (B > 65535 || H > 65535) return fail(ATTN_EINVAL, "attn_fwd: B and H must be <= 65535 for fp32");
        e = launch_prefill_f32(a);
    } else {
        CUtensorMap tq, tk, tv;
        if ((rc = make_map(&tq, q, D, Sq, bh)) || (rc = make_map(&tk, k, D, Skv, bh_kv)) ||
            (rc = make_map(&tv, v, D, Skv, bh_kv)))
            return rc;
        e = launch_prefill_tc(a, tq, tk, tv);
    }
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_fwd launch");
}

ATTN_API int attn_fwd_gqa(const void *q, const void *k, const void *v, void *out, int B, int H,
                          int H_kv, int Sq, int Skv, int D, float scale, int causal,
                          const int32_t *kv_len, int dtype, void *stream) {
    return fwd_impl(q, k, v, out, nullptr, B, H, H_kv, Sq, Skv, D, scale, causal, kv_len, 0, dtype,
                    stream);
}

// Prefill from host buffers: the batch is cut into chunks of whole
// key/value-head groups (runs of consecutive (b, h) slices, contiguous in the
// (B, H, S, D) layout), and chunk c's copy in, chunk c - 1's attention and
// chunk c - 2's copy out run at the same time on three streams.
ATTN_API int attn_fwd_host(const void *q, const void *k, const void *v, void *out, int B, int H,
                           int H_kv, int Sq, int Skv, int D, float scale, int causal,
                           const int32_t *kv_len, int dtype, void *stream) {
    g_last_error[0] = '\0';
    if (B < 1 || H < 1 || Sq < 0 || Skv < 0)
        return fail(ATTN_EINVAL, "attn_fwd_host: need B >= 1, H >= 1, Sq >= 0, Skv >= 0");
    if (H_kv < 1 || H % H_kv != 0)
        return fail(ATTN_EINVAL, "attn_fwd_host: H_kv must divide H (got H = %d, H_kv = %d)", H, H_kv);
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return fail(ATTN_EINVAL, "attn_fwd_host: unknown dtype %d", dtype);
    if (D != 64 && D != 128) return fail(ATTN_EUNSUPPORTED, "attn_fwd_host: D = %d not supported (64 or 128)", D);
    if ((Sq > 0 && (!q || !out)) || (Skv > 0 && (!k || !v)))
        return fail(ATTN_EINVAL, "attn_fwd_host: q and out (Sq > 0), k and v (Skv > 0) must not be NULL");
    if (causal && Sq > Skv) return fail(ATTN_EINVAL, "attn_fwd_host: causal needs Sq <= Skv (got %d > %d)", Sq, Skv);
    if (kv_len && causal && Sq != Skv) return fail(ATTN_EINVAL, "attn_fwd_host: causal kv_len needs Sq == Skv");
    if (Sq == 0) return ATTN_OK;
    const size_t esz = dtype == ATTN_BF16 ? 2 : 4;
    const int G = H / H_kv;
    const size_t q_head = static_cast<size_t>(Sq) * D * esz, kv_head = static_cast<size_t>(Skv) * D * esz;
    const size_t q_bytes = static_cast<size_t>(B) * H * q_head, kv_bytes = static_cast<size_t>(B) * H_kv * kv_head;
    if (overlaps(out, q_bytes, q, q_bytes) || overlaps(out, q_bytes, k, kv_bytes) || overlaps(out, q_bytes, v, kv_bytes))
        return fail(ATTN_EINVAL, "attn_fwd_host: out overlaps an input");
    int dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    HostExec &x = g_host[dev];
    std::lock_guard<std::mutex> lock(x.mutex);  // one call at a time per device: it owns the buffers
    // device copies: Q | K | V | O | kv_len, each 256-byte aligned
    auto up = [](size_t n) { return (n + 255) & ~static_cast<size_t>(255); };
    const size_t off_k = up(q_bytes), off_v = off_k + up(kv_bytes), off_o = off_v + up(kv_bytes);
    const size_t off_l = off_o + up(q_bytes), total = off_l + up(static_cast<size_t>(B) * sizeof(int32_t));
    if ((rc = x.ensure(total))) return rc;
    char *dbuf = static_cast<char *>(x.buf);
    int32_t *d_len = kv_len ? reinterpret_cast<int32_t *>(dbuf + off_l) : nullptr;
    // chunks: whole batches when one batch is below the target, else runs of key/value heads of one batch
    const size_t per_b = static_cast<size_t>(H) * q_head + 2 * static_cast<size_t>(H_kv) * kv_head;
    size_t target = (static_cast<size_t>(B) * per_b) / kHostChunks;
    target = target < kHostMinChunkBytes ? kHostMinChunkBytes : target;
    int nb = 1, kv_per = H_kv;  // batches per chunk, or key/value heads per chunk (nb == 1)
    if (per_b <= target) {
        nb = static_cast<int>(target / per_b);
        nb = nb < 1 ? 1 : (nb > B ? B : nb);
    } else {
        const size_t per_kv = static_cast<size_t>(G) * q_head + 2 * kv_head;
        kv_per = static_cast<int>((target + per_kv - 1) / per_kv);
        kv_per = kv_per < 1 ? 1 : (kv_per > H_kv ? H_kv : kv_per);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaEventRecord(x.ev_start, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(x.h2d, x.ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(x.d2h, x.ev_start, 0);
    if (e == cudaSuccess && kv_len)
        e = cudaMemcpyAsync(d_len, kv_len, static_cast<size_t>(B) * sizeof(int32_t), cudaMemcpyHostToDevice, x.h2d);
    int n_chunk = 0;
    for (int b0 = 0; b0 < B && e == cudaSuccess && rc == ATTN_OK; b0 += nb) {
        const int bn = b0 + nb <= B ? nb : B - b0;
        for (int g0 = 0; g0 < H_kv && e == cudaSuccess && rc == ATTN_OK; g0 += kv_per) {
            const int gn = g0 + kv_per <= H_kv ? kv_per : H_kv - g0;
            // slices: batches [b0, b0 + bn) x kv heads [g0, g0 + gn) (nb == 1 or gn == H_kv)
            const size_t qo = (static_cast<size_t>(b0) * H + static_cast<size_t>(g0) * G) * q_head;
            const size_t ko = (static_cast<size_t>(b0) * H_kv + g0) * kv_head;
            const size_t qn = static_cast<size_t>(bn) * gn * G * q_head, kn = static_cast<size_t>(bn) * gn * kv_head;
            cudaEvent_t ev_in = x.ev[2 * (n_chunk % kHostEvents)], ev_done = x.ev[2 * (n_chunk % kHostEvents) + 1];
            if (n_chunk >= kHostEvents) e = cudaEventSynchronize(x.ev[2 * (n_chunk % kHostEvents) + 1]);
            if (e == cudaSuccess) e = cudaMemcpyAsync(dbuf + qo, static_cast<const char *>(q) + qo, qn, cudaMemcpyHostToDevice, x.h2d);
            if (e == cudaSuccess && Skv > 0)
                e = cudaMemcpyAsync(dbuf + off_k + ko, static_cast<const char *>(k) + ko, kn, cudaMemcpyHostToDevice, x.h2d);
            if (e == cudaSuccess && Skv > 0)
                e = cudaMemcpyAsync(dbuf + off_v + ko, static_cast<const char *>(v) + ko, kn, cudaMemcpyHostToDevice, x.h2d);
            if (e == cudaSuccess) e = cudaEventRecord(ev_in, x.h2d);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_in, 0);
            if (e != cudaSuccess) break;
            rc = fwd_impl(dbuf + qo, dbuf + off_k + ko, dbuf + off_v + ko, dbuf + off_o + qo, nullptr, bn,
                          gn * G, gn, Sq, Skv, D, scale, causal, d_len ? d_len + b0 : nullptr, 0, dtype, st);
            if (rc) break;
            e = cudaEventRecord(ev_done, st);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(x.d2h, ev_done, 0);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(static_cast<char *>(out) + qo, dbuf + off_o + qo, qn, cudaMemcpyDeviceToHost, x.d2h);
            ++n_chunk;
        }
    }
    // the caller's stream resumes after the last copy out; the call returns when it is done
    cudaError_t e2 = cudaEventRecord(x.ev_end, x.d2h);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, x.ev_end, 0);
    if (e2 == cudaSuccess) e2 = cudaEventSynchronize(x.ev_end);
    if (rc) return rc;
    if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_host");
    if (e2 != cudaSuccess) return cuda_fail(e2, "attn_fwd_host (completion)");
    return ATTN_OK;
}

ATTN_API int attn_fwd_chunked(const void *q, const void *kcache, const void *vcache, void *out,
                              float *lse, int B, int H, int H_kv, int Sq, int Skv, int D, float scale,
                              const int32_t *cache_len, int dtype, void *stream) {
    return fwd_impl(q, kcache, vcache, out, lse, B, H, H_kv, Sq, Skv, D, scale, 1, cache_len, 1, dtype,
                    stream);
}

ATTN_API int attn_fwd_debug(const void *q, const void *k, const void *v, void *out, float *weights,
                            int B, int H, int H_kv, int Sq, int Skv, int Dk, int Dv, float scale,
                            int causal, const int32_t *kv_len, int dtype, void *stream) {
    g_last_error[0] = '\0';
    if (B < 1 || H < 1 || Sq < 0 || Skv < 0)
        return fail(ATTN_EINVAL, "attn_fwd_debug: need B >= 1, H >= 1, Sq >= 0, Skv >= 0");
    if (H_kv < 1 || H % H_kv != 0)
        return fail(ATTN_EINVAL, "attn_fwd_debug: H_kv must divide H (got H = %d, H_kv = %d)", H, H_kv);
    if (Dk < 1 || Dk > 256 || Dv < 1 || Dv > 256)
        return fail(ATTN_EINVAL, "attn_fwd_debug: Dk and Dv must be in [1, 256] (got %d, %d)", Dk, Dv);
    if (Skv > 16384) return fail(ATTN_EUNSUPPORTED, "attn_fwd_debug: Skv = %d above 16384", Skv);
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return fail(ATTN_EINVAL, "attn_fwd_debug: unknown dtype %d", dtype);
    if (!(scale >= 0.f) || isinf(scale)) return fail(ATTN_EINVAL, "attn_fwd_debug: scale must be finite and >= 0");
    if (causal != 0 && causal != 1) return fail(ATTN_EINVAL, "attn_fwd_debug: causal must be 0 or 1");
    if (causal && Sq > Skv) return fail(ATTN_EINVAL, "attn_fwd_debug: causal needs Sq <= Skv (got %d > %d)", Sq, Skv);
    if (kv_len && causal && Sq != Skv)
        return fail(ATTN_EINVAL, "attn_fwd_debug: causal kv_len needs Sq == Skv");
    if ((Sq > 0 && (!q || !out)) || (Skv > 0 && (!k || !v)))
        return fail(ATTN_EINVAL, "attn_fwd_debug: q and out (Sq > 0), k and v (Skv > 0) must not be NULL");
    const size_t esz = dtype == ATTN_BF16 ? 2 : 4;
    const uintptr_t amask = esz - 1;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(out)) & amask)
        return fail(ATTN_EINVAL, "attn_fwd_debug: tensors must be aligned to their element size");
    if ((kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) || (weights && (reinterpret_cast<uintptr_t>(weights) & 3u)))
        return fail(ATTN_EINVAL, "attn_fwd_debug: kv_len and weights must be 4-byte aligned");
    const long long rows = static_cast<long long>(B) * H * Sq;
    if (rows >= (1LL << 31)) return fail(ATTN_EINVAL, "attn_fwd_debug: B*H*Sq is too large");
    const long long bh_kv = static_cast<long long>(B) * H_kv;
    const size_t q_bytes = static_cast<size_t>(rows) * Dk * esz, o_bytes = static_cast<size_t>(rows) * Dv * esz;
    const size_t k_bytes = static_cast<size_t>(bh_kv) * Skv * Dk * esz, v_bytes = static_cast<size_t>(bh_kv) * Skv * Dv * esz;
    const size_t w_bytes = static_cast<size_t>(rows) * Skv * sizeof(float);
    if (overlaps(out, o_bytes, q, q_bytes) || overlaps(out, o_bytes, k, k_bytes) || overlaps(out, o_bytes, v, v_bytes) ||
        (weights && (overlaps(weights, w_bytes, q, q_bytes) || overlaps(weights, w_bytes, k, k_bytes) ||
                     overlaps(weights, w_bytes, v, v_bytes) || overlaps(weights, w_bytes, out, o_bytes))))
        return fail(ATTN_EINVAL, "attn_fwd_debug: out or weights overlaps another tensor");
    if (rows == 0) return ATTN_OK;
    DebugArgs a{q, k, v, out, weights, kv_len, B, H, H_kv, Sq, Skv, Dk, Dv, scale, causal,
                dtype == ATTN_BF16 ? 1 : 0, static_cast<cudaStream_t>(stream)};
    const cudaError_t e = launch_debug_attention(a);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_fwd_debug launch");
}

ATTN_API int attn_decode_splits(int B, int H, int Skv, int D) {
    if (B < 1 || H < 1 || Skv < 0 || (D != 64 && D != 128)) return ATTN_EINVAL;
    const int chunk = decode_chunk(B, H, Skv);
    const int n = (Skv + chunk - 1) / chunk;
    return n > 0 ? n : 1;
}

ATTN_API int attn_decode(const void *q, const void *kcache, const void *vcache, void *out, int B,
                         int H, int Skv, int D, const int32_t *kv_len, int dtype, void *stream) {
    return attn_decode_gqa(q, kcache, vcache, out, B, H, H, Skv, D, kv_len, dtype, stream);
}

ATTN_API int attn_decode_gqa(const void *q, const void *kcache, const void *vcache, void *out, int B,
                             int H, int H_kv, int Skv, int D, const int32_t *kv_len, int dtype,
                             void *stream) {
    g_last_error[0] = '\0';
    if (B < 1 || H < 1 || Skv < 0)
        return fail(ATTN_EINVAL, "attn_decode: need B >= 1, H >= 1, Skv >= 0 (got %d, %d, %d)", B, H, Skv);
    if (H_kv < 1 || H % H_kv != 0)
        return fail(ATTN_EINVAL, "attn_decode: H_kv must divide H (got H = %d, H_kv = %d)", H, H_kv);
    if (!q || !out || (Skv > 0 && (!kcache || !vcache)))
        return fail(ATTN_EINVAL, "attn_decode: q, out and (for Skv > 0) kcache, vcache must not be NULL");
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return fail(ATTN_EINVAL, "attn_decode: unknown dtype %d", dtype);
    if (D <= 0) return fail(ATTN_EINVAL, "attn_decode: D must be positive (got %d)", D);
    if (D != 64 && D != 128) return fail(ATTN_EUNSUPPORTED, "attn_decode: D = %d not supported (64 or 128)", D);
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
        return fail(ATTN_EINVAL, "attn_decode: q, kcache, vcache and out must be 16-byte aligned");
    if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u))
        return fail(ATTN_EINVAL, "attn_decode: kv_len must be 4-byte aligned");
    const long long bh = static_cast<long long>(B) * H;
    const long long bh_kv = static_cast<long long>(B) * H_kv;
    if (bh * (Skv > 1 ? Skv : 1) >= (1LL << 31) || bh >= (1LL << 31) / 64)
        return fail(ATTN_EINVAL, "attn_decode: B*H*Skv is too large");
    const size_t esz = dtype == ATTN_BF16 ? 2 : 4;
    const size_t qo_bytes = static_cast<size_t>(bh) * D * esz;
    const size_t kv_bytes = static_cast<size_t>(bh_kv) * Skv * D * esz;
    if (overlaps(out, qo_bytes, q, qo_bytes) || overlaps(out, qo_bytes, kcache, kv_bytes) ||
        overlaps(out, qo_bytes, vcache, kv_bytes))
        return fail(ATTN_EINVAL, "attn_decode: out overlaps an input");

    // bf16 with large query groups: the tensor-core kernel (the group's queries
    // are the rows of one tile); fp32: its own CUDA-core kernel
    const bool f32 = dtype == ATTN_F32;
    const int G = H / H_kv;
    const bool tc = !f32 && G >= kDecodeTcMinGroup && G <= 128 && bh_kv <= 65535;
    const int chunk = tc ? decode_tc_chunk(B, H_kv, Skv, num_sms())
                         : ((H_kv == H || f32) ? decode_chunk(B, H, Skv) : decode_chunk_gqa(B, H, H_kv, Skv));
    const int n_split = Skv > 0 ? (Skv + chunk - 1) / chunk : 1;
    const size_t o_bytes = static_cast<size_t>(bh) * n_split * D * sizeof(float);
    const size_t ml_bytes = static_cast<size_t>(bh) * n_split * 2 * sizeof(float);
    void *ws = nullptr;
    int rc = workspace(o_bytes + ml_bytes, static_cast<cudaStream_t>(stream), &ws);
    if (rc) return rc;
    int *status = nullptr;
    if ((rc = status_word(&status))) return rc;
    DecodeArgs a{q, kcache, vcache, out, kv_len, B, H, Skv, D, 1.0f / sqrtf(static_cast<float>(D)),
                 chunk, n_split, static_cast<float *>(ws),
                 reinterpret_cast<float *>(static_cast<char *>(ws) + o_bytes), status,
                 static_cast<cudaStream_t>(stream), H_kv};
    cudaError_t e;
    if (tc) {
        CUtensorMap tq, tk, tv;
        if (Skv > 0 && ((rc = make_map_rows(&tq, q, D, bh)) || (rc = make_map(&tk, kcache, D, Skv, bh_kv, 64)) ||
                        (rc = make_map(&tv, vcache, D, Skv, bh_kv, 64))))
            return rc;
        e = launch_decode_tc(a, tq, tk, tv);
    } else if (f32) {
        e = launch_decode_f32(a);
    } else {
        e = H_kv == H ? launch_decode(a) : launch_decode_gqa(a);
    }
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_decode launch");
}

ATTN_API int attn_decode_noalloc(const void *q, const void *kcache, const void *vcache, void *out, int B,
                                 int H, int Skv, int D, const int32_t *kv_len, int dtype, void *stream) {
    g_last_error[0] = '\0';
    if (B < 1 || H < 1 || Skv < 0)
        return fail(ATTN_EINVAL, "attn_decode_noalloc: need B >= 1, H >= 1, Skv >= 0 (got %d, %d, %d)", B, H, Skv);
    if (!q || !out || (Skv > 0 && (!kcache || !vcache)))
        return fail(ATTN_EINVAL, "attn_decode_noalloc: q, out and (for Skv > 0) kcache, vcache must not be NULL");
    if (dtype != ATTN_F32 && dtype != ATTN_BF16)
        return fail(ATTN_EINVAL, "attn_decode_noalloc: unknown dtype %d", dtype);
    if (D <= 0) return fail(ATTN_EINVAL, "attn_decode_noalloc: D must be positive (got %d)", D);
    if (D != 64 && D != 128)
        return fail(ATTN_EUNSUPPORTED, "attn_decode_noalloc: D = %d not supported (64 or 128)", D);
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
        return fail(ATTN_EINVAL, "attn_decode_noalloc: q, kcache, vcache and out must be 16-byte aligned");
    if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u))
        return fail(ATTN_EINVAL, "attn_decode_noalloc: kv_len must be 4-byte aligned");
    const long long bh = static_cast<long long>(B) * H;
    if (bh * (Skv > 1 ? Skv : 1) >= (1LL << 31) || bh >= (1LL << 31) / 64)
        return fail(ATTN_EINVAL, "attn_decode_noalloc: B*H*Skv is too large");
    const size_t esz = dtype == ATTN_BF16 ? 2 : 4;
    const size_t qo_bytes = static_cast<size_t>(bh) * D * esz;
    const size_t kv_bytes = static_cast<size_t>(bh) * Skv * D * esz;
    if (overlaps(out, qo_bytes, q, qo_bytes) || overlaps(out, qo_bytes, kcache, kv_bytes) ||
        overlaps(out, qo_bytes, vcache, kv_bytes))
        return fail(ATTN_EINVAL, "attn_decode_noalloc: out overlaps an input");
    const int chunk = decode_chunk(B, H, Skv);
    const int n_split = attn_decode_splits(B, H, Skv, D);
    const size_t need = static_cast<size_t>(bh) * n_split * (D + 2) * sizeof(float);
    if (need > kDecodeNoAllocScratchBytes)
        return fail(ATTN_EINVAL,
                    "attn_decode_noalloc: these sizes need %zu bytes of scratch; the library's fixed "
                    "scratch holds %zu (use attn_decode, or fewer sequences per call)",
                    need, kDecodeNoAllocScratchBytes);
    int *status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    DecodeArgs a{q, kcache, vcache, out, kv_len, B, H, Skv, D, 1.0f / sqrtf(static_cast<float>(D)),
                 chunk, n_split, nullptr, nullptr, status, static_cast<cudaStream_t>(stream), H};
    cudaError_t e = launch_decode_noalloc(a, dtype == ATTN_F32);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_decode_noalloc launch");
}

ATTN_API int attn_device_status(void *stream) {
    g_last_error[0] = '\0';
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_device_status: stream synchronize");
    int *status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    int word = 0;
    e = cudaMemcpy(&word, status, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "attn_device_status: read status word");
    if (word == 0) return ATTN_OK;
    const int zero = 0;
    e = cudaMemcpy(status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "attn_device_status: clear status word");
    if ((word & 0xff) == kStatusSchedConflict)
        return fail(ATTN_ECONFLICT,
                    "two bf16 prefill launches in flight shared one work counter (site 0x%x); "
                    "their outputs are undefined", word >> 8);
    return fail(ATTN_ETIMEOUT, "a device-side wait gave up (site 0x%x); that call's output is undefined",
                word >> 8);
}

ATTN_API int attn_selftest_wait_timeout(long long limit_cycles, void *stream) {
    g_last_error[0] = '\0';
    if (limit_cycles < 0 || limit_cycles > kWaitLimitCycles)
        return fail(ATTN_EINVAL, "attn_selftest_wait_timeout: limit must be in [0, %lld] cycles", kWaitLimitCycles);
    int *status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    cudaError_t e = launch_wait_timeout_probe(limit_cycles, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_selftest_wait_timeout launch");
}

ATTN_API void attn_release(void) {
    int dev;
    if (current_device(&dev)) return;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        Workspace &w = g_ws[dev];
        if (w.ptr) cudaFree(w.ptr);
        for (int i = 0; i < w.n_retired; ++i) cudaFree(w.retired[i]);
        w.ptr = nullptr;
        w.bytes = 0;
        w.n_retired = 0;
    }
    // outside g_mutex: attn_fwd_host takes its own lock first, then g_mutex
    g_host[dev].release();
    // work counters that a conflict (ATTN_ECONFLICT) may have left unbalanced
    reset_prefill_counters();
}

}  // extern "C"

namespace attn {

namespace {
// Waits on an mbarrier phase that nothing completes, with a short limit, so
// that the timeout path (abort flag, status word) runs without a hang.
__global__ void wait_timeout_probe_kernel(long long limit, int *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, limit)) report_timeout(status, 0x7f);
    __syncthreads();
    if (threadIdx.x == 0) mbar_arrive(&bar);  // complete the phase before the CTA exits
}

__global__ void zero_fill_kernel(uint4 *out, size_t n) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        out[i] = make_uint4(0, 0, 0, 0);
}
}  // namespace

cudaError_t launch_wait_timeout_probe(long long limit, int *status, cudaStream_t stream) {
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(limit, status);
    return cudaGetLastError();
}

cudaError_t launch_zero_fill(void *out, size_t n_bytes, cudaStream_t stream) {
    const size_t n = n_bytes / 16;
    if (n == 0) return cudaSuccess;
    size_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<uint4 *>(out), n);
    return cudaGetLastError();
}

}  // namespace attn
