// Debug attention: the general form of "Attention from Scratch" (kube-dojo),
// Part 2 -- T_q query positions, T_k key/value positions, value depth d_v that
// may differ from the query/key depth d_k -- returning the attention weights
// as well as the output (Part 4 "Self-Attention, Cross-Attention, and
// Attention Maps"; Part 7 shape tests with T_target = 4, T_source = 7).
//
// One warp per query row, fp32 arithmetic, the row's scores held in shared
// memory: meant for inspection-sized problems, not for speed.  Masks, padded
// and all-masked rows follow the library's rules (include/attn.h).
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

template <typename T>
__device__ __forceinline__ float ld(const T *p, size_t i);
template <>
__device__ __forceinline__ float ld<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void st(T *p, size_t i, float x);
template <>
__device__ __forceinline__ void st<float>(float *p, size_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(32) debug_attention_kernel(const DebugArgs a) {
    extern __shared__ float dsm[];  // [Dk] query row, then [Skv] scores / weights
    float *qs = dsm;
    float *sw = dsm + a.Dk;
    const int lane = threadIdx.x;
    const long long row = blockIdx.x;  // (b * H + h) * Sq + i
    const int i = static_cast<int>(row % a.Sq);
    const long long bh = row / a.Sq;
    const int b = static_cast<int>(bh / a.H), h = static_cast<int>(bh % a.H);
    const long long bh_kv = static_cast<long long>(b) * a.H_kv + h / (a.H / a.H_kv);
    const T *q = static_cast<const T *>(a.q) + static_cast<size_t>(row) * a.Dk;
    const T *k = static_cast<const T *>(a.k) + static_cast<size_t>(bh_kv) * a.Skv * a.Dk;
    const T *v = static_cast<const T *>(a.v) + static_cast<size_t>(bh_kv) * a.Skv * a.Dv;
    T *out = static_cast<T *>(a.out) + static_cast<size_t>(row) * a.Dv;
    float *w = a.weights ? a.weights + static_cast<size_t>(row) * a.Skv : nullptr;

    int L = a.Skv;
    if (a.kv_len) L = min(max(a.kv_len[b], 0), a.Skv);
    // visible keys: j < L, and j <= i + (Skv - Sq) when causal; a padded query
    // row of a self-attention batch (Sq == Skv, i >= L) sees none
    int lim = L;
    if (a.causal) lim = min(lim, i + (a.Skv - a.Sq) + 1);
    if (a.kv_len && a.Sq == a.Skv && i >= L) lim = 0;
    lim = max(lim, 0);

    for (int d = lane; d < a.Dk; d += 32) qs[d] = ld(q, d);
    __syncwarp();
    float m = -INFINITY;
    for (int j = lane; j < lim; j += 32) {
        float dot = 0.f;
        for (int d = 0; d < a.Dk; ++d) dot = fmaf(qs[d], ld(k, static_cast<size_t>(j) * a.Dk + d), dot);
        const float s = dot * a.scale;
        sw[j] = s;
        m = fmaxf(m, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
    for (int j = lane; j < lim; j += 32) {
        const float p = expf(sw[j] - m);
        sw[j] = p;
        z += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv = lim > 0 ? 1.f / z : 0.f;
    for (int j = lane; j < a.Skv; j += 32) {
        const float p = j < lim ? sw[j] * inv : 0.f;
        if (j < lim) sw[j] = p;
        if (w) w[j] = p;
    }
    __syncwarp();
    for (int d = lane; d < a.Dv; d += 32) {
        float acc = 0.f;
        for (int j = 0; j < lim; ++j) acc = fmaf(sw[j], ld(v, static_cast<size_t>(j) * a.Dv + d), acc);
        st(out, d, acc);
    }
}

}  // namespace

cudaError_t launch_debug_attention(const DebugArgs &a) {
    const long long rows = static_cast<long long>(a.B) * a.H * a.Sq;
    if (rows <= 0) return cudaSuccess;
    const size_t smem = (static_cast<size_t>(a.Dk) + a.Skv) * sizeof(float);
    cudaError_t e;
    if (a.dtype_bf16) {
        e = cudaFuncSetAttribute(debug_attention_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        debug_attention_kernel<__nv_bfloat16><<<static_cast<unsigned>(rows), 32, smem, a.stream>>>(a);
    } else {
        e = cudaFuncSetAttribute(debug_attention_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        debug_attention_kernel<float><<<static_cast<unsigned>(rows), 32, smem, a.stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace attn
