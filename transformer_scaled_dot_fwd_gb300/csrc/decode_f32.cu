// fp32 decode: one query per (batch, head) against an fp32 KV cache.
//
// The same split-KV computation as the bf16 decode ("Attention from First
// Principles", section 6 "Under the hood": a matrix-vector product over the
// cache), in fp32 on the CUDA cores: the tensor cores' fp32 input path (TF32,
// 10-bit mantissa) would not keep the 1e-4 tolerance.  Query head h reads
// cached head h / (H / H_kv) (grouped-query attention, "Scaled dot-product
// attention with masking", "Grouped-query attention (GQA)").
//
//   partial kernel  one CTA (4 warps) per (b, h, chunk of `chunk` keys):
//                   scores with 8 lanes per key (float4 loads of the key
//                   row), the chunk max m_c (log2 units), p_j = 2^(s_j - m_c),
//                   l_c and o_c = sum p_j v_j written as fp32 partials.  Keys
//                   j >= kv_len[b] are never loaded.
//   combine kernel  per (b, h): the exact max-shifted merge of the chunks,
//                   written as fp32; kv_len[b] == 0 gives zeros.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kF32Warps = 4;
constexpr int kF32Threads = kF32Warps * 32;
constexpr float kF32Log2e = 1.4426950408889634f;

template <int D>
__global__ void __launch_bounds__(kF32Threads) decode_f32_partial_kernel(DecodeArgs a) {
    griddep_launch_dependents();  // the combine may be placed once every CTA has started
    griddep_wait();               // launched back to back: the previous kernel's writes are visible
    __shared__ float s[kDecodeMaxChunk];  // scores, then probabilities, of the chunk
    __shared__ float red[kF32Warps][D];
    __shared__ float wred[kF32Warps];

    const int bh = blockIdx.x / a.n_split;
    const int c = blockIdx.x % a.n_split;
    const int b = bh / a.H, h = bh % a.H;
    const size_t bh_kv = static_cast<size_t>(b) * a.H_kv + h / (a.H / a.H_kv);
    int L = a.Skv;
    if (a.kv_len) L = min(max(a.kv_len[b], 0), a.Skv);
    const int k0 = c * a.chunk;
    if (k0 >= L) return;  // the combine reads only chunks below L
    const int nkeys = min(a.chunk, L - k0);
    const float *K = static_cast<const float *>(a.k) + (bh_kv * a.Skv + k0) * D;
    const float *V = static_cast<const float *>(a.v) + (bh_kv * a.Skv + k0) * D;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    // ---- scores: 8 lanes per key, 4 keys per warp step; lane t8 of group g
    // holds dims [4 t8 + 32 u, 4 t8 + 32 u + 4) of the query and of key g
    constexpr int NU = D / 32;
    const int g = lane / 8, t8 = lane % 8;
    float4 qf[NU];
    {
        const float sl2 = a.scale * kF32Log2e;
        const float4 *qp = reinterpret_cast<const float4 *>(static_cast<const float *>(a.q) + static_cast<size_t>(bh) * D);
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const float4 v = qp[u * 8 + t8];
            qf[u] = make_float4(v.x * sl2, v.y * sl2, v.z * sl2, v.w * sl2);
        }
    }
    for (int kb = warp * 4; kb < nkeys; kb += 4 * kF32Warps) {
        const int key = kb + g;
        float part = 0.f;
        if (key < nkeys) {
            const float4 *kp = reinterpret_cast<const float4 *>(K + static_cast<size_t>(key) * D);
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const float4 kv = kp[u * 8 + t8];
                part = fmaf(qf[u].x, kv.x, part);
                part = fmaf(qf[u].y, kv.y, part);
                part = fmaf(qf[u].z, kv.z, part);
                part = fmaf(qf[u].w, kv.w, part);
            }
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        part += __shfl_xor_sync(0xffffffffu, part, 4);
        if (t8 == 0 && key < nkeys) s[key] = part;
    }
    __syncthreads();

    // ---- chunk max and p_j = 2^(s_j - m_c), l_c = sum p_j
    float mx = -INFINITY;
    for (int j = tid; j < nkeys; j += kF32Threads) mx = fmaxf(mx, s[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) wred[warp] = mx;
    __syncthreads();
    float m_c = wred[0];
#pragma unroll
    for (int w = 1; w < kF32Warps; ++w) m_c = fmaxf(m_c, wred[w]);
    float lsum = 0.f;
    for (int j = tid; j < nkeys; j += kF32Threads) {
        const float p = ex2_approx(s[j] - m_c);
        s[j] = p;
        lsum += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    __syncthreads();  // every p written; wred[] free again
    if (lane == 0) wred[warp] = lsum;

    // ---- o_c = sum p_j v_j: lane owns dims [DPL lane, DPL lane + DPL); warp w keys w, w + 4, ...
    constexpr int DPL = D / 32;
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    for (int key = warp; key < nkeys; key += kF32Warps) {
        const float p = s[key];
        const float *vp = V + static_cast<size_t>(key) * D + lane * DPL;
        if constexpr (DPL == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(vp);
            acc[0] = fmaf(p, v.x, acc[0]);
            acc[1] = fmaf(p, v.y, acc[1]);
            acc[2] = fmaf(p, v.z, acc[2]);
            acc[3] = fmaf(p, v.w, acc[3]);
        } else {
            const float2 v = *reinterpret_cast<const float2 *>(vp);
            acc[0] = fmaf(p, v.x, acc[0]);
            acc[1] = fmaf(p, v.y, acc[1]);
        }
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) red[warp][lane * DPL + e] = acc[e];
    __syncthreads();
    const size_t part = static_cast<size_t>(bh) * a.n_split + c;
    for (int d = tid; d < D; d += kF32Threads) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kF32Warps; ++w) sum += red[w][d];
        a.part_o[part * D + d] = sum;
    }
    if (tid == 0) {
        float l_c = 0.f;
#pragma unroll
        for (int w = 0; w < kF32Warps; ++w) l_c += wred[w];
        a.part_ml[part * 2 + 0] = m_c;
        a.part_ml[part * 2 + 1] = l_c;
    }
}

template <int D>
__global__ void __launch_bounds__(D) decode_f32_combine_kernel(DecodeArgs a) {
    griddep_wait();  // the partial kernel's results
    const int bh = blockIdx.x;
    const int d = threadIdx.x;
    const int b = bh / a.H;
    int L = a.Skv;
    if (a.kv_len) L = min(max(a.kv_len[b], 0), a.Skv);
    const int nv = (L + a.chunk - 1) / a.chunk;  // chunks holding at least one key
    float *out = static_cast<float *>(a.out) + static_cast<size_t>(bh) * D;
    if (nv == 0) {
        out[d] = 0.f;
        return;
    }
    const float *ml = a.part_ml + static_cast<size_t>(bh) * a.n_split * 2;
    const float *po = a.part_o + static_cast<size_t>(bh) * a.n_split * D;
    float M = -INFINITY;
    for (int cc = 0; cc < nv; ++cc) M = fmaxf(M, ml[2 * cc]);
    float acc = 0.f, lsum = 0.f;
    for (int cc = 0; cc < nv; ++cc) {
        const float w = ex2_approx(ml[2 * cc] - M);
        acc = fmaf(w, po[static_cast<size_t>(cc) * D + d], acc);
        lsum = fmaf(w, ml[2 * cc + 1], lsum);
    }
    out[d] = acc / lsum;
}

template <int D>
cudaError_t launch_f32_t(const DecodeArgs &a) {
    if (a.Skv > 0) {
        const long long blocks = static_cast<long long>(a.B) * a.H * a.n_split;
        const cudaError_t e = launch_pdl(decode_f32_partial_kernel<D>, dim3(static_cast<unsigned>(blocks)),
                                         dim3(kF32Threads), 0, a.stream, a);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(decode_f32_combine_kernel<D>, dim3(static_cast<unsigned>(a.B * a.H)), dim3(D), 0, a.stream, a);
}

}  // namespace

cudaError_t launch_decode_f32(const DecodeArgs &a) {
    return a.D == 64 ? launch_f32_t<64>(a) : launch_f32_t<128>(a);
}

}  // namespace attn
