// fp32 prefill attention on the CUDA cores (FFMA only, no TF32).
//
// Computes softmax(Q K^T * scale + M) V per (batch, head) in float32 with an
// online (streaming) row softmax, for the fp32 workloads whose tolerance
// (1e-4 absolute) TF32's 10-bit mantissa could not meet.  Masking follows
// "Attention from Scratch" (kube-dojo), Part 3 (causal AND key padding,
// applied before the softmax); rows that see no key and padded query rows are
// written as zeros.
//
// Work split: one CTA per (8 query rows, head, batch), so that even the small
// fp32 workload (B2 H4 S128) spreads over 128 CTAs.  Sixteen threads share a
// query row, each holding every sixteenth element of q and of the output row
// in registers; a score is a 16-way partial dot product summed with four lane
// shuffles.  K and V tiles of 32 keys are staged in shared memory.
#include "kernels.h"
#include "ptx.cuh"

#include <math.h>

namespace attn {
namespace {

constexpr int kRows = 8;          // query rows per CTA
constexpr int kLanesPerRow = 16;  // threads sharing one query row
constexpr int kThreads = kRows * kLanesPerRow;
constexpr int kKeys = 32;         // keys per shared-memory tile
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
__global__ void __launch_bounds__(kThreads) prefill_f32_kernel(FwdArgs a) {
    constexpr int DL = D / kLanesPerRow;
    __shared__ __align__(16) float ks[kKeys][D];
    __shared__ __align__(16) float vs[kKeys][D];

    const int t = threadIdx.x % kLanesPerRow;
    const int r = threadIdx.x / kLanesPerRow;
    const int b = blockIdx.z, h = blockIdx.y;
    const int i = blockIdx.x * kRows + r;
    const size_t bh = static_cast<size_t>(b) * a.H + h;
    const size_t bh_kv = static_cast<size_t>(b) * a.H_kv + h / (a.H / a.H_kv);  // grouped-query head
    const float *Q = static_cast<const float *>(a.q) + bh * a.Sq * D;
    const float *K = static_cast<const float *>(a.k) + bh_kv * a.Skv * D;
    const float *V = static_cast<const float *>(a.v) + bh_kv * a.Skv * D;
    float *O = static_cast<float *>(a.out) + bh * a.Sq * D;

    int L = a.Skv;
    if (a.kv_len) L = min(max(a.kv_len[b], 0), a.Skv);
    // causal: key j visible from query i iff j <= i + off
    const int off = a.chunked ? L - a.Sq : a.Skv - a.Sq;
    const bool row_valid = i < a.Sq && !(!a.chunked && a.kv_len && a.Sq == a.Skv && i >= L);
    int lim = L;                   // keys [0, lim) are visible from row i
    if (a.causal) lim = min(lim, i + off + 1);
    if (!row_valid) lim = 0;
    const int last_row = min(a.Sq - 1, static_cast<int>(blockIdx.x) * kRows + kRows - 1);
    int cta_lim = L;               // keys any row of this CTA can see
    if (a.causal) cta_lim = min(cta_lim, last_row + off + 1);

    float q[DL], o[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) {
        q[d] = i < a.Sq ? Q[static_cast<size_t>(i) * D + d * kLanesPerRow + t] : 0.f;
        o[d] = 0.f;
    }
    const float sl2 = a.scale * kLog2e;  // scores kept in log2 units
    float m = -INFINITY, l = 0.f;

    for (int j0 = 0; j0 < cta_lim; j0 += kKeys) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kKeys * D / 4; idx += kThreads) {
            const int row = idx / (D / 4), c4 = idx % (D / 4);
            float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
            if (j0 + row < cta_lim) {
                kk = reinterpret_cast<const float4 *>(K + static_cast<size_t>(j0 + row) * D)[c4];
                vv = reinterpret_cast<const float4 *>(V + static_cast<size_t>(j0 + row) * D)[c4];
            }
            reinterpret_cast<float4 *>(ks[row])[c4] = kk;
            reinterpret_cast<float4 *>(vs[row])[c4] = vv;
        }
        __syncthreads();

        float s[kKeys];
        float mt = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kKeys; ++jj) {
            float part = 0.f;
#pragma unroll
            for (int d = 0; d < DL; ++d) part = fmaf(q[d], ks[jj][d * kLanesPerRow + t], part);
#pragma unroll
            for (int o16 = 1; o16 < kLanesPerRow; o16 <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o16);
            s[jj] = (j0 + jj < lim) ? part * sl2 : -INFINITY;
            mt = fmaxf(mt, s[jj]);
        }
        const float mn = fmaxf(m, mt);
        if (mn == -INFINITY) continue;  // nothing visible to this row yet
        const float corr = exp2f(m - mn);
        l *= corr;
#pragma unroll
        for (int d = 0; d < DL; ++d) o[d] *= corr;
#pragma unroll
        for (int jj = 0; jj < kKeys; ++jj) {
            const float p = exp2f(s[jj] - mn);
            l += p;
#pragma unroll
            for (int d = 0; d < DL; ++d) o[d] = fmaf(p, vs[jj][d * kLanesPerRow + t], o[d]);
        }
        m = mn;
    }

    if (i < a.Sq) {
        const bool seen = row_valid && l > 0.f;
        const float inv = seen ? 1.f / l : 0.f;
#pragma unroll
        for (int d = 0; d < DL; ++d) O[static_cast<size_t>(i) * D + d * kLanesPerRow + t] = o[d] * inv;
        // log(sum_j exp(scale * s_j)) = ln 2 * (m + log2 l), m and l in log2 units
        if (a.lse && t == 0) a.lse[bh * a.Sq + i] = seen ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_prefill_f32(const FwdArgs &a) {
    dim3 grid((a.Sq + kRows - 1) / kRows, a.H, a.B);
    if (a.D == 64)
        prefill_f32_kernel<64><<<grid, kThreads, 0, a.stream>>>(a);
    else
        prefill_f32_kernel<128><<<grid, kThreads, 0, a.stream>>>(a);
    return cudaGetLastError();
}

}  // namespace attn
