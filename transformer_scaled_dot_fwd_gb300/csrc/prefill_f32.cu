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
// shuffles.  K and V tiles of 32 keys are staged in shared memory, double-
// buffered: the next tile's asynchronous copies (cp.async, zero-filled past
// the keys the CTA needs) are in flight while this tile is computed.
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
constexpr int f32_smem_bytes() { return 2 * 2 * kKeys * D * 4; }  // [stage][K, V][key][D]

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int D>
__global__ void __launch_bounds__(kThreads) prefill_f32_kernel(FwdArgs a) {
    constexpr int DL = D / kLanesPerRow;
    griddep_launch_dependents();
    griddep_wait();  // launched back to back: the previous kernel's writes are visible
    extern __shared__ __align__(16) float f32_smem[];
    // stage st: keys ks(st)[kKeys][D], values vs(st)[kKeys][D]
    auto ks = [&](int st) { return f32_smem + (2 * st) * kKeys * D; };
    auto vs = [&](int st) { return f32_smem + (2 * st + 1) * kKeys * D; };

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

    // tile j0's keys and values into stage st; rows past cta_lim are zeros
    auto load_tile = [&](int j0, int st) {
        const uint32_t kd = static_cast<uint32_t>(__cvta_generic_to_shared(ks(st)));
        const uint32_t vd = static_cast<uint32_t>(__cvta_generic_to_shared(vs(st)));
        for (int idx = threadIdx.x; idx < kKeys * D / 4; idx += kThreads) {
            const int row = idx / (D / 4);
            const bool in = j0 + row < cta_lim;
            const size_t src = static_cast<size_t>(in ? j0 + row : 0) * D + 4 * (idx % (D / 4));
            cp_async16(kd + 16u * idx, K + src, in ? 16u : 0u);
            cp_async16(vd + 16u * idx, V + src, in ? 16u : 0u);
        }
        cp_async_commit();
    };
    const int n_tiles = (cta_lim + kKeys - 1) / kKeys;
    if (n_tiles > 0) load_tile(0, 0);
    for (int tile = 0; tile < n_tiles; ++tile) {
        const int j0 = tile * kKeys;
        const int st = tile & 1;
        if (tile + 1 < n_tiles) {
            load_tile(j0 + kKeys, st ^ 1);  // its stage was last read before the previous barrier
            cp_async_wait<1>();              // this tile's copies have landed
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float *kt = ks(st), *vt = vs(st);

        float s[kKeys];
        float mt = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kKeys; ++jj) {
            float part = 0.f;
#pragma unroll
            for (int d = 0; d < DL; ++d) part = fmaf(q[d], kt[jj * D + d * kLanesPerRow + t], part);
#pragma unroll
            for (int o16 = 1; o16 < kLanesPerRow; o16 <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o16);
            s[jj] = (j0 + jj < lim) ? part * sl2 : -INFINITY;
            mt = fmaxf(mt, s[jj]);
        }
        const float mn = fmaxf(m, mt);
        if (mn != -INFINITY) {  // else nothing is visible to this row yet
            const float corr = ex2_approx(m - mn);  // 2^-inf = 0 on the first visible tile
            l *= corr;
#pragma unroll
            for (int d = 0; d < DL; ++d) o[d] *= corr;
#pragma unroll
            for (int jj = 0; jj < kKeys; ++jj) {
                const float p = ex2_approx(s[jj] - mn);  // masked keys: 2^-inf = 0
                l += p;
#pragma unroll
                for (int d = 0; d < DL; ++d) o[d] = fmaf(p, vt[jj * D + d * kLanesPerRow + t], o[d]);
            }
            m = mn;
        }
        __syncthreads();  // every thread is done with stage st before it is refilled
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

template <int D>
cudaError_t launch_f32_t(const FwdArgs &a) {
    const dim3 grid((a.Sq + kRows - 1) / kRows, a.H, a.B);
    cudaError_t e = cudaFuncSetAttribute(prefill_f32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         f32_smem_bytes<D>());
    if (e != cudaSuccess) return e;
    return launch_pdl(prefill_f32_kernel<D>, grid, dim3(kThreads), f32_smem_bytes<D>(), a.stream, a);
}

}  // namespace

cudaError_t launch_prefill_f32(const FwdArgs &a) {
    return a.D == 64 ? launch_f32_t<64>(a) : launch_f32_t<128>(a);
}

}  // namespace attn
