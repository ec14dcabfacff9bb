// bf16 prefill attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes out = softmax(Q K^T * scale + M) V per (batch, head) ("Attention
// from First Principles", section 5 "The full multi-head computation"), with
// the causal and key-padding masks of "Attention from Scratch" (kube-dojo),
// Part 3, without ever writing the score matrix to HBM: the tiled, exact
// scheme the pages name as FlashAttention ("Scaled dot-product attention with
// masking", "The memory problem"), redesigned here for Blackwell.
//
// One CTA owns two 128-row query tiles (Q0, Q1) of one (b, h) and streams the
// 128-key K/V tiles they need through shared memory.  Roles:
//   warp 0      TMA producer: Q0/Q1 once, then K_j, V_j into a ring of
//               32 KB stages (128-byte swizzle, 64-column boxes).
//   warp 1      allocates 512 TMEM columns; lane 0 issues every MMA:
//                 S_x = Q_x K_j^T        (SS: both operands in shared memory)
//                 O_x += P_x V_j         (TS: P read from TMEM, V MN-major)
//               in the order S0_0 S1_0 | PV0_j S0_{j+1} PV1_j S1_{j+1} | ...
//               so each softmax warpgroup has two MMA slots to hide behind.
//   warps 2-5   softmax for Q0, warps 6-9 for Q1: thread = query row = TMEM
//               lane.  Load the 128 fp32 scores of the row, mask (only on
//               tiles that cross the causal diagonal or the padding edge),
//               online max/sum in log2 units, p = 2^(s*scale*log2e - m),
//               write p as bf16 over the S columns for the TS MMA.  O is
//               rescaled lazily, only when the running max grows by more
//               than 2^8, so most tiles never touch O.
//   epilogue    the same warps: O / l -> bf16 -> global; rows with no visible
//               key and padded query rows are written as exact zeros.
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D, 256+2D);
// P_x aliases the first 64 columns of S_x.
// KV tiles wholly above the causal diagonal or past kv_len are never loaded.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;       // query rows per Q tile (one TMEM lane each)
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kQTiles = 2;     // Q tiles per CTA
constexpr int kThreads = 320;  // 10 warps
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold (log2 units)

template <int D>
struct Layout {
    static constexpr int kSub = D / 64;                    // 128-byte column blocks per row
    static constexpr int kBlockBytes = 128 * 128;          // one block of a 128-row tile
    static constexpr int kTileBytes = kSub * kBlockBytes;  // 32 KB at D = 128
    static constexpr int kStages = D == 128 ? 4 : 8;       // K/V ring depth
    static constexpr int kRingOff = kQTiles * kTileBytes;
    static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
    static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // + barriers + alignment slack
    // TMEM column of S_x (and of P_x, which aliases it) and of O_x
    static __device__ __forceinline__ uint32_t s_col(int x) { return static_cast<uint32_t>(x) * 128u; }
    static __device__ __forceinline__ uint32_t o_col(int x) { return 256u + static_cast<uint32_t>(x) * D; }
};

struct Bars {
    uint64_t q_full;
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t s_full[2];
    uint64_t p_ready[2];
    uint64_t o_full[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const int n_pairs) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem + L::kRingOff;
    Bars &bars = *reinterpret_cast<Bars *>(smem + L::kBarOff);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // ---- work unit: longest query-tile pairs first (causal cost grows with the row)
    const int BH = a.B * a.H;
    const int pair = n_pairs - 1 - static_cast<int>(blockIdx.x) / BH;
    const int bh = static_cast<int>(blockIdx.x) % BH;
    const int b = bh / a.H;
    int Lb = a.Skv;
    if (a.kv_len) Lb = min(max(a.kv_len[b], 0), a.Skv);
    const int off = a.Skv - a.Sq;  // causal: key j visible from query i iff j <= i + off
    int n_kv[kQTiles];             // K/V tiles each Q tile needs
#pragma unroll
    for (int x = 0; x < kQTiles; ++x) {
        const int row0 = (pair * kQTiles + x) * kBM;
        n_kv[x] = 0;
        if (row0 < a.Sq && !(a.kv_len && row0 >= Lb)) {
            int last = min(a.Sq - 1, row0 + kBM - 1);
            if (a.kv_len) last = min(last, Lb - 1);
            const int hi = a.causal ? min(Lb, last + off + 1) : Lb;
            n_kv[x] = (hi + kBN - 1) / kBN;
        }
    }
    const int N = max(n_kv[0], n_kv[1]);

    if (threadIdx.x == 0) {
        mbar_init(&bars.q_full, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&bars.kv_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int x = 0; x < kQTiles; ++x) {
            mbar_init(&bars.s_full[x], 1);
            mbar_init(&bars.p_ready[x], 128);
            mbar_init(&bars.o_full[x], 1);
        }
        mbar_init(&bars.mma_done, 1);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0 && N > 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            uint32_t qbytes = 0;
#pragma unroll
            for (int x = 0; x < kQTiles; ++x) qbytes += n_kv[x] > 0 ? L::kTileBytes : 0;
            mbar_arrive_expect_tx(&bars.q_full, qbytes);
#pragma unroll
            for (int x = 0; x < kQTiles; ++x)
                if (n_kv[x] > 0)
#pragma unroll
                    for (int c = 0; c < L::kSub; ++c)
                        tma_load_3d(smem + x * L::kTileBytes + c * L::kBlockBytes, &tq, &bars.q_full,
                                    c * 64, (pair * kQTiles + x) * kBM, bh);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < N && ok; ++j) {
                for (int kv = 0; kv < 2; ++kv) {  // K_j, then V_j
                    const int slot = issued % L::kStages;
                    if (issued >= L::kStages &&
                        !mbar_wait(&bars.kv_empty[slot], ((issued / L::kStages) - 1) & 1, &bars.abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars.kv_full[slot], L::kTileBytes);
#pragma unroll
                    for (int c = 0; c < L::kSub; ++c)
                        tma_load_3d(ring + slot * L::kTileBytes + c * L::kBlockBytes, kv ? &tv : &tk,
                                    &bars.kv_full[slot], c * 64, j * kBN, bh);
                    ++issued;
                }
            }
            // never leave with copies still landing in shared memory
            volatile int never = 0;
            mbar_wait(&bars.q_full, 0, &never);
            for (int u = max(0, issued - L::kStages); u < issued; ++u)
                mbar_wait(&bars.kv_full[u % L::kStages], (u / L::kStages) & 1, &never);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0 && N > 0) {
            const uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0);
            const uint32_t idesc_o = idesc_bf16_f32(kBM, D, 1);
            const uint32_t q_addr = smem_u32(smem), ring_addr = smem_u32(ring);
            auto issue_s = [&](int x, int slot) {
                const uint32_t qa = q_addr + x * L::kTileBytes;
                const uint32_t ka = ring_addr + slot * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk / 4) * L::kBlockBytes + (kk % 4) * 32;
                    mma_ss(tmem + L::s_col(x), sdesc_sw128(qa + koff, 16, 1024),
                           sdesc_sw128(ka + koff, 16, 1024), idesc_s, kk > 0);
                }
            };
            auto issue_pv = [&](int x, int slot, bool acc) {
                const uint32_t va = ring_addr + slot * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(tmem + L::o_col(x), tmem + L::s_col(x) + kk * 8,
                           sdesc_sw128(va + kk * 16 * 128, L::kBlockBytes, 1024), idesc_o,
                           (acc || kk > 0) ? 1u : 0u);
            };
            int consumed = 0;
            uint32_t pr[2] = {0, 0};
            bool ok = mbar_wait(&bars.q_full, 0, &bars.abort);
            if (ok) {
                const int kslot = consumed % L::kStages;
                ok = mbar_wait(&bars.kv_full[kslot], (consumed / L::kStages) & 1, &bars.abort);
                ++consumed;
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int x = 0; x < kQTiles; ++x)
                        if (n_kv[x] > 0) {
                            issue_s(x, kslot);
                            tc_commit(&bars.s_full[x]);
                        }
                    tc_commit(&bars.kv_empty[kslot]);
                }
            }
            for (int j = 0; j < N && ok; ++j) {
                const int vslot = consumed % L::kStages;
                if (!(ok = mbar_wait(&bars.kv_full[vslot], (consumed / L::kStages) & 1, &bars.abort))) break;
                ++consumed;
                tc_fence_after();
                if (j < n_kv[0]) {
                    if (!(ok = mbar_wait(&bars.p_ready[0], pr[0], &bars.abort))) break;
                    pr[0] ^= 1;
                    tc_fence_after();
                    issue_pv(0, vslot, j > 0);
                    if (j == n_kv[0] - 1) tc_commit(&bars.o_full[0]);
                }
                const bool next = j + 1 < N;
                int nslot = 0;
                if (next) {
                    nslot = consumed % L::kStages;
                    if (!(ok = mbar_wait(&bars.kv_full[nslot], (consumed / L::kStages) & 1, &bars.abort))) break;
                    ++consumed;
                    tc_fence_after();
                    if (j + 1 < n_kv[0]) {
                        issue_s(0, nslot);  // overwrites P0_j: PV0_j was issued first
                        tc_commit(&bars.s_full[0]);
                    }
                }
                if (j < n_kv[1]) {
                    if (!(ok = mbar_wait(&bars.p_ready[1], pr[1], &bars.abort))) break;
                    pr[1] ^= 1;
                    tc_fence_after();
                    issue_pv(1, vslot, j > 0);
                    if (j == n_kv[1] - 1) tc_commit(&bars.o_full[1]);
                }
                tc_commit(&bars.kv_empty[vslot]);
                if (next) {
                    if (j + 1 < n_kv[1]) {
                        issue_s(1, nslot);
                        tc_commit(&bars.s_full[1]);
                    }
                    tc_commit(&bars.kv_empty[nslot]);
                }
            }
            // every MMA must have finished before TMEM is released
            tc_commit(&bars.mma_done);
            volatile int never = 0;
            mbar_wait(&bars.mma_done, 0, &never);
        }
    } else {
        // ================================================================ softmax + epilogue
        const int x = (warp - 2) / 4;
        const int quarter = warp % 4;  // TMEM lanes [32*quarter, 32*quarter + 32)
        const int r = quarter * 32 + lane;
        const int i = (pair * kQTiles + x) * kBM + r;  // query row
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t t_s = t_lane + L::s_col(x);
        const uint32_t t_o = t_lane + L::o_col(x);
        const int n = n_kv[x];
        const int lim = a.causal ? min(Lb, i + off + 1) : Lb;  // keys [0, lim) visible
        const float sl2 = a.scale * kLog2e;
        float m_run = -INFINITY, l = 0.f;
        uint32_t sp = 0;
        bool ok = true;

        for (int j = 0; j < n; ++j) {
            if (!(ok = mbar_wait_warp(&bars.s_full[x], sp, &bars.abort))) break;
            sp ^= 1;
            tc_fence_after();
            uint32_t s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, s + c * 32);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence32(s + c * 32);

            const int kbase = j * kBN;
            const bool need_mask = __any_sync(0xffffffffu, kbase + kBN > lim);
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (kbase + c >= lim) s[c] = f2u(-INFINITY);
            }
            float m8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) m8[e] = u2f(s[e]);
#pragma unroll
            for (int c = 8; c < 128; ++c) m8[c % 8] = fmaxf(m8[c % 8], u2f(s[c]));
            const float mraw = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            const float m_tile = mraw == -INFINITY ? -INFINITY : mraw * sl2;
            const float m_new = fmaxf(m_run, m_tile);
            const bool grow = m_new > m_run + kRescaleLog2;
            if (__any_sync(0xffffffffu, grow)) {
                const float factor = grow ? ex2_approx(m_run - m_new) : 1.f;
                if (grow) {
                    l *= factor;
                    m_run = m_new;
                }
                if (j > 0) {  // O holds earlier tiles: bring it to the new max
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(t_o + c * 32, o);
                        tmem_ld_wait();
                        reg_fence32(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = f2u(u2f(o[e]) * factor);
                        tmem_st32(t_o + c * 32, o);
                    }
                }
            }
            const float negm = m_run == -INFINITY ? 0.f : -m_run;
            float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // two halves of 64 keys -> 32 packed columns each
                uint32_t p[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float s0 = u2f(s[h * 64 + 2 * e]), s1 = u2f(s[h * 64 + 2 * e + 1]);
                    float p0 = ex2_approx(fmaf(s0, sl2, negm));
                    float p1 = ex2_approx(fmaf(s1, sl2, negm));
                    if (need_mask) {  // exact zeros, also when scale == 0
                        p0 = s0 == -INFINITY ? 0.f : p0;
                        p1 = s1 == -INFINITY ? 0.f : p1;
                    }
                    l8[(2 * e) % 8] += p0;
                    l8[(2 * e + 1) % 8] += p1;
                    p[e] = pack_bf16x2(p0, p1);
                }
                tmem_st32(t_s + h * 32, p);
            }
            l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars.p_ready[x]);
        }

        // ---- epilogue
        bool have_o = n > 0 && ok;
        if (have_o) {
            have_o = mbar_wait_warp(&bars.o_full[x], 0, &bars.abort);
            tc_fence_after();
        }
        const bool zero_row = !have_o || (a.kv_len && i >= Lb) || !(l > 0.f);
        const float inv = zero_row ? 0.f : 1.f / l;
        __nv_bfloat16 *orow =
            static_cast<__nv_bfloat16 *>(a.out) + (static_cast<size_t>(bh) * a.Sq + i) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32] = {};
            if (have_o) {
                tmem_ld32(t_o + c * 32, o);
                tmem_ld_wait();
                reg_fence32(o);
            }
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float v0 = zero_row ? 0.f : u2f(o[2 * e]) * inv;
                const float v1 = zero_row ? 0.f : u2f(o[2 * e + 1]) * inv;
                pk[e] = pack_bf16x2(v0, v1);
            }
            if (i < a.Sq) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && bars.abort) report_timeout(a.status, 0x11);
}

template <int D>
cudaError_t launch_t(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv) {
    using L = Layout<D>;
    const int n_qt = (a.Sq + kBM - 1) / kBM;
    const int n_pairs = (n_qt + kQTiles - 1) / kQTiles;
    const long long blocks = static_cast<long long>(a.B) * a.H * n_pairs;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<D><<<static_cast<unsigned>(blocks), kThreads, L::kSmemBytes, a.stream>>>(a, tq, tk, tv,
                                                                                             n_pairs);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv) {
    return a.D == 64 ? launch_t<64>(a, tq, tk, tv) : launch_t<128>(a, tq, tk, tv);
}

}  // namespace attn
