// Grouped-query and multi-query decode on the sm_103a tensor cores.
//
// One new query per head against a KV cache ("Attention from First
// Principles", section 6 "Under the hood": decode reads the cache once per
// token; "Scaled dot-product attention with masking", "Grouped-query attention
// (GQA)").  With G = H / H_kv query heads per cached head, every key and value
// row of a cached head serves G queries: for large G the CUDA-core decode
// kernels run out of FMA throughput long before HBM bandwidth, so the G
// queries become the rows of one 128-row tile and the contractions run as
// tcgen05 MMAs:
//     S = Q K_j^T        (M = 128 rows: the G heads, N = 64 keys, K = D)
//     O += P V_j          (M = 128, N = D, K = 64 keys; P from TMEM)
// One CTA per (sequence, cached head, chunk of keys); it writes the chunk's
// partial softmax state (O unnormalised, running max in log2 units, sum) and
// the decode combine kernel merges the chunks exactly.
//
// S is double-buffered in TMEM (two 64-column buffers beside O), so the MMA
// warp issues S_{j+1} before PV_j and the softmax of one tile overlaps the
// score MMA of the next: per 64-key tile the CTA costs about one softmax.
// Roles (6 warps): warp 0 TMA producer (Q once, then K_j, V_j through a ring),
// warp 1 TMEM allocation and MMA issue (whole warp, one elected lane), warps
// 2-5 softmax and epilogue, thread = row = query head (TMEM lane).  Rows past
// the group's G heads hold other heads' queries (or zeros past the tensor):
// they are computed and never written.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kTcBN = 64;        // keys per K/V tile
constexpr int kTcThreads = 192;  // 6 warps
// K/V ring stages (K_j and V_j take one each); with 4 stages a CTA needs
// 97 KB of shared memory at D = 128 and two CTAs share an SM (and its TMEM)
#ifndef ATTN_DTC_STAGES
#define ATTN_DTC_STAGES 4
#endif
constexpr int kTcStages = ATTN_DTC_STAGES;
constexpr int kTcMinBlocks = kTcStages <= 4 ? 2 : 1;
#ifndef ATTN_DTC_WAVES
#define ATTN_DTC_WAVES 6
#endif
#ifndef ATTN_DTC_MIN_TILES
#define ATTN_DTC_MIN_TILES 8
#endif
constexpr int kTcCols = 256;     // TMEM: S buffers at columns 0 and 64, O at 128
constexpr float kTcLog2e = 1.4426950408889634f;
constexpr float kTcRescaleLog2 = 8.0f;  // lazy rescale of O (log2 units)

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

template <int D>
struct TcLayout {
    static constexpr int kSub = D / 64;            // 128-byte column blocks per row
    static constexpr int kQBlock = 128 * 128;      // 128 rows x 128 bytes
    static constexpr int kQBytes = kSub * kQBlock;
    static constexpr int kKvBlock = kTcBN * 128;   // 64 rows x 128 bytes
    static constexpr int kKvBytes = kSub * kKvBlock;
    static constexpr int kRingOff = kQBytes;
    static constexpr int kBarOff = kRingOff + kTcStages * kKvBytes;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // + barriers + alignment slack
};

struct TcBars {
    uint64_t q_full;
    uint64_t kv_full[kTcStages];
    uint64_t kv_empty[kTcStages];
    uint64_t s_full[2];
    uint64_t p_ready[2];
    uint64_t o_done;  // one phase per PV MMA group
    uint64_t o_full;  // after the last PV
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(TcBars) <= 256, "barrier block");

template <int D>
__global__ void __launch_bounds__(kTcThreads, kTcMinBlocks)
    decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tq,
                     const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
    griddep_launch_dependents();  // the combine may be placed once every CTA has started
    griddep_wait();               // launched back to back: the previous kernel's writes are visible
    using L = TcLayout<D>;
    const int c = blockIdx.x;   // chunk of keys
    const int bk = blockIdx.y;  // b * H_kv + h_kv
    const int b = bk / a.H_kv;
    const int G = a.H / a.H_kv;
    int Lb = a.Skv;
    if (a.kv_len) Lb = min(max(a.kv_len[b], 0), a.Skv);
    const int k0 = c * a.chunk;
    if (k0 >= Lb) return;  // past the sequence: the combine never reads this chunk
    const int nkeys = min(a.chunk, Lb - k0);
    const int n = (nkeys + kTcBN - 1) / kTcBN;  // K/V tiles, >= 1

    extern __shared__ __align__(1024) uint8_t dsmem[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem + L::kRingOff;
    TcBars &bars = *reinterpret_cast<TcBars *>(smem + L::kBarOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        mbar_init(&bars.q_full, 1);
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&bars.kv_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars.s_full[x], 1);
            mbar_init(&bars.p_ready[x], 128);
        }
        mbar_init(&bars.o_done, 1);
        mbar_init(&bars.o_full, 1);
        mbar_init(&bars.mma_done, 1);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars.tmem_base, kTcCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            mbar_arrive_expect_tx(&bars.q_full, L::kQBytes);
#pragma unroll
            for (int cb = 0; cb < L::kSub; ++cb)
                tma_load_2d(smem + cb * L::kQBlock, &tq, &bars.q_full, cb * 64, bk * G);
            bool ok = true;
            int issued = 0;
            for (; issued < 2 * n && ok; ++issued) {
                const int j = issued / 2, kv = issued % 2, s = issued % kTcStages;
                if (issued >= kTcStages &&
                    !(ok = mbar_wait(&bars.kv_empty[s], ((issued / kTcStages) - 1) & 1, &bars.abort)))
                    break;
                mbar_arrive_expect_tx(&bars.kv_full[s], L::kKvBytes);
#pragma unroll
                for (int cb = 0; cb < L::kSub; ++cb)
                    tma_load_3d(ring + s * L::kKvBytes + cb * L::kKvBlock, kv ? &tv : &tk, &bars.kv_full[s],
                                cb * 64, k0 + j * kTcBN, bk);
            }
            // never leave with copies still landing in shared memory
            volatile int never = 0;
            mbar_wait(&bars.q_full, 0, &never);
            for (int u = max(0, issued - kTcStages); u < issued; ++u)
                mbar_wait(&bars.kv_full[u % kTcStages], (u / kTcStages) & 1, &never);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        const uint32_t idesc_s = idesc_bf16_f32(128, kTcBN, 0);
        const uint32_t idesc_o = idesc_bf16_f32(128, D, 1);
        const uint64_t dq = sdesc_sw128(smem_u32(smem), 16, 1024);
        const uint64_t dk0 = sdesc_sw128(smem_u32(ring), 16, 1024);
        const uint64_t dv0 = sdesc_sw128(smem_u32(ring), L::kKvBlock, 1024);
        // S_x = Q K^T into buffer x: K-step kk is 32 bytes into a 128-byte
        // swizzled row; 64-column blocks are kQBlock (Q) and kKvBlock (K) apart
        auto issue_s = [&](int x, int slot) {
            const uint64_t db = desc_add(dk0, (slot * L::kKvBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_ss_warp(tmem + static_cast<uint32_t>(x) * kTcBN,
                            desc_add(dq, ((kk / 4) * L::kQBlock + (kk % 4) * 32) >> 4),
                            desc_add(db, ((kk / 4) * L::kKvBlock + (kk % 4) * 32) >> 4), idesc_s, kk > 0);
        };
        // O (+)= P_x V: P is bf16 over the first 32 columns of buffer x; V is
        // MN-major, K-step kk is 16 key rows of 128 bytes
        auto issue_pv = [&](int x, int slot, bool acc) {
            const uint64_t db = desc_add(dv0, (slot * L::kKvBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kTcBN / 16; ++kk)
                mma_ts_warp(tmem + 128u, tmem + static_cast<uint32_t>(x) * kTcBN + kk * 8,
                            desc_add(db, (kk * 16 * 128) >> 4), idesc_o, (acc || kk > 0) ? 1u : 0u);
        };
        uint32_t pr0 = 0, pr1 = 0;  // p_ready parities (scalars: no runtime-indexed array)
        bool ok = mbar_wait_warp(&bars.q_full, 0, &bars.abort);
        tc_fence_after();
        // order: S_0 | S_1 PV_0 | S_2 PV_1 | ... | PV_{n-1}.  S_j reuses the
        // buffer of tile j - 2, whose P was read by PV_{j-2}, issued earlier.
        for (int j = 0; j <= n && ok; ++j) {
            if (j < n) {
                const int ks = (2 * j) % kTcStages;
                if (!(ok = mbar_wait_warp(&bars.kv_full[ks], ((2 * j) / kTcStages) & 1, &bars.abort))) break;
                tc_fence_after();
                issue_s(j & 1, ks);
                tc_commit_warp(&bars.s_full[j & 1]);
                tc_commit_warp(&bars.kv_empty[ks]);
            }
            if (j >= 1) {
                const int t = j - 1, x = t & 1, vs = (2 * t + 1) % kTcStages;
                if (!(ok = mbar_wait_warp(&bars.p_ready[x], x ? pr1 : pr0, &bars.abort))) break;
                if (x) pr1 ^= 1; else pr0 ^= 1;
                if (!(ok = mbar_wait_warp(&bars.kv_full[vs], ((2 * t + 1) / kTcStages) & 1, &bars.abort))) break;
                tc_fence_after();
                issue_pv(x, vs, t > 0);
                tc_commit_warp(&bars.o_done);
                tc_commit_warp(&bars.kv_empty[vs]);
                if (t == n - 1) tc_commit_warp(&bars.o_full);
            }
        }
        // every MMA must have finished before TMEM is released
        tc_commit_warp(&bars.mma_done);
        volatile int never = 0;
        mbar_wait_warp(&bars.mma_done, 0, &never);
    } else {
        // ================================================================ softmax + epilogue
        const int quarter = warp % 4;  // TMEM lanes [32 * quarter, 32 * quarter + 32)
        const int r = quarter * 32 + lane;  // row: query head r of the group
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const float sl2 = a.scale * kTcLog2e;  // decode scale is 1 / sqrt(D) > 0
        float m_run = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n && ok; ++j) {
            // buffer x = j & 1 is used by every other tile: its s_full parity is (j >> 1) & 1
            const int x = j & 1;
            if (!(ok = mbar_wait_warp<32>(&bars.s_full[x], (j >> 1) & 1, &bars.abort))) break;
            tc_fence_after();
            uint32_t s[kTcBN];
            tmem_ld32(t_lane + x * kTcBN, s);
            tmem_ld32(t_lane + x * kTcBN + 32, s + 32);
            tmem_ld_wait();
            reg_fence32(s);
            reg_fence32(s + 32);
            // keys past the chunk's end (last tile only) are hidden: -inf, then 2^-inf = 0
            const int t = nkeys - j * kTcBN;
            if (t < kTcBN) {
#pragma unroll
                for (int e = 0; e < kTcBN; ++e)
                    if (e >= t) s[e] = f2u(-INFINITY);
            }
            float m4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = fmaxf(u2f(s[2 * e]), u2f(s[2 * e + 1]));
#pragma unroll
            for (int cc = 8; cc < kTcBN; cc += 2) m4[(cc / 2) % 4] = fmax3(m4[(cc / 2) % 4], u2f(s[cc]), u2f(s[cc + 1]));
            // column 0 is always a key of the chunk (t >= 1): the tile max is finite
            const float m_tile = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
            const float m_new = fmaxf(m_run, m_tile);
            const bool grow = m_new > m_run + kTcRescaleLog2;
            if (__any_sync(0xffffffffu, grow)) {
                const float factor = grow ? ex2_approx(m_run - m_new) : 1.f;
                if (grow) {
                    l *= factor;
                    m_run = m_new;
                }
                if (j > 0) {
                    // O holds PV_0 .. PV_{j-1}; PV_{j-2} finished before S_j, so
                    // o_done has completed j - 1 or j phases: wait for phase j - 1
                    if (!(ok = mbar_wait_warp(&bars.o_done, (j - 1) & 1, &bars.abort))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + 128 + cc * 32, o);
                        tmem_ld_wait();
                        reg_fence32(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = f2u(u2f(o[e]) * factor);
                        tmem_st32(t_lane + 128 + cc * 32, o);
                    }
                }
            }
            // p = 2^(s * scale * log2 e - m), bf16 pairs over the first 32 columns of the buffer
            const uint64_t sl2x2 = f2_pack(sl2, sl2), negmx2 = f2_pack(-m_run, -m_run);
            uint64_t l4[4] = {0, 0, 0, 0};
            uint32_t p[kTcBN / 2];
#pragma unroll
            for (int e = 0; e < kTcBN / 2; ++e) {
                const uint64_t arg = ffma2(f2_pack(u2f(s[2 * e]), u2f(s[2 * e + 1])), sl2x2, negmx2);
                const float p0 = ex2_approx(f2_lo(arg)), p1 = ex2_approx(f2_hi(arg));
                l4[e % 4] = fadd2(l4[e % 4], f2_pack(p0, p1));
                p[e] = pack_bf16x2(p0, p1);
            }
            const uint64_t l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
            l += f2_lo(l2) + f2_hi(l2);
            tmem_st32(t_lane + x * kTcBN, p);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars.p_ready[x]);
        }
        // ---- epilogue: the chunk's partial state for rows that are heads of this group
        if (ok) {
            ok = mbar_wait_warp(&bars.o_full, 0, &bars.abort);
            tc_fence_after();
        }
        const bool write = ok && r < G;
        const size_t part = (static_cast<size_t>(b) * a.H + static_cast<size_t>(bk % a.H_kv) * G + r) * a.n_split + c;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];  // TMEM of this CTA: loaded unconditionally, stored only when valid
            tmem_ld32(t_lane + 128 + cc * 32, o);
            tmem_ld_wait();
            reg_fence32(o);
            if (write) {
                float4 *dst = reinterpret_cast<float4 *>(a.part_o + part * D + cc * 32);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(u2f(o[4 * e]), u2f(o[4 * e + 1]), u2f(o[4 * e + 2]), u2f(o[4 * e + 3]));
            }
        }
        if (write) {
            a.part_ml[part * 2 + 0] = m_run;
            a.part_ml[part * 2 + 1] = l;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        __syncwarp();
        tmem_dealloc(tmem, kTcCols);
    }
    if (threadIdx.x == 0 && bars.abort) report_timeout(a.status, 0x33);
}

template <int D>
cudaError_t launch_tc_t(const DecodeArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv) {
    using L = TcLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (a.Skv > 0) {
        const dim3 grid(static_cast<unsigned>(a.n_split), static_cast<unsigned>(a.B * a.H_kv));
        e = launch_pdl(decode_tc_kernel<D>, grid, dim3(kTcThreads), L::kSmemBytes, a.stream, a, tq, tk, tv);
        if (e != cudaSuccess) return e;
    }
    return launch_decode_combine(a);
}

}  // namespace

int decode_tc_chunk(int B, int H_kv, int Skv, int n_sm) {
    // about ATTN_DTC_WAVES waves of the CTAs an SM holds, at least
    // ATTN_DTC_MIN_TILES 64-key tiles per CTA
    const long long tiles = static_cast<long long>(B) * H_kv * ((Skv + kTcBN - 1) / kTcBN);
    const long long want = static_cast<long long>(ATTN_DTC_WAVES) * kTcMinBlocks * (n_sm > 0 ? n_sm : 1);
    long long per = (tiles + want - 1) / want;
    per = per < ATTN_DTC_MIN_TILES ? ATTN_DTC_MIN_TILES : per;
    const long long cap = (Skv + kTcBN - 1) / kTcBN;
    per = per > cap ? cap : per;
    per = per < 1 ? 1 : per;
    return static_cast<int>(per * kTcBN);
}

cudaError_t launch_decode_tc(const DecodeArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv) {
    return a.D == 64 ? launch_tc_t<64>(a, tq, tk, tv) : launch_tc_t<128>(a, tq, tk, tv);
}

}  // namespace attn
