// bf16 prefill attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes out = softmax(Q K^T * scale + M) V per (batch, head) ("Attention
// from First Principles", section 5 "The full multi-head computation"), with
// the causal and key-padding masks of "Attention from Scratch" (kube-dojo),
// Part 3, without ever writing the score matrix to HBM: the tiled, exact
// scheme the pages name as FlashAttention ("Scaled dot-product attention with
// masking", "The memory problem"), redesigned here for Blackwell.
//
// Persistent kernel, one CTA per SM.  A work item is two 128-row query tiles
// (Q0, Q1) that read the same key/value head: two consecutive query tiles of
// one head, or -- grouped-query attention with an even group size -- the same
// query tile of two heads of one group.  Items are numbered in blocks of
// heads whose keys and values fit in part of L2, longest-first inside a block
// (causal cost grows with the row), and handed out by an atomic counter, so
// each SM takes the next item when it is ready for it.  Roles (12 warps; the
// first warpgroup gives registers to the two softmax warpgroups):
//   warp 0      TMA producer: fetches and decodes the next item, publishes the
//               record to the other roles through a small ring in shared
//               memory, loads Q0/Q1 as
//               soon as the previous item's last S MMA on that buffer has
//               completed, and streams K_j, V_j through a ring of 32 KB stages
//               (128-byte swizzle, 64-column boxes).
//   warp 1      allocates 512 TMEM columns, then runs the MMA role as a
//               whole warp (uniform control flow, operands in the uniform
//               datapath); one elected lane issues every MMA:
//                 S_x = Q_x K_j^T        (SS: both operands in shared memory)
//                 O_x += P_x V_j         (TS: P read from TMEM, V MN-major)
//               in the order S0_0 S1_0 | PV0_j S0_{j+1} PV1_j S1_{j+1} | ...
//               so each softmax warpgroup has two MMA slots to hide behind.
//   warps 4-7   softmax for Q0, warps 8-11 for Q1: thread = query row = TMEM
//               lane.  Load the 128 fp32 scores of the row, online max/sum in
//               log2 units, p = 2^(s*scale*log2e - m), write p as bf16 over
//               the S columns for the TS MMA.  Tiles that cross the causal
//               diagonal or the padding edge take a separate masked path;
//               the common path carries no masking instructions at all.  O is
//               rescaled lazily, only when the running max grows by more
//               than 2^8, so most tiles never touch O.
//   epilogue    the same warps: O / l -> bf16, transposed through a 4 KB
//               per-warp buffer so that every global store writes whole
//               128-byte lines; rows with no visible key and padded query
//               rows are written as exact zeros.
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D, 256+2D);
// P_x aliases the first 64 columns of S_x.
// KV tiles wholly above the causal diagonal or past kv_len are never loaded.
#include "kernels.h"
#include "prefill_sched.cuh"
#include "ptx.cuh"

#include <atomic>
#include <mutex>

namespace attn {
namespace {

constexpr int kThreads = 384;  // 12 warps
constexpr uint32_t kRegsProducer = 64;   // warps 0-3 after setmaxnreg
constexpr uint32_t kRegsSoftmax = 216;   // warps 4-11: 128*64 + 256*216 <= 384*168
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold (log2 units)
constexpr int kItemRing = 4;          // work items in flight between the roles
constexpr int kItemReaders = 32 + 256;  // MMA warp + both softmax warpgroups

template <int D>
struct Layout {
    static constexpr int kSub = D / 64;                    // 128-byte column blocks per row
    static constexpr int kBlockBytes = 128 * 128;          // one block of a 128-row tile
    static constexpr int kTileBytes = kSub * kBlockBytes;  // 32 KB at D = 128
    static constexpr int kStages = D == 128 ? 4 : 8;       // K/V ring depth
    static constexpr int kRingOff = kQTiles * kTileBytes;
    static constexpr int kStageBytes = 32 * 128;           // per softmax warp: 32 rows x 64 columns bf16
    static constexpr int kStageOff = kRingOff + kStages * kTileBytes;
    static constexpr int kBarOff = kStageOff + 8 * kStageBytes;
    static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // + barriers + alignment slack
    // TMEM column of S_x (and of P_x, which aliases it) and of O_x
    static __device__ __forceinline__ uint32_t s_col(int x) { return static_cast<uint32_t>(x) * 128u; }
    static __device__ __forceinline__ uint32_t o_col(int x) { return 256u + static_cast<uint32_t>(x) * D; }
};

struct Bars {
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t s_full[2];
    uint64_t p_ready[2];
    uint64_t o_full[2];
    uint64_t item_full[kItemRing];
    uint64_t item_empty[kItemRing];
    uint64_t mma_done;
    Item item[kItemRing];  // published work items, decoded; N == -1: no more work
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Work counters, one slot per launch: [0] next item, [2] epoch of the launch
// using the slot (0: free); [1] and [3] unused.  Every CTA's producer takes
// items until it draws one past the end, so a launch draws exactly n_items +
// gridDim.x numbers: the CTA that draws the last one resets the slot (no CTA
// of the launch touches it after that), and the next launch on the slot
// starts from zero without a clearing step or any atomic at the end of the
// kernel.  Each CTA claims the slot (writes its epoch) at its start, before
// its first draw, which is a release operation; the last drawer fences before
// it resets the epoch, so no claim can land after the reset.  Direct launches
// take slots [0, kSchedSlots) in turn; a launch captured into a CUDA graph
// gets its own slot from the kGraphSlots after them, so replays never share a
// counter with direct launches.  A CTA that finds another launch's epoch in
// its slot reports kStatusSchedConflict: the two launches' outputs are then
// undefined.  A launch that gave up on a wait may stop drawing early and
// leave its slot claimed; later launches on that slot then report the
// conflict until the counters are cleared from the host.
__device__ unsigned int g_sched[kSchedSlots + kGraphSlots][4];

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// The producer decodes each item once and publishes the record; the other
// roles read it from the ring instead of repeating the integer divisions.
__device__ __forceinline__ void publish_item(Bars &bars, int slot, const Item &it) {
    volatile Item &d = bars.item[slot];
    d.row_base = it.row_base;
    d.row_step = it.row_step;
    d.bh_base = it.bh_base;
    d.bh_step = it.bh_step;
    d.bh_kv = it.bh_kv;
    d.Lb = it.Lb;
    d.off = it.off;
    d.n_kv[0] = it.n_kv[0];
    d.n_kv[1] = it.n_kv[1];
    d.N = it.N;
}
__device__ __forceinline__ Item read_item(Bars &bars, int k) {
    const volatile Item &sv = bars.item[k % kItemRing];
    Item it;
    it.row_base = sv.row_base;
    it.row_step = sv.row_step;
    it.bh_base = sv.bh_base;
    it.bh_step = sv.bh_step;
    it.bh_kv = sv.bh_kv;
    it.Lb = sv.Lb;
    it.off = sv.off;
    it.n_kv[0] = sv.n_kv[0];
    it.n_kv[1] = sv.n_kv[1];
    it.N = sv.N;
    return it;
}
// Wait (warp-wide) until the item in ring slot k % kItemRing is published and
// read it.  The slot stays readable until the caller releases it.  Returns
// false on a timed-out wait.
__device__ __forceinline__ bool take_item(Bars &bars, int k, Item *it) {
    const int slot = k % kItemRing;
    if (!mbar_wait_warp(&bars.item_full[slot], (k / kItemRing) & 1, &bars.abort)) return false;
    *it = read_item(bars, k);
    return true;
}
__device__ __forceinline__ void release_item(Bars &bars, int k) {
    mbar_arrive(&bars.item_empty[k % kItemRing]);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const int n_major, const int group, const int front, const int n_items,
                      unsigned int *sched, const unsigned int epoch) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem + L::kRingOff;
    Bars &bars = *reinterpret_cast<Bars *>(smem + L::kBarOff);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    unsigned int owner = 0u;
    if (threadIdx.x == 0) {
        // claim the slot for this launch (the first CTA finds it free, the
        // others this launch's epoch); the result is checked after the
        // prologue, so the atomic's round trip overlaps it
        owner = atomicExch(sched + 2, epoch);
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        for (int x = 0; x < kQTiles; ++x) {
            mbar_init(&bars.q_full[x], 1);
            mbar_init(&bars.q_empty[x], 1);
            mbar_init(&bars.s_full[x], 1);
            mbar_init(&bars.p_ready[x], 128);
            mbar_init(&bars.o_full[x], 1);
        }
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&bars.kv_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int s = 0; s < kItemRing; ++s) {
            mbar_init(&bars.item_full[s], 1);
            mbar_init(&bars.item_empty[s], kItemReaders);
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
    // Launched with programmatic stream serialisation: the prologue above may
    // overlap the previous kernel in the stream; nothing it wrote is read (and
    // nothing is written) before that kernel has finished.  The next kernel
    // may be placed as soon as every CTA of this one has started.
    griddep_launch_dependents();
    griddep_wait();

    if (warp == 0) {
        // ================================================================ TMA producer
        regs_dec<kRegsProducer>();
        if (lane == 0) {
            if (owner != 0u && owner != epoch) report_status(a.status, 0x12, kStatusSchedConflict);
            const unsigned int last_draw = static_cast<unsigned int>(n_items) + gridDim.x - 1u;
            uint32_t q_uses[kQTiles] = {0, 0};  // Q_x loads issued so far
            int issued = 0;                     // K/V ring loads issued so far
            bool ok = true;
            for (int k = 0; ok; ++k) {
                // ---- fetch the next item and publish it to the other roles
                const int slot = k % kItemRing;
                if (k >= kItemRing &&
                    !(ok = mbar_wait(&bars.item_empty[slot], ((k / kItemRing) - 1) & 1, &bars.abort)))
                    break;
                // the first draw releases this CTA's claim of the slot
                const unsigned int drawn = k == 0 ? atomic_add_release_gpu(sched, 1u) : atomicAdd(sched, 1u);
                if (drawn == last_draw) {  // the launch's last draw: free the slot
                    fence_acq_rel_gpu();
                    atomicExch(sched, 0u);
                    atomicExch(sched + 2, 0u);
                }
                const int t = static_cast<int>(drawn);
                Item it;
                if (t < n_items) {
                    it = decode_item(t, a, n_major, group, front);
                } else {
                    it = Item{0, 0, 0, 0, 0, 0, 0, {0, 0}, -1};
                }
                publish_item(bars, slot, it);
                mbar_arrive(&bars.item_full[slot]);
                if (it.N < 0) break;
                // ---- loads in the order the MMA warp consumes them: Q_0, K_0,
                // Q_1, V_0, K_1, V_1, ...  (Q_1 waits for the previous item's
                // last S1 to free its buffer; K_0 need not wait for that).
                // Q_x once the previous item's last S MMA on the buffer has completed:
                auto load_q = [&](int x) {
                    if (it.n_kv[x] == 0 || !ok) return;
                    if (q_uses[x] > 0 && !(ok = mbar_wait(&bars.q_empty[x], (q_uses[x] - 1) & 1, &bars.abort)))
                        return;
                    mbar_arrive_expect_tx(&bars.q_full[x], L::kTileBytes);
#pragma unroll
                    for (int c = 0; c < L::kSub; ++c)
                        tma_load_3d(smem + x * L::kTileBytes + c * L::kBlockBytes, &tq, &bars.q_full[x], c * 64,
                                    it.row_base + x * it.row_step, it.bh_base + x * it.bh_step);
                    ++q_uses[x];
                };
                // K_j (kv = 0) or V_j (kv = 1) into the next ring stage
                auto load_kv = [&](int j, int kv) {
                    if (!ok) return;
                    const int s = issued % L::kStages;
                    if (issued >= L::kStages &&
                        !(ok = mbar_wait(&bars.kv_empty[s], ((issued / L::kStages) - 1) & 1, &bars.abort)))
                        return;
                    mbar_arrive_expect_tx(&bars.kv_full[s], L::kTileBytes);
#pragma unroll
                    for (int c = 0; c < L::kSub; ++c)
                        tma_load_3d(ring + s * L::kTileBytes + c * L::kBlockBytes, kv ? &tv : &tk, &bars.kv_full[s],
                                    c * 64, j * kBN, it.bh_kv);
                    ++issued;
                };
                load_q(0);
                for (int j = 0; j < it.N && ok; ++j) {
                    load_kv(j, 0);
                    if (j == 0) load_q(1);
                    load_kv(j, 1);
                }
            }
            // never leave with copies still landing in shared memory
            volatile int never = 0;
            for (int x = 0; x < kQTiles; ++x)
                if (q_uses[x] > 0) mbar_wait(&bars.q_full[x], (q_uses[x] - 1) & 1, &never);
            for (int u = max(0, issued - L::kStages); u < issued; ++u)
                mbar_wait(&bars.kv_full[u % L::kStages], (u / L::kStages) & 1, &never);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        regs_dec<kRegsProducer>();
        const uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0);
        const uint32_t idesc_o = idesc_bf16_f32(kBM, D, 1);
        // Base descriptors, built once: the K-step offsets only move the
        // start-address field (low 14 bits, no carry below 256 KB).
        const uint64_t dq[2] = {sdesc_sw128(smem_u32(smem), 16, 1024),
                                sdesc_sw128(smem_u32(smem) + L::kTileBytes, 16, 1024)};
        const uint64_t dk0 = sdesc_sw128(smem_u32(ring), 16, 1024);
        const uint64_t dv0 = sdesc_sw128(smem_u32(ring), L::kBlockBytes, 1024);
        auto issue_s = [&](int x, int slot) {
            const uint64_t da = dq[x];
            const uint64_t db = desc_add(dk0, (slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t koff = ((kk / 4) * L::kBlockBytes + (kk % 4) * 32) >> 4;
                mma_ss_warp(tmem + L::s_col(x), desc_add(da, koff), desc_add(db, koff), idesc_s, kk > 0);
            }
        };
        auto issue_pv = [&](int x, int slot, bool acc) {
            const uint64_t db = desc_add(dv0, (slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                mma_ts_warp(tmem + L::o_col(x), tmem + L::s_col(x) + kk * 8, desc_add(db, (kk * 16 * 128) >> 4),
                            idesc_o, (acc || kk > 0) ? 1u : 0u);
        };
        int consumed = 0;  // K/V ring stages consumed so far
        uint32_t q_uses[kQTiles] = {0, 0}, pr[kQTiles] = {0, 0};
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Item it;
            if (!(ok = take_item(bars, k, &it))) break;
            release_item(bars, k);
            // Values read from memory are not provably warp-uniform; broadcast
            // them from lane 0 so the MMA code keeps its operands and branches
            // in the uniform datapath.
#pragma unroll
            for (int x = 0; x < kQTiles; ++x) it.n_kv[x] = __shfl_sync(0xffffffffu, it.n_kv[x], 0);
            it.N = __shfl_sync(0xffffffffu, it.N, 0);
            const int N = it.N;
            if (N < 0) break;
            if (N == 0) continue;
            // S_x_0 per query tile as soon as Q_x and K_0 are in (Q_1 may land
            // after Q_0: the previous item's last S1 freed its buffer late)
            {
                int kslot = 0;
                bool have_k = false;
#pragma unroll
                for (int x = 0; x < kQTiles; ++x) {
                    if (it.n_kv[x] == 0) continue;
                    if (!(ok = mbar_wait_warp(&bars.q_full[x], q_uses[x] & 1, &bars.abort))) break;
                    ++q_uses[x];
                    if (!have_k) {
                        kslot = consumed % L::kStages;
                        if (!(ok = mbar_wait_warp(&bars.kv_full[kslot], (consumed / L::kStages) & 1, &bars.abort)))
                            break;
                        ++consumed;
                        have_k = true;
                    }
                    tc_fence_after();
                    issue_s(x, kslot);
                    tc_commit_warp(&bars.s_full[x]);
                    if (it.n_kv[x] == 1) tc_commit_warp(&bars.q_empty[x]);  // last read of Q_x
                }
                if (!ok) break;
                tc_commit_warp(&bars.kv_empty[kslot]);
            }
            for (int j = 0; j < N && ok; ++j) {
                const int vslot = consumed % L::kStages;
                if (!(ok = mbar_wait_warp(&bars.kv_full[vslot], (consumed / L::kStages) & 1, &bars.abort))) break;
                ++consumed;
                tc_fence_after();
                if (j < it.n_kv[0]) {
                    if (!(ok = mbar_wait_warp(&bars.p_ready[0], pr[0], &bars.abort))) break;
                    pr[0] ^= 1;
                    tc_fence_after();
                    issue_pv(0, vslot, j > 0);
                    if (j == it.n_kv[0] - 1) tc_commit_warp(&bars.o_full[0]);
                }
                const bool next = j + 1 < N;
                int nslot = 0;
                if (next) {
                    nslot = consumed % L::kStages;
                    if (!(ok = mbar_wait_warp(&bars.kv_full[nslot], (consumed / L::kStages) & 1, &bars.abort))) break;
                    ++consumed;
                    tc_fence_after();
                    if (j + 1 < it.n_kv[0]) {
                        issue_s(0, nslot);  // overwrites P0_j: PV0_j was issued first
                        tc_commit_warp(&bars.s_full[0]);
                        if (j + 2 == it.n_kv[0]) tc_commit_warp(&bars.q_empty[0]);
                    }
                }
                if (j < it.n_kv[1]) {
                    if (!(ok = mbar_wait_warp(&bars.p_ready[1], pr[1], &bars.abort))) break;
                    pr[1] ^= 1;
                    tc_fence_after();
                    issue_pv(1, vslot, j > 0);
                    if (j == it.n_kv[1] - 1) tc_commit_warp(&bars.o_full[1]);
                }
                tc_commit_warp(&bars.kv_empty[vslot]);
                if (next) {
                    if (j + 1 < it.n_kv[1]) {
                        issue_s(1, nslot);
                        tc_commit_warp(&bars.s_full[1]);
                        if (j + 2 == it.n_kv[1]) tc_commit_warp(&bars.q_empty[1]);
                    }
                    tc_commit_warp(&bars.kv_empty[nslot]);
                }
            }
        }
        // every MMA must have finished before TMEM is released
        tc_commit_warp(&bars.mma_done);
        volatile int never = 0;
        mbar_wait_warp(&bars.mma_done, 0, &never);
    } else if (warp < 4) {
        regs_dec<kRegsProducer>();  // warps 2-3: no role, registers go to the softmax warps
    } else {
        // ================================================================ softmax + epilogue
        regs_inc<kRegsSoftmax>();
        const int x = (warp - 4) / 4;
        const int quarter = warp % 4;  // TMEM lanes [32*quarter, 32*quarter + 32)
        const int r = quarter * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t t_s = t_lane + L::s_col(x);
        const uint32_t t_o = t_lane + L::o_col(x);
        const float sl2 = a.scale * kLog2e;
        const uint32_t stage = smem_u32(smem + L::kStageOff + (warp - 4) * L::kStageBytes);
        uint32_t sp = 0, o_uses = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int n, lim;
            {
                Item it;
                if (!(ok = take_item(bars, k, &it))) break;
                if (it.N < 0) {
                    release_item(bars, k);
                    break;
                }
                const int i = it.row_base + x * it.row_step + r;  // query row
                n = x ? it.n_kv[1] : it.n_kv[0];  // a select: x is not a compile-time index here
                lim = a.causal ? min(it.Lb, i + it.off + 1) : it.Lb;  // keys [0, lim) visible
            }
            float m_run = -INFINITY, l = 0.f;

            for (int j = 0; j < n; ++j) {
                if (!(ok = mbar_wait_warp<32>(&bars.s_full[x], sp, &bars.abort))) break;
                sp ^= 1;
                tc_fence_after();
                uint32_t s[128];
    #pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, s + c * 32);
                tmem_ld_wait();
    #pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence32(s + c * 32);

                // This row sees columns [0, t) of the tile.  On a tile that crosses
                // the causal diagonal or the padding edge, each warp sorts its
                // 32-column chunks into seen by all its rows, hidden from all of
                // them (no max, no exp, P = 0) and partial (per-column select).
                const int t = lim - j * kBN;
                const bool need_mask = __any_sync(0xffffffffu, t < kBN);
                int t_lo = kBN, t_hi = kBN;
                if (need_mask) {
                    t_lo = __reduce_min_sync(0xffffffffu, t);
                    t_hi = __reduce_max_sync(0xffffffffu, t);
                }
                // row max over the tile: 8 chains of 3-input max
                float m8[8];
                if (!need_mask) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) m8[e] = fmaxf(u2f(s[2 * e]), u2f(s[2 * e + 1]));
#pragma unroll
                    for (int c = 16; c < 128; c += 2)
                        m8[(c / 2) % 8] = fmax3(m8[(c / 2) % 8], u2f(s[c]), u2f(s[c + 1]));
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (t_hi <= 32 * c) {  // hidden from every row of the warp
                            m8[2 * c] = m8[2 * c + 1] = -INFINITY;
                            continue;
                        }
                        if (t_lo < 32 * c + 32) {  // partial: hide columns >= t
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (32 * c + e >= t) s[32 * c + e] = f2u(-INFINITY);
                        }
                        float a0 = fmaxf(u2f(s[32 * c]), u2f(s[32 * c + 1]));
                        float a1 = fmaxf(u2f(s[32 * c + 2]), u2f(s[32 * c + 3]));
#pragma unroll
                        for (int e = 4; e < 32; e += 4) {
                            a0 = fmax3(a0, u2f(s[32 * c + e]), u2f(s[32 * c + e + 1]));
                            a1 = fmax3(a1, u2f(s[32 * c + e + 2]), u2f(s[32 * c + e + 3]));
                        }
                        m8[2 * c] = a0;
                        m8[2 * c + 1] = a1;
                    }
                }
                const float mraw = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
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
                const uint64_t sl2x2 = f2_pack(sl2, sl2), negmx2 = f2_pack(negm, negm);
                uint64_t l4[4] = {0, 0, 0, 0};  // packed partial row sums
                // p = 2^(s*scale*log2e - m), packed into bf16 pairs over the S
                // columns.  A hidden column holds -inf and 2^-inf is an exact
                // zero, except when scale == 0 (-inf * 0 is NaN: select it).
#define ATTN_EXP_PAIR(k0, pe, SELECT)                                                         \
    {                                                                                         \
        const uint64_t arg = ffma2(f2_pack(u2f(s[k0]), u2f(s[(k0) + 1])), sl2x2, negmx2);     \
        float p0 = ex2_approx(f2_lo(arg));                                                    \
        float p1 = ex2_approx(f2_hi(arg));                                                    \
        if (SELECT) {                                                                         \
            p0 = u2f(s[k0]) == -INFINITY ? 0.f : p0;                                          \
            p1 = u2f(s[(k0) + 1]) == -INFINITY ? 0.f : p1;                                    \
        }                                                                                     \
        l4[(pe) % 4] = fadd2(l4[(pe) % 4], f2_pack(p0, p1));                                  \
        p[pe] = pack_bf16x2(p0, p1);                                                          \
    }
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // two halves of 64 keys -> 32 packed columns each
                    uint32_t p[32];
                    if (!need_mask) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) ATTN_EXP_PAIR(h * 64 + 2 * e, e, false)
                    } else {
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int c = 2 * h + cc;
                            if (t_hi <= 32 * c) {  // hidden from every row of the warp
#pragma unroll
                                for (int e = 0; e < 16; ++e) p[16 * cc + e] = 0u;
                            } else if (sl2 != 0.f) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) ATTN_EXP_PAIR(32 * c + 2 * e, 16 * cc + e, false)
                            } else {
#pragma unroll
                                for (int e = 0; e < 16; ++e) ATTN_EXP_PAIR(32 * c + 2 * e, 16 * cc + e, true)
                            }
                        }
                    }
                    tmem_st32(t_s + h * 32, p);
                }
#undef ATTN_EXP_PAIR
                {
                    const uint64_t l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
                    l += f2_lo(l2) + f2_hi(l2);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars.p_ready[x]);
            }


            // ---- epilogue: O / l -> bf16.  Each warp transposes its 32 rows
            // through its own buffer (64 columns per pass, 128-byte swizzled
            // rows) so that each global store instruction writes four whole
            // 128-byte row segments.
            bool have_o = n > 0 && ok;
            if (have_o) {
                have_o = mbar_wait_warp(&bars.o_full[x], o_uses & 1, &bars.abort);
                tc_fence_after();
                ok = have_o;
            }
            if (n > 0) ++o_uses;
            // the item again, from its ring slot (nothing of it stays live through the tile loop)
            const Item it = read_item(bars, k);
            release_item(bars, k);
            const int row0 = it.row_base + x * it.row_step;
            const int i = row0 + r;
            const bool zero_row =
                !have_o || (a.kv_len && !a.chunked && a.Sq == a.Skv && i >= it.Lb) || !(l > 0.f);
            const float inv = zero_row ? 0.f : 1.f / l;
            // log(sum_j exp(scale * s_j)) = ln 2 * (m_run + log2 l): l is kept relative to
            // m_run whether or not the lazy rescale has moved it
            if (a.lse && i < a.Sq)
                a.lse[static_cast<size_t>(it.bh_base + x * it.bh_step) * a.Sq + i] =
                    zero_row ? -INFINITY : (m_run + log2f(l)) * 0.6931471805599453f;
            __nv_bfloat16 *obh = static_cast<__nv_bfloat16 *>(a.out) + static_cast<size_t>(it.bh_base + x * it.bh_step) * a.Sq * D;
            const int wrow0 = row0 + quarter * 32;  // first row of this warp
#pragma unroll
            for (int c = 0; c < L::kSub; ++c) {
                // Columns [64c, 64c + 64) of this row.  Loaded unconditionally (TMEM
                // of this CTA): without O the select below writes zeros.
                uint32_t o[64];
                {
                    tmem_ld32(t_o + c * 64, o);
                    tmem_ld32(t_o + c * 64 + 32, o + 32);
                    tmem_ld_wait();
                    reg_fence32(o);
                    reg_fence32(o + 32);
                }
                __syncwarp();  // the previous pass has read the buffer back
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {  // 16-byte chunk k8 of this row's 64 columns
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = k8 * 8 + 2 * e;
                        pk[e] = zero_row ? 0u : pack_bf16x2(u2f(o[col]) * inv, u2f(o[col + 1]) * inv);
                    }
                    st_shared_v4(stage + lane * 128 + ((k8 ^ (lane & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
                }
                __syncwarp();
#pragma unroll
                for (int s4 = 0; s4 < 8; ++s4) {  // rows 4*s4 .. 4*s4 + 3, one 16-byte chunk per lane
                    const int rr = 4 * s4 + (lane >> 3), ch = lane & 7;
                    const uint4 v = ld_shared_v4(stage + rr * 128 + ((ch ^ (rr & 7)) << 4));
                    const int row = wrow0 + rr;
                    if (row < a.Sq)
                        *reinterpret_cast<uint4 *>(obh + static_cast<size_t>(row) * D + c * 64 + ch * 8) = v;
                }
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

}  // namespace

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_sched_mutex;
unsigned int *g_sched_base[kMaxDevices];
std::atomic<unsigned int> g_sched_turn{0}, g_graph_turn{0}, g_epoch{0};

// Work counters for one launch: a slot of g_sched and a non-zero epoch.
// Direct launches take the first kSchedSlots slots in turn, so launches
// running at the same time on other streams count separately; a launch being
// captured into a CUDA graph (which keeps its slot for every replay) takes
// the next of the kGraphSlots reserved for captures.
cudaError_t sched_slot(cudaStream_t stream, unsigned int **out, unsigned int *epoch) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return e;
    unsigned int *base;
    {
        std::lock_guard<std::mutex> lock(g_sched_mutex);
        if (!g_sched_base[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_sched);
            if (e != cudaSuccess) return e;
            g_sched_base[dev] = static_cast<unsigned int *>(p);
        }
        base = g_sched_base[dev];
    }
    const unsigned int slot = cap == cudaStreamCaptureStatusNone
                                  ? g_sched_turn.fetch_add(1u) % kSchedSlots
                                  : kSchedSlots + g_graph_turn.fetch_add(1u) % kGraphSlots;
    *out = base + 4 * slot;
    unsigned int ep;
    do {
        ep = g_epoch.fetch_add(1u) + 1u;
    } while (ep == 0u);
    *epoch = ep;
    return cudaSuccess;
}

template <int D>
cudaError_t launch_t(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv) {
    using L = Layout<D>;
    ItemPlan plan;
    bool too_many = false;
    const long long sms = a.n_sm > 0 ? a.n_sm : 1;
    if (!plan_items(a, sms, &plan, &too_many)) return too_many ? cudaErrorInvalidConfiguration : cudaSuccess;
    unsigned int *sched = nullptr, epoch = 0;
    cudaError_t e = sched_slot(a.stream, &sched, &epoch);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(plan.n_items < sms ? plan.n_items : sms);
    e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: back to back with the previous kernel,
    // the launch and the prologue overlap its end (griddep_wait in the kernel)
    return launch_pdl(prefill_tc_kernel<D>, dim3(grid), dim3(kThreads), L::kSmemBytes, a.stream, a, tq, tk, tv,
                      plan.n_major, plan.group, plan.front, plan.n_items, sched, epoch);
}

}  // namespace

cudaError_t reset_prefill_counters() {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_sched);
    if (e != cudaSuccess) return e;
    return cudaMemset(p, 0, sizeof g_sched);
}

cudaError_t launch_prefill_tc(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv) {
    return a.D == 64 ? launch_t<64>(a, tq, tk, tv) : launch_t<128>(a, tq, tk, tv);
}

}  // namespace attn
