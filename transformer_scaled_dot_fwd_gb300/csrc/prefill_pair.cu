// bf16 prefill attention for D = 128 on CTA pairs of the sm_103a tensor cores
// (tcgen05 .cta_group::2, TMEM, TMA).
//
// Computes out = softmax(Q K^T * scale + M) V per (batch, head) ("Attention
// from First Principles", section 5 "The full multi-head computation"), with
// the causal and key-padding masks of "Attention from Scratch" (kube-dojo),
// Part 3, never writing the score matrix to HBM: the tiled, exact scheme that
// "Scaled dot-product attention with masking", "The memory problem", names,
// laid out here for CTA pairs.
//
// A cluster of two CTAs on two SMs works on one item at a time: two 128-row
// query tiles that read the same key/value head (prefill_sched.cuh), tile x
// in CTA x.  The even CTA issues every MMA for both, with M = 256:
//     S = Q K^T   (SS; each CTA holds its Q tile and 64 of the tile's 128 keys)
//     O += P V    (TS; P in each CTA's TMEM, each CTA holds 64 of V's 128 columns)
// so each SM reads half of every K/V tile from memory and serves one query
// tile with one softmax warpgroup.  TMEM per CTA (512 columns):
//     S_0 [0, 128)  S_1 [128, 256)   scores of consecutive key tiles
//     O_0 [256, 384) O_1 [384, 512)  output of consecutive items
// P (bf16) is written over the first 64 columns of its S buffer.  With S
// double-buffered the MMA order is S(j+1), PV(j): the scores of the next key
// tile are computed while the softmax works on this one.  With O
// double-buffered the next item's tiles start while this item's epilogue
// reads its output; the next item's first S is issued before this item's last
// PV whenever that item is already known.
//
// Roles (16 warps per CTA):
//   warp 0      TMA producer: item records (the even CTA fetches them from the
//               work counter and writes them into both CTAs' rings), the Q
//               tile and this CTA's halves of K_j and V_j in the order the
//               MMAs consume them (K_0, K_1, V_0, K_2, V_1, ..., V_{N-1}),
//               through a ring of 16 KB stages; every copy completes on the
//               even CTA's barrier.
//   warp 1      allocates the pair's TMEM; in the even CTA, issues the MMAs.
//   warps 4-11  softmax, two warpgroups taking the key tiles in turn:
//               warpgroup w takes every tile whose global number g has
//               g % 2 == w (so always S buffer w); thread = query row = TMEM
//               lane.  The running row max passes from one warpgroup to the
//               other through shared memory as soon as each tile's max is
//               known, before its exponentials, so the two warpgroups work
//               half a tile apart and hide each other's TMEM and MUFU
//               latencies.  Online max/sum in log2 units, p = 2^(s*scale*
//               log2e - m) as bf16 over S, lazy O rescale by whichever
//               warpgroup raises the max; each keeps its own partial row sum,
//               and both go to the epilogue with the max they were taken at.
//   warps 12-15 epilogue: O / l -> bf16 through a per-warp transposition
//               buffer, whole 128-byte row segments per store; exact zeros
//               for rows that see no key and for padded query rows.
// Key tiles wholly above the causal diagonal or past kv_len are never loaded.
#include "kernels.h"
#include "prefill_sched.cuh"
#include "ptx.cuh"

#include <mutex>

namespace attn {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr uint32_t kRegsLow = 40;        // warps 0-3 after setmaxnreg
constexpr uint32_t kRegsSoftmax = 200;   // warps 4-11
constexpr uint32_t kRegsEpilogue = 64;   // warps 12-15: 128 * (40 + 2 * 200 + 64) = 64512 <= 65536
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;     // lazy-rescale threshold (log2 units)
constexpr int kItemRing = 8;             // work items in flight between the roles
// Releases of one item record, one per warp: the MMA warp, 8 softmax and 4
// epilogue warps of the even CTA; the producer, 8 softmax and 4 epilogue
// warps of the odd one.
constexpr int kItemReleases = 26;
constexpr int kStages = 8;               // K/V ring stages
constexpr uint32_t kPReady = 8;          // one per warp of the tile's softmax warpgroup, both CTAs
constexpr uint32_t kOEmpty = 8;          // one per epilogue warp of both CTAs

// Shared memory (per CTA)
constexpr int kQBlock = 128 * 128;       // 128 rows x 64 columns, 128-byte swizzle
constexpr int kQBytes = 2 * kQBlock;     // one Q tile
constexpr int kKBlock = 64 * 128;        // 64 keys x 64 columns
constexpr int kStageBytes = 16384;       // K half: two 64-column blocks of 64 keys; V half: 64 columns of 128 keys
constexpr int kRingOff = 2 * kQBytes;
constexpr int kEpiOff = kRingOff + kStages * kStageBytes;
constexpr int kEpiBytes = 32 * 128;      // per epilogue warp: 32 rows x 64 columns bf16
constexpr int kStatOff = kEpiOff + 4 * kEpiBytes;  // [2][4][128] floats: per warpgroup row sum and its max
constexpr int kChainOff = kStatOff + 2 * 4 * 128 * 4;  // [2][128] floats: running max after a tile
constexpr int kBarOff = kChainOff + 2 * 128 * 4;
constexpr int kSmemBytes = kBarOff + 1024 + 1024;  // + barriers + alignment slack

struct Bars {
    uint64_t q_full[2];           // even CTA: both Q tiles in (tx)
    uint64_t q_empty[2];          // each CTA: last S MMA reading the buffer done
    uint64_t kv_full[kStages];    // even CTA: both halves in (tx)
    uint64_t kv_empty[kStages];   // each CTA: the MMA reading the stage done
    uint64_t s_full[2];           // each CTA: S MMA done
    uint64_t p_ready[2];          // even CTA: both CTAs' P written
    uint64_t pv_done;             // each CTA: one phase per PV MMA
    uint64_t o_full[2];           // each CTA: an item's last PV done
    uint64_t o_empty[2];          // even CTA: both CTAs' epilogues have read O
    uint64_t l_full[2];           // each CTA: softmax -> epilogue row statistics
    uint64_t l_empty[2];
    uint64_t m_ready[2][4];       // each CTA: running max of a tile published, per lane quarter
    uint64_t item_full[kItemRing];
    uint64_t item_empty[kItemRing];  // even CTA
    uint64_t mma_done;
    Item item[kItemRing];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 1024, "barrier block");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

constexpr int kItemWords = sizeof(Item) / 4;
static_assert(sizeof(Item) % 4 == 0, "item record");

__device__ __forceinline__ Item read_item(Bars &bars, int k) {
    const volatile int *src = reinterpret_cast<const volatile int *>(&bars.item[k % kItemRing]);
    Item it;
    int *dst = reinterpret_cast<int *>(&it);
#pragma unroll
    for (int w = 0; w < kItemWords; ++w) dst[w] = src[w];
    return it;
}

// Warp-wide: wait for record k, read it, release it.  Returns false on a
// timed-out wait.  The fields are broadcast from lane 0 so that the warp's
// control flow stays uniform.
__device__ __forceinline__ bool take_item_warp(Bars &bars, int k, bool even, uint32_t even_empty0, Item *it) {
    const int slot = k % kItemRing;
    // the odd CTA's records are written by the even CTA: acquire at cluster scope
    if (!(even ? mbar_wait_warp(&bars.item_full[slot], (k / kItemRing) & 1, &bars.abort)
               : mbar_wait_warp_cl(&bars.item_full[slot], (k / kItemRing) & 1, &bars.abort)))
        return false;
    Item v = read_item(bars, k);
    int *w = reinterpret_cast<int *>(&v);
#pragma unroll
    for (int i = 0; i < kItemWords; ++i) w[i] = __shfl_sync(0xffffffffu, w[i], 0);
    *it = v;
    __syncwarp();
    if (lane_id() == 0) {
        if (even)
            mbar_arrive(&bars.item_empty[slot]);
        else
            mbar_arrive_cluster_relaxed(even_empty0 + slot * 8);  // the record is in registers
    }
    return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tq,
                        const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                        const int n_major, const int group, const int front, const int n_items,
                        unsigned int *sched, const unsigned int epoch) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem + kRingOff;
    Bars &bars = *reinterpret_cast<Bars *>(smem + kBarOff);
    float *stat = reinterpret_cast<float *>(smem + kStatOff);

    const uint32_t rank = cluster_rank();  // 0: the even CTA, which issues the MMAs
    const bool even = rank == 0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars.q_full[x], 1);
            mbar_init(&bars.q_empty[x], 1);
            mbar_init(&bars.s_full[x], 1);
            mbar_init(&bars.p_ready[x], kPReady);
            mbar_init(&bars.o_full[x], 1);
            mbar_init(&bars.o_empty[x], kOEmpty);
            mbar_init(&bars.l_full[x], 8);
            mbar_init(&bars.l_empty[x], 4);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars.kv_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int w = 0; w < 2; ++w)
            for (int q = 0; q < 4; ++q) mbar_init(&bars.m_ready[w][q], 1);
        for (int s = 0; s < kItemRing; ++s) {
            mbar_init(&bars.item_full[s], 1);
            mbar_init(&bars.item_empty[s], kItemReleases);
        }
        mbar_init(&bars.pv_done, 1);
        mbar_init(&bars.mma_done, 1);
        bars.abort = 0;
        fence_mbar_init();
        if (even) {
            // claim the work counter for this launch (the first pair finds it
            // free, the others find this launch's epoch)
            const unsigned int owner = atomicExch(sched + 2, epoch);
            if (owner != 0u && owner != epoch) report_status(a.status, 0x22, kStatusSchedConflict);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars.tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    // barriers of the even CTA and of the other CTA, as cluster addresses
    const uint32_t peer = rank ^ 1u;

    if (warp == 0) {
        // ================================================================ TMA producer
        regs_dec<kRegsLow>();
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            const uint32_t q_full0 = cluster_addr(&bars.q_full[0], 0);
            const uint32_t kv_full0 = cluster_addr(&bars.kv_full[0], 0);
            const uint32_t item_empty0 = cluster_addr(&bars.item_empty[0], 0);
            const uint32_t peer_item_full0 = cluster_addr(&bars.item_full[0], peer);
            const uint32_t peer_item0 = cluster_addr(&bars.item[0], peer);
            int k = 0;  // item records taken so far
            // next item record: fetched and published by the even CTA, read by the odd one
            auto get_item = [&](Item *it) -> bool {
                const int slot = k % kItemRing;
                if (even) {
                    if (k >= kItemRing &&
                        !mbar_wait(&bars.item_empty[slot], ((k / kItemRing) - 1) & 1, &bars.abort))
                        return false;
                    const int t = static_cast<int>(atomicAdd(sched, 1u));
                    Item v;
                    if (t < n_items) {
                        v = decode_item(t, a, n_major, group, front);
                    } else {
                        v = Item{0, 0, 0, 0, 0, 0, 0, {0, 0}, -1};
                    }
                    const int *w = reinterpret_cast<const int *>(&v);
                    volatile int *mine = reinterpret_cast<volatile int *>(&bars.item[slot]);
#pragma unroll
                    for (int i = 0; i < kItemWords; ++i) {
                        mine[i] = w[i];
                        st_cluster_u32(peer_item0 + slot * sizeof(Item) + 4 * i, static_cast<uint32_t>(w[i]));
                    }
                    mbar_arrive(&bars.item_full[slot]);
                    mbar_arrive_cluster(peer_item_full0 + slot * 8);
                    *it = v;
                } else {
                    if (!mbar_wait_cl(&bars.item_full[slot], (k / kItemRing) & 1, &bars.abort)) return false;
                    *it = read_item(bars, k);
                    mbar_arrive_cluster_relaxed(item_empty0 + slot * 8);
                }
                ++k;
                return true;
            };
            auto next_nonempty = [&](Item *it) -> bool {
                do {
                    if (!get_item(it)) return false;
                } while (it->N == 0);
                return true;
            };
            uint32_t q_uses = 0;  // Q tiles loaded
            int issued = 0;       // ring loads issued
            auto load_q = [&](const Item &it) -> bool {
                const uint32_t qb = q_uses & 1u;
                if (q_uses >= 2 && !mbar_wait(&bars.q_empty[qb], ((q_uses >> 1) - 1) & 1, &bars.abort))
                    return false;
                if (even) mbar_arrive_expect_tx(&bars.q_full[qb], 2 * kQBytes);
                const int row = it.row_base + static_cast<int>(rank) * it.row_step;
                const int bh = it.bh_base + static_cast<int>(rank) * it.bh_step;
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    tma_load_3d_pair(smem + qb * kQBytes + c * kQBlock, &tq, q_full0 + qb * 8, c * 64, row, bh);
                ++q_uses;
                return true;
            };
            // this CTA's half of K_j (kv = 0: keys 64*rank .. +63, all columns)
            // or of V_j (kv = 1: columns 64*rank .. +63 of all 128 keys)
            auto load_kv = [&](const Item &it, int j, int kv) -> bool {
                const int s = issued % kStages;
                if (issued >= kStages &&
                    !mbar_wait(&bars.kv_empty[s], ((issued / kStages) - 1) & 1, &bars.abort))
                    return false;
                if (even) mbar_arrive_expect_tx(&bars.kv_full[s], 2 * kStageBytes);
                uint8_t *dst = ring + s * kStageBytes;
                if (kv == 0) {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d_pair(dst + c * kKBlock, &tk, kv_full0 + s * 8, c * 64,
                                         j * kBN + 64 * static_cast<int>(rank), it.bh_kv);
                } else {
                    tma_load_3d_pair(dst, &tv, kv_full0 + s * 8, 64 * static_cast<int>(rank), j * kBN, it.bh_kv);
                }
                ++issued;
                return true;
            };
            Item cur;
            bool ok = next_nonempty(&cur);
            while (ok && cur.N > 0) {
                ok = load_q(cur) && load_kv(cur, 0, 0);
                for (int j = 1; j < cur.N && ok; ++j) ok = load_kv(cur, j, 0) && load_kv(cur, j - 1, 1);
                if (ok) ok = load_kv(cur, cur.N - 1, 1);
                // every load of this item is issued before waiting for the next record
                if (ok) ok = next_nonempty(&cur);
            }
            // never leave with copies still landing in shared memory: the even
            // CTA's barriers count both CTAs' bytes
            if (even) {
                volatile int never = 0;
                for (uint32_t u = q_uses > 2 ? q_uses - 2 : 0; u < q_uses; ++u)
                    mbar_wait(&bars.q_full[u & 1], (u >> 1) & 1, &never);
                for (int u = max(0, issued - kStages); u < issued; ++u)
                    mbar_wait(&bars.kv_full[u % kStages], (u / kStages) & 1, &never);
            }
        }
    } else if (warp == 1) {
        regs_dec<kRegsLow>();
        if (even) {
            // ============================================================ MMA issuer (even CTA)
            const uint32_t idesc_s = idesc_bf16_f32(256, kBN, 0);
            const uint32_t idesc_o = idesc_bf16_f32(256, kD, 1);
            const uint64_t dq0 = sdesc_sw128(smem_u32(smem), 16, 1024);
            const uint64_t dk0 = sdesc_sw128(smem_u32(ring), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(ring), kKBlock, 1024);
            // a barrier's cluster address in either CTA: same offset from the
            // barrier block, whose base in the odd CTA comes from mapa
            const uint32_t bars_local = smem_u32(&bars), bars_odd = cluster_addr(&bars, 1);
            auto commit2 = [&](uint64_t *bar) {
                const uint32_t off = smem_u32(bar) - bars_local;
                tc_commit_pair_warp(bars_local + off);
                tc_commit_pair_warp(bars_odd + off);
            };
            // S into buffer sb from Q buffer qb and the K half in ring stage st
            auto issue_s = [&](uint32_t qb, uint32_t sb, int st) {
                const uint64_t da = desc_add(dq0, (qb * kQBytes) >> 4);
                const uint64_t db = desc_add(dk0, (st * kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t qoff = ((kk / 4) * kQBlock + (kk % 4) * 32) >> 4;
                    const uint32_t koff = ((kk / 4) * kKBlock + (kk % 4) * 32) >> 4;
                    mma_ss_pair_warp(tmem + sb * 128u, desc_add(da, qoff), desc_add(db, koff), idesc_s, kk > 0);
                }
            };
            // O_ob += P(sb) V, V half in ring stage st
            auto issue_pv = [&](uint32_t ob, uint32_t sb, int st, bool acc) {
                const uint64_t db = desc_add(dv0, (st * kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts_pair_warp(tmem + 256u + ob * 128u, tmem + sb * 128u + kk * 8, desc_add(db, (kk * 16 * 128) >> 4),
                                     idesc_o, (acc || kk > 0) ? 1u : 0u);
            };
            int k = 0;            // item records taken
            uint32_t gs = 0;      // S MMAs issued (buffer gs & 1)
            uint32_t gp = 0;      // PV MMAs issued
            uint32_t u = 0;       // items with work started (Q and O buffer u & 1)
            bool ok = true;
            auto wait_stage = [&](int idx) -> bool {
                if (!mbar_wait_warp(&bars.kv_full[idx % kStages], (idx / kStages) & 1, &bars.abort)) return false;
                tc_fence_after();
                return true;
            };
            // ring load index of K_j and V_j of an item whose first load has index b (load order
            // K_0, K_1, V_0, K_2, V_1, ..., K_{N-1}, V_{N-2}, V_{N-1})
            auto idx_k = [](int b, int j) { return j == 0 ? b : b + 2 * j - 1; };
            auto idx_v = [](int b, int j, int N) { return j == N - 1 ? b + 2 * N - 1 : b + 2 * j + 2; };
            // first S of an item (Q buffer uu & 1, K_0 at ring index b)
            auto first_s = [&](const Item &it, uint32_t uu, int b) -> bool {
                const uint32_t qb = uu & 1u;
                if (!mbar_wait_warp(&bars.q_full[qb], (uu >> 1) & 1, &bars.abort)) return false;
                if (!wait_stage(b)) return false;
                issue_s(qb, gs & 1u, b % kStages);
                commit2(&bars.s_full[gs & 1u]);
                ++gs;
                commit2(&bars.kv_empty[b % kStages]);
                if (it.N == 1) commit2(&bars.q_empty[qb]);
                return true;
            };
            Item cur;
            int base = 0;  // ring index of the current item's K_0
            bool s0 = false;
            // the first item: blocking takes (no MMA is outstanding)
            do {
                ok = take_item_warp(bars, k++, true, 0, &cur);
            } while (ok && cur.N == 0);
            while (ok && cur.N > 0) {
                const int N = cur.N;
                const uint32_t ob = u & 1u;
                if (!s0 && !(ok = first_s(cur, u, base))) break;
                s0 = false;
                Item nxt;
                bool have_nxt = false;
                for (int j = 0; j < N && ok; ++j) {
                    if (j + 1 < N) {
                        const int ik = idx_k(base, j + 1);
                        if (!(ok = wait_stage(ik))) break;
                        issue_s(ob, gs & 1u, ik % kStages);
                        commit2(&bars.s_full[gs & 1u]);
                        ++gs;
                        commit2(&bars.kv_empty[ik % kStages]);
                        if (j + 2 == N) commit2(&bars.q_empty[ob]);
                    } else {
                        // the next item's first S ahead of this item's last PV, if
                        // its record is already published (never block here: the
                        // record may wait for this item's epilogue to free a slot)
                        for (;;) {
                            const bool pub = __all_sync(0xffffffffu,
                                                        mbar_test_wait_cl(&bars.item_full[k % kItemRing], (k / kItemRing) & 1));
                            if (!pub) break;
                            if (!(ok = take_item_warp(bars, k++, true, 0, &nxt))) break;
                            if (nxt.N != 0) {
                                have_nxt = true;
                                break;
                            }
                        }
                        if (!ok) break;
                        if (have_nxt && nxt.N > 0) {
                            if (!(ok = first_s(nxt, u + 1, base + 2 * N))) break;
                            s0 = true;
                        }
                    }
                    const int iv = idx_v(base, j, N);
                    if (!(ok = wait_stage(iv))) break;
                    if (j == 0 && u >= 2 && !(ok = mbar_wait_warp(&bars.o_empty[ob], ((u >> 1) - 1) & 1, &bars.abort)))
                        break;
                    if (!(ok = mbar_wait_warp(&bars.p_ready[gp & 1u], (gp >> 1) & 1, &bars.abort))) break;
                    tc_fence_after();
                    issue_pv(ob, gp & 1u, iv % kStages, j > 0);
                    commit2(&bars.pv_done);
                    commit2(&bars.kv_empty[iv % kStages]);
                    if (j == N - 1) commit2(&bars.o_full[ob]);
                    ++gp;
                }
                if (!ok) break;
                ++u;
                base += 2 * N;
                if (have_nxt) {
                    cur = nxt;
                } else {
                    do {
                        ok = take_item_warp(bars, k++, true, 0, &cur);
                    } while (ok && cur.N == 0);
                }
            }
            // every MMA must have finished before TMEM is released
            tc_commit_pair_warp(smem_u32(&bars.mma_done));
            volatile int never = 0;
            mbar_wait_warp(&bars.mma_done, 0, &never);
        }
    } else if (warp < 4) {
        regs_dec<kRegsLow>();  // warps 2-3: no role, registers go to the softmax warps
    } else if (warp < 12) {
        // ================================================================ softmax
        regs_inc<kRegsSoftmax>();
        const uint32_t w = (warp - 4) / 4;  // this warpgroup takes the tiles g with g % 2 == w
        const int quarter = warp % 4;       // TMEM lanes [32*quarter, 32*quarter + 32)
        const int r = quarter * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t t_s = t_lane + w * 128u;  // S buffer w
        const float sl2 = a.scale * kLog2e;
        float *chain = reinterpret_cast<float *>(smem + kChainOff);
        const uint32_t item_empty0 = cluster_addr(&bars.item_empty[0], 0);
        const uint32_t p_ready0 = cluster_addr(&bars.p_ready[0], 0);
        uint32_t g = 0, u = 0;  // global tiles seen, items with work
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Item it;
            if (!(ok = take_item_warp(bars, k, even, item_empty0, &it))) break;
            if (it.N < 0) break;
            if (it.N == 0) continue;
            const int N = it.N;
            const uint32_t ob = u & 1u;
            const uint32_t t_o = t_lane + 256u + ob * 128u;
            const int i = it.row_base + static_cast<int>(rank) * it.row_step + r;  // query row
            const int n_mine = rank ? it.n_kv[1] : it.n_kv[0];
            int lim = a.causal ? min(it.Lb, i + it.off + 1) : it.Lb;  // keys [0, lim) visible
            if (n_mine == 0) lim = 0;
            // m_w: the running max this warpgroup's sum l is kept at
            float m_w = -INFINITY, l = 0.f;
            for (int j = 0; j < N; ++j, ++g) {
                if ((g & 1u) != w) continue;  // the other warpgroup's tile
                // the running max after the previous tile (every tile waits for it, so
                // that neither warpgroup runs ahead; the first tile of an item ignores it)
                float m_prev = -INFINITY;
                if (g > 0) {
                    if (!(ok = mbar_wait_warp(&bars.m_ready[w ^ 1u][quarter], ((g - 1) >> 1) & 1, &bars.abort)))
                        break;
                    if (j > 0) m_prev = chain[(w ^ 1u) * 128 + r];
                }
                if (m_prev > m_w) {  // the other warpgroup raised the max: bring l to it
                    if (m_w != -INFINITY) l *= ex2_approx(m_w - m_prev);
                    m_w = m_prev;
                }
                if (!(ok = mbar_wait_warp<32>(&bars.s_full[w], (g >> 1) & 1, &bars.abort))) break;
                tc_fence_after();
                // This row sees columns [0, t) of the tile.  A tile hidden from every
                // row of the warp skips its loads and exponentials and writes P = 0;
                // on a tile that crosses the causal diagonal or the padding edge each
                // warp sorts its 32-column chunks into seen by all its rows, hidden from
                // all of them and partial (per-column select).
                const int t = lim - j * kBN;
                const int t_hi = __reduce_max_sync(0xffffffffu, t);
                const bool hidden = t_hi <= 0;
                uint32_t s[128];
                float mraw = -INFINITY;
                bool need_mask = false;
                int t_lo = kBN;
                if (!hidden) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, s + c * 32);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c) reg_fence32(s + c * 32);
                    need_mask = __any_sync(0xffffffffu, t < kBN);
                    if (need_mask) t_lo = __reduce_min_sync(0xffffffffu, t);
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
                    mraw = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
                }
                const float m_tile = mraw == -INFINITY ? -INFINITY : mraw * sl2;
                const float m_new = fmaxf(m_w, m_tile);
                const bool grow = m_new > m_w + kRescaleLog2;
                const float m_old = m_w;
                if (grow) {
                    if (m_w != -INFINITY) l *= ex2_approx(m_w - m_new);
                    m_w = m_new;
                }
                // publish the running max after this tile to the other warpgroup
                chain[w * 128 + r] = m_w;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.m_ready[w][quarter]);
                if (j > 0 && __any_sync(0xffffffffu, grow)) {
                    // O holds earlier tiles of this item at the max m_old: bring it to
                    // the new one once the previous PV has landed (S(g) completing
                    // implies PV(g - 2) has, so only PV(g - 1) can still be running)
                    const float factor = grow && m_old != -INFINITY ? ex2_approx(m_old - m_new) : 1.f;
                    if (!(ok = mbar_wait_warp(&bars.pv_done, (g - 1) & 1, &bars.abort))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < kD / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(t_o + c * 32, o);
                        tmem_ld_wait();
                        reg_fence32(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = f2u(u2f(o[e]) * factor);
                        tmem_st32(t_o + c * 32, o);
                    }
                }
                if (hidden) {
                    uint32_t z[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) z[e] = 0u;
                    tmem_st32(t_s, z);
                    tmem_st32(t_s + 32, z);
                } else {
                    const float negm = m_w == -INFINITY ? 0.f : -m_w;
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
                    for (int hh = 0; hh < 2; ++hh) {  // two halves of 64 keys -> 32 packed columns each
                        uint32_t p[32];
                        if (!need_mask) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) ATTN_EXP_PAIR(hh * 64 + 2 * e, e, false)
                        } else {
#pragma unroll
                            for (int cc = 0; cc < 2; ++cc) {
                                const int c = 2 * hh + cc;
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
                        tmem_st32(t_s + hh * 32, p);
                    }
#undef ATTN_EXP_PAIR
                    const uint64_t l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
                    l += f2_lo(l2) + f2_hi(l2);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (even)
                        mbar_arrive(&bars.p_ready[w]);
                    else
                        mbar_arrive_cluster_relaxed(p_ready0 + w * 8);  // every lane's P is in TMEM
                }
            }
            if (!ok) break;
            // this warpgroup's row sum, and the max it is kept at, to the epilogue
            if (u >= 2 && !(ok = mbar_wait_warp(&bars.l_empty[ob], ((u >> 1) - 1) & 1, &bars.abort))) break;
            stat[(ob * 4 + 2 * w) * 128 + r] = l;
            stat[(ob * 4 + 2 * w + 1) * 128 + r] = m_w;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.l_full[ob]);
            ++u;
        }
    } else {
        // ================================================================ epilogue
        regs_dec<kRegsEpilogue>();
        const int quarter = warp % 4;
        const int r = quarter * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t stage = smem_u32(smem + kEpiOff + quarter * kEpiBytes);
        const uint32_t item_empty0 = cluster_addr(&bars.item_empty[0], 0);
        const uint32_t o_empty0 = cluster_addr(&bars.o_empty[0], 0);
        uint32_t u = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Item it;
            if (!(ok = take_item_warp(bars, k, even, item_empty0, &it))) break;
            if (it.N < 0) break;
            const int row0 = it.row_base + static_cast<int>(rank) * it.row_step;
            const int i = row0 + r;
            const int bh = it.bh_base + static_cast<int>(rank) * it.bh_step;
            bool zero_row = true;
            float inv = 0.f, m_row = -INFINITY, l = 0.f;
            uint32_t ob = 0;
            const bool have_o = it.N > 0;
            if (have_o) {
                ob = u & 1u;
                if (!(ok = mbar_wait_warp(&bars.l_full[ob], (u >> 1) & 1, &bars.abort))) break;
                // O is kept at the larger of the two warpgroups' maxima (the running
                // max after the item's last tile); each partial sum is brought to it
                const float l0 = stat[(ob * 4 + 0) * 128 + r], m0 = stat[(ob * 4 + 1) * 128 + r];
                const float l1 = stat[(ob * 4 + 2) * 128 + r], m1 = stat[(ob * 4 + 3) * 128 + r];
                m_row = fmaxf(m0, m1);
                if (m_row != -INFINITY)
                    l = (l0 > 0.f ? l0 * ex2_approx(m0 - m_row) : 0.f) + (l1 > 0.f ? l1 * ex2_approx(m1 - m_row) : 0.f);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.l_empty[ob]);
                if (!(ok = mbar_wait_warp(&bars.o_full[ob], (u >> 1) & 1, &bars.abort))) break;
                tc_fence_after();
                zero_row = (a.kv_len && !a.chunked && a.Sq == a.Skv && i >= it.Lb) || !(l > 0.f);
                inv = zero_row ? 0.f : 1.f / l;
                ++u;
            }
            // log(sum_j exp(scale * s_j)) = ln 2 * (m + log2 l): l is kept relative to
            // the running max whether or not the lazy rescale has moved it
            if (a.lse && i < a.Sq)
                a.lse[static_cast<size_t>(bh) * a.Sq + i] =
                    zero_row ? -INFINITY : (m_row + log2f(l)) * 0.6931471805599453f;
            __nv_bfloat16 *obh = static_cast<__nv_bfloat16 *>(a.out) + static_cast<size_t>(bh) * a.Sq * kD;
            const int wrow0 = row0 + quarter * 32;  // first row of this warp
            const uint32_t t_o = t_lane + 256u + ob * 128u;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                // columns [64c, 64c + 64) of this row, loaded 32 at a time
                __syncwarp();  // the previous pass has read the buffer back
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t o[32];
                    if (have_o) {
                        tmem_ld32(t_o + c * 64 + hh * 32, o);
                        tmem_ld_wait();
                        reg_fence32(o);
                        if (c == 1 && hh == 1) {  // every TMEM read of this buffer is done: hand it back
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                if (even)
                                    mbar_arrive(&bars.o_empty[ob]);
                                else
                                    mbar_arrive_cluster_relaxed(o_empty0 + ob * 8);
                            }
                        }
                    }
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {  // 16-byte chunk 4*hh + k4 of this row's 64 columns
                        const int k8 = 4 * hh + k4;
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = k4 * 8 + 2 * e;
                            pk[e] = zero_row ? 0u : pack_bf16x2(u2f(o[col]) * inv, u2f(o[col + 1]) * inv);
                        }
                        st_shared_v4(stage + lane * 128 + ((k8 ^ (lane & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
                    }
                }
                __syncwarp();
#pragma unroll
                for (int s4 = 0; s4 < 8; ++s4) {  // rows 4*s4 .. 4*s4 + 3, one 16-byte chunk per lane
                    const int rr = 4 * s4 + (lane >> 3), ch = lane & 7;
                    const uint4 v = ld_shared_v4(stage + rr * 128 + ((ch ^ (rr & 7)) << 4));
                    const int row = wrow0 + rr;
                    if (row < a.Sq)
                        *reinterpret_cast<uint4 *>(obh + static_cast<size_t>(row) * kD + c * 64 + ch * 8) = v;
                }
            }
        }
    }

    // No CTA of the pair leaves (or frees TMEM) while the other may still
    // reach its shared memory or TMEM.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        __syncwarp();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
    if (threadIdx.x == 0) {
        if (bars.abort) report_timeout(a.status, 0x21);
        if (even) {
            // Every producer of this launch has taken its last item once all
            // pairs have counted themselves here: the last one resets the slot.
            __threadfence();
            if (atomicAdd(sched + 1, 1u) == gridDim.x / 2 - 1) {
                atomicExch(sched, 0u);
                atomicExch(sched + 1, 0u);
                atomicExch(sched + 2, 0u);
                __threadfence();
            }
        }
    }
}

constexpr int kMaxDevices = 64;
std::mutex g_pair_mutex;
int g_max_clusters[kMaxDevices];

// Pairs that can be resident at once on the current device.
int max_pairs(int n_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return n_sm / 2;
    std::lock_guard<std::mutex> lock(g_pair_mutex);
    if (!g_max_clusters[dev]) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(n_sm / 2 * 2), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = n_sm / 2;
        }
        g_max_clusters[dev] = n;
    }
    return g_max_clusters[dev];
}

}  // namespace

cudaError_t launch_prefill_pair(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv) {
    cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    const int n_sm = a.n_sm > 1 ? a.n_sm : 2;
    const long long units = max_pairs(n_sm);
    ItemPlan plan;
    bool too_many = false;
    if (!plan_items(a, units, &plan, &too_many)) return too_many ? cudaErrorInvalidConfiguration : cudaSuccess;
    unsigned int *sched = nullptr, epoch = 0;
    e = sched_slot(a.stream, &sched, &epoch);
    if (e != cudaSuccess) return e;
    const long long pairs = plan.n_items < units ? plan.n_items : units;
    prefill_pair_kernel<<<static_cast<unsigned>(2 * pairs), kThreads, kSmemBytes, a.stream>>>(
        a, tq, tk, tv, plan.n_major, plan.group, plan.front, plan.n_items, sched, epoch);
    return cudaGetLastError();
}

}  // namespace attn
