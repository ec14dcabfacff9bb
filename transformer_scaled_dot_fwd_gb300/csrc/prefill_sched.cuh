// Work items of the bf16 prefill kernel (prefill_tc.cu) and their order.
//
// A work item is two 128-row query tiles that read the same key/value head.
// Items are numbered in blocks of heads whose keys and values fit in part of
// L2, longest-first inside a block (causal cost grows with the row), and
// handed out at run time by an atomic counter, so each processing unit takes
// the next item when it is ready for it.
#pragma once

#include "kernels.h"

namespace attn {

constexpr int kBM = 128;       // query rows per Q tile (one TMEM lane each)
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kQTiles = 2;     // Q tiles per work item
constexpr int kSchedSlots = 64;       // direct launches that may run at once with their own counter
constexpr int kGraphSlots = 1024;     // counters kept for launches captured into CUDA graphs
// Bytes of keys and values per block of heads in the item order (see
// decode_item); 0 puts all heads in one block.
#ifndef ATTN_L2_GROUP_MB
#define ATTN_L2_GROUP_MB 16
#endif
constexpr long long kL2GroupBytes = static_cast<long long>(ATTN_L2_GROUP_MB) << 20;
// Work per processing unit of the last block, in units of the longest item, times 10.
#ifndef ATTN_TAIL_X10
#define ATTN_TAIL_X10 20
#endif
constexpr long long kTailFactorX10 = ATTN_TAIL_X10;

// One work item: two 128-row query tiles that read the same key/value head.
// Multi-head attention (and grouped-query attention with an odd group size)
// pairs query tiles 2p and 2p + 1 of one head; grouped-query attention with an
// even group size pairs query tile qt of heads 2m and 2m + 1 of one group, so
// each K/V tile loaded into shared memory serves two heads.
struct Item {
    // Query tile x starts at row row_base + x * row_step of head bh_base + x * bh_step
    // (b * H + h); scalars, so that a runtime x never indexes a local array.
    int row_base, row_step, bh_base, bh_step;
    int bh_kv;          // b * H_kv + h / G: the key/value head both tiles read
    int Lb;
    int off;            // causal: key j visible from query row i iff j <= i + off
    int n_kv[kQTiles];  // K/V tiles each query tile needs (0: tile empty or fully padded)
    int N;              // max of n_kv
};

__device__ __forceinline__ bool pairs_heads(const FwdArgs &a) { return ((a.H / a.H_kv) & 1) == 0; }

// Work item t -> (query rows, heads).  The minor index u runs over the M
// head units (heads, or head pairs of one group), the major index over the
// n_major query-tile units (query-tile pairs per head with tile pairing, or
// query tiles with head pairing).  Head units are taken in blocks: the first
// `front` units in blocks of `group`, the rest as one last block; inside a
// block the longest rows come first.  A front block's keys and values are
// sized to stay in L2 while its items run, so the items of one head that run
// side by side share each K/V tile from L2; the last block is large enough
// that its longest items still start early (longest-processing-time order
// at the end of the launch).
__device__ __forceinline__ Item decode_item(int t, const FwdArgs &a, int n_major, int group, int front) {
    Item it;
    const int G = a.H / a.H_kv;
    const bool hp = pairs_heads(a);
    const int M = hp ? a.B * (a.H / 2) : a.B * a.H;
    int base, cg;
    if (t < front * n_major) {
        base = (t / (group * n_major)) * group;
        cg = group;
    } else {
        base = front;
        cg = M - front;
    }
    const int tt = t - base * n_major;
    const int major = n_major - 1 - tt / cg;  // longest rows first
    const int u = base + tt % cg;
    int b, h0;
    if (hp) {
        const int HP = a.H / 2;
        b = u / HP;
        h0 = 2 * (u % HP);
        it.row_base = major * kBM;
        it.row_step = 0;
        it.bh_base = b * a.H + h0;
        it.bh_step = 1;
    } else {
        b = u / a.H;
        h0 = u % a.H;
        it.row_base = major * kQTiles * kBM;
        it.row_step = kBM;
        it.bh_base = u;
        it.bh_step = 0;
    }
    it.bh_kv = b * a.H_kv + h0 / G;
    it.Lb = a.Skv;
    if (a.kv_len) it.Lb = min(max(a.kv_len[b], 0), a.Skv);
    // Chunk against a cache: the Sq queries are the last Sq positions of the
    // sequence's L_b; otherwise the last query is aligned with the last key.
    it.off = a.chunked ? it.Lb - a.Sq : a.Skv - a.Sq;
    // rows i >= L_b of a right-padded self-attention batch (with Sq != Skv,
    // non-causal cross-attention, kv_len masks keys only)
    const bool query_padding = a.kv_len && !a.chunked && a.Sq == a.Skv;
    it.N = 0;
#pragma unroll
    for (int x = 0; x < kQTiles; ++x) {
        const int row0 = it.row_base + x * it.row_step;
        int n = 0;
        if (row0 < a.Sq && !(query_padding && row0 >= it.Lb)) {
            int last = min(a.Sq - 1, row0 + kBM - 1);
            if (query_padding) last = min(last, it.Lb - 1);
            const int hi = a.causal ? min(it.Lb, last + it.off + 1) : it.Lb;
            n = (max(hi, 0) + kBN - 1) / kBN;
        }
        it.n_kv[x] = n;
        it.N = max(it.N, n);
    }
    return it;
}

// How a launch numbers its items (decode_item's parameters), for `units`
// processing units running side by side.  Returns false when there is no
// item; n_items > 2^31 - 1 is reported through *too_many.
struct ItemPlan {
    int n_major, group, front, n_items;
};

inline bool plan_items(const FwdArgs &a, long long units, ItemPlan *plan, bool *too_many) {
    const int D = a.D;
    const int n_qt = (a.Sq + kBM - 1) / kBM;
    const bool head_pairs = ((a.H / a.H_kv) & 1) == 0;  // as pairs_heads()
    const int n_major = head_pairs ? n_qt : (n_qt + kQTiles - 1) / kQTiles;
    const long long n_items = head_pairs ? static_cast<long long>(a.B) * (a.H / 2) * n_qt
                                         : static_cast<long long>(a.B) * a.H * n_major;
    *too_many = n_items > 0x7fffffffLL;
    if (n_items <= 0 || *too_many) return false;
    units = units > 0 ? units : 1;
    const long long grid = n_items < units ? n_items : units;
    // Blocks of the item order (decode_item).  Front blocks hold as many head
    // units as keep their K and V (a key/value head serves G heads, or G/2
    // head pairs) within kL2GroupBytes.  The last block holds at least
    // enough units that its work per SM is kTailFactor times the longest
    // item; with fewer units than that, one block holds them all.
    const long long M = head_pairs ? static_cast<long long>(a.B) * (a.H / 2) : static_cast<long long>(a.B) * a.H;
    long long group = M, front = 0;
    if (kL2GroupBytes > 0) {
        const long long units_per_kv = head_pairs ? (a.H / a.H_kv) / 2 : (a.H / a.H_kv);
        const long long kv_head_bytes = 2LL * a.Skv * D * 2;
        long long c_l2 = kL2GroupBytes * units_per_kv / (kv_head_bytes > 0 ? kv_head_bytes : 1);
        c_l2 = c_l2 > 1 ? c_l2 : 1;
        // K/V steps per head unit and of the longest item, all sequences at full length
        const int off = a.Skv - a.Sq;
        long long unit_steps = 0, max_steps = 0;
        for (int m = 0; m < n_major; ++m) {
            long long n = 0;
            for (int x = 0; x < (head_pairs ? 1 : kQTiles); ++x) {
                const int row0 = head_pairs ? m * kBM : (m * kQTiles + x) * kBM;
                if (row0 >= a.Sq) continue;
                const int last = row0 + kBM - 1 < a.Sq - 1 ? row0 + kBM - 1 : a.Sq - 1;
                int hi = a.causal ? (last + off + 1 < a.Skv ? last + off + 1 : a.Skv) : a.Skv;
                hi = hi > 0 ? hi : 0;
                const long long nx = (hi + kBN - 1) / kBN;
                n = nx > n ? nx : n;
            }
            unit_steps += n;
            max_steps = n > max_steps ? n : max_steps;
        }
        const long long c_tail = unit_steps > 0
            ? (kTailFactorX10 * max_steps * static_cast<long long>(grid) + 10 * unit_steps - 1) / (10 * unit_steps)
            : M;
        if (c_l2 < M && c_tail < M) {
            const long long n_front = (M - c_tail) / c_l2;
            if (n_front > 0) {
                group = c_l2;
                front = n_front * c_l2;
            }
        }
    }
    plan->n_major = n_major;
    plan->group = static_cast<int>(group);
    plan->front = static_cast<int>(front);
    plan->n_items = static_cast<int>(n_items);
    return true;
}

}  // namespace attn
