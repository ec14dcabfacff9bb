// Split-KV decode for grouped-query and multi-query attention (H_kv < H).
//
// Query head h reads key/value head h / G, G = H / H_kv ("Attention from First
// Principles", section 5 and "MHA, GQA, MQA -- the KV cache lever"; "Scaled
// dot-product attention with masking", "Grouped-query attention (GQA)").
// Decode reads the whole cache once per step; with G query heads per cached
// head, one read can serve all G of them, which raises the arithmetic
// intensity of decode from about one flop per byte to about G ("Attention
// from First Principles", section 6 "Under the hood": intensity equals the
// GQA ratio).
//
//   partial kernel  one CTA per (b, h_kv, subgroup of up to GT query heads,
//                   chunk of keys).  A producer warp streams the chunk's K
//                   rows, then its V rows, into a 4-stage shared-memory ring
//                   (64 keys per bulk copy); four consumer warps compute the
//                   GT heads' scores for each key (8 lanes per key, one K read
//                   serving every head), each head's chunk max and sum, and
//                   sum_j p_j v_j for every head from one V read.  Partials go
//                   to the same per-query-head layout as the multi-head decode,
//                   so the same combine kernel finishes the job.
//
// Groups larger than GT (16, 32) are split into subgroups of GT heads that
// each stream the chunk; their CTAs run side by side, so the repeated reads
// of a chunk mostly hit L2.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kTileKeys = 64;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxChunk = kDecodeGqaMaxChunk;  // keys per CTA (bounds the score buffer)
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int GT>
struct __align__(128) GqaSmem {
    __nv_bfloat16 tile[kStages][kTileKeys * D];
    float qs[GT][D];                    // this subgroup's queries, scaled to log2 units
    float s[kMaxChunk * GT];            // [key][head]: scores, then probabilities
    float ml[kConsumerWarps][GT];       // per-warp partial max, then sum
    uint64_t full[kStages], empty[kStages];
    int abort;
};

template <int D, int GT>
__global__ void __launch_bounds__(kThreads) decode_gqa_partial_kernel(DecodeArgs a, int n_sub) {
    griddep_launch_dependents();
    griddep_wait();  // launched back to back: the previous kernel's writes are visible
    extern __shared__ __align__(128) uint8_t smem_raw[];
    GqaSmem<D, GT> &sm = *reinterpret_cast<GqaSmem<D, GT> *>(smem_raw);

    const int G = a.H / a.H_kv;
    const int c = blockIdx.x % a.n_split;
    const int rest = blockIdx.x / a.n_split;
    const int sg = rest % n_sub;
    const int bkv = rest / n_sub;  // b * H_kv + h_kv
    const int b = bkv / a.H_kv, hkv = bkv % a.H_kv;
    const int h_first = hkv * G + sg * GT;  // first query head of this subgroup
    const int ng = min(GT, G - sg * GT);    // heads in this subgroup
    int L = a.Skv;
    if (a.kv_len) L = min(max(a.kv_len[b], 0), a.Skv);
    const int k0 = c * a.chunk;
    if (k0 >= L) return;  // the combine kernel reads only chunks below L
    const int nkeys = min(a.chunk, L - k0);
    const int ntiles = (nkeys + kTileKeys - 1) / kTileKeys;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    // queries of the subgroup (absent heads of a partial subgroup read as zero)
    const float sl2 = a.scale * kLog2e;
    for (int e = threadIdx.x; e < GT * D; e += kThreads) {
        const int g = e / D, d = e % D;
        float x = 0.f;
        if (g < ng) {
            const __nv_bfloat16 *qp =
                static_cast<const __nv_bfloat16 *>(a.q) + (static_cast<size_t>(b) * a.H + h_first + g) * D;
            x = __bfloat162float(qp[d]) * sl2;
        }
        sm.qs[g][d] = x;
    }
    __syncthreads();

    const size_t row0 = static_cast<size_t>(bkv) * a.Skv + k0;
    const __nv_bfloat16 *Kp = static_cast<const __nv_bfloat16 *>(a.k) + row0 * D;
    const __nv_bfloat16 *Vp = static_cast<const __nv_bfloat16 *>(a.v) + row0 * D;

    if (warp == kConsumerWarps) {
        // ---------------- producer: K tiles 0..ntiles-1, then V tiles
        if (lane == 0) {
            const int total = 2 * ntiles;
            int t = 0;
            for (; t < total; ++t) {
                const int slot = t % kStages;
                if (t >= kStages && !mbar_wait(&sm.empty[slot], ((t / kStages) - 1) & 1, &sm.abort)) break;
                const int tt = t < ntiles ? t : t - ntiles;
                const int rows = min(kTileKeys, nkeys - tt * kTileKeys);
                const uint32_t bytes = static_cast<uint32_t>(rows) * D * 2;
                const __nv_bfloat16 *src = (t < ntiles ? Kp : Vp) + static_cast<size_t>(tt) * kTileKeys * D;
                mbar_arrive_expect_tx(&sm.full[slot], bytes);
                bulk_load(sm.tile[slot], src, bytes, &sm.full[slot]);
            }
            // do not leave the CTA with copies still landing in shared memory
            for (int u = max(0, t - kStages); u < t; ++u) {
                volatile int never = 0;
                mbar_wait(&sm.full[u % kStages], (u / kStages) & 1, &never);
            }
            if (sm.abort) report_timeout(a.status, 0x31);
        }
        return;
    }

    // ---------------- consumers: scores.  8 lanes per key, 4 keys per warp
    // step; lane (kg, t8) owns dims [64u + 8 t8, 64u + 8 t8 + 8) of key kg and
    // keeps those dims of the GT queries in registers.
    constexpr int NQ = D / 64;
    constexpr int LG = GT >= 8 ? 3 : (GT >= 4 ? 2 : 1);  // log2(GT)
    const int kg = lane / 8, t8 = lane % 8;
    float qf[GT][NQ * 8];
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
        for (int u = 0; u < NQ; ++u)
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[g][u * 8 + e] = sm.qs[g][u * 64 + t8 * 8 + e];
    bool ok = true;
    for (int kt = 0; kt < ntiles; ++kt) {
        const int slot = kt % kStages;
        if (ok) ok = mbar_wait_warp(&sm.full[slot], (kt / kStages) & 1, &sm.abort);
        if (ok) {
            const int rows = min(kTileKeys, nkeys - kt * kTileKeys);
            const __nv_bfloat16 *tile = sm.tile[slot];
#pragma unroll 1
            for (int it = 0; it < kTileKeys / (4 * kConsumerWarps); ++it) {
                const int key = warp * (kTileKeys / kConsumerWarps) + it * 4 + kg;
                float kf[NQ * 8];
#pragma unroll
                for (int u = 0; u < NQ; ++u) {
                    // rows past the chunk's end read stale data of the ring slot: their
                    // scores are never stored
                    const uint4 raw = *reinterpret_cast<const uint4 *>(tile + key * D + u * 64 + t8 * 8);
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kf[u * 8 + 2 * e] = bf16lo_to_f32(w[e]);
                        kf[u * 8 + 2 * e + 1] = bf16hi_to_f32(w[e]);
                    }
                }
                float part[GT];
#pragma unroll
                for (int g = 0; g < GT; ++g) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < NQ * 8; ++e) acc = fmaf(qf[g][e], kf[e], acc);
                    part[g] = acc;
                }
                // Sum over the key's 8 lanes by reduce-scatter: at each of the top
                // LG lane bits a lane keeps half of its heads and adds the partner's
                // half, so lane t8 ends with head t8 >> (3 - LG); the remaining
                // bits are a plain butterfly.  7 shuffles for 8 heads instead of 24.
#pragma unroll
                for (int step = 0; step < LG; ++step) {
                    const int half = GT >> (step + 1);
                    const int bit = 4 >> step;
                    const bool upper = (t8 & bit) != 0;
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        const float send = upper ? part[i] : part[i + half];
                        const float keep = upper ? part[i + half] : part[i];
                        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
                    }
                }
#pragma unroll
                for (int bit = 4 >> LG; bit > 0; bit >>= 1) part[0] += __shfl_xor_sync(0xffffffffu, part[0], bit);
                const int head = t8 >> (3 - LG);
                if ((t8 & ((1 << (3 - LG)) - 1)) == 0 && key < rows)
                    sm.s[(kt * kTileKeys + key) * GT + head] = part[0];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[slot]);
        }
    }
    named_bar_sync(1, kConsumers);

    // ---------------- per-head chunk max m_c, p_j = 2^(s_j - m_c), l_c = sum p_j
    const int tid = threadIdx.x;
    float mx[GT];
#pragma unroll
    for (int g = 0; g < GT; ++g) mx[g] = -INFINITY;
    for (int j = tid; j < nkeys; j += kConsumers)
#pragma unroll
        for (int g = 0; g < GT; ++g) mx[g] = fmaxf(mx[g], sm.s[j * GT + g]);
#pragma unroll
    for (int g = 0; g < GT; ++g) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], o));
        if (lane == 0) sm.ml[warp][g] = mx[g];
    }
    named_bar_sync(1, kConsumers);
    float m_c[GT], lsum[GT];
#pragma unroll
    for (int g = 0; g < GT; ++g) {
        m_c[g] = sm.ml[0][g];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) m_c[g] = fmaxf(m_c[g], sm.ml[w][g]);
        lsum[g] = 0.f;
    }
    for (int j = tid; j < nkeys; j += kConsumers)
#pragma unroll
        for (int g = 0; g < GT; ++g) {
            const float p = ex2_approx(sm.s[j * GT + g] - m_c[g]);
            sm.s[j * GT + g] = p;
            lsum[g] += p;
        }
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], o);
    named_bar_sync(1, kConsumers);  // every p written; ml[] free again
    if (lane == 0)
#pragma unroll
        for (int g = 0; g < GT; ++g) sm.ml[warp][g] = lsum[g];

    // ---------------- PV: lane owns D/32 consecutive dims; warp w takes keys w, w+4, ...
    constexpr int DPL = D / 32;
    float acc[GT][DPL];
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[g][e] = 0.f;
    for (int vt = 0; vt < ntiles; ++vt) {
        const int tq = ntiles + vt;
        const int slot = tq % kStages;
        if (ok) ok = mbar_wait_warp(&sm.full[slot], (tq / kStages) & 1, &sm.abort);
        if (ok) {
            const int rows = min(kTileKeys, nkeys - vt * kTileKeys);
            const __nv_bfloat16 *tile = sm.tile[slot];
            const float *pp = sm.s + vt * kTileKeys * GT;
            for (int key = warp; key < rows; key += kConsumerWarps) {
                float vf[DPL];
                if constexpr (DPL == 4) {
                    const uint2 raw = *reinterpret_cast<const uint2 *>(tile + key * D + lane * 4);
                    vf[0] = bf16lo_to_f32(raw.x);
                    vf[1] = bf16hi_to_f32(raw.x);
                    vf[2] = bf16lo_to_f32(raw.y);
                    vf[3] = bf16hi_to_f32(raw.y);
                } else {
                    const uint32_t raw = *reinterpret_cast<const uint32_t *>(tile + key * D + lane * 2);
                    vf[0] = bf16lo_to_f32(raw);
                    vf[1] = bf16hi_to_f32(raw);
                }
#pragma unroll
                for (int g = 0; g < GT; ++g) {
                    const float p = pp[key * GT + g];
#pragma unroll
                    for (int e = 0; e < DPL; ++e) acc[g][e] = fmaf(p, vf[e], acc[g][e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[slot]);
        }
    }
    // Cross-warp sum of the PV partials through the (now idle) tile ring.
    named_bar_sync(1, kConsumers);
    float *red = reinterpret_cast<float *>(&sm.tile[0][0]);  // [warp][g][D]
    static_assert(kConsumerWarps * GT * D * sizeof(float) <= sizeof(sm.tile), "reduction space");
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
        for (int e = 0; e < DPL; ++e) red[(warp * GT + g) * D + lane * DPL + e] = acc[g][e];
    named_bar_sync(1, kConsumers);
    for (int e = tid; e < ng * D; e += kConsumers) {
        const int g = e / D, d = e % D;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) sum += red[(w * GT + g) * D + d];
        const size_t part = (static_cast<size_t>(b) * a.H + h_first + g) * a.n_split + c;
        a.part_o[part * D + d] = sum;
    }
#pragma unroll
    for (int g = 0; g < GT; ++g) {
        if (g == tid && g < ng) {  // thread g writes head g (no runtime index into m_c)
            float l_c = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) l_c += sm.ml[w][g];
            const size_t part = (static_cast<size_t>(b) * a.H + h_first + g) * a.n_split + c;
            a.part_ml[part * 2 + 0] = m_c[g];
            a.part_ml[part * 2 + 1] = l_c;
        }
    }
    if (tid == 0 && (!ok || sm.abort)) report_timeout(a.status, 0x32);
}

template <int D, int GT>
cudaError_t launch_gqa_t(const DecodeArgs &a) {
    const size_t smem = sizeof(GqaSmem<D, GT>);
    cudaError_t e = cudaFuncSetAttribute(decode_gqa_partial_kernel<D, GT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int G = a.H / a.H_kv;
    const int n_sub = (G + GT - 1) / GT;
    const long long blocks = static_cast<long long>(a.B) * a.H_kv * n_sub * a.n_split;
    if (a.Skv > 0) {
        e = launch_pdl(decode_gqa_partial_kernel<D, GT>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), smem,
                       a.stream, a, n_sub);
        if (e != cudaSuccess) return e;
    }
    return launch_decode_combine(a);
}

template <int D>
cudaError_t launch_gqa_d(const DecodeArgs &a) {
    const int GT = decode_gqa_heads_per_cta(a.H / a.H_kv);
    switch (GT) {
        case 2: return launch_gqa_t<D, 2>(a);
        case 4: return launch_gqa_t<D, 4>(a);
        default: return launch_gqa_t<D, 8>(a);
    }
}

}  // namespace

int decode_gqa_heads_per_cta(int G) { return G <= 2 ? 2 : (G <= 4 ? 4 : 8); }

cudaError_t launch_decode_gqa(const DecodeArgs &a) {
    return a.D == 64 ? launch_gqa_d<64>(a) : launch_gqa_d<128>(a);
}

}  // namespace attn
