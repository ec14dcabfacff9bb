// Split-KV decode attention: one query per (batch, head) against a bf16 KV cache.
//
// Decode is a matrix-vector product that reads the whole cache once and does
// about one flop per byte ("Attention from First Principles", section 6
// "Under the hood"), so this kernel is built for HBM bandwidth, not for the
// tensor cores:
//
//   partial kernel  one CTA per (b, h, chunk of `chunk` keys).  A producer
//                   warp streams the chunk's K rows and then its V rows,
//                   64 keys (16 KB at D = 128) per bulk copy, into a 4-stage
//                   shared-memory ring; four consumer warps compute the
//                   chunk's scores (log2 units), its max m_c, p_j = 2^(s_j-m_c),
//                   l_c = sum p_j and o_c = sum p_j v_j, written as fp32
//                   partials.  Keys j >= kv_len[b] are never loaded or used.
//   combine kernel  per (b, h): M = max_c m_c, out = sum_c 2^(m_c-M) o_c /
//                   sum_c 2^(m_c-M) l_c, rounded to bf16.  kv_len[b] == 0
//                   gives zeros.  (This merge is the exact softmax identity
//                   for a split key set; it is not on the pages.)
//
// The query sees every cached key below kv_len[b]: "Scaled dot-product
// attention with masking", "Adding the causal mask" (no mask for seq_q = 1).
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kTileKeys = 64;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct __align__(128) DecodeSmem {
    __nv_bfloat16 tile[kStages][kTileKeys * D];
    float s[kDecodeMaxChunk];         // scores, then probabilities, of the chunk
    float red[kConsumerWarps][D];     // per-warp partial outputs
    float wred[kConsumerWarps];
    uint64_t full[kStages], empty[kStages];
    int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads) decode_partial_kernel(DecodeArgs a) {
    griddep_launch_dependents();
    griddep_wait();  // launched back to back: the previous kernel's writes are visible
    extern __shared__ __align__(128) uint8_t smem_raw[];
    DecodeSmem<D> &sm = *reinterpret_cast<DecodeSmem<D> *>(smem_raw);

    const int bh = blockIdx.x / a.n_split;
    const int c = blockIdx.x % a.n_split;
    const int b = bh / a.H;
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
    __syncthreads();

    const size_t row0 = static_cast<size_t>(bh) * a.Skv + k0;
    const __nv_bfloat16 *Kp = static_cast<const __nv_bfloat16 *>(a.k) + row0 * D;
    const __nv_bfloat16 *Vp = static_cast<const __nv_bfloat16 *>(a.v) + row0 * D;

    if (warp == kConsumerWarps) {
        // ---------------- producer: K tiles 0..ntiles-1, then V tiles
        if (lane == 0) {
            const int total = 2 * ntiles;
            int t = 0;
            for (; t < total; ++t) {
                const int slot = t % kStages;
                if (t >= kStages &&
                    !mbar_wait(&sm.empty[slot], ((t / kStages) - 1) & 1, &sm.abort))
                    break;
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
            if (sm.abort) report_timeout(a.status, 0x21);
        }
        return;
    }

    // ---------------- consumers
    // Score phase mapping: 8 lanes per key, 4 keys per warp step; lane (g, t)
    // owns dims [8t, 8t+8) (and [64+8t, 64+8t+8) when D = 128) of key g.
    constexpr int NQ = D / 64;  // 16-byte chunks per lane per key
    const int g = lane / 8, t8 = lane % 8;
    float qf[NQ * 8];
    {
        const __nv_bfloat16 *qp = static_cast<const __nv_bfloat16 *>(a.q) + static_cast<size_t>(bh) * D;
        const float sl2 = a.scale * kLog2e;
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(qp + u * 64 + t8 * 8);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qf[u * 8 + 2 * e] = bf16lo_to_f32(w[e]) * sl2;
                qf[u * 8 + 2 * e + 1] = bf16hi_to_f32(w[e]) * sl2;
            }
        }
    }
    bool ok = true;
    for (int kt = 0; kt < ntiles; ++kt) {
        const int slot = kt % kStages;
        if (ok) ok = mbar_wait_warp(&sm.full[slot], (kt / kStages) & 1, &sm.abort);
        if (ok) {
            const int rows = min(kTileKeys, nkeys - kt * kTileKeys);
            const __nv_bfloat16 *tile = sm.tile[slot];
#pragma unroll
            for (int it = 0; it < kTileKeys / (4 * kConsumerWarps); ++it) {
                const int key = warp * (kTileKeys / kConsumerWarps) + it * 4 + g;
                float part = 0.f;
                if (key < rows) {
#pragma unroll
                    for (int u = 0; u < NQ; ++u) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(tile + key * D + u * 64 + t8 * 8);
                        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            part = fmaf(qf[u * 8 + 2 * e], bf16lo_to_f32(w[e]), part);
                            part = fmaf(qf[u * 8 + 2 * e + 1], bf16hi_to_f32(w[e]), part);
                        }
                    }
                }
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                part += __shfl_xor_sync(0xffffffffu, part, 4);
                if (t8 == 0 && key < rows) sm.s[kt * kTileKeys + key] = part;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[slot]);
        }
    }
    named_bar_sync(1, kConsumers);

    // chunk max and p_j = 2^(s_j - m_c), l_c = sum p_j
    const int tid = threadIdx.x;
    float mx = -INFINITY;
    for (int j = tid; j < nkeys; j += kConsumers) mx = fmaxf(mx, sm.s[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) sm.wred[warp] = mx;
    named_bar_sync(1, kConsumers);
    float m_c = sm.wred[0];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) m_c = fmaxf(m_c, sm.wred[w]);
    float lsum = 0.f;
    for (int j = tid; j < nkeys; j += kConsumers) {
        const float p = ex2_approx(sm.s[j] - m_c);
        sm.s[j] = p;
        lsum += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    named_bar_sync(1, kConsumers);  // every p written; wred[] free again
    if (lane == 0) sm.wred[warp] = lsum;

    // PV phase: lane owns D/32 consecutive dims; warp w takes keys w, w+4, ...
    constexpr int DPL = D / 32;
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    for (int vt = 0; vt < ntiles; ++vt) {
        const int tq = ntiles + vt;
        const int slot = tq % kStages;
        if (ok) ok = mbar_wait_warp(&sm.full[slot], (tq / kStages) & 1, &sm.abort);
        if (ok) {
            const int rows = min(kTileKeys, nkeys - vt * kTileKeys);
            const __nv_bfloat16 *tile = sm.tile[slot];
            const float *pp = sm.s + vt * kTileKeys;
            for (int key = warp; key < rows; key += kConsumerWarps) {
                const float p = pp[key];
                if constexpr (DPL == 4) {
                    const uint2 raw = *reinterpret_cast<const uint2 *>(tile + key * D + lane * 4);
                    acc[0] = fmaf(p, bf16lo_to_f32(raw.x), acc[0]);
                    acc[1] = fmaf(p, bf16hi_to_f32(raw.x), acc[1]);
                    acc[2] = fmaf(p, bf16lo_to_f32(raw.y), acc[2]);
                    acc[3] = fmaf(p, bf16hi_to_f32(raw.y), acc[3]);
                } else {
                    const uint32_t raw = *reinterpret_cast<const uint32_t *>(tile + key * D + lane * 2);
                    acc[0] = fmaf(p, bf16lo_to_f32(raw), acc[0]);
                    acc[1] = fmaf(p, bf16hi_to_f32(raw), acc[1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[slot]);
        }
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) sm.red[warp][lane * DPL + e] = acc[e];
    named_bar_sync(1, kConsumers);
    const size_t part = static_cast<size_t>(bh) * a.n_split + c;
    for (int d = tid; d < D; d += kConsumers) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) sum += sm.red[w][d];
        a.part_o[part * D + d] = sum;
    }
    if (tid == 0) {
        float l_c = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) l_c += sm.wred[w];
        a.part_ml[part * 2 + 0] = m_c;
        a.part_ml[part * 2 + 1] = l_c;
        if (!ok || sm.abort) report_timeout(a.status, 0x22);
    }
}

// One warp per (b, h) row, four rows per block: lane t owns output dims
// [t * D/32, (t + 1) * D/32).  Chunk maxima and sums are spread over the
// lanes and each chunk's weight is broadcast to the warp; the partial loads
// of 16 chunks carry no branch, so they are all in flight together.
constexpr int kCombineRows = 4;

template <int D>
__global__ void __launch_bounds__(32 * kCombineRows) decode_combine_kernel(DecodeArgs a) {
    constexpr int kV = D / 32;  // output dims per lane
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kCombineRows + (threadIdx.x >> 5);  // b * H + h
    const bool live = row < a.B * a.H;
    int L = a.Skv;
    if (live && a.kv_len) L = min(max(a.kv_len[row / a.H], 0), a.Skv);  // an input: read before the wait
    griddep_wait();  // the partial kernel's results (launched early: see launch_decode_combine)
    if (!live) return;
    const int nv = (L + a.chunk - 1) / a.chunk;  // chunks holding at least one key
    const float *ml = a.part_ml + static_cast<size_t>(row) * a.n_split * 2;
    const float *po = a.part_o + static_cast<size_t>(row) * a.n_split * D + lane * kV;
    float acc[kV], lsum = 0.f;
#pragma unroll
    for (int e = 0; e < kV; ++e) acc[e] = 0.f;
    // The partial outputs of 16 chunks, c0 .. c0 + 15: a load past the last
    // chunk re-reads that chunk (a valid address) and later gets weight 0, so
    // the loads carry no branch and are all in flight together.
    float v[16][kV];
    auto load16 = [&](int c0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float *p = po + static_cast<size_t>(min(c0 + i, nv - 1)) * D;
            if constexpr (kV == 4) {
                const float4 t = *reinterpret_cast<const float4 *>(p);
                v[i][0] = t.x;
                v[i][1] = t.y;
                v[i][2] = t.z;
                v[i][3] = t.w;
            } else {
                const float2 t = *reinterpret_cast<const float2 *>(p);
                v[i][0] = t.x;
                v[i][1] = t.y;
            }
        }
    };
    // chunk c0 + i carries the weight held by lane i
    auto mix16 = [&](float w) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float wi = __shfl_sync(0xffffffffu, w, i);
#pragma unroll
            for (int e = 0; e < kV; ++e) acc[e] = fmaf(wi, v[i][e], acc[e]);
        }
    };
    if (nv > 0 && nv <= 16) {
        // one round of loads: the chunk statistics and outputs together
        float mc = -INFINITY, lc = 0.f;
        if (lane < nv) {
            mc = ml[2 * lane];
            lc = ml[2 * lane + 1];
        }
        load16(0);
        float M = mc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w = lane < nv ? ex2_approx(mc - M) : 0.f;
        lsum = w * lc;
        mix16(w);
    } else if (nv > 16) {
        float M = -INFINITY;
        for (int c = lane; c < nv; c += 32) M = fmaxf(M, ml[2 * c]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        for (int c0 = 0; c0 < nv; c0 += 16) {
            const int c = c0 + lane;
            float w = 0.f;
            if (lane < 16 && c < nv) {
                w = ex2_approx(ml[2 * c] - M);
                lsum = fmaf(w, ml[2 * c + 1], lsum);
            }
            load16(c0);
            mix16(w);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = nv > 0 ? 1.f / lsum : 0.f;  // no key: exact zeros
    uint32_t pk[kV / 2];
#pragma unroll
    for (int e = 0; e < kV / 2; ++e) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
        pk[e] = *reinterpret_cast<uint32_t *>(&h2);
    }
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + static_cast<size_t>(row) * D + lane * kV;
    if constexpr (kV == 4)
        *reinterpret_cast<uint2 *>(out) = make_uint2(pk[0], pk[1]);
    else
        *reinterpret_cast<uint32_t *>(out) = pk[0];
}

template <int D>
cudaError_t launch_decode_t(const DecodeArgs &a) {
    const size_t smem = sizeof(DecodeSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const long long blocks = static_cast<long long>(a.B) * a.H * a.n_split;
    if (a.Skv > 0) {
        e = launch_pdl(decode_partial_kernel<D>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), smem, a.stream, a);
        if (e != cudaSuccess) return e;
    }
    return launch_decode_combine(a);
}

}  // namespace

// The combine is launched with programmatic stream serialization: once every
// CTA of the partial kernel has started (each signals at its start), the
// combine's blocks may be placed and wait in griddep_wait for the partial
// kernel to finish, which hides the launch gap between the two kernels.
cudaError_t launch_decode_combine(const DecodeArgs &a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a.B * a.H + kCombineRows - 1) / kCombineRows));
    cfg.blockDim = dim3(32 * kCombineRows);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
#ifndef ATTN_NO_PDL
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#endif
    return a.D == 64 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, a)
                     : cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, a);
}

cudaError_t launch_decode(const DecodeArgs &a) {
    return a.D == 64 ? launch_decode_t<64>(a) : launch_decode_t<128>(a);
}

}  // namespace attn
