// K1 - router: FP32 logits r = x W_router, the gate mode's selection score,
// top-K (top-(K+1) in sigmoid mode) and gate weights, fused in one kernel.
//
// Sources: APEX-1 docs "10 - Mixture of Experts" (MoEFFN.forward steps 2-3:
// router Linear without bias, expert bias added, top-K, softmax over the
// selected scores); APEX-1 Mathematical Reference Part 3 sections 13.2 and
// 13.5; "MoE from scratch" MoELayer.forward (softmax over all experts in
// FP32, top-K of the probabilities, renormalised); kimi_k3 StableLatentMoE
// "FP32 router and training-only QB update" (sigmoid scores, top-(K+1) of
// the bias-corrected scores, weights from the uncorrected scores).
//
// Ranking: score descending, equal scores -> lower expert id first. A NaN
// score ranks as -inf so the selected ids are always valid.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {


// The error word and the dispatch ticket that follows it start every forward at zero.
MOE_DEV void clear_status(int* w) {
    w[0] = 0;
    w[1] = 0;
}

MOE_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
MOE_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Routes token t. Lane l holds the logits of experts l + 32 j in r[j].
template <int J>
MOE_DEV void route_token_warp(const float (&r)[J], int t, const RouterArgs& a) {
    const int lane = static_cast<int>(lane_id());
    const int E = a.E, K = a.K;
    if (a.logits != nullptr) {
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (lane + 32 * j < E) a.logits[static_cast<size_t>(t) * E + lane + 32 * j] = r[j];
    }
    float c[J], s[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        const float b = (a.bias != nullptr && e < E) ? a.bias[e] : 0.0f;
        s[j] = 0.0f;
        if (a.gate == MOE_GATE_SIGMOID) {
            s[j] = 1.0f / (1.0f + expf(-r[j]));
            c[j] = s[j] + b;
        } else {
            c[j] = r[j] + b;
        }
    }
    if (a.gate == MOE_GATE_SOFTMAX_ALL_RENORM) {
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (lane + 32 * j < E) m = fmaxf(m, c[j]);
        m = warp_max(m);
        float z[J], sum = 0.0f;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            z[j] = (lane + 32 * j < E) ? expf(c[j] - m) : 0.0f;
            sum += z[j];
        }
        sum = warp_sum(sum);
#pragma unroll
        for (int j = 0; j < J; ++j) c[j] = z[j] / sum;
    }
    if (a.gate == MOE_GATE_SIGMOID && a.scores != nullptr) {
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            if (e < E) a.scores[static_cast<size_t>(t) * E + e] = s[j];
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j)
        if (!(c[j] == c[j])) c[j] = -INFINITY;

    const int nsel = (K < E) ? K + 1 : K;
    uint32_t taken = 0;
    float my_val = 0.0f;
    int my_idx = 0;
    for (int it = 0; it < nsel; ++it) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u)) {
                if (c[j] > bv || (c[j] == bv && e < bi)) {
                    bv = c[j];
                    bi = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == (bi & 31)) taken |= 1u << (bi >> 5);
        if (lane == it) {
            my_val = bv;
            my_idx = bi;
        }
    }

    float w = 0.0f;
    if (a.gate == MOE_GATE_SOFTMAX_TOPK) {
        const float m = __shfl_sync(0xffffffffu, my_val, 0);
        const float ex = (lane < K) ? expf(my_val - m) : 0.0f;
        const float sum = warp_sum(ex);
        w = ex / sum;
    } else if (a.gate == MOE_GATE_SOFTMAX_ALL_RENORM) {
        const float p = (lane < K) ? my_val : 0.0f;
        const float sum = warp_sum(p);
        w = p / sum;
    } else {
        float my_s = 0.0f;
        for (int k = 0; k < K; ++k) {
            const int e = __shfl_sync(0xffffffffu, my_idx, k);
            const int jj = e >> 5;
            float sv = 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (j == jj) sv = s[j];
            sv = __shfl_sync(0xffffffffu, sv, e & 31);
            if (lane == k) my_s = sv;
        }
        w = my_s;
        if (a.renorm) {
            const float sum = warp_sum(lane < K ? my_s : 0.0f);
            w = my_s / sum;
        }
        w *= a.scale;
    }

    const float vK1 = __shfl_sync(0xffffffffu, my_val, K - 1);
    const float vK = __shfl_sync(0xffffffffu, my_val, (K < E) ? K : K - 1);
    if (lane < K) {
        a.idx[static_cast<size_t>(t) * K + lane] = my_idx;
        a.w[static_cast<size_t>(t) * K + lane] = w;
    }
    if (a.top_scores != nullptr && a.gate == MOE_GATE_SIGMOID && lane <= K)
        a.top_scores[static_cast<size_t>(t) * (K + 1) + lane] = my_val;
    if (a.margin != nullptr && lane == 0) a.margin[t] = (K < E) ? (vK1 - vK) : INFINITY;
}

// Routes token t in one thread from all E logits in r[0..E-1] (E <= EP <= 8):
// the same selection, ranking and weights as route_token_warp, for small E
// where one lane is cheaper than the warp-wide search.
template <int EP>
MOE_DEV void route_token_seq(const float (&r)[EP], int t, const RouterArgs& a) {
    const int E = a.E, K = a.K;
    if (a.logits != nullptr) {
#pragma unroll
        for (int e = 0; e < EP; ++e)
            if (e < E) a.logits[static_cast<size_t>(t) * E + e] = r[e];
    }
    float c[EP], sg[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) {
        sg[e] = 0.0f;
        c[e] = -INFINITY;
        if (e < E) {
            const float b = a.bias != nullptr ? a.bias[e] : 0.0f;
            if (a.gate == MOE_GATE_SIGMOID) {
                sg[e] = 1.0f / (1.0f + expf(-r[e]));
                c[e] = sg[e] + b;
            } else {
                c[e] = r[e] + b;
            }
        }
    }
    if (a.gate == MOE_GATE_SOFTMAX_ALL_RENORM) {
        float m = -INFINITY;
#pragma unroll
        for (int e = 0; e < EP; ++e)
            if (e < E) m = fmaxf(m, c[e]);
        float sum = 0.0f;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            c[e] = e < E ? expf(c[e] - m) : 0.0f;
            sum += c[e];
        }
#pragma unroll
        for (int e = 0; e < EP; ++e)
            if (e < E) c[e] = c[e] / sum;
    }
    if (a.gate == MOE_GATE_SIGMOID && a.scores != nullptr) {
#pragma unroll
        for (int e = 0; e < EP; ++e)
            if (e < E) a.scores[static_cast<size_t>(t) * E + e] = sg[e];
    }
#pragma unroll
    for (int e = 0; e < EP; ++e)
        if (!(c[e] == c[e])) c[e] = -INFINITY;
    // rank of each expert: how many beat it (higher value, or equal value and
    // lower id); slot k of the top-(K+1) holds the expert of rank k
    int rank[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) {
        rank[e] = EP;
        if (e < E) {
            int n = 0;
#pragma unroll
            for (int f = 0; f < EP; ++f)
                if (f < E && (c[f] > c[e] || (c[f] == c[e] && f < e))) ++n;
            rank[e] = n;
        }
    }
    auto slot = [&](int k, float& v, int& id, float& sgv) {
        v = 0.0f;
        id = 0;
        sgv = 0.0f;
#pragma unroll
        for (int e = 0; e < EP; ++e)
            if (rank[e] == k) {
                v = c[e];
                id = e;
                sgv = sg[e];
            }
    };
    float v0, sg0;
    int id0;
    slot(0, v0, id0, sg0);
    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < EP; ++k) {
        if (k < K) {
            float v, sgv;
            int id;
            slot(k, v, id, sgv);
            sum += a.gate == MOE_GATE_SOFTMAX_TOPK ? expf(v - v0)
                   : a.gate == MOE_GATE_SOFTMAX_ALL_RENORM ? v : sgv;
        }
    }
    const bool normalise = a.gate != MOE_GATE_SIGMOID || a.renorm;
#pragma unroll
    for (int k = 0; k < EP + 1; ++k) {
        if (k <= K && k < E) {
            float v, sgv;
            int id;
            slot(k, v, id, sgv);
            if (k < K) {
                float wk = a.gate == MOE_GATE_SOFTMAX_TOPK ? expf(v - v0)
                           : a.gate == MOE_GATE_SOFTMAX_ALL_RENORM ? v : sgv;
                if (normalise) wk = wk / sum;
                if (a.gate == MOE_GATE_SIGMOID) wk *= a.scale;
                a.idx[static_cast<size_t>(t) * K + k] = id;
                a.w[static_cast<size_t>(t) * K + k] = wk;
            }
            if (a.top_scores != nullptr && a.gate == MOE_GATE_SIGMOID)
                a.top_scores[static_cast<size_t>(t) * (K + 1) + k] = v;
        }
    }
    if (a.margin != nullptr) {
        float vK1, vK, sgv;
        int id;
        slot(K - 1, vK1, id, sgv);
        slot(K, vK, id, sgv);
        a.margin[t] = (K < E) ? (vK1 - vK) : INFINITY;
    }
}

// E <= 32: one warp per token, 8 tokens per CTA. The CTA first copies its 8
// x rows into shared memory with all its loads in flight at once (one memory
// round trip), then lane l of a warp takes the d-index pairs k0 + 2l, k0 + 2l + 1,
// so the W_router row loads of a warp are contiguous; a butterfly then leaves
// every expert's full sum on every lane.
template <int EP, bool BF16>
__global__ void __launch_bounds__(256) router_small_kernel(RouterArgs a) {
    extern __shared__ __align__(16) uint8_t xsm[];
    pdl_wait();
    pdl_trigger();
    if (a.err_clear != nullptr && blockIdx.x == 0 && threadIdx.x == 0) clear_status(a.err_clear);
    const int E = a.E, d = a.d;
    const int t0 = blockIdx.x * 8;
    const int ntok = min(8, a.T - t0);
    {
        const size_t row_bytes = static_cast<size_t>(d) * (BF16 ? 2 : 4);
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.x) + t0 * row_bytes);
        uint4* dst = reinterpret_cast<uint4*>(xsm);
        const int nvec = static_cast<int>(ntok * row_bytes / 16);
        for (int i = threadIdx.x; i < nvec; i += blockDim.x) dst[i] = __ldg(src + i);
    }
    __syncthreads();
    const int wt = threadIdx.x >> 5;
    if (wt >= ntok) return;
    const int t = t0 + wt;
    const int lane = static_cast<int>(lane_id());
    const bool vec = (E == EP) && (EP % 4 == 0);
    constexpr int U = EP <= 8 ? 4 : (EP <= 16 ? 2 : 1);
    float acc[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[e] = 0.0f;
    for (int k0 = 2 * lane; k0 < d; k0 += 64 * U) {
        float x0[U], x1[U];
        float w0[U][EP], w1[U][EP];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int k = k0 + 64 * u;
            x0[u] = x1[u] = 0.0f;
#pragma unroll
            for (int e = 0; e < EP; ++e) w0[u][e] = w1[u][e] = 0.0f;
            if (k < d) {
                if (BF16) {
                    const uint32_t v = reinterpret_cast<const uint32_t*>(xsm)[(wt * d + k) >> 1];
                    x0[u] = bf16_lo(v);
                    x1[u] = bf16_hi(v);
                } else {
                    const float2 v = reinterpret_cast<const float2*>(xsm)[(wt * d + k) >> 1];
                    x0[u] = v.x;
                    x1[u] = v.y;
                }
                const float* r0 = a.W + static_cast<size_t>(k) * E;
                const float* r1 = r0 + E;
                if (vec) {
#pragma unroll
                    for (int e = 0; e < EP; e += 4) {
                        const float4 p = __ldg(reinterpret_cast<const float4*>(r0 + e));
                        const float4 q = __ldg(reinterpret_cast<const float4*>(r1 + e));
                        w0[u][e] = p.x; w0[u][e + 1] = p.y; w0[u][e + 2] = p.z; w0[u][e + 3] = p.w;
                        w1[u][e] = q.x; w1[u][e + 1] = q.y; w1[u][e + 2] = q.z; w1[u][e + 3] = q.w;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < EP; ++e)
                        if (e < E) {
                            w0[u][e] = __ldg(r0 + e);
                            w1[u][e] = __ldg(r1 + e);
                        }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int e = 0; e < EP; ++e) acc[e] = fmaf(x1[u], w1[u][e], fmaf(x0[u], w0[u][e], acc[e]));
    }
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[e] = warp_sum(acc[e]);  // every lane: all E sums
    if (EP <= 8) {
        if (lane == 0) route_token_seq<(EP <= 8 ? EP : 8)>(
            reinterpret_cast<const float(&)[(EP <= 8 ? EP : 8)]>(acc), t, a);
        return;
    }
    float r[1] = {0.0f};
#pragma unroll
    for (int e = 0; e < EP; ++e)
        if (e == lane) r[0] = acc[e];
    route_token_warp<1>(r, t, a);
}

// E > 32: a CTA computes a [32 tokens x E] logit tile with FP32 FMAs through
// shared memory, then each warp routes 4 tokens.
constexpr int RT_BT = 32;
constexpr int RT_DK = 32;

template <int J, bool BF16>
__global__ void __launch_bounds__(256) router_tiled_kernel(RouterArgs a) {
    pdl_wait();
    pdl_trigger();
    constexpr int EPAD = 32 * J;        // 64, 128 or 256
    constexpr int EI = EPAD / 64;       // experts per thread
    __shared__ float xs[RT_BT * RT_DK];
    __shared__ float wl[RT_DK * EPAD];  // W chunk, then the logit tile
    static_assert(RT_BT * EPAD <= RT_DK * EPAD, "logit tile must fit the W chunk buffer");

    const int tid = threadIdx.x;
    if (a.err_clear != nullptr && blockIdx.x == 0 && tid == 0) clear_status(a.err_clear);
    const int tg = tid >> 6;   // token group: tokens tg*8 .. tg*8+7
    const int el = tid & 63;   // experts el + 64 i
    const int t0 = blockIdx.x * RT_BT;
    const int E = a.E, d = a.d;

    float acc[8][EI];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < EI; ++j) acc[i][j] = 0.0f;

    for (int k0 = 0; k0 < d; k0 += RT_DK) {
        // x chunk: 32 tokens x 32 columns, 4 consecutive columns per thread
        {
            const int tt = tid >> 3, kk = (tid & 7) * 4;
            const int t = t0 + tt;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (t < a.T) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int k = k0 + kk + i;
                    if (k < d) {
                        if (BF16)
                            v[i] = __bfloat162float(static_cast<const __nv_bfloat16*>(
                                a.x)[static_cast<size_t>(t) * d + k]);
                        else
                            v[i] = static_cast<const float*>(a.x)[static_cast<size_t>(t) * d + k];
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) xs[tt * RT_DK + kk + i] = v[i];
        }
        for (int i = tid; i < RT_DK * EPAD; i += 256) {
            const int kk = i / EPAD, e = i % EPAD;
            const int k = k0 + kk;
            wl[i] = (k < d && e < E) ? __ldg(a.W + static_cast<size_t>(k) * E + e) : 0.0f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < RT_DK; ++kk) {
            float wv[EI];
#pragma unroll
            for (int j = 0; j < EI; ++j) wv[j] = wl[kk * EPAD + el + 64 * j];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float xv = xs[(tg * 8 + i) * RT_DK + kk];
#pragma unroll
                for (int j = 0; j < EI; ++j) acc[i][j] = fmaf(xv, wv[j], acc[i][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < EI; ++j) wl[(tg * 8 + i) * EPAD + el + 64 * j] = acc[i][j];
    __syncthreads();

    const int warp = tid >> 5, lane = tid & 31;
    for (int i = 0; i < RT_BT / 8; ++i) {
        const int tt = warp * (RT_BT / 8) + i;
        const int t = t0 + tt;
        if (t >= a.T) break;
        float r[J];
#pragma unroll
        for (int j = 0; j < J; ++j) r[j] = wl[tt * EPAD + lane + 32 * j];
        route_token_warp<J>(r, t, a);
    }
}

// Exact three-term BF16 split of the FP32 router weights for the tensor-core
// router: W = hi + mid + lo with hi = bf16(W), mid = bf16(W - hi),
// lo = bf16(W - hi - mid). Both subtractions are exact in FP32 and the last
// remainder has at most 8 significant bits, so hi + mid + lo == W exactly.
// x is BF16, so every product x * part is exact in FP32. The tensor core's
// FP32 accumulation loses precision over long chains, so the reduction is cut
// into chunks of ROUTER_CHUNK rows of W: rows are stored chunk by chunk, and
// within a chunk as lo, mid, hi (small parts first). The GEMM accumulates one
// chunk per split-K slice and the slices are summed in FP32 afterwards.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ W, int d, int E,
                                                           __nv_bfloat16* __restrict__ W3,
                                                           int* err_clear) {
    pdl_wait();
    pdl_trigger();
    if (err_clear != nullptr && blockIdx.x == 0 && threadIdx.x == 0) clear_status(err_clear);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= d * E) return;
    const int k = i / E, e = i - k * E;
    const int c = k / ROUTER_CHUNK, j = k - c * ROUTER_CHUNK;
    const float w = W[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = __fsub_rn(w, __bfloat162float(hi));
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    const size_t base = (static_cast<size_t>(c) * 3 * ROUTER_CHUNK + j) * E + e;
    const size_t part = static_cast<size_t>(ROUTER_CHUNK) * E;
    W3[base] = __float2bfloat16_rn(r2);
    W3[base + part] = mid;
    W3[base + 2 * part] = hi;
}

// Routing from precomputed logits: r[t, e] = sum over the split-K slices of
// part[s, t, e], summed in slice order; one warp per token.
template <int J>
__global__ void __launch_bounds__(256) route_from_logits_kernel(const float* __restrict__ part,
                                                                int nsplit, RouterArgs a) {
    pdl_wait();
    pdl_trigger();
    if (a.err_clear != nullptr && blockIdx.x == 0 && threadIdx.x == 0) clear_status(a.err_clear);
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= a.T) return;
    const int lane = static_cast<int>(lane_id());
    const size_t slice = static_cast<size_t>(a.T) * a.E;
    float r[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        float v = 0.0f;
        if (e < a.E) {
            // slices in order, 8 loads in flight per step
            const float* p = part + static_cast<size_t>(t) * a.E + e;
            for (int s0 = 0; s0 < nsplit; s0 += 8) {
                float q[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) q[i] = s0 + i < nsplit ? p[(s0 + i) * slice] : 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (s0 + i < nsplit) v += q[i];
            }
        }
        r[j] = v;
    }
    route_token_warp<J>(r, t, a);
}

// Few tokens, E > 32: partial logits over slices of d, one CTA per (8 tokens,
// slice) so that even a decode batch spreads over many SMs. The CTA's threads
// are (expert e, part r): R = 256 / EP parts each take a contiguous run of 64
// of the slice's CHUNK_LEN(EP) = 64 R values (W_router rows read coalesced
// across e, 8 rows in flight), the 8 tokens' x slices sit in shared memory,
// and part 0 adds the R partial sums in order. route_from_logits_kernel sums
// the slices in FP32 and routes.
__host__ __device__ constexpr int router_chunk_len(int EP) { return 64 * (256 / EP); }

template <bool BF16, int EP>
__global__ void __launch_bounds__(256) router_chunk_kernel(RouterArgs a, float* __restrict__ part) {
    constexpr int R = 256 / EP;            // parts per expert
    constexpr int LEN = router_chunk_len(EP);
    constexpr int RUN = LEN / R;           // k values per part (64)
    pdl_wait();
    pdl_trigger();
    if (a.err_clear != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        clear_status(a.err_clear);
    __shared__ float xs[8][LEN];
    __shared__ float red[R > 1 ? R - 1 : 1][8][EP];
    const int t0 = blockIdx.x * 8, k0 = blockIdx.y * LEN;
    const int kn = min(LEN, a.d - k0);
    for (int i = threadIdx.x; i < 8 * LEN; i += blockDim.x) {
        const int tt = i / LEN, k = i - tt * LEN;
        float v = 0.0f;
        if (t0 + tt < a.T && k < kn) {
            const size_t off = static_cast<size_t>(t0 + tt) * a.d + k0 + k;
            v = BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.x)[off])
                     : static_cast<const float*>(a.x)[off];
        }
        xs[tt][k] = v;
    }
    __syncthreads();
    const int e = threadIdx.x % EP, r = threadIdx.x / EP;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    if (e < a.E) {
        const int kb = r * RUN;
        const int ke = min(kb + RUN, kn);
        const float* w = a.W + static_cast<size_t>(k0) * a.E + e;
        int k = kb;
        for (; k + 8 <= ke; k += 8) {
            float wv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) wv[i] = __ldg(w + static_cast<size_t>(k + i) * a.E);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(xs[j][k + i], wv[i], acc[j]);
        }
        for (; k < ke; ++k) {
            const float wv = __ldg(w + static_cast<size_t>(k) * a.E);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = fmaf(xs[j][k], wv, acc[j]);
        }
    }
    if (R > 1) {
        if (r > 0)
#pragma unroll
            for (int j = 0; j < 8; ++j) red[r - 1][j][e] = acc[j];
        __syncthreads();
        if (r == 0)
            for (int q = 0; q < R - 1; ++q)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] += red[q][j][e];
    }
    if (r != 0 || e >= a.E) return;
    float* dst = part + (static_cast<size_t>(blockIdx.y) * a.T + t0) * a.E + e;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (t0 + j < a.T) dst[static_cast<size_t>(j) * a.E] = acc[j];
}

template <bool BF16>
cudaError_t launch_router_t(const RouterArgs& a, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (a.E <= 32) {
        const int blocks = (a.T + 7) / 8;
        const size_t smem = static_cast<size_t>(8) * a.d * (BF16 ? 2 : 4);
        if (smem > 48 * 1024) {
            static bool set = false;
            if (!set) {
                cudaFuncSetAttribute(router_small_kernel<4, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
                cudaFuncSetAttribute(router_small_kernel<8, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
                cudaFuncSetAttribute(router_small_kernel<16, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
                cudaFuncSetAttribute(router_small_kernel<32, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
                set = true;
            }
        }
        if (a.E <= 4)
            e = launch_pdl(router_small_kernel<4, BF16>, dim3(blocks), dim3(256), smem, s, a);
        else if (a.E <= 8)
            e = launch_pdl(router_small_kernel<8, BF16>, dim3(blocks), dim3(256), smem, s, a);
        else if (a.E <= 16)
            e = launch_pdl(router_small_kernel<16, BF16>, dim3(blocks), dim3(256), smem, s, a);
        else
            e = launch_pdl(router_small_kernel<32, BF16>, dim3(blocks), dim3(256), smem, s, a);
    } else {
        const int blocks = (a.T + RT_BT - 1) / RT_BT;
        if (a.E <= 64)
            e = launch_pdl(router_tiled_kernel<2, BF16>, dim3(blocks), dim3(256), 0, s, a);
        else if (a.E <= 128)
            e = launch_pdl(router_tiled_kernel<4, BF16>, dim3(blocks), dim3(256), 0, s, a);
        else
            e = launch_pdl(router_tiled_kernel<8, BF16>, dim3(blocks), dim3(256), 0, s, a);
    }
    return e;
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
    return a.x_bf16 ? launch_router_t<true>(a, s) : launch_router_t<false>(a, s);
}

cudaError_t launch_router_split(const float* W, int d, int E, void* W3, int* err_clear,
                                cudaStream_t s) {
    const int n = d * E;
    return launch_pdl(router_split_kernel, dim3((n + 255) / 256), dim3(256), 0, s, W, d, E,
                      static_cast<__nv_bfloat16*>(W3), err_clear);
}

int router_chunked_nsplit(int d, int E) {
    const int len = router_chunk_len(E <= 64 ? 64 : (E <= 128 ? 128 : 256));
    return (d + len - 1) / len;
}

cudaError_t launch_router_chunked(const RouterArgs& a, float* part, cudaStream_t s) {
    const int nsplit = router_chunked_nsplit(a.d, a.E);
    const dim3 grid((a.T + 7) / 8, nsplit);
    cudaError_t e;
#define MOE_RC(EPV)                                                                                \
    e = a.x_bf16 ? launch_pdl(router_chunk_kernel<true, EPV>, grid, dim3(256), 0, s, a, part)      \
                 : launch_pdl(router_chunk_kernel<false, EPV>, grid, dim3(256), 0, s, a, part)
    if (a.E <= 64)
        MOE_RC(64);
    else if (a.E <= 128)
        MOE_RC(128);
    else
        MOE_RC(256);
#undef MOE_RC
    if (e != cudaSuccess) return e;
    RouterArgs b = a;
    b.err_clear = nullptr;  // cleared by the partial kernel; later bits must survive
    return launch_route_from_logits(part, nsplit, b, s);
}

cudaError_t launch_route_from_logits(const float* part, int nsplit, const RouterArgs& a,
                                     cudaStream_t s) {
    const int blocks = (a.T * 32 + 255) / 256;
    cudaError_t e;
    if (a.E <= 32)
        e = launch_pdl(route_from_logits_kernel<1>, dim3(blocks), dim3(256), 0, s, part, nsplit, a);
    else if (a.E <= 64)
        e = launch_pdl(route_from_logits_kernel<2>, dim3(blocks), dim3(256), 0, s, part, nsplit, a);
    else if (a.E <= 128)
        e = launch_pdl(route_from_logits_kernel<4>, dim3(blocks), dim3(256), 0, s, part, nsplit, a);
    else
        e = launch_pdl(route_from_logits_kernel<8>, dim3(blocks), dim3(256), 0, s, part, nsplit, a);
    return e;
}

}  // namespace moe
