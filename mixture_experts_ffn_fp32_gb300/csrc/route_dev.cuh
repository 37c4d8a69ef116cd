// Routing device code shared by the router kernels and the decode front end:
// per-token routing (the gate mode's selection score, top-K (top-(K+1) in
// sigmoid mode) with ties to the lower expert id, gate weights, margin, and
// the optional raw logits for the routing diagnostics), and the split router
// GEMM for few tokens (partial logits per slice of d, and their sum).
// Sources as in router.cu.
#pragma once

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

// Block `first` of a one-launch router zeroes the counters it was given.
MOE_DEV void zero_counters(const RouterArgs& a, bool first) {
    if (first && a.zero != nullptr)
        for (int i = threadIdx.x; i < a.nzero; i += blockDim.x) a.zero[i] = 0u;
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

// Lane l's bias values for experts l + 32 j (zero without a bias).
template <int J>
MOE_DEV void load_bias_lanes(const RouterArgs& a, float (&b)[J]) {
    const int lane = static_cast<int>(lane_id());
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        b[j] = (a.bias != nullptr && e < a.E) ? a.bias[e] : 0.0f;
    }
}

// Routes token t. Lane l holds the logits of experts l + 32 j in r[j] and
// their bias in bj[j].
template <int J>
MOE_DEV void route_token_warp(const float (&r)[J], const float (&bj)[J], int t, const RouterArgs& a) {
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
        const float b = bj[j];
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

    // Selection of the nsel largest candidates (ties: the lower expert id), one
    // per step: every lane keeps its best remaining candidate as an
    // order-preserving 32-bit key (-0 counted as +0, so equal values give equal
    // keys); the warp's largest key and, among the lanes holding it, the
    // lowest expert id come from two warp reductions; the winning lane then
    // finds its next best. The same choice as comparing (value, id) pairs.
    const int nsel = (K < E) ? K + 1 : K;
    uint32_t key[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const uint32_t u = __float_as_uint(c[j] + 0.0f);
        key[j] = (lane + 32 * j < E) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
    }
    // best remaining candidate of this lane (the lowest j among equal keys)
    auto head = [&](uint32_t& hk, uint32_t& he) {
        hk = 0u;
        he = 0xffffffffu;
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (key[j] > hk) {
                hk = key[j];
                he = static_cast<uint32_t>(lane + 32 * j);
            }
    };
    uint32_t hk, he;
    head(hk, he);
    float my_val = 0.0f;
    int my_idx = 0;
    for (int it = 0; it < nsel; ++it) {
        const uint32_t mk = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t me = __reduce_min_sync(0xffffffffu, hk == mk ? he : 0xffffffffu);
        if (lane == it) {
            my_val = __uint_as_float((mk & 0x80000000u) ? (mk & 0x7fffffffu) : ~mk);
            my_idx = static_cast<int>(me);
        }
        if (he == me) {
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (static_cast<uint32_t>(lane + 32 * j) == me) key[j] = 0u;
            head(hk, he);
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

template <int J>
MOE_DEV void route_token_warp(const float (&r)[J], int t, const RouterArgs& a) {
    float b[J];
    load_bias_lanes<J>(a, b);
    route_token_warp<J>(r, b, t, a);
}

// Routes token t in one thread from all E logits in r[0..E-1] (E <= EP <= 8):
// the same selection, ranking and weights as route_token_warp, for small E
// where one lane is cheaper than the warp-wide search.
// ids_out, w_out (optional): the K expert ids and gate weights once more,
// ids_out[k] and w_out[k].
template <int EP>
MOE_DEV void route_token_seq(const float (&r)[EP], int t, const RouterArgs& a, int* ids_out = nullptr,
                             float* w_out = nullptr) {
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
    // the experts in rank order, built once (slot k: the expert of rank k; a
    // slot no expert reaches holds zeros)
    float ov[EP + 1], osg[EP + 1];
    int oid[EP + 1];
#pragma unroll
    for (int k = 0; k <= EP; ++k) {
        ov[k] = 0.0f;
        osg[k] = 0.0f;
        oid[k] = 0;
    }
#pragma unroll
    for (int k = 0; k < EP; ++k) {
        float v = 0.0f, g = 0.0f;
        int id = 0;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            const bool m = rank[e] == k;
            v = m ? c[e] : v;
            g = m ? sg[e] : g;
            id = m ? e : id;
        }
        ov[k] = v;
        osg[k] = g;
        oid[k] = id;
    }
    const float v0 = ov[0];
    float ex[EP];
    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < EP; ++k) {
        ex[k] = 0.0f;
        if (k < K) {
            ex[k] = a.gate == MOE_GATE_SOFTMAX_TOPK ? expf(ov[k] - v0)
                    : a.gate == MOE_GATE_SOFTMAX_ALL_RENORM ? ov[k] : osg[k];
            sum += ex[k];
        }
    }
    const bool normalise = a.gate != MOE_GATE_SIGMOID || a.renorm;
#pragma unroll
    for (int k = 0; k < EP + 1; ++k) {
        if (k <= K && k < E) {
            if (k < K) {
                float wk = ex[k < EP ? k : 0];
                if (normalise) wk = wk / sum;
                if (a.gate == MOE_GATE_SIGMOID) wk *= a.scale;
                a.idx[static_cast<size_t>(t) * K + k] = oid[k];
                a.w[static_cast<size_t>(t) * K + k] = wk;
                if (ids_out != nullptr) ids_out[k] = oid[k];
                if (w_out != nullptr) w_out[k] = wk;
            }
            if (a.top_scores != nullptr && a.gate == MOE_GATE_SIGMOID)
                a.top_scores[static_cast<size_t>(t) * (K + 1) + k] = ov[k];
        }
    }
    if (a.margin != nullptr) {
        // the values of rank K - 1 and K (zero where no expert has rank K)
        float vK1 = 0.0f, vK = 0.0f;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            vK1 = rank[e] == K - 1 ? c[e] : vK1;
            vK = rank[e] == K ? c[e] : vK;
        }
        a.margin[t] = (K < E) ? (vK1 - vK) : INFINITY;
    }
}


// Logits of token t from split partial sums: r[j] (expert lane + 32 j) is the
// sum of part[s, t, e] over the nsplit slices in slice order, all J x 8 loads
// of a step in flight before their sums. Read through L2, so that partials
// written by other CTAs of the same grid are seen after their ticket.
template <int J>
MOE_DEV void sum_slices(const float* __restrict__ part, int nsplit, int t, int T, int E,
                        float (&r)[J]) {
    const int lane = static_cast<int>(lane_id());
    const size_t slice = static_cast<size_t>(T) * E;
#pragma unroll
    for (int j = 0; j < J; ++j) r[j] = 0.0f;
    for (int s0 = 0; s0 < nsplit; s0 += 8) {
        float q[J][8];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            const float* p = part + static_cast<size_t>(t) * E + e;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                q[j][i] = (e < E && s0 + i < nsplit) ? __ldcg(p + (s0 + i) * slice) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < J; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (s0 + i < nsplit) r[j] += q[j][i];
    }
}

// Partial logits of 8 tokens over one slice of d, for few tokens and E > 32:
// one CTA of 256 threads per (token block bx, slice by). The threads are
// (expert e, part r): R = 256 / EP parts each take a contiguous run of 64 of
// the slice's router_chunk_len(EP) = 64 R values, reading W_router rows
// coalesced across e; the 8 tokens' x slices sit in shared memory, and part 0
// adds the R partial sums in order into part[by, t, e].
__host__ __device__ constexpr int router_chunk_len(int EP) { return 64 * (256 / EP); }

template <bool BF16, int EP>
MOE_DEV void chunk_partials(const RouterArgs& a, float* __restrict__ part, int bx, int by) {
    constexpr int R = 256 / EP;            // parts per expert
    constexpr int LEN = router_chunk_len(EP);
    constexpr int RUN = LEN / R;           // k values per part (64)
    __shared__ float xs[8][LEN];
    __shared__ float red[R > 1 ? R - 1 : 1][8][EP];
    const int t0 = bx * 8, k0 = by * LEN;
    const int kn = min(LEN, a.d - k0);
    const int e = threadIdx.x % EP, r = threadIdx.x / EP;
    const int kb = r * RUN;
    // Every load of the thread is issued before the first use: the thread's
    // run of W rows and its share of the 8 x slices. A decode batch is bound
    // by these loads' latency, so one round trip.
    float wv[RUN];
    {
        const float* w = a.W + static_cast<size_t>(k0 + kb) * a.E + e;
#pragma unroll
        for (int i = 0; i < RUN; ++i)
            wv[i] = (e < a.E && kb + i < kn) ? __ldg(w + static_cast<size_t>(i) * a.E) : 0.0f;
    }
    constexpr int XPER = 8 * LEN / 256;
    float xv[XPER];
#pragma unroll
    for (int q = 0; q < XPER; ++q) {
        const int i = threadIdx.x + 256 * q;
        const int tt = i / LEN, k = i - tt * LEN;
        xv[q] = 0.0f;
        if (t0 + tt < a.T && k < kn) {
            const size_t off = static_cast<size_t>(t0 + tt) * a.d + k0 + k;
            xv[q] = BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.x)[off])
                         : static_cast<const float*>(a.x)[off];
        }
    }
#pragma unroll
    for (int q = 0; q < XPER; ++q) {
        const int i = threadIdx.x + 256 * q;
        xs[i / LEN][i % LEN] = xv[q];
    }
    __syncthreads();
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    // zero-filled past the slice end, so the full run adds exact zeros
#pragma unroll
    for (int i = 0; i < RUN; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(xs[j][kb + i], wv[i], acc[j]);
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
    if (r == 0 && e < a.E) {
        float* dst = part + (static_cast<size_t>(by) * a.T + t0) * a.E + e;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (t0 + j < a.T) dst[static_cast<size_t>(j) * a.E] = acc[j];
    }
}

}  // namespace
}  // namespace moe
