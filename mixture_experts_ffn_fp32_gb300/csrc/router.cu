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

// E <= 32: one warp per token; lanes split d, then a butterfly leaves every
// expert's full sum on every lane.
template <int EP, bool BF16>
__global__ void __launch_bounds__(256) router_small_kernel(RouterArgs a) {
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= a.T) return;
    const int lane = static_cast<int>(lane_id());
    const int E = a.E, d = a.d;
    float acc[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[e] = 0.0f;
    // chunks of 8 consecutive x elements
    for (int k0 = lane * 8; k0 < d; k0 += 32 * 8) {
        float xv[8];
        if (BF16) {
            const uint4 v = *reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(a.x) + static_cast<size_t>(t) * d + k0);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xv[2 * i] = bf16_lo(u[i]);
                xv[2 * i + 1] = bf16_hi(u[i]);
            }
        } else {
            const float* xp = static_cast<const float*>(a.x) + static_cast<size_t>(t) * d + k0;
            const float4 p0 = *reinterpret_cast<const float4*>(xp);
            const float4 p1 = *reinterpret_cast<const float4*>(xp + 4);
            xv[0] = p0.x; xv[1] = p0.y; xv[2] = p0.z; xv[3] = p0.w;
            xv[4] = p1.x; xv[5] = p1.y; xv[6] = p1.z; xv[7] = p1.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float* wr = a.W + static_cast<size_t>(k0 + i) * E;
#pragma unroll
            for (int e = 0; e < EP; ++e)
                if (e < E) acc[e] = fmaf(xv[i], __ldg(wr + e), acc[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[e] = warp_sum(acc[e]);
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
    constexpr int EPAD = 32 * J;        // 64, 128 or 256
    constexpr int EI = EPAD / 64;       // experts per thread
    __shared__ float xs[RT_BT * RT_DK];
    __shared__ float wl[RT_DK * EPAD];  // W chunk, then the logit tile
    static_assert(RT_BT * EPAD <= RT_DK * EPAD, "logit tile must fit the W chunk buffer");

    const int tid = threadIdx.x;
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

template <bool BF16>
cudaError_t launch_router_t(const RouterArgs& a, cudaStream_t s) {
    if (a.E <= 32) {
        const int blocks = (a.T * 32 + 255) / 256;
        if (a.E <= 4)
            router_small_kernel<4, BF16><<<blocks, 256, 0, s>>>(a);
        else if (a.E <= 8)
            router_small_kernel<8, BF16><<<blocks, 256, 0, s>>>(a);
        else if (a.E <= 16)
            router_small_kernel<16, BF16><<<blocks, 256, 0, s>>>(a);
        else
            router_small_kernel<32, BF16><<<blocks, 256, 0, s>>>(a);
    } else {
        const int blocks = (a.T + RT_BT - 1) / RT_BT;
        if (a.E <= 64)
            router_tiled_kernel<2, BF16><<<blocks, 256, 0, s>>>(a);
        else if (a.E <= 128)
            router_tiled_kernel<4, BF16><<<blocks, 256, 0, s>>>(a);
        else
            router_tiled_kernel<8, BF16><<<blocks, 256, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
    note_launch();
    return a.x_bf16 ? launch_router_t<true>(a, s) : launch_router_t<false>(a, s);
}

}  // namespace moe
