// K6 - balance-bias updates.
//
// Quantile balancer (kimi_k3 "QuantileBalancer: persistent biases, no
// gradient update"): per expert j, rel[t] = thresh_t - s[t, j] in FP32 with
// thresh_t the (K+1)-th bias-corrected score of token t; the new bias is the
// 'higher' quantile at p = K/E of rel over the tokens, i.e. the value at
// 0-based sorted index q = ceil(p (T-1)); then the mean over experts is
// subtracted. Selection here is an exact 4-pass radix select over an
// order-preserving 32-bit key of each FP32 value, one CTA per expert, so the
// result is the q-th order statistic bit for bit. The mean is a sequential
// float64 sum over experts in index order, divided by E, rounded once to
// FP32, and subtracted in FP32 - a fixed order, hence bit-reproducible.
//
// Sign-bias balancer (APEX-1 Mathematical Reference Part 3, section 14.3):
// f_e = c_e / (N K), tau = 1/E, b_e <- clamp(b_e + alpha sign(tau - f_e), -1, 1).
//
// Routing diagnostics: the Switch load-balancing loss of "MoE from scratch"
// (MoELayer.forward: f_e = share of the T*K assignments on expert e, P_e =
// mean softmax router probability, aux = E sum_e f_e P_e before its alpha) and
// the router z-loss of the book-ai MoE chapter (MoELoss.router_z_loss: mean
// over tokens of the squared log-sum-exp of the logits, before its weight),
// from the raw FP32 logits the router wrote. Two fixed-order passes, so the
// result does not depend on scheduling: per CTA of STATS_TOKENS tokens the
// probability sums, expert counts and squared log-sum-exps; then one CTA adds
// the partials in CTA order.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// Monotone map FP32 -> uint32 (total order of the values; -0 and +0 equal).
MOE_DEV uint32_t f2key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0;  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MOE_DEV float key2f(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

__global__ void __launch_bounds__(512) quantile_select_kernel(const float* __restrict__ top_scores,
                                                              const float* __restrict__ scores,
                                                              int T, int E, int K, int q,
                                                              float* __restrict__ braw) {
    __shared__ int hist[256];
    __shared__ uint32_t s_prefix;
    __shared__ int s_rank;
    const int j = blockIdx.x;
    uint32_t prefix = 0, mask = 0;
    int rank = q;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int t = threadIdx.x; t < T; t += blockDim.x) {
            const float rel =
                __fsub_rn(top_scores[static_cast<size_t>(t) * (K + 1) + K], scores[static_cast<size_t>(t) * E + j]);
            const uint32_t key = f2key(rel);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int c[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = hist[lane * 8 + i];
                sum += c[i];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - sum;
            // the lane whose buckets hold the rank-th smallest remaining key
            const bool mine = (rank >= excl) && (rank < incl);
            if (mine) {
                int r = rank - excl, b = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (r >= 0 && r < c[i] && b == 0) b = i + 1;
                    if (b == 0) r -= c[i];
                }
                s_prefix = prefix | (static_cast<uint32_t>(lane * 8 + b - 1) << shift);
                s_rank = r;
            }
        }
        __syncthreads();
        prefix = s_prefix;
        rank = s_rank;
        mask |= 255u << shift;
        __syncthreads();
    }
    if (threadIdx.x == 0) braw[j] = key2f(prefix);
}

__global__ void quantile_center_kernel(const float* __restrict__ braw, int E, float* __restrict__ bias) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    double acc = 0.0;
    for (int j = 0; j < E; ++j) acc += static_cast<double>(braw[j]);
    const float mean = static_cast<float>(acc / static_cast<double>(E));
    for (int j = 0; j < E; ++j) bias[j] = __fsub_rn(braw[j], mean);
}

__global__ void sign_bias_kernel(int E, int N, int K, const int32_t* __restrict__ counts,
                                 float* __restrict__ bias, float alpha) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const double f = static_cast<double>(counts[e]) / (static_cast<double>(N) * K);
    const double tau = 1.0 / E;
    const float sg = (tau > f) ? 1.0f : ((tau < f) ? -1.0f : 0.0f);
    const float b = bias[e] + alpha * sg;
    bias[e] = fminf(1.0f, fmaxf(-1.0f, b));
}

// Waits on a shared-memory barrier that nothing completes, with the given
// limit; the bounded wait gives up, sets the error bit and the kernel returns.
__global__ void wait_selftest_kernel(int* err, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx wc{err, &abort_flag, timeout_ns};
        bounded_wait(smem_u32(&bar), 0, wc);
    }
    __syncthreads();
}

MOE_DEV float stats_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
MOE_DEV float stats_warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Partial sums of one CTA: 8 warps x STATS_TOKENS / 8 consecutive tokens each,
// lane l holds experts l + 32 j. part row: [P sums (E), counts (E), sum lse^2].
template <int J>
__global__ void __launch_bounds__(256) stats_partial_kernel(const float* __restrict__ logits,
                                                            const int32_t* __restrict__ idx, int T,
                                                            int E, int K, float* __restrict__ part) {
    pdl_wait();
    pdl_trigger();
    __shared__ float wsum[8][32 * J];
    __shared__ float wz[8];
    __shared__ int cnt[32 * J];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < 32 * J; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    float ps[J];
#pragma unroll
    for (int j = 0; j < J; ++j) ps[j] = 0.0f;
    float zs = 0.0f;
    constexpr int PER_WARP = STATS_TOKENS / 8;
    const int tw = blockIdx.x * STATS_TOKENS + warp * PER_WARP;
    for (int i = 0; i < PER_WARP; ++i) {
        const int t = tw + i;
        if (t >= T) break;
        float r[J], m = -INFINITY;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            r[j] = e < E ? logits[static_cast<size_t>(t) * E + e] : -INFINITY;
            m = fmaxf(m, r[j]);
        }
        m = stats_warp_max(m);
        float ex[J], sum = 0.0f;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            ex[j] = lane + 32 * j < E ? expf(r[j] - m) : 0.0f;
            sum += ex[j];
        }
        sum = stats_warp_sum(sum);
#pragma unroll
        for (int j = 0; j < J; ++j) ps[j] += ex[j] / sum;
        const float lse = m + logf(sum);
        zs += lse * lse;
        if (lane < K) {
            const int e = idx[static_cast<size_t>(t) * K + lane];
            if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) wsum[warp][lane + 32 * j] = ps[j];
    if (lane == 0) wz[warp] = zs;
    __syncthreads();
    float* row = part + static_cast<size_t>(blockIdx.x) * (2 * E + 1);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float acc = 0.0f;
        for (int w = 0; w < 8; ++w) acc += wsum[w][e];
        row[e] = acc;
        row[E + e] = static_cast<float>(cnt[e]);
    }
    if (threadIdx.x == 0) {
        float z = 0.0f;
        for (int w = 0; w < 8; ++w) z += wz[w];
        row[2 * E] = z;
    }
}

// out = [aux, z, P_0 .. P_{E-1}] from the partial rows, added in CTA order.
__global__ void __launch_bounds__(256) stats_final_kernel(const float* __restrict__ part, int nblk,
                                                          int T, int E, int K, float* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[8];
    const int e = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t stride = 2 * static_cast<size_t>(E) + 1;
    float P = 0.0f, fP = 0.0f;
    if (e < E) {
        long long c = 0;
        // CTA order, 8 partial rows' loads in flight per step
        for (int b0 = 0; b0 < nblk; b0 += 8) {
            float pv[8], cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                pv[i] = b0 + i < nblk ? part[(b0 + i) * stride + e] : 0.0f;
                cv[i] = b0 + i < nblk ? part[(b0 + i) * stride + E + e] : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (b0 + i < nblk) P += pv[i];
                c += static_cast<long long>(cv[i]);
            }
        }
        P /= static_cast<float>(T);
        const float f = static_cast<float>(static_cast<double>(c) / (static_cast<double>(T) * K));
        fP = f * P;
        out[2 + e] = P;
    }
    fP = stats_warp_sum(fP);
    if (lane == 0) red[warp] = fP;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.0f;
        for (int w = 0; w < 8; ++w) a += red[w];
        out[0] = static_cast<float>(E) * a;
        float z = 0.0f;
        for (int b0 = 0; b0 < nblk; b0 += 8) {
            float zv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) zv[i] = b0 + i < nblk ? part[(b0 + i) * stride + 2 * E] : 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (b0 + i < nblk) z += zv[i];
        }
        out[1] = z / static_cast<float>(T);
    }
}

}  // namespace

cudaError_t launch_quantile(int T, int E, int K, const float* top_scores, const float* scores,
                            float* braw, float* bias, cudaStream_t s, int* n_launched) {
    // 'higher' quantile index, computed in FP32 like an FP32 quantile
    const float p = static_cast<float>(static_cast<double>(K) / static_cast<double>(E));
    const float pos = p * static_cast<float>(T - 1);
    int q = static_cast<int>(ceilf(pos));
    if (q > T - 1) q = T - 1;
    if (q < 0) q = 0;
    quantile_select_kernel<<<E, 512, 0, s>>>(top_scores, scores, T, E, K, q, braw);
    quantile_center_kernel<<<1, 32, 0, s>>>(braw, E, bias);
    note_launch(2);
    if (n_launched) *n_launched = 2;
    return cudaGetLastError();
}

cudaError_t launch_sign_bias(int E, int N, int K, const int32_t* counts, float* bias, float alpha,
                             cudaStream_t s) {
    sign_bias_kernel<<<(E + 255) / 256, 256, 0, s>>>(E, N, K, counts, bias, alpha);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_routing_stats(const float* logits, const int32_t* idx, int T, int E, int K,
                                 float* part, float* out, cudaStream_t s) {
    const int nblk = (T + STATS_TOKENS - 1) / STATS_TOKENS;
    cudaError_t e;
    if (E <= 32)
        e = launch_pdl(stats_partial_kernel<1>, dim3(nblk), dim3(256), 0, s, logits, idx, T, E, K, part);
    else if (E <= 64)
        e = launch_pdl(stats_partial_kernel<2>, dim3(nblk), dim3(256), 0, s, logits, idx, T, E, K, part);
    else if (E <= 128)
        e = launch_pdl(stats_partial_kernel<4>, dim3(nblk), dim3(256), 0, s, logits, idx, T, E, K, part);
    else
        e = launch_pdl(stats_partial_kernel<8>, dim3(nblk), dim3(256), 0, s, logits, idx, T, E, K, part);
    if (e != cudaSuccess) return e;
    return launch_pdl(stats_final_kernel, dim3(1), dim3(256), 0, s, part, nblk, T, E, K, out);
}

cudaError_t launch_wait_selftest(int* err, uint64_t timeout_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
