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

cudaError_t launch_wait_selftest(int* err, uint64_t timeout_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
