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

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "route_dev.cuh"

namespace moe {
namespace {


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
    zero_counters(a, blockIdx.x == 0);
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
    float r[J];
    sum_slices<J>(part, nsplit, t, a.T, a.E, r);
    route_token_warp<J>(r, t, a);
}

// Few tokens, E > 32: partial logits over slices of d (chunk_partials), one
// CTA per (8 tokens, slice); route_from_logits_kernel sums the slices.
template <bool BF16, int EP>
__global__ void __launch_bounds__(256) router_chunk_kernel(RouterArgs a, float* __restrict__ part) {
    pdl_wait();
    pdl_trigger();
    if (a.err_clear != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        clear_status(a.err_clear);
    chunk_partials<BF16, EP>(a, part, blockIdx.x, blockIdx.y);
}

// Few tokens, E > 32, as one launch without any memory-based synchronisation:
// a thread-block cluster per block of 8 tokens, one CTA per slice of d (at
// most 8 slices). Each CTA brings its W_router rows and the 8 tokens' x
// slices into shared memory with bulk copies (one round trip), computes the
// partial logits of the slice there, and after a cluster barrier the CTAs
// sum the slices of their tokens in slice order straight from the peers'
// shared memory and route them (token c + ns w in warp w of the CTA of
// cluster rank c). WG (E up to 256, whose W_router slice does not fit shared
// memory): the slice streams through a ring of three 32-row chunks in shared
// memory (bulk copies, one thread per expert consuming each row).
constexpr int WG_ROWS = 32;  // W_router rows per streamed chunk (WG)
constexpr int WG_BUFS = 3;

struct ClusterRouterShape {
    int ns, lenc;
    bool wg;  // W_router read from global memory (more than 128 experts)
    size_t smem;
};

template <bool BF16, int EP, bool WG>
__global__ void __launch_bounds__(256) router_cluster_kernel(RouterArgs a, int lenc, uint64_t timeout_ns) {
    extern __shared__ __align__(128) uint8_t sm[];
    constexpr int R = 256 / EP;  // parts per expert
    constexpr int J = EP / 32;
    constexpr int XES = BF16 ? 2 : 4;
    const int E = a.E, d = a.d;
    const int ns = static_cast<int>(gridDim.x);  // cluster = the token block's slices
    const int c = static_cast<int>(cluster_ctarank());
    const int t0 = blockIdx.y * 8, k0 = c * lenc;
    const int kn = max(0, min(lenc, d - k0));
    const int ntok = min(8, a.T - t0);
    const int xstage_bytes = (8 * lenc * XES + 15) / 16 * 16;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm);  // [0]: x and W slice; [1..]: WG ring
    uint8_t* xstage = sm + 64;
    float* xt = reinterpret_cast<float*>(xstage + xstage_bytes);  // [lenc][8]
    float* ws = xt + 8 * lenc;  // [lenc][E]; WG: the ring [WG_BUFS][WG_ROWS][EP]
    float* part = ws + (WG ? static_cast<size_t>(WG_BUFS) * WG_ROWS * EP : static_cast<size_t>(lenc) * E);
    float* red = part + 8 * EP;                                   // [R-1][8][EP]
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(bar);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(b, 1);
        if (WG)
            for (int i = 0; i < WG_BUFS; ++i) mbar_init(b + 8u * (1 + i), 1);
        fence_mbarrier_init();
    }
    pdl_wait();
    pdl_trigger();
    if (a.err_clear != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        clear_status(a.err_clear);
    zero_counters(a, blockIdx.x == 0 && blockIdx.y == 0);
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t wbytes = WG ? 0u : static_cast<uint32_t>(kn) * E * 4;
        const uint32_t xbytes = static_cast<uint32_t>(kn) * XES;
        mbar_expect_tx(b, wbytes + xbytes * ntok);
        if (kn > 0) {
            if (!WG) bulk_load(smem_u32(ws), a.W + static_cast<size_t>(k0) * E, wbytes, b);
            for (int tt = 0; tt < ntok; ++tt)
                bulk_load(smem_u32(xstage + static_cast<size_t>(tt) * lenc * XES),
                          static_cast<const uint8_t*>(a.x) +
                              (static_cast<size_t>(t0 + tt) * d + k0) * XES,
                          xbytes, b);
        }
        if (WG) {
            // the first chunks of the W_router slice
            const int nch = (kn + WG_ROWS - 1) / WG_ROWS;
            for (int i = 0; i < WG_BUFS && i < nch; ++i) {
                const int rows = min(WG_ROWS, kn - i * WG_ROWS);
                const uint32_t bytes = static_cast<uint32_t>(rows) * E * 4;
                mbar_expect_tx(b + 8u * (1 + i), bytes);
                bulk_load(smem_u32(ws + static_cast<size_t>(i) * WG_ROWS * EP),
                          a.W + static_cast<size_t>(k0 + i * WG_ROWS) * E, bytes, b + 8u * (1 + i));
            }
        }
    }
    // the routing warps' bias values, loaded while the copies are in flight
    float bj[J];
    load_bias_lanes<J>(a, bj);
    const WaitCtx wc{a.err_clear, &abort_flag, timeout_ns};
    const bool ok = bounded_wait(b, 0, wc);
    // x slices as FP32, transposed to [k][token] (zero for missing tokens)
    for (int i = threadIdx.x; i < 8 * kn; i += blockDim.x) {
        const int tt = i / kn, k = i - tt * kn;
        float v = 0.0f;
        if (ok && tt < ntok) {
            v = BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(xstage)[tt * lenc + k])
                     : reinterpret_cast<const float*>(xstage)[tt * lenc + k];
        }
        xt[k * 8 + tt] = v;
    }
    __syncthreads();
    const int e = threadIdx.x % EP, r = threadIdx.x / EP;
    const int run = (kn + R - 1) / R;
    const int kb = r * run, ke = min(kb + run, kn);
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    if (WG) {
        // stream the slice: chunk i in buffer i % WG_BUFS, refilled with chunk
        // i + WG_BUFS once every thread has used it; rows in order, as above
        const int nch = (kn + WG_ROWS - 1) / WG_ROWS;
        bool okc = ok;
        int consumed = 0;
        for (int i = 0; i < nch; ++i) {
            const int buf = i % WG_BUFS;
            if (okc) okc = bounded_wait(b + 8u * (1 + buf), static_cast<uint32_t>((i / WG_BUFS) & 1), wc);
            if (okc) consumed = i + 1;
            const int rows = min(WG_ROWS, kn - i * WG_ROWS);
            if (okc && e < E) {
                const float* wb = ws + static_cast<size_t>(buf) * WG_ROWS * EP;
                for (int r0 = 0; r0 < rows; ++r0) {
                    const float wv = wb[r0 * E + e];
                    const int k = i * WG_ROWS + r0;
                    const float4 x0 = *reinterpret_cast<const float4*>(xt + k * 8);
                    const float4 x1 = *reinterpret_cast<const float4*>(xt + k * 8 + 4);
                    acc[0] = fmaf(x0.x, wv, acc[0]);
                    acc[1] = fmaf(x0.y, wv, acc[1]);
                    acc[2] = fmaf(x0.z, wv, acc[2]);
                    acc[3] = fmaf(x0.w, wv, acc[3]);
                    acc[4] = fmaf(x1.x, wv, acc[4]);
                    acc[5] = fmaf(x1.y, wv, acc[5]);
                    acc[6] = fmaf(x1.z, wv, acc[6]);
                    acc[7] = fmaf(x1.w, wv, acc[7]);
                }
            }
            __syncthreads();
            if (threadIdx.x == 0 && i + WG_BUFS < nch && !abort_flag) {
                const int j = i + WG_BUFS;
                const int rj = min(WG_ROWS, kn - j * WG_ROWS);
                const uint32_t bytes = static_cast<uint32_t>(rj) * E * 4;
                mbar_expect_tx(b + 8u * (1 + buf), bytes);
                bulk_load(smem_u32(ws + static_cast<size_t>(buf) * WG_ROWS * EP),
                          a.W + static_cast<size_t>(k0 + j * WG_ROWS) * E, bytes, b + 8u * (1 + buf));
            }
        }
        // copies issued and never waited for (a wait gave up) land before the exit
        if (threadIdx.x == 0 && consumed < nch) {
            const int issued = abort_flag ? min(nch, consumed + WG_BUFS) : nch;
            for (int i = consumed; i < issued; ++i)
                bounded_drain(b + 8u * (1 + i % WG_BUFS), static_cast<uint32_t>((i / WG_BUFS) & 1),
                              timeout_ns, a.err_clear);
        }
    }
    if (!WG && ok && e < E) {
        for (int k = kb; k < ke; ++k) {
            const float wv = ws[static_cast<size_t>(k) * E + e];
            const float4 x0 = *reinterpret_cast<const float4*>(xt + k * 8);
            const float4 x1 = *reinterpret_cast<const float4*>(xt + k * 8 + 4);
            acc[0] = fmaf(x0.x, wv, acc[0]);
            acc[1] = fmaf(x0.y, wv, acc[1]);
            acc[2] = fmaf(x0.z, wv, acc[2]);
            acc[3] = fmaf(x0.w, wv, acc[3]);
            acc[4] = fmaf(x1.x, wv, acc[4]);
            acc[5] = fmaf(x1.y, wv, acc[5]);
            acc[6] = fmaf(x1.z, wv, acc[6]);
            acc[7] = fmaf(x1.w, wv, acc[7]);
        }
    }
    if (R > 1) {
        if (r > 0)
#pragma unroll
            for (int j = 0; j < 8; ++j) red[((r - 1) * 8 + j) * EP + e] = acc[j];
        __syncthreads();
        if (r == 0)
            for (int q = 0; q < R - 1; ++q)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] += red[(q * 8 + j) * EP + e];
    }
    if (r == 0)
#pragma unroll
        for (int j = 0; j < 8; ++j) part[j * EP + e] = acc[j];
    // every slice's partials are in its CTA's shared memory
    cluster_sync();

    const int lane = static_cast<int>(lane_id()), w = threadIdx.x >> 5;
    const int tt = c + ns * w;
    const bool mine = tt < ntok;
    float rl[J];
#pragma unroll
    for (int j = 0; j < J; ++j) rl[j] = 0.0f;
    if (mine) {
        float q[8][J];
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
            const uint32_t src = map_shared_rank(smem_u32(part + tt * EP), static_cast<uint32_t>(sl < ns ? sl : 0));
#pragma unroll
            for (int j = 0; j < J; ++j)
                q[sl][j] = (sl < ns) ? ld_shared_cluster_f32(src + 4u * (lane + 32 * j)) : 0.0f;
        }
#pragma unroll
        for (int sl = 0; sl < 8; ++sl)
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (sl < ns) rl[j] += q[sl][j];
    }
    // the peers' partials are read: a CTA may leave once every CTA got here
    cluster_arrive();
    if (mine) route_token_warp<J>(rl, bj, t0 + tt, a);
    if (!ok) bounded_drain(b, 0, timeout_ns, a.err_clear);
    cluster_wait();
}

ClusterRouterShape cluster_router_shape(int d, int E, int x_bf16) {
    ClusterRouterShape sh{};
    const int ns0 = std::min(8, (d + 127) / 128);
    sh.lenc = ((d + ns0 - 1) / ns0 + 15) / 16 * 16;
    sh.ns = (d + sh.lenc - 1) / sh.lenc;
    sh.wg = E > 128;
    const int EP = E <= 64 ? 64 : (E <= 128 ? 128 : 256);
    const int R = 256 / EP;
    const size_t xes = x_bf16 ? 2 : 4;
    sh.smem = 64 + (8 * sh.lenc * xes + 15) / 16 * 16 + 8 * static_cast<size_t>(sh.lenc) * 4 +
              (sh.wg ? static_cast<size_t>(WG_BUFS) * WG_ROWS * EP * 4 : static_cast<size_t>(sh.lenc) * E * 4) +
              8 * EP * 4 + (R - 1) * 8 * EP * 4;
    return sh;
}

constexpr size_t CLUSTER_ROUTER_SMEM_MAX = 200 * 1024;

// Decode batches (T <= 128, 128 < E <= 256, where the cluster router would
// stream its W_router slices through a ring) in one cooperative launch that
// reads W_router once: CTA (s, eb) holds the d-slice s of every token's x row
// and the 32 W_router columns of expert block eb in shared memory and forms
// the partial logits of all tokens for those 32 experts (FP32 FMA chains over
// the slice in increasing d); the partials go to global memory, then every
// CTA stores its tag (this launch's epoch tag, release order) and waits, with
// a time limit, for all tags (no zeroed memory needed); CTA c then routes tokens
// c, c + G, ...: each expert's logit is the sum of its slices' partials in
// slice order. (The cluster router re-reads W_router once per 8-token block.)
// The slices arrive by asynchronous 16-byte copies (one memory round trip, no
// registers held); x is then transposed to [k][token] FP32. Thread layout of
// the partial phase: warp w takes tokens 16 (w % WT) .. +15 over part w / WT
// of the slice; lane l the 4 tokens 16 (w % WT) + 4 (l >> 3) .. and the 4
// experts 4 (l & 7) .., so each k costs two 16-byte shared loads for 16 FMAs.
// Parts of a slice are added in part order.
constexpr int RD_THREADS = 512;
constexpr int RD_WARPS = RD_THREADS / 32;
constexpr int RD_EB = 32;    // experts per CTA
constexpr int RD_TMAX = 128;  // tokens
constexpr int RD_MAX_SLICES = 32;
constexpr size_t RD_SMEM_MAX = 210 * 1024;

// Row stride (elements) of the staged x slice [token][k]: 16-byte aligned
// rows whose 16-byte chunks start in different bank groups for 8 consecutive
// tokens (an odd number of chunks per row).
__host__ __device__ __forceinline__ int router_decode_xs(int lens, bool bf16) {
    const int per = bf16 ? 8 : 4;  // elements per 16-byte chunk
    return ((lens / per) % 2 == 0) ? lens + per : lens;
}

struct RouterDecodeShape {
    int neb, S, lens, G, tt, wt, kp;
    size_t smem;
};

RouterDecodeShape router_decode_shape(int T, int d, int E, bool bf16) {
    RouterDecodeShape sh{};
    sh.neb = (E + RD_EB - 1) / RD_EB;
    sh.tt = (T + 15) / 16 * 16;
    sh.wt = sh.tt / 16;
    sh.kp = sh.wt > 0 ? RD_WARPS / sh.wt : 1;
    const int G0 = std::min(num_sms(), FRONT_SMALL_MAX_CTAS);
    const int s0 = std::max(1, std::min(RD_MAX_SLICES, G0 / std::max(1, sh.neb)));
    sh.lens = ((d + s0 - 1) / s0 + 7) / 8 * 8;
    sh.S = (d + sh.lens - 1) / sh.lens;
    sh.G = sh.S * sh.neb;
    const size_t stage = static_cast<size_t>(sh.tt) * router_decode_xs(sh.lens, bf16) * (bf16 ? 2 : 4);
    const size_t red = static_cast<size_t>(sh.kp - 1) * sh.wt * 32 * 16 * 4;
    sh.smem = static_cast<size_t>(sh.lens) * (RD_EB + sh.tt) * 4 + std::max(stage, red);
    return sh;
}

template <bool BF16, int EP>
__global__ void __launch_bounds__(RD_THREADS, 1) router_decode_kernel(RouterArgs a, int S, int lens, int tt, int wt,
                                                                      int kp, float* __restrict__ part,
                                                                      unsigned long long* __restrict__ tags,
                                                                      uint64_t timeout_ns) {
    extern __shared__ __align__(16) float rsm[];
    __shared__ float s_r[EP];
    constexpr int J = EP / 32;
    constexpr int ES = BF16 ? 2 : 4;  // x element bytes
    constexpr int XV = 16 / ES;       // x elements per 16-byte chunk
    pdl_wait();
    pdl_trigger();
    // this launch's tag (every thread reads the epoch before any CTA can pass the barrier)
    unsigned long long* epoch = tags + GRID_TAG_STRIDE * GRID_EPOCH_LINE;
    const unsigned long long gid = grid_epoch_tag(epoch);
    const int b = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const int T = a.T, E = a.E, d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (a.err_clear != nullptr && b == 0 && threadIdx.x == 0) clear_status(a.err_clear);
    zero_counters(a, b == 0);
    const int sl = b % S, eb = b / S;
    const int k0 = sl * lens, kn = max(0, min(lens, d - k0));  // kn: a multiple of 8
    const int e0 = eb * RD_EB;
    const int xs = router_decode_xs(lens, BF16);
    float* ws = rsm;                                     // [lens][32] W_router columns e0 ..
    float* xt = ws + static_cast<size_t>(lens) * RD_EB;  // [lens][tt] x as FP32
    uint8_t* xst = reinterpret_cast<uint8_t*>(xt + static_cast<size_t>(lens) * tt);  // [tt][xs] staged x
    float* red = reinterpret_cast<float*>(xst);  // [kp - 1][wt][32][16], once the staged x is used

    // 1. the slice of W_router and of every token's x row
    if (E % 4 == 0) {
        for (int q = threadIdx.x; q < kn * 8; q += RD_THREADS) {
            const int k = q >> 3, c4 = q & 7, e = e0 + 4 * c4;
            float* dst = ws + k * RD_EB + 4 * c4;
            if (e < E)
                cp_async_16(dst, a.W + static_cast<size_t>(k0 + k) * E + e);
            else
                *reinterpret_cast<float4*>(dst) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
    } else {
        for (int q = threadIdx.x; q < kn * RD_EB; q += RD_THREADS) {
            const int k = q >> 5, c = q & 31, e = e0 + c;
            float* dst = ws + k * RD_EB + c;
            if (e < E)
                cp_async_4(dst, a.W + static_cast<size_t>(k0 + k) * E + e);
            else
                *dst = 0.0f;
        }
    }
    const int npc = kn / XV;  // 16-byte chunks per token
    // chunk pc of token t: threads take consecutive tokens for one chunk (the
    // first (RD_THREADS / tt) * tt threads)
    const int cstep = RD_THREADS / tt;
    const bool stager = static_cast<int>(threadIdx.x) < cstep * tt;
    for (int pc = stager ? threadIdx.x / tt : npc; pc < npc; pc += cstep) {
        const int t = threadIdx.x % tt;
        uint8_t* dst = xst + (static_cast<size_t>(t) * xs + pc * XV) * ES;
        if (t < T)
            cp_async_16(dst, static_cast<const uint8_t*>(a.x) + (static_cast<size_t>(t) * d + k0 + pc * XV) * ES);
        else
            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_wait_all();
    __syncthreads();
    // x to [k][token] FP32 (16-byte chunk reads, consecutive tokens per warp)
    for (int pc = stager ? threadIdx.x / tt : npc; pc < npc; pc += cstep) {
        const int t = threadIdx.x % tt;
        const uint4 v = *reinterpret_cast<const uint4*>(xst + (static_cast<size_t>(t) * xs + pc * XV) * ES);
        float f[XV];
        if (BF16) {
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = bf16_lo(w4[i]);
                f[(2 * i + 1) % XV] = bf16_hi(w4[i]);
            }
        } else {
            f[0] = __uint_as_float(v.x);
            f[1 % XV] = __uint_as_float(v.y);
            f[2 % XV] = __uint_as_float(v.z);
            f[3 % XV] = __uint_as_float(v.w);
        }
#pragma unroll
        for (int i = 0; i < XV; ++i) xt[static_cast<size_t>(pc * XV + i) * tt + t] = f[i];
    }
    __syncthreads();

    // 2. partial logits of the slice: 4 tokens x 4 experts per thread
    const int pp = warp / wt, wtok = warp - pp * wt;
    const int eg = lane & 7, tg = lane >> 3;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    if (pp < kp) {
        const int kper = (kn + kp - 1) / kp;
        const int kb = min(kn, pp * kper), ke = min(kn, kb + kper);
        const float* wr = ws + eg * 4;
        const float* xr = xt + wtok * 16 + tg * 4;
#pragma unroll 4
        for (int k = kb; k < ke; ++k) {
            const float4 w0 = *reinterpret_cast<const float4*>(wr + k * RD_EB);
            const float4 x0 = *reinterpret_cast<const float4*>(xr + static_cast<size_t>(k) * tt);
            const float xa[4] = {x0.x, x0.y, x0.z, x0.w}, wa[4] = {w0.x, w0.y, w0.z, w0.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wa[j], acc[i][j]);
        }
        if (pp > 0) {
            float4* rp = reinterpret_cast<float4*>(red + ((static_cast<size_t>(pp - 1) * wt + wtok) * 32 + lane) * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) rp[i] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
    }
    if (kp > 1) __syncthreads();
    if (pp == 0) {
        for (int q = 1; q < kp; ++q) {
            const float4* rp =
                reinterpret_cast<const float4*>(red + ((static_cast<size_t>(q - 1) * wt + wtok) * 32 + lane) * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = rp[i];
                acc[i][0] += v.x;
                acc[i][1] += v.y;
                acc[i][2] += v.z;
                acc[i][3] += v.w;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = wtok * 16 + tg * 4 + i;
            if (t < T) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int e = e0 + eg * 4 + j;
                    if (e < E) part[(static_cast<size_t>(sl) * T + t) * E + e] = acc[i][j];
                }
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // the CTA's partials (ordered by the barrier above) before the tag
        st_release_u64(tags + GRID_TAG_STRIDE * b, gid);
    }
    const bool okb = grid_tags_wait_cta(tags, G, gid, timeout_ns, a.err_clear);
    grid_epoch_store(epoch, gid);  // every CTA has read the epoch by now
    if (!okb) return;

    // 3. route tokens b, b + G, ...: expert e's logit in thread e, its slices
    //    summed in slice order
    for (int t = b; t < T; t += G) {
        if (static_cast<int>(threadIdx.x) < EP) {
            const int e = threadIdx.x;
            float r = 0.0f;
            if (e < E) {
                float v[RD_MAX_SLICES];
#pragma unroll
                for (int q = 0; q < RD_MAX_SLICES; ++q)
                    v[q] = q < S ? __ldcg(part + (static_cast<size_t>(q) * T + t) * E + e) : 0.0f;
#pragma unroll
                for (int q = 0; q < RD_MAX_SLICES; ++q)
                    if (q < S) r += v[q];
            }
            s_r[e] = r;
        }
        __syncthreads();
        if (warp == 0) {
            float rl[J];
#pragma unroll
            for (int j = 0; j < J; ++j) rl[j] = s_r[lane + 32 * j];
            route_token_warp<J>(rl, t, a);
        }
        __syncthreads();
    }
}

}  // namespace

bool router_decode_ok(int T, int d, int E, int x_bf16) {
    // up to 128 experts the cluster router holds its W_router slices in shared
    // memory and sums them over a cluster barrier: faster than the grid barrier
    if (T < 1 || T > RD_TMAX || E <= 128 || E > 256 || d % 16) return false;
    const RouterDecodeShape sh = router_decode_shape(T, d, E, x_bf16 != 0);
    return sh.G <= std::min(num_sms(), FRONT_SMALL_MAX_CTAS) && sh.S <= RD_MAX_SLICES && sh.smem <= RD_SMEM_MAX;
}

int router_decode_slices(int T, int d, int E) { return router_decode_shape(T, d, E, true).S; }

cudaError_t launch_router_decode(const RouterArgs& a, float* part, unsigned long long* tags, cudaStream_t s) {
    if (!router_decode_ok(a.T, a.d, a.E, a.x_bf16) || a.err_clear == nullptr || tags == nullptr)
        return cudaErrorInvalidValue;
    const RouterDecodeShape sh = router_decode_shape(a.T, a.d, a.E, a.x_bf16 != 0);
    const uint64_t to = wait_timeout_ns();
#define MOE_RD(B, EPV)                                                                                 \
    {                                                                                                  \
        static bool set = false;                                                                       \
        if (!set) {                                                                                    \
            const cudaError_t ea = cudaFuncSetAttribute(router_decode_kernel<B, EPV>,                  \
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                                                        static_cast<int>(RD_SMEM_MAX));                \
            if (ea != cudaSuccess) return ea;                                                          \
            set = true;                                                                                \
        }                                                                                              \
        return launch_pdl_coop(router_decode_kernel<B, EPV>, dim3(sh.G), dim3(RD_THREADS), sh.smem, s, a, \
                               sh.S, sh.lens, sh.tt, sh.wt, sh.kp, part, tags, to);                    \
    }
    if (a.x_bf16) MOE_RD(true, 256)
    MOE_RD(false, 256)
#undef MOE_RD
}

bool router_one_launch(int T, int d, int E, int x_bf16) {
    if (E <= 32) return true;  // router_small_kernel
    if (router_decode_ok(T, d, E, x_bf16)) return true;  // router_decode_kernel (with a workspace)
    // the cluster router (launch_router_chunked with a workspace)
    return E <= 256 && T <= 512 && cluster_router_shape(d, E, x_bf16).smem <= CLUSTER_ROUTER_SMEM_MAX;
}

namespace {

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
    const ClusterRouterShape sh = cluster_router_shape(a.d, a.E, a.x_bf16);
    if (a.err_clear != nullptr && sh.smem <= CLUSTER_ROUTER_SMEM_MAX) {
        const dim3 grid(sh.ns, (a.T + 7) / 8);
        const uint64_t to = wait_timeout_ns();
#define MOE_RCL(B, EPV, WGV)                                                                       \
    {                                                                                              \
        static bool set = false;                                                                   \
        if (!set) {                                                                                \
            cudaFuncSetAttribute(router_cluster_kernel<B, EPV, WGV>,                               \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,                      \
                                 static_cast<int>(CLUSTER_ROUTER_SMEM_MAX));                       \
            set = true;                                                                            \
        }                                                                                          \
        return launch_pdl_cluster(router_cluster_kernel<B, EPV, WGV>, grid, dim3(256), sh.smem, s, \
                                  sh.ns, a, sh.lenc, to);                                          \
    }
        if (a.x_bf16) {
            if (a.E <= 64) MOE_RCL(true, 64, false)
            if (a.E <= 128) MOE_RCL(true, 128, false)
            MOE_RCL(true, 256, true)
        } else {
            if (a.E <= 64) MOE_RCL(false, 64, false)
            if (a.E <= 128) MOE_RCL(false, 128, false)
            MOE_RCL(false, 256, true)
        }
#undef MOE_RCL
    }
    // wide slices that do not fit shared memory: partials through global memory
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
