// K1+K2 in one launch for prefill batches of a BF16 layer with few experts
// (E <= 8, 1024 < T*K <= 16384, no latent projection): router, dispatch and
// row gather. It replaces the router launch and the dispatch-and-gather
// launch, whose dispatch every CTA recomputed from all T*K assignments.
//
// What it computes is exactly what those two launches compute (same logits
// bit for bit, same routing, same integer dispatch):
//   r[t, :] = x[t, :] W_router (FP32), the gate rule's top-K (APEX-1
//   Mathematical Reference Part 3 section 13.1; "MoE from scratch"
//   MoELayer.forward), then the stable counting sort of the T*K (token, slot)
//   assignments by expert (kimi_k3 StableLatentMoE "Grouped expert
//   execution": tokens of one expert in token order) and xs[pos] = x[token].
//
// Shape: one CTA per SM at most, launched cooperatively (all CTAs resident at
// once). CTA b routes a contiguous block of tokens, so its assignments are a
// contiguous range of the (token, slot) order:
//   1. its tokens' x rows into shared memory with every load in flight, one
//      warp per token (lane l takes the d-index pairs 2l + 64m in increasing m,
//      the fused multiply-adds of the standalone router in the same order,
//      then the same butterfly and the same per-token routing);
//   2. ranks inside the range (warp match) and the CTA's per-expert counts,
//      published as count words: each 64-bit word holds two experts' counts
//      (10 bits each) under a 44-bit tag taken from this launch's epoch tag
//      (one more than the workspace's epoch word, which CTA 0 advances after
//      the barrier), stored with release order; every CTA waits, with a time
//      limit, until all words carry this launch's tag - a grid barrier that
//      needs no zeroed memory (a dirty workspace and graph replays are fine)
//      and whose polls bring the counts along;
//   3. expert totals, the CTA's prefix per expert (counts of the CTAs before
//      it), offsets and tile prefixes (CTA 0 writes them), sorted_token /
//      sorted_w / inv, and the rows copied into xs from shared memory.
#include "common.cuh"
#include "internal.h"
#include "route_dev.cuh"

namespace moe {
namespace {

constexpr int FS_THREADS = 512;
constexpr int FS_WARPS = FS_THREADS / 32;
constexpr size_t FS_SMEM_MAX = 190 * 1024;  // dynamic; the static arrays take up to ~31 KB
constexpr int FS_MAX_G = 256;  // blocks at most (one per SM)

// The count words' tag: 44 bits of the launch's epoch tag, never zero (a
// zeroed word never passes for a launch's).
MOE_DEV unsigned long long fs_tag(unsigned long long ep) { return ((ep << 1) | 1ULL) & ((1ULL << 44) - 1); }

// Every thread of each CTA, once the CTA's count words were stored: the G * EP/2
// words (word q of CTA i: counts of experts 2q and 2q + 1 in bits 0-9 and 10-19)
// are watched with relaxed loads until they carry this launch's tag, and their
// counts go to s_all[i * EP + expert]. The counts travel inside the watched
// words, so no other memory needs ordering. False when timeout_ns ran out (the
// error word gets ERRBIT_TIMEOUT).
template <int EP>
MOE_DEV bool fs_wait_counts(const unsigned long long* tags, int G, unsigned long long tag, uint64_t timeout_ns,
                            int* err, int* s_all) {
    constexpr int NW = EP / 2;
    bool ok = true;
    const uint64_t start = globaltimer_ns();
    for (int i = threadIdx.x; i < G * NW && ok; i += FS_THREADS) {
        const int blk = i / NW, q = i - blk * NW;
        const unsigned long long* p = tags + GRID_TAG_STRIDE * blk + q;
        unsigned long long v = ld_relaxed_u64(p);
        while ((v >> 20) != tag) {
            if (globaltimer_ns() - start > timeout_ns) {
                ok = false;
                break;
            }
            v = ld_relaxed_u64(p);
        }
        s_all[blk * EP + 2 * q] = static_cast<int>(v & 1023u);
        s_all[blk * EP + 2 * q + 1] = static_cast<int>((v >> 10) & 1023u);
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok && threadIdx.x == 0) atomicOr(err, ERRBIT_TIMEOUT);
    return ok;
}

template <int EP>
__global__ void __launch_bounds__(FS_THREADS, 1) front_small_kernel(RouterArgs ra, DispatchArgs da, int tpc,
                                                                    void* __restrict__ xs,
                                                                    unsigned long long* __restrict__ tags,
                                                                    uint64_t timeout_ns) {
    extern __shared__ __align__(16) uint8_t xsm[];
    __shared__ int s_base[EP], s_rank[FS_WARPS][EP];
    __shared__ int s_pos[FS_WARPS * 32], s_tok[FS_WARPS * 32], s_ids[FS_WARPS * 32];
    __shared__ float s_wt[FS_WARPS * 32];  // the block's gate weights, in (token, slot) order
    __shared__ float s_logit[FS_WARPS * 32 * EP];  // the block's logits (tpc <= FS_WARPS * 32)
    __shared__ int s_all[FS_MAX_G * EP];  // every block's counts
    pdl_wait();
    pdl_trigger();
    // this launch's tag (every thread reads the epoch before any CTA can pass the barrier)
    unsigned long long* epoch = tags + GRID_TAG_STRIDE * GRID_EPOCH_LINE;
    const unsigned long long ep = grid_epoch_tag(epoch);
    const int b = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (ra.err_clear != nullptr && b == 0 && threadIdx.x == 0) clear_status(ra.err_clear);
    const int E = ra.E, K = ra.K, d = ra.d, T = ra.T;
    const int t0 = min(T, b * tpc), t1 = min(T, t0 + tpc);
    const int nt = t1 - t0;
    for (int i = threadIdx.x; i < FS_WARPS * EP; i += FS_THREADS) (&s_rank[0][0])[i] = 0;

    // 1. stage the block's x rows and W_router (EP columns, zero beyond E) with
    //    every load in flight, then route: warp w takes tokens w and w + 16
    //    together (the W_router values it reads serve both)
    const int xbytes = nt * d * 2;
    float* wsm = reinterpret_cast<float*>(xsm + ((tpc * d * 2 + 15) & ~15));
    {
        // up to 8 x pieces and 8 W_router values per thread in flight per round
        // (one round for the small layer) before any of them is stored
        const int nvec = xbytes / 16, nw = d * EP;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ra.x) +
                                                          static_cast<size_t>(t0) * d);
        uint4* dst = reinterpret_cast<uint4*>(xsm);
        const int n = nvec > nw ? nvec : nw;
        for (int base = threadIdx.x; base < n; base += 8 * FS_THREADS) {
            uint4 xv[8];
            float wv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = base + u * FS_THREADS;
                if (q < nvec) xv[u] = __ldg(src + q);
                wv[u] = 0.0f;
                if (q < nw) {
                    const int k = q / EP, e = q - k * EP;
                    if (e < E) wv[u] = __ldg(ra.W + static_cast<size_t>(k) * E + e);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = base + u * FS_THREADS;
                if (q < nvec) dst[q] = xv[u];
                if (q < nw) wsm[q] = wv[u];
            }
        }
    }
    __syncthreads();
    for (int i = warp; i < nt; i += 2 * FS_WARPS) {
        const int i2 = i + FS_WARPS;
        const bool two = i2 < nt;
        const uint32_t* xa = reinterpret_cast<const uint32_t*>(xsm) + static_cast<size_t>(i) * (d >> 1);
        const uint32_t* xb = reinterpret_cast<const uint32_t*>(xsm) + static_cast<size_t>(two ? i2 : i) * (d >> 1);
        float acc[EP], acc2[EP];
#pragma unroll
        for (int e = 0; e < EP; ++e) acc[e] = acc2[e] = 0.0f;
        // lane l: d-index pairs k = 2 l + 64 m, m increasing (the standalone
        // router's order), one fused multiply-add chain per expert
#pragma unroll 4
        for (int k = 2 * lane; k < d; k += 64) {
            const uint32_t va = xa[k >> 1], vb = xb[k >> 1];
            const float a0 = bf16_lo(va), a1 = bf16_hi(va), b0 = bf16_lo(vb), b1 = bf16_hi(vb);
            // rows k and k + 1 of W_router: 2 EP contiguous floats, 16-byte loads
            const float4* w4 = reinterpret_cast<const float4*>(wsm + static_cast<size_t>(k) * EP);
            float wr0[EP], wr1[EP];
#pragma unroll
            for (int e = 0; e < EP; e += 4) {
                const float4 p0 = w4[e / 4], p1 = w4[EP / 4 + e / 4];
                wr0[e] = p0.x; wr0[e + 1] = p0.y; wr0[e + 2] = p0.z; wr0[e + 3] = p0.w;
                wr1[e] = p1.x; wr1[e + 1] = p1.y; wr1[e + 2] = p1.z; wr1[e + 3] = p1.w;
            }
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                acc[e] = fmaf(a1, wr1[e], fmaf(a0, wr0[e], acc[e]));
                acc2[e] = fmaf(b1, wr1[e], fmaf(b0, wr0[e], acc2[e]));
            }
        }
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            acc[e] = warp_sum(acc[e]);
            acc2[e] = warp_sum(acc2[e]);
        }
        if (lane == 0) {
#pragma unroll
            for (int e = 0; e < EP; ++e) s_logit[i * EP + e] = acc[e];
        }
        if (lane == 1 && two) {
#pragma unroll
            for (int e = 0; e < EP; ++e) s_logit[i2 * EP + e] = acc2[e];
        }
    }
    __syncthreads();
    // one thread per token: the per-token routing is a serial chain, so all of
    // the block's tokens take it side by side
    if (threadIdx.x < nt) {
        float r[EP];
#pragma unroll
        for (int e = 0; e < EP; ++e) r[e] = s_logit[threadIdx.x * EP + e];
        route_token_seq<EP>(r, t0 + threadIdx.x, ra, s_ids + threadIdx.x * K, s_wt + threadIdx.x * K);
    }
    __syncthreads();  // the block's ids and gate weights are in shared memory

    // 2. ranks inside the block's range (one assignment per thread: tpc * K <=
    //    FS_THREADS), the block's counts as count words; wait for every block's
    const int j0 = t0 * K, j1 = t1 * K;
    const int j = j0 + static_cast<int>(threadIdx.x);
    const bool mine = j < j1;
    int e = mine ? s_ids[threadIdx.x] : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) s_rank[warp][e] = __popc(peers);
    __syncthreads();
    const unsigned long long tag = fs_tag(ep);
    if (threadIdx.x < EP / 2) {
        const int e0 = 2 * static_cast<int>(threadIdx.x);
        unsigned long long c0 = 0, c1 = 0;
#pragma unroll
        for (int w = 0; w < FS_WARPS; ++w) {
            c0 += static_cast<unsigned>(s_rank[w][e0]);
            c1 += static_cast<unsigned>(s_rank[w][e0 + 1]);
        }
        st_release_u64(tags + GRID_TAG_STRIDE * b + threadIdx.x, (tag << 20) | (c1 << 10) | c0);
    }
    const bool okb = fs_wait_counts<EP>(tags, G, tag, timeout_ns, da.err, s_all);
    grid_epoch_store(epoch, ep);  // every CTA has read the epoch by now
    if (!okb) return;

    // 3. warp 0: every expert's total and its count in the blocks before this
    //    one, the scan into offsets and tile prefixes, the block's base per expert
    if (warp == 0) {
        int tot_e[EP], pre_e[EP];
#pragma unroll
        for (int x = 0; x < EP; ++x) tot_e[x] = pre_e[x] = 0;
        for (int i = lane; i < G; i += 32) {
#pragma unroll
            for (int x = 0; x < EP; ++x) {
                const int c = s_all[i * EP + x];
                tot_e[x] += c;
                pre_e[x] += i < b ? c : 0;
            }
        }
        int tot = 0, pre = 0;
#pragma unroll
        for (int x = 0; x < EP; ++x) {
            const int tx = __reduce_add_sync(0xffffffffu, tot_e[x]);
            const int px = __reduce_add_sync(0xffffffffu, pre_e[x]);
            if (lane == x && x < E) {
                tot = tx;
                pre = px;
            }
        }
        const int bm = da.bm;
        const int m1 = (tot + bm - 1) / bm, m2 = (tot + 2 * bm - 1) / (2 * bm);
        int x = tot, x1 = m1, x2 = m2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            const int y1 = __shfl_up_sync(0xffffffffu, x1, o);
            const int y2 = __shfl_up_sync(0xffffffffu, x2, o);
            if (lane >= o) {
                x += y;
                x1 += y1;
                x2 += y2;
            }
        }
        if (lane < E) {
            s_base[lane] = x - tot + pre;
            if (b == 0) {
                da.counts[lane] = tot;
                da.offsets[lane] = x - tot;
                da.mt_prefix[lane] = x1 - m1;
                da.mt_prefix[E + 1 + lane] = x2 - m2;
                if (lane == E - 1) {
                    da.offsets[E] = x;
                    da.mt_prefix[E] = x1;
                    da.mt_prefix[2 * E + 1] = x2;
                }
            }
        }
    }
    __syncthreads();
    if (mine) {
        int pos = -1;
        if (e >= 0) {
            pos = s_base[e] + rank;
            for (int w = 0; w < warp; ++w) pos += s_rank[w][e];
            da.sorted_token[pos] = j / K;
            da.sorted_w[pos] = s_wt[threadIdx.x];
            da.inv[j] = pos;
        }
        s_pos[threadIdx.x] = pos;
        s_tok[threadIdx.x] = j / K - t0;
    }
    __syncthreads();
    const int vpr = d / 8;  // 16-byte pieces per row
    const uint4* rows = reinterpret_cast<const uint4*>(xsm);
    uint4* out = static_cast<uint4*>(xs);
    for (int r = warp; r < j1 - j0; r += FS_WARPS) {
        const int pos = s_pos[r];
        if (pos < 0) continue;
        const uint4* sr = rows + static_cast<size_t>(s_tok[r]) * vpr;
        uint4* dr = out + static_cast<size_t>(pos) * vpr;
        for (int v = lane; v < vpr; v += 32) dr[v] = sr[v];
    }
}

// Dynamic shared memory: the block's x rows, then W_router as [d, 8] FP32.
size_t front_small_smem(int tpc, int d) {
    return ((static_cast<size_t>(tpc) * d * 2 + 15) & ~static_cast<size_t>(15)) + static_cast<size_t>(d) * 8 * 4;
}

}  // namespace

bool front_small_ok(int T, int d, int E, int K) {
    const long long TK = static_cast<long long>(T) * K;
    if (E < 1 || E > 8 || K < 1 || TK <= 1024 || TK > DISPATCH_WIDE_MAX || d % 8) return false;
    const int G = num_sms() < FS_MAX_G ? num_sms() : FS_MAX_G;
    const int tpc = (T + G - 1) / G;
    return tpc * K <= FS_WARPS * 32 && front_small_smem(tpc, d) <= FS_SMEM_MAX;
}

cudaError_t launch_front_small(const RouterArgs& ra, const DispatchArgs& da, void* xs,
                               unsigned long long* tags, cudaStream_t s) {
    if (!front_small_ok(ra.T, ra.d, ra.E, ra.K) || !ra.x_bf16) return cudaErrorInvalidValue;
    const int G0 = num_sms() < FS_MAX_G ? num_sms() : FS_MAX_G;
    const int tpc = (ra.T + G0 - 1) / G0;
    const int G = (ra.T + tpc - 1) / tpc;
    const size_t smem = front_small_smem(tpc, ra.d);
    static bool attr_set[64][2] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const int which = ra.E <= 4 ? 0 : 1;
    if (dev >= 0 && dev < 64 && !attr_set[dev][which]) {
        const cudaError_t e = which == 0
            ? cudaFuncSetAttribute(front_small_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(FS_SMEM_MAX))
            : cudaFuncSetAttribute(front_small_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(FS_SMEM_MAX));
        if (e != cudaSuccess) return e;
        attr_set[dev][which] = true;
    }
    const uint64_t tmo = wait_timeout_ns();
    return which == 0
        ? launch_pdl_coop(front_small_kernel<4>, dim3(G), dim3(FS_THREADS), smem, s, ra, da, tpc, xs, tags, tmo)
        : launch_pdl_coop(front_small_kernel<8>, dim3(G), dim3(FS_THREADS), smem, s, ra, da, tpc, xs, tags, tmo);
}

}  // namespace moe
