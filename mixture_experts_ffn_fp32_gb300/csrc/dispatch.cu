// K2 - sorted dispatch: per-expert histogram, exclusive scan and a stable
// scatter that lists the T*K assignments expert by expert, plus the row
// gather that lays the tokens' activations out in that order.
//
// Source: kimi_k3 StableLatentMoE, "Flatten routing and recover original
// token order" and "Dispatch is a stable permutation, not token duplication
// in model state": the flat ids are sorted with a stable argsort, the sorted
// assignment at position pos belongs to token order[pos] // K, bincount gives
// the expert loads and their cumulative sums the expert slices.
//
// Here the stable argsort is a counting sort done in two launches with no
// host synchronisation: (a) each CTA histograms a chunk of 1024 consecutive
// flat assignments, and the CTA that finishes last (a ticket counter) turns
// the chunk histograms into per-expert offsets and per-chunk bases (and the
// per-expert GEMM tile prefixes), (b) each CTA ranks its chunk's assignments
// stably (warp match + per-warp counts) and writes sorted_token / sorted_w /
// inv. Integer arithmetic only, so the result is bit-exact and independent of
// scheduling.
#include <algorithm>

#include "common.cuh"
#include "dispatch_dev.cuh"
#include "internal.h"

namespace moe {
namespace {

// Exclusive scan of v over the 256 threads of the block (all threads call).
__device__ int block_exclusive_scan(int v, int* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = (lane < 8) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < 8) warp_tot[lane] = t;  // inclusive warp totals
    }
    __syncthreads();
    const int before = (warp > 0) ? warp_tot[warp - 1] : 0;
    const int excl = before + x - v;
    __syncthreads();
    return excl;
}

// Per-expert offsets, per-chunk bases and GEMM tile prefixes from the chunk
// histograms (one CTA of 256 threads, thread e = expert e). The histograms
// were written by other CTAs of the same grid: read through L2 (ld.cg).
__device__ void dispatch_scan(const int32_t* chunk_counts, int nchunks, int E, int bm,
                              int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                              int32_t* __restrict__ offsets, int32_t* __restrict__ mt_prefix) {
    __shared__ int warp_tot[8];
    const int e = threadIdx.x;
    // 8 histogram loads in flight per step rather than one round trip per chunk
    auto load8 = [&](int b0, int (&c)[8]) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            c[i] = (b0 + i < nchunks) ? __ldcg(chunk_counts + static_cast<size_t>(b0 + i) * E + e) : 0;
    };
    int running = 0;
    if (e < E) {
        for (int b0 = 0; b0 < nchunks; b0 += 8) {
            int c[8];
            load8(b0, c);
#pragma unroll
            for (int i = 0; i < 8; ++i) running += c[i];
        }
    }
    const int cnt = (e < E) ? running : 0;
    const int off = block_exclusive_scan(cnt, warp_tot);
    // tiles of bm rows per expert (mt_prefix[0..E]) and of 2 bm rows (mt_prefix[E+1..2E+1])
    const int mt = (cnt + bm - 1) / bm;
    const int mtoff = block_exclusive_scan(mt, warp_tot);
    const int mt2 = (cnt + 2 * bm - 1) / (2 * bm);
    const int mtoff2 = block_exclusive_scan(mt2, warp_tot);
    if (e < E) {
        counts[e] = cnt;
        offsets[e] = off;
        mt_prefix[e] = mtoff;
        mt_prefix[E + 1 + e] = mtoff2;
        // chunk b of expert e starts after the expert's earlier chunks
        int base = off;
        for (int b0 = 0; b0 < nchunks; b0 += 8) {
            int c[8];
            load8(b0, c);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (b0 + i < nchunks) chunk_base[static_cast<size_t>(b0 + i) * E + e] = base;
                base += c[i];
            }
        }
    }
    if (e == E - 1) {
        offsets[E] = off + cnt;
        mt_prefix[E] = mtoff + mt;
        mt_prefix[2 * E + 1] = mtoff2 + mt2;
    }
}

// (a): histogram of one chunk; the last CTA to finish then runs the scan and
// re-arms the ticket (zero) for the next dispatch.
__global__ void __launch_bounds__(256) dispatch_count_kernel(
    const int32_t* __restrict__ idx, int TK, int E, int nchunks, int bm,
    int32_t* __restrict__ chunk_counts, int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ mt_prefix,
    int* ticket, int* err) {
    pdl_wait();
    pdl_trigger();
    __shared__ int hist[256];
    __shared__ int is_last;
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int j0 = blockIdx.x * DISPATCH_CHUNK;
    const int j1 = min(j0 + DISPATCH_CHUNK, TK);
    bool bad = false;
    for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
        const int e = idx[j];
        if (e >= 0 && e < E)
            atomicAdd(&hist[e], 1);
        else
            bad = true;
    }
    if (bad) atomicOr(err, ERRBIT_INDEX);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_counts[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];
    // publish this chunk's histogram, then take a ticket
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(ticket, 1) == nchunks - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    if (threadIdx.x == 0) *ticket = 0;
    dispatch_scan(chunk_counts, nchunks, E, bm, chunk_base, counts, offsets, mt_prefix);
}

__global__ void __launch_bounds__(DISPATCH_CHUNK) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, int TK, int K, int E,
    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ sorted_token,
    float* __restrict__ sorted_w, int32_t* __restrict__ inv) {
    pdl_wait();
    pdl_trigger();
    __shared__ int wcnt[32][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 32 * 256; i += blockDim.x) (&wcnt[0][0])[i] = 0;
    __syncthreads();
    const int j = blockIdx.x * DISPATCH_CHUNK + threadIdx.x;
    int e = (j < TK) ? idx[j] : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
        int run = 0;
        for (int ww = 0; ww < 32; ++ww) {
            const int c = wcnt[ww][x];
            wcnt[ww][x] = run;
            run += c;
        }
    }
    __syncthreads();
    if (e >= 0) {
        const int pos = chunk_base[static_cast<size_t>(blockIdx.x) * E + e] + wcnt[warp][e] + rank;
        sorted_token[pos] = j / K;
        sorted_w[pos] = w[j];
        inv[j] = pos;
    }
}

// All of the dispatch for at most DISPATCH_CHUNK assignments (a decode batch)
// in one CTA of 1024 threads (dispatch_block): the same integer results as
// the two-launch path, one launch.
__global__ void __launch_bounds__(DISPATCH_CHUNK) dispatch_single_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, int TK, int K, int E, int bm,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ mt_prefix,
    int32_t* __restrict__ sorted_token, float* __restrict__ sorted_w, int32_t* __restrict__ inv,
    int* err) {
    pdl_wait();
    pdl_trigger();
    dispatch_block<DISPATCH_CHUNK, 256>(idx, w, TK, K, E, bm, true, counts, offsets, mt_prefix,
                                        sorted_token, sorted_w, inv, err);
}

// Dispatch and row gather of a decode batch (at most DISPATCH_CHUNK
// assignments) in one launch: every CTA runs the whole dispatch on its own
// (dispatch_block: the same integer results in each) and CTA 0 writes it out;
// each CTA then copies its rows of the gathered operand from the positions it
// computed itself, so nothing passes between CTAs. One warp per row, rows
// blockIdx.x * 8 + warp with a stride of 8 gridDim.x.
template <int EMAX>
__global__ void __launch_bounds__(256) dispatch_gather_kernel(DispatchArgs a,
                                                              const uint4* __restrict__ src,
                                                              int vec_per_row,
                                                              uint4* __restrict__ dst) {
    __shared__ int32_t tok[DISPATCH_CHUNK];
    // every row index defined even if an id were invalid (its row then copies token 0)
    for (int i = threadIdx.x; i < DISPATCH_CHUNK; i += blockDim.x) tok[i] = 0;
    pdl_wait();
    pdl_trigger();
    const int TK = a.T * a.K;
    dispatch_block<256, EMAX>(a.idx, a.w, TK, a.K, a.E, a.bm, blockIdx.x == 0, a.counts,
                              a.offsets, a.mt_prefix, a.sorted_token, a.sorted_w, a.inv, a.err,
                              tok);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < TK; r += gridDim.x * 8) {
        const size_t so = static_cast<size_t>(tok[r]) * vec_per_row;
        const size_t d = static_cast<size_t>(r) * vec_per_row;
        for (int v0 = lane; v0 < vec_per_row; v0 += 128) {
            uint4 buf[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (v0 + 32 * i < vec_per_row) buf[i] = __ldg(src + so + v0 + 32 * i);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (v0 + 32 * i < vec_per_row) dst[d + v0 + 32 * i] = buf[i];
        }
    }
}

// Dispatch and row gather of up to DISPATCH_WIDE_MAX assignments in one
// launch over many CTAs, with nothing passed between them: every CTA counts
// all assignments per expert itself (the totals, and the counts before its
// own range of per_cta consecutive assignments, a multiple of 32), which
// places each assignment of its range in the stable expert order; CTA 0
// writes the counts, offsets and tile prefixes; each CTA writes sorted_token
// / sorted_w / inv of its range and copies the range's rows (one warp per
// row, several rows of a warp in flight). The same integer results as the
// two-launch dispatch. E <= 8: 1024 threads, per-thread counters packed as
// 16-bit fields of two 64-bit words; otherwise 256 threads and per-warp
// counters in shared memory.
template <int EMAX, int NT>
__global__ void __launch_bounds__(NT) dispatch_gather_wide_kernel(DispatchArgs a, int per_cta,
                                                                  const uint4* __restrict__ src,
                                                                  int vpr, uint4* __restrict__ dst) {
    constexpr int NW = NT / 32;
    constexpr bool REG = EMAX <= 8;
    constexpr int RB = NT >= 1024 ? 2 : 4;  // rows of a warp in flight in the gather
    static_assert(DISPATCH_WIDE_MAX < 65536 && EMAX <= 256 && (REG || NT == 256), "wide dispatch shape");
    __shared__ int s_all[NW][EMAX];
    __shared__ int s_pre[NW][EMAX];
    __shared__ int s_rank[8][EMAX];
    __shared__ int s_tot[EMAX];
    __shared__ int s_base[EMAX];
    __shared__ int s_pos[256];
    __shared__ int s_tok[256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < NW * EMAX; i += NT) {
        (&s_all[0][0])[i] = 0;
        (&s_pre[0][0])[i] = 0;
    }
    for (int i = threadIdx.x; i < 8 * EMAX; i += NT) (&s_rank[0][0])[i] = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    const int TK = a.T * a.K, E = a.E;
    const int j0 = blockIdx.x * per_cta;
    const int j1 = min(j0 + per_cta, TK);
    bool bad = false;

    // 1. counts of all assignments per expert, and of those before j0 (packed
    //    fields: a CTA sees at most DISPATCH_WIDE_MAX ids, no field overflows)
    {
        unsigned long long all0 = 0, all1 = 0, pre0 = 0, pre1 = 0;
        auto count = [&](int j, int e) {
            if (e < 0 || e >= E) {
                bad = true;
                return;
            }
            if (REG) {
                const unsigned long long inc = 1ull << (16 * (e & 3));
                const bool hi = e >= 4, before = j < j0;
                all0 += hi ? 0ull : inc;
                all1 += hi ? inc : 0ull;
                pre0 += (before && !hi) ? inc : 0ull;
                pre1 += (before && hi) ? inc : 0ull;
            } else {
                atomicAdd(&s_all[warp][e], 1);
                if (j < j0) atomicAdd(&s_pre[warp][e], 1);
            }
        };
        const int nv = TK / 4;  // ids four at a time, up to four loads in flight per thread
        const int4* iv = reinterpret_cast<const int4*>(a.idx);
        for (int i0 = threadIdx.x; i0 < nv; i0 += 4 * NT) {
            int4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * NT;
                v[u] = i < nv ? __ldcg(iv + i) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * NT;
                if (i < nv) {
                    count(4 * i, v[u].x);
                    count(4 * i + 1, v[u].y);
                    count(4 * i + 2, v[u].z);
                    count(4 * i + 3, v[u].w);
                }
            }
        }
        for (int j = 4 * nv + threadIdx.x; j < TK; j += NT) count(j, __ldcg(a.idx + j));
        if (REG) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                all0 += __shfl_xor_sync(0xffffffffu, all0, o);
                all1 += __shfl_xor_sync(0xffffffffu, all1, o);
                pre0 += __shfl_xor_sync(0xffffffffu, pre0, o);
                pre1 += __shfl_xor_sync(0xffffffffu, pre1, o);
            }
            if (lane < EMAX) {
                const unsigned long long wa = lane < 4 ? all0 : all1, wp = lane < 4 ? pre0 : pre1;
                s_all[warp][lane] = static_cast<int>((wa >> (16 * (lane & 3))) & 0xFFFFull);
                s_pre[warp][lane] = static_cast<int>((wp >> (16 * (lane & 3))) & 0xFFFFull);
            }
        }
    }
    if (bad && blockIdx.x == 0) atomicOr(a.err, ERRBIT_INDEX);
    __syncthreads();

    // 2. per-expert totals; warp 0 scans them (and in CTA 0 writes the outputs)
    for (int e = threadIdx.x; e < EMAX; e += NT) {
        int tot = 0, pre = 0;
        if (e < E) {
#pragma unroll 8
            for (int w = 0; w < NW; ++w) {
                tot += s_all[w][e];
                pre += s_pre[w][e];
            }
        }
        s_tot[e] = tot;
        s_base[e] = pre;
    }
    __syncthreads();
    if (warp == 0) {
        constexpr int EPL = EMAX >= 32 ? EMAX / 32 : 1;  // experts per lane
        const int bm = a.bm;
        int c[EPL], m1[EPL], m2[EPL], sc = 0, s1 = 0, s2 = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int ex = EPL * lane + i;
            c[i] = ex < E && ex < EMAX ? s_tot[ex] : 0;
            m1[i] = (c[i] + bm - 1) / bm;
            m2[i] = (c[i] + 2 * bm - 1) / (2 * bm);
            sc += c[i];
            s1 += m1[i];
            s2 += m2[i];
        }
        int x = sc, x1 = s1, x2 = s2;
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
        int b = x - sc, b1 = x1 - s1, b2 = x2 - s2;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int ex = EPL * lane + i;
            if (ex < E && ex < EMAX) {
                s_base[ex] += b;
                if (blockIdx.x == 0) {
                    a.counts[ex] = c[i];
                    a.offsets[ex] = b;
                    a.mt_prefix[ex] = b1;
                    a.mt_prefix[E + 1 + ex] = b2;
                    if (ex == E - 1) {
                        a.offsets[E] = b + c[i];
                        a.mt_prefix[E] = b1 + m1[i];
                        a.mt_prefix[2 * E + 1] = b2 + m2[i];
                    }
                }
            }
            b += c[i];
            b1 += m1[i];
            b2 += m2[i];
        }
    }
    __syncthreads();

    // 3. stable ranks within the range: warp w < 8 takes assignments j0 + 32 w + lane
    {
        const bool mine = warp < 8 && 32 * warp < per_cta;
        const int j = j0 + 32 * warp + lane;
        int e = (mine && j < j1) ? __ldcg(a.idx + j) : -1;
        if (e < 0 || e >= E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) s_rank[warp][e] = __popc(peers);
        __syncthreads();
        if (mine && j < j1) {
            int pos = -1;
            if (e >= 0) {
                pos = s_base[e] + rank;
                for (int w = 0; w < warp; ++w) pos += s_rank[w][e];
                a.sorted_token[pos] = j / a.K;
                a.sorted_w[pos] = __ldcg(a.w + j);
                a.inv[j] = pos;
            }
            s_pos[j - j0] = pos;
            s_tok[j - j0] = j / a.K;
        }
    }
    __syncthreads();

    // 4. the range's rows: RB rows of a warp in flight, 4 vectors per lane each
    const int n = j1 - j0;
    for (int r0 = RB * warp; r0 < n; r0 += RB * NW) {
        for (int v0 = lane; v0 < vpr; v0 += 128) {
            uint4 buf[RB][4];
#pragma unroll
            for (int q = 0; q < RB; ++q) {
                const int r = r0 + q;
                if (r < n && s_pos[r] >= 0) {
                    const size_t so = static_cast<size_t>(s_tok[r]) * vpr;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (v0 + 32 * i < vpr) buf[q][i] = __ldg(src + so + v0 + 32 * i);
                }
            }
#pragma unroll
            for (int q = 0; q < RB; ++q) {
                const int r = r0 + q;
                if (r < n && s_pos[r] >= 0) {
                    const size_t d = static_cast<size_t>(s_pos[r]) * vpr;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (v0 + 32 * i < vpr) dst[d + v0 + 32 * i] = buf[q][i];
                }
            }
        }
    }
}

// One warp per destination row; 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src,
                                                          const int32_t* __restrict__ rowidx,
                                                          int rows, int vec_per_row,
                                                          uint4* __restrict__ dst) {
    pdl_wait();
    pdl_trigger();
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (r >= rows) return;
    const int lane = threadIdx.x & 31;
    const size_t s = static_cast<size_t>(rowidx[r]) * vec_per_row;
    const size_t d = static_cast<size_t>(r) * vec_per_row;
    // 4 loads per lane in flight before their stores
    for (int v0 = lane; v0 < vec_per_row; v0 += 128) {
        uint4 buf[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (v0 + 32 * i < vec_per_row) buf[i] = __ldg(src + s + v0 + 32 * i);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (v0 + 32 * i < vec_per_row) dst[d + v0 + 32 * i] = buf[i];
    }
}

// K5 - combine: out[t, c] = sum_k ys[inv[t, k], c] (+ addend[t, c]) in FP32, k in
// ascending slot order, the addend last; one warp per token, 8 columns per
// lane step. A fixed order and no atomics, so the result is deterministic
// (APEX-1 Mathematical Reference Part 3 section 13.2: shared output plus the
// gate-weighted routed outputs; kimi_k3 StableLatentMoE's index_add_ scatter
// written as a gather through the inverse permutation).
template <bool OUT_BF16, int KMAX, int NB>
__global__ void __launch_bounds__(256) gather_sum_kernel(const float* __restrict__ ys,
                                                         const int32_t* __restrict__ inv, int T,
                                                         int K, int cols,
                                                         const float* __restrict__ addend,
                                                         void* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    int pos[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) pos[k] = (k < K) ? inv[static_cast<size_t>(t) * K + k] : 0;
    // NB column blocks of 256 per batch, every load of the batch issued before the sums
    // column batches; few tokens: the batches of a token spread over gridDim.y CTAs
    for (int cb = blockIdx.y * 256 * NB; cb < cols; cb += gridDim.y * 256 * NB) {
        float4 y[NB][KMAX][2];
        float4 ad[NB][2];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int c0 = cb + 256 * b + lane * 8;
            if (c0 < cols) {
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    if (k < K) {
                        const float* p = ys + static_cast<size_t>(pos[k]) * cols + c0;
                        y[b][k][0] = __ldg(reinterpret_cast<const float4*>(p));
                        y[b][k][1] = __ldg(reinterpret_cast<const float4*>(p + 4));
                    }
                }
                if (addend != nullptr) {
                    const float* p = addend + static_cast<size_t>(t) * cols + c0;
                    ad[b][0] = __ldg(reinterpret_cast<const float4*>(p));
                    ad[b][1] = __ldg(reinterpret_cast<const float4*>(p + 4));
                }
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int c0 = cb + 256 * b + lane * 8;
            if (c0 >= cols) continue;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
                if (k < K) {
                    acc[0] += y[b][k][0].x; acc[1] += y[b][k][0].y; acc[2] += y[b][k][0].z; acc[3] += y[b][k][0].w;
                    acc[4] += y[b][k][1].x; acc[5] += y[b][k][1].y; acc[6] += y[b][k][1].z; acc[7] += y[b][k][1].w;
                }
            }
            if (addend != nullptr) {
                acc[0] += ad[b][0].x; acc[1] += ad[b][0].y; acc[2] += ad[b][0].z; acc[3] += ad[b][0].w;
                acc[4] += ad[b][1].x; acc[5] += ad[b][1].y; acc[6] += ad[b][1].z; acc[7] += ad[b][1].w;
            }
            const size_t o = static_cast<size_t>(t) * cols + c0;
            if (OUT_BF16) {
                uint4 v;
                v.x = pack_bf16x2(acc[0], acc[1]);
                v.y = pack_bf16x2(acc[2], acc[3]);
                v.z = pack_bf16x2(acc[4], acc[5]);
                v.w = pack_bf16x2(acc[6], acc[7]);
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + o) = v;
            } else {
                float* q = static_cast<float*>(out) + o;
                *reinterpret_cast<float4*>(q) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4*>(q + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
        }
    }
}

// The combine with the routed rows in the 24-bit blocked layout (ys24): one
// warp per (token, 256-column block), a lane's 8 columns being 16 bytes of
// high parts and 8 of low parts in each routed row. Every row's raw parts are
// loaded before the first is converted, and they are summed as they are put
// back (exactly), in the same order as the FP32 combine.
template <bool OUT_BF16, int KMAX>
__global__ void __launch_bounds__(256) gather_sum_f24_kernel(const uint8_t* __restrict__ ys24,
                                                             const int32_t* __restrict__ inv, int T,
                                                             int K, int cols,
                                                             const float* __restrict__ addend,
                                                             void* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    int pos[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) pos[k] = (k < K) ? inv[static_cast<size_t>(t) * K + k] : 0;
    const size_t pitch = static_cast<size_t>(cols) * 3;
    for (int cb = blockIdx.y * YS24_BLOCK; cb < cols; cb += gridDim.y * YS24_BLOCK) {
        const int c0 = cb + lane * 8;
        const size_t boff = static_cast<size_t>(cb / YS24_BLOCK) * (3 * YS24_BLOCK);
        uint4 h[KMAX];
        uint2 l[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            if (k < K) {
                const uint8_t* blk = ys24 + static_cast<size_t>(pos[k]) * pitch + boff;
                h[k] = __ldg(reinterpret_cast<const uint4*>(blk + 16 * lane));
                l[k] = __ldg(reinterpret_cast<const uint2*>(blk + 2 * YS24_BLOCK + 8 * lane));
            }
        }
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
        if (addend != nullptr) {
            const float* p = addend + static_cast<size_t>(t) * cols + c0;
            a0 = __ldg(reinterpret_cast<const float4*>(p));
            a1 = __ldg(reinterpret_cast<const float4*>(p + 4));
        }
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            if (k < K) {
                acc[0] += f24_to_f32(h[k].x & 0xFFFFu, l[k].x & 0xFFu);
                acc[1] += f24_to_f32(h[k].x >> 16, (l[k].x >> 8) & 0xFFu);
                acc[2] += f24_to_f32(h[k].y & 0xFFFFu, (l[k].x >> 16) & 0xFFu);
                acc[3] += f24_to_f32(h[k].y >> 16, l[k].x >> 24);
                acc[4] += f24_to_f32(h[k].z & 0xFFFFu, l[k].y & 0xFFu);
                acc[5] += f24_to_f32(h[k].z >> 16, (l[k].y >> 8) & 0xFFu);
                acc[6] += f24_to_f32(h[k].w & 0xFFFFu, (l[k].y >> 16) & 0xFFu);
                acc[7] += f24_to_f32(h[k].w >> 16, l[k].y >> 24);
            }
        }
        if (addend != nullptr) {
            acc[0] += a0.x; acc[1] += a0.y; acc[2] += a0.z; acc[3] += a0.w;
            acc[4] += a1.x; acc[5] += a1.y; acc[6] += a1.z; acc[7] += a1.w;
        }
        const size_t o = static_cast<size_t>(t) * cols + c0;
        if (OUT_BF16) {
            uint4 v;
            v.x = pack_bf16x2(acc[0], acc[1]);
            v.y = pack_bf16x2(acc[2], acc[3]);
            v.z = pack_bf16x2(acc[4], acc[5]);
            v.w = pack_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + o) = v;
        } else {
            float* q = static_cast<float*>(out) + o;
            *reinterpret_cast<float4*>(q) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4*>(q + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
}

// gather_sum stored as a BF16 hi/lo pair (see launch_gather_sum_split).
__global__ void __launch_bounds__(256) gather_sum_split_kernel(const float* __restrict__ ys,
                                                               const int32_t* __restrict__ inv,
                                                               int T, int K, int cols, int cols_pad,
                                                               __nv_bfloat16* __restrict__ out2) {
    pdl_wait();
    pdl_trigger();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    __nv_bfloat16* hi = out2 + static_cast<size_t>(t) * 2 * cols_pad;
    __nv_bfloat16* lo = hi + cols_pad;
    for (int c0 = lane * 8; c0 < cols; c0 += 32 * 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < K; ++k) {
            const float* p = ys + static_cast<size_t>(inv[static_cast<size_t>(t) * K + k]) * cols + c0;
            const float4 a = __ldg(reinterpret_cast<const float4*>(p));
            const float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        uint32_t h[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            h[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
            l[i] = pack_bf16x2(acc[2 * i] - bf16_lo(h[i]), acc[2 * i + 1] - bf16_hi(h[i]));
        }
        *reinterpret_cast<uint4*>(hi + c0) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(lo + c0) = make_uint4(l[0], l[1], l[2], l[3]);
    }
    const __nv_bfloat16 z = __float2bfloat16_rn(0.0f);
    for (int c = cols + lane; c < cols_pad; c += 32) {
        hi[c] = z;
        lo[c] = z;
    }
}

}  // namespace

cudaError_t launch_gather_sum_split(const float* ys, const int32_t* inv, int T, int K, int cols,
                                    int cols_pad, void* out2, cudaStream_t s) {
    const int blocks = (T * 32 + 255) / 256;
    return launch_pdl(gather_sum_split_kernel, dim3(blocks), dim3(256), 0, s, ys, inv, T, K, cols,
                      cols_pad, static_cast<__nv_bfloat16*>(out2));
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s, int* n_launched) {
    const int TK = a.T * a.K;
    if (a.nchunks == 1) {
        if (n_launched) *n_launched = 1;
        return launch_pdl(dispatch_single_kernel, dim3(1), dim3(DISPATCH_CHUNK), 0, s, a.idx, a.w,
                          TK, a.K, a.E, a.bm, a.counts, a.offsets, a.mt_prefix, a.sorted_token,
                          a.sorted_w, a.inv, a.err);
    }
    cudaError_t e = launch_pdl(dispatch_count_kernel, dim3(a.nchunks), dim3(256), 0, s, a.idx, TK,
                               a.E, a.nchunks, a.bm, a.chunk_counts, a.chunk_base, a.counts,
                               a.offsets, a.mt_prefix, a.ticket, a.err);
    if (e != cudaSuccess) return e;
    e = launch_pdl(dispatch_scatter_kernel, dim3(a.nchunks), dim3(DISPATCH_CHUNK), 0, s, a.idx, a.w,
                   TK, a.K, a.E, a.chunk_base, a.sorted_token, a.sorted_w, a.inv);
    if (n_launched) *n_launched = 2;
    return e;
}

cudaError_t launch_dispatch_gather(const DispatchArgs& a, const void* src, int row_bytes, void* dst,
                                   cudaStream_t s) {
    const int TK = a.T * a.K;
    if (TK > DISPATCH_CHUNK || a.E > 256) return cudaErrorInvalidValue;
    const int blocks = std::max(1, std::min((TK + 7) / 8, num_sms()));
    const uint4* sv = static_cast<const uint4*>(src);
    uint4* dv = static_cast<uint4*>(dst);
    const int vpr = row_bytes / 16;
    if (a.E <= 64)
        return launch_pdl(dispatch_gather_kernel<64>, dim3(blocks), dim3(256), 0, s, a, sv, vpr, dv);
    if (a.E <= 128)
        return launch_pdl(dispatch_gather_kernel<128>, dim3(blocks), dim3(256), 0, s, a, sv, vpr, dv);
    return launch_pdl(dispatch_gather_kernel<256>, dim3(blocks), dim3(256), 0, s, a, sv, vpr, dv);
}

cudaError_t launch_dispatch_gather_wide(const DispatchArgs& a, const void* src, int row_bytes,
                                        void* dst, cudaStream_t s) {
    const int TK = a.T * a.K;
    if (TK > DISPATCH_WIDE_MAX || a.E > 256 || a.E < 1 || row_bytes % 16 ||
        (reinterpret_cast<uintptr_t>(a.idx) & 15u))
        return cudaErrorInvalidValue;
    // ranges of a multiple of 32 assignments, about one CTA per SM (each CTA
    // counts every assignment, so more CTAs cost more than their rows save)
    const int want = num_sms();
    int per_cta = (TK + want - 1) / want;
    per_cta = std::min(256, std::max(32, (per_cta + 31) / 32 * 32));
    const int blocks = (TK + per_cta - 1) / per_cta;
    const uint4* sv = static_cast<const uint4*>(src);
    uint4* dv = static_cast<uint4*>(dst);
    const int vpr = row_bytes / 16;
#define MOE_DGW(EM, NT) \
    return launch_pdl(dispatch_gather_wide_kernel<EM, NT>, dim3(blocks), dim3(NT), 0, s, a, per_cta, sv, vpr, dv)
    if (a.E <= 8) MOE_DGW(8, 1024);
    if (a.E <= 64) MOE_DGW(64, 256);
    MOE_DGW(256, 256);
#undef MOE_DGW
}

cudaError_t launch_gather_rows(const void* src, const int32_t* rowidx, int rows, int row_bytes,
                               void* dst, cudaStream_t s) {
    const int vpr = row_bytes / 16;
    const int blocks = (rows * 32 + 255) / 256;
    return launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, s,
                      static_cast<const uint4*>(src), rowidx, rows, vpr, static_cast<uint4*>(dst));
}

cudaError_t launch_gather_sum_f24(const void* ys24, const int32_t* inv, int T, int K, int cols,
                                  const float* addend, void* out, int out_bf16, cudaStream_t s) {
    if (cols % YS24_BLOCK || K > 16) return cudaErrorInvalidValue;
    const int blocks = (T * 32 + 255) / 256;
    // the blocks of a token on separate CTAs when that keeps every SM busy
    const int batches = cols / YS24_BLOCK;
    const int want = (2 * num_sms() + blocks - 1) / blocks;
    const dim3 g(blocks, static_cast<unsigned>(batches < want ? batches : (want > 0 ? want : 1)));
    const uint8_t* y = static_cast<const uint8_t*>(ys24);
#define MOE_GS24(KM)                                                                                  \
    return out_bf16 ? launch_pdl(gather_sum_f24_kernel<true, KM>, g, dim3(256), 0, s, y, inv, T, K,    \
                                 cols, addend, out)                                                  \
                    : launch_pdl(gather_sum_f24_kernel<false, KM>, g, dim3(256), 0, s, y, inv, T, K,   \
                                 cols, addend, out)
    if (K <= 2) MOE_GS24(2);
    if (K <= 4) MOE_GS24(4);
    if (K <= 8) MOE_GS24(8);
    MOE_GS24(16);
#undef MOE_GS24
}

cudaError_t launch_gather_sum(const float* ys, const int32_t* inv, int T, int K, int cols,
                              const float* addend, void* out, int out_bf16, cudaStream_t s) {
    const int blocks = (T * 32 + 255) / 256;
    // about 16 float4 loads in flight per lane per batch; with few tokens the
    // column batches go to separate CTAs so that at least ~2 CTAs per SM work
    auto ysplit = [&](int nb) {
        const int batches = (cols + 256 * nb - 1) / (256 * nb);
        const int want = (2 * num_sms() + blocks - 1) / blocks;
        return dim3(blocks, static_cast<unsigned>(batches < want ? batches : (want > 0 ? want : 1)));
    };
#define MOE_GS(KM, NB)                                                                            \
    return out_bf16 ? launch_pdl(gather_sum_kernel<true, KM, NB>, ysplit(NB), dim3(256), 0, s, ys, \
                                 inv, T, K, cols, addend, out)                                   \
                    : launch_pdl(gather_sum_kernel<false, KM, NB>, ysplit(NB), dim3(256), 0, s, ys, \
                                 inv, T, K, cols, addend, out)
    // Many tokens: one 256-column batch per warp, the batches of a token on
    // separate CTAs, so that few registers keep every warp resident (NB > 1
    // holds more loads per lane in flight, for batches of few tokens).
    const int batches1 = (cols + 255) / 256;
    if (K <= 4 && static_cast<long long>(T) * batches1 >= 64LL * num_sms()) {
        const dim3 g1(blocks, static_cast<unsigned>(batches1));
        if (K <= 2)
            return out_bf16 ? launch_pdl(gather_sum_kernel<true, 2, 1>, g1, dim3(256), 0, s, ys, inv, T, K, cols, addend, out)
                            : launch_pdl(gather_sum_kernel<false, 2, 1>, g1, dim3(256), 0, s, ys, inv, T, K, cols, addend, out);
        return out_bf16 ? launch_pdl(gather_sum_kernel<true, 4, 1>, g1, dim3(256), 0, s, ys, inv, T, K, cols, addend, out)
                        : launch_pdl(gather_sum_kernel<false, 4, 1>, g1, dim3(256), 0, s, ys, inv, T, K, cols, addend, out);
    }
    if (K <= 2) MOE_GS(2, 4);
    if (K <= 4) MOE_GS(4, 2);
    if (K <= 8) MOE_GS(8, 1);
    MOE_GS(16, 1);
#undef MOE_GS
}

}  // namespace moe
