// K2 in one launch for prefill batches of 16384 < T*K <= 1024 * CTAs assignments
// (BF16 rows): the stable counting sort of the (token, slot) assignments by
// expert and the row gather, without the two-launch histogram/scatter path.
//
// What it computes is exactly what the two-launch dispatch and the row gather
// compute (kimi_k3 StableLatentMoE, "Flatten routing and recover original
// token order": a stable argsort of the flat expert ids; sorted position pos
// holds token order[pos] // K): counts, offsets, tile prefixes, sorted_token,
// sorted_w, inv, and xs[pos] = x[sorted_token[pos]].
//
// One cooperative launch, one CTA of 1024 threads per SM, CTA b owning the
// contiguous range of assignments [b n, (b + 1) n):
//   1. each thread reads one assignment's expert id; warp match gives its rank
//      among the warp's equal ids and the warp's count per expert;
//   2. the CTA's count per expert goes to its row of a global table, then its
//      tag (this launch's epoch tag, release order); every CTA waits, with a
//      time limit, until all tags carry it - no zeroed memory needed;
//   3. each CTA sums the table (its expert totals, and the counts of the CTAs
//      before it), scans the totals into offsets and tile prefixes (CTA 0
//      writes them), places its assignments (offset + earlier CTAs + earlier
//      warps + rank in warp) and copies their rows.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int DO_THREADS = 1024;
constexpr int DO_WARPS = DO_THREADS / 32;

template <int EMAX>
__global__ void __launch_bounds__(DO_THREADS, 1) dispatch_onepass_kernel(DispatchArgs a, int per_cta,
                                                                         const uint4* __restrict__ src,
                                                                         int vpr, uint4* __restrict__ dst,
                                                                         unsigned long long* __restrict__ tags,
                                                                         int* __restrict__ cnt,
                                                                         uint64_t timeout_ns) {
    constexpr int P = DO_THREADS / EMAX;  // threads summing one expert's column of the table
    __shared__ unsigned short s_w[DO_WARPS][EMAX];  // per-warp counts (at most 32)
    __shared__ int s_part[P][EMAX][2];    // partial totals and prefixes of the table's column
    __shared__ int s_base[EMAX];
    __shared__ int s_wtot[8][3];
    __shared__ int s_pos[DO_THREADS], s_tok[DO_THREADS];
    pdl_wait();
    pdl_trigger();
    // this launch's tag (every thread reads the epoch before any CTA can pass the barrier)
    unsigned long long* epoch = tags + GRID_TAG_STRIDE * GRID_EPOCH_LINE;
    const unsigned long long gid = grid_epoch_tag(epoch);
    const int b = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int TK = a.T * a.K, E = a.E;
    const int j0 = b * per_cta, j1 = min(TK, j0 + per_cta);
    for (int i = threadIdx.x; i < DO_WARPS * EMAX; i += DO_THREADS) (&s_w[0][0])[i] = 0;
    __syncthreads();

    // 1. this thread's assignment: its expert, its rank in the warp, the warp's counts
    const int j = j0 + threadIdx.x;
    int e = -1;
    if (j < j1) {
        e = __ldcg(a.idx + j);
        if (e < 0 || e >= E) {
            e = -1;
            atomicOr(a.err, ERRBIT_INDEX);
        }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) s_w[warp][e] = static_cast<unsigned short>(__popc(peers));
    __syncthreads();

    // 2. the CTA's counts, its tag, and the wait for every CTA's
    for (int x = threadIdx.x; x < EMAX; x += DO_THREADS) {
        int t = 0;
#pragma unroll 8
        for (int w = 0; w < DO_WARPS; ++w) t += s_w[w][x];
        if (x < E) cnt[static_cast<size_t>(b) * E + x] = t;
    }
    __threadfence();  // each writer orders its counts before the tag below
    __syncthreads();
    if (threadIdx.x == 0) st_release_u64(tags + GRID_TAG_STRIDE * b, gid);
    const bool okb = grid_tags_wait_cta(tags, G, gid, timeout_ns, a.err);
    grid_epoch_store(epoch, gid);  // every CTA has read the epoch by now
    if (!okb) return;

    // 3. expert totals and the counts of the CTAs before this one
    {
        const int x = threadIdx.x % EMAX, part = threadIdx.x / EMAX;
        const int i0 = part * G / P, i1 = (part + 1) * G / P;
        int tot = 0, pre = 0;
        if (x < E) {
            int i = i0;
            for (; i + 7 < i1; i += 8) {
                int c[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) c[u] = __ldcg(cnt + static_cast<size_t>(i + u) * E + x);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    tot += c[u];
                    pre += (i + u < b) ? c[u] : 0;
                }
            }
            for (; i < i1; ++i) {
                const int c = __ldcg(cnt + static_cast<size_t>(i) * E + x);
                tot += c;
                pre += i < b ? c : 0;
            }
        }
        s_part[part][x][0] = tot;
        s_part[part][x][1] = pre;
    }
    __syncthreads();
    // offsets and tile prefixes: an exclusive scan over the experts (threads < 256)
    int tot = 0, pre = 0, m1 = 0, m2 = 0, xo = 0, x1 = 0, x2 = 0;
    if (threadIdx.x < 256) {
        const int x = threadIdx.x;
        if (x < E) {
#pragma unroll
            for (int q = 0; q < P; ++q) {
                tot += s_part[q][x][0];
                pre += s_part[q][x][1];
            }
        }
        m1 = (tot + a.bm - 1) / a.bm;
        m2 = (tot + 2 * a.bm - 1) / (2 * a.bm);
        xo = tot;
        x1 = m1;
        x2 = m2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, xo, o);
            const int y1 = __shfl_up_sync(0xffffffffu, x1, o);
            const int y2 = __shfl_up_sync(0xffffffffu, x2, o);
            if (lane >= o) {
                xo += y;
                x1 += y1;
                x2 += y2;
            }
        }
        if (lane == 31) {
            s_wtot[warp][0] = xo;
            s_wtot[warp][1] = x1;
            s_wtot[warp][2] = x2;
        }
    }
    __syncthreads();
    if (threadIdx.x < 256) {
        const int x = threadIdx.x;
        for (int w = 0; w < warp; ++w) {
            xo += s_wtot[w][0];
            x1 += s_wtot[w][1];
            x2 += s_wtot[w][2];
        }
        if (x < E) {
            s_base[x] = xo - tot + pre;
            if (b == 0) {
                a.counts[x] = tot;
                a.offsets[x] = xo - tot;
                a.mt_prefix[x] = x1 - m1;
                a.mt_prefix[E + 1 + x] = x2 - m2;
                if (x == E - 1) {
                    a.offsets[E] = xo;
                    a.mt_prefix[E] = x1;
                    a.mt_prefix[2 * E + 1] = x2;
                }
            }
        }
    }
    __syncthreads();

    // positions of this CTA's assignments
    int pos = -1;
    if (e >= 0) {
        pos = s_base[e] + rank;
        for (int w = 0; w < warp; ++w) pos += s_w[w][e];
        a.sorted_token[pos] = j / a.K;
        a.sorted_w[pos] = __ldcg(a.w + j);
        a.inv[j] = pos;
    }
    s_pos[threadIdx.x] = pos;
    s_tok[threadIdx.x] = j / a.K;
    __syncthreads();

    // 4. the rows: one warp per row, four 16-byte pieces per lane in flight
    for (int r = warp; r < j1 - j0; r += DO_WARPS) {
        const int p = s_pos[r];
        if (p < 0) continue;
        const uint4* sr = src + static_cast<size_t>(s_tok[r]) * vpr;
        uint4* dr = dst + static_cast<size_t>(p) * vpr;
        for (int v0 = lane; v0 < vpr; v0 += 128) {
            uint4 buf[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (v0 + 32 * i < vpr) buf[i] = __ldg(sr + v0 + 32 * i);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (v0 + 32 * i < vpr) dr[v0 + 32 * i] = buf[i];
        }
    }
}

}  // namespace

bool dispatch_onepass_ok(int T, int K, int E) {
    const long long TK = static_cast<long long>(T) * K;
    const int G = num_sms() < DISPATCH_ONEPASS_MAX_CTAS ? num_sms() : DISPATCH_ONEPASS_MAX_CTAS;
    return E >= 1 && E <= 256 && TK > DISPATCH_WIDE_MAX && TK <= static_cast<long long>(G) * DO_THREADS;
}

cudaError_t launch_dispatch_gather_onepass(const DispatchArgs& a, const void* src, int row_bytes, void* dst,
                                           unsigned long long* tags, int* cnt, cudaStream_t s) {
    if (!dispatch_onepass_ok(a.T, a.K, a.E) || row_bytes % 16) return cudaErrorInvalidValue;
    const int TK = a.T * a.K;
    const int G0 = num_sms() < DISPATCH_ONEPASS_MAX_CTAS ? num_sms() : DISPATCH_ONEPASS_MAX_CTAS;
    const int per_cta = (TK + G0 - 1) / G0;
    const int G = (TK + per_cta - 1) / per_cta;
    const uint4* sv = static_cast<const uint4*>(src);
    uint4* dv = static_cast<uint4*>(dst);
    const int vpr = row_bytes / 16;
    const uint64_t tmo = wait_timeout_ns();
    if (a.E <= 64)
        return launch_pdl_coop(dispatch_onepass_kernel<64>, dim3(G), dim3(DO_THREADS), 0, s, a, per_cta, sv, vpr,
                               dv, tags, cnt, tmo);
    if (a.E <= 128)
        return launch_pdl_coop(dispatch_onepass_kernel<128>, dim3(G), dim3(DO_THREADS), 0, s, a, per_cta, sv,
                               vpr, dv, tags, cnt, tmo);
    return launch_pdl_coop(dispatch_onepass_kernel<256>, dim3(G), dim3(DO_THREADS), 0, s, a, per_cta, sv, vpr,
                           dv, tags, cnt, tmo);
}

}  // namespace moe
