// The whole dispatch of at most DISPATCH_CHUNK (1024) assignments in one CTA,
// shared by the single-CTA dispatch kernel and the decode dispatch + gather.
//
// Source: kimi_k3 StableLatentMoE, "Flatten routing and recover original
// token order": a stable argsort of the flat expert ids; the sorted
// assignment at position pos belongs to token order[pos] // K, bincount gives
// the expert loads and their cumulative sums the expert slices.
//
// Here: the flat assignments j = 0 .. TK-1 fall into 32 groups of 32
// consecutive j ("virtual warps"; a CTA of NT threads takes them in
// 1024 / NT rounds). Each group ranks its assignments stably with a warp
// match, the per-expert counts of the groups are prefix-summed in group
// order, and one warp scans the expert totals (and the tile counts of both
// GEMM tile heights). Integer arithmetic only: the result is bit-exact and
// does not depend on NT.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// Scratch of dispatch_block_impl: NG x EMAX per-group counts (then their
// prefixes: at most DISPATCH_CHUNK, so 16 bits hold them) and EMAX offsets.
template <int EMAX>
struct DispatchScratch {
    unsigned short wcnt[DISPATCH_CHUNK / 32][EMAX];
    int off[EMAX];
};
static_assert(DISPATCH_CHUNK < 65536, "per-group prefixes in 16 bits");

// idx and w are read through L2. EMAX: a multiple of 32 that is at least E.
// The calling threads are tid = 0 .. NT-1 (whole warps, tid 0 starting a warp)
// of a group that sync() synchronises; sc is their shared scratch.
// write_out: write counts, offsets, mt_prefix, sorted_token, sorted_w and inv;
// tok_local / w_local / inv_local (optional): get sorted_token, sorted_w and
// inv too (e.g. in shared memory), and off_local the E + 1 offsets.
template <int NT, int EMAX, typename Sync>
MOE_DEV void dispatch_block_impl(int tid, Sync sync, DispatchScratch<EMAX>& sc, const int32_t* idx,
                                 const float* w, int TK, int K, int E, int bm, bool write_out,
                                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                 int32_t* __restrict__ mt_prefix, int32_t* __restrict__ sorted_token,
                                 float* __restrict__ sorted_w, int32_t* __restrict__ inv, int* err,
                                 int32_t* tok_local, float* w_local = nullptr,
                                 int32_t* inv_local = nullptr, int32_t* off_local = nullptr) {
    constexpr int ROUNDS = DISPATCH_CHUNK / NT;
    constexpr int NG = DISPATCH_CHUNK / 32;  // groups of 32 consecutive assignments
    constexpr int EPL = EMAX / 32;           // experts per lane in the scan
    static_assert(NT * ROUNDS == DISPATCH_CHUNK && EMAX % 32 == 0, "dispatch_block shape");
    auto& wcnt = sc.wcnt;
    auto& off = sc.off;
    const int warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < NG * EMAX; i += NT) (&wcnt[0][0])[i] = 0;
    // all of the thread's ids and weights in flight at once
    int ev[ROUNDS];
    float wv[ROUNDS];
#pragma unroll
    for (int q = 0; q < ROUNDS; ++q) {
        const int j = q * NT + tid;
        ev[q] = (j < TK) ? __ldcg(idx + j) : -1;
        wv[q] = (j < TK) ? __ldcg(w + j) : 0.0f;
    }
    sync();
    int rk[ROUNDS];
#pragma unroll
    for (int q = 0; q < ROUNDS; ++q) {
        const int j = q * NT + tid;
        int e = ev[q];
        if (j < TK && (e < 0 || e >= E)) atomicOr(err, ERRBIT_INDEX);
        if (e < 0 || e >= E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        rk[q] = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rk[q] == 0) wcnt[q * (NT / 32) + warp][e] = __popc(peers);
        ev[q] = e;
    }
    sync();
    // per-group exclusive prefixes and the expert totals
    for (int x = tid; x < EMAX; x += NT) {
        int run = 0;
        for (int g = 0; g < NG; ++g) {
            const int c = wcnt[g][x];
            wcnt[g][x] = run;
            run += c;
        }
        off[x] = x < E ? run : 0;
    }
    sync();
    if (warp == 0) {
        // exclusive scan of the totals (and of the tile counts of both heights)
        int c[EPL], m1[EPL], m2[EPL], s = 0, s1 = 0, s2 = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            c[i] = off[EPL * lane + i];
            m1[i] = (c[i] + bm - 1) / bm;
            m2[i] = (c[i] + 2 * bm - 1) / (2 * bm);
            s += c[i];
            s1 += m1[i];
            s2 += m2[i];
        }
        int x = s, x1 = s1, x2 = s2;
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
        int b = x - s, b1 = x1 - s1, b2 = x2 - s2;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int ex = EPL * lane + i;
            if (write_out && ex < E) {
                counts[ex] = c[i];
                offsets[ex] = b;
                mt_prefix[ex] = b1;
                mt_prefix[E + 1 + ex] = b2;
            }
            if (off_local != nullptr && ex < E) off_local[ex] = b;
            if (off_local != nullptr && ex == E - 1) off_local[E] = b + c[i];
            if (write_out && ex == E - 1) {
                offsets[E] = b + c[i];
                mt_prefix[E] = b1 + m1[i];
                mt_prefix[2 * E + 1] = b2 + m2[i];
            }
            off[ex] = b;
            b += c[i];
            b1 += m1[i];
            b2 += m2[i];
        }
    }
    sync();
#pragma unroll
    for (int q = 0; q < ROUNDS; ++q) {
        const int e = ev[q];
        if (e >= 0) {
            const int j = q * NT + tid;
            const int pos = off[e] + wcnt[q * (NT / 32) + warp][e] + rk[q];
            if (tok_local != nullptr) tok_local[pos] = j / K;
            if (w_local != nullptr) w_local[pos] = wv[q];
            if (inv_local != nullptr) inv_local[j] = pos;
            if (write_out) {
                sorted_token[pos] = j / K;
                sorted_w[pos] = wv[q];
                inv[j] = pos;
            }
        }
    }
}


// The whole CTA (NT threads) with its own static scratch.
template <int NT, int EMAX>
MOE_DEV void dispatch_block(const int32_t* idx, const float* w, int TK, int K, int E, int bm,
                            bool write_out, int32_t* __restrict__ counts,
                            int32_t* __restrict__ offsets, int32_t* __restrict__ mt_prefix,
                            int32_t* __restrict__ sorted_token, float* __restrict__ sorted_w,
                            int32_t* __restrict__ inv, int* err, int32_t* tok_local = nullptr) {
    __shared__ DispatchScratch<EMAX> sc;
    dispatch_block_impl<NT, EMAX>(static_cast<int>(threadIdx.x), [] { __syncthreads(); }, sc, idx, w, TK,
                                  K, E, bm, write_out, counts, offsets, mt_prefix, sorted_token,
                                  sorted_w, inv, err, tok_local);
}

}  // namespace
}  // namespace moe
