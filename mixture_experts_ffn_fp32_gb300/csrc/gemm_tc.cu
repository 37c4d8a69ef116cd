// K3/K4/K7 - grouped GEMM over ragged expert segments on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), operands fed by TMA.
//
// What it computes (APEX-1 Mathematical Reference Part 3, section 12.2,
// FFN(x) = W_down(SiLU(x W_gate) (.) x W_up), applied per expert to the rows
// the dispatch grouped for it, as in kimi_k3 StableLatentMoE "The actual
// grouped GEMM, and the gradient path"):
//   SwiGLU kernel : h[r, :]  = SiLU(A[r, :] W_gate[z]) * (A[r, :] W_up[z])
//   its backward  : from a = A W_gate[z], u = A W_up[z] and the upstream dh:
//                   da = g dh u SiLU'(a), du = g dh SiLU(a), g h (backward pass)
//   plain kernel  : y[r, :]  = rowscale[r] * (A[r, :] B[z])   (routed down x gate weight)
//                   y[t, :]  = A[t, :] B (+ addend[t, :])       (shared down, projections)
// Two segment groups share one persistent launch, each with its own
// reduction length: group 0 = the E routed experts over the expert-sorted
// rows (segment bounds read from device memory, never from the host),
// group 1 = S dense segments over all token rows (the shared experts, or a
// single dense projection).
//
// Tile: 128 rows x 256 accumulator columns per CTA (SwiGLU: 128 gate + 128
// up columns of the same output tile), K step 64 (one 128-byte swizzle row),
// a ring of TMA stages, two 256-column TMEM accumulators so the epilogue of
// one tile overlaps the main loop of the next. Warp 0 issues TMA, warp 1
// issues tcgen05.mma (BF16 in, FP32 accumulate), warps 2-9 drain TMEM (two
// warps per 32-lane quarter, each taking half of the columns), apply the
// epilogue and store. The weights stay in the caller's [Z, K, N] layout (N
// contiguous) and are read as an MN-major operand.
//
// Two forms. CTA pair (MMA N = 128 or 256; for routed segments of 512 rows on
// average or more, and for dense groups): a cluster of two
// CTAs on neighbouring SMs computes a 256-row tile with cta_group::2 MMAs
// (M = 256) issued by the even CTA; each CTA loads its own 128 rows of A and
// one half of B's columns, so every SM brings in 32 KB per K step instead of
// 48 KB for the same tensor work. Both CTAs' copies complete on the even
// CTA's stage barrier; the MMA commits arrive on both CTAs' barriers. A pair
// stage holds two k-blocks, as handing a stage over between the two SMs
// costs more than within one. Single CTA: M = 128 (any MMA N).
//
// Every wait is bounded (see common.cuh): on timeout the CTA stops, drains
// its copies and MMAs, frees TMEM and flags the error word.
#include <cstdlib>

#include "common.cuh"
#include "internal.h"
#include "warp_stage.cuh"

namespace moe {
namespace {

constexpr int BM = TC_BM;          // rows per CTA
constexpr int BK = 64;             // one k-block: a 128-byte swizzle row of BF16
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int STRIP_BYTES = BK * 64 * 2;    // 8 KB: 64 k rows x 64 columns
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int MAXE = 256;
constexpr int STG_BYTES = 32 * 64;  // per epilogue warp: 32 rows x 64 bytes

// Shared-memory plan: a 192 KB ring of stages, barriers, the segment tables
// and the epilogue staging buffers. Single CTA: 4 stages of one k-block (16 KB
// A + 32 KB B). Pair: 3 stages of two k-blocks (2 x (16 KB A + 16 KB B half)):
// a pair stage costs more to hand over than a single one, so it carries more.
template <bool PAIR>
struct Geo {
    static constexpr int STAGES = PAIR ? 3 : 4;
    static constexpr int KPS = PAIR ? 2 : 1;  // k-blocks per stage
    static constexpr int SUB_BYTES = A_BYTES + (PAIR ? 2 : 4) * STRIP_BYTES;
    static constexpr int STAGE_BYTES = KPS * SUB_BYTES;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int NBARS = 2 * STAGES + 4 + 1;
    static constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;
    static constexpr int SCHED_OFF = ((MISC_OFF + 16) + 15) / 16 * 16;
    static constexpr int STG_OFF = (SCHED_OFF + 2 * (MAXE + 1) * 4 + 127) / 128 * 128;
    static constexpr int SMEM_BYTES = STG_OFF + EPI_WARPS * STG_BYTES + 1024;
};

struct TcParams {
    CUtensorMap mapA[2];
    CUtensorMap mapB0[2];
    CUtensorMap mapB1[2];
    int enabled[2];
    int rows[2];
    int N[2];
    int nt[2];
    int Z[2];
    void* out[2];
    int out_ld[2];
    int out_f32[2];
    int kblocks[2];
    int a_kmod[2], b_kmod[2], a_kgroup[2], a_krep[2];
    int b_wide[2];       // B maps are 4-D strip maps: one copy fetches all strips a CTA needs
    int nstrip;          // plain kernel: 64-column B strips per tile (MMA N = 64 * nstrip)
    int bno;             // output columns per tile
    uint32_t idesc;      // instruction descriptor (M = 128 or 256, N = 64 * nstrip)
    int ksplit1, kbs1;   // group 1 split-K: slices and k-blocks per slice
    int kchunk1;         // TC_PLAIN_ACC: k-blocks per tensor-memory chunk
    // group 1, single-CTA plain: a second reduction segment (TcGroup::A2/B2)
    // from k-block kseg2 on (0: none)
    CUtensorMap mapA2, mapB2;
    int kseg2, b2_wide;
    int E, mt1;
    const int32_t* offsets;
    const int32_t* mt_prefix;  // group 0 tiles of this kernel's rows (128, pair 256) per segment
    const float* rowscale0;
    const float* addend;
    int add_ld;
    // TC_SWIGLU: also the gate and up products, BF16 in out's layout (TcGroup)
    __nv_bfloat16* a_out[2];
    __nv_bfloat16* u_out[2];
    // TC_SWIGLU_BWD (see TcGroup)
    const float* dh[2];
    int dh_ld[2];
    __nv_bfloat16* da[2];
    __nv_bfloat16* du[2];
    __nv_bfloat16* hw[2];
    float* dgpart;
    const int32_t* poff;
    int* err;
    unsigned long long timeout_ns;
};

// One work unit: `rows` (> 0) rows from row0 (at most 128; pair: 256, the
// even CTA the first 128) by one tile of output columns, reduction k-blocks
// [kb0, kb1).
struct Unit {
    int g, row0, rows, zb, n0, out_row0, out_col0, kb0, kb1;
};

// Group 0 units tile each expert's segment (mt_prefix counts the tiles),
// group 1 units the dense rows; tiles of 128 rows, or 256 for a pair.
template <bool PAIR>
MOE_DEV Unit decode_unit(int u, const TcParams& p, int total0, const int* s_mtp, const int* s_off) {
    constexpr int UROWS = PAIR ? 2 * BM : BM;
    const int BNO = p.bno;
    Unit t;
    if (u < total0) {
        // An expert's units are consecutive. Single CTA: its row tiles innermost,
        // so the units reading one weight strip (one column tile) are neighbours,
        // and the CTAs that take them (neighbours too) read the strip at about the
        // same time: all but the first find it in L2 (large prefill: 23 % -> 7.5 %
        // weight re-reads). Pair: its column tiles innermost (measured faster
        // there: segments of many row tiles keep their weights in L2 anyway).
        const int nt = p.nt[0];
        const int mt = u / nt;
        int lo = 0, hi = p.E;  // s_mtp[lo] <= mt < s_mtp[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_mtp[mid] <= mt)
                lo = mid;
            else
                hi = mid;
        }
        int n, m;
        if (PAIR) {
            n = u - mt * nt;
            m = mt - s_mtp[lo];
        } else {
            const int me = s_mtp[lo + 1] - s_mtp[lo];  // row tiles of expert lo (>= 1)
            const int l = u - s_mtp[lo] * nt;
            n = l / me;
            m = l - n * me;
        }
        t.g = 0;
        t.row0 = s_off[lo] + m * UROWS;
        t.rows = min(UROWS, s_off[lo + 1] - t.row0);
        t.zb = lo;
        t.n0 = n * BNO;
        t.out_row0 = t.row0;
        t.out_col0 = t.n0;
        t.kb0 = 0;
        t.kb1 = p.kblocks[0];
    } else {
        const int u1 = u - total0;
        const int nt = p.nt[1];
        const int nseg = p.ksplit1 > 1 ? p.ksplit1 : p.Z[1];
        const int per_m = nseg * nt;
        const int m = u1 / per_m;
        const int rem = u1 - m * per_m;
        const int s = rem / nt;
        const int n = rem - s * nt;
        t.g = 1;
        t.row0 = m * UROWS;
        t.rows = min(UROWS, p.rows[1] - t.row0);
        t.n0 = n * BNO;
        if (p.ksplit1 > 1) {
            t.zb = 0;
            t.kb0 = s * p.kbs1;
            t.kb1 = min(t.kb0 + p.kbs1, p.kblocks[1]);
            t.out_row0 = s * p.rows[1] + t.row0;
            t.out_col0 = t.n0;
        } else {
            t.zb = s;
            t.kb0 = 0;
            t.kb1 = p.kblocks[1];
            t.out_row0 = t.row0;
            t.out_col0 = s * p.N[1] + t.n0;
        }
    }
    return t;
}

// The copies one CTA makes for unit t, prepared once per unit: for each
// k-block, its A rows and its B strips into sA / sB, completing on `bar`
// (pair: the even CTA's barrier, a shared::cluster address).
template <bool SWIGLU, bool PAIR>
struct UnitCopies {
    const CUtensorMap* mA;
    const CUtensorMap* mB0;   // pair: this CTA's B (SwiGLU: gate for the even CTA, up for the odd)
    const CUtensorMap* mB1;
    int akm, bkm, akg, akr;   // k-block remaps (0: none)
    int arow, nb, zb, bstrips;
    bool loadA, wide;
    const CUtensorMap* mA2;   // second reduction segment (group 1, single-CTA plain): from k-block kbs2
    const CUtensorMap* mB2;
    int kbs2;
    bool wide2;

    MOE_DEV UnitCopies(const TcParams& p, const Unit& t, int rank, int bstrips_) {
        mA2 = &p.mapA2;
        mB2 = &p.mapB2;
        kbs2 = (t.g == 1 && p.kseg2 > 0) ? p.kseg2 : 0x7fffffff;
        wide2 = p.b2_wide != 0;
        mA = &p.mapA[t.g];
        mB0 = (PAIR && SWIGLU && rank) ? &p.mapB1[t.g] : &p.mapB0[t.g];
        mB1 = &p.mapB1[t.g];
        akm = p.a_kmod[t.g];
        bkm = p.b_kmod[t.g];
        akg = p.a_kgroup[t.g];
        akr = p.a_krep[t.g];
        arow = t.row0 + rank * BM;
        loadA = t.rows > rank * BM;  // pair: the odd CTA of a short unit has no rows
        bstrips = bstrips_;
        // pair, plain: each CTA one half of the tile's strips
        nb = (PAIR && !SWIGLU) ? t.n0 + 64 * bstrips * rank : t.n0;
        zb = t.zb;
        wide = p.b_wide[t.g] != 0;
    }

    MOE_DEV void issue(int kb, uint32_t sA, uint32_t sB, uint32_t bar) const {
        if (!PAIR && !SWIGLU && kb >= kbs2) {
            // second segment: A2 [rows, K2] against B2 [1, K2, N], no remaps
            const int kc2 = (kb - kbs2) * BK;
            tma_load_2d(sA, mA2, kc2, arow, bar);
            if (wide2) {
                tma_load_4d(sB, mB2, 0, kc2, nb >> 6, 0, bar);
            } else {
                for (int j = 0; j < bstrips; ++j) tma_load_3d(sB + j * STRIP_BYTES, mB2, nb + 64 * j, kc2, 0, bar);
            }
            return;
        }
        const int kc = kb * BK;
        int kca = akm ? kc % akm : kc;
        if (akg) kca = ((kb / (akg * akr)) * akg + kb % akg) * BK;
        const int kcb = bkm ? kc % bkm : kc;
        if (PAIR) {
            if (loadA) tma_load_2d_pair(sA, mA, kca, arow, bar);
            if (wide) {
                tma_load_4d_pair(sB, mB0, 0, kcb, nb >> 6, zb, bar);
            } else {
                for (int j = 0; j < bstrips; ++j)
                    tma_load_3d_pair(sB + j * STRIP_BYTES, mB0, nb + 64 * j, kcb, zb, bar);
            }
        } else {
            tma_load_2d(sA, mA, kca, arow, bar);
            if (wide) {
                tma_load_4d(sB, mB0, 0, kcb, nb >> 6, zb, bar);
                if (SWIGLU) tma_load_4d(sB + 2 * STRIP_BYTES, mB1, 0, kcb, nb >> 6, zb, bar);
            } else if (SWIGLU) {
                tma_load_3d(sB, mB0, nb, kcb, zb, bar);
                tma_load_3d(sB + STRIP_BYTES, mB0, nb + 64, kcb, zb, bar);
                tma_load_3d(sB + 2 * STRIP_BYTES, mB1, nb, kcb, zb, bar);
                tma_load_3d(sB + 3 * STRIP_BYTES, mB1, nb + 64, kcb, zb, bar);
            } else {
                for (int j = 0; j < bstrips; ++j)
                    tma_load_3d(sB + j * STRIP_BYTES, mB0, nb + 64 * j, kcb, zb, bar);
            }
        }
    }
};

template <int MODE, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1) tc_grouped_gemm_kernel(const __grid_constant__ TcParams p) {
    constexpr bool SWIGLU = MODE == TC_SWIGLU || MODE == TC_SWIGLU_BWD;
    static_assert(MODE != TC_PLAIN_ACC || !PAIR, "chunk accumulation runs in the single-CTA form");
    using G = Geo<PAIR>;
    constexpr int STAGES = G::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + G::BAR_OFF;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::MISC_OFF + 4);
    int* s_mtp = reinterpret_cast<int*>(smem + G::SCHED_OFF);
    int* s_off = s_mtp + (MAXE + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // pair: rank 0 issues the MMAs; work is distributed per cluster
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int ustep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), PAIR ? 2 * EPI_WARPS : EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int g = 0; g < 2; ++g) {
            if (!p.enabled[g]) continue;
            tma_prefetch_map(&p.mapA[g]);
            tma_prefetch_map(&p.mapB0[g]);
            if (SWIGLU) tma_prefetch_map(&p.mapB1[g]);
        }
        if (p.kseg2 > 0) {
            tma_prefetch_map(&p.mapA2);
            tma_prefetch_map(&p.mapB2);
        }
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish();
        }
    }
    // everything above overlaps the previous kernel; its outputs are read below
    pdl_wait();
    pdl_trigger();
    if (p.enabled[0]) {
        for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
            s_mtp[i] = p.mt_prefix[i];
            s_off[i] = p.offsets[i];
        }
    }
    __syncwarp();
    tc_fence_before();
    if (PAIR)
        cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total0 = p.enabled[0] ? s_mtp[p.E] * p.nt[0] : 0;
    const int total =
        total0 + (p.enabled[1] ? p.mt1 * (p.ksplit1 > 1 ? p.ksplit1 : p.Z[1]) * p.nt[1] : 0);
    const WaitCtx wc{p.err, abort_flag, p.timeout_ns};
    const int nstrip = SWIGLU ? 4 : p.nstrip;
    const int bstrips = PAIR ? (SWIGLU ? 2 : nstrip / 2) : nstrip;  // strips this CTA loads

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int u = unit0; u < total && ok; u += ustep) {
                const Unit t = decode_unit<PAIR>(u, p, total0, s_mtp, s_off);
                const UnitCopies<SWIGLU, PAIR> cp(p, t, rank, bstrips);
                // pair: the even CTA's barrier counts both CTAs' bytes
                const uint32_t own = (cp.loadA ? A_BYTES : 0) + bstrips * STRIP_BYTES;
                const uint32_t peer = (t.rows > BM ? A_BYTES : 0) + bstrips * STRIP_BYTES;
                const uint32_t sub_bytes = PAIR ? own + peer : own;
                for (int kb = t.kb0; kb < t.kb1; kb += G::KPS) {
                    const int nk = min(G::KPS, t.kb1 - kb);
                    if (!bounded_wait(empty_bar(stage), phase ^ 1u, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sS = sbase + stage * G::STAGE_BYTES;
                    const uint32_t fb = PAIR ? map_shared_rank(full_bar(stage), 0) : full_bar(stage);
                    if (rank == 0) mbar_expect_tx(full_bar(stage), nk * sub_bytes);
                    for (int j = 0; j < nk; ++j) {
                        const uint32_t sA = sS + j * G::SUB_BYTES;
                        cp.issue(kb + j, sA, sA + A_BYTES, fb);
                    }
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy this thread issued has landed before the CTA can exit:
            // its stage was filled (even CTA: the barrier counts both CTAs'
            // bytes) or, in the odd CTA, consumed by the pair's MMAs
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u)
                    bounded_drain(rank == 0 ? full_bar(s) : empty_bar(s), (last_par >> s) & 1u,
                                  p.timeout_ns, p.err);
        }
    } else if (warp == 1 && PAIR && rank == 1) {
        // the odd CTA of a pair issues no MMAs
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            // Descriptors of stage 0, k-block 0, k-step 0; the others differ only in
            // the start-address field (16-byte units, no carry out of it below 256 KB).
            const uint64_t adesc0 = smem_desc_sw128(sbase, 16, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(sbase + A_BYTES, STRIP_BYTES, 1024);
            for (int u = unit0; u < total && ok; u += ustep) {
                const Unit t = decode_unit<PAIR>(u, p, total0, s_mtp, s_off);
                // one accumulator per unit; TC_PLAIN_ACC: one per chunk of kchunk1 k-blocks
                const int kstep = MODE == TC_PLAIN_ACC ? p.kchunk1 : t.kb1 - t.kb0;
                for (int cs = t.kb0; cs < t.kb1; cs += kstep) {
                    const int ce = min(cs + kstep, t.kb1);
                    if (!bounded_wait(tempty_bar(acc), acc_phase ^ 1u, wc, PAIR)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
                    for (int kb = cs; kb < ce; kb += G::KPS) {
                        const int nk = min(G::KPS, ce - kb);
                        if (!bounded_wait(full_bar(stage), phase, wc, PAIR)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t soff = static_cast<uint64_t>(stage * G::STAGE_BYTES) >> 4;
                        const uint32_t first = kb == cs ? 0u : 1u;  // 0: overwrite the accumulator
#pragma unroll
                        for (int j = 0; j < G::KPS; ++j) {
                            if (j < nk) {
#pragma unroll
                                for (int ks = 0; ks < BK / 16; ++ks) {
                                    const uint64_t ad = adesc0 + soff + (j * G::SUB_BYTES + ks * 32) / 16;
                                    const uint64_t bd = bdesc0 + soff + (j * G::SUB_BYTES + ks * 2048) / 16;
                                    const uint32_t accum = (j != 0 || ks != 0) ? 1u : first;
                                    if (PAIR)
                                        tc_mma_bf16_pair(d_tmem, ad, bd, p.idesc, accum);
                                    else
                                        tc_mma_bf16(d_tmem, ad, bd, p.idesc, accum);
                                }
                            }
                        }
                        if (PAIR)
                            tc_commit_pair_mc(empty_bar(stage), 3);
                        else
                            tc_commit(empty_bar(stage));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    if (PAIR)
                        tc_commit_pair_mc(tfull_bar(acc), 3);
                    else
                        tc_commit(tfull_bar(acc));
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                }
            }
            if (PAIR)
                tc_commit_pair(drain_bar);
            else
                tc_commit(drain_bar);
            bounded_drain(drain_bar, 0, p.timeout_ns, p.err);
        }
    } else {
        // ---------------- epilogue warps 2..9 ----------------
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;  // which half of the tile's columns
        uint4* stg = reinterpret_cast<uint4*>(smem + G::STG_OFF + (warp - 2) * STG_BYTES);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = unit0; u < total; u += ustep) {
            const Unit t = decode_unit<PAIR>(u, p, total0, s_mtp, s_off);
            if constexpr (MODE == TC_PLAIN_ACC) {
                // the unit's chunks, each from its own accumulator, summed in FP32 in
                // chunk order in this thread's registers (its row, `span` columns)
                const int span = 32 * p.nstrip;  // <= 128
                float av[128];
#pragma unroll
                for (int i = 0; i < 128; ++i) av[i] = 0.0f;
                bool okc = true;
                for (int cs = t.kb0; cs < t.kb1; cs += p.kchunk1) {
                    int okw = 1;
                    if (lane == 0) okw = bounded_wait(tfull_bar(acc), acc_phase, wc) ? 1 : 0;
                    okw = __shfl_sync(0xffffffffu, okw, 0);
                    if (!okw) {
                        okc = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * ACC_COLS) +
                                        (static_cast<uint32_t>(q * 32) << 16) +
                                        static_cast<uint32_t>(half * span);
#pragma unroll
                    for (int c = 0; c < 128; c += 32) {
                        if (c < span) {
                            uint32_t r0[16], r1[16];
                            tc_ld_32x32b_x16(tb + c, r0);
                            tc_ld_32x32b_x16(tb + c + 16, r1);
                            tc_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                av[c + i] += __uint_as_float(r0[i]);
                                av[c + 16 + i] += __uint_as_float(r1[i]);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(acc));
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                }
                if (!okc) break;
                const int valid_rows = min(BM, t.rows) - q * 32;
                if (valid_rows > 0) {
                    const int N = p.N[t.g];
                    const size_t pitch = static_cast<size_t>(p.out_ld[t.g]) * 4;
                    char* out_rows = static_cast<char*>(p.out[t.g]) +
                                     static_cast<size_t>(t.out_row0 + q * 32) * pitch;
#pragma unroll
                    for (int c = 0; c < 128; c += 16) {
                        if (c < span) {
                            const int cc = half * span + c;
                            const int lim = N - (t.n0 + cc);
                            uint4 blk[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                blk[j] = make_uint4(__float_as_uint(av[c + 4 * j]), __float_as_uint(av[c + 4 * j + 1]),
                                                    __float_as_uint(av[c + 4 * j + 2]), __float_as_uint(av[c + 4 * j + 3]));
                            const int vch = lim > 0 ? (lim >= 16 ? 4 : lim / 4) : 0;
                            warp_store_block(stg, blk, lane, out_rows + static_cast<size_t>(t.out_col0 + cc) * 4,
                                             pitch, valid_rows, vch);
                        }
                    }
                }
                continue;
            }
            int ok = 1;
            if (lane == 0) ok = bounded_wait(tfull_bar(acc), acc_phase, wc) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb =
                tmem_base + static_cast<uint32_t>(acc * ACC_COLS) + (static_cast<uint32_t>(q * 32) << 16);
            // this CTA's rows of the unit, then this warp's 32 of them
            const int my_rows = min(BM, t.rows - rank * BM);
            const int valid_rows = my_rows - q * 32;
            const int my_out0 = t.out_row0 + rank * BM;
            const size_t orow = static_cast<size_t>(my_out0 + q * 32 + lane);
            const int N = p.N[t.g];
            const int ld = p.out_ld[t.g];
            const int of32 = p.out_f32[t.g];
            const size_t es = of32 ? 4 : 2;
            const size_t pitch = static_cast<size_t>(ld) * es;
            char* out_rows = static_cast<char*>(p.out[t.g]) +
                             static_cast<size_t>(my_out0 + q * 32) * pitch;
            if (MODE == TC_SWIGLU_BWD) {
                // Output rows of this warp: group 0 in the expert-padded row layout
                // (the segment's rows, then its padding rows, written as zeros),
                // group 1 the token rows. dh is read in the same layout.
                long long rbase;
                int nrow;
                if (t.g == 0) {
                    rbase = p.poff[t.zb] + (static_cast<long long>(my_out0 + q * 32) - s_off[t.zb]);
                    const long long left = p.poff[t.zb + 1] - rbase;
                    nrow = left < 32 ? static_cast<int>(left) : 32;
                } else {
                    rbase = my_out0 + q * 32;
                    nrow = valid_rows;
                }
                const bool row_valid = lane < valid_rows;
                const long long drow = rbase + lane;
                const float g = (t.g == 0 && p.rowscale0 != nullptr && row_valid) ? p.rowscale0[orow] : 1.0f;
                const size_t bpitch = static_cast<size_t>(ld) * 2;
                char* da_rows = reinterpret_cast<char*>(p.da[t.g]) + static_cast<size_t>(rbase) * bpitch;
                char* du_rows = reinterpret_cast<char*>(p.du[t.g]) + static_cast<size_t>(rbase) * bpitch;
                char* hw_rows = reinterpret_cast<char*>(p.hw[t.g]) + static_cast<size_t>(rbase) * bpitch;
                float part = 0.0f;
#pragma unroll 1
                for (int c = half * 64; c < half * 64 + 64; c += 32) {
                    uint32_t pda[16], pdu[16], phw[16];
#pragma unroll
                    for (int hc = 0; hc < 32; hc += 16) {
                        uint32_t gv[16], uv[16];
                        tc_ld_32x32b_x16(tb + c + hc, gv);
                        tc_ld_32x32b_x16(tb + 128 + c + hc, uv);
                        tc_wait_ld();
                        const int lim = N - (t.n0 + c + hc);
                        float dh[16];
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            float4 d4 = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (row_valid && i < lim)
                                d4 = *reinterpret_cast<const float4*>(
                                    p.dh[t.g] + drow * p.dh_ld[t.g] + t.out_col0 + c + hc + i);
                            dh[i] = d4.x;
                            dh[i + 1] = d4.y;
                            dh[i + 2] = d4.z;
                            dh[i + 3] = d4.w;
                        }
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            float o_da[2], o_du[2], o_hw[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float a = __uint_as_float(gv[i + e]), uu = __uint_as_float(uv[i + e]);
                                const float sg = 1.0f / (1.0f + expf(-a));
                                const float si = a * sg;
                                const float h = si * uu;
                                const float dv = dh[i + e];
                                o_da[e] = row_valid ? g * dv * uu * (sg * (1.0f + a * (1.0f - sg))) : 0.0f;
                                o_du[e] = row_valid ? g * dv * si : 0.0f;
                                o_hw[e] = row_valid ? g * h : 0.0f;
                                part += row_valid ? dv * h : 0.0f;
                            }
                            pda[(hc + i) / 2] = pack_bf16x2(o_da[0], o_da[1]);
                            pdu[(hc + i) / 2] = pack_bf16x2(o_du[0], o_du[1]);
                            phw[(hc + i) / 2] = pack_bf16x2(o_hw[0], o_hw[1]);
                        }
                    }
                    // 32 BF16 of each row through the staging buffer, padding rows included
                    const int vch = (N - (t.n0 + c)) / 8;
                    const size_t col = static_cast<size_t>(t.out_col0 + c) * 2;
                    const uint4 va[4] = {make_uint4(pda[0], pda[1], pda[2], pda[3]), make_uint4(pda[4], pda[5], pda[6], pda[7]),
                                         make_uint4(pda[8], pda[9], pda[10], pda[11]), make_uint4(pda[12], pda[13], pda[14], pda[15])};
                    warp_store_block(stg, va, lane, da_rows + col, bpitch, nrow, vch);
                    const uint4 vu[4] = {make_uint4(pdu[0], pdu[1], pdu[2], pdu[3]), make_uint4(pdu[4], pdu[5], pdu[6], pdu[7]),
                                         make_uint4(pdu[8], pdu[9], pdu[10], pdu[11]), make_uint4(pdu[12], pdu[13], pdu[14], pdu[15])};
                    warp_store_block(stg, vu, lane, du_rows + col, bpitch, nrow, vch);
                    const uint4 vh[4] = {make_uint4(phw[0], phw[1], phw[2], phw[3]), make_uint4(phw[4], phw[5], phw[6], phw[7]),
                                         make_uint4(phw[8], phw[9], phw[10], phw[11]), make_uint4(phw[12], phw[13], phw[14], phw[15])};
                    warp_store_block(stg, vh, lane, hw_rows + col, bpitch, nrow, vch);
                }
                if (t.g == 0 && p.dgpart != nullptr && row_valid)
                    p.dgpart[orow * static_cast<size_t>(2 * p.nt[0]) + 2 * (t.n0 / 128) + half] = part;
            } else if (valid_rows <= 0) {
                // none of this warp's 32 rows exist (the odd CTA of a short pair unit)
            } else if (SWIGLU) {
                // 2 blocks of 32 BF16 columns per warp
#pragma unroll 1
                for (int c = half * 64; c < half * 64 + 64; c += 32) {
                    uint32_t g0[16], g1[16], u0[16], u1[16];
                    tc_ld_32x32b_x16(tb + c, g0);
                    tc_ld_32x32b_x16(tb + c + 16, g1);
                    tc_ld_32x32b_x16(tb + 128 + c, u0);
                    tc_ld_32x32b_x16(tb + 128 + c + 16, u1);
                    tc_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float ga = __uint_as_float(g0[2 * i]), gb = __uint_as_float(g0[2 * i + 1]);
                        pk[i] = pack_bf16x2(__fdividef(ga, 1.0f + __expf(-ga)) * __uint_as_float(u0[2 * i]),
                                            __fdividef(gb, 1.0f + __expf(-gb)) * __uint_as_float(u0[2 * i + 1]));
                        ga = __uint_as_float(g1[2 * i]);
                        gb = __uint_as_float(g1[2 * i + 1]);
                        pk[8 + i] = pack_bf16x2(__fdividef(ga, 1.0f + __expf(-ga)) * __uint_as_float(u1[2 * i]),
                                                __fdividef(gb, 1.0f + __expf(-gb)) * __uint_as_float(u1[2 * i + 1]));
                    }
                    const uint4 v[4] = {make_uint4(pk[0], pk[1], pk[2], pk[3]), make_uint4(pk[4], pk[5], pk[6], pk[7]),
                                        make_uint4(pk[8], pk[9], pk[10], pk[11]),
                                        make_uint4(pk[12], pk[13], pk[14], pk[15])};
                    const int vch = (N - (t.n0 + c)) / 8;  // valid 16-byte chunks (8 BF16 each)
                    warp_store_block(stg, v, lane, out_rows + static_cast<size_t>(t.out_col0 + c) * 2,
                                     pitch, valid_rows, vch);
                    if (p.a_out[t.g] != nullptr) {
                        // the products themselves, kept for the backward pass
                        const size_t ro = static_cast<size_t>(my_out0 + q * 32) * pitch +
                                          static_cast<size_t>(t.out_col0 + c) * 2;
                        uint32_t pa[16], pu[16];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            pa[i] = pack_bf16x2(__uint_as_float(g0[2 * i]), __uint_as_float(g0[2 * i + 1]));
                            pa[8 + i] = pack_bf16x2(__uint_as_float(g1[2 * i]), __uint_as_float(g1[2 * i + 1]));
                            pu[i] = pack_bf16x2(__uint_as_float(u0[2 * i]), __uint_as_float(u0[2 * i + 1]));
                            pu[8 + i] = pack_bf16x2(__uint_as_float(u1[2 * i]), __uint_as_float(u1[2 * i + 1]));
                        }
                        const uint4 va[4] = {make_uint4(pa[0], pa[1], pa[2], pa[3]), make_uint4(pa[4], pa[5], pa[6], pa[7]),
                                             make_uint4(pa[8], pa[9], pa[10], pa[11]),
                                             make_uint4(pa[12], pa[13], pa[14], pa[15])};
                        warp_store_block(stg, va, lane, reinterpret_cast<char*>(p.a_out[t.g]) + ro, pitch,
                                         valid_rows, vch);
                        const uint4 vu[4] = {make_uint4(pu[0], pu[1], pu[2], pu[3]), make_uint4(pu[4], pu[5], pu[6], pu[7]),
                                             make_uint4(pu[8], pu[9], pu[10], pu[11]),
                                             make_uint4(pu[12], pu[13], pu[14], pu[15])};
                        warp_store_block(stg, vu, lane, reinterpret_cast<char*>(p.u_out[t.g]) + ro, pitch,
                                         valid_rows, vch);
                    }
                }
            } else {
                float rs = 1.0f;
                if (t.g == 0 && p.rowscale0 != nullptr && lane < valid_rows) rs = p.rowscale0[orow];
                // the addend's rows of this warp, read row-major (8 rows x 64 contiguous
                // bytes per load instruction) before the accumulator is waited for, then
                // turned into the lane = row layout through the staging buffer
                const bool add = t.g == 1 && p.addend != nullptr;
                const size_t apitch = static_cast<size_t>(p.add_ld) * 4;
                const char* add_rows = add ? reinterpret_cast<const char*>(p.addend) +
                                                 static_cast<size_t>(my_out0 + q * 32) * apitch
                                           : nullptr;
                auto add_issue = [&](uint4 (&w)[4], int col) {
                    const int lim = N - (t.n0 + col);  // valid columns from col
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = 8 * i + (lane >> 2), ch = lane & 3;
                        w[i] = make_uint4(0u, 0u, 0u, 0u);
                        if (row < valid_rows && 4 * ch + 4 <= lim)
                            w[i] = *reinterpret_cast<const uint4*>(
                                add_rows + row * apitch + static_cast<size_t>(t.out_col0 + col) * 4 + ch * 16);
                    }
                };
                const int span = 32 * p.nstrip;  // this warp's columns: [half * span, +span)
                // blocks of 64 bytes per row: 16 FP32 or 32 BF16 columns
                const int bc = of32 ? 16 : 32;
#pragma unroll 1
                for (int c = half * span; c < half * span + span; c += bc) {
                    float v[32];
                    uint4 aw[4];
                    if (add) add_issue(aw, c);
                    uint32_t r0[16], r1[16];
                    tc_ld_32x32b_x16(tb + c, r0);
                    if (!of32) tc_ld_32x32b_x16(tb + c + 16, r1);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        v[i] = rs * __uint_as_float(r0[i]);
                        v[16 + i] = of32 ? 0.0f : rs * __uint_as_float(r1[i]);
                    }
                    const int lim = N - (t.n0 + c);
                    if (add) {
                        uint4 av[4];
                        warp_load_finish(stg, aw, av, lane);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            v[4 * j] += __uint_as_float(av[j].x);
                            v[4 * j + 1] += __uint_as_float(av[j].y);
                            v[4 * j + 2] += __uint_as_float(av[j].z);
                            v[4 * j + 3] += __uint_as_float(av[j].w);
                        }
                        if (!of32) {
                            add_issue(aw, c + 16);
                            warp_load_finish(stg, aw, av, lane);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                v[16 + 4 * j] += __uint_as_float(av[j].x);
                                v[16 + 4 * j + 1] += __uint_as_float(av[j].y);
                                v[16 + 4 * j + 2] += __uint_as_float(av[j].z);
                                v[16 + 4 * j + 3] += __uint_as_float(av[j].w);
                            }
                        }
                    }
                    uint4 blk[4];
                    if (of32) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            blk[j] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                                __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            blk[j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                                pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                                pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
                    }
                    const int vch = lim > 0 ? static_cast<int>(lim * es / 16) : 0;
                    warp_store_block(stg, blk, lane, out_rows + static_cast<size_t>(t.out_col0 + c) * es,
                                     pitch, valid_rows, vch);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && rank == 1)
                    mbar_arrive_remote(map_shared_rank(tempty_bar(acc), 0));
                else
                    mbar_arrive(tempty_bar(acc));
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    if (PAIR) {
        // no CTA of the pair leaves while the other may still touch its
        // shared memory, barriers or tensor memory
        __syncwarp();
        tc_fence_before();
        cluster_sync();
        if (warp == 1) {
            __syncwarp();
            tc_fence_after();
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        }
    } else {
        __syncthreads();
        if (warp == 1) {
            __syncwarp();
            tc_fence_after();
            tmem_dealloc(tmem_base, TMEM_COLS);
        }
    }
}

// ---------------------------------------------------------------------------
// Token-column form (CTA pair). The weights are the MMA's A operand: M = 256
// output features, 128 rows of A in each CTA, read MN-major straight from the
// [Z, K, N] weights (the same 64-column strips as the row-tile forms). The
// unit's tokens are its B operand: N = the unit's token count rounded up to
// 16 (at most 256), the first half in the even CTA, read K-major from the
// row-major activations. A segment of n rows thus costs n rounded up to 16
// MMA columns instead of whole 128- or 256-row tiles.
//
// Units: a segment of n rows is cut into ceil(n / 256) token tiles of nearly
// equal size (the 256-row tile counts of the dispatch); each unit covers 128
// output features per CTA. SwiGLU: gate and up of those features, two MMAs
// into two 256-column accumulators that take all of tensor memory, a stage
// of 48 KB (16 KB of token rows, 32 KB of weights: twice the tensor work of
// the single-CTA row-tile form per byte), 4 stages; the epilogue of a unit
// runs before the MMAs of the next, while the copies of the next run ahead.
// Plain: one MMA into one of two 256-column accumulators, so that the
// epilogue of a unit overlaps the MMAs of the next; a stage of 32 KB, 6
// stages. An expert's token tiles are innermost, so the CTA pairs that share
// a weight tile run side by side.
//
// An accumulator holds features on its lanes and tokens on its columns; the
// epilogue warps transpose 32 x 32 (BF16) or 16 x 32 (FP32) blocks through
// their staging buffers so that the stores stay row-major. Same per-element
// arithmetic as the row-tile epilogues, and the tensor core's sums do not
// depend on which operand is A: the outputs equal the row-tile forms' bit
// for bit (measured).
// ---------------------------------------------------------------------------
constexpr int SW_TOK = 256;  // tokens per unit at most
constexpr int SW_FPC = 128;  // output features of one CTA per unit

template <bool SWIGLU>
struct TGeo {
    static constexpr int STAGES = SWIGLU ? 4 : 6;
    static constexpr int WSTRIPS = SWIGLU ? 4 : 2;  // weight strips per stage
    static constexpr int STAGE_BYTES = A_BYTES + WSTRIPS * STRIP_BYTES;
    static constexpr int NACC = SWIGLU ? 1 : 2;     // accumulators (TMEM: 512 columns)
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int NBARS = 2 * STAGES + 2 * NACC + 1;
    static constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;
    static constexpr int SCHED_OFF = ((MISC_OFF + 16) + 15) / 16 * 16;
    static constexpr int STG_OFF = (SCHED_OFF + 2 * (MAXE + 1) * 4 + 127) / 128 * 128;
    static constexpr int SMEM_BYTES = STG_OFF + EPI_WARPS * STG_BYTES + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "token-column shared memory");
};

struct SUnit {
    int g, row0, n, zb, f0, out_col0;
};

MOE_DEV SUnit decode_sunit(int u, const TcParams& p, int total0, const int* s_mtp2, const int* s_off) {
    SUnit t;
    if (u < total0) {
        const int nt = p.nt[0];
        const int mt = u / nt;
        int lo = 0, hi = p.E;  // s_mtp2[lo] <= mt < s_mtp2[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_mtp2[mid] <= mt)
                lo = mid;
            else
                hi = mid;
        }
        const int me = s_mtp2[lo + 1] - s_mtp2[lo];  // token tiles of expert lo (>= 1)
        const int l = u - s_mtp2[lo] * nt;
        const int n = l / me, m = l - n * me;
        const long long rows = s_off[lo + 1] - s_off[lo];
        const int r0 = static_cast<int>(m * rows / me), r1 = static_cast<int>((m + 1) * rows / me);
        t.g = 0;
        t.row0 = s_off[lo] + r0;
        t.n = r1 - r0;
        t.zb = lo;
        t.f0 = n * p.bno;
        t.out_col0 = t.f0;
    } else {
        const int u1 = u - total0;
        const int m = u1 % p.mt1;
        const int rest = u1 / p.mt1;
        const int n = rest % p.nt[1];
        const int s = rest / p.nt[1];
        const long long rows = p.rows[1];
        const int r0 = static_cast<int>(m * rows / p.mt1), r1 = static_cast<int>((m + 1) * rows / p.mt1);
        t.g = 1;
        t.row0 = r0;
        t.n = r1 - r0;
        t.zb = s;
        t.f0 = n * p.bno;
        t.out_col0 = s * p.N[1] + t.f0;
    }
    return t;
}

template <bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1) tc_token_pair_kernel(const __grid_constant__ TcParams p) {
    using G = TGeo<SWIGLU>;
    constexpr int STAGES = G::STAGES;
    constexpr int NACC = G::NACC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + G::BAR_OFF;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + NACC + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * NACC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::MISC_OFF + 4);
    int* s_mtp = reinterpret_cast<int*>(smem + G::SCHED_OFF);
    int* s_off = s_mtp + (MAXE + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int unit0 = static_cast<int>(blockIdx.x >> 1);
    const int ustep = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int g = 0; g < 2; ++g) {
            if (!p.enabled[g]) continue;
            tma_prefetch_map(&p.mapA[g]);
            tma_prefetch_map(&p.mapB0[g]);
            if (SWIGLU) tma_prefetch_map(&p.mapB1[g]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    // everything above overlaps the previous kernel; its outputs are read below
    pdl_wait();
    pdl_trigger();
    if (p.enabled[0]) {
        for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
            s_mtp[i] = p.mt_prefix[i];
            s_off[i] = p.offsets[i];
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total0 = p.enabled[0] ? s_mtp[p.E] * p.nt[0] : 0;
    const int total = total0 + (p.enabled[1] ? p.mt1 * p.Z[1] * p.nt[1] : 0);
    const WaitCtx wc{p.err, abort_flag, p.timeout_ns};

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int u = unit0; u < total && ok; u += ustep) {
                const SUnit t = decode_sunit(u, p, total0, s_mtp, s_off);
                const int nh = ((t.n + 15) & ~15) >> 1;  // token columns held by each CTA
                const int arow = t.row0 + rank * nh;
                const int fc = t.f0 + SW_FPC * rank;   // this CTA's first output feature
                const CUtensorMap* mA = &p.mapA[t.g];
                const CUtensorMap* mB0 = &p.mapB0[t.g];
                const CUtensorMap* mB1 = &p.mapB1[t.g];
                const bool wide = p.b_wide[t.g] != 0;
                for (int kb = 0; kb < p.kblocks[t.g]; ++kb) {
                    if (!bounded_wait(empty_bar(stage), phase ^ 1u, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sX = sbase + stage * G::STAGE_BYTES;
                    const uint32_t sW = sX + A_BYTES;
                    const uint32_t fb = map_shared_rank(full_bar(stage), 0);
                    if (rank == 0) mbar_expect_tx(full_bar(stage), 2 * G::STAGE_BYTES);
                    const int kc = kb * BK;
                    tma_load_2d_pair(sX, mA, kc, arow, fb);
                    if (wide) {
                        tma_load_4d_pair(sW, mB0, 0, kc, fc >> 6, t.zb, fb);
                        if (SWIGLU) tma_load_4d_pair(sW + 2 * STRIP_BYTES, mB1, 0, kc, fc >> 6, t.zb, fb);
                    } else {
                        tma_load_3d_pair(sW, mB0, fc, kc, t.zb, fb);
                        tma_load_3d_pair(sW + STRIP_BYTES, mB0, fc + 64, kc, t.zb, fb);
                        if (SWIGLU) {
                            tma_load_3d_pair(sW + 2 * STRIP_BYTES, mB1, fc, kc, t.zb, fb);
                            tma_load_3d_pair(sW + 3 * STRIP_BYTES, mB1, fc + 64, kc, t.zb, fb);
                        }
                    }
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy this thread issued has landed before the CTA can exit
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u)
                    bounded_drain(rank == 0 ? full_bar(s) : empty_bar(s), (last_par >> s) & 1u,
                                  p.timeout_ns, p.err);
        }
    } else if (warp == 1 && rank == 1) {
        // the odd CTA of a pair issues no MMAs
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer (even CTA) ----------------
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            // token rows: K-major B; weight strips: MN-major A (8 KB between
            // 64-feature strips, 1 KB between 8-row k groups)
            const uint64_t bdesc0 = smem_desc_sw128(sbase, 16, 1024);
            const uint64_t adesc0 = smem_desc_sw128(sbase + A_BYTES, STRIP_BYTES, 1024);
            const uint32_t idesc0 = idesc_bf16_f32(2 * BM, 0, 0) | (1u << 15);  // A MN-major
            for (int u = unit0; u < total && ok; u += ustep) {
                const SUnit t = decode_sunit(u, p, total0, s_mtp, s_off);
                const uint32_t idesc = idesc0 | (static_cast<uint32_t>(((t.n + 15) & ~15) >> 3) << 17);
                if (!bounded_wait(tempty_bar(acc), acc_phase ^ 1u, wc, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
                for (int kb = 0; kb < p.kblocks[t.g]; ++kb) {
                    if (!bounded_wait(full_bar(stage), phase, wc, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t soff = static_cast<uint64_t>(stage * G::STAGE_BYTES) >> 4;
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {
                        const uint64_t bd = bdesc0 + soff + (ks * 32) / 16;
                        const uint32_t accum = (kb != 0 || ks != 0) ? 1u : 0u;
                        // SwiGLU: gate strips into columns 0-255, up strips into 256-511
#pragma unroll
                        for (int j = 0; j < (SWIGLU ? 2 : 1); ++j) {
                            const uint64_t ad = adesc0 + soff + (j * 2 * STRIP_BYTES + ks * 2048) / 16;
                            tc_mma_bf16_pair(d_tmem + static_cast<uint32_t>(256 * j), ad, bd, idesc, accum);
                        }
                    }
                    tc_commit_pair_mc(empty_bar(stage), 3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_mc(tfull_bar(acc), 3);
                if (++acc == NACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            tc_commit_pair(drain_bar);
            bounded_drain(drain_bar, 0, p.timeout_ns, p.err);
        }
    } else {
        // ---------------- epilogue warps 2..9 (both CTAs) ----------------
        const int q = warp & 3;            // TMEM lane quarter: features 32q .. 32q + 31
        const int half = (warp - 2) >> 2;  // token columns [128 half, 128 half + 128)
        uint4* stg = reinterpret_cast<uint4*>(smem + G::STG_OFF + (warp - 2) * STG_BYTES);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = unit0; u < total; u += ustep) {
            const SUnit t = decode_sunit(u, p, total0, s_mtp, s_off);
            int ok = 1;
            if (lane == 0) ok = bounded_wait(tfull_bar(acc), acc_phase, wc) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * 256) + (static_cast<uint32_t>(q * 32) << 16);
            const int N = p.N[t.g];
            const int fl = SW_FPC * rank + 32 * q;  // this warp's first feature in the unit
            const int lim = N - (t.f0 + fl);
            const int c0 = 128 * half;
            if (SWIGLU) {
                const size_t pitch = static_cast<size_t>(p.out_ld[t.g]) * 2;
                const int vch = lim <= 0 ? 0 : (lim >= 32 ? 4 : lim / 8);
                char* base = static_cast<char*>(p.out[t.g]) + static_cast<size_t>(t.out_col0 + fl) * 2;
                const int c1 = min(c0 + 128, t.n);
#pragma unroll 1
                for (int c = c0; c < c1; c += 32) {
                    uint32_t g0[16], g1[16], u0[16], u1[16];
                    tc_ld_32x32b_x16(tb + c, g0);
                    tc_ld_32x32b_x16(tb + c + 16, g1);
                    tc_ld_32x32b_x16(tb + 256 + c, u0);
                    tc_ld_32x32b_x16(tb + 256 + c + 16, u1);
                    tc_wait_ld();
                    float h[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float ga = __uint_as_float(g0[i]), gb = __uint_as_float(g1[i]);
                        h[i] = __fdividef(ga, 1.0f + __expf(-ga)) * __uint_as_float(u0[i]);
                        h[16 + i] = __fdividef(gb, 1.0f + __expf(-gb)) * __uint_as_float(u1[i]);
                    }
                    warp_stage_bf16_column(stg, lane, h);
                    warp_flush_block(stg, lane, base + static_cast<size_t>(t.row0 + c) * pitch, pitch,
                                     t.n - c, vch);
                }
            } else {
                // FP32 rows, or the 24-bit blocked layout (a 256-feature pair unit is one block)
                const bool f24 = p.out_f32[t.g] == 2;
                const size_t pitch = static_cast<size_t>(p.out_ld[t.g]) * (f24 ? 3 : 4);
                const int vch = lim <= 0 ? 0 : (lim >= 32 ? 8 : lim / 4);
                const int col = t.out_col0 + fl;
                const size_t blk = static_cast<size_t>(col / YS24_BLOCK) * (3 * YS24_BLOCK);
                const size_t hi_off = blk + 2 * (col % YS24_BLOCK), lo_off = blk + 2 * YS24_BLOCK + col % YS24_BLOCK;
                char* rows0 = static_cast<char*>(p.out[t.g]);
                char* base = rows0 + static_cast<size_t>(col) * 4;
                // the row scales of this warp's 128 tokens, lane l holding tokens c0 + 32 j + l
                float rs[4];
                const bool scale = t.g == 0 && p.rowscale0 != nullptr;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ti = c0 + 32 * j + lane;
                    rs[j] = (scale && ti < t.n) ? p.rowscale0[t.row0 + ti] : 1.0f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = c0 + 16 * i;
                    if (c < t.n) {
                        uint32_t r[16];
                        tc_ld_32x32b_x16(tb + c, r);
                        tc_wait_ld();
                        float v[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            v[e] = __shfl_sync(0xffffffffu, rs[i >> 1], 16 * (i & 1) + e) * __uint_as_float(r[e]);
                        if (f24)
                            warp_store_f24_columns(stg, lane, v, rows0 + static_cast<size_t>(t.row0 + c) * pitch, pitch,
                                                   t.n - c, hi_off, lo_off);
                        else
                            warp_store_f32_columns(stg, lane, v, base + static_cast<size_t>(t.row0 + c) * pitch,
                                                   pitch, t.n - c, vch);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 1)
                    mbar_arrive_remote(map_shared_rank(tempty_bar(acc), 0));
                else
                    mbar_arrive(tempty_bar(acc));
            }
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    // no CTA of the pair leaves while the other may still touch its shared
    // memory, barriers or tensor memory
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

bool make_A_map(CUtensorMap* m, const void* A, int rows, int K, int lda) {
    // K: the columns of A the reduction reads
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(lda) * 2};
    const uint32_t box[2] = {64, BM};
    return encode_tmap(m, A, 2, dims, strides, box);
}

// B [Z, K, N] seen as [Z, N/64 strips, K, 64]: one box of `strips` strips lands
// in shared memory strip after strip (8 KB each), the layout the MMA reads.
// Needs N % 64 == 0 so that no strip runs past the end of a row.
bool make_B_strip_map(CUtensorMap* m, const void* B, int Z, int K, int N, int strips) {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(K), static_cast<uint64_t>(N / 64),
                              static_cast<uint64_t>(Z)};
    const uint64_t strides[3] = {static_cast<uint64_t>(N) * 2, 128,
                                 static_cast<uint64_t>(K) * N * 2};
    const uint32_t box[4] = {64, 64, static_cast<uint32_t>(strips), 1};
    return encode_tmap(m, B, 4, dims, strides, box);
}

bool make_B_map(CUtensorMap* m, const void* B, int Z, int K, int N) {
    const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                              static_cast<uint64_t>(Z)};
    const uint64_t strides[2] = {static_cast<uint64_t>(N) * 2, static_cast<uint64_t>(K) * N * 2};
    const uint32_t box[3] = {64, 64, 1};
    return encode_tmap(m, B, 3, dims, strides, box);
}

template <int MODE, bool PAIR>
bool prepare_kernel(int dev) {
    static bool attr_set[64] = {};
    if (dev < 0 || dev >= 64) return false;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(tc_grouped_gemm_kernel<MODE, PAIR>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Geo<PAIR>::SMEM_BYTES) != cudaSuccess)
            return false;
        attr_set[dev] = true;
    }
    return true;
}

// How many CTA pairs of the pair kernel fit on the device at once (0: none,
// or the query failed; the single-CTA form is used then).
template <int MODE>
int pair_slots(int dev) {
    static int cache[64] = {};
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = -1;
        if (prepare_kernel<MODE, true>(dev)) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * static_cast<unsigned>(num_sms()));
            cfg.blockDim = dim3(THREADS);
            cfg.dynamicSmemBytes = Geo<true>::SMEM_BYTES;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int c = 0;
            if (cudaOccupancyMaxActiveClusters(&c, tc_grouped_gemm_kernel<MODE, true>, &cfg) ==
                    cudaSuccess &&
                c > 0)
                n = c;
            else
                cudaGetLastError();  // clear a failed query
        }
        cache[dev] = n;
    }
    return cache[dev] > 0 ? cache[dev] : 0;
}

template <int MODE, bool PAIR>
cudaError_t launch_tc_t(const TcGemmArgs& a, int nstrip, int slots, cudaStream_t s) {
    constexpr bool SWIGLU = MODE == TC_SWIGLU || MODE == TC_SWIGLU_BWD;
    constexpr int UROWS = PAIR ? 2 * BM : BM;
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.nstrip = nstrip;
    p.bno = SWIGLU ? 128 : 64 * p.nstrip;
    p.idesc = idesc_bf16_f32(PAIR ? 2 * BM : BM, 64 * p.nstrip, /*b_mn_major=*/1);
    const int BNO = p.bno;
    // strips of B one CTA loads per stage
    const int strips = PAIR ? (SWIGLU ? 2 : nstrip / 2) : (SWIGLU ? 2 : nstrip);
    long long units_bound = 0;
    for (int g = 0; g < 2; ++g) {
        const TcGroup& G = a.g[g];
        p.enabled[g] = G.enabled;
        if (!G.enabled) continue;
        const int KA = G.a_kmod ? G.a_kmod : (G.a_kgroup ? G.K / (G.a_krep > 0 ? G.a_krep : 1) : G.K);
        const int KB = G.b_rows ? G.b_rows : (G.b_kmod ? G.b_kmod : G.K);
        if ((G.a_kmod && G.a_kmod % BK) || (G.b_kmod && G.b_kmod % BK)) return cudaErrorInvalidValue;
        if (G.ksplit > 1 && (g != 1 || G.Z != 1)) return cudaErrorInvalidValue;
        if (!make_A_map(&p.mapA[g], G.A, G.rows, KA, G.lda)) return cudaErrorInvalidValue;
        p.b_wide[g] = G.N % 64 == 0 && make_B_strip_map(&p.mapB0[g], G.B0, G.Z, KB, G.N, strips) &&
                      (!SWIGLU || make_B_strip_map(&p.mapB1[g], G.B1, G.Z, KB, G.N, strips));
        if (!p.b_wide[g]) {
            if (!make_B_map(&p.mapB0[g], G.B0, G.Z, KB, G.N)) return cudaErrorInvalidValue;
            if (SWIGLU && !make_B_map(&p.mapB1[g], G.B1, G.Z, KB, G.N)) return cudaErrorInvalidValue;
        }
        p.kblocks[g] = (G.K + BK - 1) / BK;
        if (G.A2 != nullptr) {
            // a second reduction segment: group 1 of a single-CTA plain launch, whole k-blocks
            if (g != 1 || PAIR || MODE != TC_PLAIN || G.K % BK || G.ksplit > 1 || G.K2 <= 0 || G.Z != 1)
                return cudaErrorInvalidValue;
            if (!make_A_map(&p.mapA2, G.A2, G.rows, G.K2, G.lda2)) return cudaErrorInvalidValue;
            p.b2_wide = G.N % 64 == 0 && make_B_strip_map(&p.mapB2, G.B2, 1, G.K2, G.N, strips);
            if (!p.b2_wide && !make_B_map(&p.mapB2, G.B2, 1, G.K2, G.N)) return cudaErrorInvalidValue;
            p.kseg2 = p.kblocks[g];
            p.kblocks[g] += (G.K2 + BK - 1) / BK;
        }
        p.a_kmod[g] = G.a_kmod;
        p.b_kmod[g] = G.b_kmod;
        p.a_kgroup[g] = G.a_kgroup;
        p.a_krep[g] = G.a_krep > 0 ? G.a_krep : 1;
        if (g == 1) {
            const int ks = G.ksplit > 1 ? G.ksplit : 1;
            p.kbs1 = (p.kblocks[1] + ks - 1) / ks;
            if (MODE == TC_PLAIN_ACC) {
                // whole chunks per slice
                if (G.kchunk <= 0) return cudaErrorInvalidValue;
                p.kchunk1 = G.kchunk;
                p.kbs1 = (p.kbs1 + G.kchunk - 1) / G.kchunk * G.kchunk;
            }
            p.ksplit1 = ks > 1 ? (p.kblocks[1] + p.kbs1 - 1) / p.kbs1 : 1;
        }
        p.rows[g] = G.rows;
        p.N[g] = G.N;
        p.nt[g] = (G.N + BNO - 1) / BNO;
        p.Z[g] = G.Z;
        p.out[g] = G.out;
        p.out_ld[g] = G.out_ld;
        p.out_f32[g] = G.out_f32;
        p.a_out[g] = static_cast<__nv_bfloat16*>(G.a_out);
        p.u_out[g] = static_cast<__nv_bfloat16*>(G.u_out);
        if ((G.a_out != nullptr) != (G.u_out != nullptr) || (G.a_out && (MODE != TC_SWIGLU || G.out_f32)))
            return cudaErrorInvalidValue;
        p.dh[g] = G.dh;
        p.dh_ld[g] = G.dh_ld;
        p.da[g] = static_cast<__nv_bfloat16*>(G.da);
        p.du[g] = static_cast<__nv_bfloat16*>(G.du);
        p.hw[g] = static_cast<__nv_bfloat16*>(G.hw);
        if (MODE == TC_SWIGLU_BWD && (!G.dh || !G.da || !G.du || !G.hw || G.dh_ld % 4))
            return cudaErrorInvalidValue;
        if (g == 0)
            units_bound += static_cast<long long>((G.rows + UROWS - 1) / UROWS + a.E) * p.nt[0];
        else
            units_bound += static_cast<long long>((G.rows + UROWS - 1) / UROWS) *
                           (p.ksplit1 > 1 ? p.ksplit1 : G.Z) * p.nt[1];
    }
    p.E = a.E;
    p.mt1 = a.g[1].enabled ? (a.g[1].rows + UROWS - 1) / UROWS : 0;
    p.offsets = a.offsets;
    p.mt_prefix = a.mt_prefix ? a.mt_prefix + (PAIR ? a.E + 1 : 0) : nullptr;
    p.rowscale0 = a.rowscale0;
    p.addend = a.addend;
    p.add_ld = a.add_ld;
    p.poff = a.poff;
    p.dgpart = a.g[0].dgpart;
    if (MODE == TC_SWIGLU_BWD && a.g[0].enabled && a.poff == nullptr) return cudaErrorInvalidValue;
    p.err = a.err;
    p.timeout_ns = wait_timeout_ns();
    long long grid = slots;  // persistent: one CTA (pair) per slot, at most one per unit
    if (units_bound < grid) grid = units_bound;
    if (grid < 1) grid = 1;
    if constexpr (PAIR)
        return launch_pdl_cluster(tc_grouped_gemm_kernel<MODE, true>,
                                  dim3(2 * static_cast<unsigned>(grid)), dim3(THREADS),
                                  Geo<true>::SMEM_BYTES, s, 2, p);
    else
        return launch_pdl(tc_grouped_gemm_kernel<MODE, false>, dim3(static_cast<unsigned>(grid)),
                          dim3(THREADS), Geo<false>::SMEM_BYTES, s, p);
}

// The token-column CTA-pair form (tc_token_pair_kernel).
template <bool SWIGLU>
bool prepare_token_kernel(int dev) {
    static bool attr_set[64] = {};
    if (dev < 0 || dev >= 64) return false;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(tc_token_pair_kernel<SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TGeo<SWIGLU>::SMEM_BYTES) != cudaSuccess)
            return false;
        attr_set[dev] = true;
    }
    return true;
}

template <bool SWIGLU>
int token_pair_slots(int dev) {
    static int cache[64] = {};
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = -1;
        if (prepare_token_kernel<SWIGLU>(dev)) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * static_cast<unsigned>(num_sms()));
            cfg.blockDim = dim3(THREADS);
            cfg.dynamicSmemBytes = TGeo<SWIGLU>::SMEM_BYTES;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int c = 0;
            if (cudaOccupancyMaxActiveClusters(&c, tc_token_pair_kernel<SWIGLU>, &cfg) == cudaSuccess && c > 0)
                n = c;
            else
                cudaGetLastError();  // clear a failed query
        }
        cache[dev] = n;
    }
    return cache[dev] > 0 ? cache[dev] : 0;
}

// Whether a forward launch takes the token-column form: the SwiGLU or the
// plain product (FP32 output, no addend), no k remaps or split, no gate/up
// products kept, and routed segments of 128 to 511 rows on average, where
// the row-tile forms would run single-CTA 128-row tiles that pad each
// segment by 64 rows on average. Shorter segments leave the pair's 256 MMA
// rows of weights for few tokens; from 512 rows on the row-tile CTA pair,
// whose epilogue overlaps the next tile, measured faster (medium prefill
// gate/up 1116 against 1198 us). The environment variable MOE_GEMM_FORM
// overrides the choice for tests and tuning: "rows" never takes the token
// form, "tokens" takes it whenever the product allows it.
template <int MODE>
bool token_form_ok(const TcGemmArgs& a) {
    if (MODE != TC_SWIGLU && MODE != TC_PLAIN) return false;
    if (a.addend != nullptr || !a.g[0].enabled || a.mt_prefix == nullptr) return false;
    for (int g = 0; g < 2; ++g) {
        const TcGroup& G = a.g[g];
        if (!G.enabled) continue;
        if (G.a_kmod || G.b_kmod || G.a_kgroup || G.ksplit > 1 || G.a_out != nullptr ||
            (G.b_rows && G.b_rows != G.K))
            return false;
        if (MODE == TC_PLAIN && G.out_f32 != 1) return false;
        if (MODE == TC_SWIGLU && G.out_f32 != 0) return false;
    }
    const char* e = getenv("MOE_GEMM_FORM");
    if (e != nullptr && (e[0] == 'r' || e[0] == 's')) return false;
    if (e != nullptr && e[0] == 't') return true;
    const long long E = a.E > 0 ? a.E : 1;
    return a.g[0].rows >= 128LL * E && a.g[0].rows < 512LL * E;
}

template <bool SWIGLU>
cudaError_t launch_token_t(const TcGemmArgs& a, int slots, cudaStream_t s) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.bno = 2 * SW_FPC;  // output features of a pair per unit
    const int strips = 2;  // 64-column strips per matrix and CTA
    long long units_bound = 0;
    for (int g = 0; g < 2; ++g) {
        const TcGroup& G = a.g[g];
        p.enabled[g] = G.enabled;
        if (!G.enabled) continue;
        if (!make_A_map(&p.mapA[g], G.A, G.rows, G.K, G.lda)) return cudaErrorInvalidValue;
        p.b_wide[g] = G.N % 64 == 0 && make_B_strip_map(&p.mapB0[g], G.B0, G.Z, G.K, G.N, strips) &&
                      (!SWIGLU || make_B_strip_map(&p.mapB1[g], G.B1, G.Z, G.K, G.N, strips));
        if (!p.b_wide[g]) {
            if (!make_B_map(&p.mapB0[g], G.B0, G.Z, G.K, G.N)) return cudaErrorInvalidValue;
            if (SWIGLU && !make_B_map(&p.mapB1[g], G.B1, G.Z, G.K, G.N)) return cudaErrorInvalidValue;
        }
        p.kblocks[g] = (G.K + BK - 1) / BK;
        p.rows[g] = G.rows;
        p.N[g] = G.N;
        p.nt[g] = (G.N + p.bno - 1) / p.bno;
        p.Z[g] = G.Z;
        p.out[g] = G.out;
        p.out_ld[g] = G.out_ld;
        p.out_f32[g] = G.out_f32;
        // routed rows of a plain product in the 24-bit blocked layout, where allowed
        if (!SWIGLU && g == 0 && a.f24_ok && G.out_f32 == 1 && G.N % YS24_BLOCK == 0) p.out_f32[g] = 2;
        const long long mt = (G.rows + SW_TOK - 1) / SW_TOK;
        units_bound += g == 0 ? (mt + a.E) * p.nt[0] : mt * G.Z * p.nt[1];
    }
    p.E = a.E;
    p.mt1 = a.g[1].enabled ? (a.g[1].rows + SW_TOK - 1) / SW_TOK : 0;
    p.offsets = a.offsets;
    p.mt_prefix = a.mt_prefix + a.E + 1;  // tiles of 256 rows per expert
    p.rowscale0 = a.rowscale0;
    p.err = a.err;
    p.timeout_ns = wait_timeout_ns();
    long long grid = slots;
    if (units_bound < grid) grid = units_bound;
    if (grid < 1) grid = 1;
    if (a.used_f24 != nullptr) *a.used_f24 = p.enabled[0] && p.out_f32[0] == 2 ? 1 : 0;
    return launch_pdl_cluster(tc_token_pair_kernel<SWIGLU>, dim3(2 * static_cast<unsigned>(grid)),
                              dim3(THREADS), TGeo<SWIGLU>::SMEM_BYTES, s, 2, p);
}

template <int MODE>
cudaError_t launch_tc_s(const TcGemmArgs& a, cudaStream_t s) {
    constexpr bool SWIGLU = MODE == TC_SWIGLU || MODE == TC_SWIGLU_BWD;
    int dev = 0;
    cudaGetDevice(&dev);
    int nmax = 0;
    for (int g = 0; g < 2; ++g)
        if (a.g[g].enabled && a.g[g].N > nmax) nmax = a.g[g].N;
    const int nstrip = SWIGLU ? 4 : (nmax >= 256 ? 4 : (nmax + 63) / 64);
    // The pair form splits B's strips between the two CTAs (an even count).
    // Its routed tiles are 256 rows, so a segment wastes 128 padded rows on
    // average instead of 64: it is used when segments average >= 512 rows.
    // Dense projections alone (no routed group, single product: the latent
    // down and up projections, the router) measured faster in the single-CTA
    // form (latent up projection 69 -> 60 us).
    const bool even = SWIGLU || nstrip % 2 == 0;
    const char* form = getenv("MOE_GEMM_FORM");  // 's': single-CTA row tiles (tests, tuning)
    const bool long_segments =
        (form == nullptr || form[0] != 's') &&
        (!a.g[0].enabled || static_cast<long long>(a.g[0].rows) >= 512LL * (a.E > 0 ? a.E : 1));
    const bool dense_plain = MODE == TC_PLAIN && !a.g[0].enabled;
    if constexpr (MODE == TC_SWIGLU || MODE == TC_PLAIN) {
        if (token_form_ok<MODE>(a)) {
            const int slots = token_pair_slots<MODE == TC_SWIGLU>(dev);
            if (slots > 0) return launch_token_t<MODE == TC_SWIGLU>(a, slots, s);
        }
    }
    if constexpr (MODE != TC_PLAIN_ACC) {
        const int slots = (even && long_segments && !dense_plain) ? pair_slots<MODE>(dev) : 0;
        if (slots > 0) return launch_tc_t<MODE, true>(a, nstrip, slots, s);
    } else {
        (void)even;
        (void)long_segments;
        (void)dense_plain;
        if (a.g[0].enabled || !a.g[1].enabled) return cudaErrorInvalidValue;
    }
    if (!prepare_kernel<MODE, false>(dev)) return cudaErrorInvalidValue;
    return launch_tc_t<MODE, false>(a, nstrip, num_sms(), s);
}

}  // namespace

cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t s) {
    if (a.used_f24 != nullptr) *a.used_f24 = 0;  // set by the token-column launch where it applies
    if (a.swiglu == TC_SWIGLU_BWD) return launch_tc_s<TC_SWIGLU_BWD>(a, s);
    if (a.swiglu == TC_PLAIN && a.g[1].enabled && a.g[1].kchunk > 0)
        return launch_tc_s<TC_PLAIN_ACC>(a, s);
    return a.swiglu ? launch_tc_s<TC_SWIGLU>(a, s) : launch_tc_s<TC_PLAIN>(a, s);
}

}  // namespace moe
