// Fused decode back end: for a batch of at most 128 tokens (BF16 layer, no
// latent projection), everything after the router in ONE persistent launch:
// the stable dispatch, the row gather, the grouped gate/up GEMM with the
// SiLU(gate)*up epilogue, the grouped down GEMM scaled by the gate weights,
// the shared experts, and the deterministic combine.
//
// What it computes is the forward of APEX-1 Mathematical Reference Part 3,
// sections 12.2 and 13.2 (FFN(x) = W_down(SiLU(x W_gate) * x W_up); MoE(x) =
// sum of the shared experts + sum_k g_k Expert_{e_k}(x)), grouped as in
// kimi_k3 StableLatentMoE "Flatten routing and recover original token order"
// and "Grouped expert execution and sparse gradients", with the same tiles,
// reduction order and combine order as the separate launches, so the result
// is the same to the bit. The pages run it as a host loop over the experts
// with a host read of each expert's token count ("MoE from scratch"
// MoELayer.forward); here nothing leaves the device.
//
// Work units, in this order, dealt to the CTAs round robin:
//   0  shared gate/up   128 token rows x 128 hidden columns of shared expert s
//   1  routed gate/up   expert e's rows (at most 128) x 128 hidden columns
//   2  shared down      token rows x 256 output columns (all shared hidden columns)
//   3  routed down      expert e's rows x 256 output columns, times the gate weight
// then the combine. Every CTA computes the dispatch itself (a few microseconds,
// the same integers everywhere), so units 0 and 1 wait for nothing; a unit of
// kind 2 or 3 waits for the gate/up units it reads (a counter per expert and
// one for the shared experts, released by each epilogue warp after its
// stores), and the combine waits for every down unit. A unit only waits on
// units of lower index, and every CTA works through its units in index
// order, so with the CTAs resident together (one per SM) every wait ends;
// each one is bounded anyway. The counters are zeroed by the router launch
// that precedes this one.
//
// Rows of a routed gate/up unit with at most GATHER_MAX rows come straight
// from x with TMA row gathers (four rows per copy); every CTA also copies its
// share of the rows into the gathered-row buffer (which the backward pass
// reads), and a heavier unit loads its rows from there as tiles once every
// CTA has released its share (one more counter).
#include "common.cuh"
#include "dispatch_dev.cuh"
#include "internal.h"
#include "warp_stage.cuh"

namespace moe {
namespace {

constexpr int BM = TC_BM;                 // 128 rows per unit
constexpr int BK = 64;                    // k-block
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int STRIP_BYTES = BK * 64 * 2;  // 8 KB
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int STAGE_BYTES = A_BYTES + 4 * STRIP_BYTES;  // 48 KB
constexpr int STG_BYTES = 32 * 64;
constexpr int EMAXF = 256;
constexpr int GATHER_MAX = 32;  // routed rows a unit gathers from x itself
constexpr int MAX_STAGES = 4;
constexpr int NBARS = 2 * MAX_STAGES + 4 + 2;  // full, empty, tfull x2, tempty x2, drain, dispatch

// Shared memory after the 1024-aligned ring. The dispatch scratch and the
// epilogue's staging buffers share their space (the epilogue warps use one,
// then the other).
template <int EMAXT>
struct Smem {
    uint64_t bars[NBARS];
    uint32_t tmem_slot;
    int abort_flag;
    int nused;
    int pad_;
    union {
        DispatchScratch<EMAXT> disp;
        uint4 stg[EPI_WARPS][STG_BYTES / 16];
    };
    int32_t tok[DISPATCH_CHUNK];   // sorted position -> token
    float wloc[DISPATCH_CHUNK];    // sorted position -> gate weight
    int32_t invl[DISPATCH_CHUNK];  // assignment t*K+k -> sorted position
    int32_t off[EMAXT + 1];        // expert offsets
    int32_t used[EMAXT];           // experts with rows, ascending
};

// Ring stages: 4 (192 KB of weight tiles in flight).
template <int EMAXT>
constexpr int stages_for() { return 4; }
template <int EMAXT>
constexpr size_t smem_bytes() { return 1024 + stages_for<EMAXT>() * STAGE_BYTES + sizeof(Smem<EMAXT>); }
static_assert(smem_bytes<64>() <= 227 * 1024 && smem_bytes<128>() <= 227 * 1024 &&
              smem_bytes<256>() <= 227 * 1024, "fused decode shared memory");

struct DecodeParams {
    CUtensorMap mapX;    // x [T, d], box 64 x 128 (shared experts' rows)
    CUtensorMap mapXg;   // x [T, d], box 64 x 1 (row gathers)
    CUtensorMap mapWg;   // W_gate [E, d, F] as 64-column strips, 2 strips a box
    CUtensorMap mapWu;   // W_up
    CUtensorMap mapSg;   // Ws_gate [S, d, Fs], 2 strips
    CUtensorMap mapSu;   // Ws_up
    CUtensorMap mapH;    // h [T*K, F], box 64 x 128
    CUtensorMap mapHs;   // hs [T, S*Fs], box 64 x 128
    CUtensorMap mapWd;   // W_down [E, F, d], 4 strips
    CUtensorMap mapSd;   // Ws_down as [1, S*Fs, d], 4 strips
    CUtensorMap mapXs;   // gathered rows xs [T*K, d], box 64 x 128
    uint32_t idesc;
    int T, d, F, E, K, S, Fs;
    const int32_t* idx;  // router output [T, K]
    const float* w;      // [T, K]
    const void* x;       // [T, d] BF16
    // dispatch results (written by CTA 0), gathered rows, hidden rows, outputs
    int32_t* counts;
    int32_t* offsets;
    int32_t* mt_prefix;
    int32_t* sorted_token;
    float* sorted_w;
    int32_t* inv;
    __nv_bfloat16* xs;
    __nv_bfloat16* h;
    __nv_bfloat16* hs;
    float* ys;  // routed rows times their gate weight
    float* shout;
    void* out;
    int out_f32;
    unsigned* ctr;  // [E + 3]: per-expert gate/up warps, shared gate/up warps, down warps,
                    // gather warps
    int* err;
    unsigned long long timeout_ns;
};

// One unit: kind (0..3), its matrix z (expert or shared expert), A rows
// [row0, row0 + rows), output column n0, and its k-blocks.
struct DUnit {
    int kind, z, row0, rows, n0, kblocks;
};

struct Counts {
    int nt_g, nt_gs, nt_d, U1, U2, U3, U4, nused;
    MOE_DEV int total() const { return U1 + U2 + U3 + U4; }
};

MOE_DEV Counts unit_counts(const DecodeParams& p, int nused) {
    Counts c;
    c.nt_g = (p.F + 127) / 128;
    c.nt_gs = p.S ? (p.Fs + 127) / 128 : 0;
    c.nt_d = (p.d + 255) / 256;
    c.U1 = p.S * c.nt_gs;
    c.U2 = nused * c.nt_g;
    c.U3 = p.S ? c.nt_d : 0;
    c.U4 = nused * c.nt_d;
    c.nused = nused;
    return c;
}

template <class SM>
MOE_DEV DUnit decode_dunit(int u, const DecodeParams& p, const Counts& c, const SM& sm) {
    DUnit t;
    if (u < c.U1) {
        const int s = u / c.nt_gs;
        t.kind = 0;
        t.z = s;
        t.row0 = 0;
        t.rows = p.T;
        t.n0 = (u - s * c.nt_gs) * 128;
        t.kblocks = (p.d + BK - 1) / BK;
        return t;
    }
    u -= c.U1;
    if (u < c.U2) {
        const int j = u / c.nt_g;
        const int e = sm.used[j];
        t.kind = 1;
        t.z = e;
        t.row0 = sm.off[e];
        t.rows = sm.off[e + 1] - sm.off[e];
        t.n0 = (u - j * c.nt_g) * 128;
        t.kblocks = (p.d + BK - 1) / BK;
        return t;
    }
    u -= c.U2;
    if (u < c.U3) {
        t.kind = 2;
        t.z = 0;
        t.row0 = 0;
        t.rows = p.T;
        t.n0 = u * 256;
        t.kblocks = (p.S * p.Fs + BK - 1) / BK;
        return t;
    }
    u -= c.U3;
    const int j = u / c.nt_d;
    const int e = sm.used[j];
    t.kind = 3;
    t.z = e;
    t.row0 = sm.off[e];
    t.rows = sm.off[e + 1] - sm.off[e];
    t.n0 = (u - j * c.nt_d) * 256;
    t.kblocks = (p.F + BK - 1) / BK;
    return t;
}

// Counter a unit releases (and the value its readers wait for).
MOE_DEV unsigned* unit_counter(const DecodeParams& p, const DUnit& t) {
    if (t.kind == 0) return p.ctr + p.E;
    if (t.kind == 1) return p.ctr + t.z;
    return p.ctr + p.E + 1;
}

MOE_DEV void epi_bar_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int EMAXT>
__global__ void __launch_bounds__(THREADS, 1) decode_fused_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int STAGES = stages_for<EMAXT>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Smem<EMAXT>& sm = *reinterpret_cast<Smem<EMAXT>*>(ring + STAGES * STAGE_BYTES);
    const uint32_t sbase = smem_u32(ring);
    const uint32_t bar0 = smem_u32(&sm.bars[0]);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    const uint32_t disp_bar = bar0 + 8u * (2 * STAGES + 5);
    volatile int* abort_flag = &sm.abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        mbar_init(disp_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.mapX);
        tma_prefetch_map(&p.mapXg);
        tma_prefetch_map(&p.mapWg);
        tma_prefetch_map(&p.mapWu);
        tma_prefetch_map(&p.mapH);
        tma_prefetch_map(&p.mapWd);
        tma_prefetch_map(&p.mapXs);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    // the router's outputs and the zeroed counters are read below
    pdl_wait();
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_slot;
    const WaitCtx wc{p.err, abort_flag, p.timeout_ns};
    const int TK = p.T * p.K;
    const Counts c0 = unit_counts(p, 0);  // only U1 is valid before the dispatch

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            bool ok = true, have = false, gathered = false;
            Counts c = c0;
            for (int u = blockIdx.x; ok; u += gridDim.x) {
                if (!have && u >= c.U1) {
                    if (!bounded_wait(disp_bar, 0, wc)) break;
                    c = unit_counts(p, sm.nused);
                    have = true;
                }
                if (u >= (have ? c.total() : c.U1)) break;
                const DUnit t = decode_dunit(u, p, c, sm);
                const bool tiled = t.kind == 1 && t.rows > GATHER_MAX;  // rows from xs
                if (tiled && !gathered) {
                    // every CTA's share of the gathered rows is in xs
                    if (!bounded_wait_count(p.ctr + p.E + 2, EPI_WARPS * gridDim.x, wc)) break;
                    fence_proxy_async_global();
                    gathered = true;
                }
                if (t.kind >= 2) {
                    // the hidden rows this unit reads: every epilogue warp of their units done
                    const unsigned target = EPI_WARPS * (t.kind == 2 ? c.U1 : c.nt_g);
                    if (!bounded_wait_count(t.kind == 2 ? p.ctr + p.E : p.ctr + t.z, target, wc)) break;
                    fence_proxy_async_global();
                }
                const int ng = (t.rows + 3) / 4;  // row gathers of a routed gate/up k-block
                const uint32_t abytes = (t.kind == 1 && !tiled) ? static_cast<uint32_t>(ng) * 512u : A_BYTES;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!bounded_wait(empty_bar(stage), phase ^ 1u, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = sbase + stage * STAGE_BYTES, sB = sA + A_BYTES;
                    const uint32_t fb = full_bar(stage);
                    mbar_expect_tx(fb, abytes + 4 * STRIP_BYTES);
                    const int kc = kb * BK;
                    if (t.kind == 0) {
                        tma_load_2d(sA, &p.mapX, kc, 0, fb);
                        tma_load_4d(sB, &p.mapSg, 0, kc, t.n0 >> 6, t.z, fb);
                        tma_load_4d(sB + 2 * STRIP_BYTES, &p.mapSu, 0, kc, t.n0 >> 6, t.z, fb);
                    } else if (tiled) {
                        tma_load_2d(sA, &p.mapXs, kc, t.row0, fb);
                        tma_load_4d(sB, &p.mapWg, 0, kc, t.n0 >> 6, t.z, fb);
                        tma_load_4d(sB + 2 * STRIP_BYTES, &p.mapWu, 0, kc, t.n0 >> 6, t.z, fb);
                    } else if (t.kind == 1) {
                        for (int g = 0; g < ng; ++g) {
                            int r[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) r[i] = sm.tok[t.row0 + min(4 * g + i, t.rows - 1)];
                            tma_gather4(sA + g * 512, &p.mapXg, kc, r[0], r[1], r[2], r[3], fb);
                        }
                        tma_load_4d(sB, &p.mapWg, 0, kc, t.n0 >> 6, t.z, fb);
                        tma_load_4d(sB + 2 * STRIP_BYTES, &p.mapWu, 0, kc, t.n0 >> 6, t.z, fb);
                    } else if (t.kind == 2) {
                        tma_load_2d(sA, &p.mapHs, kc, 0, fb);
                        tma_load_4d(sB, &p.mapSd, 0, kc, t.n0 >> 6, 0, fb);
                    } else {
                        tma_load_2d(sA, &p.mapH, kc, t.row0, fb);
                        tma_load_4d(sB, &p.mapWd, 0, kc, t.n0 >> 6, t.z, fb);
                    }
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy issued has landed before the CTA can exit
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u) bounded_drain(full_bar(s), (last_par >> s) & 1u, p.timeout_ns, p.err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, have = false;
            Counts c = c0;
            const uint64_t adesc0 = smem_desc_sw128(sbase, 16, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(sbase + A_BYTES, STRIP_BYTES, 1024);
            for (int u = blockIdx.x; ok; u += gridDim.x) {
                if (!have && u >= c.U1) {
                    if (!bounded_wait(disp_bar, 0, wc)) break;
                    c = unit_counts(p, sm.nused);
                    have = true;
                }
                if (u >= (have ? c.total() : c.U1)) break;
                const DUnit t = decode_dunit(u, p, c, sm);
                if (!bounded_wait(tempty_bar(acc), acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!bounded_wait(full_bar(stage), phase, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t soff = static_cast<uint64_t>(stage * STAGE_BYTES) >> 4;
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {
                        const uint64_t ad = adesc0 + soff + (ks * 32) / 16;
                        const uint64_t bd = bdesc0 + soff + (ks * 2048) / 16;
                        tc_mma_bf16(d_tmem, ad, bd, p.idesc, (kb != 0 || ks != 0) ? 1u : 0u);
                    }
                    tc_commit(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(tfull_bar(acc));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            tc_commit(drain_bar);
            bounded_drain(drain_bar, 0, p.timeout_ns, p.err);
        }
    } else {
        // ---------------- epilogue warps 2..9 ----------------
        const int tid = threadIdx.x - 64;
        // the dispatch, the same in every CTA (CTA 0 also writes it out)
        dispatch_block_impl<256, EMAXT>(tid, [] { epi_bar_sync(); }, sm.disp, p.idx, p.w, TK, p.K, p.E,
                                        BM, blockIdx.x == 0, p.counts, p.offsets, p.mt_prefix,
                                        p.sorted_token, p.sorted_w, p.inv, p.err, sm.tok, sm.wloc,
                                        sm.invl, sm.off);
        epi_bar_sync();
        if (tid < 32) {
            // the experts with rows, ascending
            int has[EMAXT / 32];
            int n = 0;
#pragma unroll
            for (int i = 0; i < EMAXT / 32; ++i) {
                const int e = lane * (EMAXT / 32) + i;
                has[i] = (e < p.E && sm.off[e + 1] > sm.off[e]) ? 1 : 0;
                n += has[i];
            }
            int incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int at = incl - n;
#pragma unroll
            for (int i = 0; i < EMAXT / 32; ++i)
                if (has[i]) sm.used[at++] = lane * (EMAXT / 32) + i;
            if (lane == 31) sm.nused = incl;
        }
        epi_bar_sync();
        if (tid == 0) mbar_arrive(disp_bar);
        // gathered rows for the backward pass: rows r of this CTA, one warp a row
        {
            const int vpr = p.d / 8;  // 16-byte vectors per row
            const uint4* src = static_cast<const uint4*>(p.x);
            uint4* dst = reinterpret_cast<uint4*>(p.xs);
            for (int r = blockIdx.x + gridDim.x * (tid >> 5); r < TK; r += gridDim.x * EPI_WARPS) {
                const size_t so = static_cast<size_t>(sm.tok[r]) * vpr, d0 = static_cast<size_t>(r) * vpr;
                for (int v = lane; v < vpr; v += 32) dst[d0 + v] = __ldg(src + so + v);
            }
            // release this warp's rows to the tiled loads of heavier units
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) {
                __threadfence();
                release_add_gpu(p.ctr + p.E + 2, 1u);
            }
        }
        const Counts c = unit_counts(p, sm.nused);
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        uint4* stg = sm.stg[warp - 2];
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < c.total(); u += gridDim.x) {
            const DUnit t = decode_dunit(u, p, c, sm);
            int ok = 1;
            if (lane == 0) ok = bounded_wait(tfull_bar(acc), acc_phase, wc) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * ACC_COLS) + (static_cast<uint32_t>(q * 32) << 16);
            const int valid_rows = t.rows - q * 32;
            if (valid_rows > 0 && t.kind <= 1) {
                // h = SiLU(gate) * up as BF16: routed rows into h, shared rows into hs
                const int N = t.kind == 1 ? p.F : p.Fs;
                const size_t pitch = static_cast<size_t>(t.kind == 1 ? p.F : p.S * p.Fs) * 2;
                char* rows = reinterpret_cast<char*>(t.kind == 1 ? p.h : p.hs) +
                             static_cast<size_t>(t.row0 + q * 32) * pitch;
                const int col0 = t.kind == 1 ? t.n0 : t.z * p.Fs + t.n0;
#pragma unroll 1
                for (int cc = half * 64; cc < half * 64 + 64; cc += 32) {
                    uint32_t g0[16], g1[16], u0[16], u1[16];
                    tc_ld_32x32b_x16(tb + cc, g0);
                    tc_ld_32x32b_x16(tb + cc + 16, g1);
                    tc_ld_32x32b_x16(tb + 128 + cc, u0);
                    tc_ld_32x32b_x16(tb + 128 + cc + 16, u1);
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
                    const int vch = (N - (t.n0 + cc)) / 8;
                    warp_store_block(stg, v, lane, rows + static_cast<size_t>(col0 + cc) * 2, pitch, valid_rows, vch);
                }
            } else if (valid_rows > 0) {
                // FP32 rows: routed rows times their gate weight into ys, shared into shout
                const float rs = (t.kind == 3 && lane < valid_rows) ? sm.wloc[t.row0 + q * 32 + lane] : 1.0f;
                const size_t pitch = static_cast<size_t>(p.d) * 4;
                char* rows = reinterpret_cast<char*>(t.kind == 3 ? p.ys : p.shout) +
                             static_cast<size_t>(t.row0 + q * 32) * pitch;
#pragma unroll 1
                for (int cc = half * 128; cc < half * 128 + 128; cc += 16) {
                    uint32_t r0[16];
                    tc_ld_32x32b_x16(tb + cc, r0);
                    tc_wait_ld();
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = rs * __uint_as_float(r0[i]);
                    uint4 blk[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        blk[j] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                            __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                    const int lim = p.d - (t.n0 + cc);
                    const int vch = lim > 0 ? lim * 4 / 16 : 0;
                    warp_store_block(stg, blk, lane, rows + static_cast<size_t>(t.n0 + cc) * 4, pitch, valid_rows, vch);
                }
            }
            tc_fence_before();
            // this warp's stores, then the unit's counter
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(tempty_bar(acc));
                __threadfence();
                release_add_gpu(unit_counter(p, t), 1u);
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    // ---------------- combine: out[t] = sum_k ys[inv[t, k]] + shout[t] ----------------
    __syncthreads();
    __shared__ int comb_ok;
    if (threadIdx.x == 0) {
        const Counts c = unit_counts(p, sm.nused);
        comb_ok = bounded_wait_count(p.ctr + p.E + 1, EPI_WARPS * (c.U3 + c.U4), wc) ? 1 : 0;
    }
    __syncthreads();
    if (comb_ok) {
        const int nchunk = (p.d + 1023) / 1024;  // 1024-column pieces, 4 columns a thread
        for (int pr = blockIdx.x; pr < p.T * nchunk; pr += gridDim.x) {
            const int tt = pr / nchunk;
            const int c0 = (pr - tt * nchunk) * 1024 + 4 * threadIdx.x;
            if (threadIdx.x < 256 && c0 < p.d) {
                float a4[4] = {0.f, 0.f, 0.f, 0.f};
                for (int k = 0; k < p.K; ++k) {
                    const float4 y = __ldcg(reinterpret_cast<const float4*>(
                        p.ys + static_cast<size_t>(sm.invl[tt * p.K + k]) * p.d + c0));
                    a4[0] += y.x;
                    a4[1] += y.y;
                    a4[2] += y.z;
                    a4[3] += y.w;
                }
                if (p.S) {
                    const float4 y = __ldcg(reinterpret_cast<const float4*>(p.shout + static_cast<size_t>(tt) * p.d + c0));
                    a4[0] += y.x;
                    a4[1] += y.y;
                    a4[2] += y.z;
                    a4[3] += y.w;
                }
                const size_t o = static_cast<size_t>(tt) * p.d + c0;
                if (p.out_f32) {
                    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                } else {
                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + o) =
                        make_uint2(pack_bf16x2(a4[0], a4[1]), pack_bf16x2(a4[2], a4[3]));
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// 2-D row-major BF16 [rows, cols] (pitch ld elements), box 64 columns x box_rows.
bool map2d(CUtensorMap* m, const void* base, int rows, int cols, int ld, int box_rows) {
    const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(ld) * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(box_rows)};
    return encode_tmap(m, base, 2, dims, strides, box);
}

// B [Z, K, N] as [Z, N/64 strips, K, 64]: one box = `strips` 64-column strips
// of 64 k rows, landing strip after strip (the layout the MMA reads).
bool map_strips(CUtensorMap* m, const void* B, int Z, int K, int N, int strips) {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(K), static_cast<uint64_t>(N / 64),
                              static_cast<uint64_t>(Z)};
    const uint64_t strides[3] = {static_cast<uint64_t>(N) * 2, 128, static_cast<uint64_t>(K) * N * 2};
    const uint32_t box[4] = {64, 64, static_cast<uint32_t>(strips), 1};
    return encode_tmap(m, B, 4, dims, strides, box);
}

}  // namespace

bool decode_fused_shape_ok(int T, int d, int F, int E, int K, int S, int Fs) {
    return T >= 1 && T <= TC_BM && static_cast<long long>(T) * K <= DISPATCH_CHUNK && E >= 1 &&
           E <= EMAXF && d % 64 == 0 && F % 64 == 0 && (S == 0 || Fs % 64 == 0);
}

cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s) {
    if (!decode_fused_shape_ok(a.T, a.d, a.F, a.E, a.K, a.S, a.Fs)) return cudaErrorInvalidValue;
    DecodeParams p;
    memset(&p, 0, sizeof(p));
    const int TK = a.T * a.K, SF = a.S * a.Fs;
    bool ok = map2d(&p.mapX, a.x, a.T, a.d, a.d, TC_BM) && map2d(&p.mapXg, a.x, a.T, a.d, a.d, 1) &&
              map_strips(&p.mapWg, a.W_gate, a.E, a.d, a.F, 2) &&
              map_strips(&p.mapWu, a.W_up, a.E, a.d, a.F, 2) &&
              map2d(&p.mapH, a.h, TK, a.F, a.F, TC_BM) &&
              map_strips(&p.mapWd, a.W_down, a.E, a.F, a.d, 4) &&
              map2d(&p.mapXs, a.xs, TK, a.d, a.d, TC_BM);
    if (ok && a.S)
        ok = map_strips(&p.mapSg, a.Ws_gate, a.S, a.d, a.Fs, 2) &&
             map_strips(&p.mapSu, a.Ws_up, a.S, a.d, a.Fs, 2) && map2d(&p.mapHs, a.hs, a.T, SF, SF, TC_BM) &&
             map_strips(&p.mapSd, a.Ws_down, 1, SF, a.d, 4);
    if (!ok) return cudaErrorInvalidValue;
    p.idesc = idesc_bf16_f32(TC_BM, 256, /*b_mn_major=*/1);
    p.T = a.T; p.d = a.d; p.F = a.F; p.E = a.E; p.K = a.K; p.S = a.S; p.Fs = a.Fs;
    p.idx = a.idx; p.w = a.w; p.x = a.x;
    p.counts = a.counts; p.offsets = a.offsets; p.mt_prefix = a.mt_prefix;
    p.sorted_token = a.sorted_token; p.sorted_w = a.sorted_w; p.inv = a.inv;
    p.xs = static_cast<__nv_bfloat16*>(a.xs);
    p.h = static_cast<__nv_bfloat16*>(a.h);
    p.hs = static_cast<__nv_bfloat16*>(a.hs);
    p.ys = a.ys; p.shout = a.shout; p.out = a.out; p.out_f32 = a.out_f32;
    p.ctr = a.ctr; p.err = a.err;
    p.timeout_ns = wait_timeout_ns();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const dim3 grid(static_cast<unsigned>(num_sms()));
#define MOE_DF(EM)                                                                                  \
    {                                                                                               \
        static bool attr_set[64] = {};                                                              \
        if (!attr_set[dev]) {                                                                       \
            const cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel<EM>,                     \
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                                       static_cast<int>(smem_bytes<EM>()));         \
            if (e != cudaSuccess) return e;                                                         \
            attr_set[dev] = true;                                                                   \
        }                                                                                           \
        return launch_pdl(decode_fused_kernel<EM>, grid, dim3(THREADS), smem_bytes<EM>(), s, p);   \
    }
    if (a.E <= 64) MOE_DF(64)
    if (a.E <= 128) MOE_DF(128)
    MOE_DF(256)
#undef MOE_DF
}

}  // namespace moe
