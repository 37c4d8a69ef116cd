// Grouped "NT" GEMM on the 5th-generation tensor cores for the backward pass:
//   C[m, n] (+)= sum_k A[m, k] B[n, k]
// with BOTH operands K-major BF16 (rows of K contiguous) - the layout every
// backward contraction has once its operands are laid out for it: the
// transposed weight products dh = gy W_down^T and dz = da W_gate^T + du W_up^T
// read the caller's weights as they are ([E, F, d_e] and [E, d_e, F] rows),
// and the weight gradients read transposed, expert-padded copies of the
// activations that the backward writes for them. FP32 accumulation in tensor
// memory, FP32 output (stored or accumulated).
//
// Ways to cut the work (the forward's grouping, extended to the reduction):
//   NT_MSEG  : the rows of segment z are offsets[z] .. offsets[z+1] (routed
//              rows in expert order); B is the 3-D map's slice z
//   NT_KSEG  : the reduction of segment z runs over columns koff[z] ..
//              koff[z+1] (each a multiple of 64: every expert's rows padded
//              with zero columns); C advanced by z c_zs; an empty segment
//              writes nothing (no gradient for an expert without rows)
//   NT_DENSE : Z problems of one shape; A rows, B rows and B's slice advanced
//              by z a_zrow, z b_zrow, z b_z3; C by z c_zs
// A unit accumulates one or two phases (e.g. da W_gate^T then du W_up^T),
// each with its own pair of tensor maps and coordinate offsets.
// Either operand may instead be stored MN-major (K rows of its M or N
// columns, a_mn / b_mn): the weight gradients then read the row-major
// activations as they are, C = A^T B over the rows (no transposed copies).
//
// Tile 128 x BN (BN = 256 when N >= 256, else 128), K step 64 (a 128-byte
// swizzle row), a 192 KB ring of TMA stages (4 of 48 KB, or 6 of 32 KB), two
// BN-column TMEM accumulators. Warp 0 issues TMA, warp 1 the MMAs
// (tcgen05.mma kind::f16, M = 128, N = BN, both operands K-major), warps 2-9
// drain TMEM (two warps per lane quarter, each half of the columns) and
// write FP32 rows through a per-warp staging buffer, 8 rows x 64 contiguous
// bytes per store. Every wait is bounded; on timeout the CTA stops, drains
// and flags the error word.
// Shapes: every K, N and row count the maps see is handled by TMA bounds and
// masks, but each phase's K must be a multiple of 64 (the caller's choice).
#include "common.cuh"
#include "internal.h"
#include "warp_stage.cuh"

namespace moe {
namespace {

constexpr int NBM = 128, NBK = 64;
constexpr int NT_A_BYTES = NBM * NBK * 2;  // 16 KB
constexpr int NT_THREADS = 320;
constexpr int NT_EPI_WARPS = 8;

template <int BN>
struct NtGeo {
    static constexpr int B_BYTES = BN * NBK * 2;
    static constexpr int STAGE_BYTES = NT_A_BYTES + B_BYTES;
    static constexpr int STAGES = (192 * 1024) / STAGE_BYTES;
    static constexpr int ACC_COLS = BN;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int NBARS = 2 * STAGES + 4 + 1;
    static constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;
    static constexpr int SCHED_OFF = (MISC_OFF + 16 + 15) / 16 * 16;
    static constexpr int STG_OFF = (SCHED_OFF + 2 * (MAXSEG + 1) * 4 + 127) / 128 * 128;
    static constexpr int STG_BYTES = 32 * 16 * 4;  // per epilogue warp: 32 rows x 16 FP32
    static constexpr int SMEM_BYTES = STG_OFF + NT_EPI_WARPS * STG_BYTES + 1024;
};

struct NtParams {
    CUtensorMap mapA[2];
    CUtensorMap mapB[2];
    int nph;
    int a_kofs[2], b_zc[2];
    int mode, M, N, Z, kblocks;
    int a_zrow, b_zrow, b_z3;
    int a_mn, b_mn;  // operand stored MN-major: K rows of its M (N) columns
    const int32_t* offsets;
    float* C;
    long long ldc, c_zs;
    int accumulate;
    // SwiGLU-backward epilogue (NtGemm)
    const __nv_bfloat16* sg_a;
    const __nv_bfloat16* sg_u;
    const int32_t* sg_off;
    long long sg_ld;
    const float* sg_g;
    __nv_bfloat16* sg_da;
    __nv_bfloat16* sg_du;
    __nv_bfloat16* sg_hw;
    float* sg_part;
    int sg_npart;
    uint32_t idesc;
    int* err;
    unsigned long long timeout_ns;
};

struct NtUnit {
    int z, arow, rows, m0, n0, kb0, nkb;
    bool skip;
};

// s_tp: m-tile prefix per segment (NT_MSEG), s_off: offsets (NT_MSEG, NT_KSEG)
template <int NBN>
MOE_DEV NtUnit nt_unit(int u, const NtParams& p, int nt, int mt, const int* s_tp, const int* s_off) {
    NtUnit t;
    t.skip = false;
    if (p.mode == NT_MSEG) {
        const int m = u / nt;
        t.n0 = (u - m * nt) * NBN;
        int lo = 0, hi = p.Z;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_tp[mid] <= m)
                lo = mid;
            else
                hi = mid;
        }
        t.z = lo;
        t.arow = s_off[lo] + (m - s_tp[lo]) * NBM;
        t.rows = min(NBM, s_off[lo + 1] - t.arow);
        t.m0 = t.arow;
        t.kb0 = 0;
        t.nkb = p.kblocks;
    } else {
        const int per = mt * nt;
        t.z = u / per;
        const int rem = u - t.z * per;
        const int m = rem / nt;
        t.m0 = m * NBM;
        t.n0 = (rem - m * nt) * NBN;
        t.rows = min(NBM, p.M - t.m0);
        t.arow = t.m0 + t.z * p.a_zrow;
        if (p.mode == NT_KSEG) {
            t.kb0 = s_off[t.z] / NBK;
            t.nkb = (s_off[t.z + 1] - s_off[t.z]) / NBK;
            t.skip = t.nkb <= 0;
        } else {
            t.kb0 = 0;
            t.nkb = p.kblocks;
        }
    }
    return t;
}

template <int NBN>
__global__ void __launch_bounds__(NT_THREADS, 1) nt_gemm_kernel(const __grid_constant__ NtParams p) {
    using G = NtGeo<NBN>;
    constexpr int NT_STAGES = G::STAGES;
    constexpr int NT_STAGE_BYTES = G::STAGE_BYTES;
    constexpr int NT_ACC_COLS = G::ACC_COLS;
    constexpr int NT_TMEM_COLS = G::TMEM_COLS;
    constexpr int NT_BAR_OFF = G::BAR_OFF;
    constexpr int NT_MISC_OFF = G::MISC_OFF;
    constexpr int NT_SCHED_OFF = G::SCHED_OFF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + NT_BAR_OFF;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (NT_STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * NT_STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * NT_STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * NT_STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + NT_MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + NT_MISC_OFF + 4);
    int* s_tp = reinterpret_cast<int*>(smem + NT_SCHED_OFF);
    int* s_off = s_tp + (MAXSEG + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NT_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), NT_EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0)
        for (int ph = 0; ph < p.nph; ++ph) {
            tma_prefetch_map(&p.mapA[ph]);
            tma_prefetch_map(&p.mapB[ph]);
        }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), NT_TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    if (p.mode != NT_DENSE) {
        for (int i = threadIdx.x; i <= p.Z; i += blockDim.x) s_off[i] = p.offsets[i];
    }
    __syncthreads();
    if (p.mode == NT_MSEG && threadIdx.x == 0) {
        int acc = 0;
        for (int z = 0; z < p.Z; ++z) {
            s_tp[z] = acc;
            acc += (s_off[z + 1] - s_off[z] + NBM - 1) / NBM;
        }
        s_tp[p.Z] = acc;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nt = (p.N + NBN - 1) / NBN;
    const int mt = (p.M + NBM - 1) / NBM;
    const int total = p.mode == NT_MSEG ? s_tp[p.Z] * nt : p.Z * mt * nt;
    const WaitCtx wc{p.err, abort_flag, p.timeout_ns};

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                const NtUnit t = nt_unit<NBN>(u, p, nt, mt, s_tp, s_off);
                if (t.skip) continue;
                const int brow = t.n0 + t.z * p.b_zrow;
                for (int ph = 0; ph < p.nph && ok; ++ph) {
                    const int bz = p.b_zc[ph] + (p.mode == NT_MSEG ? t.z : t.z * p.b_z3);
                    for (int kb = t.kb0; kb < t.kb0 + t.nkb; ++kb) {
                        if (!bounded_wait(empty_bar(stage), phase ^ 1u, wc)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sA = sbase + stage * NT_STAGE_BYTES;
                        mbar_expect_tx(full_bar(stage), NT_STAGE_BYTES);
                        if (p.a_mn)  // two 64-column strips of 64 k rows
                            tma_load_3d(sA, &p.mapA[ph], 0, kb * NBK + p.a_kofs[ph], t.arow / 64, full_bar(stage));
                        else
                            tma_load_2d(sA, &p.mapA[ph], kb * NBK + p.a_kofs[ph], t.arow, full_bar(stage));
                        if (p.b_mn)  // NBN / 64 strips
                            tma_load_3d(sA + NT_A_BYTES, &p.mapB[ph], 0, kb * NBK, brow / 64, full_bar(stage));
                        else
                            tma_load_3d(sA + NT_A_BYTES, &p.mapB[ph], kb * NBK, brow, bz, full_bar(stage));
                        issued |= 1u << stage;
                        last_par = (last_par & ~(1u << stage)) | (phase << stage);
                        if (++stage == NT_STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            for (int s = 0; s < NT_STAGES; ++s)
                if ((issued >> s) & 1u) bounded_drain(full_bar(s), (last_par >> s) & 1u, p.timeout_ns, p.err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            // K-major tiles: rows of 64 k (lbo unused), a 16-deep k-step is 32 bytes;
            // MN-major tiles: 8 KB strips of 64 columns x 64 k rows (lbo = the strip
            // pitch), a 16-deep k-step is 16 rows = 2048 bytes
            const uint64_t adesc0 = smem_desc_sw128(sbase, p.a_mn ? 8192 : 16, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(sbase + NT_A_BYTES, p.b_mn ? 8192 : 16, 1024);
            const uint32_t a_ks = p.a_mn ? 128 : 2, b_ks = p.b_mn ? 128 : 2;  // 16-byte units
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                const NtUnit t = nt_unit<NBN>(u, p, nt, mt, s_tp, s_off);
                if (t.skip) continue;
                if (!bounded_wait(tempty_bar(acc), acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NT_ACC_COLS);
                const int nkb = t.nkb * p.nph;
                for (int i = 0; i < nkb; ++i) {
                    if (!bounded_wait(full_bar(stage), phase, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t soff = static_cast<uint64_t>(stage * NT_STAGE_BYTES) >> 4;
#pragma unroll
                    for (int ks = 0; ks < NBK / 16; ++ks) {
                        const uint32_t accum = (i != 0 || ks != 0) ? 1u : 0u;
                        tc_mma_bf16(d_tmem, adesc0 + soff + ks * a_ks, bdesc0 + soff + ks * b_ks, p.idesc,
                                    accum);
                    }
                    tc_commit(empty_bar(stage));
                    if (++stage == NT_STAGES) {
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
        const int q = warp & 3;            // TMEM lane quarter of this warp
        const int half = (warp - 2) >> 2;  // which half of the tile's columns
        // staging: a row's 16 values in, then 8 rows x 64 contiguous bytes per
        // store instruction out (16-byte slots XOR-swizzled by row: both
        // directions bank-conflict free)
        float4* stg = reinterpret_cast<float4*>(smem + G::STG_OFF + (warp - 2) * G::STG_BYTES);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const NtUnit t = nt_unit<NBN>(u, p, nt, mt, s_tp, s_off);
            if (t.skip) continue;
            int ok = 1;
            if (lane == 0) ok = bounded_wait(tfull_bar(acc), acc_phase, wc) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * NT_ACC_COLS) +
                                (static_cast<uint32_t>(q * 32) << 16);
            if (p.sg_a != nullptr) {
                // SwiGLU backward, 32 columns at a time: a and u of the warp's 32 rows
                // come in and da, du, g h go out as row-major 64-byte row segments
                // through the warp's staging buffer; lane = row in between
                uint4* stg4 = reinterpret_cast<uint4*>(stg);
                const int wr0 = t.m0 + q * 32;                        // the warp's first row
                const int tile_rows = max(0, min(32, t.rows - q * 32));  // rows written
                int real_rows = tile_rows;                            // rows with a and u
                long long arow0 = wr0;
                if (p.mode == NT_MSEG) {
                    const int i0 = wr0 - s_off[t.z];
                    real_rows = max(0, min(tile_rows, p.sg_off[t.z + 1] - p.sg_off[t.z] - i0));
                    arow0 = p.sg_off[t.z] + i0;
                }
                const bool real = lane < real_rows;
                const float g = (real && p.sg_g != nullptr) ? p.sg_g[arow0 + lane] : 1.0f;
                const long long obase = (p.mode == NT_MSEG ? 0 : t.z * p.c_zs) + static_cast<long long>(wr0) * p.ldc + t.n0;
                const long long abase = p.mode == NT_MSEG ? arow0 * p.sg_ld + t.n0 : obase;
                const size_t apitch = static_cast<size_t>(p.mode == NT_MSEG ? p.sg_ld : p.ldc) * 2;
                const size_t opitch = static_cast<size_t>(p.ldc) * 2;
                float part = 0.0f;
                const int c_beg = half * (NBN / 2), c_end = (half + 1) * (NBN / 2);
                // a and u of a 32-column block: both arrays' loads in flight together
                // (N is a multiple of 64: a block is wholly inside or outside it)
                const char* a_row0 = reinterpret_cast<const char*>(p.sg_a + abase);
                const char* u_row0 = reinterpret_cast<const char*>(p.sg_u + abase);
#pragma unroll 1
                for (int c = c_beg; c < c_end; c += 32) {
                    const bool col_ok = t.n0 + c < p.N;
                    uint32_t v0[16], v1[16];
                    tc_ld_32x32b_x16(tb + c, v0);
                    tc_ld_32x32b_x16(tb + c + 16, v1);
                    uint4 av[4], uv[4];
                    {
                        uint4 wa[4], wu[4];
                        warp_load_issue(wa, lane, a_row0 + 2 * c, apitch, col_ok ? real_rows : 0);
                        warp_load_issue(wu, lane, u_row0 + 2 * c, apitch, col_ok ? real_rows : 0);
                        warp_load_finish(stg4, wa, av, lane);
                        warp_load_finish(stg4, wu, uv, lane);
                    }
                    tc_wait_ld();
                    const uint32_t* aw = reinterpret_cast<const uint32_t*>(av);
                    const uint32_t* uw = reinterpret_cast<const uint32_t*>(uv);
                    uint32_t pda[16], pdu[16], phw[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float o_da[2], o_du[2], o_hw[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float a = e ? bf16_hi(aw[j]) : bf16_lo(aw[j]);
                            const float uu = e ? bf16_hi(uw[j]) : bf16_lo(uw[j]);
                            const float dv = __uint_as_float(j < 8 ? v0[2 * j + e] : v1[2 * j - 16 + e]);
                            const float sg = 1.0f / (1.0f + expf(-a));
                            const float si = a * sg;
                            const float h = si * uu;
                            o_da[e] = real ? g * dv * uu * (sg * (1.0f + a * (1.0f - sg))) : 0.0f;
                            o_du[e] = real ? g * dv * si : 0.0f;
                            o_hw[e] = real ? g * h : 0.0f;
                            part += real ? dv * h : 0.0f;
                        }
                        pda[j] = pack_bf16x2(o_da[0], o_da[1]);
                        pdu[j] = pack_bf16x2(o_du[0], o_du[1]);
                        phw[j] = pack_bf16x2(o_hw[0], o_hw[1]);
                    }
                    const int wrows = col_ok ? tile_rows : 0;
                    const uint4 vd[4] = {make_uint4(pda[0], pda[1], pda[2], pda[3]), make_uint4(pda[4], pda[5], pda[6], pda[7]),
                                         make_uint4(pda[8], pda[9], pda[10], pda[11]), make_uint4(pda[12], pda[13], pda[14], pda[15])};
                    warp_store_block(stg4, vd, lane, reinterpret_cast<char*>(p.sg_da + obase + c), opitch, wrows, 4);
                    const uint4 vu[4] = {make_uint4(pdu[0], pdu[1], pdu[2], pdu[3]), make_uint4(pdu[4], pdu[5], pdu[6], pdu[7]),
                                         make_uint4(pdu[8], pdu[9], pdu[10], pdu[11]), make_uint4(pdu[12], pdu[13], pdu[14], pdu[15])};
                    warp_store_block(stg4, vu, lane, reinterpret_cast<char*>(p.sg_du + obase + c), opitch, wrows, 4);
                    const uint4 vh[4] = {make_uint4(phw[0], phw[1], phw[2], phw[3]), make_uint4(phw[4], phw[5], phw[6], phw[7]),
                                         make_uint4(phw[8], phw[9], phw[10], phw[11]), make_uint4(phw[12], phw[13], phw[14], phw[15])};
                    warp_store_block(stg4, vh, lane, reinterpret_cast<char*>(p.sg_hw + obase + c), opitch, wrows, 4);
                    if (((t.n0 + c + 32) & 63) == 0) {
                        // a 64-column group is complete
                        if (real && col_ok && p.sg_part != nullptr)
                            p.sg_part[(arow0 + lane) * p.sg_npart + (t.n0 + c) / 64] = part;
                        part = 0.0f;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
                continue;
            }
            float* cbase = p.C + (p.mode == NT_MSEG ? 0 : t.z * p.c_zs);
#pragma unroll 1
            for (int c = half * (NBN / 2); c < (half + 1) * (NBN / 2); c += 16) {
                uint32_t v[16];
                tc_ld_32x32b_x16(tb + c, v);
                tc_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    stg[lane * 4 + (j ^ ((lane >> 1) & 3))] =
                        make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                    __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                __syncwarp();
                if (t.n0 + c < p.N) {
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int rr = it * 8 + (lane >> 2), qq = lane & 3;
                        const int r = q * 32 + rr;
                        if (r < t.rows) {
                            float4 o = stg[rr * 4 + (qq ^ ((rr >> 1) & 3))];
                            float4* dst = reinterpret_cast<float4*>(
                                              cbase + static_cast<long long>(t.m0 + r) * p.ldc + t.n0 + c) +
                                          qq;
                            if (p.accumulate) {
                                const float4 a = *dst;
                                o.x += a.x;
                                o.y += a.y;
                                o.z += a.z;
                                o.w += a.w;
                            }
                            *dst = o;
                        }
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, NT_TMEM_COLS);
    }
}

// MN-major operand: K rows of `cols` columns (pitch ld), seen as
// [cols/64 strips, K, 64]; a box is `strips` strips of 64 k rows (8 KB each),
// the layout the MMA reads as an MN-major tile.
bool make_nt_strips(CUtensorMap* m, const void* X, long long cols, long long K, long long ld, int strips) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(K), static_cast<uint64_t>(cols / 64)};
    const uint64_t strides[2] = {static_cast<uint64_t>(ld) * 2, 128};
    const uint32_t box[3] = {64, NBK, static_cast<uint32_t>(strips)};
    return encode_tmap(m, X, 3, dims, strides, box);
}

// A: rows x K_total, row pitch lda elements (K-major), box 64 x 128 rows
bool make_nt_A(CUtensorMap* m, const void* A, long long rows, long long K, long long lda) {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(lda) * 2};
    const uint32_t box[2] = {NBK, NBM};
    return encode_tmap(m, A, 2, dims, strides, box);
}

// B: Z slices of rows x K (K-major), row pitch ldb, slice pitch zstride elements; box 64 x bn rows
bool make_nt_B(CUtensorMap* m, const void* B, long long Z, long long rows, long long K, long long ldb,
               long long zstride, int bn) {
    const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows),
                              static_cast<uint64_t>(Z)};
    const uint64_t strides[2] = {static_cast<uint64_t>(ldb) * 2, static_cast<uint64_t>(zstride) * 2};
    const uint32_t box[3] = {NBK, static_cast<uint32_t>(bn), 1};
    return encode_tmap(m, B, 3, dims, strides, box);
}


template <int NBN>
cudaError_t launch_nt_t(const NtGemm& g, cudaStream_t s) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidValue;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(nt_gemm_kernel<NBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 NtGeo<NBN>::SMEM_BYTES) != cudaSuccess)
            return cudaErrorInvalidValue;
        attr_set[dev] = true;
    }
    NtParams p;
    memset(&p, 0, sizeof(p));
    for (int ph = 0; ph < g.nph; ++ph) {
        const NtOperand& a = g.A[ph];
        const NtOperand& b = g.B[ph];
        if (g.a_mn ? !make_nt_strips(&p.mapA[ph], a.p, a.rows, a.K, a.ld, NBM / 64)
                   : !make_nt_A(&p.mapA[ph], a.p, a.rows, a.K, a.ld))
            return cudaErrorInvalidValue;
        if (g.b_mn ? !make_nt_strips(&p.mapB[ph], b.p, b.rows, b.K, b.ld, NBN / 64)
                   : !make_nt_B(&p.mapB[ph], b.p, b.Z > 0 ? b.Z : 1, b.rows, b.K, b.ld, b.zstride, NBN))
            return cudaErrorInvalidValue;
        p.a_kofs[ph] = g.a_kofs[ph];
        p.b_zc[ph] = g.b_zc[ph];
    }
    p.nph = g.nph;
    p.mode = g.mode;
    p.M = g.M;
    p.N = g.N;
    p.Z = g.Z;
    p.kblocks = g.K / NBK;
    p.a_zrow = g.a_zrow;
    p.b_zrow = g.b_zrow;
    p.b_z3 = g.b_z3;
    p.a_mn = g.a_mn;
    p.b_mn = g.b_mn;
    p.offsets = g.offsets;
    p.C = g.C;
    p.ldc = g.ldc;
    p.c_zs = g.c_zs;
    p.accumulate = g.accumulate;
    p.sg_a = g.sg_a;
    p.sg_u = g.sg_u;
    p.sg_off = g.sg_off;
    p.sg_ld = g.sg_ld;
    p.sg_g = g.sg_g;
    p.sg_da = g.sg_da;
    p.sg_du = g.sg_du;
    p.sg_hw = g.sg_hw;
    p.sg_part = g.sg_part;
    p.sg_npart = g.sg_npart;
    p.idesc = idesc_bf16_f32(NBM, NBN, g.b_mn ? 1 : 0) | (g.a_mn ? (1u << 15) : 0u);  // bit 15: A MN-major
    p.err = g.err;
    p.timeout_ns = wait_timeout_ns();
    const long long nt = (g.N + NBN - 1) / NBN;
    long long units;
    if (g.mode == NT_MSEG)
        units = ((g.M + NBM - 1) / NBM + g.Z) * nt;
    else
        units = static_cast<long long>(g.Z) * ((g.M + NBM - 1) / NBM) * nt;
    long long grid = num_sms();
    if (units < grid) grid = units;
    if (grid < 1) grid = 1;
    return launch_pdl(nt_gemm_kernel<NBN>, dim3(static_cast<unsigned>(grid)), dim3(NT_THREADS),
                      NtGeo<NBN>::SMEM_BYTES, s, p);
}

}  // namespace

cudaError_t launch_nt_gemm(const NtGemm& g, cudaStream_t s) {
    if (g.nph < 1 || g.nph > 2 || g.Z < 1 || (g.mode != NT_DENSE && g.Z > MAXSEG))
        return cudaErrorInvalidValue;
    if (g.N % 16 || g.K % NBK) return cudaErrorInvalidValue;
    if (g.sg_a != nullptr) {
        // SwiGLU-backward epilogue: BF16 rows of 16-byte aligned 16-column blocks
        if (!g.sg_u || !g.sg_da || !g.sg_du || !g.sg_hw || g.N % 64 || g.ldc % 8 || g.c_zs % 8 ||
            g.mode == NT_KSEG || (g.mode == NT_MSEG && (!g.sg_off || g.sg_ld % 8)) ||
            (g.sg_part != nullptr && g.sg_npart < (g.N + 63) / 64))
            return cudaErrorInvalidValue;
    }
    // MN-major operands: whole 64-column strips, no row segments, no B slices
    for (int ph = 0; ph < g.nph; ++ph) {
        if (g.a_mn && (g.mode == NT_MSEG || g.A[ph].rows % 64 || g.A[ph].ld % 8 || g.a_zrow % 64))
            return cudaErrorInvalidValue;
        if (g.b_mn && (g.B[ph].rows % 64 || g.B[ph].ld % 8 || g.b_zrow % 64 || g.b_z3 || g.b_zc[ph] ||
                       g.mode == NT_MSEG))
            return cudaErrorInvalidValue;
    }
    // 128 x 256 tiles halve the A re-reads, but only while they still give
    // every SM a unit, and (grouped by expert) while the segments average 256
    // rows or more: short segments stream weights or store FP32 gradients,
    // which narrower tiles spread over more SMs
    bool wide = g.N >= 256;
    if (g.mode == NT_MSEG) {
        wide = wide && static_cast<long long>(g.M) >= 256LL * g.Z;
    } else if (g.mode == NT_KSEG && static_cast<long long>(g.K) < 256LL * g.Z) {
        wide = false;  // short reductions: the tiles' FP32 stores dominate; spread them
    } else {
        const long long units256 = static_cast<long long>(g.Z) * ((g.M + NBM - 1) / NBM) * ((g.N + 255) / 256);
        wide = wide && units256 >= num_sms();
    }
    return wide ? launch_nt_t<256>(g, s) : launch_nt_t<128>(g, s);
}

}  // namespace moe
