// Backward pass of the layer: gradients of L = sum(dout * out) with the
// routing of the forward held fixed (the top-K selection carries no
// gradient). Source: kimi_k3 StableLatentMoE, "The actual grouped GEMM, and
// the gradient path" (backpropagation through the scatter, both grouped GEMMs
// and the gate weights to the selected router scores) and "Grouped expert
// execution and sparse gradients" (experts without rows get no gradient); the
// forward it differentiates is APEX-1 Mathematical Reference Part 3, sections
// 12.2 and 13.2.
//
// Per routed assignment at sorted position pos (token t, expert e, gate g)
// with upstream gy = dout[t] (latent: dout[t] W_up_latent^T):
//   dh' = gy W_down[e]^T                          (G1, unweighted)
//   a, u = z W_gate[e], z W_up[e] (recomputed), h = SiLU(a) u
//   da = g dh' u SiLU'(a), du = g dh' SiLU(a)     (SwiGLU backward epilogue)
//   dg = sum dh' h  (= gy . y)                    (gate weight gradient)
//   dz = da W_gate[e]^T + du W_up[e]^T            (G3)
//   dW_down[e] += (g h)^T gy, dW_gate[e] += z^T da, dW_up[e] += z^T du
// The shared experts the same with g = 1 on every token; the router logits
// get dr from dg through the gate mode's formula, dW_router = x^T dr and
// dx += dr W_router^T; the latent projections their two GEMMs. All sums are
// plain stores and accumulations in a fixed order: the result is
// reproducible bit for bit. This first form runs every contraction on the
// CUDA cores in FP32 (gemm_gen.cu), BF16 operands converted exactly.
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// dr[t, :] from the gate-weight gradients of token t, one warp per token.
// dg of slot k is the fixed-order sum of the SwiGLU epilogue's column-tile
// partials of its sorted position. Softmax modes (both select on and weight
// by a softmax over the selected logits): dr_e(k) = g_k (dg_k - sum_j g_j dg_j).
// Sigmoid: ds_k = scale dg_k, renormalised: scale (dg_k - sum_j dg_j s_j / S) / S
// with S = sum_j s_j; dr = ds s (1 - s). Unselected experts: 0.
__global__ void __launch_bounds__(256) router_bwd_kernel(const float* __restrict__ dwpart, int ntf,
                                                         const int32_t* __restrict__ inv,
                                                         const int32_t* __restrict__ idx,
                                                         const float* __restrict__ w,
                                                         const float* __restrict__ scores, int T,
                                                         int K, int E, int gate, int renorm,
                                                         float scale, float* __restrict__ dr,
                                                         float* __restrict__ dg_out,
                                                         float* __restrict__ cp,
                                                         const int32_t* __restrict__ invp,
                                                         const float* __restrict__ WrT, int d,
                                                         float* __restrict__ dx) {
    pdl_wait();
    pdl_trigger();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    float dg = 0.0f, gk = 0.0f, sk = 0.0f;
    int ek = 0;
    if (lane < K) {
        const int pos = inv[static_cast<size_t>(t) * K + lane];
        const float* pp = dwpart + static_cast<size_t>(pos) * ntf;
        for (int i = 0; i < ntf; ++i) dg += pp[i];
        ek = idx[static_cast<size_t>(t) * K + lane];
        gk = w[static_cast<size_t>(t) * K + lane];
        if (gate == MOE_GATE_SIGMOID) sk = scores[static_cast<size_t>(t) * E + ek];
        if (dg_out != nullptr) dg_out[static_cast<size_t>(t) * K + lane] = dg;
    }
    float drk;
    if (gate == MOE_GATE_SIGMOID) {
        float ds;
        if (renorm) {
            float S = lane < K ? sk : 0.0f, sd = lane < K ? dg * sk : 0.0f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                S += __shfl_xor_sync(0xffffffffu, S, o);
                sd += __shfl_xor_sync(0xffffffffu, sd, o);
            }
            ds = scale * (dg - sd / S) / S;
        } else {
            ds = scale * dg;
        }
        drk = ds * sk * (1.0f - sk);
    } else {
        float sgd = lane < K ? gk * dg : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sgd += __shfl_xor_sync(0xffffffffu, sgd, o);
        drk = gk * (dg - sgd);
    }
    float* row = dr + static_cast<size_t>(t) * E;
    for (int e = lane; e < E; e += 32) row[e] = 0.0f;
    __syncwarp();
    if (lane < K) row[ek] = drk;
    // the router's coefficient of each assignment at its expert-padded row
    if (cp != nullptr && lane < K) cp[invp[static_cast<size_t>(t) * K + lane]] = drk;
    // dx[t, :] += sum_k dr_k W_router[:, e_k] (slot order), from W_router^T rows
    if (WrT != nullptr) {
        float* xr = dx + static_cast<size_t>(t) * d;
        for (int j = lane; j < d; j += 32) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                const float dk = __shfl_sync(0xffffffffu, drk, k);
                const int e = __shfl_sync(0xffffffffu, ek, k);
                acc = fmaf(dk, WrT[static_cast<size_t>(e) * d + j], acc);
            }
            xr[j] += acc;
        }
    }
}

// Partial router weight gradients over 64 expert-padded rows (all of one
// expert): part[chunk, j] = sum over the chunk's rows k (in order) of
// rows[k, j] cp[k]; cp is zero on padding rows.
__global__ void __launch_bounds__(256) router_wgrad_part_kernel(const __nv_bfloat16* __restrict__ rows,
                                                                const float* __restrict__ cp, int d,
                                                                float* __restrict__ part) {
    pdl_wait();
    pdl_trigger();
    const int j = blockIdx.y * 256 + threadIdx.x;
    const int k0 = blockIdx.x * 64;
    __shared__ float c[64];
    if (threadIdx.x < 64) c[threadIdx.x] = cp[k0 + threadIdx.x];
    __syncthreads();
    if (j >= d) return;
    float acc = 0.0f;
#pragma unroll 8
    for (int k = 0; k < 64; ++k)
        acc = fmaf(__bfloat162float(rows[static_cast<size_t>(k0 + k) * d + j]), c[k], acc);
    part[static_cast<size_t>(blockIdx.x) * d + j] = acc;
}

// dW_router[j, e] = sum over expert e's chunks (in order) of part[chunk, j].
__global__ void __launch_bounds__(256) router_wgrad_reduce_kernel(const float* __restrict__ part,
                                                                  const int32_t* __restrict__ poff,
                                                                  int d, int E,
                                                                  float* __restrict__ dW) {
    pdl_wait();
    pdl_trigger();
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<long long>(d) * E) return;
    const int j = static_cast<int>(i / E), e = static_cast<int>(i - static_cast<long long>(j) * E);
    float v = 0.0f;
    for (int ch = poff[e] / 64; ch < poff[e + 1] / 64; ++ch) v += part[static_cast<size_t>(ch) * d + j];
    dW[i] = v;
}

// out [cols, rows] = in [rows, cols]^T, FP32, 32 x 32 tiles.
__global__ void __launch_bounds__(256) transpose_f32_kernel(const float* __restrict__ in, int rows,
                                                            int cols, float* __restrict__ out) {
    __shared__ float tile[32][33];
    pdl_wait();
    pdl_trigger();
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < 32; r += 8)
        if (r0 + r < rows && c0 + tx < cols) tile[r][tx] = in[static_cast<size_t>(r0 + r) * cols + c0 + tx];
    __syncthreads();
    for (int c = ty; c < 32; c += 8)
        if (c0 + c < cols && r0 + tx < rows) out[static_cast<size_t>(c0 + c) * rows + r0 + tx] = tile[tx][c];
}

GenOp op(const void* p, int bf16, long long s0, long long s1, long long zs = 0,
         const int32_t* idx0 = nullptr, const int32_t* idx1 = nullptr) {
    GenOp o;
    o.p = p;
    o.bf16 = bf16;
    o.s0 = s0;
    o.s1 = s1;
    o.zs = zs;
    o.idx0 = idx0;
    o.idx1 = idx1;
    return o;
}

GenGemm gemm(int mode, int M, int N, int K, int Z, GenOp A, int a_m_contig, GenOp B,
             int b_n_contig, float* C, long long ldc, long long c_zs = 0,
             const int32_t* offsets = nullptr) {
    GenGemm g;
    memset(&g, 0, sizeof(g));
    g.mode = mode;
    g.offsets = offsets;
    g.M = M;
    g.N = N;
    g.K = K;
    g.Z = Z;
    g.A = A;
    g.B0 = B;
    g.B1 = B;
    g.a_m_contig = a_m_contig;
    g.b_n_contig = b_n_contig;
    g.C = C;
    g.ldc = ldc;
    g.c_zs = c_zs;
    return g;
}

// A dense CUDA-core product whose reduction runs over the tokens (weight
// gradients of the router and the latent projections): split-K into `part`.
cudaError_t run_splitk(GenGemm g, int epi, float* part, size_t part_floats, cudaStream_t s) {
    g.ksplit = gen_gemm_ksplit(g, part_floats);
    g.part = part;
    return launch_gen_gemm(g, epi, s);
}

const void* offset_elems(const void* p, long long n, int bf16) {
    return static_cast<const uint8_t*>(p) + n * (bf16 ? 2 : 4);
}

}  // namespace

bool bwd_on_tensor_cores(const moe_config& c) {
    const int de = c.latent_dim ? c.latent_dim : c.d;
    return c.dtype == MOE_BF16 && c.d % 64 == 0 && c.d_ff % 64 == 0 && de % 64 == 0 &&
           (c.n_shared == 0 || c.shared_d_ff % 64 == 0);
}

BwdLayout plan_backward(const moe_config& c) {
    BwdLayout B;
    memset(&B, 0, sizeof(B));
    const size_t T = c.T, TK = T * c.K, F = c.d_ff, E = c.E;
    const size_t de = c.latent_dim ? c.latent_dim : c.d;
    const size_t SF = static_cast<size_t>(c.n_shared) * (c.n_shared ? c.shared_d_ff : 0);
    const size_t L = c.latent_dim;
    const size_t ntf = gen_gemm_ntiles(c.d_ff);
    B.tc = bwd_on_tensor_cores(c) ? 1 : 0;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + bytes + 255) & ~static_cast<size_t>(255);
        return at;
    };
    B.dxs = take(TK * de * 4);
    {
        const size_t plane = std::max(static_cast<size_t>(c.d) * E, static_cast<size_t>(c.d) * L);
        B.kpart_floats = std::min<size_t>(size_t(4) << 20, 64 * plane);
        B.kpart = take(B.kpart_floats * 4);
    }
    B.dr = take(T * E * 4);
    B.dg = take(TK * 4);
    B.glat = L ? take(T * L * 4) : 0;
    B.routed = L ? take(T * L * 4) : 0;
    B.dz = L ? take(T * L * 4) : 0;
    if (!B.tc) {
        B.dhp = take(TK * F * 4);
        B.da = take(TK * F * 4);
        B.du = take(TK * F * 4);
        B.hw = take(TK * F * 4);
        B.dwpart = take(TK * ntf * 4);
        B.dhs = SF ? take(T * SF * 4) : 0;
        B.das = SF ? take(T * SF * 4) : 0;
        B.dus = SF ? take(T * SF * 4) : 0;
        B.hs = SF ? take(T * SF * 4) : 0;
    } else {
        // expert-padded row layout: each expert's rows, then zero rows up to a multiple of 64
        B.tkpad = static_cast<long long>((TK + 63) / 64 * 64 + 64 * E);  // >= padded total
        B.tpad = static_cast<long long>((T + 63) / 64 * 64);
        const size_t kp = static_cast<size_t>(B.tkpad);
        B.poff = take((E + 1) * 4);
        B.invp = take(TK * 4);
        B.gys = take(kp * de * 2);
        B.zs = take(kp * de * 2);
        B.saved = c.save_gate_up != 0;  // the forward kept the gate / up products
        B.dhp = B.saved ? 0 : take(kp * F * 4);
        B.dab = take(kp * F * 2);
        B.dub = take(kp * F * 2);
        B.hwb = take(kp * F * 2);
        B.dwrow = take(TK * 2 * ((F + 127) / 128) * 4);  // per-row partials of dg, one per 64 columns
                                                           // (>= F / 64 of them)
        B.dxsp = take(kp * de * 4);
        B.wrt = take(static_cast<size_t>(c.d) * E * 4);
        B.cp = take(kp * 4);
        B.rpart = take(kp / 64 * c.d * 4);
        if (SF || L) B.doutb = take(T * c.d * 2);
        if (L) {
            B.routedb = take(T * L * 2);
            B.dzb = take(T * L * 2);
        }
        if (SF) {
            B.dhs = B.saved ? 0 : take(T * SF * 4);
            B.dasb = take(T * SF * 2);
            B.dusb = take(T * SF * 2);
            B.hsb = take(T * SF * 2);
        }
    }
    B.total = o;
    return B;
}

static moe_status backward_tc(const moe_config& c, const void* x, const moe_weights& w,
                              const float* dout, const moe_grads& gr, uint8_t* ws, uint8_t* bws,
                              cudaStream_t s);

moe_status backward_impl(const moe_config& c, const void* x, const moe_weights& w, const float* dout,
                         const moe_grads& gr, uint8_t* ws, uint8_t* bws, cudaStream_t s) {
    const WsLayout L = plan_workspace(c);
    const BwdLayout BL = plan_backward(c);
    if (BL.tc) return backward_tc(c, x, w, dout, gr, ws, bws, s);
    const int bf = c.dtype == MOE_BF16 ? 1 : 0;
    const int T = c.T, K = c.K, E = c.E, TK = T * K, F = c.d_ff, d = c.d;
    const int lat = c.latent_dim, de = lat ? lat : d;
    const int S = c.n_shared, Fs = S ? c.shared_d_ff : 0, SF = S * Fs;
    auto WP = [&](size_t off) { return static_cast<void*>(ws + off); };
    auto BP = [&](size_t off) { return reinterpret_cast<float*>(bws + off); };
    const int32_t* stok = static_cast<const int32_t*>(WP(L.sorted_token));
    const float* sw = static_cast<const float*>(WP(L.sorted_w));
    const int32_t* inv = static_cast<const int32_t*>(WP(L.inv));
    const int32_t* offsets = static_cast<const int32_t*>(WP(L.offsets));
    const int32_t* tidx = static_cast<const int32_t*>(WP(L.topk_idx));
    const float* tw = static_cast<const float*>(WP(L.topk_w));
    const float* scores = L.scores ? static_cast<const float*>(WP(L.scores)) : nullptr;
    float *dhp = BP(BL.dhp), *da = BP(BL.da), *du = BP(BL.du), *hw = BP(BL.hw);
    float *dwpart = BP(BL.dwpart), *dxs = BP(BL.dxs), *dr = BP(BL.dr), *dg = BP(BL.dg);
    const int ntf = gen_gemm_ntiles(F);
    cudaError_t e;
#define RUN(G, EPI)                                                      \
    do {                                                                 \
        if ((e = launch_gen_gemm((G), (EPI), s)) != cudaSuccess) return MOE_ERR_CUDA; \
    } while (0)

    // upstream gradient of the routed sum, and the rows the experts act on
    const float* gy = dout;
    long long ld_gy = d;
    const void* zsrc = x;
    long long ld_z = d;
    int z_bf = bf;
    if (lat) {
        float* glat = BP(BL.glat);
        float* routed = BP(BL.routed);
        // gy = dout W_up_latent^T
        RUN(gemm(GEN_DENSE, T, lat, d, 1, op(dout, 0, d, 1), 0, op(w.W_up_latent, bf, 1, d), 0,
                 glat, lat),
            GEN_EPI_STORE);
        if (gr.dW_up_latent) {
            // routed sum of the forward (latent width), then dW_up_latent = routed^T dout
            if ((e = launch_gather_sum(static_cast<const float*>(WP(L.ys)), inv, T, K, lat, nullptr,
                                       routed, 0, s)) != cudaSuccess)
                return MOE_ERR_CUDA;
            if ((e = run_splitk(gemm(GEN_DENSE, lat, d, T, 1, op(routed, 0, 1, lat), 1,
                                     op(dout, 0, d, 1), 1, gr.dW_up_latent, d),
                                GEN_EPI_STORE, BP(BL.kpart), BL.kpart_floats, s)) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        gy = glat;
        ld_gy = lat;
        zsrc = WP(L.z);
        ld_z = lat;
        z_bf = 1;
    }

    // routed experts
    // G1: dh' = gy[tok] W_down[e]^T
    RUN(gemm(GEN_MSEG, TK, F, de, E, op(gy, 0, ld_gy, 1, 0, stok), 0,
             op(w.W_down, bf, 1, de, static_cast<long long>(F) * de), 0, dhp, F, 0, offsets),
        GEN_EPI_STORE);
    // a, u recomputed; SwiGLU backward with the gate weights
    {
        GenGemm g = gemm(GEN_MSEG, TK, F, de, E, op(zsrc, z_bf, ld_z, 1, 0, stok), 0,
                         op(w.W_gate, bf, F, 1, static_cast<long long>(de) * F), 1, nullptr, F);
        g.B1 = op(w.W_up, bf, F, 1, static_cast<long long>(de) * F);
        g.offsets = offsets;
        g.rowscale = sw;
        g.dh = dhp;
        g.da = da;
        g.du = du;
        g.hw = hw;
        g.dwpart = dwpart;
        RUN(g, GEN_EPI_SWIGLU_BWD);
    }
    // G3: dz rows = da W_gate[e]^T + du W_up[e]^T
    {
        GenGemm g = gemm(GEN_MSEG, TK, de, F, E, op(da, 0, F, 1), 0,
                         op(w.W_gate, bf, 1, F, static_cast<long long>(de) * F), 0, dxs, de);
        g.offsets = offsets;
        RUN(g, GEN_EPI_STORE);
        g.A = op(du, 0, F, 1);
        g.B0 = op(w.W_up, bf, 1, F, static_cast<long long>(de) * F);
        RUN(g, GEN_EPI_ACCUM);
    }
    // expert weight gradients, reduced over each expert's rows
    if (gr.dW_down) {
        GenGemm g = gemm(GEN_KSEG, F, de, TK, E, op(hw, 0, 1, F), 1,
                         op(gy, 0, ld_gy, 1, 0, stok), 1, gr.dW_down, de,
                         static_cast<long long>(F) * de);
        g.offsets = offsets;
        RUN(g, GEN_EPI_STORE);
    }
    if (gr.dW_gate || gr.dW_up) {
        GenGemm g = gemm(GEN_KSEG, de, F, TK, E, op(zsrc, z_bf, 1, ld_z, 0, nullptr, stok), 1,
                         op(da, 0, F, 1), 1, gr.dW_gate, F, static_cast<long long>(de) * F);
        g.offsets = offsets;
        if (gr.dW_gate) RUN(g, GEN_EPI_STORE);
        g.B0 = op(du, 0, F, 1);
        g.C = gr.dW_up;
        if (gr.dW_up) RUN(g, GEN_EPI_STORE);
    }

    // dx from the routed experts (latent: through dz and W_down_latent)
    if (!lat) {
        if ((e = launch_gather_sum(dxs, inv, T, K, d, nullptr, gr.dx, 0, s)) != cudaSuccess)
            return MOE_ERR_CUDA;
    } else {
        float* dz = BP(BL.dz);
        if ((e = launch_gather_sum(dxs, inv, T, K, lat, nullptr, dz, 0, s)) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (gr.dW_down_latent &&
            (e = run_splitk(gemm(GEN_DENSE, d, lat, T, 1, op(x, bf, 1, d), 1, op(dz, 0, lat, 1), 1,
                                 gr.dW_down_latent, lat),
                            GEN_EPI_STORE, BP(BL.kpart), BL.kpart_floats, s)) != cudaSuccess)
            return MOE_ERR_CUDA;
        RUN(gemm(GEN_DENSE, T, d, lat, 1, op(dz, 0, lat, 1), 0, op(w.W_down_latent, bf, 1, lat), 0,
                 gr.dx, d),
            GEN_EPI_STORE);
    }

    // shared experts (g = 1 on every token)
    if (S) {
        float *dhs = BP(BL.dhs), *das = BP(BL.das), *dus = BP(BL.dus), *hs = BP(BL.hs);
        RUN(gemm(GEN_DENSE, T, Fs, d, S, op(dout, 0, d, 1), 0,
                 op(w.Ws_down, bf, 1, d, static_cast<long long>(Fs) * d), 0, dhs, SF, Fs),
            GEN_EPI_STORE);
        {
            GenGemm g = gemm(GEN_DENSE, T, Fs, d, S, op(x, bf, d, 1), 0,
                             op(w.Ws_gate, bf, Fs, 1, static_cast<long long>(d) * Fs), 1, nullptr,
                             SF, Fs);
            g.B1 = op(w.Ws_up, bf, Fs, 1, static_cast<long long>(d) * Fs);
            g.dh = dhs;
            g.da = das;
            g.du = dus;
            g.hw = hs;
            RUN(g, GEN_EPI_SWIGLU_BWD);
        }
        for (int z = 0; z < S; ++z) {
            const long long wz = static_cast<long long>(z) * d * Fs;
            RUN(gemm(GEN_DENSE, T, d, Fs, 1, op(das + z * Fs, 0, SF, 1), 0,
                     op(offset_elems(w.Ws_gate, wz, bf), bf, 1, Fs), 0, gr.dx, d),
                GEN_EPI_ACCUM);
            RUN(gemm(GEN_DENSE, T, d, Fs, 1, op(dus + z * Fs, 0, SF, 1), 0,
                     op(offset_elems(w.Ws_up, wz, bf), bf, 1, Fs), 0, gr.dx, d),
                GEN_EPI_ACCUM);
        }
        if (gr.dWs_down)
            RUN(gemm(GEN_DENSE, Fs, d, T, S, op(hs, 0, 1, SF, Fs), 1, op(dout, 0, d, 1), 1,
                     gr.dWs_down, d, static_cast<long long>(Fs) * d),
                GEN_EPI_STORE);
        if (gr.dWs_gate)
            RUN(gemm(GEN_DENSE, d, Fs, T, S, op(x, bf, 1, d), 1, op(das, 0, SF, 1, Fs), 1,
                     gr.dWs_gate, Fs, static_cast<long long>(d) * Fs),
                GEN_EPI_STORE);
        if (gr.dWs_up)
            RUN(gemm(GEN_DENSE, d, Fs, T, S, op(x, bf, 1, d), 1, op(dus, 0, SF, 1, Fs), 1,
                     gr.dWs_up, Fs, static_cast<long long>(d) * Fs),
                GEN_EPI_STORE);
    }

    // router: dg -> dr -> dW_router and dx
    if ((e = launch_pdl(router_bwd_kernel, dim3((T * 32 + 255) / 256), dim3(256), 0, s, dwpart, ntf,
                        inv, tidx, tw, scores, T, K, E, c.gate, c.renormalize, c.routed_scale, dr,
                        dg, static_cast<float*>(nullptr), static_cast<const int32_t*>(nullptr),
                        static_cast<const float*>(nullptr), 0, static_cast<float*>(nullptr))) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (gr.dW_router &&
        (e = run_splitk(gemm(GEN_DENSE, d, E, T, 1, op(x, bf, 1, d), 1, op(dr, 0, E, 1), 1,
                             gr.dW_router, E),
                        GEN_EPI_STORE, BP(BL.kpart), BL.kpart_floats, s)) != cudaSuccess)
        return MOE_ERR_CUDA;
    RUN(gemm(GEN_DENSE, T, d, E, 1, op(dr, 0, E, 1), 0, op(w.W_router, 0, 1, E), 0, gr.dx, d),
        GEN_EPI_ACCUM);
#undef RUN
    return MOE_OK;
}

// The tensor-core form (BF16 layers, widths multiples of 64). The routed
// rows live in the expert-padded row layout (each expert's rows, then zero
// rows up to a multiple of 64), so every per-expert reduction covers whole
// 64-row k-blocks of its own rows. dh = gy W_down^T and dz = da W_gate^T +
// du W_up^T run on the NT kernel (both operands K-major: the weights as they
// are); the gate and up products are recomputed by the forward's grouped
// GEMM, whose backward epilogue writes da, du and g h; the weight gradients
// run on the NT kernel with both operands MN-major (the row-major
// activations as they are, C = A^T B over the rows). Upstream and activation
// gradients enter the tensor cores rounded to BF16; every sum is FP32.
static moe_status backward_tc(const moe_config& c, const void* x, const moe_weights& w,
                              const float* dout, const moe_grads& gr, uint8_t* ws, uint8_t* bws,
                              cudaStream_t s) {
    const WsLayout L = plan_workspace(c);
    const BwdLayout BL = plan_backward(c);
    const int T = c.T, K = c.K, E = c.E, TK = T * c.K, F = c.d_ff, d = c.d;
    const int lat = c.latent_dim, de = lat ? lat : d;
    const int S = c.n_shared, Fs = S ? c.shared_d_ff : 0, SF = S * Fs;
    const int kp = static_cast<int>(BL.tkpad), tp = static_cast<int>(BL.tpad);
    int* err = reinterpret_cast<int*>(ws + L.err);
    auto WP = [&](size_t off) { return static_cast<void*>(ws + off); };
    auto BF = [&](size_t off) { return reinterpret_cast<float*>(bws + off); };
    auto BH = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(bws + off); };
    const int32_t* stok = static_cast<const int32_t*>(WP(L.sorted_token));
    const float* sw = static_cast<const float*>(WP(L.sorted_w));
    const int32_t* inv = static_cast<const int32_t*>(WP(L.inv));
    const int32_t* offsets = static_cast<const int32_t*>(WP(L.offsets));
    const int32_t* tidx = static_cast<const int32_t*>(WP(L.topk_idx));
    const float* tw = static_cast<const float*>(WP(L.topk_w));
    const float* scores = L.scores ? static_cast<const float*>(WP(L.scores)) : nullptr;
    int32_t* poff = reinterpret_cast<int32_t*>(bws + BL.poff);
    int32_t* invp = reinterpret_cast<int32_t*>(bws + BL.invp);
    float *dr = BF(BL.dr), *dg = BF(BL.dg);
    cudaError_t e;
#define CK(call)                                                  \
    do {                                                          \
        if ((e = (call)) != cudaSuccess) return MOE_ERR_CUDA;     \
    } while (0)
    // K-major operand: rows x K (pitch ld), optionally Z slices; MN-major:
    // K rows of `rows` columns (pitch ld)
    auto opnd = [](const void* p, long long rows, long long K_, long long ld, long long Z = 1,
                   long long zstride = 0) {
        NtOperand o;
        o.p = p;
        o.rows = rows;
        o.K = K_;
        o.ld = ld;
        o.Z = Z;
        o.zstride = zstride;
        return o;
    };
    auto nt = [&](int mode, int M, int N, int K_, int Z, NtOperand A, NtOperand B, float* C,
                  long long ldc, long long c_zs = 0, const int32_t* offs = nullptr) {
        NtGemm g;
        memset(&g, 0, sizeof(g));
        g.mode = mode;
        g.M = M;
        g.N = N;
        g.K = K_;
        g.Z = Z;
        g.nph = 1;
        g.A[0] = A;
        g.B[0] = B;
        g.offsets = offs;
        g.C = C;
        g.ldc = ldc;
        g.c_zs = c_zs;
        g.err = err;
        return g;
    };
    auto tn = [&](int mode, int M, int N, int K_, int Z, NtOperand A, NtOperand B, float* C,
                  long long ldc, long long c_zs = 0, const int32_t* offs = nullptr) {
        NtGemm g = nt(mode, M, N, K_, Z, A, B, C, ldc, c_zs, offs);
        g.a_mn = 1;
        g.b_mn = 1;
        return g;
    };

    // BF16 copy of dout: the shared experts' and the latent projections' operand
    __nv_bfloat16* doutb = nullptr;
    if (S || lat) {
        doutb = BH(BL.doutb);
        CK(launch_gather_bf16(dout, 0, d, nullptr, T, d, doutb, s));
    }

    // upstream gradient of the routed sum (FP32) and the rows the experts act on
    const float* gy = dout;
    long long ld_gy = d;
    const void* zsrc = x;
    long long ld_z = d;
    if (lat) {
        float* glat = BF(BL.glat);
        // gy = dout W_up_latent^T: W_up_latent [L, d] rows are K-major for this product
        CK(launch_nt_gemm(nt(NT_DENSE, T, lat, d, 1, opnd(doutb, T, d, d), opnd(w.W_up_latent, lat, d, d),
                             glat, lat),
                          s));
        if (gr.dW_up_latent) {
            // routed sum of the forward (latent width), then dW_up_latent = routed^T dout
            float* routed = BF(BL.routed);
            __nv_bfloat16* routedb = BH(BL.routedb);
            CK(launch_gather_sum(static_cast<const float*>(WP(L.ys)), inv, T, K, lat, nullptr,
                                 routed, 0, s));
            CK(launch_gather_bf16(routed, 0, lat, nullptr, T, lat, routedb, s));
            CK(launch_nt_gemm(tn(NT_DENSE, lat, d, tp, 1, opnd(routedb, lat, T, lat), opnd(doutb, d, T, d),
                                 gr.dW_up_latent, d),
                              s));
        }
        gy = glat;
        ld_gy = lat;
        zsrc = WP(L.z);
        ld_z = lat;
    }

    // ---- the expert-padded row layout: offsets, positions, gathered rows ----
    CK(launch_pad_offsets(offsets, E, poff, s));
    CK(launch_pad_inverse(inv, tidx, TK, poff, offsets, invp, s));
    __nv_bfloat16 *gys = BH(BL.gys), *zs = BH(BL.zs);
    CK(launch_gather_pad_bf16(gy, 0, ld_gy, stok, TK, de, poff, offsets, E, kp, gys, s));
    CK(launch_gather_pad_bf16(zsrc, 1, ld_z, stok, TK, de, poff, offsets, E, kp, zs, s));

    // ---- dh = gy W_down^T per expert (padded rows), dout Ws_down^T (shared),
    //      then the SwiGLU backward: da, du, g h and the gate-gradient partials ----
    __nv_bfloat16 *dab = BH(BL.dab), *dub = BH(BL.dub), *hwb = BH(BL.hwb);
    float* dgpart = BF(BL.dwrow);
    __nv_bfloat16 *dasb = S ? BH(BL.dasb) : nullptr, *dusb = S ? BH(BL.dusb) : nullptr,
                  *hsb = S ? BH(BL.hsb) : nullptr;
    int npart;  // gate-gradient partials per row
    if (BL.saved) {
        // the forward kept the gate and up products: the SwiGLU backward runs in
        // the epilogue of the dh products, nothing is recomputed
        NtGemm g = nt(NT_MSEG, kp, F, de, E, opnd(gys, kp, de, de),
                      opnd(w.W_down, F, de, de, E, static_cast<long long>(F) * de), nullptr, F, 0, poff);
        g.sg_a = static_cast<const __nv_bfloat16*>(WP(L.ga));
        g.sg_u = static_cast<const __nv_bfloat16*>(WP(L.gu));
        g.sg_off = offsets;
        g.sg_ld = F;
        g.sg_g = sw;
        g.sg_da = dab;
        g.sg_du = dub;
        g.sg_hw = hwb;
        g.sg_part = dgpart;
        g.sg_npart = F / 64;
        CK(launch_nt_gemm(g, s));
        if (S) {
            NtGemm g2 = nt(NT_DENSE, T, Fs, d, S, opnd(doutb, T, d, d),
                           opnd(w.Ws_down, Fs, d, d, S, static_cast<long long>(Fs) * d), nullptr, SF, Fs);
            g2.b_z3 = 1;
            g2.sg_a = static_cast<const __nv_bfloat16*>(WP(L.gas));
            g2.sg_u = static_cast<const __nv_bfloat16*>(WP(L.gus));
            g2.sg_da = dasb;
            g2.sg_du = dusb;
            g2.sg_hw = hsb;
            CK(launch_nt_gemm(g2, s));
        }
        npart = F / 64;
    } else {
        float* dhp = BF(BL.dhp);
        CK(launch_nt_gemm(nt(NT_MSEG, kp, F, de, E, opnd(gys, kp, de, de),
                             opnd(w.W_down, F, de, de, E, static_cast<long long>(F) * de), dhp, F, 0, poff),
                          s));
        float* dhs = nullptr;
        if (S) {
            dhs = BF(BL.dhs);
            NtGemm g = nt(NT_DENSE, T, Fs, d, S, opnd(doutb, T, d, d),
                          opnd(w.Ws_down, Fs, d, d, S, static_cast<long long>(Fs) * d), dhs, SF, Fs);
            g.b_z3 = 1;
            CK(launch_nt_gemm(g, s));
        }
        // the gate and up products recomputed by the forward's GEMM; its SwiGLU
        // backward epilogue writes da, du, g h and the gate-gradient partials
        TcGemmArgs g{};
        g.g[0] = TcGroup{1, de, WP(L.xs), de, TK, w.W_gate, w.W_up, E, F, nullptr, F, 0};
        g.g[0].dh = dhp;
        g.g[0].dh_ld = F;
        g.g[0].da = dab;
        g.g[0].du = dub;
        g.g[0].hw = hwb;
        g.g[0].dgpart = dgpart;
        if (S) {
            g.g[1] = TcGroup{1, d, x, d, T, w.Ws_gate, w.Ws_up, S, Fs, nullptr, SF, 0};
            g.g[1].dh = dhs;
            g.g[1].dh_ld = SF;
            g.g[1].da = dasb;
            g.g[1].du = dusb;
            g.g[1].hw = hsb;
        }
        g.E = E;
        g.offsets = offsets;
        g.mt_prefix = static_cast<const int32_t*>(WP(L.mt_prefix));
        g.swiglu = TC_SWIGLU_BWD;
        g.rowscale0 = sw;
        g.poff = poff;
        g.err = err;
        CK(launch_tc_gemm(g, s));
        npart = 2 * ((F + 127) / 128);
    }

    // ---- dz rows = da W_gate^T + du W_up^T (padded rows, two phases) ----
    float* dxsp = BF(BL.dxsp);
    {
        NtGemm g = nt(NT_MSEG, kp, de, F, E, opnd(dab, kp, F, F),
                      opnd(w.W_gate, de, F, F, E, static_cast<long long>(de) * F), dxsp, de, 0, poff);
        g.nph = 2;
        g.A[1] = opnd(dub, kp, F, F);
        g.B[1] = opnd(w.W_up, de, F, F, E, static_cast<long long>(de) * F);
        CK(launch_nt_gemm(g, s));
    }
    // ---- expert weight gradients: sums over each expert's padded rows of the
    //      row-major operands (both MN-major) ----
    if (gr.dW_down)
        CK(launch_nt_gemm(tn(NT_KSEG, F, de, kp, E, opnd(hwb, F, kp, F), opnd(gys, de, kp, de), gr.dW_down,
                             de, static_cast<long long>(F) * de, poff),
                          s));
    if (gr.dW_gate)
        CK(launch_nt_gemm(tn(NT_KSEG, de, F, kp, E, opnd(zs, de, kp, de), opnd(dab, F, kp, F), gr.dW_gate, F,
                             static_cast<long long>(de) * F, poff),
                          s));
    if (gr.dW_up)
        CK(launch_nt_gemm(tn(NT_KSEG, de, F, kp, E, opnd(zs, de, kp, de), opnd(dub, F, kp, F), gr.dW_up, F,
                             static_cast<long long>(de) * F, poff),
                          s));

    // ---- dx from the routed experts (latent: through dz and W_down_latent) ----
    if (!lat) {
        CK(launch_gather_sum(dxsp, invp, T, K, d, nullptr, gr.dx, 0, s));
    } else {
        float* dz = BF(BL.dz);
        __nv_bfloat16* dzb = BH(BL.dzb);
        CK(launch_gather_sum(dxsp, invp, T, K, lat, nullptr, dz, 0, s));
        CK(launch_gather_bf16(dz, 0, lat, nullptr, T, lat, dzb, s));
        if (gr.dW_down_latent)  // dW_down_latent = x^T dz
            CK(launch_nt_gemm(tn(NT_DENSE, d, lat, tp, 1, opnd(x, d, T, d), opnd(dzb, lat, T, lat),
                                 gr.dW_down_latent, lat),
                              s));
        // dx = dz W_down_latent^T: W_down_latent [d, L] rows are K-major for this product
        CK(launch_nt_gemm(nt(NT_DENSE, T, d, lat, 1, opnd(dzb, T, lat, lat),
                             opnd(w.W_down_latent, d, lat, lat), gr.dx, d),
                          s));
    }

    // ---- shared experts: dx, weight gradients ----
    if (S) {
        for (int z = 0; z < S; ++z) {
            NtGemm g = nt(NT_DENSE, T, d, Fs, 1, opnd(dasb, T, SF, SF),
                          opnd(w.Ws_gate, d, Fs, Fs, S, static_cast<long long>(d) * Fs), gr.dx, d);
            g.nph = 2;
            g.A[1] = opnd(dusb, T, SF, SF);
            g.B[1] = opnd(w.Ws_up, d, Fs, Fs, S, static_cast<long long>(d) * Fs);
            g.a_kofs[0] = g.a_kofs[1] = z * Fs;
            g.b_zc[0] = g.b_zc[1] = z;
            g.accumulate = 1;
            CK(launch_nt_gemm(g, s));
        }
        if (gr.dWs_down) {  // dWs_down[s] = hs_s^T dout
            NtGemm g = tn(NT_DENSE, Fs, d, tp, S, opnd(hsb, SF, T, SF), opnd(doutb, d, T, d), gr.dWs_down, d,
                          static_cast<long long>(Fs) * d);
            g.a_zrow = Fs;
            CK(launch_nt_gemm(g, s));
        }
        for (int which = 0; which < 2; ++which) {  // dWs_gate[s] = x^T das_s, dWs_up[s] = x^T dus_s
            float* C = which ? gr.dWs_up : gr.dWs_gate;
            if (!C) continue;
            NtGemm g = tn(NT_DENSE, d, Fs, tp, S, opnd(x, d, T, d), opnd(which ? dusb : dasb, SF, T, SF), C, Fs,
                          static_cast<long long>(d) * Fs);
            g.b_zrow = Fs;
            CK(launch_nt_gemm(g, s));
        }
    }

    // ---- router: dg -> dr; dx += dr W_router^T (K nonzeros per token, read
    //      from W_router^T rows); dW_router over each expert's padded rows of
    //      x (the latent variant: a split-K product over the tokens) ----
    float* wrt = BF(BL.wrt);
    float* cp = lat ? nullptr : BF(BL.cp);
    if (cp != nullptr) CK(cudaMemsetAsync(cp, 0, static_cast<size_t>(kp) * sizeof(float), s));
    CK(launch_pdl(transpose_f32_kernel, dim3((E + 31) / 32, (d + 31) / 32), dim3(256), 0, s,
                  static_cast<const float*>(w.W_router), d, E, wrt));
    CK(launch_pdl(router_bwd_kernel, dim3((T * 32 + 255) / 256), dim3(256), 0, s,
                  static_cast<const float*>(dgpart), npart, inv, tidx, tw, scores, T, K, E,
                  c.gate, c.renormalize, c.routed_scale, dr, dg, cp, static_cast<const int32_t*>(invp),
                  static_cast<const float*>(wrt), d, gr.dx));
    if (gr.dW_router) {
        if (!lat) {
            float* rp = BF(BL.rpart);
            CK(launch_pdl(router_wgrad_part_kernel, dim3(kp / 64, (d + 255) / 256), dim3(256), 0, s,
                          static_cast<const __nv_bfloat16*>(zs), static_cast<const float*>(cp), d, rp));
            CK(launch_pdl(router_wgrad_reduce_kernel, dim3((d * E + 255) / 256), dim3(256), 0, s,
                          static_cast<const float*>(rp), static_cast<const int32_t*>(poff), d, E,
                          gr.dW_router));
        } else {
            CK(run_splitk(gemm(GEN_DENSE, d, E, T, 1, op(x, 1, 1, d), 1, op(dr, 0, E, 1), 1, gr.dW_router, E),
                          GEN_EPI_STORE, BF(BL.kpart), BL.kpart_floats, s));
        }
    }
#undef CK
    return MOE_OK;
}

}  // namespace moe
