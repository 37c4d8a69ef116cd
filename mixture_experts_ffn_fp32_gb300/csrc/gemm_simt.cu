// FP32 grouped GEMM on the CUDA cores (FFMA), for the FP32 layer. Same
// segment groups and epilogues as the tcgen05 kernel (gemm_tc.cu):
//   SwiGLU : h[r, :] = SiLU(A[a_row(r), :] W_gate[z]) * (A[a_row(r), :] W_up[z])
//   plain  : y[r, :] = rowscale[r] * (A[r, :] B[z])                       (group 0)
//            out[t, :] = A[t, :] B + sum_k ys[inv[t, k], :]                (group 1)
// (APEX-1 Mathematical Reference Part 3, section 12.2; the layer sum of
// section 13.2). The routed gate/up step reads its A rows through the
// dispatch's sorted_token list, so no gathered copy of x is made.
// The 5th-generation tensor cores have no FP32-exact input kind, and TF32
// inputs would not meet a 1e-4 absolute error on this layer, so FP32 stays
// on FFMA. Tile 64 x 64 x 16, 256 threads, 4 x 4 outputs per thread and
// operand, one tile per CTA (grid over an upper bound of the tile count;
// tiles past the device-side count exit at once).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = SIMT_BM, BN = 64, BK = 16;

struct SimtParams {
    SimtGroup g[2];
    int K, E, nt0, nt1, mt1;
    const int32_t* offsets;
    const int32_t* mt_prefix;
    const float* rowscale0;
    const int32_t* inv;
    const float* ys;
    int ys_ld, Kr;
};

template <bool SWIGLU>
__global__ void __launch_bounds__(256) simt_grouped_gemm_kernel(SimtParams p) {
    constexpr int NB = SWIGLU ? 2 : 1;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[NB][BK][BN + 4];
    pdl_wait();
    pdl_trigger();

    const int total0 = p.g[0].enabled ? p.mt_prefix[p.E] * p.nt0 : 0;
    const int total = total0 + (p.g[1].enabled ? p.mt1 * p.g[1].Z * p.nt1 : 0);
    const int u = blockIdx.x;
    if (u >= total) return;

    int g, row0, rows, z, n0, out_col0;
    if (u < total0) {
        const int mt = u / p.nt0, n = u - mt * p.nt0;
        int lo = 0, hi = p.E;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.mt_prefix[mid] <= mt)
                lo = mid;
            else
                hi = mid;
        }
        g = 0;
        row0 = p.offsets[lo] + (mt - p.mt_prefix[lo]) * BM;
        rows = min(BM, p.offsets[lo + 1] - row0);
        z = lo;
        n0 = n * BN;
        out_col0 = n0;
    } else {
        const int u1 = u - total0;
        const int per_m = p.g[1].Z * p.nt1;
        const int m = u1 / per_m, rem = u1 - m * per_m;
        g = 1;
        z = rem / p.nt1;
        n0 = (rem - z * p.nt1) * BN;
        row0 = m * BM;
        rows = min(BM, p.g[1].rows - row0);
        out_col0 = z * p.g[1].N + n0;
    }
    const SimtGroup& G = p.g[g];
    const int N = G.N, K = p.K;
    const float* B0 = G.B0 + static_cast<size_t>(z) * K * N;
    const float* B1 = SWIGLU ? G.B1 + static_cast<size_t>(z) * K * N : nullptr;

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    // A loader: row lr = tid / 4, 4 consecutive k at (tid % 4) * 4
    const int lr = tid >> 2, lk = (tid & 3) * 4;
    const bool lrow_ok = lr < rows;
    const int arow = lrow_ok ? (G.a_rows ? G.a_rows[row0 + lr] : row0 + lr) : 0;
    // B loader: k row tid / 16, 4 consecutive n at (tid % 16) * 4
    const int bk = tid >> 4, bn = (tid & 15) * 4;

    float acc[NB][4][4];
#pragma unroll
    for (int o = 0; o < NB; ++o)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[o][i][j] = 0.0f;

    for (int k0 = 0; k0 < K; k0 += BK) {
        {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lrow_ok && k0 + lk < K)
                v = *reinterpret_cast<const float4*>(G.A + static_cast<size_t>(arow) * G.lda + k0 + lk);
            As[lk + 0][lr] = v.x;
            As[lk + 1][lr] = v.y;
            As[lk + 2][lr] = v.z;
            As[lk + 3][lr] = v.w;
        }
#pragma unroll
        for (int o = 0; o < NB; ++o) {
            const float* B = (o == 0) ? B0 : B1;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            const int kk = k0 + bk, nn = n0 + bn;
            if (kk < K && nn < N) v = *reinterpret_cast<const float4*>(B + static_cast<size_t>(kk) * N + nn);
            *reinterpret_cast<float4*>(&Bs[o][bk][bn]) = v;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float av[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int o = 0; o < NB; ++o) {
                float bv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[j] = Bs[o][kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[o][i][j] = fmaf(av[i], bv[j], acc[o][i][j]);
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty * 4 + i;
        if (r >= rows) continue;
        const size_t orow = static_cast<size_t>(row0 + r);
        const float rs = (!SWIGLU && g == 0 && p.rowscale0) ? p.rowscale0[orow] : 1.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float v;
            if (SWIGLU) {
                const float a = acc[0][i][j];
                v = a / (1.0f + expf(-a)) * acc[1][i][j];
            } else {
                v = rs * acc[0][i][j];
                if (g == 1 && p.inv) {
                    for (int k = 0; k < p.Kr; ++k)
                        v += p.ys[static_cast<size_t>(p.inv[orow * p.Kr + k]) * p.ys_ld + out_col0 + tx * 4 + j];
                }
            }
            G.out[orow * G.out_ld + out_col0 + tx * 4 + j] = v;
        }
    }
}

template <bool SWIGLU>
cudaError_t launch_simt_t(const SimtGemmArgs& a, cudaStream_t s) {
    SimtParams p;
    memset(&p, 0, sizeof(p));
    p.g[0] = a.g[0];
    p.g[1] = a.g[1];
    p.K = a.K;
    p.E = a.E;
    p.nt0 = a.g[0].enabled ? (a.g[0].N + BN - 1) / BN : 0;
    p.nt1 = a.g[1].enabled ? (a.g[1].N + BN - 1) / BN : 0;
    p.mt1 = a.g[1].enabled ? (a.g[1].rows + BM - 1) / BM : 0;
    p.offsets = a.offsets;
    p.mt_prefix = a.mt_prefix;
    p.rowscale0 = a.rowscale0;
    p.inv = a.inv;
    p.ys = a.ys;
    p.ys_ld = a.ys_ld;
    p.Kr = a.Kr;
    long long bound = 0;
    if (a.g[0].enabled) bound += static_cast<long long>((a.g[0].rows + BM - 1) / BM + a.E) * p.nt0;
    if (a.g[1].enabled) bound += static_cast<long long>(p.mt1) * a.g[1].Z * p.nt1;
    if (bound < 1) bound = 1;
    return launch_pdl(simt_grouped_gemm_kernel<SWIGLU>, dim3(static_cast<unsigned>(bound)), dim3(256),
                      0, s, p);
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemmArgs& a, cudaStream_t s) {
    return a.swiglu ? launch_simt_t<true>(a, s) : launch_simt_t<false>(a, s);
}

}  // namespace moe
