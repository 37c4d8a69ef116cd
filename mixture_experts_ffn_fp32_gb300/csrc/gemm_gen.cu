// Strided grouped GEMM on the CUDA cores (FP32 FFMA, FP32 or BF16 operands),
// for the backward pass of the layer. Every contraction of the backward is
//   C[m, n] (+)= sum_k A(m, k) B(k, n)
// with each operand read through two strides and an optional index list on
// either of its dimensions, so transposed operands and rows gathered through
// the dispatch (sorted_token) need no copies. Three ways to cut the work:
//   GEN_DENSE : Z independent problems of the same shape, operand and output
//               bases advanced by z * zs (shared experts, projections, router)
//   GEN_MSEG  : the rows m of segment z are offsets[z] .. offsets[z+1] (the
//               expert-sorted rows of the routed experts); B advanced by z
//   GEN_KSEG  : the reduction k of segment z runs over offsets[z] ..
//               offsets[z+1] (an expert's weight gradient, summed over its
//               rows); C advanced by z. Empty segments write nothing: an
//               expert without rows gets no gradient (kimi_k3
//               StableLatentMoE, "Grouped expert execution and sparse
//               gradients").
// Epilogues: store, accumulate, and the SwiGLU backward, which takes the
// recomputed gate and up products a, u of the row (two B operands) with the
// upstream gradient dh of the hidden vector and the row's gate weight g:
//   h = SiLU(a) u, da = g dh u SiLU'(a), du = g dh SiLU(a), hw = g h,
//   dwpart[m, tile] = sum over the tile's columns of dh h
// (the chain rule of APEX-1 Mathematical Reference Part 3, section 12.2;
// SiLU'(a) = sigma(a) (1 + a (1 - sigma(a))), from section 12.3's SiLU).
// Tile 64 x 64 x 16, 256 threads, 4 x 4 outputs per thread, one tile per CTA.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int GBM = 64, GBN = 64, GBK = 16;

MOE_DEV float ld_op(const GenOp& o, long long off) {
    return o.bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(o.p)[off])
                  : static_cast<const float*>(o.p)[off];
}

// Element (i, j) of an operand: dimension 0 is m for A and k for B.
MOE_DEV long long op_off(const GenOp& o, int i, int j, long long zoff) {
    const long long ii = o.idx0 ? o.idx0[i] : i;
    const long long jj = o.idx1 ? o.idx1[j] : j;
    return zoff + ii * o.s0 + jj * o.s1;
}

template <int EPI>
__global__ void __launch_bounds__(256) gen_gemm_kernel(GenGemm p) {
    constexpr int NB = EPI == GEN_EPI_SWIGLU_BWD ? 2 : 1;
    __shared__ float As[GBK][GBM + 4];
    __shared__ float Bs[NB][GBK][GBN + 4];
    __shared__ int s_tp[MAXSEG + 1];
    pdl_wait();
    pdl_trigger();

    const int nt = (p.N + GBN - 1) / GBN;
    const int mt_dense = (p.M + GBM - 1) / GBM;
    int total;
    if (p.mode == GEN_MSEG) {
        // m-tiles per segment, prefix-summed by one thread (at most MAXSEG segments)
        if (threadIdx.x == 0) {
            int acc = 0;
            for (int z = 0; z < p.Z; ++z) {
                s_tp[z] = acc;
                acc += (p.offsets[z + 1] - p.offsets[z] + GBM - 1) / GBM;
            }
            s_tp[p.Z] = acc;
        }
        __syncthreads();
        total = s_tp[p.Z] * nt;
    } else {
        total = p.Z * mt_dense * nt;
    }
    const int u = blockIdx.x;
    if (u >= total) return;

    int z, m0, rows, n0, k0 = 0, k1 = p.K;
    long long a_z = 0, b_z = 0, c_z = 0;
    if (p.ksplit > 1) {
        // split-K: this CTA's slice of the reduction, into its own partial plane
        const int kc = (p.K + p.ksplit - 1) / p.ksplit;
        k0 = blockIdx.y * kc;
        k1 = min(p.K, k0 + kc);
    }
    if (p.mode == GEN_MSEG) {
        const int mt = u / nt;
        n0 = (u - mt * nt) * GBN;
        int lo = 0, hi = p.Z;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_tp[mid] <= mt)
                lo = mid;
            else
                hi = mid;
        }
        z = lo;
        m0 = p.offsets[z] + (mt - s_tp[z]) * GBM;
        rows = min(GBM, p.offsets[z + 1] - m0);
        b_z = z * p.B0.zs;
    } else {
        const int per = mt_dense * nt;
        z = u / per;
        const int rem = u - z * per;
        const int mt = rem / nt;
        m0 = mt * GBM;
        rows = min(GBM, p.M - m0);
        n0 = (rem - mt * nt) * GBN;
        a_z = z * p.A.zs;
        b_z = z * p.B0.zs;
        c_z = z * p.c_zs;
        if (p.mode == GEN_KSEG) {
            k0 = p.offsets[z];
            k1 = p.offsets[z + 1];
            if (k1 <= k0) return;  // no rows: no gradient for this segment
            a_z = 0;
            b_z = 0;
        }
    }
    const long long b1_z = (p.mode == GEN_KSEG) ? 0 : z * p.B1.zs;

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    float acc[NB][4][4];
#pragma unroll
    for (int o = 0; o < NB; ++o)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[o][i][j] = 0.0f;

    for (int kb = k0; kb < k1; kb += GBK) {
        // A tile [GBM x GBK]: consecutive threads walk the operand's contiguous dimension
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = tid + 256 * q;
            int mm, kk;
            if (p.a_m_contig) {
                mm = e & (GBM - 1);
                kk = e >> 6;
            } else {
                kk = e & (GBK - 1);
                mm = e >> 4;
            }
            float v = 0.0f;
            if (mm < rows && kb + kk < k1) v = ld_op(p.A, op_off(p.A, m0 + mm, kb + kk, a_z));
            As[kk][mm] = v;
        }
#pragma unroll
        for (int o = 0; o < NB; ++o) {
            const GenOp& B = o == 0 ? p.B0 : p.B1;
            const long long bz = o == 0 ? b_z : b1_z;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = tid + 256 * q;
                int kk, nn;
                if (p.b_n_contig) {
                    nn = e & (GBN - 1);
                    kk = e >> 6;
                } else {
                    kk = e & (GBK - 1);
                    nn = e >> 4;
                }
                float v = 0.0f;
                if (kb + kk < k1 && n0 + nn < p.N) v = ld_op(B, op_off(B, kb + kk, n0 + nn, bz));
                Bs[o][kk][nn] = v;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GBK; ++kk) {
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

    if (EPI == GEN_EPI_SWIGLU_BWD) {
        // per-row partial of sum_n dh h over this tile's columns: 16 threads share a row
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            if (r >= rows) continue;
            const long long row = m0 + r;
            const float g = p.rowscale ? p.rowscale[row] : 1.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx * 4 + j;
                if (n >= p.N) continue;
                const long long o = c_z + row * p.ldc + n;
                const float a = acc[0][i][j], uu = acc[1][i][j];
                const float sg = 1.0f / (1.0f + expf(-a));
                const float si = a * sg;
                const float dh = p.dh[o];
                const float h = si * uu;
                p.da[o] = g * dh * uu * (sg * (1.0f + a * (1.0f - sg)));
                p.du[o] = g * dh * si;
                p.hw[o] = g * h;
                part[i] += dh * h;
            }
        }
        if (p.dwpart != nullptr) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // fixed-order sum over the 16 threads of the row (tx = 0..15)
                float v = part[i];
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                const int r = ty * 4 + i;
                if (tx == 0 && r < rows) p.dwpart[static_cast<long long>(m0 + r) * nt + n0 / GBN] = v;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            if (r >= rows) continue;
            const long long row = m0 + r;
            const float g = p.rowscale ? p.rowscale[row] : 1.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx * 4 + j;
                if (n >= p.N) continue;
                const float v = g * acc[0][i][j];
                if (p.ksplit > 1) {
                    p.part[((static_cast<long long>(blockIdx.y) * p.Z + z) * p.M + row) * p.N + n] = v;
                    continue;
                }
                float* c = p.C + c_z + row * p.ldc + n;
                if (EPI == GEN_EPI_ACCUM)
                    *c += v;
                else
                    *c = v;
            }
        }
    }
}

// C (=|+=) sum over the ksplit partial planes, in plane order.
__global__ void __launch_bounds__(256) gen_reduce_kernel(const float* __restrict__ part, int ksplit,
                                                         int Z, int M, int N, float* __restrict__ C,
                                                         long long ldc, long long c_zs, int accumulate) {
    pdl_wait();
    pdl_trigger();
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long plane = static_cast<long long>(Z) * M * N;
    if (i >= plane) return;
    float v = 0.0f;
    for (int k = 0; k < ksplit; ++k) v += part[k * plane + i];
    const long long z = i / (static_cast<long long>(M) * N);
    const long long rem = i - z * M * N;
    const long long m = rem / N, n = rem - m * N;
    float* c = C + z * c_zs + m * ldc + n;
    if (accumulate)
        *c += v;
    else
        *c = v;
}

}  // namespace

int gen_gemm_ksplit(const GenGemm& p, size_t part_floats) {
    if (p.mode != GEN_DENSE) return 1;
    const long long tiles = static_cast<long long>(p.Z) * ((p.M + GBM - 1) / GBM) * ((p.N + GBN - 1) / GBN);
    const long long plane = static_cast<long long>(p.Z) * p.M * p.N;
    long long ks = (4LL * num_sms() + tiles - 1) / tiles;      // about four CTAs per SM
    ks = std::min<long long>(ks, (p.K + 63) / 64);             // at least 64 k per slice
    ks = std::max<long long>(ks, (p.K + 1023) / 1024);         // and at most 1024 k per slice: its k-steps are not pipelined
    ks = std::min<long long>(ks, plane > 0 ? static_cast<long long>(part_floats) / plane : 1);
    return ks > 1 ? static_cast<int>(std::min<long long>(ks, 1024)) : 1;
}

cudaError_t launch_gen_gemm(const GenGemm& p, int epi, cudaStream_t s) {
    if (p.mode == GEN_MSEG && p.Z > MAXSEG) return cudaErrorInvalidValue;
    const long long nt = (p.N + GBN - 1) / GBN;
    long long tiles;
    if (p.mode == GEN_MSEG)
        tiles = ((p.M + GBM - 1) / GBM + p.Z) * nt;  // at most one partial tile per segment
    else
        tiles = static_cast<long long>(p.Z) * ((p.M + GBM - 1) / GBM) * nt;
    if (tiles < 1) return cudaSuccess;
    if (p.ksplit > 1) {
        if (p.mode != GEN_DENSE || epi == GEN_EPI_SWIGLU_BWD || p.part == nullptr)
            return cudaErrorInvalidValue;
        const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(p.ksplit));
        cudaError_t e = launch_pdl(gen_gemm_kernel<GEN_EPI_STORE>, grid, dim3(256), 0, s, p);
        if (e != cudaSuccess) return e;
        const long long plane = static_cast<long long>(p.Z) * p.M * p.N;
        return launch_pdl(gen_reduce_kernel, dim3(static_cast<unsigned>((plane + 255) / 256)), dim3(256), 0,
                          s, static_cast<const float*>(p.part), p.ksplit, p.Z, p.M, p.N, p.C, p.ldc,
                          p.c_zs, epi == GEN_EPI_ACCUM ? 1 : 0);
    }
    const dim3 grid(static_cast<unsigned>(tiles));
    if (epi == GEN_EPI_SWIGLU_BWD) return launch_pdl(gen_gemm_kernel<GEN_EPI_SWIGLU_BWD>, grid, dim3(256), 0, s, p);
    if (epi == GEN_EPI_ACCUM) return launch_pdl(gen_gemm_kernel<GEN_EPI_ACCUM>, grid, dim3(256), 0, s, p);
    return launch_pdl(gen_gemm_kernel<GEN_EPI_STORE>, grid, dim3(256), 0, s, p);
}

int gen_gemm_ntiles(int N) { return (N + GBN - 1) / GBN; }

}  // namespace moe
