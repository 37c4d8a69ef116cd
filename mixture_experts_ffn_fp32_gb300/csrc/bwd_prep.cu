// Operand preparation for the tensor-core backward (gemm_nt.cu reads both
// operands K-major): BF16 copies of gathered rows, transposed copies laid out
// per expert with each expert's rows padded to a multiple of 64 columns
// (zero columns between experts, so an expert's weight-gradient reduction
// covers whole k-blocks of its own rows only), and the SwiGLU backward of
// each row. Sources: the chain rule of APEX-1 Mathematical Reference Part 3,
// section 12.2 (SwiGLU) and 12.3 (SiLU), as in backward.cu.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void pad_offsets_kernel(const int32_t* __restrict__ offsets, int E,
                                   int32_t* __restrict__ poff) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int acc = 0;
    for (int z = 0; z < E; ++z) {
        poff[z] = acc;
        acc += (offsets[z + 1] - offsets[z] + 63) / 64 * 64;
    }
    poff[E] = acc;
}

MOE_DEV float ld_any(const void* p, int bf16, long long off) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[off])
                : static_cast<const float*>(p)[off];
}

// one warp per row, 8 columns per lane step
__global__ void __launch_bounds__(256) gather_bf16_kernel(const void* __restrict__ src, int src_bf16,
                                                          long long ld, const int32_t* __restrict__ idx,
                                                          int rows, int cols,
                                                          __nv_bfloat16* __restrict__ dst) {
    pdl_wait();
    pdl_trigger();
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (r >= rows) return;
    const int lane = threadIdx.x & 31;
    const long long sr = idx ? idx[r] : r;
    for (int c = lane * 8; c < cols; c += 256) {
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            pk[i] = pack_bf16x2(ld_any(src, src_bf16, sr * ld + c + 2 * i),
                                ld_any(src, src_bf16, sr * ld + c + 2 * i + 1));
        *reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * cols + c) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
}

// 32 x 32 tiles through shared memory: reads along a source row, writes
// along a destination row. blockIdx.x: 32-column block of j, blockIdx.y: of c.
__global__ void __launch_bounds__(256) transpose_pad_kernel(
    const void* __restrict__ src, int src_bf16, long long ld, const int32_t* __restrict__ idx,
    int nrows, int cols, const int32_t* __restrict__ poff, const int32_t* __restrict__ offsets,
    int E, int kpad, __nv_bfloat16* __restrict__ dst) {
    __shared__ float tile[32][33];
    pdl_wait();
    pdl_trigger();
    const int j0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of 32 per pass
    for (int jj = ty; jj < 32; jj += 8) {
        const int j = j0 + jj;
        long long row = -1;
        if (j < kpad) {
            if (poff == nullptr) {
                if (j < nrows) row = j;
            } else {
                int lo = 0, hi = E;  // poff[lo] <= j < poff[hi]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (poff[mid] <= j)
                        lo = mid;
                    else
                        hi = mid;
                }
                const int k = j - poff[lo];
                if (k < offsets[lo + 1] - offsets[lo]) row = offsets[lo] + k;
            }
        }
        float v = 0.0f;
        const int c = c0 + tx;
        if (row >= 0 && c < cols) {
            const long long sr = idx ? idx[row] : row;
            v = ld_any(src, src_bf16, sr * ld + c);
        }
        tile[jj][tx] = v;
    }
    __syncthreads();
    for (int cc = ty; cc < 32; cc += 8) {
        const int c = c0 + cc, j = j0 + tx;
        if (c < cols && j < kpad) dst[static_cast<long long>(c) * kpad + j] = __float2bfloat16_rn(tile[tx][cc]);
    }
}

// one warp per row; dg summed over the row in a fixed order (lane-strided
// partials, then a fixed shuffle tree)
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const float* __restrict__ a,
                                                         const float* __restrict__ u,
                                                         const float* __restrict__ dh, long long ld,
                                                         int rows, int F,
                                                         const float* __restrict__ rowscale,
                                                         __nv_bfloat16* __restrict__ da,
                                                         __nv_bfloat16* __restrict__ du,
                                                         __nv_bfloat16* __restrict__ hw,
                                                         float* __restrict__ dg) {
    pdl_wait();
    pdl_trigger();
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (r >= rows) return;
    const int lane = threadIdx.x & 31;
    const float g = rowscale ? rowscale[r] : 1.0f;
    const long long base = static_cast<long long>(r) * ld;
    const long long ob = static_cast<long long>(r) * F;
    float part = 0.0f;
    for (int c = lane * 4; c < F; c += 128) {
        const float4 av = *reinterpret_cast<const float4*>(a + base + c);
        const float4 uv = *reinterpret_cast<const float4*>(u + base + c);
        const float4 dv = *reinterpret_cast<const float4*>(dh + base + c);
        const float aa[4] = {av.x, av.y, av.z, av.w}, uu[4] = {uv.x, uv.y, uv.z, uv.w};
        const float dd[4] = {dv.x, dv.y, dv.z, dv.w};
        float o_da[4], o_du[4], o_hw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float sg = 1.0f / (1.0f + expf(-aa[i]));
            const float si = aa[i] * sg;
            const float h = si * uu[i];
            o_da[i] = g * dd[i] * uu[i] * (sg * (1.0f + aa[i] * (1.0f - sg)));
            o_du[i] = g * dd[i] * si;
            o_hw[i] = g * h;
            part += dd[i] * h;
        }
        *reinterpret_cast<uint2*>(da + ob + c) = make_uint2(pack_bf16x2(o_da[0], o_da[1]), pack_bf16x2(o_da[2], o_da[3]));
        *reinterpret_cast<uint2*>(du + ob + c) = make_uint2(pack_bf16x2(o_du[0], o_du[1]), pack_bf16x2(o_du[2], o_du[3]));
        *reinterpret_cast<uint2*>(hw + ob + c) = make_uint2(pack_bf16x2(o_hw[0], o_hw[1]), pack_bf16x2(o_hw[2], o_hw[3]));
    }
    if (dg != nullptr) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) dg[r] = part;
    }
}

}  // namespace

cudaError_t launch_pad_offsets(const int32_t* offsets, int E, int32_t* poff, cudaStream_t s) {
    return launch_pdl(pad_offsets_kernel, dim3(1), dim3(32), 0, s, offsets, E, poff);
}

cudaError_t launch_gather_bf16(const void* src, int src_bf16, long long ld, const int32_t* idx,
                               int rows, int cols, __nv_bfloat16* dst, cudaStream_t s) {
    if (cols % 8) return cudaErrorInvalidValue;
    return launch_pdl(gather_bf16_kernel, dim3((rows * 32 + 255) / 256), dim3(256), 0, s, src,
                      src_bf16, ld, idx, rows, cols, dst);
}

cudaError_t launch_transpose_pad(const void* src, int src_bf16, long long ld, const int32_t* idx,
                                 int nrows, int cols, const int32_t* poff, const int32_t* offsets,
                                 int E, int kpad, __nv_bfloat16* dst, cudaStream_t s) {
    const dim3 grid((kpad + 31) / 32, (cols + 31) / 32);
    return launch_pdl(transpose_pad_kernel, grid, dim3(256), 0, s, src, src_bf16, ld, idx, nrows,
                      cols, poff, offsets, E, kpad, dst);
}

cudaError_t launch_swiglu_bwd(const float* a, const float* u, const float* dh, long long ld, int rows,
                              int F, const float* rowscale, __nv_bfloat16* da, __nv_bfloat16* du,
                              __nv_bfloat16* hw, float* dg, cudaStream_t s) {
    if (F % 4 || ld % 4) return cudaErrorInvalidValue;
    return launch_pdl(swiglu_bwd_kernel, dim3((rows * 32 + 255) / 256), dim3(256), 0, s, a, u, dh,
                      ld, rows, F, rowscale, da, du, hw, dg);
}

}  // namespace moe
