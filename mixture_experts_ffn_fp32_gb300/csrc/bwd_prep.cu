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

// Source row of padded column j (-1: a zero column).
MOE_DEV long long pad_row(int j, int nrows, int kpad, const int32_t* poff, const int32_t* offsets,
                          int E) {
    if (j >= kpad) return -1;
    if (poff == nullptr) return j < nrows ? j : -1;
    int lo = 0, hi = E;  // poff[lo] <= j < poff[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (poff[mid] <= j)
            lo = mid;
        else
            hi = mid;
    }
    const int k = j - poff[lo];
    return k < offsets[lo + 1] - offsets[lo] ? offsets[lo] + k : -1;
}

// 64 x 64 tiles through shared memory, 16-byte accesses on both sides:
// 8 BF16 (or 4 FP32) consecutive source columns per load, 8 consecutive
// destination columns per store. blockIdx.x: 64-block of j, blockIdx.y: of c.
// cols is a multiple of 8.
template <bool SRC_BF16>
__global__ void __launch_bounds__(256) transpose_pad_kernel(
    const void* __restrict__ src, long long ld, const int32_t* __restrict__ idx, int nrows, int cols,
    const int32_t* __restrict__ poff, const int32_t* __restrict__ offsets, int E, int kpad,
    __nv_bfloat16* __restrict__ dst) {
    __shared__ float tile[64][65];
    __shared__ long long srow[64];
    pdl_wait();
    pdl_trigger();
    const int j0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
    if (threadIdx.x < 64) {
        const long long r = pad_row(j0 + threadIdx.x, nrows, kpad, poff, offsets, E);
        srow[threadIdx.x] = r < 0 ? -1 : (idx ? idx[r] : r);
    }
    __syncthreads();
    if (SRC_BF16) {
        // 64 rows x 8 chunks of 8 BF16: two chunks per thread
        for (int i = threadIdx.x; i < 64 * 8; i += 256) {
            const int jj = i >> 3, ch = i & 7;
            const int c = c0 + ch * 8;
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (srow[jj] >= 0 && c < cols) {
                const uint4 q = *reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(src) + srow[jj] * ld + c);
                v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
                v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) tile[jj][ch * 8 + t] = v[t];
        }
    } else {
        // 64 rows x 16 chunks of 4 FP32: four chunks per thread
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int jj = i >> 4, ch = i & 15;
            const int c = c0 + ch * 4;
            float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
            if (srow[jj] >= 0 && c < cols)
                q = *reinterpret_cast<const float4*>(static_cast<const float*>(src) + srow[jj] * ld + c);
            tile[jj][ch * 4] = q.x;
            tile[jj][ch * 4 + 1] = q.y;
            tile[jj][ch * 4 + 2] = q.z;
            tile[jj][ch * 4 + 3] = q.w;
        }
    }
    __syncthreads();
    // 64 destination rows (c) x 8 chunks of 8 BF16 (j)
    for (int i = threadIdx.x; i < 64 * 8; i += 256) {
        const int cc = i >> 3, ch = i & 7;
        const int c = c0 + cc, j = j0 + ch * 8;
        if (c >= cols || j >= kpad) continue;
        uint32_t pk[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
            pk[t] = pack_bf16x2(tile[ch * 8 + 2 * t][cc], tile[ch * 8 + 2 * t + 1][cc]);
        *reinterpret_cast<uint4*>(dst + static_cast<long long>(c) * kpad + j) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
}

// The SwiGLU backward of a 64 x 64 block (64 padded columns j of the
// expert layout, i.e. 64 rows, by 64 hidden columns c): da, du row-major BF16
// for the rows that exist, and da, du, g h transposed into the padded layout
// (zero columns for padding), plus dgpart[row, c / 64] = sum over the block's
// c of dh h. One pass over a, u, dh instead of a row pass and three
// transposes.
__global__ void __launch_bounds__(256) swiglu_bwd_t_kernel(
    const float* __restrict__ a, const float* __restrict__ u, const float* __restrict__ dh,
    long long ld, int nrows, int F, const float* __restrict__ rowscale,
    const int32_t* __restrict__ poff, const int32_t* __restrict__ offsets, int E, int kpad,
    __nv_bfloat16* __restrict__ da, __nv_bfloat16* __restrict__ du, __nv_bfloat16* __restrict__ daT,
    __nv_bfloat16* __restrict__ duT, __nv_bfloat16* __restrict__ hwT, float* __restrict__ dgpart) {
    __shared__ __nv_bfloat16 t_da[64][66], t_du[64][66], t_hw[64][66];  // [row j][c]
    __shared__ float s_part[64][17];
    __shared__ long long srow[64];
    pdl_wait();
    pdl_trigger();
    const int j0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
    if (threadIdx.x < 64) srow[threadIdx.x] = pad_row(j0 + threadIdx.x, nrows, kpad, poff, offsets, E);
    __syncthreads();
    // 64 rows x 16 chunks of 4 columns: four chunks per thread
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
        const int jj = i >> 4, ch = i & 15;
        const int c = c0 + ch * 4;
        const long long r = srow[jj];
        float o_da[4] = {0.f, 0.f, 0.f, 0.f}, o_du[4] = {0.f, 0.f, 0.f, 0.f}, o_hw[4] = {0.f, 0.f, 0.f, 0.f};
        float part = 0.0f;
        if (r >= 0 && c < F) {
            const float g = rowscale ? rowscale[r] : 1.0f;
            const float4 av = *reinterpret_cast<const float4*>(a + r * ld + c);
            const float4 uv = *reinterpret_cast<const float4*>(u + r * ld + c);
            const float4 dv = *reinterpret_cast<const float4*>(dh + r * ld + c);
            const float aa[4] = {av.x, av.y, av.z, av.w}, uu[4] = {uv.x, uv.y, uv.z, uv.w};
            const float dd[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float sg = 1.0f / (1.0f + expf(-aa[q]));
                const float si = aa[q] * sg;
                const float h = si * uu[q];
                o_da[q] = g * dd[q] * uu[q] * (sg * (1.0f + aa[q] * (1.0f - sg)));
                o_du[q] = g * dd[q] * si;
                o_hw[q] = g * h;
                part += dd[q] * h;
            }
            const long long o = r * F + c;
            *reinterpret_cast<uint2*>(da + o) = make_uint2(pack_bf16x2(o_da[0], o_da[1]), pack_bf16x2(o_da[2], o_da[3]));
            *reinterpret_cast<uint2*>(du + o) = make_uint2(pack_bf16x2(o_du[0], o_du[1]), pack_bf16x2(o_du[2], o_du[3]));
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            t_da[jj][ch * 4 + q] = __float2bfloat16_rn(o_da[q]);
            t_du[jj][ch * 4 + q] = __float2bfloat16_rn(o_du[q]);
            t_hw[jj][ch * 4 + q] = __float2bfloat16_rn(o_hw[q]);
        }
        s_part[jj][ch] = part;
    }
    __syncthreads();
    if (dgpart != nullptr && threadIdx.x < 64 && srow[threadIdx.x] >= 0) {
        float v = 0.0f;
        for (int ch = 0; ch < 16; ++ch) v += s_part[threadIdx.x][ch];
        dgpart[srow[threadIdx.x] * ((F + 63) / 64) + blockIdx.y] = v;
    }
    // transposed: 64 destination rows (c) x 8 chunks of 8 padded columns (j)
    for (int i = threadIdx.x; i < 64 * 8; i += 256) {
        const int cc = i >> 3, ch = i & 7;
        const int c = c0 + cc, j = j0 + ch * 8;
        if (c >= F || j >= kpad) continue;
        uint32_t p0[4], p1[4], p2[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int r0 = ch * 8 + 2 * t;
            p0[t] = static_cast<uint32_t>(__bfloat16_as_ushort(t_da[r0][cc])) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(t_da[r0 + 1][cc])) << 16);
            p1[t] = static_cast<uint32_t>(__bfloat16_as_ushort(t_du[r0][cc])) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(t_du[r0 + 1][cc])) << 16);
            p2[t] = static_cast<uint32_t>(__bfloat16_as_ushort(t_hw[r0][cc])) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(t_hw[r0 + 1][cc])) << 16);
        }
        const long long o = static_cast<long long>(c) * kpad + j;
        *reinterpret_cast<uint4*>(daT + o) = make_uint4(p0[0], p0[1], p0[2], p0[3]);
        *reinterpret_cast<uint4*>(duT + o) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
        *reinterpret_cast<uint4*>(hwT + o) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
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
    if (cols % 8 || kpad % 8 || ld % 8) return cudaErrorInvalidValue;
    const dim3 grid((kpad + 63) / 64, (cols + 63) / 64);
    if (src_bf16)
        return launch_pdl(transpose_pad_kernel<true>, grid, dim3(256), 0, s, src, ld, idx, nrows, cols,
                          poff, offsets, E, kpad, dst);
    return launch_pdl(transpose_pad_kernel<false>, grid, dim3(256), 0, s, src, ld, idx, nrows, cols,
                      poff, offsets, E, kpad, dst);
}

cudaError_t launch_swiglu_bwd_t(const float* a, const float* u, const float* dh, long long ld,
                                int nrows, int F, const float* rowscale, const int32_t* poff,
                                const int32_t* offsets, int E, int kpad, __nv_bfloat16* da,
                                __nv_bfloat16* du, __nv_bfloat16* daT, __nv_bfloat16* duT,
                                __nv_bfloat16* hwT, float* dgpart, cudaStream_t s) {
    if (F % 64 || ld % 4 || kpad % 64) return cudaErrorInvalidValue;
    const dim3 grid(kpad / 64, F / 64);
    return launch_pdl(swiglu_bwd_t_kernel, grid, dim3(256), 0, s, a, u, dh, ld, nrows, F, rowscale,
                      poff, offsets, E, kpad, da, du, daT, duT, hwT, dgpart);
}

}  // namespace moe
