// Operand preparation for the tensor-core backward (gemm_nt.cu reads both
// operands K-major): BF16 copies of gathered rows, transposed copies laid out
// per expert with each expert's rows padded to a multiple of 64 columns
// (zero columns between experts, so an expert's weight-gradient reduction
// covers whole k-blocks of its own rows only). The SwiGLU backward itself
// runs in the epilogue of the recomputing gate/up GEMM (gemm_tc.cu).
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

}  // namespace moe
