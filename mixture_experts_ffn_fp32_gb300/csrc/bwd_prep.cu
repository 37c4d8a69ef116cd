// Operand preparation for the tensor-core backward: BF16 copies of rows, and
// the expert-padded row layout (each expert's rows, then zero rows up to a
// multiple of 64, so an expert's weight-gradient reduction covers whole
// 64-row k-blocks of its own rows only): padded offsets, padded positions of
// the assignments, rows gathered into it. The SwiGLU backward itself runs in
// the epilogue of the recomputing gate/up GEMM (gemm_tc.cu).
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

// Row gather into the expert-padded row layout: dst row j (of kpad) =
// BF16(src[idx[pos(j)], :cols]) for the rows of the experts, zero for the
// padding rows. One warp per row, 8 columns per lane step.
__global__ void __launch_bounds__(256) gather_pad_bf16_kernel(
    const void* __restrict__ src, int src_bf16, long long ld, const int32_t* __restrict__ idx,
    int nrows, int cols, const int32_t* __restrict__ poff, const int32_t* __restrict__ offsets, int E,
    int kpad, __nv_bfloat16* __restrict__ dst) {
    pdl_wait();
    pdl_trigger();
    const int j = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (j >= kpad) return;
    const int lane = threadIdx.x & 31;
    const long long r = pad_row(j, nrows, kpad, poff, offsets, E);
    const long long sr = r < 0 ? -1 : (idx ? idx[r] : r);
    for (int c = lane * 8; c < cols; c += 256) {
        uint32_t pk[4] = {0u, 0u, 0u, 0u};
        if (sr >= 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                pk[i] = pack_bf16x2(ld_any(src, src_bf16, sr * ld + c + 2 * i),
                                    ld_any(src, src_bf16, sr * ld + c + 2 * i + 1));
        }
        *reinterpret_cast<uint4*>(dst + static_cast<long long>(j) * cols + c) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
}

// Padded position of every assignment: inv_pad = poff[e] + inv - offsets[e].
__global__ void __launch_bounds__(256) pad_inverse_kernel(const int32_t* __restrict__ inv,
                                                          const int32_t* __restrict__ idx, int TK,
                                                          const int32_t* __restrict__ poff,
                                                          const int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ inv_pad) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= TK) return;
    const int e = idx[i];
    inv_pad[i] = poff[e] + inv[i] - offsets[e];
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

cudaError_t launch_gather_pad_bf16(const void* src, int src_bf16, long long ld, const int32_t* idx,
                                   int nrows, int cols, const int32_t* poff, const int32_t* offsets,
                                   int E, int kpad, __nv_bfloat16* dst, cudaStream_t s) {
    if (cols % 8) return cudaErrorInvalidValue;
    return launch_pdl(gather_pad_bf16_kernel, dim3((kpad * 32 + 255) / 256), dim3(256), 0, s, src,
                      src_bf16, ld, idx, nrows, cols, poff, offsets, E, kpad, dst);
}

cudaError_t launch_pad_inverse(const int32_t* inv, const int32_t* idx, int TK, const int32_t* poff,
                               const int32_t* offsets, int32_t* inv_pad, cudaStream_t s) {
    return launch_pdl(pad_inverse_kernel, dim3((TK + 255) / 256), dim3(256), 0, s, inv, idx, TK, poff,
                      offsets, inv_pad);
}

}  // namespace moe
