// moe_dispatch_noalloc: the sorted dispatch of moe_dispatch for callers that
// cannot allocate device memory. Some callers run where cudaMalloc is not
// available to them: an embedding runtime that owns all device memory and
// hands out only the tensors it manages, or code that must not allocate
// after start-up because allocation can synchronise the device or fail under
// memory pressure. moe_dispatch needs a caller-provided workspace for its
// per-chunk histograms; this variant keeps that scratch in a fixed array in
// the library's own device memory instead, so the caller passes only the
// inputs and outputs.
//
// The array is sized for at most NOALLOC_MAX_TK = 65536 assignments (T * K)
// and E <= 256 experts: about 130 KB, which every GPU that loads the library
// keeps until the process exits. All calls share it, so calls whose work
// overlaps on the GPU (different streams without ordering between them) race
// on it and give wrong results; calls ordered on one stream are fine.
#include "common.cuh"
#include "internal.h"

#include <mutex>

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

constexpr int NOALLOC_MAX_TK = 65536;
constexpr int NOALLOC_MAX_E = 256;
constexpr int NOALLOC_CHUNKS = NOALLOC_MAX_TK / DISPATCH_CHUNK;

// [0, 64): error word and dispatch ticket (cleared at the start of every call)
// then chunk_counts and chunk_base [NOALLOC_CHUNKS * E], then mt_prefix [2 (E + 1)]
constexpr size_t NOALLOC_WORDS =
    64 + 2 * static_cast<size_t>(NOALLOC_CHUNKS) * NOALLOC_MAX_E + 2 * (NOALLOC_MAX_E + 1);

static __device__ __align__(256) int32_t g_dispatch_scratch[NOALLOC_WORDS];

// Identity of the current context: its process-unique id (cuCtxGetId), so
// that a context destroyed and made again (cudaDeviceReset, for one) is seen
// as new even if its handle value comes back. Driver entry points are taken
// through the runtime; the library does not link libcuda.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array, looked up once per device and context with
// that device current (in host code the symbol is only a stand-in for the
// address). The lookup is redone when the device's context is not the one the
// cached address was taken in.
int32_t* scratch_address(cudaError_t* err) {
    static std::mutex mu;
    static int32_t* addr[64] = {};
    static unsigned long long ctx_of[64] = {};
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    // cudaSetDevice makes the device's primary context current (and creates it
    // if no call has yet)
    *err = cudaSetDevice(dev);
    if (*err != cudaSuccess) return nullptr;
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) {
        *err = cudaErrorDeviceUninitialized;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (addr[dev] == nullptr || ctx_of[dev] != ctx) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (*err != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int32_t*>(p);
        ctx_of[dev] = ctx;
    }
    return addr[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx,
                                        const float* topk_w, int32_t* counts, int32_t* offsets,
                                        int32_t* sorted_token, float* sorted_w, int32_t* inv,
                                        void* stream) {
    if (!cfg || !topk_idx || !topk_w || !counts || !offsets || !sorted_token || !sorted_w || !inv)
        return MOE_ERR_INVALID_ARG;
    const moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    const long long TK = static_cast<long long>(cfg->T) * cfg->K;
    if (TK > NOALLOC_MAX_TK || cfg->E > NOALLOC_MAX_E) return MOE_ERR_UNSUPPORTED;
    cudaError_t e = cudaSuccess;
    int32_t* base = scratch_address(&e);
    if (base == nullptr) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the error word and the dispatch ticket must start at zero; everything
    // else is fully rewritten
    if (cudaMemsetAsync(base, 0, 2 * sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    const int nchunks = static_cast<int>((TK + DISPATCH_CHUNK - 1) / DISPATCH_CHUNK);
    DispatchArgs da{};
    da.idx = topk_idx;
    da.w = topk_w;
    da.T = cfg->T;
    da.K = cfg->K;
    da.E = cfg->E;
    da.nchunks = nchunks;
    da.bm = cfg->dtype == MOE_BF16 ? TC_BM : SIMT_BM;
    da.chunk_counts = base + 64;
    da.chunk_base = base + 64 + static_cast<size_t>(nchunks) * cfg->E;
    da.mt_prefix = base + 64 + 2 * static_cast<size_t>(NOALLOC_CHUNKS) * NOALLOC_MAX_E;
    da.counts = counts;
    da.offsets = offsets;
    da.sorted_token = sorted_token;
    da.sorted_w = sorted_w;
    da.inv = inv;
    da.err = base;
    da.ticket = base + 1;
    return launch_dispatch(da, s, nullptr) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
