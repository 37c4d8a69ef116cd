// Internal declarations shared by the translation units of libmoe (not part
// of the public C ABI in include/moe.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Count of kernels launched by the library (moe_launch_count).
void note_launch(int n = 1);
// Wait limit of device-side bounded waits, in ns.
uint64_t wait_timeout_ns();
// Number of SMs of the current device (cached per device).
int num_sms();

// ---------------------------------------------------------------------------
// Workspace layout. Every region is 256-byte aligned; offsets in bytes.
// ---------------------------------------------------------------------------
constexpr int DISPATCH_CHUNK = 1024;   // assignments per dispatch CTA
constexpr int TC_BM = 128;             // rows per tcgen05 GEMM tile
constexpr int SIMT_BM = 64;            // rows per FP32 SIMT GEMM tile

struct WsLayout {
    size_t err, topk_idx, topk_w, margin, top_scores, scores;
    size_t chunk_counts, chunk_base, counts, offsets, mt_prefix;
    size_t sorted_token, sorted_w, inv;
    size_t xs, z, h, hs, ys, routed, shout, xstage, ostage, qb;
    size_t total;
    int nchunks;
};

WsLayout plan_workspace(const moe_config& c);
moe_status validate_config(const moe_config& c);

// ---------------------------------------------------------------------------
// Kernel launchers (each returns cudaGetLastError() of its launch)
// ---------------------------------------------------------------------------
struct RouterArgs {
    const void* x;
    int x_bf16;
    const float* W;
    const float* bias;
    int T, d, E, K, gate, renorm;
    float scale;
    int32_t* idx;
    float* w;
    float* margin;
    float* top_scores;
    float* scores;
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);

struct DispatchArgs {
    const int32_t* idx;
    const float* w;
    int T, K, E, nchunks, bm;
    int32_t* chunk_counts;
    int32_t* chunk_base;
    int32_t* counts;
    int32_t* offsets;
    int32_t* mt_prefix;
    int32_t* sorted_token;
    float* sorted_w;
    int32_t* inv;
    int* err;
};
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s, int* n_launched);

// dst[r, :] = src[rowidx[r], :] for r < rows, row_bytes a multiple of 16.
cudaError_t launch_gather_rows(const void* src, const int32_t* rowidx, int rows, int row_bytes,
                               void* dst, cudaStream_t s);

// out[t, :] = sum_k ys[inv[t, k], :] (+ addend[t, :]) in FP32, stored BF16 or FP32.
cudaError_t launch_gather_sum(const void* ys, int ys_bf16, const int32_t* inv, int T, int K,
                              int cols, void* out, int out_bf16, cudaStream_t s);

// ---- tcgen05 grouped GEMM -------------------------------------------------
// A segment group: rows of A multiplied by a per-segment B matrix.
//   Group 0 ("routed"): E segments, segment e = A rows [offsets[e], offsets[e+1]),
//     B = expert e's matrix; output rows = the same A rows.
//   Group 1 ("dense"): S segments all over A rows [0, rows1), B = matrix s;
//     output columns [s*N1, (s+1)*N1).
struct TcGroup {
    int enabled;
    const void* A;      // [rows, K] BF16, row pitch lda elements
    int lda;
    int rows;           // group 0: T*K (rows of A), group 1: rows1
    const void* B0;     // [Z, K, N] BF16 (gate / down / plain)
    const void* B1;     // [Z, K, N] BF16 (up), only for the SwiGLU kernel
    int Z;              // number of B matrices (E or S)
    int N;              // output columns per segment
    void* out;          // [rows, out_ld] BF16 or FP32
    int out_ld;
    int out_f32;
};

struct TcGemmArgs {
    TcGroup g[2];
    int K;                       // reduction length
    int E;                       // group 0 segment count
    const int32_t* offsets;      // group 0 [E+1]
    const int32_t* mt_prefix;    // group 0 [E+1], m-tiles of TC_BM rows
    int swiglu;                  // 1: h = SiLU(A B0) * (A B1); 0: single product
    const float* rowscale0;      // group 0: multiply row r by rowscale0[r]
    const int32_t* inv;          // group 1: add sum_k ys[inv[r*Kr + k]]
    const void* ys;              // BF16 [*, ys_ld]
    int ys_ld, Kr;
    const float* addend;         // group 1: add addend[r, col] (FP32 [rows1, add_ld])
    int add_ld;
    int* err;
};
cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t s);

// ---- FP32 SIMT grouped GEMM (same groups, FP32 everywhere) ----------------
struct SimtGroup {
    int enabled;
    const float* A;
    int lda;
    const int32_t* a_rows;   // group 0: A row of output row r is a_rows[r] (NULL: r)
    int rows;
    const float* B0;
    const float* B1;
    int Z, N;
    float* out;
    int out_ld;
};
struct SimtGemmArgs {
    SimtGroup g[2];
    int K, E;
    const int32_t* offsets;
    const int32_t* mt_prefix;    // m-tiles of SIMT_BM rows
    int swiglu;
    const float* rowscale0;
    const int32_t* inv;
    const float* ys;
    int ys_ld, Kr;
};
cudaError_t launch_simt_gemm(const SimtGemmArgs& a, cudaStream_t s);

// ---- balancers --------------------------------------------------------------
cudaError_t launch_quantile(int T, int E, int K, const float* top_scores, const float* scores,
                            float* braw, float* bias, cudaStream_t s, int* n_launched);
cudaError_t launch_sign_bias(int E, int N, int K, const int32_t* counts, float* bias,
                             float alpha, cudaStream_t s);

// ---- self-test of bounded waits --------------------------------------------
cudaError_t launch_wait_selftest(int* err, uint64_t timeout_ns, cudaStream_t s);

// Tensor-map encoder (driver entry point, resolved once).
bool encode_tmap(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace moe
