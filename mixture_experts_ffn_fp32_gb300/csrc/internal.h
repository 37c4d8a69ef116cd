// Internal declarations shared by the translation units of libmoe (not part
// of the public C ABI in include/moe.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// Count of kernels launched by the library (moe_launch_count).
void note_launch(int n = 1);

// Launch with programmatic stream serialisation (see pdl_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_launch();
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// The same with thread-block clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, int cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    note_launch();
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// The same as a cooperative launch (every CTA resident at once; the grid must
// fit the device). Programmatic serialisation is requested too; where the
// runtime refuses the pair, the launch goes without it (decided once).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_coop(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args&&... args) {
    static int with_pdl = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = with_pdl ? 2 : 1;
    note_launch();
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess && with_pdl) {
        cudaGetLastError();
        with_pdl = 0;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, args...);
    }
    return e;
}
// Wait limit of device-side bounded waits, in ns.
uint64_t wait_timeout_ns();
// Number of SMs of the current device (cached per device).
int num_sms();

// ---------------------------------------------------------------------------
// Workspace layout. Every region is 256-byte aligned; offsets in bytes.
// ---------------------------------------------------------------------------
constexpr int DISPATCH_CHUNK = 1024;   // assignments per dispatch CTA
constexpr int TC_BM = 128;             // rows per tcgen05 GEMM tile of one CTA (a pair: 2 TC_BM)
constexpr int SIMT_BM = 64;            // rows per FP32 SIMT GEMM tile
constexpr int ROUTER_CHUNK = 256;      // tensor-core router: reduction chunk per split-K slice

struct WsLayout {
    size_t err, topk_idx, topk_w, margin, top_scores, scores;
    size_t chunk_counts, chunk_base, counts, offsets, mt_prefix;
    size_t sorted_token, sorted_w, inv;
    size_t xs, z, h, hs, ys, routed, shout, xstage, ostage, qb, w3, rpart;
    size_t ga, gu, gas, gus;  // saved gate / up products (save_gate_up): routed rows, shared
    size_t logits, stats_part;  // routing diagnostics: r [T, E], per-CTA partial sums
    size_t dctr;                // fused decode back end: counters [E + 3]
    size_t fs_tags, fs_cnt;     // one-launch front end / dispatch: CTA tag lines, CTA counts (dispatch)
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
    int* err_clear;   // if set, block 0 zeroes this error word and the dispatch ticket after
                      // it (first kernel of a forward)
    float* logits;    // if set: the raw FP32 logits r [T, E] (routing diagnostics)
    unsigned* zero = nullptr;  // if set (one-launch routers): block 0 zeroes zero[0, nzero)
    int nzero = 0;             //   (the fused decode back end's counters)
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);
// Whether the router of this layer runs as one launch that honours RouterArgs::zero.
bool router_one_launch(int T, int d, int E, int x_bf16);
// Tensor-core router pieces: W3 [3, d, E] BF16 = exact split of W [d, E];
// routing from logits summed over nsplit partial slices part [nsplit, T, E].
cudaError_t launch_router_split(const float* W, int d, int E, void* W3, int* err_clear,
                                cudaStream_t s);
cudaError_t launch_route_from_logits(const float* part, int nsplit, const RouterArgs& a,
                                     cudaStream_t s);
// Tensor-core router used when x is BF16, E > 32, E % 8 == 0 and d % ROUTER_CHUNK == 0.
bool router_on_tensor_cores(const moe_config& c);
// Decode batches (T <= 128, 128 < E <= 256, d a multiple of 8 (BF16 x) or 4):
// one cooperative launch reading W_router once (router.cu); part: [S, T, E]
// FP32 (S = router_decode_slices), tags: FRONT_SMALL_MAX_CTAS 128-byte lines
// and the epoch line (no initial state needed); a.err_clear must be set.
bool router_decode_ok(int T, int d, int E, int x_bf16);
int router_decode_slices(int T, int d, int E);
cudaError_t launch_router_decode(const RouterArgs& a, float* part, unsigned long long* tags, cudaStream_t s);
// Few tokens and E > 32: FP32 partial logits per 256-long slice of d on many
// CTAs, summed and routed by route_from_logits (needs a workspace's rpart).
bool router_chunked(const moe_config& c);
cudaError_t launch_router_chunked(const RouterArgs& a, float* part, cudaStream_t s);
int router_chunked_nsplit(int d, int E);  // slices of the chunked router
// Split-K slices of the tensor-core router GEMM (one per chunk of d).
int router_ksplit(int T, int d);

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
    int* ticket;   // zero when no dispatch is running; the word after *err in a workspace
};
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s, int* n_launched);
// Dispatch + gather of the routed rows (row_bytes each, from src into dst in
// expert order) in one launch, for T*K <= DISPATCH_CHUNK.
cudaError_t launch_dispatch_gather(const DispatchArgs& a, const void* src, int row_bytes, void* dst,
                                   cudaStream_t s);

// The same for T*K <= DISPATCH_WIDE_MAX, over many CTAs (each counts all
// assignments itself and places its own range of them).
constexpr int DISPATCH_WIDE_MAX = 16384;
cudaError_t launch_dispatch_gather_wide(const DispatchArgs& a, const void* src, int row_bytes,
                                        void* dst, cudaStream_t s);

// Router, dispatch and row gather in one cooperative launch (front_small.cu)
// for BF16 x, E <= 8, 1024 < T*K <= DISPATCH_WIDE_MAX. tags: FRONT_SMALL_MAX_CTAS
// 128-byte lines, each CTA's count words at the start of its line, then the
// epoch line (no initial state needed).
constexpr int FRONT_SMALL_MAX_CTAS = 256;

// Dispatch and row gather in one cooperative launch (dispatch_onepass.cu) for
// DISPATCH_WIDE_MAX < T*K <= 1024 * CTAs, E <= 256. tags: DISPATCH_ONEPASS_MAX_CTAS
// 128-byte lines (one 64-bit tag each) and the epoch line, cnt: DISPATCH_ONEPASS_MAX_CTAS * E
// ints of scratch (no initial state needed).
constexpr int DISPATCH_ONEPASS_MAX_CTAS = 256;
bool dispatch_onepass_ok(int T, int K, int E);
cudaError_t launch_dispatch_gather_onepass(const DispatchArgs& a, const void* src, int row_bytes, void* dst,
                                           unsigned long long* tags, int* cnt, cudaStream_t s);
bool front_small_ok(int T, int d, int E, int K);
cudaError_t launch_front_small(const RouterArgs& ra, const DispatchArgs& da, void* xs,
                               unsigned long long* tags, cudaStream_t s);

// dst[r, :] = src[rowidx[r], :] for r < rows, row_bytes a multiple of 16.
cudaError_t launch_gather_rows(const void* src, const int32_t* rowidx, int rows, int row_bytes,
                               void* dst, cudaStream_t s);

// out[t, :] = sum_k ys[inv[t, k], :] (+ addend[t, :]) in FP32 (k ascending, addend
// last), stored BF16 or FP32. ys and addend are FP32; addend may be NULL.
cudaError_t launch_gather_sum(const float* ys, const int32_t* inv, int T, int K, int cols,
                              const float* addend, void* out, int out_bf16, cudaStream_t s);
// The same with the routed rows in the 24-bit blocked layout (ys24; cols % 256 == 0).
cudaError_t launch_gather_sum_f24(const void* ys24, const int32_t* inv, int T, int K, int cols,
                                  const float* addend, void* out, int out_bf16, cudaStream_t s);
// Same sum, stored as two BF16 parts hi = bf16(v), lo = bf16(v - hi) in
// out2 [T, 2*cols_pad]: hi in columns [0, cols), lo in [cols_pad, cols_pad + cols),
// zeros elsewhere (hi + lo carries ~16 significant bits of v).
cudaError_t launch_gather_sum_split(const float* ys, const int32_t* inv, int T, int K, int cols,
                                    int cols_pad, void* out2, cudaStream_t s);

// ---- tcgen05 grouped GEMM -------------------------------------------------
// A segment group: rows of A multiplied by a per-segment B matrix.
//   Group 0 ("routed"): E segments, segment e = A rows [offsets[e], offsets[e+1]),
//     B = expert e's matrix; output rows = the same A rows.
//   Group 1 ("dense"): S segments all over A rows [0, rows1), B = matrix s;
//     output columns [s*N1, (s+1)*N1).
// tc_grouped_gemm epilogues (TcGemmArgs::swiglu)
// TC_PLAIN_ACC: the single product of group 1 (split-K slices), each slice's
// k-range reduced in chunks of TcGroup::kchunk k-blocks: every chunk's product
// goes through tensor memory on its own and the epilogue adds the chunks in
// FP32, in order, before it stores the slice (the tensor-core router: short
// accumulation chains, few partial slices).
enum { TC_PLAIN = 0, TC_SWIGLU = 1, TC_SWIGLU_BWD = 2, TC_PLAIN_ACC = 3 };
struct TcGroup {
    int enabled;
    int K;              // reduction length of this group
    const void* A;      // [rows, K] BF16, row pitch lda elements (see a_kmod)
    int lda;
    int rows;           // group 0: T*K (rows of A), group 1: rows1
    const void* B0;     // [Z, K, N] BF16 (gate / down / plain)
    const void* B1;     // [Z, K, N] BF16 (up), only for the SwiGLU kernel
    int Z;              // number of B matrices (E or S)
    int N;              // output columns per segment
    void* out;          // [rows, out_ld] BF16 or FP32
    int out_ld;
    int out_f32;
    int a_kmod = 0;     // > 0: A is [rows, a_kmod] and reduction index k reads A column k % a_kmod
    int a_kgroup = 0;   // > 0 (k-blocks of 64): reduction k-block kb reads A k-block
    int a_krep = 1;     //   (kb / (a_kgroup * a_krep)) * a_kgroup + kb % a_kgroup
    int b_kmod = 0;     // > 0: reduction index k reads B row k % b_kmod
    int b_rows = 0;     // > 0: B has b_rows rows per matrix (rows beyond read as zero)
    int ksplit = 1;     // group 1 only: split K into ksplit slices; slice s writes the partial
                        // product to out rows [s*rows, (s+1)*rows) (needs Z == 1)
    int kchunk = 0;     // TC_PLAIN_ACC, group 1: k-blocks per chunk (each slice a whole
                        // number of chunks)
    // A second reduction segment (group 1 of a plain product, Z == 1, K a multiple
    // of 64): out += A2 [rows, K2] (pitch lda2) times B2 [K2, N], accumulated with
    // the first segment's product in one pass (the remaps above apply to the first).
    const void* A2 = nullptr;
    int lda2 = 0;
    const void* B2 = nullptr;
    int K2 = 0;
    // TC_SWIGLU: a_out / u_out (optional, both or neither, BF16 like out): the gate
    // and up products a = A B0, u = A B1 themselves, in out's rows, columns and pitch.
    void* a_out = nullptr;
    void* u_out = nullptr;
    // TC_SWIGLU_BWD: with a, u the gate and up products of row r, column c (the
    // SwiGLU layout of `out`, pitch out_ld), the upstream gradient dh of h
    // (FP32, pitch dh_ld) and the row's gate weight g (group 0: rowscale0,
    // group 1: 1): da = g dh u SiLU'(a), du = g dh SiLU(a) and g h as BF16
    // rows of da / du / hw (pitch out_ld). Group 0 reads dh and writes in the
    // expert-padded row layout (TcGemmArgs::poff; padding rows zeroed), group 1
    // in token rows; group 0 also dgpart[r, 2 tile + half] = sum of dh h over
    // each 64 of the tile's columns (r the unpadded row).
    const float* dh = nullptr;
    int dh_ld = 0;
    void* da = nullptr;
    void* du = nullptr;
    void* hw = nullptr;
    float* dgpart = nullptr;
};

struct TcGemmArgs {
    TcGroup g[2];
    int E;                       // group 0 segment count
    const int32_t* offsets;      // group 0 [E+1]
    const int32_t* mt_prefix;    // group 0 [2(E+1)]: tiles of TC_BM rows, then of 2 TC_BM rows
    int swiglu;                  // TC_SWIGLU: h = SiLU(A B0) * (A B1); TC_PLAIN: single product;
                                 // TC_SWIGLU_BWD: the SwiGLU backward epilogue (TcGroup)
    const int32_t* poff;         // TC_SWIGLU_BWD group 0: padded column offsets [E+1]
    const float* rowscale0;      // group 0: multiply row r by rowscale0[r]
    const float* addend;         // group 1: add addend[r, col] (FP32 [rows1, add_ld])
    int add_ld;
    int* err;
    // Group 0 of a plain product with FP32 output may instead be stored in the
    // 24-bit blocked layout (ys24 below) where the launch takes a form that
    // writes it: f24_ok allows it, *used_f24 (if set) tells whether it did.
    int f24_ok = 0;
    int* used_f24 = nullptr;
};
cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t s);

// The 24-bit blocked row layout of routed rows (ys24): each row of N columns
// (N % 256 == 0) is N / 256 blocks of 768 bytes; block b holds columns
// 256 b .. 256 b + 255 as 256 16-bit high parts, then 256 8-bit low parts
// (f32_to_f24). Row pitch 3 N bytes.
constexpr int YS24_BLOCK = 256;

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

// ---- routing diagnostics -----------------------------------------------------
constexpr int STATS_TOKENS = 64;  // tokens per CTA of the partial-sum kernel
cudaError_t launch_routing_stats(const float* logits, const int32_t* idx, int T, int E, int K,
                                 float* part, float* out, cudaStream_t s);

// ---- balancers --------------------------------------------------------------
cudaError_t launch_quantile(int T, int E, int K, const float* top_scores, const float* scores,
                            float* braw, float* bias, cudaStream_t s, int* n_launched);
cudaError_t launch_sign_bias(int E, int N, int K, const int32_t* counts, float* bias,
                             float alpha, cudaStream_t s);

// ---- self-test of bounded waits --------------------------------------------
cudaError_t launch_wait_selftest(int* err, uint64_t timeout_ns, cudaStream_t s);

// Tensor-map encoder (driver entry point, resolved once).
// ---- fused decode back end (decode_fused.cu) ---------------------------------
// Everything after the router of a batch of at most 128 tokens in one launch:
// dispatch (written to counts .. inv), row gather (xs, for the backward pass),
// gate/up (h, hs), down (ys, shout), combine (out). ctr [E + 3] must be zero
// (the router launch zeroes it).
struct DecodeArgs {
    int T, d, F, E, K, S, Fs;
    const void* x;
    const int32_t* idx;
    const float* w;
    const void *W_gate, *W_up, *W_down, *Ws_gate, *Ws_up, *Ws_down;
    int32_t *counts, *offsets, *mt_prefix, *sorted_token;
    float* sorted_w;
    int32_t* inv;
    void *xs, *h, *hs;
    float *ys, *shout;
    void* out;
    int out_f32;
    unsigned* ctr;
    int* err;
};
bool decode_fused_shape_ok(int T, int d, int F, int E, int K, int S, int Fs);
cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s);

bool encode_tmap(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box);


// ---------------------------------------------------------------------------
// Backward pass (gemm_gen.cu, backward.cu)
// ---------------------------------------------------------------------------
// One operand of gen_gemm: element (i, j) at p + zoff + I(i) s0 + J(j) s1,
// I / J the optional index lists idx0 / idx1; dimension 0 is m for A and k
// for B. zs advances the base per problem (GEN_DENSE; B of GEN_MSEG).
struct GenOp {
    const void* p;
    int bf16;
    long long s0, s1, zs;
    const int32_t* idx0;
    const int32_t* idx1;
};
enum { GEN_DENSE = 0, GEN_MSEG = 1, GEN_KSEG = 2 };
enum { GEN_EPI_STORE = 0, GEN_EPI_ACCUM = 1, GEN_EPI_SWIGLU_BWD = 2 };
constexpr int MAXSEG = 256;
struct GenGemm {
    int mode, M, N, K, Z;
    const int32_t* offsets;  // [Z+1] device: GEN_MSEG rows / GEN_KSEG reduction ranges
    GenOp A, B0, B1;         // B1: the up operand of the SwiGLU backward
    float* C;                // output (store / accumulate), element (m, n) at C + z c_zs + m ldc + n
    long long ldc, c_zs;
    int a_m_contig, b_n_contig;  // which index of A / B is the contiguous one
    const float* rowscale;   // optional per-row factor (gate weight)
    const float* dh;         // SwiGLU backward: upstream gradient of h, same layout as C
    float *da, *du, *hw;     // SwiGLU backward outputs, same layout as C
    float* dwpart;           // optional [rows, column tiles] partials of sum dh h
    int ksplit;              // GEN_DENSE store/accumulate: > 1 splits the reduction
    float* part;             // ksplit x Z x M x N FP32 partials (ksplit > 1)
};
cudaError_t launch_gen_gemm(const GenGemm& p, int epi, cudaStream_t s);
// ksplit a GEN_DENSE product should use with `part_floats` of scratch (1: none).
int gen_gemm_ksplit(const GenGemm& p, size_t part_floats);
int gen_gemm_ntiles(int N);  // column tiles of a gen_gemm output of width N

// NT grouped GEMM on the tensor cores (gemm_nt.cu): C (+)= A B^T, both
// operands K-major BF16. A: rows x K (pitch ld); B: Z slices of rows x K.
enum { NT_DENSE = 0, NT_MSEG = 1, NT_KSEG = 2 };
struct NtOperand {
    const void* p;
    long long rows, K, ld, Z, zstride;
};
struct NtGemm {
    int mode, M, N, K, Z, nph;  // K: per-phase reduction (multiple of 64); NT_KSEG: offsets
    NtOperand A[2], B[2];
    int a_kofs[2], b_zc[2];     // per phase: A column offset, B slice offset
    int a_zrow, b_zrow, b_z3;   // NT_DENSE: per-problem A row, B row and B slice steps
    int a_mn = 0, b_mn = 0;     // operand stored MN-major: K rows of its rows-many columns
                                // (pitch ld; rows a multiple of 64; not with NT_MSEG)
    const int32_t* offsets;     // [Z+1] device: NT_MSEG rows / NT_KSEG reduction columns
    float* C;
    long long ldc, c_zs;
    int accumulate;
    int* err;
    // SwiGLU-backward epilogue (sg_a set; C unused): the accumulator at output row r,
    // column c is dh, the gradient of h = SiLU(a) u. With a = sg_a, u = sg_u (BF16
    // gate and up products; NT_MSEG: row i of segment z read at row sg_off[z] + i
    // of pitch sg_ld, the segment's rows past sg_off[z+1] - sg_off[z] are padding;
    // otherwise at the output's own index, pitch ldc) and g = sg_g[that row] (NULL:
    // 1), writes BF16 da = g dh u SiLU'(a), du = g dh SiLU(a), g h at the output
    // index (pitch ldc, NT_DENSE slices c_zs apart; zeros on padding rows), and
    // sg_part[row * sg_npart + c / 64] = the sum of dh h over each 64 columns
    // (NULL: not written). N a multiple of 64.
    const __nv_bfloat16* sg_a = nullptr;
    const __nv_bfloat16* sg_u = nullptr;
    const int32_t* sg_off = nullptr;
    long long sg_ld = 0;
    const float* sg_g = nullptr;
    __nv_bfloat16* sg_da = nullptr;
    __nv_bfloat16* sg_du = nullptr;
    __nv_bfloat16* sg_hw = nullptr;
    float* sg_part = nullptr;
    int sg_npart = 0;
};
cudaError_t launch_nt_gemm(const NtGemm& g, cudaStream_t s);

// Backward operand preparation (bwd_prep.cu).
// poff[z] = sum over z' < z of cnt_z' rounded up to 64 (cnt from offsets), z <= E.
cudaError_t launch_pad_offsets(const int32_t* offsets, int E, int32_t* poff, cudaStream_t s);
// dst[r, :cols] = BF16(src[idx ? idx[r] : r, :cols]) for r < rows; src FP32 or BF16.
cudaError_t launch_gather_bf16(const void* src, int src_bf16, long long ld, const int32_t* idx,
                               int rows, int cols, __nv_bfloat16* dst, cudaStream_t s);
// Rows gathered into the expert-padded row layout: dst [kpad, cols] BF16,
// row j = poff[z] + i holds src row idx[offsets[z] + i] for i < cnt_z (the
// rows of segment z), zero rows up to poff[z + 1]; without poff, row j = j
// for j < nrows.
cudaError_t launch_gather_pad_bf16(const void* src, int src_bf16, long long ld, const int32_t* idx,
                                   int nrows, int cols, const int32_t* poff, const int32_t* offsets,
                                   int E, int kpad, __nv_bfloat16* dst, cudaStream_t s);
// inv_pad[i] = poff[idx[i]] + inv[i] - offsets[idx[i]] for i < TK.
cudaError_t launch_pad_inverse(const int32_t* inv, const int32_t* idx, int TK, const int32_t* poff,
                               const int32_t* offsets, int32_t* inv_pad, cudaStream_t s);

// Backward scratch (FP32 arrays, byte offsets into the backward workspace).
struct BwdLayout {
    int tc;  // the tensor-core form (bwd_on_tensor_cores)
    size_t dhp, da, du, hw, dwpart, dxs, dhs, das, dus, hs, dr, dg, glat, routed, dz;
    // tensor-core form only, in the expert-padded row layout where routed: BF16
    // operand copies, the SwiGLU backward's outputs, padded positions
    size_t poff, invp, gys, zs, dab, dub, hwb, dwrow, dxsp;
    size_t doutb, dasb, dusb, hsb, routedb, dzb;
    size_t wrt, cp, rpart;  // W_router^T; router coefficient per padded row; per-64-row partials
    long long tkpad, tpad;
    size_t kpart, kpart_floats;  // split-K partials of the long-reduction CUDA-core products
    bool saved = false;          // tensor-core form on the forward's saved gate / up products
    size_t total;
};
// BF16 layers whose widths are multiples of 64 run the backward's expert
// contractions on the tensor cores (gemm_nt.cu); the others on gemm_gen.cu.
bool bwd_on_tensor_cores(const moe_config& c);
BwdLayout plan_backward(const moe_config& c);
// Enqueue the backward on s; ws holds the forward's routing and dispatch.
moe_status backward_impl(const moe_config& c, const void* x, const moe_weights& w, const float* dout,
                         const moe_grads& g, uint8_t* ws, uint8_t* bws, cudaStream_t s);

}  // namespace moe
