// C ABI of libmoe (declared in include/moe.h): host-side validation,
// workspace planning and the forward pipeline that enqueues the kernels of
// router.cu, dispatch.cu, gemm_tc.cu / gemm_simt.cu and balance.cu.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

static std::atomic<unsigned long long> g_launches{0};
static std::atomic<long long> g_timeout_ns{1000LL * 1000LL * 1000LL};

void note_launch(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }
uint64_t wait_timeout_ns() { return static_cast<uint64_t>(g_timeout_ns.load()); }

int num_sms() {
    static int cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

// ---------------------------------------------------------------------------
// Tensor-map encoding through the driver entry point (no libcuda link).
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode_tmap(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box) {
    EncodeTiledFn fn = get_encoder();
    if (!fn) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                          const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Validation and workspace layout
// ---------------------------------------------------------------------------
moe_status validate_config(const moe_config& c) {
    if (c.T < 1 || c.d < 1 || c.d_ff < 1 || c.E < 1 || c.K < 1) return MOE_ERR_INVALID_ARG;
    if (c.K > c.E) return MOE_ERR_INVALID_ARG;
    if (c.gate != MOE_GATE_SOFTMAX_TOPK && c.gate != MOE_GATE_SOFTMAX_ALL_RENORM &&
        c.gate != MOE_GATE_SIGMOID)
        return MOE_ERR_INVALID_ARG;
    if (c.gate == MOE_GATE_SIGMOID && c.K + 1 > c.E) return MOE_ERR_INVALID_ARG;
    if (c.dtype != MOE_F32 && c.dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c.out_dtype != MOE_F32 && c.out_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c.dtype == MOE_F32 && c.out_dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
    if (c.n_shared < 0 || (c.n_shared > 0 && c.shared_d_ff < 1)) return MOE_ERR_INVALID_ARG;
    if (c.latent_dim < 0) return MOE_ERR_INVALID_ARG;
    if (!(c.routed_scale == c.routed_scale)) return MOE_ERR_INVALID_ARG;
    if (c.save_gate_up != 0 && c.save_gate_up != 1) return MOE_ERR_INVALID_ARG;
    if (c.E > 256 || c.K > 16) return MOE_ERR_UNSUPPORTED;
    // row pitches feed 16-byte vector accesses and TMA strides; tiles store 16 columns at a time
    if (c.d % 16 || c.d_ff % 16) return MOE_ERR_UNSUPPORTED;
    if (c.n_shared > 0 && c.shared_d_ff % 16) return MOE_ERR_UNSUPPORTED;
    if (c.latent_dim > 0 && (c.latent_dim % 16 || c.dtype != MOE_BF16)) return MOE_ERR_UNSUPPORTED;
    const long long TK = static_cast<long long>(c.T) * c.K;
    if (TK > (1LL << 30) || static_cast<long long>(c.T) * c.d > (1LL << 40)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

static size_t align_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool router_on_tensor_cores(const moe_config& c) {
    return c.dtype == MOE_BF16 && c.E > 32 && c.E % 8 == 0 && c.d % ROUTER_CHUNK == 0;
}

// Up to 512 tokens the FP32 cluster router (one launch; slices of d summed
// through distributed shared memory) is faster than the tensor-core router
// (three launches): up to 128 experts with W_router slices in shared memory,
// up to 256 reading them from global memory. (Where a slice of x and
// W_router would not fit shared memory, the chunked two-launch form runs.)
bool router_chunked(const moe_config& c) { return c.E > 32 && c.E <= 256 && c.T <= 512; }

// Partial slices of the tensor-core router: each slice is a run of whole
// ROUTER_CHUNK-long chunks of d, and the GEMM adds a slice's chunks in FP32 in
// its epilogue. The count minimises the chunks the busiest SM reduces (units
// = 128-token row tiles x slices, spread over 152 SMs) plus a quarter chunk
// per slice for writing and reading the partial logits: the 8192-token
// layers take 2.
int router_ksplit(int T, int d) {
    const int chunks = d / ROUTER_CHUNK;
    const int tiles = (T + TC_BM - 1) / TC_BM;
    int best = 1;
    double best_cost = 1e30;
    for (int sl = 1; sl <= chunks; ++sl) {
        const int per = (chunks + sl - 1) / sl;
        const int real = (chunks + per - 1) / per;
        if (real != sl) continue;
        const int rounds = (tiles * sl + 151) / 152;
        const double cost = static_cast<double>(rounds) * per + 0.25 * sl;
        if (cost < best_cost) {
            best_cost = cost;
            best = sl;
        }
    }
    return best;
}

// The router GEMM: x [T, d] against the chunk-interleaved split weights W3
// [3d, E]; reduction k-block kb reads x k-block (kb / 12) * 4 + kb % 4; each
// chunk of 12 k-blocks (the lo, mid and hi parts of 256 rows of W_router)
// accumulates in tensor memory on its own.
static TcGroup router_group(const void* x, int T, int d, int E, void* w3, void* rpart) {
    TcGroup g{1, 3 * d, x, d, T, w3, nullptr, 1, E, rpart, E, 1};
    g.a_kgroup = ROUTER_CHUNK / 64;
    g.a_krep = 3;
    g.ksplit = router_ksplit(T, d);
    g.kchunk = 3 * ROUTER_CHUNK / 64;
    return g;
}

static int latent_pad(int L) { return (L + 63) / 64 * 64; }

static_assert(GRID_EPOCH_LINE >= FRONT_SMALL_MAX_CTAS && GRID_EPOCH_LINE >= DISPATCH_ONEPASS_MAX_CTAS,
              "the grid barrier's epoch line follows every CTA's tag line");

WsLayout plan_workspace(const moe_config& c) {
    WsLayout L;
    memset(&L, 0, sizeof(L));
    const size_t T = c.T, K = c.K, E = c.E, TK = T * K;
    const size_t es = (c.dtype == MOE_BF16) ? 2 : 4;
    const size_t de = c.latent_dim ? c.latent_dim : c.d;
    L.nchunks = static_cast<int>((TK + DISPATCH_CHUNK - 1) / DISPATCH_CHUNK);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes);
        return at;
    };
    L.err = take(256);
    L.topk_idx = take(TK * 4);
    L.topk_w = take(TK * 4);
    L.margin = take(T * 4);
    const bool sig = c.gate == MOE_GATE_SIGMOID;
    L.top_scores = sig ? take(T * (K + 1) * 4) : 0;
    L.scores = sig ? take(T * E * 4) : 0;
    L.chunk_counts = take(static_cast<size_t>(L.nchunks) * E * 4);
    L.chunk_base = take(static_cast<size_t>(L.nchunks) * E * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.mt_prefix = take(2 * (E + 1) * 4);  // tiles of bm and of 2 bm rows
    L.sorted_token = take(TK * 4);
    L.sorted_w = take(TK * 4);
    L.inv = take(TK * 4);
    const bool bf = c.dtype == MOE_BF16;
    L.xs = bf ? take(TK * de * es) : 0;
    L.z = c.latent_dim ? take(T * de * es) : 0;
    L.h = take(TK * c.d_ff * es);
    const size_t SF = static_cast<size_t>(c.n_shared) * (c.n_shared ? c.shared_d_ff : 0);
    L.hs = SF ? take(T * SF * es) : 0;
    // the gate and up products, kept for a backward pass on the tensor cores
    const bool sv = bf && c.save_gate_up && bwd_on_tensor_cores(c);
    L.ga = sv ? take(TK * c.d_ff * 2) : 0;
    L.gu = sv ? take(TK * c.d_ff * 2) : 0;
    L.gas = (sv && SF) ? take(T * SF * 2) : 0;
    L.gus = (sv && SF) ? take(T * SF * 2) : 0;
    L.ys = take(TK * de * 4);  // FP32: the K routed rows are summed before one final rounding
    // latent routed sum as a BF16 hi/lo pair, each part padded to a multiple of 64 columns
    L.routed = c.latent_dim ? take(T * 2 * static_cast<size_t>(latent_pad(c.latent_dim)) * 2) : 0;
    // FP32 shared-expert output (latent layers add the shared product inside the up-projection)
    L.shout = (c.n_shared && !c.latent_dim) ? take(T * c.d * 4) : 0;
    L.xstage = take(T * c.d * es);
    L.ostage = take(T * c.d * (c.out_dtype == MOE_BF16 ? 2 : 4));
    L.qb = take(E * 4);
    const bool chk = router_chunked(c);
    const bool tcr = router_on_tensor_cores(c) && !chk;
    L.w3 = tcr ? take(3 * static_cast<size_t>(c.d) * E * 2) : 0;
    // (decode batches: the one-launch decode router's partials, at most 32 slices)
    const bool rdec = chk && c.T <= 128 && c.E > 128;
    size_t nsplit = chk ? router_chunked_nsplit(c.d, c.E) : router_ksplit(c.T, c.d);
    if (rdec && nsplit < 32) nsplit = 32;
    L.rpart = (tcr || chk) ? take(nsplit * T * E * 4) : 0;
    L.logits = take(T * E * 4);
    L.stats_part = take(((T + STATS_TOKENS - 1) / STATS_TOKENS) * (2 * E + 1) * 4);
    L.dctr = take((E + 3) * 4);
    // one-launch front end (E <= 8), one-launch dispatch (larger batches) or decode
    // router: CTA tag lines (the front end's count words), the dispatch's per-CTA
    // count table
    const bool fsw = bf && c.latent_dim == 0 && E <= 8 && TK > 1024 && TK <= DISPATCH_WIDE_MAX;
    const bool dow = bf && E <= 256 && TK > DISPATCH_WIDE_MAX && TK <= 1024ull * DISPATCH_ONEPASS_MAX_CTAS;
    L.fs_tags = (fsw || dow || rdec) ? take((GRID_EPOCH_LINE + 1) * 128) : 0;  // + the epoch line
    L.fs_cnt = dow ? take(static_cast<size_t>(DISPATCH_ONEPASS_MAX_CTAS) * (E > 8 ? E : 8) * 4) : 0;
    L.total = o;
    return L;
}

// ---------------------------------------------------------------------------
// Stage timing (instrumentation)
// ---------------------------------------------------------------------------
enum Stage { ST_ROUTE = 0, ST_LATENT_DOWN, ST_DISPATCH, ST_GATHER, ST_GATEUP, ST_DOWN, ST_COMBINE,
             ST_LATENT_UP, ST_FUSED, ST_FRONT, ST_COUNT };
static const char* kStageNames[ST_COUNT] = {"router", "latent_down", "dispatch", "gather",
                                            "gate_up", "down", "combine", "latent_up",
                                            "decode_fused", "route_dispatch_gather"};

struct Timing {
    std::mutex mu;
    bool on = false;
    uint32_t mask = 0xFFFFFFFFu;
    int max_calls = 0, calls = 0;
    std::vector<cudaEvent_t> ev;  // [max_calls][ST_COUNT][2]
    std::vector<char> used;       // [max_calls][ST_COUNT]
};
static Timing g_timing;

struct StageRec {
    int call = -1;
    cudaStream_t s = nullptr;
    void begin(int st) {
        if (call >= 0 && ((g_timing.mask >> st) & 1u))
            cudaEventRecord(g_timing.ev[(call * ST_COUNT + st) * 2], s);
    }
    void end(int st) {
        if (call >= 0 && ((g_timing.mask >> st) & 1u)) {
            cudaEventRecord(g_timing.ev[(call * ST_COUNT + st) * 2 + 1], s);
            g_timing.used[call * ST_COUNT + st] = 1;
        }
    }
};

static StageRec stage_rec(cudaStream_t s) {
    StageRec r;
    r.s = s;
    std::lock_guard<std::mutex> lk(g_timing.mu);
    if (g_timing.on && g_timing.calls < g_timing.max_calls) r.call = g_timing.calls++;
    return r;
}

static moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static moe_status check_weights(const moe_config& c, const moe_weights* w) {
    if (!w || !w->W_router || !w->W_gate || !w->W_up || !w->W_down) return MOE_ERR_INVALID_ARG;
    if (c.n_shared > 0 && (!w->Ws_gate || !w->Ws_up || !w->Ws_down)) return MOE_ERR_INVALID_ARG;
    if (c.latent_dim > 0 && (!w->W_down_latent || !w->W_up_latent)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {w->W_router, w->W_gate, w->W_up, w->W_down, w->Ws_gate, w->Ws_up,
                          w->Ws_down, w->W_down_latent, w->W_up_latent};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (w->bias && (reinterpret_cast<uintptr_t>(w->bias) & 3u)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// The router of cfg on x into ra's outputs (ws optional: with it, the
// workspace error word is cleared and the chunked or tensor-core paths may run).
static moe_status run_router(const moe_config& c, RouterArgs ra, const float* W_router,
                             const void* x, uint8_t* ws, const WsLayout& L, cudaStream_t s) {
    if (ws != nullptr) ra.err_clear = reinterpret_cast<int*>(ws + L.err);
    if (ws != nullptr && router_chunked(c)) {
        if (L.fs_tags != 0 && router_decode_ok(c.T, c.d, c.E, ra.x_bf16))
            return cuda_status(launch_router_decode(ra, reinterpret_cast<float*>(ws + L.rpart),
                                                    reinterpret_cast<unsigned long long*>(ws + L.fs_tags), s));
        return cuda_status(launch_router_chunked(ra, reinterpret_cast<float*>(ws + L.rpart), s));
    }
    if (ws != nullptr && router_on_tensor_cores(c)) {
        ra.err_clear = nullptr;
        int* err = reinterpret_cast<int*>(ws + L.err);
        cudaError_t e;
        if ((e = launch_router_split(W_router, c.d, c.E, ws + L.w3, err, s)) != cudaSuccess)
            return cuda_status(e);
        const int ks = router_ksplit(c.T, c.d);
        TcGemmArgs g{};
        g.g[1] = router_group(x, c.T, c.d, c.E, ws + L.w3, ws + L.rpart);
        g.err = err;
        if ((e = launch_tc_gemm(g, s)) != cudaSuccess) return cuda_status(e);
        return cuda_status(
            launch_route_from_logits(reinterpret_cast<const float*>(ws + L.rpart), ks, ra, s));
    }
    return cuda_status(launch_router(ra, s));
}

static RouterArgs router_args(const moe_config& c, const void* x, const float* W_router,
                              const float* bias) {
    RouterArgs ra{};
    ra.x = x;
    ra.x_bf16 = c.dtype == MOE_BF16;
    ra.W = W_router;
    ra.bias = bias;
    ra.T = c.T; ra.d = c.d; ra.E = c.E; ra.K = c.K; ra.gate = c.gate;
    ra.renorm = c.renormalize; ra.scale = c.routed_scale;
    return ra;
}

// A decode batch of a BF16 layer without latent projection (at most 128
// tokens, the router in one launch) runs everything after the router in one
// persistent launch (decode_fused.cu): two launches for the whole forward.
static bool decode_fused(const moe_config& c) {
    return c.dtype == MOE_BF16 && c.latent_dim == 0 && !c.save_gate_up &&
           decode_fused_shape_ok(c.T, c.d, c.d_ff, c.E, c.K, c.n_shared, c.n_shared ? c.shared_d_ff : 0) &&
           router_one_launch(c.T, c.d, c.E, 1);
}

// Enqueue the whole forward on s. x and out are device pointers.
static moe_status forward_impl(const moe_config& c, const void* x, const moe_weights& w, void* out,
                               uint8_t* ws, cudaStream_t s) {
    const WsLayout L = plan_workspace(c);
    const bool bf = c.dtype == MOE_BF16;
    const int T = c.T, K = c.K, E = c.E, TK = T * K;
    const int de = c.latent_dim ? c.latent_dim : c.d;
    const int S = c.n_shared, Fs = c.shared_d_ff, SF = S * (S ? Fs : 0);
    const size_t es = bf ? 2 : 4;
    const int of32 = c.out_dtype == MOE_F32 ? 1 : 0;
    int* err = reinterpret_cast<int*>(ws + L.err);
    auto P = [&](size_t off) { return static_cast<void*>(ws + off); };
    int32_t* idx = static_cast<int32_t*>(P(L.topk_idx));
    float* tw = static_cast<float*>(P(L.topk_w));
    int32_t* offsets = static_cast<int32_t*>(P(L.offsets));
    int32_t* mt_prefix = static_cast<int32_t*>(P(L.mt_prefix));
    int32_t* sorted_token = static_cast<int32_t*>(P(L.sorted_token));
    float* sorted_w = static_cast<float*>(P(L.sorted_w));
    int32_t* inv = static_cast<int32_t*>(P(L.inv));
    StageRec rec = stage_rec(s);
    cudaError_t e;

    DispatchArgs da{};
    da.idx = idx;
    da.w = tw;
    da.T = T; da.K = K; da.E = E; da.nchunks = L.nchunks;
    da.bm = bf ? TC_BM : SIMT_BM;
    da.chunk_counts = static_cast<int32_t*>(P(L.chunk_counts));
    da.chunk_base = static_cast<int32_t*>(P(L.chunk_base));
    da.counts = static_cast<int32_t*>(P(L.counts));
    da.offsets = offsets;
    da.mt_prefix = mt_prefix;
    da.sorted_token = sorted_token;
    da.sorted_w = sorted_w;
    da.inv = inv;
    da.err = err;
    da.ticket = err + 1;

    // 1. router (with the dispatch, for a decode batch)
    RouterArgs ra = router_args(c, x, static_cast<const float*>(w.W_router),
                                static_cast<const float*>(w.bias));
    ra.idx = idx;
    ra.w = tw;
    ra.margin = static_cast<float*>(P(L.margin));
    ra.top_scores = L.top_scores ? static_cast<float*>(P(L.top_scores)) : nullptr;
    ra.scores = L.scores ? static_cast<float*>(P(L.scores)) : nullptr;
    const bool fused = decode_fused(c);
    if (fused) {
        ra.zero = static_cast<unsigned*>(P(L.dctr));
        ra.nzero = E + 3;
    }
    // few experts, a prefill batch: router, dispatch and row gather in one launch
    const bool front = !fused && L.fs_tags != 0 && front_small_ok(T, c.d, E, K);
    if (front) {
        rec.begin(ST_FRONT);
        ra.err_clear = err;
        if ((e = launch_front_small(ra, da, P(L.xs), static_cast<unsigned long long*>(P(L.fs_tags)), s)) !=
            cudaSuccess)
            return cuda_status(e);
        rec.end(ST_FRONT);
    } else {
        rec.begin(ST_ROUTE);
        const moe_status rs = run_router(c, ra, static_cast<const float*>(w.W_router), x, ws, L, s);
        if (rs != MOE_OK) return rs;
        rec.end(ST_ROUTE);
    }

    if (fused) {
        // 2. everything else in one launch
        rec.begin(ST_FUSED);
        DecodeArgs a{};
        a.T = T; a.d = c.d; a.F = c.d_ff; a.E = E; a.K = K; a.S = S; a.Fs = S ? Fs : 0;
        a.x = x; a.idx = idx; a.w = tw;
        a.W_gate = w.W_gate; a.W_up = w.W_up; a.W_down = w.W_down;
        a.Ws_gate = w.Ws_gate; a.Ws_up = w.Ws_up; a.Ws_down = w.Ws_down;
        a.counts = da.counts; a.offsets = offsets; a.mt_prefix = mt_prefix;
        a.sorted_token = sorted_token; a.sorted_w = sorted_w; a.inv = inv;
        a.xs = P(L.xs); a.h = P(L.h); a.hs = S ? P(L.hs) : nullptr;
        a.ys = static_cast<float*>(P(L.ys));
        a.shout = S ? static_cast<float*>(P(L.shout)) : nullptr;
        a.out = out; a.out_f32 = of32;
        a.ctr = static_cast<unsigned*>(P(L.dctr));
        a.err = err;
        if ((e = launch_decode_fused(a, s)) != cudaSuccess) return cuda_status(e);
        rec.end(ST_FUSED);
        return MOE_OK;
    }

    // 1b. latent compression z = x W_down_latent (once per token)
    const void* ex_src = x;  // rows the routed experts act on
    if (c.latent_dim) {
        rec.begin(ST_LATENT_DOWN);
        TcGemmArgs g{};
        g.g[1] = TcGroup{1, c.d, x, c.d, T, w.W_down_latent, nullptr, 1, c.latent_dim, P(L.z),
                         c.latent_dim, 0};
        g.err = err;
        if ((e = launch_tc_gemm(g, s)) != cudaSuccess) return cuda_status(e);
        ex_src = P(L.z);
        rec.end(ST_LATENT_DOWN);
    }

    // 2. dispatch (BF16 batches of up to DISPATCH_WIDE_MAX assignments: with the row
    //    gather, one launch)
    // (a stage without a launch records no events: its time is nil)
    const bool dg1 = bf && L.nchunks == 1;
    const bool dgw = bf && !dg1 && TK <= DISPATCH_WIDE_MAX;
    const bool onepass = bf && !dg1 && !dgw && L.fs_tags != 0 && dispatch_onepass_ok(T, K, E);
    const bool dg = dg1 || dgw || front || onepass;
    if (!front) rec.begin(ST_DISPATCH);
    if (front) {
        // done by the front-end launch
    } else if (onepass) {
        if ((e = launch_dispatch_gather_onepass(da, ex_src, de * 2, P(L.xs),
                                                static_cast<unsigned long long*>(P(L.fs_tags)),
                                                static_cast<int*>(P(L.fs_cnt)), s)) != cudaSuccess)
            return cuda_status(e);
    } else if (dg1) {
        if ((e = launch_dispatch_gather(da, ex_src, de * 2, P(L.xs), s)) != cudaSuccess)
            return cuda_status(e);
    } else if (dgw) {
        if ((e = launch_dispatch_gather_wide(da, ex_src, de * 2, P(L.xs), s)) != cudaSuccess)
            return cuda_status(e);
    } else if ((e = launch_dispatch(da, s, nullptr)) != cudaSuccess) {
        return cuda_status(e);
    }
    if (!front) rec.end(ST_DISPATCH);

    if (bf) {
        float* ys = static_cast<float*>(P(L.ys));
        int ys_f24 = 0;  // routed rows stored in the 24-bit blocked layout (ys24)
        float* shout = L.shout ? static_cast<float*>(P(L.shout)) : nullptr;
        // 3. gather the routed rows into expert order
        if (!dg) {
            rec.begin(ST_GATHER);
            if ((e = launch_gather_rows(ex_src, sorted_token, TK, de * 2, P(L.xs), s)) != cudaSuccess)
                return cuda_status(e);
            rec.end(ST_GATHER);
        }

        // 4. gate/up with the SiLU(gate) * up epilogue: routed experts (group 0, on the
        //    sorted rows) and shared experts (group 1, on x) in one launch
        rec.begin(ST_GATEUP);
        {
            TcGemmArgs g{};
            g.g[0] = TcGroup{1, de, P(L.xs), de, TK, w.W_gate, w.W_up, E, c.d_ff, P(L.h), c.d_ff, 0};
            if (S) g.g[1] = TcGroup{1, c.d, x, c.d, T, w.Ws_gate, w.Ws_up, S, Fs, P(L.hs), SF, 0};
            if (L.ga) {
                g.g[0].a_out = P(L.ga);
                g.g[0].u_out = P(L.gu);
                if (S) {
                    g.g[1].a_out = P(L.gas);
                    g.g[1].u_out = P(L.gus);
                }
            }
            g.E = E; g.offsets = offsets; g.mt_prefix = mt_prefix; g.swiglu = 1; g.err = err;
            if ((e = launch_tc_gemm(g, s)) != cudaSuccess) return cuda_status(e);
        }
        rec.end(ST_GATEUP);

        // 5. down projections in one launch: routed rows scaled by their gate weight
        //    (group 0, FP32 ys) and the shared experts summed over their concatenated
        //    hidden width (group 1, FP32 shared output)
        rec.begin(ST_DOWN);
        {
            TcGemmArgs g{};
            g.g[0] = TcGroup{1, c.d_ff, P(L.h), c.d_ff, TK, w.W_down, nullptr, E, de, ys, de, 1};
            // (latent layers: the shared experts' down product joins the up-projection below)
            if (S && !c.latent_dim)
                g.g[1] = TcGroup{1, SF, P(L.hs), SF, T, w.Ws_down, nullptr, 1, c.d, shout, c.d, 1};
            g.E = E; g.offsets = offsets; g.mt_prefix = mt_prefix; g.swiglu = 0;
            g.rowscale0 = sorted_w; g.err = err;
            // routed rows in the 24-bit blocked layout where the launch's form writes it
            g.f24_ok = c.latent_dim == 0;
            g.used_f24 = &ys_f24;
            if ((e = launch_tc_gemm(g, s)) != cudaSuccess) return cuda_status(e);
        }
        rec.end(ST_DOWN);

        // 6. deterministic combine of the K routed rows of each token (+ shared)
        rec.begin(ST_COMBINE);
        if (!c.latent_dim) {
            if ((e = ys_f24 ? launch_gather_sum_f24(ys, inv, T, K, de, shout, out, !of32, s)
                            : launch_gather_sum(ys, inv, T, K, de, shout, out, !of32, s)) != cudaSuccess)
                return cuda_status(e);
            rec.end(ST_COMBINE);
        } else {
            // routed sum in latent width as a BF16 hi/lo pair: the up projection reads
            // [hi | lo] against W_up_latent twice, so the sum keeps ~16 bits into it
            const int Lp = latent_pad(de);
            if ((e = launch_gather_sum_split(ys, inv, T, K, de, Lp, P(L.routed), s)) != cudaSuccess)
                return cuda_status(e);
            rec.end(ST_COMBINE);
            rec.begin(ST_LATENT_UP);
            TcGemmArgs g{};
            // out = [routed hi | routed lo] [W_up_latent; W_up_latent] + hs Ws_down: the
            // shared experts' down product as a second reduction segment of the same
            // accumulation (no FP32 shared output written and read back)
            g.g[1] = TcGroup{1, 2 * Lp, P(L.routed), 2 * Lp, T, w.W_up_latent, nullptr, 1, c.d, out,
                             c.d, of32};
            g.g[1].b_kmod = Lp;
            g.g[1].b_rows = de;
            if (S) {
                g.g[1].A2 = P(L.hs);
                g.g[1].lda2 = SF;
                g.g[1].B2 = w.Ws_down;
                g.g[1].K2 = SF;
            }
            g.swiglu = 0; g.err = err;
            if ((e = launch_tc_gemm(g, s)) != cudaSuccess) return cuda_status(e);
            rec.end(ST_LATENT_UP);
        }
    } else {
        // FP32 layer on the CUDA cores; routed A rows read through sorted_token
        const float* xf = static_cast<const float*>(x);
        rec.begin(ST_GATEUP);
        {
            SimtGemmArgs g{};
            g.g[0] = SimtGroup{1, xf, c.d, sorted_token, TK, static_cast<const float*>(w.W_gate),
                               static_cast<const float*>(w.W_up), E, c.d_ff,
                               static_cast<float*>(P(L.h)), c.d_ff};
            if (S)
                g.g[1] = SimtGroup{1, xf, c.d, nullptr, T, static_cast<const float*>(w.Ws_gate),
                                   static_cast<const float*>(w.Ws_up), S, Fs,
                                   static_cast<float*>(P(L.hs)), SF};
            g.K = c.d; g.E = E; g.offsets = offsets; g.mt_prefix = mt_prefix; g.swiglu = 1;
            if ((e = launch_simt_gemm(g, s)) != cudaSuccess) return cuda_status(e);
        }
        rec.end(ST_GATEUP);
        rec.begin(ST_DOWN);
        {
            SimtGemmArgs g{};
            g.g[0] = SimtGroup{1, static_cast<const float*>(P(L.h)), c.d_ff, nullptr, TK,
                               static_cast<const float*>(w.W_down), nullptr, E, c.d,
                               static_cast<float*>(P(L.ys)), c.d};
            g.K = c.d_ff; g.E = E; g.offsets = offsets; g.mt_prefix = mt_prefix; g.swiglu = 0;
            g.rowscale0 = sorted_w;
            if ((e = launch_simt_gemm(g, s)) != cudaSuccess) return cuda_status(e);
        }
        rec.end(ST_DOWN);
        rec.begin(ST_COMBINE);
        if (S) {
            SimtGemmArgs g{};
            g.g[1] = SimtGroup{1, static_cast<const float*>(P(L.hs)), SF, nullptr, T,
                               static_cast<const float*>(w.Ws_down), nullptr, 1, c.d,
                               static_cast<float*>(out), c.d};
            g.K = SF; g.swiglu = 0; g.inv = inv; g.ys = static_cast<const float*>(P(L.ys));
            g.ys_ld = c.d; g.Kr = K;
            if ((e = launch_simt_gemm(g, s)) != cudaSuccess) return cuda_status(e);
        } else {
            if ((e = launch_gather_sum(static_cast<const float*>(P(L.ys)), inv, T, K, c.d, nullptr,
                                       out, 0, s)) != cudaSuccess)
                return cuda_status(e);
        }
        rec.end(ST_COMBINE);
    }
    (void)es;
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

MOE_API const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_DEVICE_INDEX: return "expert id out of range";
    }
    return "unknown status";
}

MOE_API const char* moe_version(void) { return "0.1.0"; }

MOE_API moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
    if (!cfg || !bytes) return MOE_ERR_INVALID_ARG;
    const moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    *bytes = plan_workspace(*cfg).total;
    return MOE_OK;
}

MOE_API moe_status moe_get_workspace_views(const moe_config* cfg, void* ws, moe_workspace_views* v) {
    if (!cfg || !ws || !v) return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_config(*cfg);
    if (st != MOE_OK) return st;
    const WsLayout L = plan_workspace(*cfg);
    uint8_t* b = static_cast<uint8_t*>(ws);
    v->topk_idx = reinterpret_cast<int32_t*>(b + L.topk_idx);
    v->topk_w = reinterpret_cast<float*>(b + L.topk_w);
    v->margin = reinterpret_cast<float*>(b + L.margin);
    v->top_scores = L.top_scores ? reinterpret_cast<float*>(b + L.top_scores) : nullptr;
    v->scores = L.scores ? reinterpret_cast<float*>(b + L.scores) : nullptr;
    v->counts = reinterpret_cast<int32_t*>(b + L.counts);
    v->offsets = reinterpret_cast<int32_t*>(b + L.offsets);
    v->sorted_token = reinterpret_cast<int32_t*>(b + L.sorted_token);
    v->sorted_w = reinterpret_cast<float*>(b + L.sorted_w);
    v->inv = reinterpret_cast<int32_t*>(b + L.inv);
    return MOE_OK;
}

MOE_API moe_status moe_route(const moe_config* cfg, const void* x, const float* W_router,
                             const float* bias, int32_t* topk_idx, float* topk_w, float* margin,
                             float* top_scores, float* scores, void* ws, size_t ws_bytes,
                             void* stream) {
    if (!cfg || !x || !W_router || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    const moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    if (!aligned16(x) || !aligned16(W_router)) return MOE_ERR_INVALID_ARG;
    if (ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = plan_workspace(*cfg);
    if (ws != nullptr && ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    RouterArgs ra = router_args(*cfg, x, W_router, bias);
    ra.idx = topk_idx; ra.w = topk_w; ra.margin = margin;
    ra.top_scores = top_scores;
    ra.scores = scores;
    return run_router(*cfg, ra, W_router, x, static_cast<uint8_t*>(ws), L,
                      static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_routing_stats(const moe_config* cfg, const void* x, const float* W_router,
                                     const float* bias, float* out, void* ws, size_t ws_bytes,
                                     void* stream) {
    if (!cfg || !x || !W_router || !out || !ws) return MOE_ERR_INVALID_ARG;
    const moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    if (!aligned16(x) || !aligned16(W_router) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = plan_workspace(*cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    uint8_t* b = static_cast<uint8_t*>(ws);
    RouterArgs ra = router_args(*cfg, x, W_router, bias);
    ra.idx = reinterpret_cast<int32_t*>(b + L.topk_idx);
    ra.w = reinterpret_cast<float*>(b + L.topk_w);
    ra.margin = reinterpret_cast<float*>(b + L.margin);
    ra.top_scores = L.top_scores ? reinterpret_cast<float*>(b + L.top_scores) : nullptr;
    ra.scores = L.scores ? reinterpret_cast<float*>(b + L.scores) : nullptr;
    ra.logits = reinterpret_cast<float*>(b + L.logits);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const moe_status st = run_router(*cfg, ra, W_router, x, b, L, s);
    if (st != MOE_OK) return st;
    return cuda_status(launch_routing_stats(ra.logits, ra.idx, cfg->T, cfg->E, cfg->K,
                                            reinterpret_cast<float*>(b + L.stats_part), out, s));
}

MOE_API moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const float* topk_w,
                                int32_t* counts, int32_t* offsets, int32_t* sorted_token,
                                float* sorted_w, int32_t* inv, void* ws, size_t ws_bytes,
                                void* stream) {
    if (!cfg || !topk_idx || !topk_w || !counts || !offsets || !sorted_token || !sorted_w || !inv || !ws)
        return MOE_ERR_INVALID_ARG;
    const moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    const WsLayout L = plan_workspace(*cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    uint8_t* b = static_cast<uint8_t*>(ws);
    DispatchArgs da{};
    da.idx = topk_idx; da.w = topk_w;
    da.T = cfg->T; da.K = cfg->K; da.E = cfg->E; da.nchunks = L.nchunks;
    da.bm = cfg->dtype == MOE_BF16 ? TC_BM : SIMT_BM;
    da.chunk_counts = reinterpret_cast<int32_t*>(b + L.chunk_counts);
    da.chunk_base = reinterpret_cast<int32_t*>(b + L.chunk_base);
    da.counts = counts; da.offsets = offsets;
    da.mt_prefix = reinterpret_cast<int32_t*>(b + L.mt_prefix);
    da.sorted_token = sorted_token; da.sorted_w = sorted_w; da.inv = inv;
    da.err = reinterpret_cast<int*>(b + L.err);
    da.ticket = da.err + 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the error word and the dispatch ticket start at zero
    if (cudaMemsetAsync(da.err, 0, 2 * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(launch_dispatch(da, s, nullptr));
}

MOE_API moe_status moe_forward(const moe_config* cfg, const void* x, const moe_weights* w, void* out,
                               void* ws, size_t ws_bytes, void* stream) {
    if (!cfg || !x || !out || !ws) return MOE_ERR_INVALID_ARG;
    moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    if ((v = check_weights(*cfg, w)) != MOE_OK) return v;
    if (!aligned16(x) || !aligned16(out) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < plan_workspace(*cfg).total) return MOE_ERR_WORKSPACE;
    return forward_impl(*cfg, x, *w, out, static_cast<uint8_t*>(ws), static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes) {
    if (!cfg || !bytes) return MOE_ERR_INVALID_ARG;
    const moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    *bytes = plan_backward(*cfg).total;
    return MOE_OK;
}

MOE_API moe_status moe_backward(const moe_config* cfg, const void* x, const moe_weights* w,
                                const float* dout, const moe_grads* grads, void* ws,
                                size_t ws_bytes, void* bws, size_t bws_bytes, void* stream) {
    if (!cfg || !x || !dout || !grads || !grads->dx || !ws || !bws) return MOE_ERR_INVALID_ARG;
    moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    if ((v = check_weights(*cfg, w)) != MOE_OK) return v;
    if (!aligned16(x) || !aligned16(dout) || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
        (reinterpret_cast<uintptr_t>(bws) & 255u))
        return MOE_ERR_INVALID_ARG;
    const float* outs[] = {grads->dx, grads->dW_router, grads->dW_gate, grads->dW_up,
                           grads->dW_down, grads->dWs_gate, grads->dWs_up, grads->dWs_down,
                           grads->dW_down_latent, grads->dW_up_latent};
    for (const float* p : outs)
        if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if ((grads->dWs_gate || grads->dWs_up || grads->dWs_down) && cfg->n_shared == 0)
        return MOE_ERR_INVALID_ARG;
    if ((grads->dW_down_latent || grads->dW_up_latent) && cfg->latent_dim == 0)
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < plan_workspace(*cfg).total || bws_bytes < plan_backward(*cfg).total)
        return MOE_ERR_WORKSPACE;
    return backward_impl(*cfg, x, *w, dout, *grads, static_cast<uint8_t*>(ws),
                         static_cast<uint8_t*>(bws), static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_forward_host(const moe_config* cfg, const void* x_host, const moe_weights* w,
                                    void* out_host, void* ws, size_t ws_bytes, void* stream) {
    if (!cfg || !x_host || !out_host || !ws) return MOE_ERR_INVALID_ARG;
    moe_status v = validate_config(*cfg);
    if (v != MOE_OK) return v;
    if ((v = check_weights(*cfg, w)) != MOE_OK) return v;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_INVALID_ARG;
    const WsLayout L = plan_workspace(*cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* b = static_cast<uint8_t*>(ws);
    const size_t xbytes = static_cast<size_t>(cfg->T) * cfg->d * (cfg->dtype == MOE_BF16 ? 2 : 4);
    const size_t obytes = static_cast<size_t>(cfg->T) * cfg->d * (cfg->out_dtype == MOE_BF16 ? 2 : 4);
    if (cudaMemcpyAsync(b + L.xstage, x_host, xbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    v = forward_impl(*cfg, b + L.xstage, *w, b + L.ostage, b, s);
    if (v != MOE_OK) return v;
    if (cudaMemcpyAsync(out_host, b + L.ostage, obytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
}

MOE_API size_t moe_quantile_workspace_size(int32_t T, int32_t E) {
    (void)T;
    return 256 + ((static_cast<size_t>(E > 0 ? E : 0) * 4 + 255) & ~static_cast<size_t>(255));
}

MOE_API moe_status moe_quantile_bias_update(int32_t T, int32_t E, int32_t K, const float* top_scores,
                                            const float* scores, float* bias, void* ws,
                                            size_t ws_bytes, void* stream) {
    if (T < 1 || E < 2 || K < 1 || K + 1 > E || !top_scores || !scores || !bias || !ws)
        return MOE_ERR_INVALID_ARG;
    if (E > 256) return MOE_ERR_UNSUPPORTED;
    if (ws_bytes < moe_quantile_workspace_size(T, E)) return MOE_ERR_WORKSPACE;
    // the FP32 pre-centring biases live right after the 256-byte error word
    float* braw = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
    return cuda_status(launch_quantile(T, E, K, top_scores, scores, braw, bias,
                                       static_cast<cudaStream_t>(stream), nullptr));
}

MOE_API moe_status moe_sign_bias_update(int32_t E, int32_t N, int32_t K, const int32_t* counts,
                                        float* bias, float alpha, void* stream) {
    if (E < 1 || N < 1 || K < 1 || !counts || !bias || !(alpha == alpha)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_sign_bias(E, N, K, counts, bias, alpha, static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status moe_workspace_status(void* ws, void* stream) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&h, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (h != 0 && cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    if (h & ERRBIT_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (h & ERRBIT_INDEX) return MOE_ERR_DEVICE_INDEX;
    return MOE_OK;
}

MOE_API moe_status moe_timing_begin(int32_t max_calls, uint32_t stage_mask) {
    if (max_calls < 1) return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_timing.mu);
    g_timing.mask = stage_mask;
    for (cudaEvent_t e : g_timing.ev) cudaEventDestroy(e);
    g_timing.ev.assign(static_cast<size_t>(max_calls) * ST_COUNT * 2, nullptr);
    g_timing.used.assign(static_cast<size_t>(max_calls) * ST_COUNT, 0);
    for (auto& e : g_timing.ev)
        if (cudaEventCreate(&e) != cudaSuccess) return MOE_ERR_CUDA;
    g_timing.max_calls = max_calls;
    g_timing.calls = 0;
    g_timing.on = true;
    return MOE_OK;
}

MOE_API moe_status moe_timing_end(float* stage_ms, int32_t max_stages, int32_t* n_stages,
                                  int32_t* n_calls) {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    if (!g_timing.on) return MOE_ERR_INVALID_ARG;
    g_timing.on = false;
    moe_status st = MOE_OK;
    std::vector<float> sum(ST_COUNT, 0.0f);
    for (int c = 0; c < g_timing.calls; ++c)
        for (int k = 0; k < ST_COUNT; ++k) {
            if (!g_timing.used[c * ST_COUNT + k]) continue;
            float ms = 0.0f;
            cudaEvent_t b = g_timing.ev[(c * ST_COUNT + k) * 2], e = g_timing.ev[(c * ST_COUNT + k) * 2 + 1];
            if (cudaEventSynchronize(e) != cudaSuccess || cudaEventElapsedTime(&ms, b, e) != cudaSuccess)
                st = MOE_ERR_CUDA;
            sum[k] += ms;
        }
    if (stage_ms)
        for (int k = 0; k < ST_COUNT && k < max_stages; ++k) stage_ms[k] = sum[k];
    if (n_stages) *n_stages = ST_COUNT;
    if (n_calls) *n_calls = g_timing.calls;
    for (cudaEvent_t e : g_timing.ev) cudaEventDestroy(e);
    g_timing.ev.clear();
    g_timing.used.clear();
    g_timing.calls = 0;
    return st;
}

MOE_API const char* moe_stage_name(int32_t stage) {
    return (stage >= 0 && stage < ST_COUNT) ? kStageNames[stage] : nullptr;
}

MOE_API uint64_t moe_launch_count(void) { return g_launches.load(); }

MOE_API moe_status moe_set_wait_timeout_ms(int32_t ms) {
    if (ms < 1) return MOE_ERR_INVALID_ARG;
    g_timeout_ns.store(static_cast<long long>(ms) * 1000000LL);
    return MOE_OK;
}

MOE_API moe_status moe_selftest_wait_timeout(int32_t ms, void* ws, void* stream) {
    if (ms < 1 || ms > 10000 || !ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_wait_selftest(static_cast<int*>(ws), static_cast<uint64_t>(ms) * 1000000ull, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return moe_workspace_status(ws, stream);
}
