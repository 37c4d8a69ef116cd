/*
 * moe.h - C ABI of the GB300 (sm_103a) forward (and backward) pass of a
 * top-K routed Mixture-of-Experts SwiGLU FFN layer with always-on shared
 * experts.
 *
 * The layer (APEX-1 Mathematical Reference Part 3, section 13.2):
 *
 *     MoE(x) = sum_{s<S} Shared_s(x) + sum_{k<K} g_k * Expert_{e_k}(x)
 *     Expert(x) = W_down( SiLU(x W_gate) (.) x W_up )          (section 12.2)
 *
 * with router logits r = x W_router in FP32, an optional per-expert balance
 * bias, top-K selection and one of three gate rules (see moe_gate). In the
 * latent variant (kimi_k3 "StableLatentMoE and QuantileBalancer") the routed
 * experts act on z = x W_down_latent and their weighted sum is projected back
 * by W_up_latent before the shared output is added.
 *
 * Conventions for every entry point:
 *  - Every array is row-major and contiguous. "Device" pointers must point to
 *    memory of the current CUDA device; "host" pointers to host memory.
 *  - The caller owns every buffer. The library allocates no device memory;
 *    scratch space is the caller's workspace (see moe_workspace_size).
 *  - Work is enqueued on the given stream (a cudaStream_t passed as void*,
 *    NULL = the legacy default stream) and the call returns without
 *    synchronising, except where a function says otherwise.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns an error code and enqueues nothing.
 *  - Expert ids are int32; FP32 is IEEE binary32; BF16 is bfloat16 (the
 *    upper 16 bits of a binary32), rounded to nearest-even where produced.
 *  - No entry point is thread-safe with respect to a workspace: concurrent
 *    calls must use distinct workspaces.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, K > E, ... */
    MOE_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement (e.g. E > 256) */
    MOE_ERR_WORKSPACE = 3,    /* workspace smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    MOE_ERR_TIMEOUT = 5,      /* a device-side wait ran out of time (see moe_workspace_status) */
    MOE_ERR_DEVICE_INDEX = 6  /* a kernel met an expert id outside [0, E) */
} moe_status;

typedef enum moe_dtype {
    MOE_F32 = 0,   /* FP32 activations and expert weights, FP32 FMA arithmetic */
    MOE_BF16 = 1   /* BF16 activations and expert weights, FP32 accumulation (tcgen05) */
} moe_dtype;

/* Gate rule. c denotes the selection score, b the balance bias.
 * Top-K ranks by c descending; equal scores rank the lower expert id first;
 * slot k of every [T, K] output holds the k-th ranked expert. */
typedef enum moe_gate {
    /* c = r + b; top-K of c; g = softmax over the K selected c.
     * (APEX-1 docs "10 - Mixture of Experts", MoEFFN.forward steps 2-3;
     *  APEX-1 Math Ref Part 3 section 13.2) */
    MOE_GATE_SOFTMAX_TOPK = 0,
    /* p = softmax over all E of (r + b); c = p; top-K of p; g = p_sel / sum p_sel.
     * ("MoE from scratch" tutorial, MoELayer.forward) */
    MOE_GATE_SOFTMAX_ALL_RENORM = 1,
    /* s = sigmoid(r); c = s + b; top-(K+1) of c, the first K used; g = s at the
     * selected experts (uncorrected), divided by its sum if renormalize, times
     * routed_scale. (kimi_k3 StableLatentMoE, "FP32 router and training-only QB
     * update", "Flatten routing and recover original token order") */
    MOE_GATE_SIGMOID = 2
} moe_gate;

/* Problem description. */
typedef struct moe_config {
    int32_t T;            /* tokens (batch x sequence flattened), >= 1 */
    int32_t d;            /* model width (M of the latent page) */
    int32_t d_ff;         /* routed expert hidden width (I of the latent page) */
    int32_t E;            /* routed experts, 1..256 */
    int32_t K;            /* active experts per token, 1..min(E,16); K+1 <= E in sigmoid mode */
    int32_t n_shared;     /* always-on shared experts S >= 0 */
    int32_t shared_d_ff;  /* hidden width of each shared expert */
    int32_t latent_dim;   /* 0: experts act on x; L > 0: experts act on z = x W_down_latent */
    int32_t dtype;        /* moe_dtype of x, out and every expert/shared/latent weight */
    int32_t gate;         /* moe_gate */
    int32_t renormalize;  /* sigmoid mode: divide the K weights by their sum */
    float routed_scale;   /* sigmoid mode: factor on the routed weights (1.0 = none) */
    int32_t out_dtype;    /* moe_dtype of out: MOE_F32 (the FP32 accumulation, unrounded) or
                             MOE_BF16 (rounded once to nearest-even); must be MOE_F32 when
                             dtype is MOE_F32 */
    int32_t save_gate_up; /* 0 or 1. 1, for a layer whose moe_backward runs on the tensor
                             cores (BF16, widths multiples of 64): moe_forward also keeps
                             the gate and up products a = z W_gate, u = z W_up of every
                             routed row and shared expert (BF16) in the workspace, and
                             moe_backward reads them instead of recomputing them (the
                             workspace grows by 4 (T K d_ff + T n_shared shared_d_ff)
                             bytes). The forward and the backward of one step must use the
                             same value. Ignored by other layers. */
} moe_config;

/* Weights, all device pointers. d_e = latent_dim ? latent_dim : d.
 * W_router  [d, E] FP32                       (always FP32, always read as FP32)
 * bias      [E]   FP32, or NULL for no bias
 * W_gate    [E, d_e, d_ff]  W_up [E, d_e, d_ff]  W_down [E, d_ff, d_e]      (dtype)
 * Ws_gate   [S, d, shared_d_ff]  Ws_up [S, d, shared_d_ff]
 * Ws_down   [S, shared_d_ff, d]                                              (dtype)
 * W_down_latent [d, L], W_up_latent [L, d]   (dtype; NULL unless latent_dim > 0)
 * Matrices multiply row vectors from the right: h = x W_gate, y = h W_down. */
typedef struct moe_weights {
    const float* W_router;
    const float* bias;
    const void* W_gate;
    const void* W_up;
    const void* W_down;
    const void* Ws_gate;
    const void* Ws_up;
    const void* Ws_down;
    const void* W_down_latent;
    const void* W_up_latent;
} moe_weights;

/* Device pointers into a workspace after moe_forward: the routing and
 * dispatch results of the last forward that used the workspace. */
typedef struct moe_workspace_views {
    int32_t* topk_idx;      /* [T, K]   selected experts, slot order */
    float* topk_w;          /* [T, K]   gate weights */
    float* margin;          /* [T]      c at rank K minus c at rank K+1 (+inf if K == E) */
    float* top_scores;      /* [T, K+1] sigmoid mode: the K+1 largest c, descending; else NULL */
    float* scores;          /* [T, E]   sigmoid mode: s = sigmoid(r); else NULL */
    int32_t* counts;        /* [E]      assignments per expert */
    int32_t* offsets;       /* [E+1]    exclusive prefix sum of counts */
    int32_t* sorted_token;  /* [T*K]    token of each expert-sorted assignment */
    float* sorted_w;        /* [T*K]    gate weight of each expert-sorted assignment */
    int32_t* inv;           /* [T, K]   sorted position of assignment (t, k) */
} moe_workspace_views;

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status s);

/* Library version, e.g. "0.1.0" (static storage). */
const char* moe_version(void);

/* Bytes of device workspace moe_forward / moe_dispatch /
 * moe_quantile_bias_update need for cfg (host only, no CUDA call).
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for an invalid config. */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Pointers to the routing/dispatch results inside a workspace of cfg
 * (host only; NULL members where the mode has no such array). */
moe_status moe_get_workspace_views(const moe_config* cfg, void* ws, moe_workspace_views* v);

/* Router: logits r = x W_router in FP32 (x read as FP32 when dtype is BF16,
 * which is exact), the mode's selection score, top-K (top-(K+1) in sigmoid
 * mode) and gate weights.
 *   x [T, d] (dtype), W_router [d, E] FP32, bias [E] FP32 or NULL.
 *   Outputs (device): topk_idx [T, K] int32, topk_w [T, K] FP32, required;
 *   margin [T] FP32, top_scores [T, K+1] FP32 and scores [T, E] FP32 optional
 *   (NULL = not written); top_scores/scores are only produced in sigmoid mode.
 *   ws: NULL, or a workspace of moe_workspace_size(cfg) bytes. With a
 *   workspace, BF16 layers with E > 32, E % 8 == 0 and d % 64 == 0 compute
 *   the logits on the tensor cores from an exact three-part BF16 split of
 *   W_router (the same path moe_forward takes); otherwise, and without a
 *   workspace, one fused FP32 FMA kernel computes them. Both are FP32-accurate
 *   but sum in different orders, so near-tie tokens may rank differently.
 * Sources: APEX-1 docs "10 - Mixture of Experts" steps 2-3; APEX-1 Math Ref
 * Part 3 sections 13.2 and 13.5; "MoE from scratch" MoELayer.forward;
 * kimi_k3 StableLatentMoE "FP32 router and training-only QB update". */
moe_status moe_route(const moe_config* cfg, const void* x, const float* W_router,
                     const float* bias, int32_t* topk_idx, float* topk_w, float* margin,
                     float* top_scores, float* scores, void* ws, size_t ws_bytes, void* stream);

/* Sorted dispatch of the T*K assignments by expert id: a stable counting sort
 * of the flat assignments j = t*K + k (kimi_k3 StableLatentMoE, "Flatten
 * routing and recover original token order" and "Dispatch is a stable
 * permutation").
 *   topk_idx [T, K] int32 (device), topk_w [T, K] FP32 (device).
 *   Outputs (device): counts [E], offsets [E+1] (exclusive prefix sums,
 *   offsets[E] = T*K), sorted_token [T*K] (= j / K of the assignment at each
 *   sorted position), sorted_w [T*K], inv [T, K] (sorted position of (t, k)).
 *   ws: device workspace of at least moe_workspace_size(cfg) bytes.
 * No host synchronisation. An expert id outside [0, E) is skipped and
 * recorded in the workspace (moe_workspace_status returns MOE_ERR_DEVICE_INDEX). */
moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const float* topk_w,
                        int32_t* counts, int32_t* offsets, int32_t* sorted_token,
                        float* sorted_w, int32_t* inv, void* ws, size_t ws_bytes,
                        void* stream);

/* moe_dispatch for callers that cannot allocate device memory: for example a
 * runtime that owns all device memory and only hands out the tensors it
 * manages, or code that must not call cudaMalloc after start-up because an
 * allocation can synchronise the device or fail under memory pressure.
 * The pages have no counterpart of this call; it exists for such callers.
 * Same inputs, outputs and results as moe_dispatch, but no workspace: its
 * scratch is a fixed array in the library's own device memory, sized for
 * T*K <= 65536 and E <= 256 (about 130 KB, held by every GPU that loads the
 * library until the process exits); larger calls return MOE_ERR_UNSUPPORTED.
 * The first call on each device looks up the array's device address with
 * that device current; make that first call before any stream capture. The
 * address is kept per device and context: after cudaDeviceReset (or anything
 * else that makes a new context) the next call looks it up again, so make
 * that call before any capture too.
 * Every call reuses the same array, so calls that overlap on the GPU (for
 * example on two streams with no ordering between them) race and corrupt
 * each other's results; order such calls on one stream. Expert ids outside
 * [0, E) are skipped, the other assignments dispatched as moe_dispatch does;
 * the caller detects skipped ids by offsets[E] falling short of T*K by their
 * number. Calls no allocating function. */
moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx,
                                const float* topk_w, int32_t* counts, int32_t* offsets,
                                int32_t* sorted_token, float* sorted_w, int32_t* inv,
                                void* stream);

/* Whole layer forward: route -> dispatch -> grouped gate/up GEMM with
 * SiLU(.)*up epilogue -> grouped down GEMM scaled by the gate weight ->
 * shared experts -> deterministic combine (no float atomics).
 *   x [T, d] (dtype, device), out [T, d] (out_dtype, device).
 *   The routing and dispatch results stay in ws (moe_get_workspace_views).
 *   The balance bias is read, never written (use moe_quantile_bias_update).
 *   No host synchronisation and no allocation: after a first call on the
 *   device (which sets kernel attributes), calls can be captured into a CUDA
 *   graph; so can moe_backward.
 *   The grouped GEMMs pick their tile form from the shapes; the environment
 *   variable MOE_GEMM_FORM, read at each call, overrides the choice for tests
 *   and tuning ("rows": row-tile forms only; "single": single-CTA row tiles
 *   only; "tokens": the token-column form wherever the product allows it).
 *   The forms give the same bits except
 *   that the token-column down product stores its routed rows rounded to 16
 *   significant bits (a relative error of at most 2^-17 per routed row).
 * Sources: APEX-1 Math Ref Part 3 sections 12.2 and 13.2; APEX-1 docs
 * "10 - Mixture of Experts" MoEFFN.forward; kimi_k3 StableLatentMoE
 * "Grouped expert execution" and "Return to model width"; "MoE from scratch"
 * MoELayer.forward. */
moe_status moe_forward(const moe_config* cfg, const void* x, const moe_weights* w, void* out,
                       void* ws, size_t ws_bytes, void* stream);

/* moe_forward with HOST input and output: copies x_host [T, d] (dtype) to the
 * device (inside ws), runs the forward and copies out [T, d] (out_dtype) back to
 * out_host, all on `stream`, then synchronises the stream before returning.
 * Pinned host memory makes the copies asynchronous DMA; pageable works too. */
moe_status moe_forward_host(const moe_config* cfg, const void* x_host, const moe_weights* w,
                            void* out_host, void* ws, size_t ws_bytes, void* stream);

/* Quantile balancer update (kimi_k3 "QuantileBalancer: persistent biases, no
 * gradient update"): with p = K/E,
 *     thresh_t = top_scores[t, K]            (the (K+1)-th corrected score)
 *     rel[t, j] = thresh_t - scores[t, j]    (FP32)
 *     b_j = rel[:, j] at sorted index ceil(p (T-1))   ('higher' quantile; the
 *           index computed in FP32 as the FP32 quantile does)
 *     bias = b - mean(b)   (mean: sequential float64 sum over j, divided by E,
 *                           rounded to FP32; FP32 subtraction)
 * Bit-exact for given inputs. top_scores [T, K+1], scores [T, E], bias [E]
 * (output, replaced), all FP32 device. ws: at least moe_workspace_size of a
 * config with the same T, E, K (or moe_quantile_workspace_size bytes). */
moe_status moe_quantile_bias_update(int32_t T, int32_t E, int32_t K, const float* top_scores,
                                    const float* scores, float* bias, void* ws, size_t ws_bytes,
                                    void* stream);

/* Workspace bytes moe_quantile_bias_update needs on its own. */
size_t moe_quantile_workspace_size(int32_t T, int32_t E);

/* Routing diagnostics of one batch: runs the router of cfg on x (as
 * moe_route with a workspace; its selection and logits stay in ws) and
 * writes to out (device, FP32, 2 + E values):
 *     out[0] = aux = E * sum_e f_e P_e      Switch load-balancing loss before
 *                                           its alpha ("MoE from scratch",
 *                                           MoELayer.forward)
 *     out[1] = z = (1/T) sum_t (log sum_e exp r_te)^2   router z-loss before
 *                                           its weight (book-ai MoE chapter,
 *                                           MoELoss.router_z_loss)
 *     out[2 + e] = P_e = (1/T) sum_t softmax(r_t)_e
 * with r = x W_router the raw FP32 logits (no balance bias) and f_e the share
 * of the T*K selected (token, slot) pairs on expert e (the selection uses the
 * bias, as the forward's does). Sums run in a fixed order: the result is
 * reproducible bit for bit. ws: required, at least moe_workspace_size(cfg)
 * bytes, 256-byte aligned; x and W_router 16-byte aligned. */
moe_status moe_routing_stats(const moe_config* cfg, const void* x, const float* W_router,
                             const float* bias, float* out, void* ws, size_t ws_bytes,
                             void* stream);

/* Sign-bias balancing (APEX-1 Math Ref Part 3, section 14.3): with
 * f_e = counts[e] / (N K) and tau = 1/E,
 *     bias[e] <- clamp(bias[e] + alpha * sign(tau - f_e), -1, 1)
 * counts [E] int32 (device, e.g. the workspace's counts after a forward with
 * N = T tokens), bias [E] FP32 device, updated in place. */
moe_status moe_sign_bias_update(int32_t E, int32_t N, int32_t K, const int32_t* counts,
                                float* bias, float alpha, void* stream);

/* Gradients written by moe_backward: FP32 device arrays, row-major. dx is
 * required; any other pointer may be NULL (that gradient is not computed). */
typedef struct moe_grads {
    float* dx;              /* [T, d] */
    float* dW_router;       /* [d, E] */
    float* dW_gate;         /* [E, d_e, d_ff]  d_e = latent_dim ? latent_dim : d */
    float* dW_up;           /* [E, d_e, d_ff] */
    float* dW_down;         /* [E, d_ff, d_e] */
    float* dWs_gate;        /* [S, d, shared_d_ff] */
    float* dWs_up;          /* [S, d, shared_d_ff] */
    float* dWs_down;        /* [S, shared_d_ff, d] */
    float* dW_down_latent;  /* [d, latent_dim] */
    float* dW_up_latent;    /* [latent_dim, d] */
} moe_grads;

/* Bytes of the backward's own scratch workspace (bws of moe_backward). */
moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes);

/* Backward pass: the gradients of L = sum(dout * out) of the forward that
 * last ran on `ws` (moe_forward with the same cfg, x and weights; its routing
 * and dispatch, and for the latent variant z and the routed rows, are read
 * from ws), with that forward's expert selection held fixed - the top-K
 * indices carry no gradient (kimi_k3 StableLatentMoE, "The actual grouped
 * GEMM, and the gradient path"):
 *     gate weights g -> router logits r -> W_router and x, through the gate
 *     rule's formula (the balance bias is a buffer without gradient);
 *     the routed and shared SwiGLU experts, their weights and their input;
 *     the latent projections.
 * Experts that no token selected get no gradient: their slices of dW_gate,
 * dW_up and dW_down are NOT written (kimi_k3 StableLatentMoE, "Grouped
 * expert execution and sparse gradients"); the workspace's counts tell which.
 * Every other requested gradient is overwritten. Sums run in a fixed order:
 * bit-reproducible.
 *   x [T, d] (dtype), dout [T, d] FP32 device; x, dout and every gradient
 *   16-byte aligned.
 * BF16 layers whose d, d_ff, latent_dim and shared_d_ff are multiples of 64
 * run the expert contractions on the tensor cores with BF16 operands (the
 * upstream and activation gradients rounded to BF16, FP32 sums); the others
 * on the CUDA cores in FP32. On the tensor cores, cfg->save_gate_up = 1 takes
 * the gate and up products the forward kept (BF16) instead of recomputing
 * them; the forward must then have run with save_gate_up = 1 as well.
 *   ws: the forward's workspace (moe_workspace_size bytes, 256-byte aligned).
 *   bws: moe_backward_workspace_size bytes, 256-byte aligned. */
moe_status moe_backward(const moe_config* cfg, const void* x, const moe_weights* w,
                        const float* dout, const moe_grads* grads, void* ws, size_t ws_bytes,
                        void* bws, size_t bws_bytes, void* stream);

/* Synchronises `stream`, then reads and clears the device-side error word of
 * the workspace: MOE_OK, MOE_ERR_TIMEOUT (a bounded device wait ran out and
 * its kernel stopped early; outputs of that call are invalid) or
 * MOE_ERR_DEVICE_INDEX. moe_forward and moe_dispatch clear the word when
 * they start, so the status covers the calls since the last of those. */
moe_status moe_workspace_status(void* ws, void* stream);

/* Instrumentation. While enabled, each moe_forward records CUDA events
 * around each of its kernel stages selected by stage_mask (bit i = stage i;
 * 0xFFFFFFFF = all) on the caller's stream, for up to max_calls calls.
 * moe_timing_end synchronises those events and returns, per stage, the summed
 * milliseconds over the recorded calls. Stage names via moe_stage_name.
 * Events are created/destroyed by the library. Recording an event between
 * two kernels stops the second from overlapping the first's tail, so time
 * only the stages you need. */
moe_status moe_timing_begin(int32_t max_calls, uint32_t stage_mask);
moe_status moe_timing_end(float* stage_ms, int32_t max_stages, int32_t* n_stages,
                          int32_t* n_calls);
const char* moe_stage_name(int32_t stage);

/* Number of kernels this library has launched in this process. */
uint64_t moe_launch_count(void);

/* Sets the limit of every bounded device-side wait (default 1000 ms). */
moe_status moe_set_wait_timeout_ms(int32_t ms);

/* Self-test of the bounded-wait machinery: launches one kernel that waits on
 * a shared-memory barrier nothing ever completes, with a `ms` millisecond
 * limit, then synchronises. Returns MOE_ERR_TIMEOUT when the wait gave up
 * as designed (and the context stays usable), MOE_OK never. */
moe_status moe_selftest_wait_timeout(int32_t ms, void* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
