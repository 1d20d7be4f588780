/*
 * moe.h -- C ABI of the single-GPU Mixture-of-Experts layer forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The method ("Cross-Platform Fused MoE Dispatch in Triton: Portable Expert
 * Routing Without CUDA", review page, section "The reading"): tokens are
 * scored by a router, reordered onto experts, run through variable-size
 * expert GEMMs, then scattered back with their routing weights.  The expert
 * is SwiGLU with the gate and up projections fused so that SiLU(gate)*up is
 * finished in registers ("What carries the argument").  The router, top-k and
 * SwiGLU equations are the standard ones of Mixtral, DeepSeek-V3 and
 * Qwen2-MoE ("Assumptions & free parameters", Eq. (1)-(4)).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *    16-byte aligned.  bf16 tensors are passed as void*.  Weights use the
 *    [out_features, in_features] layout (both GEMM operands K-major).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and never synchronise the host, except
 *    moe_device_error().  Nothing is freed by the library.
 *  - Arguments are checked before any launch; a bad argument returns a
 *    status code and launches nothing.  No entry point aborts or throws.
 *  - Kernels never trap.  Problems found on the device (an expert id out of
 *    range, a pipeline wait that timed out) set a device error word that
 *    moe_device_error() reads and clears.
 *  - Shape limits: 1 <= k <= E <= 256, k <= 16, H and F multiples of 128,
 *    T >= 0 (T == 0 is a no-op that returns MOE_OK).
 */
#ifndef MOE_GB300_MOE_H
#define MOE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_VALUE = 1,  /* null pointer, bad size, misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,    /* shape outside the limits above */
    MOE_ERR_WORKSPACE = 3,      /* workspace too small */
    MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
    MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait gave up */
    MOE_ERR_DEVICE_BOUNDS = 6   /* a device-side index check failed */
} moe_status_t;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_t;

/*
 * Activation of the gated expert FFN, h = act(x W_gate^T) * (x W_up^T):
 * SiLU (SwiGLU, the default) or GELU in its exact erf form (GEGLU),
 * GELU(g) = g/2 * (1 + erf(g / sqrt(2))).  The review of "Cross-Platform
 * Fused MoE Dispatch in Triton" names GEGLU as a dual-projection activation
 * the same fused tile carries with only the element-wise op changed
 * ("Editorial extensions", "Reading between the lines").
 */
typedef enum { MOE_ACT_SILU = 0, MOE_ACT_GELU = 1 } moe_activation_t;

/*
 * Routing variant and optional shared expert.
 *  score:        softmax over all E logits, or sigmoid of each logit.
 *  renormalize:  divide the k selected scores by their sum.
 *  route_scale:  multiply the routing weights (1.0; DeepSeek-V3 uses 2.5).
 *  n_group, topk_group, group_topn: group-limited top-k (DeepSeek-V3 router):
 *                experts are split into n_group equal consecutive groups,
 *                a group's score is the sum of its top group_topn scores,
 *                the topk_group best groups are kept and the k experts are
 *                chosen among them.  n_group <= 1 switches it off.
 *                Limits: n_group <= 16, group_topn <= 4.
 *  logit_bias:   [E] fp32 added to the logits before the score function,
 *                or NULL.
 *  F_shared:     width of one always-on shared SwiGLU expert (0 = none);
 *                ws_gate, ws_up: bf16 [F_shared, H]; ws_down: bf16 [H, F_shared].
 *  w_shared_gate: bf16 [H] or NULL.  When set, the shared expert's output is
 *                scaled by sigmoid(x . w_shared_gate) (Qwen2-MoE); when NULL
 *                it is added with scale 1 (DeepSeek-V3).
 * Selection ties go to the lower expert (group) index.
 */
typedef struct {
    int score;
    int renormalize;
    float route_scale;
    int n_group;
    int topk_group;
    int group_topn;
    const float* logit_bias;
    int F_shared;
    const void* ws_gate;
    const void* ws_up;
    const void* ws_down;
    const void* w_shared_gate;
    int activation; /* moe_activation_t, for the routed and the shared experts */
} moe_config_t;

/* Fill cfg with the Mixtral routing: softmax, renormalised top-k, scale 1,
 * no groups, no bias, no shared expert. */
MOE_API void moe_config_default(moe_config_t* cfg);

/*
 * Router scoring and top-k selection ("The reading": tokens are scored).
 * logits = x . W_r^T (+ logit_bias) with fp32 accumulation on the tensor
 * cores (the K dimension split over the CTAs of a thread-block cluster, the
 * partial logits added in rank order in shared memory), then the score
 * function, top-k and weights as in moe_config_t, in the same launch.
 *   x:            bf16 [T, H]
 *   w_router:     bf16 [E, H]
 *   topk_idx:     int32 [T, k] out, slot order = descending score
 *   topk_w:       fp32 [T, k] out, routing weights in the same order
 *   shared_scale: fp32 [T] out, sigmoid(x . w_shared_gate); may be NULL
 *                 when cfg->w_shared_gate is NULL.
 *   scratch:      device memory of at least moe_route_scratch_bytes(cfg, T,
 *                 H, E) bytes; too little returns MOE_ERR_WORKSPACE.  This
 *                 version needs none (moe_route_scratch_bytes returns 0), so
 *                 scratch may be NULL; the argument stays for callers that
 *                 size it from moe_route_scratch_bytes.
 * cfg may be NULL (moe_config_default).
 */
MOE_API size_t moe_route_scratch_bytes(const moe_config_t* cfg, int T, int H, int E);
MOE_API moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       int T, int H, int E, int k,
                       int32_t* topk_idx, float* topk_w, float* shared_scale,
                       void* scratch, size_t scratch_bytes, moe_stream_t stream);

/*
 * Token permutation ("The reading": tokens are reordered onto experts).
 * Row q = t*k + j is token t's j-th choice.  Rows are grouped by expert and
 * kept in token order inside an expert (stable).
 *   topk_idx: int32 [T, k] in; ids outside [0, E) set MOE_ERR_DEVICE_BOUNDS
 *             on the device and the row is dropped
 *   x:        bf16 [T, H] in
 *   counts:   int32 [E] out, rows per expert
 *   offsets:  int32 [E + 1] out, exclusive scan of counts (offsets[E] = T*k)
 *   perm:     int32 [T*k] out, perm[r] = q of grouped row r
 *   inv:      int32 [T*k] out, inv[q] = r
 *   x_perm:   bf16 [T*k, H] out, x_perm[r] = x[perm[r] / k]
 *   scratch:  device memory of at least moe_permute_scratch_bytes(T, E) bytes
 */
MOE_API size_t moe_permute_scratch_bytes(int T, int E);
MOE_API moe_status_t moe_permute(const int32_t* topk_idx, const void* x, int T, int H, int E, int k,
                         int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                         void* x_perm, void* scratch, size_t scratch_bytes,
                         moe_stream_t stream);

/*
 * moe_permute without caller scratch.  The paper has no counterpart: this
 * entry point exists for callers that cannot allocate device memory, such as
 * serving engines that plan all device memory at start-up and forbid any
 * allocation afterwards, plugins that run inside a host application which
 * owns the CUDA allocator, and code with latency bounds that cannot afford
 * cudaMalloc's implicit synchronisation.
 * Same arguments and results as moe_permute, minus scratch: the token bitmaps
 * live in a 512 KiB array built into the library's device image (every GPU
 * that loads the library holds it until the process exits).  Limits: all of
 * moe_permute's, plus ceil(T/32) * E <= 65536 (e.g. T <= 8192 at E = 256);
 * larger calls return MOE_ERR_WORKSPACE and launch nothing.  The first call
 * on each device looks up that device's copy of the array, so make it before
 * any stream capture.  Every call on a device shares the one array: calls
 * that overlap on the GPU (different streams, or concurrent host threads)
 * race and must be serialised by the caller.  Nothing in the array needs to
 * start at zero; each call writes every word it reads.  Allocates nothing
 * (no cudaMalloc, cudaFree or allocating library call).
 */
MOE_API moe_status_t moe_permute_noalloc(const int32_t* topk_idx, const void* x, int T, int H, int E, int k,
                                         int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                         void* x_perm, moe_stream_t stream);

/*
 * Expert SwiGLU FFN over grouped rows ("What carries the argument": a fused
 * gate+up GEMM that finishes SiLU(gate)*up in registers, then a grouped
 * down-projection GEMM; one persistent kernel each, with a tile schedule
 * built on the device from `offsets`).
 *   x_perm:  bf16 [rows, H] in, grouped by expert
 *   offsets: int32 [E + 1] in, group g owns rows [offsets[g], offsets[g+1]),
 *            offsets[E] == rows; or NULL, meaning one group of all rows
 *            (then E must be 1: a dense SwiGLU MLP, used for shared experts)
 *   w_gate, w_up: bf16 [E, F, H];  w_down: bf16 [E, H, F]
 *   h:       bf16 [rows, F] out, SiLU(x W_gate^T) * (x W_up^T) rounded to bf16
 *   y:       fp16 [rows, H] out, h W_down^T accumulated in fp32 and rounded
 *            once to fp16 (a 16-bit intermediate, as the pages' byte model
 *            counts; fp16 rather than bf16 for its 8x finer rounding).  A
 *            value beyond the fp16 range (|y| > 65504) becomes inf and sets
 *            MOE_ERR_DEVICE_BOUNDS (site bit 18) in the device error word.
 */
MOE_API moe_status_t moe_expert_ffn(const void* x_perm, const int32_t* offsets, int rows,
                            int H, int F, int E,
                            const void* w_gate, const void* w_up, const void* w_down,
                            void* h, void* y, moe_stream_t stream);

/* moe_expert_ffn with the activation chosen (moe_activation_t; an unknown
 * value returns MOE_ERR_INVALID_VALUE). */
MOE_API moe_status_t moe_expert_ffn_ex(const void* x_perm, const int32_t* offsets, int rows,
                               int H, int F, int E,
                               const void* w_gate, const void* w_up, const void* w_down,
                               int activation, void* h, void* y, moe_stream_t stream);

/*
 * Fusion ablation, for measurement: the same grouped FFN with the gate and up
 * projections run as two grouped GEMMs whose bf16 outputs g, u [rows, F] go
 * to global memory, then h = act(g) * u as an element-wise pass, then the
 * down projection ("What carries the argument": fusing gate and up removes
 * those intermediates; the referee's minor comment 1 on the paper's section
 * 3.3 gives the byte counts).  Arguments as moe_expert_ffn_ex plus the
 * caller's g and u buffers (bf16 [rows, F], 16-byte aligned).  g and u are
 * each rounded to bf16 before the activation, so h can differ from the fused
 * result in the last bit.
 */
MOE_API moe_status_t moe_expert_ffn_unfused(const void* x_perm, const int32_t* offsets, int rows,
                                    int H, int F, int E,
                                    const void* w_gate, const void* w_up, const void* w_down,
                                    int activation, void* g, void* u, void* h, void* y,
                                    moe_stream_t stream);

/*
 * Schedule ablation, for measurement: the grouped SwiGLU FFN (as
 * moe_expert_ffn) run the way the pages' design schedules it ("Load-bearing
 * premise": a compile-time fixed tile size and a static expert-to-block
 * schedule; the referee's minor comment 5 on its host-device sync).  The
 * expert offsets are copied back to the host and the call WAITS for them
 * (cudaStreamSynchronize on `stream`), every tile has block_m token rows
 * (16, 32, 64, 128 or 256; an expert's rows are split into equal tiles of at
 * most block_m rows), and each GEMM is launched with one CTA per tile (no
 * persistent CTAs, no CTA pairs, one 128-row weight tile per CTA).  offsets
 * must not be NULL.  The results equal moe_expert_ffn's bit for bit.  Not
 * capturable in a CUDA graph.
 */
MOE_API moe_status_t moe_expert_ffn_static(const void* x_perm, const int32_t* offsets, int rows,
                                   int H, int F, int E,
                                   const void* w_gate, const void* w_up, const void* w_down,
                                   int block_m, void* h, void* y, moe_stream_t stream);

/*
 * Weighted scatter-back ("The reading": scattered back with weights).
 * out[t] = sum_{j=0..k-1} topk_w[t,j] * y_perm[inv[t*k+j]]
 *          (+ s_t * y_shared[t]), summed in fp32 in that fixed order and
 * rounded once to bf16 (round to nearest even); deterministic.
 *   y_perm:       fp16 [T*k, H] (moe_expert_ffn's y)
 *   inv:          int32 [T*k]
 *   topk_w:       fp32 [T, k]
 *   y_shared:     fp16 [T, H] or NULL (no shared expert)
 *   shared_scale: fp32 [T] or NULL (scale 1)
 *   out:          bf16 [T, H], fully overwritten
 */
MOE_API moe_status_t moe_combine(const void* y_perm, const int32_t* inv, const float* topk_w,
                         const void* y_shared, const float* shared_scale,
                         int T, int H, int k, void* out, moe_stream_t stream);

/*
 * The whole layer: moe_route -> moe_permute -> moe_expert_ffn (routed
 * experts and the shared expert in the same two persistent launches) ->
 * moe_combine, all enqueued on `stream` with no host synchronisation.
 * moe_forward_ex takes caller workspace of at least moe_workspace_bytes().
 */
MOE_API size_t moe_workspace_bytes(const moe_config_t* cfg, int T, int H, int F, int E, int k);
MOE_API moe_status_t moe_forward_ex(const moe_config_t* cfg, const void* x, const void* w_router,
                            const void* w_gate, const void* w_up, const void* w_down,
                            int T, int H, int F, int E, int k, void* out,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_forward_ex with the Mixtral routing (moe_config_default) and a
 * workspace the library keeps per device, grown (cudaFreeAsync of the old
 * one, cudaMallocAsync of the new one, both on `stream`) when a larger call
 * arrives.  Calls on one device are ordered through an event the library
 * records after each call: a call's work waits for the previous call's work,
 * on whatever stream it ran, so the shared workspace is never used by two
 * calls at once nor freed under a call still running.  Calls on different
 * streams therefore serialise on the device; callers that want them to
 * overlap use moe_forward_ex with their own workspaces.  Not for stream
 * capture (returns MOE_ERR_UNSUPPORTED on a capturing stream): capture
 * moe_forward_ex with a caller workspace instead.
 */
MOE_API moe_status_t moe_forward(const void* x, const void* w_router, const void* w_gate,
                         const void* w_up, const void* w_down, int T, int H, int F, int E,
                         int k, void* out, moe_stream_t stream);

/*
 * How many kernels one moe_forward_ex / moe_forward call launches for these
 * shapes and this configuration (cfg NULL: the defaults), or -1 if the
 * arguments would be rejected.  Host only, no device work.
 */
MOE_API int moe_forward_launches(const moe_config_t* cfg, int T, int H, int F, int E, int k);

/*
 * Kernels this library has launched since it was loaded (all entry points,
 * all devices; a host-side count of successful launches).
 */
MOE_API unsigned long long moe_launches_issued(void);

/* Human-readable name of a status code (static storage). */
MOE_API const char* moe_status_string(moe_status_t status);

/*
 * Synchronise `stream`, read and clear the current device's error word.
 * Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_BOUNDS (or
 * MOE_ERR_CUDA if the synchronisation itself failed).  *raw (may be NULL)
 * receives the raw word: bit 0 timeout, bit 1 bounds, bits 8.. the site.
 */
MOE_API moe_status_t moe_device_error(moe_stream_t stream, uint32_t* raw);

/*
 * Failure-path self-test: launch one block whose single bounded wait has no
 * producer, so it gives up after limit_us microseconds (1..1000000) and sets
 * MOE_ERR_DEVICE_TIMEOUT (site bit 17) in the device error word, exactly as a
 * stalled pipeline wait in the GEMM or router kernels would.  The context
 * stays usable.  Read the result with moe_device_error().
 */
MOE_API moe_status_t moe_selftest_wait_timeout(uint32_t limit_us, moe_stream_t stream);

/*
 * Stage tracing.  When set, every later moe_forward_ex / moe_forward call on
 * any stream records events[i] (cudaEvent_t handles created by the caller)
 * on its stream just before stage i and events[count-1] after the last:
 * stage 0 route (router GEMM + top-k, shared gate), 1 permute, 2 gate+up
 * GEMM, 3 down GEMM, 4 combine; count must be 6.  An entry may be NULL (no
 * event at that boundary; not all of them).  Pass NULL/0 to switch it off.
 * An event between two kernels ends the launch overlap between them, so
 * record only the boundaries you need.  Process-wide setting meant for
 * profiling; not thread-safe.
 */
MOE_API moe_status_t moe_set_trace_events(void* const* events, int count);

/* ABI version of this header (major * 100 + minor). */
MOE_API int moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H */
