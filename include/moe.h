/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse Mixture-of-Experts layer.
 *
 * One GPU, one layer: router GEMM -> softmax -> top-k gating with a capacity
 * limit -> permutation into expert-contiguous rows -> grouped two-layer expert
 * FFN -> gate-weighted combine -> aux load-balance statistics, and the
 * backward pass of all of it.
 *
 * Sources (the web pages that state the layer):
 *   [LLaMA4-MoE] "Hand-building a LLaMA4-MoE" guide, §2.4 (router + softmax,
 *                top-K index [B,K], sort by expert id, per-expert split,
 *                two-layer FFN experts, gate-weighted sum, gradients through
 *                the routing weights), §3.2 (Switch aux loss, gate noise).
 *   [ZeRO3-MoE]  "DeepSpeed ZeRO-3 and MoE memory accounting" guide, §3.1 and
 *                §3.4 (per-expert capacity, capacity_factor 1.2, gate_noise),
 *                §3.2 (variance aux loss), §5.3 (gating computed in fp32).
 *   [Twinkle]    "Twinkle adapts DeepSeek-V4 training" notes, §3.1
 *                (scores = W_router x, softmax, top-k with k = 2).
 *   Shared experts (experts every token passes through, [LLaMA4-MoE] §5.2)
 *   are optional: moe_config.f_shared > 0 and a moe_shared_ffn block.
 *
 * Conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer unless stated, owned by the
 *     caller; the library never allocates or frees device memory.  Scratch
 *     space is the caller's workspace of moe_workspace_size() bytes.
 *   - Row-major tensors.  Expert weights are stacked per expert:
 *     W_up[E,d,f], W_gate[E,d,f], W_down[E,f,d]; router W_r[d,E].
 *   - "act" tensors have the layer dtype (fp32 or bf16, bit pattern uint16);
 *     logits, gates, probabilities, statistics, bias, noise and dgate/dlogits
 *     are always fp32; indices are int32.
 *   - All pointers must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  No call synchronises the host on the hot path:
 *     row counts decided on the device (offsets) are read by later kernels
 *     on the device; buffers of permuted rows are sized for the worst case
 *     returned by moe_rows_capacity().
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_*.  Host-side argument
 *     checks run before anything is launched.  Conditions found on the
 *     device (a bounded wait that ran out, non-finite logits) are recorded
 *     in a device status word read by moe_last_device_status().
 *   - Fail fast after a timeout: once a bounded wait has run out
 *     (MOE_ERR_TIMEOUT in the status word), every other wait on the device
 *     gives up at its next check, and the router and grouped-GEMM kernels
 *     launched before the host reads the status skip their work.  Outputs of
 *     calls made between the timeout and that read are undefined.
 *   - Per-device state (the status word's address, kernel attributes, the
 *     no-allocation router's scratch address) is looked up once per device and
 *     kept for the life of the process.  After cudaDeviceReset on a device
 *     those cached values are stale: do not call this library on that device
 *     again in the same process.
 *   - Gradients are written, never accumulated into.
 *   - Results are deterministic: no floating-point atomics; reruns on the
 *     same inputs give identical bytes.
 */
#ifndef GB300_MOE_H
#define GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same handle as cudaStream_t */

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* ---- status codes ---- */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)   /* bad shape, null or misaligned pointer      */
#define MOE_ERR_UNSUPPORTED (-2)   /* valid but not implemented (see moe_check_config) */
#define MOE_ERR_CUDA (-3)          /* a CUDA runtime call failed                 */
#define MOE_ERR_TIMEOUT (-4)       /* device: a bounded wait gave up             */
#define MOE_ERR_NONFINITE (-5)     /* device: a router logit was NaN or infinite */
#define MOE_ERR_DEVICE_BOUNDS (-6) /* device: an index read from memory was out of range */
#define MOE_ERR_SCRATCH_LIMIT (-7) /* moe_route_noalloc: the configuration needs more scratch
                                      than MOE_ROUTE_NOALLOC_SCRATCH_BYTES                */

/* ---- configuration ---- */
#define MOE_DTYPE_F32 0
#define MOE_DTYPE_BF16 1
#define MOE_FFN_SILU 0   /* y = W_down^T silu(W_up^T x)                        */
#define MOE_FFN_SWIGLU 1 /* y = W_down^T (silu(W_gate^T x) * (W_up^T x))        */

typedef struct {
    int32_t T;               /* tokens                                          */
    int32_t d;               /* model width                                     */
    int32_t f;               /* expert hidden width                             */
    int32_t E;               /* experts, 1..64                                  */
    int32_t k;               /* experts per token, 1..min(E, 8)                 */
    float capacity_factor;   /* <= 0: no limit; else C = ceil(cf*T*k/E), in IEEE
                                double from this fp32 value, clamped to T        */
    int32_t ffn;             /* MOE_FFN_SILU or MOE_FFN_SWIGLU                   */
    int32_t dtype;           /* MOE_DTYPE_F32 or MOE_DTYPE_BF16                  */
    int32_t normalize_gates; /* 1: gates = softmax over the k selected logits (sum
                                to 1 before drops); 0: raw softmax probabilities */
    float aux_coef;          /* lambda of L_aux = lambda * sum_e (pbar_e - 1/E)^2 */
    int32_t pad_m;           /* rows of each expert segment are padded to a
                                multiple of pad_m; bf16 needs a multiple of 128  */
    float temperature;       /* softmax temperature tau: p = softmax(logits / tau)
                                ([Twinkle] §3.1, [ZeRO3-MoE] §3.2); 0 means 1     */
    int32_t straight_through;/* 1: Gumbel top-k with a straight-through estimator
                                ([Twinkle] §3.1): experts are selected on
                                logits + noise (noise = the caller's Gumbel draws),
                                `logits` stays noise-free, gates are 1 in the
                                forward, and the backward flows through
                                softmax(logits / tau) at the selected experts     */
    int32_t f_shared;        /* hidden width of the shared experts' FFN, 0 = none
                                ([LLaMA4-MoE] §5.2).  n shared experts of width
                                f_e are one FFN of width n f_e (weight blocks
                                side by side); bf16 needs a multiple of 128      */
} moe_config;

/* Shared experts ([LLaMA4-MoE] §5.2: a fixed set of experts joins every
 * token's computation).  They are one dense FFN of width f_shared, of the
 * routed experts' kind (cfg->ffn), added to every token's output with weight
 * 1 -- padding tokens included, since the token mask concerns expert
 * selection only.  Ts = moe_shared_rows(cfg) rows (T rounded up to 128 for
 * bf16; rows >= T of h, act and y are zeros).  Entry points that take a
 * `const moe_shared_ffn*` require it iff cfg->f_shared > 0 (NULL otherwise);
 * each reads or writes only the fields listed for it.                        */
typedef struct {
    const void* x;        /* [T, d] layer input                (ffn, ffn_backward)   */
    const void* W_up;     /* [d, f_shared]                     (ffn, ffn_backward)   */
    const void* W_gate;   /* [d, f_shared], SwiGLU only, else NULL                   */
    const void* W_down;   /* [f_shared, d]                     (ffn, ffn_backward)   */
    void* h;              /* [nh, Ts, f_shared] h, or g then u (ffn writes)          */
    void* act;            /* [Ts, f_shared]                    (ffn writes)          */
    void* y;              /* [Ts, d] shared output (ffn writes, moe_combine reads)   */
    const void* dout;     /* [T, d] gradient of the layer output (ffn_backward reads)*/
    void* dh;             /* [nh, Ts, f_shared] intermediate   (ffn_backward writes) */
    void* dx;             /* [Ts, d] the shared FFN's input gradient (ffn_backward
                             writes; moe_router_backward adds it into dx)           */
    void* dW_up;          /* [d, f_shared] weight gradients    (ffn_backward writes) */
    void* dW_gate;        /* [d, f_shared], SwiGLU only                              */
    void* dW_down;        /* [f_shared, d]                                           */
} moe_shared_ffn;

/* ---- statistics vector written by moe_route / moe_permute (fp32, 9 + E) ----
 * Means run over the routed tokens (tokens not masked out).                  */
#define MOE_STAT_AUX_LOSS 0      /* lambda * sum_e (pbar_e - 1/E)^2   [ZeRO3-MoE] §3.2 */
#define MOE_STAT_AUX_SWITCH 1    /* E * sum_e f_e pbar_e, f = counts/(T k) [LLaMA4-MoE] §3.2 */
#define MOE_STAT_ENTROPY 2       /* mean over tokens of -sum_e p log p  [LLaMA4-MoE] §3.3 */
#define MOE_STAT_NONFINITE 3     /* tokens with a NaN/Inf logit                      */
#define MOE_STAT_DROPPED 4       /* assignments dropped by capacity (moe_permute)    */
#define MOE_STAT_MAX_OVER_MEAN_KEPT 5  /* max_e kept_e / mean_e kept_e (moe_permute) */
#define MOE_STAT_COUNT_CV 6      /* std/mean of counts over experts                  */
#define MOE_STAT_MAX_OVER_MEAN_COUNT 7
#define MOE_STAT_TOKENS 8        /* routed tokens (not masked out)                   */
#define MOE_STAT_PBAR 9          /* pbar[0..E): mean softmax probability per expert  */
#define MOE_STATS_LEN(E) (9 + (E))

/* Validate a configuration.  MOE_OK, MOE_ERR_INVALID_ARG (impossible shape)
 * or MOE_ERR_UNSUPPORTED (bf16 needs d % 128 == 0, f % 128 == 0 and
 * pad_m % 128 == 0; E <= 64; k <= 8).                                         */
MOE_API int moe_check_config(const moe_config* cfg);

/* Per-expert capacity C (T when there is no limit).  [ZeRO3-MoE] §3.1, §3.4  */
MOE_API int moe_capacity(const moe_config* cfg, int32_t* capacity);

/* Worst-case row count of the permuted buffers (x_perm, act, y_perm, ...):
 * min(T*k, E*C) + E*(pad_m - 1).  Each buffer holds rows_cap rows.            */
MOE_API int moe_rows_capacity(const moe_config* cfg, int64_t* rows_cap);

/* Rows Ts of the shared experts' buffers (h, act, y, dh, dx of moe_shared_ffn):
 * T rounded up to a multiple of 128 for bf16, T for fp32; 0 if f_shared = 0. */
MOE_API int moe_shared_rows(const moe_config* cfg, int64_t* rows);

/* Bytes of scratch `ws` that every entry point below may use (the maximum
 * over all of them, including moe_backward's intermediate gradients).        */
MOE_API int moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* ---- forward ---- */

/* Router: logits = x W_r (+ bias) (+ noise) in fp32 accumulation; softmax of
 * logits / tau; top-k (largest logits; ties to the lowest expert id; NaN ranks
 * lowest), slot j = rank j; gates; per-expert selection counts; statistics.
 *   x[T,d] act dtype; W_r[d,E] act dtype; bias[E] fp32 or NULL;
 *   noise[T,E] fp32 or NULL: gate noise drawn by the caller ([LLaMA4-MoE] §3.2),
 *     added to the logits; in straight-through mode the Gumbel draws that
 *     perturb only the selection;
 *   token_mask[T] uint8 or NULL: 0 marks a padding token, which takes no part
 *     in routing ([LLaMA4-MoE] §4.1): topk -1, gates 0, no counts, no output,
 *     no gradient, and it is left out of every statistic;
 *   out: logits[T,E] fp32, topk_idx[T,k] int32, gate[T,k] fp32,
 *        counts[E] int32, stats[9+E] fp32 (entries 4 and 5 by moe_permute).
 * [LLaMA4-MoE] §2.4; [Twinkle] §3.1; [ZeRO3-MoE] §5.3.                         */
MOE_API int moe_route(const moe_config* cfg, const void* x, const void* W_r, const float* bias,
              const float* noise, const uint8_t* token_mask, float* logits, int32_t* topk_idx,
              float* gate, int32_t* counts, float* stats, void* ws, moe_stream_t stream);

/* Router for callers that cannot allocate device memory (no counterpart in the
 * pages: it exists for embedding).  Some hosts own all device memory through
 * their own pool and forbid side allocations once running, and some latency
 * paths cannot afford cudaMalloc's cost and implicit synchronisation; such
 * callers cannot hand moe_route a workspace.  This entry point runs the same
 * kernels as moe_route, with the same arguments minus `ws`; its scratch is a
 * static device array of MOE_ROUTE_NOALLOC_SCRATCH_BYTES that every GPU loading
 * the library holds until the process exits.  It calls no allocator.
 *   - Configurations needing more scratch than that (moe_workspace_size's
 *     router share: per-CTA partials plus E_pad*d bf16 transposed router
 *     weights) return MOE_ERR_SCRATCH_LIMIT before anything is launched.
 *   - The first call on each device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is cached for the life of the process, so it is stale after
 *     a cudaDeviceReset of that device (see the conventions above).
 *   - All calls share the array and it keeps the last call's contents (every
 *     word is written before it is read, so nothing needs clearing); calls
 *     whose kernels overlap on the GPU race on it.                            */
#define MOE_ROUTE_NOALLOC_SCRATCH_BYTES (2u * 1024u * 1024u)
MOE_API int moe_route_noalloc(const moe_config* cfg, const void* x, const void* W_r,
                              const float* bias, const float* noise, const uint8_t* token_mask,
                              float* logits, int32_t* topk_idx, float* gate, int32_t* counts,
                              float* stats, moe_stream_t stream);

/* Capacity + permutation: rank each assignment (t, j) among its expert's
 * assignments in ascending token order; keep it iff rank < C; lay experts out
 * contiguously (segment e = rows offsets[e]..offsets[e+1], kept[e] real rows
 * then zero rows up to a multiple of pad_m) and gather x rows into x_perm.
 *   in : x[T,d], topk_idx[T,k]
 *   out: x_perm[rows_cap,d] (rows >= offsets[E] untouched), perm_token[rows_cap]
 *        (token of each row, -1 on padding rows), slot_of[T,k] (row of (t,j),
 *        -1 if dropped), kept[E], offsets[E+1]; stats (may be NULL) gets
 *        MOE_STAT_DROPPED and MOE_STAT_MAX_OVER_MEAN_KEPT.
 * [LLaMA4-MoE] §2.4 (sort by expert id, split by counts); [ZeRO3-MoE] §3.1.   */
MOE_API int moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                void* x_perm, int32_t* perm_token, int32_t* slot_of, int32_t* kept,
                int32_t* offsets, float* stats, void* ws, moe_stream_t stream);

/* Grouped expert FFN over the segments given by offsets (read on the device).
 *   SiLU  : h = x_perm W_up[e]; act = silu(h); y = act W_down[e]
 *   SwiGLU: g = x_perm W_gate[e]; u = x_perm W_up[e]; act = silu(g)*u; y = act W_down[e]
 *   h_saved[nh,rows_cap,f] (nh = 1: h; nh = 2: g then u), act[rows_cap,f],
 *   y_perm[rows_cap,d]; all act dtype; W_gate may be NULL for SiLU.
 *   shared: the shared experts' FFN on all T tokens, run in the same GEMM
 *   launches as the routed experts (reads x, W_*; writes h, act, y).
 * [LLaMA4-MoE] §2.4 (each expert a two-layer FFN), §5.2 (shared experts).    */
MOE_API int moe_grouped_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                    const void* W_up, const void* W_gate, const void* W_down,
                    void* h_saved, void* act, void* y_perm, const moe_shared_ffn* shared,
                    void* ws, moe_stream_t stream);

/* Combine: out[t] = sum over kept slots j (ascending) of gate[t,j] * y_perm[slot_of[t,j]]
 * (+ shared->y[t] with weight 1), fp32 accumulation; a token whose slots were
 * all dropped gets only the shared output (zeros without shared experts).
 * [LLaMA4-MoE] §2.4 (weighted by the post-softmax routing score).             */
MOE_API int moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* slot_of,
                const float* gate, const moe_shared_ffn* shared, void* out,
                moe_stream_t stream);

/* ---- backward of  L = <dout, out> + L_aux  ---- */

/* Combine backward: dy_perm[r] = gate[t,j] * dout[t] for r = slot_of[t,j],
 * zero on padding rows; dgate[t,j] = <dout[t], y_perm[r]> (0 if dropped).     */
MOE_API int moe_combine_backward(const moe_config* cfg, const void* dout, const void* y_perm,
                         const float* gate, const int32_t* slot_of, const int32_t* perm_token,
                         const int32_t* offsets, void* dy_perm, float* dgate,
                         moe_stream_t stream);

/* Grouped FFN backward.  dact = dy W_down[e]^T; dh = dact * silu'(h)
 * (SwiGLU: du = dact * silu(g), dg = dact * u * silu'(g));
 * dW_down[e] = act_e^T dy_e; dW_up[e] = x_e^T dh_e (dW_gate[e] = x_e^T dg_e),
 * each summed over expert e's rows only (a variable-length reduction);
 * dx_perm = dh W_up[e]^T (+ dg W_gate[e]^T).
 *   dh[nh,rows_cap,f] act dtype is an output buffer of intermediate gradients
 *   (nh as h_saved: dh, or dg then du); dx_perm[rows_cap,d];
 *   dW_up/dW_gate[E,d,f], dW_down[E,f,d] act dtype.
 *   shared: the same for the shared FFN with dy = dout (weight 1), in the same
 *   launches (reads x, W_*, h, act, dout; writes dh, dx, dW_*).               */
MOE_API int moe_grouped_ffn_backward(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                             const void* W_up, const void* W_gate, const void* W_down,
                             const void* h_saved, const void* act, const void* dy_perm,
                             void* dh, void* dx_perm, void* dW_up, void* dW_gate, void* dW_down,
                             const moe_shared_ffn* shared, void* ws, moe_stream_t stream);

/* Router backward.  dlogits[t] = gate softmax Jacobian applied to dgate
 * (selected logits only; raw and straight-through gates through the full
 * softmax) + aux term lambda*2(pbar-1/E)/T_routed through the full softmax,
 * all divided by tau; masked tokens get none; dx[t] = sum over kept slots of
 * dx_perm[slot] + dlogits[t] W_r^T (+ shared->dx[t]);
 * dW_r = x^T dlogits; dbias = sum_t dlogits (if non-NULL).
 *   stats: the moe_route statistics of the same forward (pbar is used).
 *   dlogits[T,E] fp32 output (may be NULL: then ws is used).
 * [LLaMA4-MoE] §2.4 (do not detach the routing weights).                      */
MOE_API int moe_router_backward(const moe_config* cfg, const void* x, const void* W_r,
                        const float* logits, const int32_t* topk_idx, const float* gate,
                        const int32_t* slot_of, const float* dgate, const void* dx_perm,
                        const moe_shared_ffn* shared, const float* stats, void* dx, void* dW_r,
                        float* dbias, float* dlogits, void* ws, moe_stream_t stream);

/* Whole backward: moe_combine_backward -> moe_grouped_ffn_backward ->
 * moe_router_backward, intermediates in ws.  Saved forward tensors as above;
 * with shared experts, shared->dout is taken to be `dout` and shared->dh /
 * shared->dx may be NULL (the workspace then holds them).                    */
MOE_API int moe_backward(const moe_config* cfg, const void* x, const void* W_r, const void* W_up,
                 const void* W_gate, const void* W_down, const float* logits,
                 const int32_t* topk_idx, const float* gate, const int32_t* slot_of,
                 const int32_t* perm_token, const int32_t* offsets, const void* x_perm,
                 const void* h_saved, const void* act, const void* y_perm, const float* stats,
                 const void* dout, void* dx, void* dW_r, float* dbias, void* dW_up,
                 void* dW_gate, void* dW_down, const moe_shared_ffn* shared, void* ws,
                 moe_stream_t stream);

/* ---- status and bookkeeping ---- */

/* Text of a status code (static storage). */
MOE_API const char* moe_error_string(int code);

/* Synchronise `stream`, then read and clear the device status word of the
 * current device (*status = MOE_OK or a MOE_ERR_* recorded by a kernel).     */
MOE_API int moe_last_device_status(moe_stream_t stream, int* status);

/* Number of kernels this library has launched in this process (host counter). */
MOE_API uint64_t moe_launch_count(void);

/* Self-test of the failure path (no counterpart in the pages): launches one
 * kernel that waits, with the bounded wait every TMA-fed kernel uses, on an
 * mbarrier that nothing arrives on.  The wait gives up after limit_ns
 * nanoseconds (1 ns .. 1 s, else MOE_ERR_INVALID_ARG), records MOE_ERR_TIMEOUT
 * in the device status word and the kernel returns; read it with
 * moe_last_device_status.  The GPU context stays usable.                     */
MOE_API int moe_selftest_bounded_wait(unsigned long long limit_ns, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GB300_MOE_H */
