/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse MoE FFN layer library, libmoe.so.
 *
 * The layer ["MoE 路由与专家流式加载" §1 (moe: DeepSeek-V3-style sparse routing)]:
 *   1. router: logit = x . W_router[e]; sig = sigmoid(logit); the selection
 *      bias steers which experts are chosen but the applied gate is the
 *      unbiased sig (noaux_tc); top-k by iterated argmax; optional adaptive
 *      top-p; norm_topk_prob; routed_scaling_factor            (§1.1, §1.2)
 *   2. batch-union: the experts chosen by all tokens of the batch are
 *      deduplicated; each unique expert's weights are read once and applied
 *      to every token routed to it                              (§1.3)
 *   3. expert FFN: gate/up/SiLU/down on int4 group-quantised weights (64 per
 *      group, fp32 scale per group, unsigned nibble with zero point 8) against
 *      per-token int8 activations; int32 dot per group, then the group scale
 *      ["colibri 开发演进实录" §2.1 (int4-gs64), §2.2 (K1/K1b integer dot)]
 *   4. combine: gated sum of the kept experts plus the always-on shared
 *      expert                                                   (§1.4)
 *
 * Conventions (every entry point):
 *   - Tensor pointers are DEVICE pointers, allocated and owned by the caller,
 *     16-byte aligned, row major.  The library never allocates: scratch comes
 *     from a caller-provided device workspace of at least
 *     moe_workspace_size(cfg, max_tokens) bytes (256-byte aligned).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work on it and return; they never
 *     synchronise, except moe_layer_forward with MOE_FLAG_SYNC_CHECK.
 *     Kernels are launched with programmatic dependent launch: a kernel may
 *     start while the previous work on the stream finishes, and the router
 *     reads w_router and bias before it waits for that work (the down
 *     projection likewise starts reading its weights before the h
 *     quantisation ahead of it ends).  Weights and
 *     bias are parameters: do not write them with the kernel enqueued just
 *     before a call on the same stream (an event, a copy or a host sync in
 *     between orders such a write).
 *   - Arguments are validated on the host before anything is enqueued; a bad
 *     argument returns a negative MOE_ERR_* code and enqueues nothing.
 *     moe_last_error_string() (thread-local) describes the last failure.
 *   - Weight layout, canonical (the one a checkpoint converter writes):
 *       w_gate, w_up [E][F][H/2] u8    s_gate, s_up [E][F][H/64] fp32
 *       w_down       [E][H][F/2] u8    s_down       [E][H][F/64] fp32
 *     byte j of a row holds element 2j in its low nibble and element 2j+1 in
 *     its high nibble ["colibrì 深度拆解" §5.2 pack order]; a code u in 0..15
 *     stands for (u - 8) * scale ["colibri 开发演进实录" §2.2].
 *     The shared expert uses the same layout with E = 1 and F = d_ff_shared.
 *   - Limits: H, F and Fs multiples of 64 in [64, 8192]; 1 <= E <= 512;
 *     1 <= K <= min(E, 16); 0 <= T <= 1,000,000, and (T*(K+1) + 513) *
 *     max(F, Fs)/16 and (T*(K+1) + 513) * H/64 below 1e9.  Inputs must be finite.
 *   - Alignment: weight, activation and output tensors 16 bytes; index arrays,
 *     bias and routing weights 4 bytes; the workspace 256 bytes.
 *   - The workspace's first 256 bytes hold a device error word and a counter
 *     that the kernels return to zero themselves: zero them once before the
 *     workspace is first used (e.g. allocate it zeroed).  moe_check_errors
 *     zeroes them again after it reports an error.
 *   - Determinism: every output is a deterministic function of the inputs
 *     (no floating-point atomics; reductions run in a fixed order).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define MOE_OK               0
#define MOE_ERR_ARG         -1  /* null pointer, negative count, bad flag */
#define MOE_ERR_SHAPE       -2  /* config or size outside the limits above */
#define MOE_ERR_ALIGN       -3  /* a pointer is not 16-byte aligned */
#define MOE_ERR_CUDA        -4  /* a CUDA launch or runtime call failed */
#define MOE_ERR_TIMEOUT     -5  /* a bounded device-side wait gave up */
#define MOE_ERR_UNSUPPORTED -6  /* no device of compute capability 10.3 */
#define MOE_ERR_WORKSPACE   -7  /* workspace missing or smaller than required */
#define MOE_ERR_DEVICE      -8  /* a kernel found invalid data (e.g. an expert id out of range) */

/* flags of moe_layer_forward */
#define MOE_FLAG_SYNC_CHECK    1  /* synchronise the stream and report device-side errors */
#define MOE_FLAG_STAGE_EVENTS  2  /* record a CUDA event pair around each stage (moe_stage_times) */

/* stages of moe_layer_forward, for moe_stage_times.  Batches of at most 64 tokens take the
 * decode route: ROUTER also quantises x and SELECT also runs the batch-union and the FFN
 * plan, so PERMUTE, PLAN and QUANT launch nothing; larger batches use one kernel per stage. */
#define MOE_STAGE_ROUTER   0  /* router logits (1 kernel) */
#define MOE_STAGE_SELECT   1  /* top-k, top-p, norm, scale (1 kernel) */
#define MOE_STAGE_PERMUTE  2  /* batch-union counting sort */
#define MOE_STAGE_PLAN     3  /* FFN tile plan */
#define MOE_STAGE_QUANT    4  /* int8 quantisation of x */
#define MOE_STAGE_GATE_UP  5  /* expert gate/up + SiLU*up (1 kernel) */
#define MOE_STAGE_QUANT_H  6  /* int8 quantisation of SiLU(gate)*up (1 kernel) */
#define MOE_STAGE_DOWN     7  /* expert down projection (1 kernel) */
#define MOE_STAGE_COMBINE  8  /* gated sum + shared expert (1 kernel) */
#define MOE_N_STAGES       9

typedef struct moe_config {
    int32_t hidden;                /* H */
    int32_t n_experts;             /* E, routed experts */
    int32_t top_k;                 /* K, experts per token (the g_topk override is a smaller K) */
    int32_t d_ff;                  /* F, routed expert width */
    int32_t n_shared;              /* 0 or 1 shared expert */
    int32_t d_ff_shared;           /* Fs, shared expert width */
    int32_t group_size;            /* must be 64 */
    int32_t norm_topk_prob;        /* 1: renormalise the kept gates to sum 1 */
    float routed_scaling_factor;   /* multiplies the applied gates */
    float top_p;                   /* in (0,1): adaptive top-p; otherwise off (keff = K) */
} moe_config;

typedef struct moe_expert_weights {
    const uint8_t *w_gate; const float *s_gate;
    const uint8_t *w_up;   const float *s_up;
    const uint8_t *w_down; const float *s_down;
} moe_expert_weights;

/* Optional probes of moe_expert_ffn (device pointers, each nullable), indexed
 * by pair p in permuted order (p < offsets[E]):
 *   acc_gate, acc_up [P][F][H/64] int32: per-group sum (u - 8) * xq
 *   acc_down [P][H][F/64] int32:         per-group sum (u - 8) * hq
 *   hq [P][F] int8, h_scale [P] fp32:    the quantised SiLU(gate)*up rows
 * Writing them adds stores only; the arithmetic is the same. */
typedef struct moe_ffn_probe {
    int32_t *acc_gate; int32_t *acc_up; int32_t *acc_down;
    int8_t *hq; float *h_scale;
} moe_ffn_probe;

/* Optional routing outputs of moe_layer_forward (device pointers, each
 * nullable): ids [T][K], w [T][K], keff [T], as moe_route writes them. */
typedef struct moe_routing {
    int32_t *ids; float *w; int32_t *keff;
} moe_routing;

/* Bytes of device workspace every call below needs for up to max_tokens
 * tokens.  Returns 0 for an invalid config or max_tokens < 0. */
size_t moe_workspace_size(const moe_config *cfg, int max_tokens);

/* Router look-ahead ["MoE 路由与专家流式加载" §5, la_predict]: predicts a
 * layer's top-K from a residual state with the layer's own routing pipeline.
 *   x [T][H] fp32: the residual state (e.g. an earlier layer's
 *     post-attention state); norm_w [H] fp32: the layer's RMSNorm weight;
 *     eps: the RMSNorm epsilon, finite and >= 0.
 *   The rows are normalised, x / sqrt(mean(x^2) + eps) * norm_w, into the
 *   workspace (a row with mean square + eps = 0 becomes zeros), and routed
 *   exactly like moe_route with w_router / bias (the layer's router).
 *   ids, w, keff: as moe_route writes them.
 * Same errors as moe_route, plus MOE_ERR_ARG for a bad eps. */
int moe_route_lookahead(const moe_config *cfg, const float *x, const float *norm_w, float eps,
                        const float *w_router, const float *bias, int T, int32_t *ids, float *w,
                        int32_t *keff, void *workspace, size_t workspace_bytes, void *stream);

/* Hit count of a predicted routing against the true one, per token, behind
 * the pages' recall figure ["MoE 路由与专家流式加载" §5: 71.6% of the true
 * top-8].  ids_* [T][K] int32 and keff_* [T] int32 as moe_route writes them
 * (keff values are clamped to [0, K]).  hits [T] int32: how many of the
 * first keff_pred[t] predicted ids appear among the first keff_true[t] true
 * ids.  recall = sum(hits) / sum(keff_true).  No workspace; device
 * pointers; asynchronous on stream. */
int moe_topk_hits(const moe_config *cfg, const int32_t *ids_pred, const int32_t *keff_pred,
                  const int32_t *ids_true, const int32_t *keff_true, int T, int32_t *hits,
                  void *stream);

/* Offline weight quantiser: fp32 -> the int4-gs64 layout every call above
 * reads ["colibri 开发演进实录" §2.1 int4-gs64; the pages' converter is
 * `coli convert`, §9].
 *   w [rows][K] fp32 (device, 16-byte aligned), K a multiple of 64.
 *   packed [rows][K/2] u8 and scales [rows][K/64] fp32 (device, 16-byte
 *   aligned), written in full: per 64-weight group, scale = amax / 7 and
 *   u = clamp(rint(w * (7 / amax)), -7, 7) + 8 (fp32, round half to even),
 *   byte j = element 2j (low nibble) | element 2j+1 (high); an all-zero
 *   group gets scale 0 and codes 8.
 * A whole expert set converts in one call: rows = E * F for w_gate / w_up
 * ([E][F][H], K = H), E * H for w_down (K = F).  MOE_ERR_SHAPE for rows < 0
 * or a bad K.  Asynchronous on stream. */
int moe_quantize_int4_gs64(const float *w, int rows, int K, uint8_t *packed, float *scales,
                           void *stream);

/* Offline weight quantiser to the 3-bit variant int3-g64 (fmt=5,
 * "colibri 开发演进实录" §8.3: 3-bit weights with a scale per 64 weights).  The
 * layer calls above read int4-gs64 only; this converts checkpoints to the
 * smaller container.
 *   w [rows][K] fp32 (device, 16-byte aligned), K a multiple of 64.
 *   packed [rows][3K/8] u8 and scales [rows][K/64] fp32 (device, scales 4-byte
 *   aligned), written in full: per 64-weight group, scale = amax / 3 and
 *   u = clamp(rint(w * (3 / amax)), -3, 3) + 4 (fp32, round half to even), the
 *   value standing for scale * (u - 4); the group's 64 codes fill 24 bytes, code k
 *   in bits 3k .. 3k+2 of the group's little-endian bit string (bit b in byte
 *   b / 8 at bit b % 8); an all-zero group gets scale 0 and codes 4.
 * MOE_ERR_SHAPE for rows < 0 or a bad K.  Asynchronous on stream. */
int moe_quantize_int3_g64(const float *w, int rows, int K, uint8_t *packed, float *scales,
                          void *stream);

/* Diagnostic of the error path of the kernels' bounded device-side waits:
 * one CTA polls, `polls` times (1 .. 2^24), an mbarrier that nothing arrives
 * at, gives up and records the timeout in the workspace's error word exactly
 * as the tcgen05 pipeline's waits do.  Nothing faults or hangs; the next
 * moe_check_errors on the workspace returns MOE_ERR_TIMEOUT and clears the
 * word.  workspace: any workspace of the library (>= 256 bytes, 256-byte
 * aligned).  Asynchronous on stream. */
int moe_selftest_wait_timeout(void *workspace, size_t workspace_bytes, int polls, void *stream);

/* Which grouped expert-FFN kernels a call with T tokens runs (host-side, no
 * device work): 1 = the tcgen05 tensor-core grouped GEMM, 0 = the GEMV-shaped
 * kernels.  The tensor path takes layers whose matrices have hidden, d_ff and
 * d_ff_shared in multiples of 512: on narrow ones (hidden or d_ff under 1024)
 * every batch of 32 tokens or more, otherwise batches beyond the decode route
 * (T > 64) whose expected tokens per routed expert T*K/U (U = E*(1-(1-K/E)^T),
 * the distinct experts of uniform routing) is at least 10.  1 means the tensor
 * path runs at least the down projection (moe_ffn_path / moe_ffn_path_down tell
 * each projection's kernel).  Returns -1 for an invalid config or T < 0.
 * ["MoE 路由与专家流式加载" §1.3: the expert FFN turns from a weight-streaming
 * GEMV into a dense contraction once tokens per expert grow.] */
int moe_ffn_uses_tensor_cores(const moe_config *cfg, int T);

/* Which grouped expert-FFN kernel a call with T tokens runs for gate/up
 * (moe_ffn_path) and for down (moe_ffn_path_down) (host-side, no device
 * work): MOE_FFN_TENSOR when moe_ffn_uses_tensor_cores says so -- except
 * gate/up of a narrow layer (d_ff and d_ff_shared under 1024, hidden 1024 or
 * more) with 64 tokens or fewer, and gate/up of a wide layer beyond 64 tokens
 * with under 14 expected tokens per routed expert, which take the row GEMV
 * where its shape conditions hold; otherwise
 * MOE_FFN_ROW_GEMV (one weight pass per 8 tokens, TMA-fed) when hidden, d_ff
 * and d_ff_shared are multiples of 256 and T >= 3, else MOE_FFN_WARP_GEMV.
 * Returns -1 for an invalid config or T < 0.
 * ["colibri 开发演进实录" §2.2 K1/K1b: the integer dot both GEMV kernels run.] */
#define MOE_FFN_WARP_GEMV 0
#define MOE_FFN_TENSOR    1
#define MOE_FFN_ROW_GEMV  2
int moe_ffn_path(const moe_config *cfg, int T);
int moe_ffn_path_down(const moe_config *cfg, int T);

/* Router ["MoE 路由与专家流式加载" §1.1, §1.2].
 *   x [T][H] fp32, w_router [E][H] fp32, bias [E] fp32 (selection only).
 *   ids [T][K] int32: kept experts first, in selection order (descending
 *     sig + bias; equal scores go to the lower index) or, with top-p on, in
 *     descending gate order; -1 in slots >= keff.
 *   w [T][K] fp32: applied weights (0 in slots >= keff).  keff [T] int32. */
int moe_route(const moe_config *cfg, const float *x, const float *w_router, const float *bias,
              int T, int32_t *ids, float *w, int32_t *keff,
              void *workspace, size_t workspace_bytes, void *stream);

/* moe_route without a workspace.  The pages have no counterpart of this entry
 * point; it exists for callers that cannot allocate device memory themselves,
 * e.g. a plugin inside a host engine that owns every device allocation and
 * forbids its extensions to call cudaMalloc, or a decode loop that cannot
 * afford the device synchronisation a cudaMalloc/cudaFree may cause.
 *   Same arguments, results and errors as moe_route, minus the workspace.  The
 *   router's scratch (partial logits, router_splits(T) * T * E floats) lives in
 *   a fixed 8 MiB array in device memory that libmoe.so defines; every GPU
 *   that loads the library holds it until the process exits.  A call whose
 *   scratch would exceed 2,097,152 floats returns MOE_ERR_SHAPE (for E = 256
 *   every batch up to T = 4096 fits; larger ones use moe_route with a workspace).
 *   The call allocates nothing.  Its first call on each device looks up the
 *   array's device address (cudaGetSymbolAddress) with that device current:
 *   make that first call before any stream capture.  The address is looked up
 *   again when the device's current context changes (after cudaDeviceReset, for
 *   instance); make the first call after such a reset outside stream capture too.
 *   All calls share the one array and it keeps the last call's contents; the
 *   router overwrites every scratch entry before reading it, so nothing needs
 *   clearing.  Calls that overlap on the GPU (other streams or host threads)
 *   race on the array: serialise them, e.g. on one stream. */
int moe_route_noalloc(const moe_config *cfg, const float *x, const float *w_router,
                      const float *bias, int T, int32_t *ids, float *w, int32_t *keff,
                      void *stream);

/* Batch-union ["MoE 路由与专家流式加载" §1.3] by a stable counting sort
 * ["Colibri 是什么" §3.3].  Pairs (t, i < keff[t]) are grouped by expert:
 *   counts [E], offsets [E+1] (exclusive prefix of counts),
 *   tok [T*K], slot [T*K]: pair p's token and slot t*K + i, ascending token
 *     within each expert; entries >= offsets[E] are left untouched,
 *   uniq [E]: experts with a nonzero count, ascending; n_uniq [1].
 * A kept slot whose id is outside [0, E) is left out of the lists, and a keff
 * outside [0, K] is clamped; either sets the workspace's device error word,
 * which moe_check_errors reports. */
int moe_permute(const moe_config *cfg, const int32_t *ids, const int32_t *keff, int T,
                int32_t *counts, int32_t *offsets, int32_t *tok, int32_t *slot,
                int32_t *uniq, int32_t *n_uniq,
                void *workspace, size_t workspace_bytes, void *stream);

/* Routed expert FFN over a permutation ["MoE 路由与专家流式加载" §1.3;
 * "colibri 开发演进实录" §2.2].  x [T][H] fp32 is quantised per token inside.
 * For every pair p of expert e (offsets[e] <= p < offsets[e+1]) and token
 * t = tok[p]: y_pairs[p] = down(quant(silu(gate(x_t)) * up(x_t))); y_pairs is
 * [T*K][H] fp32 and rows >= offsets[E] are left untouched.
 * offsets/tok/uniq/n_uniq as moe_permute writes them.  probe nullable. */
int moe_expert_ffn(const moe_config *cfg, const float *x, int T,
                   const moe_expert_weights *routed, const int32_t *offsets,
                   const int32_t *tok, const int32_t *uniq, const int32_t *n_uniq,
                   float *y_pairs, const moe_ffn_probe *probe,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Combine ["MoE 路由与专家流式加载" §1.3, §1.4]:
 *   y[t] = sum_{i < keff[t]} w[t][i] * y_pairs[pair(t, i)] + shared(x_t)
 * summed in slot order, then the shared expert term (when `shared` is
 * non-null and cfg->n_shared == 1; x is then needed, else it may be NULL).
 * pair(t, i) is found in expert ids[t][i]'s token list (offsets, tok); a slot
 * whose expert id is out of range or whose list lacks t adds nothing. */
int moe_combine(const moe_config *cfg, const float *y_pairs, const int32_t *ids,
                const int32_t *keff, const float *w, const int32_t *offsets,
                const int32_t *tok, int T, const float *x,
                const moe_expert_weights *shared, float *y,
                void *workspace, size_t workspace_bytes, void *stream);

/* The whole layer: route, batch-union, routed and shared expert FFN, combine.
 * y [T][H] fp32.  `shared` is required when cfg->n_shared == 1 and ignored
 * otherwise.  routing (nullable) receives the routing.  flags:
 * MOE_FLAG_SYNC_CHECK ends the call with moe_check_errors; MOE_FLAG_STAGE_EVENTS
 * brackets each stage with CUDA events on `stream` (see moe_stage_times). */
int moe_layer_forward(const moe_config *cfg, const float *x, int T, const float *w_router,
                      const float *bias, const moe_expert_weights *routed,
                      const moe_expert_weights *shared, float *y, const moe_routing *routing,
                      void *workspace, size_t workspace_bytes, int flags, void *stream);

/* moe_layer_forward on host buffers: x_host [T][H] and y_host [T][H] fp32 in
 * host memory (pinned, e.g. cudaHostAlloc, for the copies to run
 * asynchronously; pageable memory works but the copies then hold the host).
 * On the stream: x is copied into the workspace, the layer runs there, y is
 * copied back.  Every other argument, error and flag as moe_layer_forward;
 * the workspace (moe_workspace_size) holds both device copies.  Returns with
 * the work enqueued: y_host is complete once the stream has reached it. */
int moe_layer_forward_host(const moe_config *cfg, const float *x_host, int T,
                           const float *w_router, const float *bias,
                           const moe_expert_weights *routed, const moe_expert_weights *shared,
                           float *y_host, const moe_routing *routing, void *workspace,
                           size_t workspace_bytes, int flags, void *stream);

/* Synchronises `stream`, then returns MOE_ERR_DEVICE if a kernel that used
 * this workspace since the last check found invalid data (see moe_permute),
 * MOE_ERR_TIMEOUT if a bounded device-side wait gave up, and clears the record;
 * MOE_OK otherwise.  Not for use inside stream capture. */
int moe_check_errors(void *workspace, size_t workspace_bytes, void *stream);

/* Per-stage device time of the moe_layer_forward calls made on this thread
 * with MOE_FLAG_STAGE_EVENTS since the last reset: waits for their events,
 * then writes the summed milliseconds ms[MOE_N_STAGES] and the number of
 * kernel launches launches[MOE_N_STAGES] (either pointer nullable, host
 * memory).  reset != 0 clears the sums afterwards. */
int moe_stage_times(double *ms, long long *launches, int reset);

/* Description of the last error returned on this thread ("" if none). */
const char *moe_last_error_string(void);

#ifdef __cplusplus
}
#endif
#endif
