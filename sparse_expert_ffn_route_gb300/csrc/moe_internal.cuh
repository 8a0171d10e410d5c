// moe_internal.cuh -- internal declarations shared by the translation units of libmoe.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "moe.h"
#include "ffn_tiles.cuh"

namespace moe {

constexpr int kGroup = 64;        // int4 group size (one fp32 scale per 64 weights)
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 16;
constexpr int kMaxSlots = kMaxExperts + 1;  // routed experts plus the shared one
constexpr int kMaxDim = 8192;
// batches up to this many tokens take the decode route: cluster router (with the x
// quantisation) and one CTA for selection, batch-union and FFN plan
constexpr int kRouteClusterMaxT = 64;
// decode-route batches of at least this many tokens take the tensor path on narrow matrices
constexpr int kTensorMinTNarrow = 32;
// the combine adds up to this many slice planes of y, so down rows are sliced only up to
// this many 1024-input slices
constexpr int kMaxCombinePlanes = 2;

// The router's partial logits ([splits][T][E] floats) stay within this many floats whenever
// one split fits: the bound of the fixed scratch array behind moe_route_noalloc (8 MiB).
constexpr size_t kRouteScratchFloats = size_t(2) << 20;

// device-side error word bits (workspace `err`)
constexpr int kErrBadExpertId = 1;
constexpr int kErrBadKeff = 2;
constexpr int kErrTimeout = 4;     // a bounded device-side wait gave up

// ---------------------------------------------------------------------------
// Work plan of the grouped expert FFN.  A "slot" is one expert applied to its
// token list: slot 0 is the shared expert when there is one, the routed
// experts follow in ascending id.  A slot's work is cut into tiles of
// (row block, token chunk); tiles of all slots are numbered consecutively.
// ---------------------------------------------------------------------------
struct FfnPlan {
    int32_t n_slots;
    int32_t gu_tiles;                 // total gate/up tasks
    int32_t dn_tiles;                 // total down tasks
    // task counters of the kernels that hand out tasks on demand (ffn_rows.cu): the next
    // task and the CTAs finished, [0] gate/up, [1] down; zero between launches
    int32_t next[2], done[2];
    int32_t pad;
    int32_t expert[kMaxSlots];        // expert id, -1 for the shared expert
    int32_t ntok[kMaxSlots];          // tokens routed to the slot
    int32_t tokbase[kMaxSlots];       // first entry of the slot's list in tok[] (routed)
    int32_t rowbase[kMaxSlots];       // first output row of the slot
    int32_t gu_prefix[kMaxSlots + 1]; // exclusive prefix of gate/up tasks per slot
    int32_t dn_prefix[kMaxSlots + 1];
    int64_t gu_cost[kMaxSlots + 1];   // exclusive prefix of gate/up task cost per slot
    int64_t dn_cost[kMaxSlots + 1];
};

// Quantised activations: per row n int8 codes stored with each run of 8
// elements as [e0 e2 e4 e6 | e1 e3 e5 e7] (the even/odd split that the packed
// nibbles' low/high halves line up with), the row scale, and the sum of the
// codes of every 32-element chunk (for the zero-point-8 correction).
// (cuda_bf16.h is included above)
struct QuantRows {
    int8_t *q;       // [rows][q_ld]
    float *scale;    // [rows]
    int32_t *csum;   // [rows][c_ld], c_ld >= n/32
    int q_ld, c_ld;
    __nv_bfloat16 *bf16;   // nullable: [rows][q_ld] the codes again as bf16, element order
};

struct FfnArgs {
    // problem
    int H, F, Fs, E, K, T, n_shared;
    int32_t *err;                     // device error word (pipeline timeouts)
    int include_routed;               // 0: shared expert only
    // routed and shared weights (canonical layout)
    moe_expert_weights routed, shared;
    // routing lists
    const int32_t *offsets, *tok;
    const FfnPlan *plan;
    // activations
    QuantRows xq;                     // [T][H]
    float *h;                         // [rows][hstride] fp32 SiLU(gate)*up
    int hstride;
    QuantRows hq;                     // [rows][hstride] quantised h
    float *y;                         // [S_down][plane_rows][H] fp32 output rows (plane 0
                                      // holds the result when down rows are not sliced)
    float *gpart, *upart;             // [S_gate/up][plane_rows][hstride] partial gate / up
    int plane_rows;                   // output rows of the call (shared rows + routed pairs)
    int slice_gu, slice_dn;           // rows cut into 1024-input slices
    int tensor, tensor_dn;            // the tcgen05 path (ffn_tc.cu) runs gate/up / down
    int rows, rows_dn;                // the row GEMV (ffn_rows.cu) runs gate/up / down
    __nv_bfloat16 *x_bf16;            // [rows][H] the codes of x per output row as bf16 (tensor path)
    __nv_bfloat16 *h_bf16;            // [rows][hstride] the codes of h as bf16 (tensor path)
    int tc_gu, tc_dn;                 // token chunk per task
    Geo geo_gu[2], geo_dn[2];         // task geometry: [0] routed experts, [1] shared expert
    moe_ffn_probe probe;              // routed pairs only; row index = pair
    int routed_rowbase;               // output row of routed pair 0
    // the row GEMV's gate/up may run the shared expert's tasks before its dependency wait:
    // set only when the x codes come from a kernel at least two launches earlier
    int shared_early;
};

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
struct WsLayout {
    size_t ids, w, keff;              // routing (layer_forward)
    size_t counts, offsets, tok, slot, uniq, n_uniq, pair_of;
    size_t logits;                    // router partial logits [S][T][E]
    size_t xq, xscale, xcsum;         // quantised x
    size_t h;                         // [rows][Fmax] fp32
    size_t hp, hp_plane_floats;       // partial gate planes then partial up planes
    size_t xbf, hbf;                  // bf16 codes of x and h (tensor path)
    size_t xn;                        // [T][H] fp32 RMSNorm output (router look-ahead)
    size_t xs, ys;                    // [T][H] fp32 device copies of host x and y (host call)
    size_t hq, hscale, hcsum;         // quantised h
    size_t y;                         // [rows][H] fp32 (shared rows, then routed pairs)
    size_t plan;                      // FfnPlan
    size_t err;                       // int32 device error word
    size_t total;
};

WsLayout ws_layout(const moe_config &c, int max_tokens);
int router_splits(const moe_config &c, int T);

// ---------------------------------------------------------------------------
// launchers (return cudaError_t of the launch)
// ---------------------------------------------------------------------------
// router logits into `scratch` ([T][E] final logits for T <= kRouteClusterMaxT, else
// [splits][T][E] partial sums); with xq non-null (decode route only) also quantises x
cudaError_t launch_router_logits(const moe_config &c, const float *x, const float *wr, int T,
                                 float *scratch, const QuantRows *xq, int *splits, cudaStream_t st);
cudaError_t launch_router_select(const moe_config &c, const float *scratch, int splits,
                                 const float *bias, int T, int32_t *ids, float *w, int32_t *keff,
                                 cudaStream_t st);
// logits + selection (moe_route)
cudaError_t launch_router(const moe_config &c, const float *x, const float *wr, const float *bias,
                          int T, float *scratch, int32_t *ids, float *w, int32_t *keff,
                          cudaStream_t st);
// outputs of the batch-union
struct PermuteOut {
    int32_t *counts, *offsets, *tok, *slot, *uniq, *n_uniq, *err;
    int32_t *pair_of;   // nullable: [T*K] list position of pair (t, i), -1 for i >= keff[t]
};
// one CTA: selection from final logits [T][E] (T <= kRouteClusterMaxT), then, when perm is
// non-null, the batch-union, then, when plan_args is non-null, the FFN plan
cudaError_t launch_route_tail(const moe_config &c, const float *logits, const float *bias, int T,
                              int32_t *ids, float *w, int32_t *keff, const PermuteOut *perm,
                              const FfnArgs *plan_args, cudaStream_t st);
cudaError_t launch_permute(const moe_config &c, const int32_t *ids, const int32_t *keff, int T,
                           const PermuteOut &o, cudaStream_t st);
cudaError_t launch_plan(const FfnArgs &a, const int32_t *uniq, const int32_t *n_uniq,
                        FfnPlan *plan, cudaStream_t st);
cudaError_t launch_quant_rows(const float *src, int rows, int n, int src_stride, QuantRows dst,
                              cudaStream_t st);
// quantise the h rows of an FFN call: `first_rows` rows of n_first values, then the routed
// pair rows (count read on the device from offsets[n_experts]) of n_rest values
cudaError_t launch_quant_h(const FfnArgs &a, int first_rows, int n_first, int n_rest,
                           int max_rows, cudaStream_t st);
// the x codes of every output row of an FFN call as bf16 (tensor-core path): `first_rows`
// shared-expert rows, then the routed pair rows (count read on the device)
cudaError_t launch_gather_x_bf16(const FfnArgs &a, int first_rows, int max_rows, cudaStream_t st);
// host-side choice of the FFN kernels' tile shape and pipeline depth
void ffn_configure(FfnArgs &a);
cudaError_t launch_ffn_gate_up(const FfnArgs &a, cudaStream_t st);
// tensor-core path (ffn_tc.cu): whole 128-row tiles of every matrix of the call
bool ffn_tc_supported(const FfnArgs &a);
// the tcgen05 path takes an FFN call when its batch is beyond the decode route, its matrices
// are supported, and it has enough tokens per routed expert (ffn_gemv.cu)
bool ffn_use_tensor_cores(const FfnArgs &a);
cudaError_t launch_ffn_tc(bool gate_up, const FfnArgs &a, cudaStream_t st);
// row GEMV (ffn_rows.cu): reductions that are multiples of 256 inputs, 16-byte aligned
// operands; one pass over each 64-row weight block per chunk of up to 16 tokens
bool ffn_rows_supported(const FfnArgs &a);
// a narrow decode-route layer whose gate/up takes the row GEMV and down the tensor path
bool ffn_split_paths(const FfnArgs &a);
cudaError_t launch_ffn_rows(bool gate_up, const FfnArgs &a, cudaStream_t st);
cudaError_t launch_ffn_down(const FfnArgs &a, cudaStream_t st);
// pair_of (nullable) gives each (t, i) its list position directly; without it the position
// is found by binary search in the expert's token list.  S_r / S_s slice planes (plane
// stride `plane` floats) hold the routed / shared rows' partial sums.
cudaError_t launch_combine(const moe_config &c, const float *y_routed, int64_t routed_row_stride,
                           const float *y_shared, const int32_t *ids, const int32_t *keff,
                           const float *w, const int32_t *offsets, const int32_t *tok,
                           const int32_t *pair_of, int S_r, int S_s, int64_t plane, int T,
                           float *y, cudaStream_t st);

// router look-ahead (lookahead.cu): RMSNorm of [T][H] rows, and the per-token count of the
// experts two routings both keep
cudaError_t launch_rmsnorm(const float *x, const float *g, float eps, int T, int H, float *out,
                           cudaStream_t st);
cudaError_t launch_topk_hits(const int32_t *ids_pred, const int32_t *keff_pred,
                             const int32_t *ids_true, const int32_t *keff_true, int T, int K,
                             int32_t *hits, cudaStream_t st);

// offline fp32 -> int4-gs64 weight quantiser (quantize_weights.cu)
cudaError_t launch_quantize_int4(const float *w, int rows, int K, uint8_t *packed, float *scales,
                                 cudaStream_t st);
cudaError_t launch_quantize_int3(const float *w, int rows, int K, uint8_t *packed, float *scales,
                                 cudaStream_t st);

// diagnostic: one bounded wait on an mbarrier nothing arrives at (selftest.cu)
cudaError_t launch_selftest_wait(int32_t *err, int polls, cudaStream_t st);

// host helpers shared with the entry points outside moe_api.cu
int set_error(int code, const char *fmt, ...);   // records the thread's last error message
int require_device();                            // MOE_OK on a compute capability 10.3 device
int validate_route_args(const moe_config *cfg, const float *x, const float *w_router,
                        const float *bias, int T, const int32_t *ids, const float *w,
                        const int32_t *keff);

int num_sms();

}  // namespace moe
