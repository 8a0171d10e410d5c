// moe_api.cu -- the extern "C" entry points of libmoe.so: argument validation, workspace
// layout and the launch sequence of each call.  See include/moe.h for the contract.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "ffn_tiles.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

thread_local char g_err[512];

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok()
{
    g_err[0] = 0;
    return MOE_OK;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kMaxTokens = 1000000;

int check_config(const moe_config *c)
{
    if (!c) return fail(MOE_ERR_ARG, "cfg is NULL");
    if (c->group_size != kGroup) return fail(MOE_ERR_SHAPE, "group_size must be 64 (got %d)", c->group_size);
    if (c->hidden < kGroup || c->hidden > kMaxDim || c->hidden % kGroup)
        return fail(MOE_ERR_SHAPE, "hidden must be a multiple of 64 in [64, %d] (got %d)", kMaxDim, c->hidden);
    if (c->n_experts < 1 || c->n_experts > kMaxExperts)
        return fail(MOE_ERR_SHAPE, "n_experts must be in [1, %d] (got %d)", kMaxExperts, c->n_experts);
    if (c->top_k < 1 || c->top_k > kMaxTopK || c->top_k > c->n_experts)
        return fail(MOE_ERR_SHAPE, "top_k must be in [1, min(n_experts, %d)] (got %d)", kMaxTopK, c->top_k);
    if (c->d_ff < kGroup || c->d_ff > kMaxDim || c->d_ff % kGroup)
        return fail(MOE_ERR_SHAPE, "d_ff must be a multiple of 64 in [64, %d] (got %d)", kMaxDim, c->d_ff);
    if (c->n_shared != 0 && c->n_shared != 1)
        return fail(MOE_ERR_SHAPE, "n_shared must be 0 or 1 (got %d)", c->n_shared);
    if (c->n_shared && (c->d_ff_shared < kGroup || c->d_ff_shared > kMaxDim || c->d_ff_shared % kGroup))
        return fail(MOE_ERR_SHAPE, "d_ff_shared must be a multiple of 64 in [64, %d] (got %d)", kMaxDim,
                    c->d_ff_shared);
    if (c->norm_topk_prob != 0 && c->norm_topk_prob != 1)
        return fail(MOE_ERR_ARG, "norm_topk_prob must be 0 or 1 (got %d)", c->norm_topk_prob);
    if (!(c->routed_scaling_factor == c->routed_scaling_factor) ||
        c->routed_scaling_factor > 3.0e38f || c->routed_scaling_factor < -3.0e38f)
        return fail(MOE_ERR_ARG, "routed_scaling_factor must be finite");
    if (!(c->top_p == c->top_p)) return fail(MOE_ERR_ARG, "top_p must not be NaN");
    return MOE_OK;
}

int check_tokens(int T)
{
    if (T < 0 || T > kMaxTokens) return fail(MOE_ERR_SHAPE, "T must be in [0, %d] (got %d)", kMaxTokens, T);
    return MOE_OK;
}

// The FFN kernels number their tiles with int32: bound the count for the worst routing
// (every pair in its own one-token chunk).
int check_tile_count(const moe_config &c, int T)
{
    const double pairs = (double)T * c.top_k + (c.n_shared ? (double)T : 0.0) + kMaxSlots;
    const int fm = c.n_shared && c.d_ff_shared > c.d_ff ? c.d_ff_shared : c.d_ff;
    const double gu = pairs * ((fm + 7) / 8), dn = pairs * ((c.hidden + 7) / 8);
    if (gu > 1.0e9 || dn > 1.0e9)
        return fail(MOE_ERR_SHAPE, "T=%d is too large for this layer (tile count would exceed 1e9)", T);
    return MOE_OK;
}

#define REQUIRE_PTR(p, a)                                                                      \
    do {                                                                                       \
        if (!(p)) return fail(MOE_ERR_ARG, "%s is NULL", #p);                                  \
        if (!aligned((p), (a))) return fail(MOE_ERR_ALIGN, "%s is not %d-byte aligned", #p, (int)(a)); \
    } while (0)

int check_weights(const moe_expert_weights *w, const char *name)
{
    if (!w) return fail(MOE_ERR_ARG, "%s weights are NULL", name);
    const void *p[6] = {w->w_gate, w->s_gate, w->w_up, w->s_up, w->w_down, w->s_down};
    static const char *nm[6] = {"w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down"};
    for (int i = 0; i < 6; ++i) {
        if (!p[i]) return fail(MOE_ERR_ARG, "%s.%s is NULL", name, nm[i]);
        if (!aligned(p[i], 16)) return fail(MOE_ERR_ALIGN, "%s.%s is not 16-byte aligned", name, nm[i]);
    }
    return MOE_OK;
}

// compute capability 10.3 check, cached per device
std::atomic<int> g_dev_ok[64];
std::atomic<int> g_dev_sms[64];

int check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fail(MOE_ERR_UNSUPPORTED, "no CUDA device is available");
    }
    int st = g_dev_ok[dev].load();
    if (st == 0) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaGetLastError();
        st = (major == 10 && minor == 3) ? 1 : -1;
        g_dev_sms[dev].store(sms > 0 ? sms : 1);
        g_dev_ok[dev].store(st);
    }
    if (st < 0) return fail(MOE_ERR_UNSUPPORTED, "libmoe.so is built for sm_103a; device %d is not compute capability 10.3", dev);
    return MOE_OK;
}

int check_ws(const moe_config &c, int T, void *ws, size_t bytes, WsLayout *L)
{
    *L = ws_layout(c, T);
    if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_ALIGN, "workspace is not 256-byte aligned");
    if (bytes < L->total)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes; %zu needed for T=%d", bytes, L->total, T);
    return MOE_OK;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

template <typename P>
P *at(void *ws, size_t off)
{
    return reinterpret_cast<P *>(static_cast<char *>(ws) + off);
}

size_t logits_rows(const moe_config &c, int T)
{
    // max over T' <= T of S(T') * T' (monotone in T, so regions never shrink as T grows)
    size_t best = 0;
    const int tiles = (T + 63) / 64;
    for (int ct = 1; ct <= tiles; ++ct) {
        const int tp = ct * 64 < T ? ct * 64 : T;
        const int s = router_splits(c, tp);
        const size_t v = (size_t)s * tp;
        if (v > best) best = v;
        if (s == 1) {
            if ((size_t)T > best) best = T;
            break;
        }
    }
    return best;
}

int fmax_of(const moe_config &c) { return c.n_shared && c.d_ff_shared > c.d_ff ? c.d_ff_shared : c.d_ff; }

// Fields common to every FFN call; the caller sets n_shared / include_routed / weights /
// lists / outputs and then calls configure_ffn().
FfnArgs base_args(const moe_config &c, int T, void *ws, const WsLayout &L)
{
    FfnArgs a;
    memset(&a, 0, sizeof a);
    a.H = c.hidden;
    a.F = c.d_ff;
    a.Fs = c.n_shared ? c.d_ff_shared : c.d_ff;
    a.E = c.n_experts;
    a.K = c.top_k;
    a.T = T;
    a.err = at<int32_t>(ws, L.err);
    a.plan = at<FfnPlan>(ws, L.plan);
    a.xq.q = at<int8_t>(ws, L.xq);
    a.xq.scale = at<float>(ws, L.xscale);
    a.xq.csum = at<int32_t>(ws, L.xcsum);
    a.xq.q_ld = c.hidden;
    a.xq.c_ld = c.hidden / 32;
    a.h = at<float>(ws, L.h);
    a.gpart = at<float>(ws, L.hp);
    a.upart = a.gpart + L.hp_plane_floats;
    a.slice_gu = 1;
    a.hstride = fmax_of(c);
    a.hq.q = at<int8_t>(ws, L.hq);
    a.hq.scale = at<float>(ws, L.hscale);
    a.hq.csum = at<int32_t>(ws, L.hcsum);
    a.hq.q_ld = a.hstride;
    a.hq.c_ld = a.hstride / 32;
    return a;
}

// the bf16 copies of the codes feed the tensor-core path only
void configure_ffn(FfnArgs &a, void *ws, const WsLayout &L)
{
    ffn_configure(a);
    a.xq.bf16 = nullptr;
    a.hq.bf16 = a.tensor_dn ? at<__nv_bfloat16>(ws, L.hbf) : nullptr;
    a.x_bf16 = a.tensor ? at<__nv_bfloat16>(ws, L.xbf) : nullptr;
    a.h_bf16 = a.hq.bf16;
}

// gate/up -> quantise h -> down, each stage optionally bracketed by events
template <typename Scope>
cudaError_t run_ffn(const FfnArgs &a, int T, int ns, bool routed_rows, bool ev, cudaStream_t st)
{
    cudaError_t e;
    {
        Scope sc(ev, MOE_STAGE_GATE_UP, st, a.tensor ? 2 : 1);   // tensor path: + x gather
        e = launch_ffn_gate_up(a, st);
        sc.finish();
    }
    if (e == cudaSuccess) {
        Scope sc(ev, MOE_STAGE_QUANT_H, st);
        const int max_rows = T * ns + (routed_rows ? T * a.K : 0);
        e = launch_quant_h(a, T * ns, a.Fs, a.F, max_rows, st);
        sc.finish();
    }
    if (e == cudaSuccess) {
        Scope sc(ev, MOE_STAGE_DOWN, st);
        e = launch_ffn_down(a, st);
        sc.finish();
    }
    return e;
}

// ---- per-stage CUDA-event timing (MOE_FLAG_STAGE_EVENTS) ----
struct StageRec {
    int stage, launches;
    cudaEvent_t start, stop;
};
thread_local std::vector<StageRec> t_pending;
thread_local std::vector<cudaEvent_t> t_spare;
thread_local double t_ms[MOE_N_STAGES];
thread_local long long t_launches[MOE_N_STAGES];

cudaEvent_t take_event()
{
    if (!t_spare.empty()) {
        cudaEvent_t e = t_spare.back();
        t_spare.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

struct StageScope {
    // records a start event now and a stop event when finished (only when enabled)
    StageScope(bool on, int stage, cudaStream_t st, int launches = 1) : on_(on), st_(st)
    {
        rec_.stage = stage;
        rec_.launches = launches;
        rec_.start = rec_.stop = nullptr;
        if (on_ && (rec_.start = take_event()) != nullptr) cudaEventRecord(rec_.start, st_);
    }
    void finish()
    {
        if (!on_ || !rec_.start) return;
        rec_.stop = take_event();
        if (rec_.stop && cudaEventRecord(rec_.stop, st_) == cudaSuccess) t_pending.push_back(rec_);
        on_ = false;
    }
    bool on_;
    cudaStream_t st_;
    StageRec rec_;
};

// the shape fields of an FFN call, as the path queries see them (no buffers)
FfnArgs query_args(const moe_config &c, int T)
{
    FfnArgs a;
    memset(&a, 0, sizeof a);
    a.H = c.hidden;
    a.F = c.d_ff;
    a.n_shared = c.n_shared;
    a.Fs = c.n_shared ? c.d_ff_shared : c.d_ff;
    a.E = c.n_experts;
    a.K = c.top_k;
    a.T = T;
    a.hstride = fmax_of(c);
    a.xq.q_ld = c.hidden;
    a.hq.q_ld = a.hstride;
    return a;
}

}  // namespace

int set_error(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int require_device() { return check_device(); }

cudaError_t ensure_dynamic_smem(const void *kernel, size_t bytes)
{
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> set;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    size_t &have = set[{dev, kernel}];
    if (have >= bytes) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

int validate_route_args(const moe_config *cfg, const float *x, const float *w_router,
                        const float *bias, int T, const int32_t *ids, const float *w,
                        const int32_t *keff)
{
    int rc;
    if ((rc = check_config(cfg)) || (rc = check_tokens(T))) return rc;
    if (T == 0) return ok();
    REQUIRE_PTR(x, 16);
    REQUIRE_PTR(w_router, 16);
    REQUIRE_PTR(bias, 4);
    REQUIRE_PTR(ids, 4);
    REQUIRE_PTR(w, 4);
    REQUIRE_PTR(keff, 4);
    return MOE_OK;
}

int num_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    const int v = g_dev_sms[dev].load();
    return v > 0 ? v : 1;
}

WsLayout ws_layout(const moe_config &c, int T)
{
    WsLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += round_up(bytes > 0 ? bytes : 1, 256);
        return o;
    };
    const size_t TK = (size_t)T * c.top_k, E = c.n_experts, H = c.hidden;
    const size_t ns = c.n_shared ? 1 : 0;
    L.err = take(4);
    L.plan = take(sizeof(FfnPlan));
    L.ids = take(TK * 4);
    L.w = take(TK * 4);
    L.keff = take((size_t)T * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.tok = take(TK * 4);
    L.slot = take(TK * 4);
    L.uniq = take(E * 4);
    L.n_uniq = take(4);
    L.pair_of = take(TK * 4);
    L.logits = take(E * 4 * logits_rows(c, T));
    L.xq = take((size_t)T * H);
    L.xscale = take((size_t)T * 4);
    L.xcsum = take((size_t)T * (H / 32) * 4);
    const size_t rows = (size_t)T * ns + TK;
    const size_t fm = (size_t)fmax_of(c);
    // sliced rows (batches of at most kRouteClusterMaxT tokens): per-slice partial planes
    const int ts = T < kRouteClusterMaxT ? T : kRouteClusterMaxT;
    const size_t rows_s = (size_t)ts * ns + (size_t)ts * c.top_k;
    const size_t s_gu = (H + 32 * kSliceChunks - 1) / (32 * kSliceChunks);
    const size_t s_dn = (fm + 32 * kSliceChunks - 1) / (32 * kSliceChunks);
    L.h = take(rows * fm * 4);
    // gate/up planes: per-slice planes of the decode route, or one plane per matrix on the
    // tensor-core path (batches beyond kRouteClusterMaxT, and decode-route batches of narrow
    // layers: see ffn_use_tensor_cores)
    const bool narrow = c.hidden < 1024 || c.d_ff < 1024;
    const bool tensor_possible = T > kRouteClusterMaxT || (narrow && T >= kTensorMinTNarrow);
    const size_t hp_sliced = s_gu > 1 ? s_gu * rows_s * fm : 0;
    const size_t hp_tensor = tensor_possible ? rows * fm : 0;
    L.hp_plane_floats = hp_sliced > hp_tensor ? hp_sliced : hp_tensor;
    L.hp = take(2 * L.hp_plane_floats * 4);
    L.xbf = take(tensor_possible ? rows * H * 2 : 0);
    L.hbf = take(tensor_possible ? rows * fm * 2 : 0);
    L.hq = take(rows * fm);
    L.hscale = take(rows * 4);
    L.hcsum = take(rows * (fm / 32) * 4);
    L.y = take((rows > s_dn * rows_s ? rows : s_dn * rows_s) * H * 4);
    L.xn = take((size_t)T * H * 4);
    L.xs = take((size_t)T * H * 4);
    L.ys = take((size_t)T * H * 4);
    L.total = off;
    return L;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_config *cfg, int max_tokens)
{
    if (check_config(cfg) != MOE_OK) return 0;
    if (max_tokens < 0 || max_tokens > kMaxTokens) return 0;
    return ws_layout(*cfg, max_tokens).total;
}

const char *moe_last_error_string(void) { return g_err; }

int moe_route_lookahead(const moe_config *cfg, const float *x, const float *norm_w, float eps,
                        const float *w_router, const float *bias, int T, int32_t *ids, float *w,
                        int32_t *keff, void *workspace, size_t workspace_bytes, void *stream)
{
    int rc;
    if ((rc = validate_route_args(cfg, x, w_router, bias, T, ids, w, keff))) return rc;
    if (T == 0) return ok();
    REQUIRE_PTR(norm_w, 16);
    if (!(eps >= 0.0f) || std::isinf(eps)) return fail(MOE_ERR_ARG, "eps must be finite and >= 0 (got %g)", (double)eps);
    WsLayout L;
    if ((rc = check_ws(*cfg, T, workspace, workspace_bytes, &L)) || (rc = check_device())) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    float *xn = at<float>(workspace, L.xn);
    cudaError_t e = launch_rmsnorm(x, norm_w, eps, T, cfg->hidden, xn, st);
    if (e == cudaSuccess)
        e = launch_router(*cfg, xn, w_router, bias, T, at<float>(workspace, L.logits), ids, w, keff, st);
    if (e != cudaSuccess) return cuda_fail(e, "router look-ahead launch");
    return ok();
}

int moe_topk_hits(const moe_config *cfg, const int32_t *ids_pred, const int32_t *keff_pred,
                  const int32_t *ids_true, const int32_t *keff_true, int T, int32_t *hits,
                  void *stream)
{
    int rc;
    if ((rc = check_config(cfg)) || (rc = check_tokens(T))) return rc;
    if (T == 0) return ok();
    REQUIRE_PTR(ids_pred, 4);
    REQUIRE_PTR(keff_pred, 4);
    REQUIRE_PTR(ids_true, 4);
    REQUIRE_PTR(keff_true, 4);
    REQUIRE_PTR(hits, 4);
    if ((rc = check_device())) return rc;
    const cudaError_t e = launch_topk_hits(ids_pred, keff_pred, ids_true, keff_true, T, cfg->top_k,
                                           hits, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "top-k hit count launch");
    return ok();
}

int moe_quantize_int4_gs64(const float *w, int rows, int K, uint8_t *packed, float *scales,
                           void *stream)
{
    if (rows < 0) return fail(MOE_ERR_SHAPE, "rows must be >= 0 (got %d)", rows);
    if (K <= 0 || K % kGroup) return fail(MOE_ERR_SHAPE, "K must be a positive multiple of 64 (got %d)", K);
    if (rows == 0) return ok();
    REQUIRE_PTR(w, 16);
    REQUIRE_PTR(packed, 16);
    REQUIRE_PTR(scales, 16);
    int rc;
    if ((rc = check_device())) return rc;
    const cudaError_t e = launch_quantize_int4(w, rows, K, packed, scales, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "weight quantiser launch");
    return ok();
}

int moe_quantize_int3_g64(const float *w, int rows, int K, uint8_t *packed, float *scales,
                          void *stream)
{
    if (rows < 0) return fail(MOE_ERR_SHAPE, "rows must be >= 0 (got %d)", rows);
    if (K <= 0 || K % kGroup) return fail(MOE_ERR_SHAPE, "K must be a positive multiple of 64 (got %d)", K);
    if (rows == 0) return ok();
    REQUIRE_PTR(w, 16);
    REQUIRE_PTR(packed, 1);
    REQUIRE_PTR(scales, 4);
    int rc;
    if ((rc = check_device())) return rc;
    const cudaError_t e = launch_quantize_int3(w, rows, K, packed, scales, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "int3 weight quantiser launch");
    return ok();
}

int moe_selftest_wait_timeout(void *workspace, size_t workspace_bytes, int polls, void *stream)
{
    if (!workspace) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(workspace, 256)) return fail(MOE_ERR_ALIGN, "workspace is not 256-byte aligned");
    if (workspace_bytes < 256) return fail(MOE_ERR_WORKSPACE, "workspace is smaller than 256 bytes");
    if (polls < 1 || polls > (1 << 24)) return fail(MOE_ERR_ARG, "polls must be in [1, 2^24] (got %d)", polls);
    int rc;
    if ((rc = check_device())) return rc;
    const cudaError_t e = launch_selftest_wait(static_cast<int32_t *>(workspace), polls, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return ok();
}

int moe_ffn_uses_tensor_cores(const moe_config *cfg, int T)
{
    if (check_config(cfg) != MOE_OK || T < 0) return -1;
    return ffn_use_tensor_cores(query_args(*cfg, T)) ? 1 : 0;
}

// the paths ffn_configure picks (the row GEMV's shape conditions hold for the operands'
// 16-byte alignment of every call that passes validation: weights are checked, the workspace
// regions are aligned)
static int ffn_path_of(const moe_config *cfg, int T, bool down)
{
    const int tc = moe_ffn_uses_tensor_cores(cfg, T);
    if (tc < 0) return tc;
    const FfnArgs a = query_args(*cfg, T);
    if (tc) return down || !ffn_split_paths(a) ? MOE_FFN_TENSOR : MOE_FFN_ROW_GEMV;
    return T >= kRowGemvMinT && ffn_rows_supported(a) ? MOE_FFN_ROW_GEMV : MOE_FFN_WARP_GEMV;
}

int moe_ffn_path(const moe_config *cfg, int T) { return ffn_path_of(cfg, T, false); }

int moe_ffn_path_down(const moe_config *cfg, int T) { return ffn_path_of(cfg, T, true); }

int moe_route(const moe_config *cfg, const float *x, const float *w_router, const float *bias,
              int T, int32_t *ids, float *w, int32_t *keff, void *workspace,
              size_t workspace_bytes, void *stream)
{
    int rc;
    if ((rc = check_config(cfg)) || (rc = check_tokens(T))) return rc;
    if (T == 0) return ok();
    REQUIRE_PTR(x, 16);
    REQUIRE_PTR(w_router, 16);
    REQUIRE_PTR(bias, 4);
    REQUIRE_PTR(ids, 4);
    REQUIRE_PTR(w, 4);
    REQUIRE_PTR(keff, 4);
    WsLayout L;
    if ((rc = check_ws(*cfg, T, workspace, workspace_bytes, &L)) || (rc = check_device())) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = launch_router(*cfg, x, w_router, bias, T, at<float>(workspace, L.logits), ids,
                                  w, keff, st);
    if (e != cudaSuccess) return cuda_fail(e, "router launch");
    return ok();
}

int moe_permute(const moe_config *cfg, const int32_t *ids, const int32_t *keff, int T,
                int32_t *counts, int32_t *offsets, int32_t *tok, int32_t *slot, int32_t *uniq,
                int32_t *n_uniq, void *workspace, size_t workspace_bytes, void *stream)
{
    int rc;
    if ((rc = check_config(cfg)) || (rc = check_tokens(T))) return rc;
    if (T > 0) {
        REQUIRE_PTR(ids, 4);
        REQUIRE_PTR(keff, 4);
        REQUIRE_PTR(tok, 4);
        REQUIRE_PTR(slot, 4);
    }
    REQUIRE_PTR(counts, 4);
    REQUIRE_PTR(offsets, 4);
    REQUIRE_PTR(uniq, 4);
    REQUIRE_PTR(n_uniq, 4);
    WsLayout L;
    if ((rc = check_ws(*cfg, T, workspace, workspace_bytes, &L)) || (rc = check_device())) return rc;
    const PermuteOut o{counts, offsets, tok, slot, uniq, n_uniq, at<int32_t>(workspace, L.err),
                       nullptr};
    cudaError_t e = launch_permute(*cfg, ids, keff, T, o, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "permute launch");
    return ok();
}

int moe_expert_ffn(const moe_config *cfg, const float *x, int T, const moe_expert_weights *routed,
                   const int32_t *offsets, const int32_t *tok, const int32_t *uniq,
                   const int32_t *n_uniq, float *y_pairs, const moe_ffn_probe *probe,
                   void *workspace, size_t workspace_bytes, void *stream)
{
    int rc;
    if ((rc = check_config(cfg)) || (rc = check_tokens(T))) return rc;
    if (T == 0) return ok();
    if ((rc = check_tile_count(*cfg, T))) return rc;
    REQUIRE_PTR(x, 16);
    if ((rc = check_weights(routed, "routed"))) return rc;
    REQUIRE_PTR(offsets, 4);
    REQUIRE_PTR(tok, 4);
    REQUIRE_PTR(uniq, 4);
    REQUIRE_PTR(n_uniq, 4);
    REQUIRE_PTR(y_pairs, 16);
    WsLayout L;
    if ((rc = check_ws(*cfg, T, workspace, workspace_bytes, &L)) || (rc = check_device())) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    FfnArgs a = base_args(*cfg, T, workspace, L);
    a.n_shared = 0;
    a.include_routed = 1;
    a.routed = *routed;
    a.offsets = offsets;
    a.tok = tok;
    a.y = y_pairs;
    a.routed_rowbase = 0;
    a.plane_rows = T * cfg->top_k;
    a.slice_dn = 0;   // y_pairs holds one plane
    if (probe) a.probe = *probe;
    configure_ffn(a, workspace, L);
    cudaError_t e = launch_quant_rows(x, T, cfg->hidden, cfg->hidden, a.xq, st);
    if (e == cudaSuccess) e = launch_plan(a, uniq, n_uniq, at<FfnPlan>(workspace, L.plan), st);
    if (e == cudaSuccess) e = run_ffn<StageScope>(a, T, 0, true, false, st);
    if (e != cudaSuccess) return cuda_fail(e, "expert FFN launch");
    return ok();
}

int moe_combine(const moe_config *cfg, const float *y_pairs, const int32_t *ids,
                const int32_t *keff, const float *w, const int32_t *offsets, const int32_t *tok,
                int T, const float *x, const moe_expert_weights *shared, float *y,
                void *workspace, size_t workspace_bytes, void *stream)
{
    int rc;
    if ((rc = check_config(cfg)) || (rc = check_tokens(T))) return rc;
    if (T == 0) return ok();
    if ((rc = check_tile_count(*cfg, T))) return rc;
    REQUIRE_PTR(y_pairs, 16);
    REQUIRE_PTR(ids, 4);
    REQUIRE_PTR(keff, 4);
    REQUIRE_PTR(w, 4);
    REQUIRE_PTR(offsets, 4);
    REQUIRE_PTR(tok, 4);
    REQUIRE_PTR(y, 16);
    const bool use_shared = shared != nullptr && cfg->n_shared == 1;
    if (use_shared) {
        REQUIRE_PTR(x, 16);
        if ((rc = check_weights(shared, "shared"))) return rc;
    }
    WsLayout L;
    if ((rc = check_ws(*cfg, T, workspace, workspace_bytes, &L)) || (rc = check_device())) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    const float *ys = nullptr;
    int s_sh = 1;
    int64_t plane = 0;
    if (use_shared) {
        FfnArgs a = base_args(*cfg, T, workspace, L);
        a.n_shared = 1;
        a.include_routed = 0;
        a.shared = *shared;
        a.y = at<float>(workspace, L.y);
        a.routed_rowbase = T;
        a.plane_rows = T;
        a.slice_dn = 1;
        configure_ffn(a, workspace, L);
        a.shared_early = 1;   // the plan kernel runs between the x quantisation and gate/up
        e = launch_quant_rows(x, T, cfg->hidden, cfg->hidden, a.xq, st);
        if (e == cudaSuccess) e = launch_plan(a, nullptr, nullptr, at<FfnPlan>(workspace, L.plan), st);
        if (e == cudaSuccess) e = run_ffn<StageScope>(a, T, 1, false, false, st);
        ys = a.y;
        s_sh = a.slice_dn ? a.geo_dn[1].S : 1;
        plane = (int64_t)a.plane_rows * cfg->hidden;
    }
    if (e == cudaSuccess)
        e = launch_combine(*cfg, y_pairs, cfg->hidden, ys, ids, keff, w, offsets, tok, nullptr, 1,
                           s_sh, plane, T, y, st);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return ok();
}

int moe_check_errors(void *workspace, size_t workspace_bytes, void *stream)
{
    if (!workspace) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(workspace, 256)) return fail(MOE_ERR_ALIGN, "workspace is not 256-byte aligned");
    if (workspace_bytes < 256) return fail(MOE_ERR_WORKSPACE, "workspace is smaller than 256 bytes");
    int rc;
    if ((rc = check_device())) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t flag = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemcpy(&flag, workspace, 4, cudaMemcpyDeviceToHost);
    // the error word and the route tail's ticket (a launch stopped midway may leave it set)
    if (e == cudaSuccess && flag) e = cudaMemsetAsync(workspace, 0, 256, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "error check");
    if (flag & kErrBadExpertId) return fail(MOE_ERR_DEVICE, "an expert id outside [0, n_experts) was skipped");
    if (flag & kErrBadKeff) return fail(MOE_ERR_DEVICE, "a keff outside [0, top_k] was clamped");
    if (flag & kErrTimeout) return fail(MOE_ERR_TIMEOUT, "a bounded device-side wait gave up; the kernel stopped early and its outputs are incomplete");
    if (flag) return fail(MOE_ERR_DEVICE, "device error word 0x%x", flag);
    return ok();
}

int moe_layer_forward(const moe_config *cfg, const float *x, int T, const float *w_router,
                      const float *bias, const moe_expert_weights *routed,
                      const moe_expert_weights *shared, float *y, const moe_routing *routing,
                      void *workspace, size_t workspace_bytes, int flags, void *stream)
{
    int rc;
    if ((rc = check_config(cfg)) || (rc = check_tokens(T))) return rc;
    if (flags & ~(MOE_FLAG_SYNC_CHECK | MOE_FLAG_STAGE_EVENTS)) return fail(MOE_ERR_ARG, "unknown flags 0x%x", flags);
    if (T == 0) return ok();
    if ((rc = check_tile_count(*cfg, T))) return rc;
    REQUIRE_PTR(x, 16);
    REQUIRE_PTR(w_router, 16);
    REQUIRE_PTR(bias, 4);
    REQUIRE_PTR(y, 16);
    if ((rc = check_weights(routed, "routed"))) return rc;
    if (cfg->n_shared && (rc = check_weights(shared, "shared"))) return rc;
    WsLayout L;
    if ((rc = check_ws(*cfg, T, workspace, workspace_bytes, &L)) || (rc = check_device())) return rc;
    int32_t *ids = at<int32_t>(workspace, L.ids);
    float *w = at<float>(workspace, L.w);
    int32_t *keff = at<int32_t>(workspace, L.keff);
    if (routing) {
        if (routing->ids) { REQUIRE_PTR(routing->ids, 4); ids = routing->ids; }
        if (routing->w) { REQUIRE_PTR(routing->w, 4); w = routing->w; }
        if (routing->keff) { REQUIRE_PTR(routing->keff, 4); keff = routing->keff; }
    }
    cudaStream_t st = (cudaStream_t)stream;
    const int ns = cfg->n_shared;
    int32_t *offsets = at<int32_t>(workspace, L.offsets);
    int32_t *tok = at<int32_t>(workspace, L.tok);
    int32_t *uniq = at<int32_t>(workspace, L.uniq);
    int32_t *n_uniq = at<int32_t>(workspace, L.n_uniq);

    FfnArgs a = base_args(*cfg, T, workspace, L);
    a.n_shared = ns;
    a.include_routed = 1;
    a.routed = *routed;
    if (ns) a.shared = *shared;
    a.offsets = offsets;
    a.tok = tok;
    a.y = at<float>(workspace, L.y);
    a.routed_rowbase = T * ns;
    a.plane_rows = T * ns + T * cfg->top_k;
    a.slice_dn = 1;
    configure_ffn(a, workspace, L);
    // decode route: the router kernel writes the x codes and the route tail runs between it
    // and gate/up (the prefill route quantises x right before gate/up)
    a.shared_early = T <= kRouteClusterMaxT ? 1 : 0;

    const bool ev = (flags & MOE_FLAG_STAGE_EVENTS) != 0;
    float *logits = at<float>(workspace, L.logits);
    const PermuteOut perm{at<int32_t>(workspace, L.counts), offsets, tok,
                          at<int32_t>(workspace, L.slot), uniq, n_uniq,
                          at<int32_t>(workspace, L.err), at<int32_t>(workspace, L.pair_of)};
    cudaError_t e;
    int splits = 1;
    if (T <= kRouteClusterMaxT) {
        // decode route: router + x quantisation, then selection + batch-union + plan
        {
            StageScope sc(ev, MOE_STAGE_ROUTER, st);
            e = launch_router_logits(*cfg, x, w_router, T, logits, &a.xq, &splits, st);
            sc.finish();
        }
        if (e == cudaSuccess) {
            StageScope sc(ev, MOE_STAGE_SELECT, st);
            e = launch_route_tail(*cfg, logits, bias, T, ids, w, keff, &perm, &a, st);
            sc.finish();
        }
    } else {
        {
            StageScope sc(ev, MOE_STAGE_ROUTER, st);
            e = launch_router_logits(*cfg, x, w_router, T, logits, nullptr, &splits, st);
            sc.finish();
        }
        if (e == cudaSuccess) {
            StageScope sc(ev, MOE_STAGE_SELECT, st);
            e = launch_router_select(*cfg, logits, splits, bias, T, ids, w, keff, st);
            sc.finish();
        }
        if (e == cudaSuccess) {
            StageScope sc(ev, MOE_STAGE_PERMUTE, st);
            e = launch_permute(*cfg, ids, keff, T, perm, st);
            sc.finish();
        }
        if (e == cudaSuccess) {
            StageScope sc(ev, MOE_STAGE_PLAN, st);
            e = launch_plan(a, uniq, n_uniq, at<FfnPlan>(workspace, L.plan), st);
            sc.finish();
        }
        if (e == cudaSuccess) {
            StageScope sc(ev, MOE_STAGE_QUANT, st);
            e = launch_quant_rows(x, T, cfg->hidden, cfg->hidden, a.xq, st);
            sc.finish();
        }
    }
    if (e == cudaSuccess) e = run_ffn<StageScope>(a, T, ns, true, ev, st);
    if (e == cudaSuccess) {
        StageScope sc(ev, MOE_STAGE_COMBINE, st);
        e = launch_combine(*cfg, a.y + (size_t)T * ns * cfg->hidden, cfg->hidden,
                           ns ? a.y : nullptr, ids, keff, w, offsets, tok, perm.pair_of,
                           a.slice_dn ? a.geo_dn[0].S : 1, a.slice_dn ? a.geo_dn[1].S : 1,
                           (int64_t)a.plane_rows * cfg->hidden, T, y, st);
        sc.finish();
    }
    if (e != cudaSuccess) return cuda_fail(e, "layer launch");
    if (flags & MOE_FLAG_SYNC_CHECK) return moe_check_errors(workspace, workspace_bytes, stream);
    return ok();
}

int moe_layer_forward_host(const moe_config *cfg, const float *x_host, int T,
                           const float *w_router, const float *bias,
                           const moe_expert_weights *routed, const moe_expert_weights *shared,
                           float *y_host, const moe_routing *routing, void *workspace,
                           size_t workspace_bytes, int flags, void *stream)
{
    int rc;
    if ((rc = check_config(cfg)) || (rc = check_tokens(T))) return rc;
    if (T == 0) return ok();
    if (!x_host) return fail(MOE_ERR_ARG, "x_host is NULL");
    if (!y_host) return fail(MOE_ERR_ARG, "y_host is NULL");
    WsLayout L;
    if ((rc = check_ws(*cfg, T, workspace, workspace_bytes, &L)) || (rc = check_device())) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    float *xd = at<float>(workspace, L.xs), *yd = at<float>(workspace, L.ys);
    const size_t bytes = (size_t)T * cfg->hidden * sizeof(float);
    cudaError_t e = cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "copy of x to the device");
    if ((rc = moe_layer_forward(cfg, xd, T, w_router, bias, routed, shared, yd, routing, workspace,
                                workspace_bytes, flags, stream)))
        return rc;
    e = cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "copy of y to the host");
    return ok();
}

int moe_stage_times(double *ms, long long *launches, int reset)
{
    for (const StageRec &r : t_pending) {
        float v = 0.0f;
        if (cudaEventSynchronize(r.stop) == cudaSuccess &&
            cudaEventElapsedTime(&v, r.start, r.stop) == cudaSuccess) {
            t_ms[r.stage] += v;
            t_launches[r.stage] += r.launches;
        } else {
            cudaGetLastError();
        }
        t_spare.push_back(r.start);
        t_spare.push_back(r.stop);
    }
    t_pending.clear();
    for (int i = 0; i < MOE_N_STAGES; ++i) {
        if (ms) ms[i] = t_ms[i];
        if (launches) launches[i] = t_launches[i];
        if (reset) {
            t_ms[i] = 0.0;
            t_launches[i] = 0;
        }
    }
    return ok();
}

}  // extern "C"
