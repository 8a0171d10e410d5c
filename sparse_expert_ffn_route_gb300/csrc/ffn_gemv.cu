// ffn_gemv.cu -- host side of the grouped expert FFN: chooses the kernel (tcgen05 grouped
// GEMM, row GEMV or warp GEMV), the warp GEMV's variant (chunks per lane, tokens per chunk,
// rows in flight) and the task geometry, and launches.
#include "ffn_kernels.cuh"
#include "launch.cuh"

#include <cmath>
#include <map>
#include <mutex>

namespace moe {

namespace {

using ffn_impl::FfnKernel;
using ffn_impl::Variant;

Variant variant(bool gu, int nc, int tc)
{
    switch ((nc + 1) / 2) {
    case 1: return gu ? ffn_variant_gu_12(nc, tc) : ffn_variant_dn_12(nc, tc);
    case 2: return gu ? ffn_variant_gu_34(nc, tc) : ffn_variant_dn_34(nc, tc);
    case 3: return gu ? ffn_variant_gu_56(nc, tc) : ffn_variant_dn_56(nc, tc);
    case 4: return gu ? ffn_variant_gu_78(nc, tc) : ffn_variant_dn_78(nc, tc);
    }
    return {};
}

struct Chosen {
    FfnKernel k;
    int ru;
    size_t smem;
};

Chosen choose(bool gu, int nc, int tc, bool probe)
{
    const Variant v = variant(gu, nc, tc);
    return {probe ? v.kprobe : v.k, v.ru, v.smem};
}

int max_nc(const Geo (&g)[2], bool both) { return both && g[1].nc > g[0].nc ? g[1].nc : g[0].nc; }

cudaError_t launch(Chosen c, const FfnArgs &a, cudaStream_t st)
{
    if (!c.k) return cudaErrorInvalidConfiguration;
    // one CTA of 8 warps per SM (the rings take most of shared memory)
    return launch_kernel(c.k, dim3(num_sms()), dim3(kFfnThreads), c.smem, st, 1, a);
}

bool probes_gu(const FfnArgs &a) { return a.probe.acc_gate != nullptr || a.probe.acc_up != nullptr; }
bool probes_dn(const FfnArgs &a) { return a.probe.acc_down != nullptr; }

// tokens per chunk (one pass over the expert's weights per chunk): enough for the tokens an
// expert is expected to receive, as far as their activations fit the registers
// (ffn_impl::tc_max) -- the routed experts' expected share T*K/U, U the expected number of
// distinct experts under uniform routing, and with a shared expert its T tokens.
int pick_tc(int nc, int T, int K, int E, bool shared)
{
    const double U = E * (1.0 - pow(1.0 - (double)K / E, (double)T));
    double want = U > 0.0 ? (double)T * K / U : 1.0;
    if (shared && T > want) want = T;
    int tc = 1;
    while (tc < ffn_impl::tc_max(nc) && tc < want) tc *= 2;
    return tc;
}

}  // namespace

bool ffn_use_tensor_cores(const FfnArgs &a)
{
    if (!ffn_tc_supported(a)) return false;
    // On narrow matrices the row GEMV's tasks are one or two stages long and its dp4a work
    // grows with every token, so decode-route batches of kTensorMinTNarrow tokens or more
    // take the tensor path too (A3B-style layer, T = 64, top-p 0.7: 27 unique experts of
    // about 12 tokens each).
    const bool narrow = a.H < 1024 || a.F < 1024;
    if (a.T <= kRouteClusterMaxT) return narrow && a.T >= kTensorMinTNarrow;
    // Measured on GB300 (gate/up + down): a tensor-core tile pays about the same per 64-input
    // group whatever its width, while the row GEMV streams an expert's weights once per 8 of
    // its tokens.  On wide matrices the row GEMV is faster below about 10 tokens per routed
    // expert (GLM T=256, 8 per expert: 2.35 vs 3.11 ms; wide layer T=256: 2.78 vs 4.46 ms),
    // level near 10 (wide layer T=512: 5.18 vs 5.08 ms) and slower above (GLM T=512: 4.39 vs
    // 3.46 ms).  On narrow ones (hidden or d_ff under 1024) its tasks are too short and the
    // tensor path wins from the first batch past the decode route (A3B T=128: 0.092 vs 0.143 ms).
    if (narrow) return true;
    const double U = a.E * (1.0 - pow(1.0 - (double)a.K / a.E, (double)a.T));
    return U > 0.0 && (double)a.T * a.K / U >= 10.0;
}

// Where the tensor path takes a layer, it runs down only in two cases.  On a narrow layer in
// the decode route: gate/up, whose reduction over H is long, is faster on the row GEMV, while
// down's short reduction over d_ff makes one-stage row-GEMV tasks (A3B-style layer, T = 64:
// gate/up 38.7 µs on the row GEMV against 48.6 on the tensor path, down 41.2 against 31.1).
// Past the decode route, on wide layers, down crosses to the tensor path at fewer tokens
// per expert than gate/up: between 10 and kSplitMaxPerExpert expected tokens per routed
// expert gate/up stays on the row GEMV (wide layer, T = 512, 10.7 per expert: gate/up 2.86 ms
// on the row GEMV against 3.32 on the tensor path, down 2.33 against 1.76).
constexpr double kSplitMaxPerExpert = 14.0;

bool ffn_split_paths(const FfnArgs &a)
{
    if (a.T < kRowGemvMinT || !ffn_rows_supported(a)) return false;
    const bool narrow = a.H < 1024 || a.F < 1024;
    if (a.T <= kRouteClusterMaxT)
        return a.H >= 1024 && a.F < 1024 && (!a.n_shared || a.Fs < 1024);
    if (narrow) return false;
    const double U = a.E * (1.0 - pow(1.0 - (double)a.K / a.E, (double)a.T));
    return U > 0.0 && (double)a.T * a.K / U < kSplitMaxPerExpert;
}

void ffn_configure(FfnArgs &a)
{
    const bool sh = a.n_shared != 0;
    const bool small = a.T <= kRouteClusterMaxT;
    // the tensor-core grouped GEMM (ffn_tc.cu) where ffn_use_tensor_cores takes it (down
    // only, when ffn_split_paths says so), the row GEMV where its shapes allow and the batch
    // has kRowGemvMinT tokens or more, else the warp GEMV below
    const bool tc = ffn_use_tensor_cores(a);
    const bool split = tc && ffn_split_paths(a);
    const bool rows = !tc && a.T >= kRowGemvMinT && ffn_rows_supported(a);
    a.tensor = tc && !split ? 1 : 0;
    a.tensor_dn = tc ? 1 : 0;
    a.rows = rows || split ? 1 : 0;
    a.rows_dn = rows ? 1 : 0;
    if (a.tensor || a.rows) {   // gate/up
        a.slice_gu = 0;
        a.tc_gu = a.tensor ? 128 : kRowTok;
        a.geo_gu[0] = a.tensor ? make_tc_geo(a.H, a.F, 2) : make_rows_geo(a.H, a.F, kRowTaskGateUp);
        a.geo_gu[1] = a.tensor ? make_tc_geo(a.H, a.Fs, 2) : make_rows_geo(a.H, a.Fs, kRowTaskGateUp);
    }
    if (a.tensor_dn || a.rows_dn) {   // down
        a.slice_dn = 0;
        a.tc_dn = a.tensor_dn ? 128 : kRowTok;
        a.geo_dn[0] = a.tensor_dn ? make_tc_geo(a.F, a.H, 1) : make_rows_geo(a.F, a.H, kRowTaskDown);
        a.geo_dn[1] = a.tensor_dn ? make_tc_geo(a.Fs, a.H, 1) : make_rows_geo(a.Fs, a.H, kRowTaskDown);
    }
    if (a.tensor || a.rows) return;   // both projections are set (the split pairs row GEMV + tensor)
    const int fmax = sh && a.Fs > a.F ? a.Fs : a.F;
    const bool slice = small && a.T >= kSliceMinT;
    const bool sgu = slice && a.slice_gu && a.H > 32 * kSliceChunks;
    const bool sdn = slice && a.slice_dn && fmax > 32 * kSliceChunks &&
                     fmax <= 32 * kSliceChunks * kMaxCombinePlanes;
    a.slice_gu = sgu ? 1 : 0;
    a.slice_dn = sdn ? 1 : 0;
    // gate/up: both matrices reduce over H
    const int ncg = make_geo(a.H, a.F, 1, false, sgu).nc;
    a.tc_gu = pick_tc(ncg, a.T, a.K, a.E, sh);
    const int ru_gu = choose(true, ncg, a.tc_gu, probes_gu(a)).ru;
    a.geo_gu[0] = make_geo(a.H, a.F, ru_gu > 0 ? ru_gu : 1, ncg > 1, sgu);
    a.geo_gu[1] = make_geo(a.H, a.Fs, ru_gu > 0 ? ru_gu : 1, ncg > 1, sgu);
    // down: the routed matrix reduces over F, the shared one over Fs
    const int nd0 = make_geo(a.F, a.H, 1, false, sdn).nc, nd1 = make_geo(a.Fs, a.H, 1, false, sdn).nc;
    const int ncd = sh && nd1 > nd0 ? nd1 : nd0;
    a.tc_dn = pick_tc(ncd, a.T, a.K, a.E, sh);
    const int ru_dn = choose(false, ncd, a.tc_dn, probes_dn(a)).ru;
    a.geo_dn[0] = make_geo(a.F, a.H, ru_dn > 0 ? ru_dn : 1, ncd > 1, sdn);
    a.geo_dn[1] = make_geo(a.Fs, a.H, ru_dn > 0 ? ru_dn : 1, ncd > 1, sdn);
}

cudaError_t launch_ffn_gate_up(const FfnArgs &a, cudaStream_t st)
{
    if (a.tensor) return launch_ffn_tc(true, a, st);
    if (a.rows) return launch_ffn_rows(true, a, st);
    return launch(choose(true, max_nc(a.geo_gu, a.n_shared != 0), a.tc_gu, probes_gu(a)), a, st);
}

cudaError_t launch_ffn_down(const FfnArgs &a, cudaStream_t st)
{
    if (a.tensor_dn) return launch_ffn_tc(false, a, st);
    if (a.rows_dn) return launch_ffn_rows(false, a, st);
    return launch(choose(false, max_nc(a.geo_dn, a.n_shared != 0), a.tc_dn, probes_dn(a)), a, st);
}

}  // namespace moe
