// ffn_gemv.cu -- host side of the grouped expert FFN: chooses the kernel variant (chunks
// per lane, tokens per chunk, rows in flight) and the task geometry, and launches.
#include "ffn_kernels.cuh"

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

// true when ptxas kept the kernel in registers (no local-memory spills)
bool spill_free(FfnKernel k)
{
    static std::mutex mu;
    static std::map<FfnKernel, bool> known;
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(k);
    if (it != known.end()) return it->second;
    cudaFuncAttributes at{};
    const bool ok = cudaFuncGetAttributes(&at, k) == cudaSuccess && at.localSizeBytes == 0;
    known[k] = ok;
    return ok;
}

struct Chosen {
    FfnKernel k;
    int ru;
};

Chosen choose(bool gu, int nc, int tc, bool probe)
{
    const Variant v = variant(gu, nc, tc);
    if (!v.k1) return {nullptr, 0};
    if (probe) return {v.kprobe, v.ru1};
    if (spill_free(v.k2)) return {v.k2, v.ru2};
    return {v.k1, v.ru1};
}

int max_nc(const Geo (&g)[2], bool both) { return both && g[1].nc > g[0].nc ? g[1].nc : g[0].nc; }

cudaError_t launch(Chosen c, const FfnArgs &a, cudaStream_t st)
{
    if (!c.k) return cudaErrorInvalidConfiguration;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, c.k, kFfnThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    c.k<<<per_sm * num_sms(), kFfnThreads, 0, st>>>(a);
    return cudaGetLastError();
}

bool probes_gu(const FfnArgs &a) { return a.probe.acc_gate != nullptr || a.probe.acc_up != nullptr; }
bool probes_dn(const FfnArgs &a) { return a.probe.acc_down != nullptr; }

// tokens per chunk (one pass over the expert's weights per chunk): 1 while experts see
// about one token each, more once the batch gives each expert several, as far as the
// activations of a chunk fit 64 registers per lane (16 warps per SM)
int pick_tc(int nc, int T, int K, int E)
{
    const double tpe = (double)T * K / E;
    int tc = 1;
    while (tc < 8 && tc < tpe && nc * 8 * (tc * 2) <= 64) tc *= 2;
    return tc;
}

}  // namespace

void ffn_configure(FfnArgs &a)
{
    const bool sh = a.n_shared != 0;
    // gate/up: both matrices reduce over H
    const int ncg = make_geo(a.H, a.F, 1, false).nc;
    a.tc_gu = pick_tc(ncg, a.T, a.K, a.E);
    const int ru_gu = choose(true, ncg, a.tc_gu, probes_gu(a)).ru;
    a.geo_gu[0] = make_geo(a.H, a.F, ru_gu > 0 ? ru_gu : 1, ncg > 1);
    a.geo_gu[1] = make_geo(a.H, a.Fs, ru_gu > 0 ? ru_gu : 1, ncg > 1);
    // down: the routed matrix reduces over F, the shared one over Fs
    const int nd0 = make_geo(a.F, a.H, 1, false).nc, nd1 = make_geo(a.Fs, a.H, 1, false).nc;
    const int ncd = sh && nd1 > nd0 ? nd1 : nd0;
    a.tc_dn = pick_tc(ncd, a.T, a.K, a.E);
    const int ru_dn = choose(false, ncd, a.tc_dn, probes_dn(a)).ru;
    a.geo_dn[0] = make_geo(a.F, a.H, ru_dn > 0 ? ru_dn : 1, ncd > 1);
    a.geo_dn[1] = make_geo(a.Fs, a.H, ru_dn > 0 ? ru_dn : 1, ncd > 1);
}

cudaError_t launch_ffn_gate_up(const FfnArgs &a, cudaStream_t st)
{
    return launch(choose(true, max_nc(a.geo_gu, a.n_shared != 0), a.tc_gu, probes_gu(a)), a, st);
}

cudaError_t launch_ffn_down(const FfnArgs &a, cudaStream_t st)
{
    return launch(choose(false, max_nc(a.geo_dn, a.n_shared != 0), a.tc_dn, probes_dn(a)), a, st);
}

}  // namespace moe
