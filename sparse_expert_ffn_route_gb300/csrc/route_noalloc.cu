// route_noalloc.cu -- moe_route_noalloc: the router without a caller-provided workspace.
//
// The router's only scratch is the buffer of partial logits [S][T][E] (fp32).  Here it
// lives in a fixed array defined by this library in device memory, so the caller passes
// inputs and outputs only and nothing is allocated by the call.  Meant for callers that
// cannot allocate device memory themselves: e.g. a plugin inside a host engine that owns
// every device allocation and forbids its extensions to call cudaMalloc, or a decode loop
// that cannot afford the device synchronisation a cudaMalloc/cudaFree may cause.
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {

// 2,097,152 floats = 8 MiB of router scratch; every GPU that loads libmoe.so holds it
// until the process exits.
static __device__ __align__(256) float g_route_scratch[kRouteScratchFloats];

std::mutex g_setup_mu;
// device address of g_route_scratch per device, and the context it was looked up in (a
// device reset or a primary-context teardown reloads the module, so the address is looked up
// again whenever the current context differs from the one recorded)
float *g_scratch_dev[64];
void *g_scratch_ctx[64];

// the current driver context, through the runtime's driver entry point (no libcuda link)
void *current_context()
{
    using GetCtx = int (*)(void **);
    static std::once_flag once;
    static GetCtx fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<GetCtx>(p);
        else
            cudaGetLastError();
    });
    void *ctx = nullptr;
    if (fn == nullptr || fn(&ctx) != 0) return nullptr;
    return ctx;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_route_noalloc(const moe_config *cfg, const float *x, const float *w_router,
                                 const float *bias, int T, int32_t *ids, float *w,
                                 int32_t *keff, void *stream)
{
    int rc = validate_route_args(cfg, x, w_router, bias, T, ids, w, keff);
    if (rc != MOE_OK || T == 0) return rc;
    const size_t need = (size_t)router_splits(*cfg, T) * (size_t)T * (size_t)cfg->n_experts;
    if (need > kRouteScratchFloats)
        return set_error(MOE_ERR_SHAPE,
                         "moe_route_noalloc: T=%d with %d experts needs %zu floats of router "
                         "scratch; the built-in array holds %zu (use moe_route with a workspace)",
                         T, cfg->n_experts, need, kRouteScratchFloats);
    if ((rc = require_device()) != MOE_OK) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return set_error(MOE_ERR_CUDA, "moe_route_noalloc: no current CUDA device");
    }
    float *scratch = nullptr;
    {
        // first call on this device (or in a new context of it): look up the array's device
        // address with the device current
        void *ctx = current_context();
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_scratch_dev[dev] || g_scratch_ctx[dev] != ctx) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
            if (e != cudaSuccess || p == nullptr) {
                cudaGetLastError();   // leave no sticky error behind for unrelated callers
                g_scratch_dev[dev] = nullptr;
                return set_error(MOE_ERR_CUDA, "moe_route_noalloc: cudaGetSymbolAddress failed: %s",
                                 cudaGetErrorString(e));
            }
            g_scratch_dev[dev] = static_cast<float *>(p);
            g_scratch_ctx[dev] = ctx;
        }
        scratch = g_scratch_dev[dev];
    }
    const cudaError_t e = launch_router(*cfg, x, w_router, bias, T, scratch, ids, w, keff,
                                        (cudaStream_t)stream);
    if (e != cudaSuccess)
        return set_error(MOE_ERR_CUDA, "moe_route_noalloc: router launch: %s", cudaGetErrorString(e));
    return set_error(MOE_OK, "");
}
