"""GB300 (sm_103a) sparse MoE FFN layer: router, batch-union, int4 x int8 expert FFN, combine.

The compute lives in ``libmoe.so`` (CUDA kernels behind the C ABI of
``include/moe.h``); this package is its thin ctypes binding.  Build the library
with ``python -m sparse_expert_ffn_route_gb300.build``.
"""
from .binding import (EXPORTS, LIBRARY_PATH, MOE_ERR_ALIGN, MOE_ERR_ARG, MOE_ERR_CUDA,  # noqa: F401
                      MOE_ERR_DEVICE, MOE_ERR_SHAPE, MOE_ERR_TIMEOUT, MOE_ERR_UNSUPPORTED,
                      MOE_ERR_WORKSPACE, MOE_FFN_ROW_GEMV, MOE_FFN_TENSOR, MOE_FFN_WARP_GEMV,
                      MOE_FLAG_STAGE_EVENTS, MOE_FLAG_SYNC_CHECK, MOE_OK, STAGES, ExpertWeights, FfnProbe,
                      MoeConfig, MoeError, Routing, alloc_workspace, last_error, load_library,
                      moe_check_errors, moe_combine, moe_expert_ffn, moe_layer_forward,
                      moe_permute, moe_route, moe_route_noalloc, moe_stage_times,
                      moe_workspace_size, moe_ffn_uses_tensor_cores,
                      moe_route_lookahead, moe_topk_hits, moe_quantize_int4_gs64, moe_quantize_int3_g64,
                      moe_selftest_wait_timeout, moe_layer_forward_host, moe_ffn_path,
                      moe_ffn_path_down)
