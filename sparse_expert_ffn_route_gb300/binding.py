"""Thin ctypes binding of libmoe.so (include/moe.h): argument marshalling only.

Every function takes CUDA torch tensors, passes their device pointers and the
current CUDA stream to the C entry point of the same name, and raises
``MoeError`` with the library's message on a nonzero return code.  All the
layer's arithmetic runs in the library's kernels; there is no other code path.
If libmoe.so is missing, loading raises ``ImportError``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_SHAPE = -2
MOE_ERR_ALIGN = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_UNSUPPORTED = -6
MOE_ERR_WORKSPACE = -7
MOE_ERR_DEVICE = -8
MOE_FLAG_SYNC_CHECK = 1
MOE_FLAG_STAGE_EVENTS = 2
MOE_FFN_WARP_GEMV = 0
MOE_FFN_TENSOR = 1
MOE_FFN_ROW_GEMV = 2
STAGES = ("router", "select", "permute", "plan", "quant", "gate_up", "quant_h", "down", "combine")

# every symbol include/moe.h declares
EXPORTS = ("moe_workspace_size", "moe_route", "moe_permute", "moe_expert_ffn", "moe_combine",
           "moe_layer_forward", "moe_check_errors", "moe_stage_times", "moe_last_error_string",
           "moe_route_noalloc", "moe_ffn_uses_tensor_cores", "moe_route_lookahead",
           "moe_topk_hits", "moe_quantize_int4_gs64", "moe_quantize_int3_g64",
           "moe_selftest_wait_timeout",
           "moe_layer_forward_host", "moe_ffn_path", "moe_ffn_path_down")


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__("%s failed (%d): %s" % (where, code, msg))
        self.code = code


class MoeConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("d_ff_shared", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("norm_topk_prob", ctypes.c_int32),
                ("routed_scaling_factor", ctypes.c_float), ("top_p", ctypes.c_float)]

    @classmethod
    def make(cls, hidden, n_experts, top_k, d_ff, n_shared=0, d_ff_shared=0, norm_topk_prob=1,
             routed_scaling_factor=1.0, top_p=0.0, group_size=64) -> "MoeConfig":
        return cls(hidden, n_experts, top_k, d_ff, n_shared, d_ff_shared, group_size,
                   norm_topk_prob, routed_scaling_factor, top_p)


class ExpertWeights(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("s_gate", ctypes.c_void_p),
                ("w_up", ctypes.c_void_p), ("s_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("s_down", ctypes.c_void_p)]

    @classmethod
    def of(cls, d: Dict[str, torch.Tensor]) -> "ExpertWeights":
        return cls(*[_ptr(d[k]) for k in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")])


class FfnProbe(ctypes.Structure):
    _fields_ = [("acc_gate", ctypes.c_void_p), ("acc_up", ctypes.c_void_p),
                ("acc_down", ctypes.c_void_p), ("hq", ctypes.c_void_p),
                ("h_scale", ctypes.c_void_p)]


class Routing(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("w", ctypes.c_void_p), ("keff", ctypes.c_void_p)]


_lib = None


def load_library():
    """Load libmoe.so (ImportError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY_PATH):
        raise ImportError("libmoe.so not found at %s; build it with "
                          "`python -m sparse_expert_ffn_route_gb300.build`" % LIBRARY_PATH)
    L = ctypes.CDLL(LIBRARY_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.moe_workspace_size.argtypes = [vp, i32]
    L.moe_workspace_size.restype = sz
    L.moe_ffn_uses_tensor_cores.argtypes = [vp, i32]
    L.moe_ffn_uses_tensor_cores.restype = i32
    L.moe_ffn_path.argtypes = [vp, i32]
    L.moe_ffn_path.restype = i32
    L.moe_ffn_path_down.argtypes = [vp, i32]
    L.moe_ffn_path_down.restype = i32
    L.moe_route.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
    L.moe_route_lookahead.argtypes = [vp, vp, vp, ctypes.c_float, vp, vp, i32, vp, vp, vp, vp, sz, vp]
    L.moe_topk_hits.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp]
    L.moe_quantize_int4_gs64.argtypes = [vp, i32, i32, vp, vp, vp]
    L.moe_quantize_int3_g64.argtypes = [vp, i32, i32, vp, vp, vp]
    L.moe_selftest_wait_timeout.argtypes = [vp, sz, i32, vp]
    L.moe_permute.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_expert_ffn.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_combine.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
    L.moe_layer_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, i32, vp]
    L.moe_layer_forward_host.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, i32, vp]
    L.moe_check_errors.argtypes = [vp, sz, vp]
    L.moe_stage_times.argtypes = [vp, vp, i32]
    L.moe_route_noalloc.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp]
    L.moe_last_error_string.argtypes = []
    L.moe_last_error_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where, load_library().moe_last_error_string().decode())


def last_error() -> str:
    return load_library().moe_last_error_string().decode()


def moe_workspace_size(cfg: MoeConfig, max_tokens: int) -> int:
    return int(load_library().moe_workspace_size(ctypes.byref(cfg), max_tokens))


def moe_ffn_uses_tensor_cores(cfg: MoeConfig, T: int) -> int:
    """1 if a call with T tokens runs the tensor-core grouped GEMM, 0 for the GEMV kernels,
    -1 for an invalid config or T."""
    return int(load_library().moe_ffn_uses_tensor_cores(ctypes.byref(cfg), T))


def moe_ffn_path(cfg: MoeConfig, T: int) -> int:
    """The grouped expert-FFN kernel a call with T tokens runs for gate/up:
    MOE_FFN_WARP_GEMV, MOE_FFN_TENSOR or MOE_FFN_ROW_GEMV; -1 for an invalid config or T."""
    return int(load_library().moe_ffn_path(ctypes.byref(cfg), T))


def moe_ffn_path_down(cfg: MoeConfig, T: int) -> int:
    """The same for the down projection."""
    return int(load_library().moe_ffn_path_down(ctypes.byref(cfg), T))


def alloc_workspace(cfg: MoeConfig, max_tokens: int, device="cuda") -> torch.Tensor:
    """Zeroed device workspace for up to ``max_tokens`` tokens (uint8 tensor)."""
    n = moe_workspace_size(cfg, max_tokens)
    if n == 0:
        raise MoeError(MOE_ERR_SHAPE, "moe_workspace_size", "invalid config or token count")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_route(cfg, x, w_router, bias, ids, w, keff, workspace, stream=None):
    T = x.shape[0]
    _check(load_library().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), T,
                                     _ptr(ids), _ptr(w), _ptr(keff), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "moe_route")


def moe_route_lookahead(cfg, x, norm_w, eps, w_router, bias, ids, w, keff, workspace, stream=None):
    """A layer's top-K predicted from the residual state x: RMSNorm with norm_w and eps, then
    the layer's router (w_router, bias); outputs as moe_route."""
    T = x.shape[0]
    _check(load_library().moe_route_lookahead(ctypes.byref(cfg), _ptr(x), _ptr(norm_w), float(eps),
                                               _ptr(w_router), _ptr(bias), T, _ptr(ids), _ptr(w),
                                               _ptr(keff), _ptr(workspace), workspace.numel(),
                                               _stream(stream)), "moe_route_lookahead")


def moe_topk_hits(cfg, ids_pred, keff_pred, ids_true, keff_true, hits, stream=None):
    """Per token, how many experts the predicted and the true routing both keep."""
    T = keff_pred.shape[0]
    _check(load_library().moe_topk_hits(ctypes.byref(cfg), _ptr(ids_pred), _ptr(keff_pred),
                                         _ptr(ids_true), _ptr(keff_true), T, _ptr(hits),
                                         _stream(stream)), "moe_topk_hits")


def moe_quantize_int3_g64(w, packed, scales, stream=None):
    """fp32 weights w [rows][K] (K a multiple of 64) -> int3-g64: packed [rows][3K/8] uint8
    and scales [rows][K/64] float32 (every leading dimension flattened into rows)."""
    K = w.shape[-1]
    rows = w.numel() // K if K else 0
    _check(load_library().moe_quantize_int3_g64(_ptr(w), rows, K, _ptr(packed), _ptr(scales),
                                                 _stream(stream)), "moe_quantize_int3_g64")


def moe_quantize_int4_gs64(w, packed, scales, stream=None):
    """fp32 weights w [rows][K] (K a multiple of 64) -> int4-gs64: packed [rows][K/2] uint8
    and scales [rows][K/64] float32 (every leading dimension flattened into rows)."""
    K = w.shape[-1]
    rows = w.numel() // K if K else 0
    _check(load_library().moe_quantize_int4_gs64(_ptr(w), rows, K, _ptr(packed), _ptr(scales),
                                                  _stream(stream)), "moe_quantize_int4_gs64")


def moe_selftest_wait_timeout(workspace, polls: int = 4096, stream=None):
    """Make one bounded device wait run out on purpose; moe_check_errors then reports
    MOE_ERR_TIMEOUT (the error path of the kernels' waits, with no fault or hang)."""
    _check(load_library().moe_selftest_wait_timeout(_ptr(workspace), workspace.numel(), int(polls),
                                                     _stream(stream)), "moe_selftest_wait_timeout")


def moe_route_noalloc(cfg, x, w_router, bias, ids, w, keff, stream=None):
    """moe_route without a workspace (the router scratch is a fixed array inside libmoe.so,
    so the call allocates nothing); same outputs as moe_route, batches up to its limit."""
    T = x.shape[0]
    _check(load_library().moe_route_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(w_router),
                                             _ptr(bias), T, _ptr(ids), _ptr(w), _ptr(keff),
                                             _stream(stream)), "moe_route_noalloc")


def moe_permute(cfg, ids, keff, counts, offsets, tok, slot, uniq, n_uniq, workspace, stream=None):
    T = keff.shape[0]
    _check(load_library().moe_permute(ctypes.byref(cfg), _ptr(ids), _ptr(keff), T, _ptr(counts),
                                       _ptr(offsets), _ptr(tok), _ptr(slot), _ptr(uniq),
                                       _ptr(n_uniq), _ptr(workspace), workspace.numel(),
                                       _stream(stream)), "moe_permute")


def moe_expert_ffn(cfg, x, routed: Dict[str, torch.Tensor], offsets, tok, uniq, n_uniq, y_pairs,
                   workspace, probe: Optional[Dict[str, torch.Tensor]] = None, stream=None):
    T = x.shape[0]
    rw = ExpertWeights.of(routed)
    pr = None
    if probe is not None:
        pr = FfnProbe(*[_ptr(probe.get(k)) for k in ("acc_gate", "acc_up", "acc_down", "hq",
                                                       "h_scale")])
    _check(load_library().moe_expert_ffn(ctypes.byref(cfg), _ptr(x), T, ctypes.byref(rw),
                                          _ptr(offsets), _ptr(tok), _ptr(uniq), _ptr(n_uniq),
                                          _ptr(y_pairs), ctypes.byref(pr) if pr else None,
                                          _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_expert_ffn")


def moe_combine(cfg, y_pairs, ids, keff, w, offsets, tok, y, workspace, x=None,
                shared: Optional[Dict[str, torch.Tensor]] = None, stream=None):
    T = keff.shape[0]
    sw = ExpertWeights.of(shared) if shared is not None else None
    _check(load_library().moe_combine(ctypes.byref(cfg), _ptr(y_pairs), _ptr(ids), _ptr(keff),
                                       _ptr(w), _ptr(offsets), _ptr(tok), T, _ptr(x),
                                       ctypes.byref(sw) if sw else None, _ptr(y),
                                       _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_combine")


def moe_layer_forward(cfg, x, w_router, bias, routed, shared, y, workspace, routing=None,
                      flags: int = 0, stream=None):
    T = x.shape[0]
    rw = ExpertWeights.of(routed)
    sw = ExpertWeights.of(shared) if shared is not None else None
    ro = None
    if routing is not None:
        ro = Routing(_ptr(routing.get("ids")), _ptr(routing.get("w")), _ptr(routing.get("keff")))
    _check(load_library().moe_layer_forward(ctypes.byref(cfg), _ptr(x), T, _ptr(w_router),
                                             _ptr(bias), ctypes.byref(rw),
                                             ctypes.byref(sw) if sw else None, _ptr(y),
                                             ctypes.byref(ro) if ro else None, _ptr(workspace),
                                             workspace.numel(), flags, _stream(stream)),
           "moe_layer_forward")


def moe_layer_forward_host(cfg, x_host, w_router, bias, routed, shared, y_host, workspace,
                           routing=None, flags: int = 0, stream=None):
    """moe_layer_forward on host tensors x_host / y_host (CPU, pinned for asynchronous
    copies): the library copies x in, runs the layer and copies y out on the stream."""
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("moe_layer_forward_host takes CPU tensors for x and y")
    T = x_host.shape[0]
    rw = ExpertWeights.of(routed)
    sw = ExpertWeights.of(shared) if shared is not None else None
    ro = None
    if routing is not None:
        ro = Routing(_ptr(routing.get("ids")), _ptr(routing.get("w")), _ptr(routing.get("keff")))
    _check(load_library().moe_layer_forward_host(ctypes.byref(cfg), _ptr(x_host), T, _ptr(w_router),
                                                  _ptr(bias), ctypes.byref(rw),
                                                  ctypes.byref(sw) if sw else None, _ptr(y_host),
                                                  ctypes.byref(ro) if ro else None, _ptr(workspace),
                                                  workspace.numel(), flags, _stream(stream)),
           "moe_layer_forward_host")


def moe_check_errors(workspace, stream=None):
    _check(load_library().moe_check_errors(_ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_check_errors")


def moe_stage_times(reset: bool = True):
    """Per-stage device milliseconds and kernel launches of the layer calls made with
    MOE_FLAG_STAGE_EVENTS on this thread since the last reset: {stage: (ms, launches)}."""
    ms = (ctypes.c_double * len(STAGES))()
    n = (ctypes.c_longlong * len(STAGES))()
    _check(load_library().moe_stage_times(ms, n, 1 if reset else 0), "moe_stage_times")
    return {name: (ms[i], int(n[i])) for i, name in enumerate(STAGES)}
