"""CPU oracle of the sparse MoE FFN layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  It wraps ``libmoe_ref.so`` (plain C99, built from
``moe_ref.c`` with gcc) through ctypes and takes numpy arrays or CPU torch
tensors.  It shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_ref.c")
_HDR = os.path.join(_HERE, "moe_ref.h")
_LIB = os.path.join(_HERE, "libmoe_ref.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile libmoe_ref.so with gcc (-O2, OpenMP, no FP contraction)."""
    fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if fresh and not force:
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("d_ff_shared", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32),
                ("routed_scaling_factor", ctypes.c_float), ("top_p", ctypes.c_float)]


class Weights(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("s_gate", ctypes.c_void_p),
                ("w_up", ctypes.c_void_p), ("s_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("s_down", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.moe_ref_route.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp]
        L.moe_ref_permute.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]
        L.moe_ref_quant_row.argtypes = [vp, i32, vp, vp]
        L.moe_ref_quant_row.restype = None
        L.moe_ref_quant_row_pre.argtypes = [vp, i32, vp, vp, vp]
        L.moe_ref_quant_row_pre.restype = None
        L.moe_ref_group_dot.argtypes = [vp, vp, i32]
        L.moe_ref_expert_apply.argtypes = [i32, i32] + [vp] * 6 + [vp, ctypes.c_float] + [vp] * 9
        L.moe_ref_expert_ffn.argtypes = [vp, vp, i32, vp, vp, vp, vp] + [vp] * 8
        L.moe_ref_shared_ffn.argtypes = [vp, vp, i32, vp, vp]
        L.moe_ref_combine.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp]
        L.moe_ref_layer_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_ref_threads.argtypes = []
        L.moe_ref_rmsnorm.argtypes = [vp, vp, ctypes.c_float, i32, i32, vp]
        L.moe_ref_route_lookahead.argtypes = [vp, vp, vp, ctypes.c_float, vp, vp, i32, vp, vp, vp, vp]
        L.moe_ref_topk_hits.argtypes = [i32, i32, vp, vp, vp, vp, vp]
        L.moe_ref_quantize_int4.argtypes = [vp, i32, i32, vp, vp]
        L.moe_ref_quantize_int3.argtypes = [vp, i32, i32, vp, vp]
        L.moe_ref_dequant_int3.argtypes = [vp, vp, i32, i32, vp]
        _lib = L
    return _lib


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _np(a, dtype=None) -> np.ndarray:
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (np.dtype(dtype), a.dtype))
    return a


def _p(a) -> Optional[int]:
    return None if a is None else a.ctypes.data


def make_config(hidden, n_experts, top_k, d_ff, n_shared=0, d_ff_shared=0, norm_topk_prob=1,
                routed_scaling_factor=1.0, top_p=0.0) -> Config:
    return Config(hidden, n_experts, top_k, d_ff, n_shared, d_ff_shared, norm_topk_prob,
                  routed_scaling_factor, top_p)


def config_of(wl) -> Config:
    """Config of a ``synth.Workload``."""
    return make_config(wl.hidden, wl.n_experts, wl.top_k, wl.d_ff, wl.n_shared, wl.d_ff_shared,
                       wl.norm_topk_prob, wl.routed_scaling_factor, wl.top_p)


def _weights(d: Dict) -> (Weights, list):
    keep = [_np(d[k]) for k in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")]
    for a, dt in zip(keep, (np.uint8, np.float32) * 3):
        if a.dtype != dt:
            raise TypeError("weight dtype %s, expected %s" % (a.dtype, np.dtype(dt)))
    return Weights(*[_p(a) for a in keep]), keep


def _check(rc, name):
    if rc != 0:
        raise RuntimeError("%s failed with %d" % (name, rc))


# --------------------------------------------------------------------------
# API
# --------------------------------------------------------------------------

def route(cfg: Config, x, w_router, bias, with_logits: bool = False):
    x = _np(x, np.float32); wr = _np(w_router, np.float32); b = _np(bias, np.float32)
    T = x.shape[0]
    K, E = cfg.top_k, cfg.n_experts
    ids = np.zeros((T, K), np.int32); w = np.zeros((T, K), np.float32)
    keff = np.zeros(T, np.int32)
    logits = np.zeros((T, E), np.float32) if with_logits else None
    _check(lib().moe_ref_route(ctypes.byref(cfg), _p(x), _p(wr), _p(b), T, _p(ids), _p(w),
                               _p(keff), _p(logits)), "moe_ref_route")
    out = {"ids": ids, "w": w, "keff": keff}
    if with_logits:
        out["logits"] = logits
    return out


def quantize_int4(w):
    """fp32 weights [rows][K] -> (packed nibbles [rows][K/2] u8, scales [rows][K/64] fp32)."""
    w = _np(w, np.float32)
    rows, K = w.shape
    packed = np.zeros((rows, K // 2), np.uint8)
    scales = np.zeros((rows, K // 64), np.float32)
    _check(lib().moe_ref_quantize_int4(_p(w), rows, K, _p(packed), _p(scales)), "moe_ref_quantize_int4")
    return packed, scales


def quantize_int3(w):
    """fp32 weights [rows][K] -> (packed int3-g64 [rows][3K/8] u8, scales [rows][K/64] fp32)."""
    w = _np(w, np.float32)
    rows, K = w.shape
    packed = np.zeros((rows, 3 * K // 8), np.uint8)
    scales = np.zeros((rows, K // 64), np.float32)
    _check(lib().moe_ref_quantize_int3(_p(w), rows, K, _p(packed), _p(scales)), "moe_ref_quantize_int3")
    return packed, scales


def dequant_int3(packed, scales):
    """The fp32 values [rows][K] an int3-g64 matrix stands for."""
    packed = _np(packed, np.uint8); scales = _np(scales, np.float32)
    rows, G = scales.shape
    out = np.zeros((rows, 64 * G), np.float32)
    _check(lib().moe_ref_dequant_int3(_p(packed), _p(scales), rows, 64 * G, _p(out)), "moe_ref_dequant_int3")
    return out


def rmsnorm(x, g, eps: float):
    """RMSNorm of each row of x [T][H] with weight g [H] (["MoE 路由与专家流式加载" §5])."""
    x = _np(x, np.float32); g = _np(g, np.float32)
    T, H = x.shape
    out = np.zeros((T, H), np.float32)
    _check(lib().moe_ref_rmsnorm(_p(x), _p(g), float(eps), T, H, _p(out)), "moe_ref_rmsnorm")
    return out


def route_lookahead(cfg: Config, x, norm_w, eps: float, w_router, bias, with_logits: bool = False):
    """The router applied to RMSNorm(x): a later layer's predicted top-K (la_predict)."""
    x = _np(x, np.float32); g = _np(norm_w, np.float32)
    wr = _np(w_router, np.float32); b = _np(bias, np.float32)
    T = x.shape[0]
    K, E = cfg.top_k, cfg.n_experts
    ids = np.zeros((T, K), np.int32); w = np.zeros((T, K), np.float32)
    keff = np.zeros(T, np.int32)
    logits = np.zeros((T, E), np.float32) if with_logits else None
    _check(lib().moe_ref_route_lookahead(ctypes.byref(cfg), _p(x), _p(g), float(eps), _p(wr),
                                         _p(b), T, _p(ids), _p(w), _p(keff), _p(logits)),
           "moe_ref_route_lookahead")
    out = {"ids": ids, "w": w, "keff": keff}
    if with_logits:
        out["logits"] = logits
    return out


def topk_hits(ids_pred, keff_pred, ids_true, keff_true):
    """Per token, the number of experts kept by both routings."""
    ip = _np(ids_pred, np.int32); kp = _np(keff_pred, np.int32)
    it = _np(ids_true, np.int32); kt = _np(keff_true, np.int32)
    T, K = ip.shape
    hits = np.zeros(T, np.int32)
    _check(lib().moe_ref_topk_hits(T, K, _p(ip), _p(kp), _p(it), _p(kt), _p(hits)),
           "moe_ref_topk_hits")
    return hits


def permute(cfg: Config, ids, keff):
    ids = _np(ids, np.int32); keff = _np(keff, np.int32)
    T, K, E = keff.shape[0], cfg.top_k, cfg.n_experts
    counts = np.zeros(E, np.int32); offsets = np.zeros(E + 1, np.int32)
    tok = np.zeros(max(T * K, 1), np.int32); slot = np.zeros(max(T * K, 1), np.int32)
    uniq = np.zeros(E, np.int32); n_uniq = np.zeros(1, np.int32)
    _check(lib().moe_ref_permute(ctypes.byref(cfg), _p(ids), _p(keff), T, _p(counts),
                                 _p(offsets), _p(tok), _p(slot), _p(uniq), _p(n_uniq)),
           "moe_ref_permute")
    P = int(offsets[E]); U = int(n_uniq[0])
    return {"counts": counts, "offsets": offsets, "tok": tok[:P], "slot": slot[:P],
            "uniq": uniq[:U], "n_uniq": U}


def quant_row(v):
    v = _np(v, np.float32)
    q = np.zeros(v.shape[-1], np.int8); s = np.zeros(1, np.float32)
    lib().moe_ref_quant_row(_p(v), v.shape[-1], _p(q), _p(s))
    return q, float(s[0])


def quant_row_pre(v):
    """quant_row plus the fp32 value each code rounds (v * 127 / amax)."""
    v = _np(v, np.float32)
    q = np.zeros(v.shape[-1], np.int8); s = np.zeros(1, np.float32)
    pre = np.zeros(v.shape[-1], np.float32)
    lib().moe_ref_quant_row_pre(_p(v), v.shape[-1], _p(q), _p(s), _p(pre))
    return q, float(s[0]), pre


def quant_rows(m):
    m = _np(m, np.float32)
    q = np.zeros(m.shape, np.int8); s = np.zeros(m.shape[0], np.float32)
    for i in range(m.shape[0]):
        q[i], s[i] = quant_row(m[i])
    return q, s


def group_dot(row, q, g: int) -> int:
    row = _np(row, np.uint8); q = _np(q, np.int8)
    return int(lib().moe_ref_group_dot(_p(row), _p(q), g))


def expert_apply(H, F, expert: Dict, xq, sx: float, probes: bool = False, hq_in=None,
                 hs_in: Optional[float] = None):
    """One expert (its own [F, H/2] ... tensors) on one quantised token."""
    wt, keep = _weights(expert)
    xq = _np(xq, np.int8)
    y = np.zeros(H, np.float64)
    ag = au = ad = hq = hs = hp = None
    if probes:
        ag = np.zeros((F, H // 64), np.int32); au = np.zeros((F, H // 64), np.int32)
        ad = np.zeros((H, F // 64), np.int32); hq = np.zeros(F, np.int8); hs = np.zeros(1, np.float32)
        hp = np.zeros(F, np.float32)
    hqi = _np(hq_in, np.int8)
    hsi = None if hs_in is None else np.array([hs_in], np.float32)
    _check(lib().moe_ref_expert_apply(H, F, wt.w_gate, wt.s_gate, wt.w_up, wt.s_up, wt.w_down,
                                      wt.s_down, _p(xq), sx, _p(y), _p(ag), _p(au), _p(ad),
                                      _p(hq), _p(hs), _p(hqi), _p(hsi), _p(hp)), "moe_ref_expert_apply")
    out = {"y": y}
    if probes:
        out.update(acc_gate=ag, acc_up=au, acc_down=ad, hq=hq, hs=float(hs[0]), h_pre=hp)
    return out


def expert_ffn(cfg: Config, x, routed: Dict, offsets, tok, probes: bool = False,
               hq_in=None, hs_in=None):
    x = _np(x, np.float32); offsets = _np(offsets, np.int32); tok = _np(tok, np.int32)
    wt, keep = _weights(routed)
    T, H, F = x.shape[0], cfg.hidden, cfg.d_ff
    P = int(offsets[cfg.n_experts])
    y = np.zeros((max(P, 1), H), np.float64)
    ag = au = ad = hq = hs = hp = None
    if probes:
        ag = np.zeros((P, F, H // 64), np.int32); au = np.zeros((P, F, H // 64), np.int32)
        ad = np.zeros((P, H, F // 64), np.int32); hq = np.zeros((P, F), np.int8)
        hs = np.zeros(P, np.float32); hp = np.zeros((P, F), np.float32)
    hqi = _np(hq_in, np.int8); hsi = _np(hs_in, np.float32)
    tokp = tok if tok.size else np.zeros(1, np.int32)
    _check(lib().moe_ref_expert_ffn(ctypes.byref(cfg), _p(x), T, ctypes.byref(wt), _p(offsets),
                                    _p(tokp), _p(y), _p(ag), _p(au), _p(ad), _p(hq), _p(hs),
                                    _p(hqi), _p(hsi), _p(hp)), "moe_ref_expert_ffn")
    out = {"y_pairs": y[:P]}
    if probes:
        out.update(acc_gate=ag, acc_up=au, acc_down=ad, hq=hq, hs=hs, h_pre=hp)
    return out


def shared_ffn(cfg: Config, x, shared: Dict):
    x = _np(x, np.float32)
    wt, keep = _weights({k: (v[0] if getattr(v, "ndim", 0) == 3 else v) for k, v in shared.items()})
    ys = np.zeros((x.shape[0], cfg.hidden), np.float64)
    _check(lib().moe_ref_shared_ffn(ctypes.byref(cfg), _p(x), x.shape[0], ctypes.byref(wt),
                                    _p(ys)), "moe_ref_shared_ffn")
    return ys


def combine(cfg: Config, y_pairs, slot, offsets, w, keff, ys=None):
    yp = _np(y_pairs, np.float64); slot = _np(slot, np.int32); offsets = _np(offsets, np.int32)
    w = _np(w, np.float32); keff = _np(keff, np.int32); ys = _np(ys, np.float64)
    T = keff.shape[0]
    y = np.zeros((T, cfg.hidden), np.float64)
    ypp = yp if yp.size else np.zeros(1, np.float64)
    slp = slot if slot.size else np.zeros(1, np.int32)
    _check(lib().moe_ref_combine(ctypes.byref(cfg), _p(ypp), _p(slp), _p(offsets), _p(w),
                                 _p(keff), T, _p(ys), _p(y)), "moe_ref_combine")
    return y


def layer_forward(cfg: Config, x, w_router, bias, routed: Dict, shared: Optional[Dict]):
    x = _np(x, np.float32); wr = _np(w_router, np.float32); b = _np(bias, np.float32)
    T, K = x.shape[0], cfg.top_k
    rw, keep1 = _weights(routed)
    sw = None
    if shared is not None:
        sw, keep2 = _weights({k: (v[0] if getattr(v, "ndim", 0) == 3 else v)
                              for k, v in shared.items()})
    y = np.zeros((T, cfg.hidden), np.float64)
    ids = np.zeros((T, K), np.int32); w = np.zeros((T, K), np.float32); keff = np.zeros(T, np.int32)
    _check(lib().moe_ref_layer_forward(ctypes.byref(cfg), _p(x), T, _p(wr), _p(b),
                                       ctypes.byref(rw), ctypes.byref(sw) if sw else None,
                                       _p(y), _p(ids), _p(w), _p(keff)), "moe_ref_layer_forward")
    return {"y": y, "ids": ids, "w": w, "keff": keff}


def threads() -> int:
    return int(lib().moe_ref_threads())
