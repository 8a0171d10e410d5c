"""Shared helpers of the GPU parity tests: inputs on both sides, routing margins.

Inputs for the CUDA path and for the oracle come from the same seeded generator
(``synth``); nothing computed by the CUDA path is ever handed to the oracle.
"""
from __future__ import annotations

from dataclasses import replace
from typing import Dict, Optional

import numpy as np
import torch

import oracle
import parity
import synth

_DEV_CACHE: Dict[tuple, Dict[str, torch.Tensor]] = {}


def device_experts(wl: synth.Workload, shared: bool = False) -> Dict[str, torch.Tensor]:
    """All routed experts (or the shared one) of a workload, generated on the GPU (cached)."""
    key = (wl.hidden, wl.n_experts, wl.d_ff, wl.d_ff_shared, wl.seed, wl.scale_lo, wl.scale_hi, shared)
    if key not in _DEV_CACHE:
        _DEV_CACHE[key] = synth.gen_experts(wl, shared=shared, device="cuda")
    return _DEV_CACHE[key]


def drop_device_cache():
    _DEV_CACHE.clear()
    torch.cuda.empty_cache()


def moe_cfg(wl: synth.Workload):
    import sparse_expert_ffn_route_gb300 as moe
    return moe.MoeConfig.make(wl.hidden, wl.n_experts, wl.top_k, wl.d_ff, wl.n_shared,
                              wl.d_ff_shared, wl.norm_topk_prob, wl.routed_scaling_factor,
                              wl.top_p)


def compact_experts(wl: synth.Workload, experts) -> Dict[str, np.ndarray]:
    """Host copies of just the listed experts (for per-token oracle checks at full size)."""
    d = synth.gen_experts(wl, experts=list(experts))
    return {k: v.numpy() for k, v in d.items()}


def oracle_tokens(wl: synth.Workload, x_rows: np.ndarray, ids: np.ndarray, w: np.ndarray,
                  keff: np.ndarray):
    """The oracle's layer reference (``parity.layer_reference``) of a few tokens whose routing
    (ids, w, keff) the oracle chose, regenerating only the experts those tokens use.  The
    routed expert ids are remapped to 0..U-1 so the oracle runs on a compact expert set
    (index bookkeeping only)."""
    T, K = ids.shape
    used = sorted({int(e) for t in range(T) for e in ids[t, :keff[t]]})
    remap = {e: i for i, e in enumerate(used)}
    ids_c = np.full_like(ids, -1)
    for t in range(T):
        for i in range(keff[t]):
            ids_c[t, i] = remap[int(ids[t, i])]
    wl_c = replace(wl, n_experts=len(used))
    cfg = oracle.config_of(wl_c)
    R = compact_experts(wl, used)
    S = None
    if wl.n_shared:
        S = {k: v.numpy() for k, v in synth.gen_experts(wl, shared=True).items()}
    return parity.layer_reference(oracle, cfg, x_rows, ids_c, w, keff, R, S)


def host_experts(wl: synth.Workload, shared: bool = False) -> Dict[str, np.ndarray]:
    return {k: v.numpy() for k, v in synth.gen_experts(wl, shared=shared).items()}


def rel_err(a: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2)))
    return float(np.max(np.abs(np.asarray(a, np.float64) - ref))) / max(rms, 1e-30)
