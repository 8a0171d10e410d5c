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


def sig64(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, np.float64)))


def routing_margins(logits: np.ndarray, bias: np.ndarray, K: int, top_p: float) -> np.ndarray:
    """Per token, the smallest distance (in fp64) of any decision the router takes to its
    tie point: between consecutive choices among the top K+1, and, with top-p, between the
    running gate sum and p * total at the cut and just before it."""
    choice = sig64(logits) + bias.astype(np.float64)[None, :]
    T, E = choice.shape
    out = np.empty(T)
    for t in range(T):
        order = np.argsort(-choice[t], kind="stable")
        top = choice[t, order[:min(K + 1, E)]]
        m = np.min(np.abs(np.diff(top))) if top.size > 1 else np.inf
        if 0.0 < top_p < 1.0:
            g = np.sort(sig64(logits[t, order[:K]]))[::-1]
            if g.size > 1:
                m = min(m, np.min(np.abs(np.diff(g))))
            cum = np.cumsum(g)
            m = min(m, np.min(np.abs(cum - top_p * cum[-1])))
        out[t] = m
    return out


def compact_experts(wl: synth.Workload, experts) -> Dict[str, np.ndarray]:
    """Host copies of just the listed experts (for per-token oracle checks at full size)."""
    d = synth.gen_experts(wl, experts=list(experts))
    return {k: v.numpy() for k, v in d.items()}


def oracle_tokens(wl: synth.Workload, x_rows: np.ndarray, ids: np.ndarray, w: np.ndarray,
                  keff: np.ndarray) -> np.ndarray:
    """Oracle output rows of a few tokens whose routing (ids, w, keff) the oracle chose,
    regenerating only the experts those tokens use.  The routed expert ids are remapped to
    0..U-1 so the oracle runs on a compact expert set (index bookkeeping only)."""
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
    perm = oracle.permute(cfg, ids_c, keff)
    ffn = oracle.expert_ffn(cfg, x_rows, R, perm["offsets"], perm["tok"])
    ys = None
    if wl.n_shared:
        S = {k: v[0].numpy() for k, v in synth.gen_experts(wl, shared=True).items()}
        ys = oracle.shared_ffn(cfg, x_rows, S)
    return oracle.combine(cfg, ffn["y_pairs"], perm["slot"], perm["offsets"], w, keff, ys)


def tokens_within(y: np.ndarray, ref: np.ndarray, tol: float, flip_tol: float = 20e-3,
                  max_share: float = 0.05) -> None:
    """Layer outputs [tokens, H] against the oracle.  Every token within tol x RMS except a
    few (at most max(1, max_share of them)), which stay within flip_tol x RMS: an int8 code
    of h = SiLU(gate)*up lying at a rounding boundary may legitimately land on either side
    (fp32 sums in another order than the oracle's), and one such code moves its token's
    output by one code step's contribution, measured at up to ~6e-3 x RMS."""
    rms = float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2)))
    err = np.max(np.abs(np.asarray(y, np.float64) - ref), axis=1) / max(rms, 1e-30)
    over = int(np.sum(err > tol))
    allowed = max(1, int(np.ceil(max_share * len(err))))
    assert over <= allowed, "%d of %d tokens beyond %.1g x RMS (max %.3g)" % (over, len(err), tol, err.max())
    assert err.max() <= flip_tol, "a token beyond the one-code-step bound: %.3g x RMS" % err.max()


def rel_err(a: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2)))
    return float(np.max(np.abs(np.asarray(a, np.float64) - ref))) / max(rms, 1e-30)
