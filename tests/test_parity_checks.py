"""The parity checks themselves (``tests/parity.py``), on the CPU: every mistake is planted in
a copy of the oracle's own results, never in anything the CUDA path computed.

A check that accepts the oracle's results unchanged, accepts a code flipped at a rounding
boundary (with the down projection recomputed by the oracle on the flipped codes), and
rejects a flip away from a boundary, an inconsistent down accumulator, a moved output and an
invalid routing, is one the GPU tests can rely on.
"""
import numpy as np
import pytest

import parity
import synth


def _case(ref, H=2048, F=512, E=4, K=2, T=8):
    wl = synth.Workload("chk", H, E, K, F, 1, F, (T,), 1, 1.0, 0.0, 0.1)
    cfg = ref.config_of(wl)
    x = synth.gen_x(wl, T).numpy()
    wr, bias = synth.gen_router(wl)
    r = ref.route(cfg, x, wr, bias, with_logits=True)
    perm = ref.permute(cfg, r["ids"], r["keff"])
    R = {k: v.numpy() for k, v in synth.gen_experts(wl).items()}
    out = ref.expert_ffn(cfg, x, R, perm["offsets"], perm["tok"], probes=True)
    xq, sx = ref.quant_rows(x)
    g = {"acc_gate": out["acc_gate"].copy(), "acc_up": out["acc_up"].copy(),
         "acc_down": out["acc_down"].copy(), "hq": out["hq"].copy(),
         "h_scale": out["hs"].copy(), "y": out["y_pairs"].astype(np.float32)}
    return wl, cfg, x, wr, bias, r, perm, R, out, xq, sx, g


def _expert_of(perm, p):
    return int(np.searchsorted(perm["offsets"], p, side="right") - 1)


def _closest_flip(R, perm, out, xq, sx):
    """The pair and h code lying closest to a rounding boundary, relative to the bound."""
    best = None
    for p in range(len(perm["tok"])):
        e, t = _expert_of(perm, p), int(perm["tok"][p])
        G = R["s_gate"].shape[-1]
        Dg = parity.half_sums(R["w_gate"][e], xq[[t]])
        Du = parity.half_sums(R["w_up"][e], xq[[t]])
        eps = parity.h_pre_bound(sx[[t]], R["s_gate"][e], Dg, R["s_up"][e], Du,
                                 out["h_pre"][[p]], depth=G + 16)[0]
        off = out["h_pre"][p].astype(np.float64) - out["hq"][p]
        ratio = (0.5 - np.abs(off)) / eps
        k = int(np.argmin(np.where(off != 0, ratio, np.inf)))
        if best is None or ratio[k] < best[0]:
            best = (float(ratio[k]), p, k, int(np.sign(off[k])))
    return best


def _planted_flip(ref, x, R, perm, out, xq, sx, g, p, k, sgn):
    e = _expert_of(perm, p)
    hq = out["hq"][p].copy()
    hq[k] += sgn
    ex = {kk: v[e] for kk, v in R.items()}
    H, F = R["w_down"].shape[1], hq.size
    t = int(perm["tok"][p])
    r = ref.expert_apply(H, F, ex, xq[t], float(sx[t]), probes=True, hq_in=hq,
                         hs_in=float(out["hs"][p]))
    g["hq"][p] = hq
    g["acc_down"][p] = r["acc_down"]
    g["y"][p] = r["y"].astype(np.float32)


def test_unchanged_oracle_results_pass(ref):
    _, _, x, _, _, _, perm, R, out, xq, sx, g = _case(ref)
    c = parity.check_ffn_pairs(g, out, x, R, perm["offsets"], perm["tok"], xq, sx)
    assert c["h_flips"] == 0


def test_flip_at_a_boundary_passes_and_elsewhere_fails(ref):
    _, _, x, _, _, _, perm, R, out, xq, sx, g0 = _case(ref)
    ratio, p, k, sgn = _closest_flip(R, perm, out, xq, sx)
    assert ratio < 1.0, "no h code of this case lies within its bound of a boundary"
    g = {kk: v.copy() for kk, v in g0.items()}
    _planted_flip(ref, x, R, perm, out, xq, sx, g, p, k, sgn)
    c = parity.check_ffn_pairs(g, out, x, R, perm["offsets"], perm["tok"], xq, sx)
    assert c["h_flips"] == 1
    # the same flip without the down projection following it
    g2 = {kk: v.copy() for kk, v in g.items()}
    g2["acc_down"][p] = out["acc_down"][p]
    with pytest.raises(AssertionError, match="brute force"):
        parity.check_ffn_pairs(g2, out, x, R, perm["offsets"], perm["tok"], xq, sx)
    # a code flipped far from any boundary
    off = np.abs(out["h_pre"][p].astype(np.float64) - out["hq"][p])
    kf = int(np.argmin(off))          # a value sitting on its code: 0.5 from both boundaries
    g3 = {kk: v.copy() for kk, v in g0.items()}
    _planted_flip(ref, x, R, perm, out, xq, sx, g3, p, kf, 1 if out["hq"][p][kf] < 127 else -1)
    with pytest.raises(AssertionError, match="not at a rounding boundary"):
        parity.check_ffn_pairs(g3, out, x, R, perm["offsets"], perm["tok"], xq, sx)
    # an output moved by 2e-3 x RMS
    g4 = {kk: v.copy() for kk, v in g0.items()}
    g4["y"][3, 5] += 2e-3 * parity.rms(out["y_pairs"])
    with pytest.raises(AssertionError, match="y_pairs beyond"):
        parity.check_ffn_pairs(g4, out, x, R, perm["offsets"], perm["tok"], xq, sx)
    # a gate accumulator off by one
    g5 = {kk: v.copy() for kk, v in g0.items()}
    g5["acc_gate"][0, 0, 0] += 1
    with pytest.raises(AssertionError, match="acc_gate"):
        parity.check_ffn_pairs(g5, out, x, R, perm["offsets"], perm["tok"], xq, sx)


def test_layer_token_explained_by_a_flip_and_noise_rejected(ref):
    wl, cfg, x, wr, bias, r, perm, R, out, xq, sx, _ = _case(ref)
    S = {k: v.numpy() for k, v in synth.gen_experts(wl, shared=True).items()}
    L = parity.layer_reference(ref, cfg, x, r["ids"], r["w"], r["keff"], R, S)
    T = x.shape[0]
    assert parity.explain_tokens(L["y"].astype(np.float32), L, range(T))["tokens_over"] == 0
    # move one token by the exact effect of a boundary flip in one of its routed pairs
    ratio, p, k, sgn = _closest_flip(R, perm, out, xq, sx)
    assert ratio < 1.0
    t = int(perm["tok"][p])
    i = int(perm["slot"][p]) - t * cfg.top_k
    e = _expert_of(perm, p)
    hq = out["hq"][p].copy()
    hq[k] += sgn
    H, F = cfg.hidden, cfg.d_ff
    alt = ref.expert_apply(H, F, {kk: v[e] for kk, v in R.items()}, xq[t], float(sx[t]),
                           hq_in=hq, hs_in=float(out["hs"][p]))["y"]
    y = L["y"].copy()
    y[t] += float(r["w"][t, i]) * (alt - out["y_pairs"][p])
    assert np.abs(y[t] - L["y"][t]).max() > parity.TOL * parity.rms(L["y"])
    c = parity.explain_tokens(y, L, range(T))
    assert c["tokens_over"] == 1 and c["flips"] == 1
    # noise that no set of flips explains
    y2 = L["y"].copy()
    y2[1] += 5e-3 * parity.rms(L["y"]) * np.sin(np.arange(H))
    with pytest.raises(AssertionError, match="not explained|no h code"):
        parity.explain_tokens(y2, L, range(T))


def test_valid_routing_hand_cases():
    # 6 experts; experts 2 and 4 tie for the 3rd choice (K = 3)
    logits = np.log(np.array([0.9, 0.8, 0.5, 0.1, 0.5, 0.3]) / (1 - np.array([0.9, 0.8, 0.5, 0.1, 0.5, 0.3])))
    bias = np.zeros(6)
    gate = parity.sig64(logits)

    def w_of(ids):
        g = gate[ids]
        return g / g.sum()
    for third in (2, 4):
        ids = np.array([0, 1, third])
        assert parity.valid_routing(logits, bias, ids, w_of(ids), 3, 3, 0.0, 1, 1.0) == ""
    ids = np.array([0, 1, 5])              # the 4th-best expert
    assert "top K" in parity.valid_routing(logits, bias, ids, w_of(ids), 3, 3, 0.0, 1, 1.0)
    ids = np.array([1, 0, 2])              # wrong order
    assert "order" in parity.valid_routing(logits, bias, ids, w_of(ids), 3, 3, 0.0, 1, 1.0)
    ids = np.array([0, 1, 2])
    assert "weights" in parity.valid_routing(logits, bias, ids, w_of(ids) * 1.01, 3, 3, 0.0, 1, 1.0)
    # top-p = 0.4 of gates {0.9, 0.8, 0.5}: total 2.2, threshold 0.88 -> keep 1 expert
    ids = np.array([0, -1, -1])
    w = np.array([1.0, 0.0, 0.0])
    assert parity.valid_routing(logits, bias, ids, w, 1, 3, 0.4, 1, 1.0) == ""
    ids = np.array([0, 1, -1])             # one expert too many for this cut
    w = np.concatenate([w_of(np.array([0, 1])), [0.0]])
    assert "top-p" in parity.valid_routing(logits, bias, ids, w, 2, 3, 0.4, 1, 1.0)
    # a cut exactly at the threshold: p * total = cum_1 (0.9 = p * 2.2), so keeping 1 or 2 is
    # valid under the tie margin
    p = 0.9 / 2.2
    for k in (1, 2):
        ids = np.array([0, 1, -1][:k] + [-1] * (3 - k))
        w = np.concatenate([w_of(ids[:k]), np.zeros(3 - k)])
        assert parity.valid_routing(logits, bias, ids, w, k, 3, p, 1, 1.0) == "", k
