"""Parity checks for the two places where floating point decides an integer.

1. Routing.  The router's fp32 logits are summed in another order on the two sides, so a
   token whose decision (the K-th against the (K+1)-th choice, or the top-p cut) lies within
   TIE of a tie may route either way.  Every other token must match the oracle exactly; a
   near-tie token must still be a valid routing under TIE (``valid_routing``).

2. The int8 codes of h = SiLU(gate) * up ["MoE 路由与专家流式加载" §1.3: the down projection
   runs on the integer-dot path too, so h is quantised].  gate and up are fp32 sums of group
   terms in a kernel-specific order, so a code whose pre-rounding value h * 127 / amax lies at
   a .5 boundary may land on either side.  A differing code counts as such a flip only if
   the oracle's pre-rounding value lies within a proven error bound of the boundary between
   the two codes (``h_pre_bound``); the down projection of a row with flips is then checked
   bit for bit against an int64 brute force on the GPU's own codes, and its output against
   the oracle's output moved by exactly those flips.  Layer outputs beyond 1e-3 x RMS must
   be explained by a set of such flips (``explain_token``), found by least squares and
   accepted only with integer (0/1) coefficients and a residual within 1e-3 x RMS.

The error bound.  For one h element with exact integer half-group sums D_h (32 inputs each;
every kernel's fp32 terms are sums over whole halves or groups, and the sum of |terms| over
any such grouping is at most the sum over halves) and group scales s_g:
    E      = sx * sum_h |s_g(h) * D_h|                      (the terms' absolute sum)
    |dgate| <= (depth + 2) u E + u |gate|                   (any summation tree of that depth,
                                                            the token-scale product)
    |dh|   <= |silu'| |dgate| (|up| + |dup|) + |silu| |dup| + 11 u |h|
                                                            (expf within 2 ulp, add, IEEE
                                                            divide and multiply on the GPU;
                                                            the oracle's fp64 h rounded once)
    |dpre| <= (127/amax) |dh| + |pre| max|dh| / (amax - max|dh|) + 4 u |pre|
with u = 2^-24 and depth = groups per row + 16, the deepest fp32 addition chain of the three
FFN kernels (a lane's sequential chain plus the cross-lane and cross-slice adds).  The
expf bound is the CUDA math library's documented 2-ulp maximum error.

Test infrastructure only: imports nothing from the CUDA package.
"""
from __future__ import annotations

import itertools
from typing import Dict, List, Optional, Sequence

import numpy as np

U32 = 2.0 ** -24
TOL = 1e-3        # max-abs error relative to the oracle output's RMS
TIE = 1e-5        # routing margin below which a token is a near tie


def sig64(v):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-np.asarray(v, np.float64)))


def rms(a) -> float:
    return float(np.sqrt(np.mean(np.asarray(a, np.float64) ** 2)))


# ---------------------------------------------------------------------------------- codes

def codes_of(packed) -> np.ndarray:
    """Packed int4 rows [..., K/2] u8 -> signed weights u - 8 [..., K] (element 2j in the low
    nibble of byte j ["colibrì 深度拆解" §5.2], zero point 8 ["colibri 开发演进实录" §2.2])."""
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.int8)
    out[..., 0::2] = (p & 0x0F).astype(np.int8) - 8
    out[..., 1::2] = (p >> 4).astype(np.int8) - 8
    return out


def half_sums(packed, q, chunk: int = 32) -> np.ndarray:
    """Exact sums of (u - 8) * q over every 32-input half group: [nt, rows, K/32] float64
    (integers, exact in fp64).  packed [rows][K/2] u8, q [nt][K] int8."""
    W = codes_of(packed).astype(np.float64)
    rows, K = W.shape
    nh = K // 32
    Wh = W.reshape(rows, nh, 32).transpose(1, 0, 2)            # [nh, rows, 32]
    q = np.asarray(q, np.float64).reshape(-1, nh, 32)
    out = np.empty((q.shape[0], rows, nh))
    for t0 in range(0, q.shape[0], chunk):
        Qh = q[t0:t0 + chunk].transpose(1, 2, 0)               # [nh, 32, nt]
        out[t0:t0 + chunk] = (Wh @ Qh).transpose(2, 1, 0)
    return out


def group_sums_down(packed_down, hq) -> np.ndarray:
    """int64 brute force of the down projection's group sums: [rows, F/64] for one h row."""
    W = codes_of(packed_down).astype(np.int64)
    rows, F = W.shape
    return np.einsum("rgk,gk->rg", W.reshape(rows, F // 64, 64),
                     np.asarray(hq, np.int64).reshape(F // 64, 64))


# ---------------------------------------------------------------------------------- bound

def h_pre_bound(sx, s_gate, Dg, s_up, Du, pre, depth: int) -> np.ndarray:
    """Upper bound on |pre_gpu - pre_oracle| for every h element of nt rows of one expert.

    sx [nt] token scales; s_gate / s_up [F][G] group scales; Dg / Du [nt][F][2G] exact half-
    group sums; pre [nt][F] the oracle's pre-rounding values; depth as in the module text."""
    sx = np.asarray(sx, np.float64)[:, None]

    def side(s, D):
        sh = np.repeat(np.asarray(s, np.float64), 2, axis=1)[None]   # scale of each half
        t = D * sh
        v = sx * t.sum(-1)
        E = sx * np.abs(t).sum(-1)
        return v, (depth + 2) * U32 * E + U32 * np.abs(v)

    gate, bg = side(s_gate, Dg)
    up, bu = side(s_up, Du)
    sg = sig64(gate)
    silu = gate * sg
    dsilu = np.minimum(1.1, np.abs(sg * (1.0 + gate * (1.0 - sg))) + bg)
    h = silu * up
    dh = dsilu * bg * (np.abs(up) + bu) + np.abs(silu) * bu + 11 * U32 * np.abs(h)
    amax = np.abs(h).max(-1, keepdims=True)
    dam = dh.max(-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(amax > 0, 127.0 / amax, 0.0)
        rel = np.where(amax > dam, dam / (amax - dam), np.inf)
    p = np.abs(np.asarray(pre, np.float64))
    return 1.01 * (inv * dh + p * rel) + 4 * U32 * p + 1e-7


def justify_h_flips(hq_gpu, hq_ref, pre, eps, what: str = "h") -> Dict[str, float]:
    """Every code where the GPU and the oracle differ must be one step away and the oracle's
    pre-rounding value must lie within eps of the boundary between the two codes."""
    d = hq_gpu.astype(np.int32) - hq_ref.astype(np.int32)
    assert np.abs(d).max(initial=0) <= 1, "%s: a code differs by %d steps" % (what, np.abs(d).max())
    idx = np.nonzero(d)
    b = hq_ref[idx].astype(np.float64) + 0.5 * d[idx]
    dist = np.abs(np.asarray(pre, np.float64)[idx] - b)
    bound = np.asarray(eps)[idx]
    bad = dist > bound
    assert not bad.any(), ("%s: %d of %d differing codes are not at a rounding boundary "
                           "(worst: %.3g from it, bound %.3g)"
                           % (what, int(bad.sum()), dist.size, dist[bad].max(), bound[bad][np.argmax(dist[bad])]))
    return {"flips": int(dist.size), "max_dist": float(dist.max(initial=0.0)),
            "max_dist_over_bound": float((dist / np.maximum(bound, 1e-30)).max(initial=0.0))}


# ---------------------------------------------------------------------- FFN (with probes)

def check_ffn_pairs(g: Dict[str, np.ndarray], ref: Dict[str, np.ndarray], x, experts: Dict,
                    offsets, tok, xq, sx, report: Optional[list] = None) -> Dict[str, int]:
    """moe_expert_ffn outputs with probes (``g``) against the oracle's (``ref``).

    Exact: acc_gate and acc_up everywhere; acc_down on rows whose h codes match the oracle's.
    Justified: every differing h code (``justify_h_flips``); acc_down of such rows equals an
    int64 brute force on the GPU's codes; every output row within TOL x RMS of the oracle's
    output moved by exactly the flipped codes' contribution."""
    assert np.array_equal(g["acc_gate"], ref["acc_gate"]), "acc_gate differs"
    assert np.array_equal(g["acc_up"], ref["acc_up"]), "acc_up differs"
    np.testing.assert_allclose(g["h_scale"], ref["hs"], rtol=1e-5)
    offsets = np.asarray(offsets)
    E = offsets.size - 1
    y_exp = np.array(ref["y_pairs"], np.float64, copy=True)
    flips = rows_flipped = 0
    worst = dmax = 0.0
    for e in range(E):
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        if p1 == p0:
            continue
        diff = np.any(g["hq"][p0:p1] != ref["hq"][p0:p1], axis=1)
        same = ~diff
        assert np.array_equal(g["acc_down"][p0:p1][same], ref["acc_down"][p0:p1][same]), \
            "acc_down differs on rows with identical h codes (expert %d)" % e
        if not diff.any():
            continue
        ps = p0 + np.nonzero(diff)[0]
        tks = np.asarray(tok)[ps]
        G = experts["s_gate"].shape[-1]
        Dg = half_sums(experts["w_gate"][e], xq[tks])
        Du = half_sums(experts["w_up"][e], xq[tks])
        eps = h_pre_bound(sx[tks], experts["s_gate"][e], Dg, experts["s_up"][e], Du,
                          ref["h_pre"][ps], depth=G + 16)
        r = justify_h_flips(g["hq"][ps], ref["hq"][ps], ref["h_pre"][ps], eps, "expert %d" % e)
        flips += r["flips"]
        rows_flipped += len(ps)
        worst = max(worst, r["max_dist_over_bound"])
        dmax = max(dmax, r["max_dist"])
        sd = np.asarray(experts["s_down"][e], np.float64)
        for p in ps:
            A = group_sums_down(experts["w_down"][e], g["hq"][p])
            assert np.array_equal(g["acc_down"][p], A), "acc_down of pair %d differs from the brute force" % p
            dA = A - ref["acc_down"][p].astype(np.int64)
            y_exp[p] += float(ref["hs"][p]) * (sd * dA).sum(-1)
    err = np.abs(np.asarray(g["y"], np.float64) - y_exp).max(initial=0.0) / max(rms(ref["y_pairs"]), 1e-30)
    assert err <= TOL, "y_pairs beyond %.0e x RMS after accounting for the h-code flips: %.3g" % (TOL, err)
    out = {"h_flips": flips, "rows_with_flips": rows_flipped}
    if report is not None:
        report.append(dict(out, max_dist=dmax, max_dist_over_bound=round(worst, 4), y_err=err))
    print("h-code flips justified: %d codes in %d rows (largest distance of a flipped value from "
          "its boundary %.2g code steps, %.3f of its bound); y within %.2e x RMS"
          % (flips, rows_flipped, dmax, worst, err))
    return out


# ------------------------------------------------------------------------- layer outputs

def layer_reference(oracle, cfg, x, ids, w, keff, routed: Dict, shared: Optional[Dict]):
    """The oracle's layer output for tokens x with the given routing, plus what
    ``explain_tokens`` needs: every pair's h codes, their pre-rounding values and the x
    codes.  routed / shared: host weight dicts ([E, ...] and [1, ...] or [...])."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    T = x.shape[0]
    perm = oracle.permute(cfg, ids, keff)
    ffn = oracle.expert_ffn(cfg, x, routed, perm["offsets"], perm["tok"], probes=True)
    xq, sx = oracle.quant_rows(x)
    out = {"perm": perm, "ffn": ffn, "xq": xq, "sx": sx, "routed": routed, "shared": None,
           "w": np.asarray(w, np.float32), "keff": np.asarray(keff), "K": cfg.top_k}
    ys = None
    if shared is not None:
        sh = {k: (np.asarray(v)[0] if np.asarray(v).ndim == 3 else np.asarray(v))[None]
              for k, v in shared.items()}
        Fs = sh["w_gate"].shape[1]
        csh = oracle.make_config(cfg.hidden, 1, 1, Fs)
        sf = oracle.expert_ffn(csh, x, sh, np.array([0, T], np.int32), np.arange(T, dtype=np.int32),
                               probes=True)
        ys = sf["y_pairs"]
        out["shared"] = sh
        out["sffn"] = sf
    out["y"] = oracle.combine(cfg, ffn["y_pairs"], perm["slot"], perm["offsets"], w, keff, ys)
    return out


def _flip_columns(L, e_weights, row_probe, xq_t, sx_t, weight):
    """Candidate h-code flips of one (token, expert) row and each one's effect on the
    token's output: columns [H, n] and the candidates' distance / bound."""
    W = e_weights
    G = W["s_gate"].shape[-1]
    Dg = half_sums(W["w_gate"], xq_t[None])
    Du = half_sums(W["w_up"], xq_t[None])
    pre = row_probe["h_pre"][None]
    eps = h_pre_bound(np.array([sx_t]), W["s_gate"], Dg, W["s_up"], Du, pre, depth=G + 16)[0]
    q = row_probe["hq"].astype(np.float64)
    off = pre[0].astype(np.float64) - q
    dist = 0.5 - np.abs(off)                 # distance of the value to the nearest boundary
    cand = np.nonzero((dist <= eps) & (off != 0.0))[0]
    if cand.size == 0:
        return np.zeros((W["s_down"].shape[0], 0)), cand
    sgn = np.sign(off[cand])                 # the neighbouring code lies on this side
    U = codes_of(W["w_down"]).astype(np.float64)[:, cand]            # [H, n]
    sd = np.asarray(W["s_down"], np.float64)[:, cand // 64]          # [H, n]
    cols = weight * float(row_probe["hs"]) * sd * U * sgn[None]
    return cols, cand


def explain_tokens(y_gpu, L, tokens: Sequence[int], ref_rms: Optional[float] = None,
                   what: str = "layer") -> Dict[str, int]:
    """Every listed token's GPU output must lie within TOL x RMS of the oracle's, or be the
    oracle's output moved by a set of justified h-code flips (0/1 least-squares coefficients,
    residual within TOL x RMS).  Returns the counts."""
    y_ref = L["y"]
    R = ref_rms if ref_rms is not None else rms(y_ref[list(tokens)])
    perm, ffn, K = L["perm"], L["ffn"], L["K"]
    pair_of = {}
    for p, s in enumerate(perm["slot"]):
        pair_of[int(s)] = p
    offsets = perm["offsets"]
    exp_of = np.searchsorted(offsets, np.arange(len(perm["tok"])), side="right") - 1
    n_over = n_explained = n_flips = 0
    for t in tokens:
        r = np.asarray(y_gpu[t], np.float64) - y_ref[t]
        if np.abs(r).max() <= TOL * R:
            continue
        n_over += 1
        cols = []
        for i in range(int(L["keff"][t])):
            p = pair_of[t * K + i]
            e = int(exp_of[p])
            We = {k: np.asarray(v[e]) for k, v in L["routed"].items()}
            probe = {"hq": ffn["hq"][p], "hs": ffn["hs"][p], "h_pre": ffn["h_pre"][p]}
            c, _ = _flip_columns(L, We, probe, L["xq"][t], L["sx"][t], float(L["w"][t, i]))
            cols.append(c)
        if L["shared"] is not None:
            sf = L["sffn"]
            Ws = {k: np.asarray(v[0]) for k, v in L["shared"].items()}
            probe = {"hq": sf["hq"][t], "hs": sf["hs"][t], "h_pre": sf["h_pre"][t]}
            c, _ = _flip_columns(L, Ws, probe, L["xq"][t], L["sx"][t], 1.0)
            cols.append(c)
        D = np.concatenate(cols, axis=1) if cols else np.zeros((r.size, 0))
        assert D.shape[1] > 0, ("%s: token %d is %.3g x RMS off and has no h code at a rounding "
                                "boundary" % (what, t, np.abs(r).max() / R))
        c, *_ = np.linalg.lstsq(D, r, rcond=None)
        cr = np.clip(np.rint(c), 0, 1)
        resid = np.abs(r - D @ cr).max() / R
        assert np.abs(c - cr).max() <= 0.3 and resid <= TOL, (
            "%s: token %d (%.3g x RMS off) is not explained by flips of its %d boundary codes "
            "(coefficient off by %.2f, residual %.3g x RMS)"
            % (what, t, np.abs(r).max() / R, D.shape[1], np.abs(c - cr).max(), resid))
        n_explained += 1
        n_flips += int(cr.sum())
    print("%s: %d of %d tokens beyond %.0e x RMS, each explained by justified h-code flips "
          "(%d flips)" % (what, n_over, len(tokens), TOL, n_flips))
    return {"tokens_over": n_over, "explained": n_explained, "flips": n_flips}


# --------------------------------------------------------------------------------- routing

def routing_margins(logits, bias, K: int, top_p: float) -> np.ndarray:
    """Per token, the smallest distance (fp64) of any decision the router takes to its tie
    point: between consecutive choices among the top K+1, and, with top-p, between sorted
    gates and between the running gate sum and p * total at every position."""
    choice = sig64(logits) + np.asarray(bias, np.float64)[None, :]
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


def valid_routing(logits_t, bias, ids, w, keff, K, top_p, norm, scale, eps=TIE):
    """Is (ids, w, keff) of one token a correct routing when every choice, gate and running
    sum may move by eps ["MoE 路由与专家流式加载" §1.1, §1.2]?  Returns '' or the reason."""
    gate = sig64(logits_t)
    choice = gate + np.asarray(bias, np.float64)
    E = choice.size
    k = int(keff)
    if not 1 <= k <= K:
        return "keff %d outside [1, %d]" % (k, K)
    kept = [int(e) for e in ids[:k]]
    if len(set(kept)) != k or min(kept) < 0 or max(kept) >= E:
        return "kept ids not distinct or out of range"
    if np.any(np.asarray(ids[k:]) != -1) or np.any(np.asarray(w[k:]) != 0):
        return "slots past keff not cleared"
    order = np.argsort(-choice, kind="stable")
    cK = choice[order[K - 1]]
    if np.any(choice[kept] < cK - eps):
        return "a kept expert is not among the top K"
    topp = 0.0 < top_p < 1.0
    if not topp:
        if k != K:
            return "keff %d without top-p" % k
        if np.any(np.diff(choice[kept]) > eps):
            return "ids not in descending choice order"
        S_ok = True
    else:
        gk = gate[kept]
        if np.any(np.diff(gk) > eps):
            return "kept ids not in descending gate order"
        definite = [int(e) for e in order if choice[e] > cK + eps and int(e) not in kept]
        band = [int(e) for e in order if abs(choice[e] - cK) <= eps and int(e) not in kept
                and int(e) not in definite]
        need = K - k - len(definite)
        S_ok = False
        if need >= 0:
            for extra in itertools.combinations(band, need):
                rest = definite + list(extra)
                if rest and gate[rest].max() > gk.min() + eps:
                    continue
                g_all = np.concatenate([gk, np.sort(gate[rest])[::-1]]) if rest else gk
                cum = np.cumsum(g_all)
                thr = top_p * cum[-1]
                prev = cum[k - 2] if k >= 2 else 0.0
                if prev < thr + K * eps and cum[k - 1] >= thr - K * eps:
                    S_ok = True
                    break
        if not S_ok:
            return "no valid top-K set whose top-p cut keeps these %d experts" % k
    gk = gate[kept]
    w_exp = (gk / gk.sum() if norm else gk) * scale
    if not np.allclose(np.asarray(w[:k], np.float64), w_exp, rtol=1e-4, atol=1e-7):
        return "applied weights differ from the gates of the kept experts"
    return ""


def check_routing(gpu, ref_ids, ref_w, ref_keff, logits, bias, K, top_p, norm, scale,
                  tie=TIE) -> int:
    """Exact ids / keff (and w within rtol 2e-5) on every token whose margin exceeds tie;
    a valid routing under tie on the rest.  Returns the number of near-tie tokens."""
    ids, w, keff = gpu
    margin = routing_margins(logits, bias, K, top_p)
    clear = margin > tie
    assert np.array_equal(ids[clear], ref_ids[clear]), "ids differ on tokens away from ties"
    assert np.array_equal(keff[clear], ref_keff[clear]), "keff differs on tokens away from ties"
    np.testing.assert_allclose(w[clear], ref_w[clear], rtol=2e-5, atol=1e-7)
    for t in np.nonzero(~clear)[0]:
        why = valid_routing(logits[t], bias, ids[t], w[t], keff[t], K, top_p, norm, scale, tie)
        assert not why, "near-tie token %d: %s" % (t, why)
    return int((~clear).sum())
