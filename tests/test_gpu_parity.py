"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Bars: selected expert ids, keff, per-expert token lists, unique lists and int32
per-group accumulators exact; fp32 outputs within max-abs 1e-3 x RMS of the
oracle's output.  Where floating point decides an integer, ``parity`` compares
what is unique and proves the rest valid: a token whose routing decision sits
within 1e-5 of a tie must still be a valid routing under that margin (the tiny
workload must have none), and an int8 code of h that differs from the oracle's
must sit at a rounding boundary within a proven error bound, with its effect on
the down accumulators and on the output accounted for exactly.  Downstream
calls are fed the oracle's routing, never the other way round.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
import parity
from helpers import device_experts, host_experts, moe_cfg, oracle_tokens, rel_err
from parity import TIE, TOL, routing_margins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_expert_ffn_route_gb300 as m
    m.load_library()
    return m


def _inputs(wl, T, batch=0):
    x = synth.gen_x(wl, T, batch)
    wr, bias = synth.gen_router(wl)
    return x, wr, bias


def _route_both(moe, wl, T, batch=0):
    x, wr, bias = _inputs(wl, T, batch)
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    K = wl.top_k
    ids = torch.empty(T, K, dtype=torch.int32, device="cuda")
    w = torch.empty(T, K, dtype=torch.float32, device="cuda")
    keff = torch.empty(T, dtype=torch.int32, device="cuda")
    moe.moe_route(cfg, x.cuda(), wr.cuda(), bias.cuda(), ids, w, keff, ws)
    torch.cuda.synchronize()
    ref = oracle.route(oracle.config_of(wl), x, wr, bias, with_logits=True)
    margin = routing_margins(ref["logits"], bias.numpy(), K, wl.top_p)
    return x, wr, bias, (ids.cpu().numpy(), w.cpu().numpy(), keff.cpu().numpy()), ref, margin


def _check_routing(wl, gpu, ref, bias):
    """Exact routing away from ties, a valid routing under the tie margin at them."""
    return parity.check_routing(gpu, ref["ids"], ref["w"], ref["keff"], ref["logits"],
                                np.asarray(bias), wl.top_k, wl.top_p, wl.norm_topk_prob,
                                wl.routed_scaling_factor)


# (a3b 45 and 64: the route tail selects over several CTAs, the last one ragged at 45)
ROUTE_CASES = [("tiny", 16), ("tiny", 1), ("a3b_decode", 45), ("a3b_decode", 64), ("glm_decode", 1),
               ("glm_decode", 32), ("wide", 8), ("wide", 512), ("prefill", 4096)]


@pytest.mark.parametrize("name,T", ROUTE_CASES)
def test_route(moe, name, T):
    wl = synth.WORKLOADS[name]
    _, _, bias, gpu, ref, margin = _route_both(moe, wl, T)
    near = _check_routing(wl, gpu, ref, bias)
    print("%s T=%d: %d near-tie token(s), each a valid routing" % (name, T, near))
    if name == "tiny":
        assert near == 0
    assert near <= max(1, T // 50)


def test_route_top_p_variants(moe):
    from dataclasses import replace
    base = synth.WORKLOADS["a3b_decode"]
    for top_p, norm, scale, K in ((0.5, 1, 1.0, 8), (0.9, 0, 2.5, 6), (0.0, 1, 1.0, 16),
                                  (0.3, 1, 1.0, 1)):
        wl = replace(base, top_p=top_p, norm_topk_prob=norm, routed_scaling_factor=scale,
                     top_k=K)
        _, _, bias, gpu, ref, margin = _route_both(moe, wl, 200)
        assert _check_routing(wl, gpu, ref, bias) <= 4


def _permute_gpu(moe, wl, ids, keff):
    T, K, E = keff.shape[0], wl.top_k, wl.n_experts
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    d = dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
             offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
             tok=torch.full((max(T * K, 1),), -7, dtype=torch.int32, device="cuda"),
             slot=torch.full((max(T * K, 1),), -7, dtype=torch.int32, device="cuda"),
             uniq=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
             n_uniq=torch.empty(1, dtype=torch.int32, device="cuda"))
    moe.moe_permute(cfg, torch.from_numpy(ids).cuda(), torch.from_numpy(keff).cuda(),
                    d["counts"], d["offsets"], d["tok"], d["slot"], d["uniq"], d["n_uniq"], ws)
    moe.moe_check_errors(ws)
    return {k: v.cpu().numpy() for k, v in d.items()}, ws


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 0), ("a3b_decode", 64),
                                    ("glm_decode", 32), ("prefill", 4096), ("wide", 8192)])
def test_permute(moe, name, T):
    wl = synth.WORKLOADS[name]
    x, wr, bias = _inputs(wl, max(T, 1))
    ref_r = oracle.route(oracle.config_of(wl), x[:T], wr, bias)
    g, _ = _permute_gpu(moe, wl, ref_r["ids"], ref_r["keff"])
    ref = oracle.permute(oracle.config_of(wl), ref_r["ids"], ref_r["keff"])
    P = int(ref["offsets"][-1])
    assert np.array_equal(g["counts"], ref["counts"])
    assert np.array_equal(g["offsets"], ref["offsets"])
    assert np.array_equal(g["tok"][:P], ref["tok"]) and np.array_equal(g["slot"][:P], ref["slot"])
    assert int(g["n_uniq"][0]) == ref["n_uniq"]
    assert np.array_equal(g["uniq"][:ref["n_uniq"]], ref["uniq"])
    if P < g["tok"].size:
        assert np.all(g["tok"][P:] == -7)   # entries past offsets[E] untouched


def test_permute_skewed_and_invalid(moe):
    wl = synth.Workload("skew", 64, 16, 4, 64, 0, 0, (3000,))
    rng = np.random.default_rng(0)
    T, K = 3000, 4
    ids = np.stack([rng.permutation(16)[:K] for _ in range(T)]).astype(np.int32)
    ids[:1500, 0] = 3                     # one expert takes half the tokens first
    for t in range(1500):
        if 3 in ids[t, 1:]:
            ids[t, 1:] = [e for e in rng.permutation(16) if e != 3][:K - 1]
    keff = rng.integers(1, K + 1, T).astype(np.int32)
    for t in range(T):
        ids[t, keff[t]:] = -1
    g, _ = _permute_gpu(moe, wl, ids, keff)
    ref = oracle.permute(oracle.config_of(wl), ids, keff)
    P = int(ref["offsets"][-1])
    assert np.array_equal(g["offsets"], ref["offsets"])
    assert np.array_equal(g["tok"][:P], ref["tok"]) and np.array_equal(g["slot"][:P], ref["slot"])
    # an id out of range is skipped and reported, without a fault
    bad = ids.copy()
    bad[5, 0] = 99
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    dev = {k: torch.zeros(n, dtype=torch.int32, device="cuda")
           for k, n in (("c", 16), ("o", 17), ("t", T * K), ("s", T * K), ("u", 16), ("n", 1))}
    moe.moe_permute(cfg, torch.from_numpy(bad).cuda(), torch.from_numpy(keff).cuda(), dev["c"],
                    dev["o"], dev["t"], dev["s"], dev["u"], dev["n"], ws)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_check_errors(ws)
    assert ei.value.code == moe.MOE_ERR_DEVICE
    moe.moe_check_errors(ws)   # the record is cleared
    assert int(dev["o"][-1]) == P - 1


def _ffn_both(moe, wl, T, batch=0, probes=True, routing=None):
    """GPU moe_expert_ffn on the oracle's routing (or a given (ids, keff)) vs the oracle.
    The oracle's result also carries what the h-code checks need (x, its codes, weights)."""
    x, wr, bias = _inputs(wl, T, batch)
    cfg_r = oracle.config_of(wl)
    r = oracle.route(cfg_r, x, wr, bias) if routing is None else {"ids": routing[0], "keff": routing[1]}
    perm = oracle.permute(cfg_r, r["ids"], r["keff"])
    P, E, H, F = int(perm["offsets"][-1]), wl.n_experts, wl.hidden, wl.d_ff
    R_dev = device_experts(wl)
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    y = torch.full((max(P, 1), H), float("nan"), device="cuda")
    probe = None
    if probes:
        probe = dict(acc_gate=torch.zeros(P, F, H // 64, dtype=torch.int32, device="cuda"),
                     acc_up=torch.zeros(P, F, H // 64, dtype=torch.int32, device="cuda"),
                     acc_down=torch.zeros(P, H, F // 64, dtype=torch.int32, device="cuda"),
                     hq=torch.zeros(P, F, dtype=torch.int8, device="cuda"),
                     h_scale=torch.zeros(P, dtype=torch.float32, device="cuda"))
    moe.moe_expert_ffn(cfg, x.cuda(), R_dev, torch.from_numpy(perm["offsets"]).cuda(),
                       torch.from_numpy(perm["tok"]).cuda(),
                       torch.from_numpy(np.pad(perm["uniq"], (0, E - perm["n_uniq"]))).cuda(),
                       torch.tensor([perm["n_uniq"]], dtype=torch.int32, device="cuda"), y, ws,
                       probe=probe)
    torch.cuda.synchronize()
    R_host = host_experts(wl)
    ref = oracle.expert_ffn(cfg_r, x, R_host, perm["offsets"], perm["tok"], probes=probes)
    ref["x"] = x.numpy()
    ref["xq"], ref["sx"] = oracle.quant_rows(x)
    ref["experts"] = R_host
    g = {k: v.cpu().numpy() for k, v in (probe or {}).items()}
    g["y"] = y[:P].cpu().numpy()
    return g, ref, perm


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 3), ("a3b_decode", 64),
                                    ("a3b_decode", 65), ("a3b_decode", 96), ("a3b_decode", 200)])
def test_expert_ffn_exact_accumulators(moe, name, T):
    wl = synth.WORKLOADS[name]
    g, ref, perm = _ffn_both(moe, wl, T)
    _check_ffn(g, ref, perm)


def test_expert_ffn_exact_accumulators_sliced_warp_gemv(moe):
    """The warp GEMV on 1024-input slices: reductions that are not multiples of 256 (hidden and
    d_ff 1088: a full slice and a ragged one of 2 chunks) keep the row GEMV out, and 8 tokens
    are past the whole-row batches, so gate/up ends in slice planes that the h quantisation
    adds in slice order ["colibri 开发演进实录" §2.2 K1b, per-group int32 dot]."""
    from dataclasses import replace
    wl = replace(synth.WORKLOADS["tiny"], name="sliced", hidden=1088, d_ff=1088, n_shared=0,
                 d_ff_shared=0, n_experts=16, top_k=4)
    T = 8
    assert moe.moe_ffn_path(moe_cfg(wl), T) == moe.MOE_FFN_WARP_GEMV
    g, ref, perm = _ffn_both(moe, wl, T)
    _check_ffn(g, ref, perm)


def test_expert_ffn_exact_accumulators_split_paths(moe):
    """A wide layer past the decode route at about 12 tokens per routed expert: gate/up on the
    row GEMV, down on the tensor path (the paths are chosen per projection)."""
    from dataclasses import replace
    wl = replace(synth.WORKLOADS["wide"], name="split_mid", hidden=1024, d_ff=1024,
                 d_ff_shared=1024, n_experts=64)
    T = 96
    assert moe.moe_ffn_path(moe_cfg(wl), T) == moe.MOE_FFN_ROW_GEMV
    assert moe.moe_ffn_path_down(moe_cfg(wl), T) == moe.MOE_FFN_TENSOR
    g, ref, perm = _ffn_both(moe, wl, T)
    _check_ffn(g, ref, perm)


@pytest.mark.parametrize("T", [24, 64])
def test_expert_ffn_exact_accumulators_row_gemv(moe, T):
    """Row GEMV (decode-sized batch, reductions in multiples of 256) on a mid-sized shape:
    gate/up rows of 2048 inputs take two 1024-input stages, down rows of 768 inputs one stage
    whose last line lies past the row (zero-filled), down tasks take two 64-row blocks, and
    routed experts with more than 8 tokens run in several token chunks."""
    from dataclasses import replace
    wl = replace(synth.WORKLOADS["a3b_decode"], name="rows_mid", hidden=2048, d_ff=768,
                 d_ff_shared=768, n_experts=16, top_k=4)
    assert moe.moe_ffn_path(moe_cfg(wl), T) == moe.MOE_FFN_ROW_GEMV
    g, ref, perm = _ffn_both(moe, wl, T)
    assert np.diff(perm["offsets"]).max() > 8
    _check_ffn(g, ref, perm)


def test_expert_ffn_tensor_tile_edges(moe):
    """Tensor-core path (a3b shape, T = 300) on a constructed routing: experts with 129 tokens
    (a full 128-token tile plus a one-token tile), exactly 128, 127, 1 and 0 tokens."""
    wl = synth.WORKLOADS["a3b_decode"]
    T, K, E = 300, wl.top_k, wl.n_experts
    ids = np.full((T, K), -1, np.int32)
    keff = np.full(T, K, np.int32)
    for t in range(T):
        row = [8 + (t * 7 + 3 * i) % (E - 8) for i in range(K)]
        ids[t] = row
    ids[:129, 0] = 0          # expert 0: tokens 0..128
    ids[:128, 1] = 1          # expert 1: tokens 0..127
    ids[150:277, 0] = 2       # expert 2: 127 tokens
    ids[299, 1] = 3           # expert 3: one token; expert 4..7: none
    for t in range(T):        # keep every row's ids distinct after the overrides
        seen = set()
        for i in range(K):
            while ids[t, i] in seen:
                ids[t, i] = 8 + (ids[t, i] - 8 + 1) % (E - 8)
            seen.add(int(ids[t, i]))
    keff[::17] = 5            # some shorter kept sets
    ids[::17, 5:] = -1
    g, ref, perm = _ffn_both(moe, wl, T, routing=(ids, keff))
    cnt = np.diff(perm["offsets"])
    assert cnt[0] == 129 and cnt[1] == 128 and cnt[2] >= 127 and cnt[3] >= 1 and (cnt[4:8] == 0).all()
    _check_ffn(g, ref, perm)


def _check_ffn(g, ref, perm):
    """Exact gate/up accumulators; every differing h code justified; down accumulators exact
    (oracle's on matching rows, int64 brute force on the GPU's codes elsewhere); outputs within
    1e-3 x RMS of the oracle's, moved by exactly the justified flips."""
    return parity.check_ffn_pairs(g, ref, ref["x"], ref["experts"], perm["offsets"], perm["tok"],
                                  ref["xq"], ref["sx"])


@pytest.mark.parametrize("T", [2, 3])
def test_expert_ffn_glm_full_width(moe, T):
    """Full GLM-decode widths (H=6144, F=2048) at the two sides of the warp / row GEMV
    crossover: T=2 the warp GEMV (whole rows), T=3 the row GEMV."""
    wl = replace(synth.WORKLOADS["glm_decode"], n_experts=48)
    want = moe.MOE_FFN_WARP_GEMV if T < 3 else moe.MOE_FFN_ROW_GEMV
    assert moe.moe_ffn_path(moe_cfg(wl), T) == want
    g, ref, perm = _ffn_both(moe, wl, T)
    _check_ffn(g, ref, perm)


def test_expert_ffn_exact_accumulators_glm_row_gemv(moe):
    """The benchmarked decode kernel at the shape it runs at: the row GEMV on GLM widths
    (H=6144, F=2048) with T=32 tokens over 32 experts, so experts receive more than 8 tokens
    and run in several token chunks ["colibri 开发演进实录" §2.2 K1b, per-group int32 dot]."""
    wl = replace(synth.WORKLOADS["glm_decode"], n_experts=32)
    T = 32
    assert moe.moe_ffn_path(moe_cfg(wl), T) == moe.MOE_FFN_ROW_GEMV
    g, ref, perm = _ffn_both(moe, wl, T)
    assert np.diff(perm["offsets"]).max() > 8
    _check_ffn(g, ref, perm)


def test_expert_ffn_exact_accumulators_glm_tensor(moe):
    """The tcgen05 grouped GEMM at prefill widths (H=6144, F=2048): 32 experts, 320 tokens,
    top-2, a skewed routing in which expert 0 takes 300 tokens (two full 128-token tiles and a
    44-token tile), expert 1 takes 257 (two full tiles and a one-token tile), and the rest
    follow a Zipf(1.1) popularity, some with no token at all."""
    wl = replace(synth.WORKLOADS["prefill"], n_experts=32, top_k=2)
    T, K, E = 320, 2, 32
    assert moe.moe_ffn_path(moe_cfg(wl), T) == moe.MOE_FFN_TENSOR
    rng = np.random.default_rng(7)
    p = 1.0 / np.arange(1, E - 1, dtype=np.float64) ** 1.1
    p /= p.sum()
    ids = np.empty((T, K), np.int32)
    for t in range(T):
        a = 0 if t < 300 else 2 + int(rng.choice(E - 2, p=p))
        b = 1 if 20 <= t < 277 else 2 + int(rng.choice(E - 2, p=p))
        while b == a:
            b = 2 + int(rng.choice(E - 2, p=p))
        ids[t] = (a, b)
    keff = np.full(T, K, np.int32)
    g, ref, perm = _ffn_both(moe, wl, T, routing=(ids, keff))
    cnt = np.diff(perm["offsets"])
    assert cnt[0] == 300 and cnt[1] == 257 and (cnt == 0).any()
    _check_ffn(g, ref, perm)


def _layer_gpu(moe, wl, x, wr, bias, routing=True):
    T, K = x.shape[0], wl.top_k
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    y = torch.full((T, wl.hidden), float("nan"), device="cuda")
    rt = dict(ids=torch.empty(T, K, dtype=torch.int32, device="cuda"),
              w=torch.empty(T, K, dtype=torch.float32, device="cuda"),
              keff=torch.empty(T, dtype=torch.int32, device="cuda"))
    moe.moe_layer_forward(cfg, x.cuda(), wr.cuda(), bias.cuda(), device_experts(wl),
                          device_experts(wl, shared=True) if wl.n_shared else None, y, ws,
                          routing=rt, flags=moe.MOE_FLAG_SYNC_CHECK)
    return y.cpu().numpy(), {k: v.cpu().numpy() for k, v in rt.items()}


def _check_layer(wl, x, wr, bias, y, rt, routed=None, shared=None, what="layer"):
    """A layer call's routing against the oracle's (exact away from ties, valid at them) and
    its outputs on every token away from a tie: within 1e-3 x RMS of the oracle's, or
    explained exactly by justified h-code flips.  routed / shared: host weights (default:
    the workload's generated experts)."""
    cfg = oracle.config_of(wl)
    r = oracle.route(cfg, x, wr, bias, with_logits=True)
    near = _check_routing(wl, (rt["ids"], rt["w"], rt["keff"]), r, bias)
    assert np.isfinite(y).all()
    clear = routing_margins(r["logits"], bias.numpy(), wl.top_k, wl.top_p) > TIE
    R = host_experts(wl) if routed is None else {k: np.asarray(v) for k, v in routed.items()}
    S = None
    if wl.n_shared:
        S = host_experts(wl, shared=True) if shared is None else {k: np.asarray(v) for k, v in shared.items()}
    L = parity.layer_reference(oracle, cfg, x, r["ids"], r["w"], r["keff"], R, S)
    toks = np.nonzero(clear)[0]
    out = parity.explain_tokens(y, L, toks, ref_rms=parity.rms(L["y"][toks]), what=what)
    return near, out


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 1), ("tiny", 45), ("a3b_decode", 64),
                                    ("a3b_decode", 128)])
def test_layer_forward(moe, name, T):
    wl = synth.WORKLOADS[name]
    x, wr, bias = _inputs(wl, T)
    y, rt = _layer_gpu(moe, wl, x, wr, bias)
    near, _ = _check_layer(wl, x, wr, bias, y, rt, what="%s T=%d" % (name, T))
    if name == "tiny":
        assert near == 0


@pytest.mark.parametrize("name,T,sample", [("glm_decode", 1, [0]), ("glm_decode", 2, [0, 1]),
                                           ("glm_decode", 32, [0, 13, 31]),
                                           ("glm_decode", 128, [0, 77, 127]),
                                           ("wide", 64, [0, 40]), ("prefill", 4096, [0, 2047, 4095])])
def test_layer_forward_full_size_sampled(moe, name, T, sample):
    """Full-size layer through moe_layer_forward (the call the benchmark times); routing of
    every token against the oracle, outputs of sampled tokens against the oracle run on just
    the experts those tokens use."""
    wl = synth.WORKLOADS[name]
    x, wr, bias = _inputs(wl, T)
    y, rt = _layer_gpu(moe, wl, x, wr, bias)
    assert np.isfinite(y).all()
    ref = oracle.route(oracle.config_of(wl), x, wr, bias, with_logits=True)
    margin = routing_margins(ref["logits"], bias.numpy(), wl.top_k, wl.top_p)
    _check_routing(wl, (rt["ids"], rt["w"], rt["keff"]), ref, bias)
    rows = [t for t in sample if margin[t] > TIE]
    assert rows
    L = oracle_tokens(wl, x.numpy()[rows], ref["ids"][rows], ref["w"][rows], ref["keff"][rows])
    parity.explain_tokens(y[rows], L, range(len(rows)), what="%s T=%d sampled" % (name, T))


def test_combine_with_shared(moe):
    wl = synth.WORKLOADS["tiny"]
    T = 16
    x, wr, bias = _inputs(wl, T)
    cfg_r = oracle.config_of(wl)
    r = oracle.route(cfg_r, x, wr, bias)
    perm = oracle.permute(cfg_r, r["ids"], r["keff"])
    ffn = oracle.expert_ffn(cfg_r, x, synth.gen_experts(wl), perm["offsets"], perm["tok"])
    S = synth.gen_experts(wl, shared=True)
    ys = oracle.shared_ffn(cfg_r, x, S)
    ref = oracle.combine(cfg_r, ffn["y_pairs"], perm["slot"], perm["offsets"], r["w"], r["keff"], ys)
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    y = torch.empty(T, wl.hidden, device="cuda")
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    moe.moe_combine(cfg, cu(ffn["y_pairs"].astype(np.float32)), cu(r["ids"]), cu(r["keff"]),
                    cu(r["w"]), cu(perm["offsets"]), cu(perm["tok"]), y, ws, x=x.cuda(),
                    shared=device_experts(wl, shared=True))
    assert rel_err(y.cpu().numpy(), ref) <= TOL
    # without the shared expert
    ref0 = oracle.combine(cfg_r, ffn["y_pairs"], perm["slot"], perm["offsets"], r["w"], r["keff"])
    moe.moe_combine(cfg, cu(ffn["y_pairs"].astype(np.float32)), cu(r["ids"]), cu(r["keff"]),
                    cu(r["w"]), cu(perm["offsets"]), cu(perm["tok"]), y, ws)
    assert rel_err(y.cpu().numpy(), ref0) <= TOL


EDGE = [
    # name, H, E, K, F, ns, Fs, T, top_p, norm, scale
    ("dense_E1", 256, 1, 1, 192, 0, 0, 33, 0.0, 1, 1.0),
    ("H64_tiny_groups", 64, 4, 2, 64, 1, 128, 9, 0.0, 1, 1.0),
    ("ragged_odd_groups", 704, 12, 3, 320, 1, 192, 37, 0.6, 0, 2.5),
    ("K_equals_E", 128, 4, 4, 128, 0, 0, 10, 0.0, 1, 1.0),
    ("one_token", 512, 64, 8, 256, 1, 256, 1, 0.7, 1, 2.5),
    ("wide_groups", 7168, 16, 4, 192, 1, 64, 5, 0.0, 1, 1.0),
    # routed rows of 6 chunks beside shared rows of 64: one down launch serves both widths
    ("mixed_widths", 256, 8, 2, 192, 1, 2048, 12, 0.0, 1, 1.0),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: c[0])
def test_edge_cases(moe, case):
    name, H, E, K, F, ns, Fs, T, top_p, norm, scale = case
    wl = synth.Workload(name, H, E, K, F, ns, Fs, (T,), norm, scale, top_p, 0.3)
    x, wr, bias = _inputs(wl, T)
    y, rt = _layer_gpu(moe, wl, x, wr, bias)
    _check_layer(wl, x, wr, bias, y, rt, what=name)
    g, refp, perm = _ffn_both(moe, wl, T)
    _check_ffn(g, refp, perm)


def test_zero_tokens_and_deterministic(moe):
    wl = synth.WORKLOADS["tiny"]
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, 16)
    x = torch.empty(0, wl.hidden, device="cuda")
    y = torch.empty(0, wl.hidden, device="cuda")
    wr, bias = synth.gen_router(wl)
    moe.moe_layer_forward(cfg, x, wr.cuda(), bias.cuda(), device_experts(wl),
                          device_experts(wl, shared=True), y, ws, flags=moe.MOE_FLAG_SYNC_CHECK)
    x, wr, bias = _inputs(wl, 16)
    y1, _ = _layer_gpu(moe, wl, x, wr, bias)
    y2, _ = _layer_gpu(moe, wl, x, wr, bias)
    assert np.array_equal(y1, y2)


def test_generator_identical_on_gpu(moe):
    wl = synth.WORKLOADS["a3b_decode"]
    d = device_experts(wl)
    h = synth.gen_experts(wl, experts=[0, 77, 255])
    for k in h:
        assert torch.equal(d[k][[0, 77, 255]].cpu(), h[k])


# ----------------------------------------------------------------------------------------------
# Router look-ahead ["MoE 路由与专家流式加载" §5]: RMSNorm of a residual state, then the router.
# ----------------------------------------------------------------------------------------------

LOOKAHEAD_CASES = [("tiny", 16), ("glm_decode", 1), ("glm_decode", 32), ("a3b_decode", 64),
                   ("wide", 512), ("prefill", 4096)]


@pytest.mark.parametrize("name,T", LOOKAHEAD_CASES)
def test_route_lookahead(moe, name, T):
    wl = synth.WORKLOADS[name]
    h, g, wr, bias = synth.gen_lookahead(wl, T, batch=1)
    eps = 1e-5
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    K = wl.top_k
    ids = torch.empty(T, K, dtype=torch.int32, device="cuda")
    w = torch.empty(T, K, dtype=torch.float32, device="cuda")
    keff = torch.empty(T, dtype=torch.int32, device="cuda")
    moe.moe_route_lookahead(cfg, h.cuda(), g.cuda(), eps, wr.cuda(), bias.cuda(), ids, w, keff, ws)
    torch.cuda.synchronize()
    ref = oracle.route_lookahead(oracle.config_of(wl), h, g, eps, wr, bias, with_logits=True)
    near = _check_routing(wl, (ids.cpu().numpy(), w.cpu().numpy(), keff.cpu().numpy()), ref, bias)
    if name == "tiny":
        assert near == 0
    assert near <= max(1, T // 50)


def test_route_lookahead_zero_rows_and_eps(moe):
    # all-zero rows normalise to zeros (mean square + eps = 0 with eps 0): every logit is 0,
    # so the choice is the bias alone on both sides
    wl = synth.WORKLOADS["tiny"]
    h, g, wr, bias = synth.gen_lookahead(wl, 8)
    h[2] = 0.0
    h[5] = 0.0
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, 8)
    K = wl.top_k
    for eps in (0.0, 0.25):
        ids = torch.empty(8, K, dtype=torch.int32, device="cuda")
        w = torch.empty(8, K, dtype=torch.float32, device="cuda")
        keff = torch.empty(8, dtype=torch.int32, device="cuda")
        moe.moe_route_lookahead(cfg, h.cuda(), g.cuda(), eps, wr.cuda(), bias.cuda(), ids, w, keff, ws)
        ref = oracle.route_lookahead(oracle.config_of(wl), h, g, eps, wr, bias, with_logits=True)
        assert np.array_equal(ids.cpu().numpy(), ref["ids"])
        assert np.array_equal(keff.cpu().numpy(), ref["keff"])
        np.testing.assert_allclose(w.cpu().numpy(), ref["w"], rtol=2e-5, atol=1e-7)
    with pytest.raises(moe.MoeError):
        moe.moe_route_lookahead(cfg, h.cuda(), g.cuda(), -1.0, wr.cuda(), bias.cuda(), ids, w, keff, ws)


def test_topk_hits(moe):
    # the look-ahead prediction against the routing of a later state (the same state plus a
    # perturbation), and against itself: integer counts, compared exactly
    wl = synth.WORKLOADS["glm_decode"]
    T, K = 32, wl.top_k
    h, g, wr, bias = synth.gen_lookahead(wl, T, batch=2)
    pert, _, _, _ = synth.gen_lookahead(wl, T, batch=3)
    cfg = oracle.config_of(wl)
    pred = oracle.route_lookahead(cfg, h, g, 1e-5, wr, bias)
    true = oracle.route_lookahead(cfg, h + 0.5 * pert, g, 1e-5, wr, bias)
    true["keff"][::5] = np.minimum(true["keff"][::5], 3)   # some shorter kept sets
    mcfg = moe_cfg(wl)
    for (ip, kp, it, kt) in ((pred["ids"], pred["keff"], true["ids"], true["keff"]),
                             (pred["ids"], pred["keff"], pred["ids"], pred["keff"])):
        hits = torch.full((T,), -9, dtype=torch.int32, device="cuda")
        moe.moe_topk_hits(mcfg, torch.from_numpy(ip).cuda(), torch.from_numpy(kp).cuda(),
                          torch.from_numpy(it).cuda(), torch.from_numpy(kt).cuda(), hits)
        assert np.array_equal(hits.cpu().numpy(), oracle.topk_hits(ip, kp, it, kt))


# ----------------------------------------------------------------------------------------------
# Offline fp32 -> int4-gs64 weight quantiser ("colibri 开发演进实录" §2.1): codes and scales are
# single-rounded fp32 operations on both sides, so they must agree bit for bit.
# ----------------------------------------------------------------------------------------------

def _quantize_gpu(moe, w):
    rows, K = w.shape
    packed = torch.full((rows, K // 2), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows, K // 64), -1.0, dtype=torch.float32, device="cuda")
    moe.moe_quantize_int4_gs64(w.cuda(), packed, scales)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("rows,K", [(1, 64), (37, 320), (2048, 6144)])
def test_quantize_int4_exact(moe, rows, K):
    wl = synth.WORKLOADS["glm_decode"]
    w = synth.gen_dense_weights(wl, rows, K, matrix=rows)
    if rows > 1:
        w[1, 64:128] = 0.0                                     # an empty group
        w[2, :64] = torch.arange(64, dtype=torch.float32) - 31.5   # half-way products: ties
        w[3, :64] = -w[3, :64].abs()                          # one-signed group
    packed, scales = _quantize_gpu(moe, w)
    ref_p, ref_s = oracle.quantize_int4(w)
    assert np.array_equal(scales.view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(packed, ref_p)


@pytest.mark.parametrize("rows,K", [(1, 64), (37, 320), (2048, 6144)])
def test_quantize_int3_exact(moe, rows, K):
    """int3-g64 (fmt=5, "colibri 开发演进实录" §8.3): codes and scales bit for bit."""
    wl = synth.WORKLOADS["glm_decode"]
    w = synth.gen_dense_weights(wl, rows, K, matrix=rows + 7)
    if rows > 1:
        w[1, 64:128] = 0.0                                         # an empty group
        w[2, :64] = (torch.arange(64, dtype=torch.float32) % 7 - 3) * 0.5 + 0.25   # ties
        w[3, :64] = -w[3, :64].abs()
    packed = torch.full((rows, 3 * K // 8), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows, K // 64), -1.0, dtype=torch.float32, device="cuda")
    moe.moe_quantize_int3_g64(w.cuda(), packed, scales)
    torch.cuda.synchronize()
    ref_p, ref_s = oracle.quantize_int3(w)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(packed.cpu().numpy(), ref_p)


def test_quantize_int4_feeds_the_layer(moe):
    # weights quantised on the GPU run through the layer exactly like the oracle's own codes
    wl = synth.WORKLOADS["tiny"]
    H, F, E = wl.hidden, wl.d_ff, wl.n_experts
    def quantised(shared):
        d = {}
        n = 1 if shared else E
        for m, (name, rows, K) in enumerate((("gate", F, H), ("up", F, H), ("down", H, F))):
            w = synth.gen_dense_weights(wl, n * rows, K, matrix=100 * shared + m)
            p, s = _quantize_gpu(moe, w)
            rp, rs = oracle.quantize_int4(w)
            assert np.array_equal(p, rp) and np.array_equal(s.view(np.uint32), rs.view(np.uint32))
            d["w_" + name] = torch.from_numpy(p.reshape(n, rows, K // 2))
            d["s_" + name] = torch.from_numpy(s.reshape(n, rows, K // 64))
        return d
    routed, shared = quantised(0), quantised(1)
    T = 16
    x, wr, bias = _inputs(wl, T)
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    y = torch.empty(T, H, device="cuda")
    K = wl.top_k
    rt = dict(ids=torch.empty(T, K, dtype=torch.int32, device="cuda"),
              w=torch.empty(T, K, dtype=torch.float32, device="cuda"),
              keff=torch.empty(T, dtype=torch.int32, device="cuda"))
    moe.moe_layer_forward(cfg, x.cuda(), wr.cuda(), bias.cuda(),
                          {k: v.cuda() for k, v in routed.items()},
                          {k: v.cuda() for k, v in shared.items()}, y, ws, routing=rt)
    torch.cuda.synchronize()
    _check_layer(wl, x, wr, bias, y.cpu().numpy(), {k: v.cpu().numpy() for k, v in rt.items()},
                 routed={k: v.numpy() for k, v in routed.items()},
                 shared={k: v.numpy() for k, v in shared.items()}, what="quantised weights")


def test_layer_forward_tensor_path_wider_shared_expert(moe):
    """Tensor-core path with the shared expert wider than the routed ones (d_ff_shared 1024,
    d_ff 512): the shared slot's tiles reduce over 1024 inputs in the down projection."""
    from dataclasses import replace
    wl = replace(synth.WORKLOADS["a3b_decode"], name="a3b_wide_shared", d_ff_shared=1024)
    T = 100
    assert moe.moe_ffn_uses_tensor_cores(moe_cfg(wl), T) == 1
    x, wr, bias = _inputs(wl, T)
    y, rt = _layer_gpu(moe, wl, x, wr, bias)
    _check_layer(wl, x, wr, bias, y, rt, what="a3b, wider shared expert")


def test_bounded_wait_reports_timeout_and_context_survives(moe):
    """A device wait that runs out (a flag nothing sets) ends the kernel with an error status
    that moe_check_errors returns as MOE_ERR_TIMEOUT; the context stays usable."""
    wl = synth.WORKLOADS["tiny"]
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, 16)
    moe.moe_check_errors(ws)                      # clean to begin with
    moe.moe_selftest_wait_timeout(ws, polls=4096)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_check_errors(ws)
    assert ei.value.code == moe.MOE_ERR_TIMEOUT
    moe.moe_check_errors(ws)                      # the record is cleared
    # the same context still runs a layer correctly
    x, wr, bias = _inputs(wl, 16)
    y, rt = _layer_gpu(moe, wl, x, wr, bias)
    near, _ = _check_layer(wl, x, wr, bias, y, rt, what="after a timeout")
    assert near == 0


@pytest.mark.parametrize("name,T", [("tiny", 16), ("glm_decode", 8), ("a3b_decode", 128)])
def test_layer_forward_host_buffers(moe, name, T):
    """moe_layer_forward_host (host x in, host y out) gives the device call's output bit for bit."""
    wl = synth.WORKLOADS[name]
    x, wr, bias = _inputs(wl, T)
    cfg = moe_cfg(wl)
    ws = moe.alloc_workspace(cfg, T)
    routed = device_experts(wl)
    shared = device_experts(wl, shared=True) if wl.n_shared else None
    y_dev = torch.empty(T, wl.hidden, device="cuda")
    moe.moe_layer_forward(cfg, x.cuda(), wr.cuda(), bias.cuda(), routed, shared, y_dev, ws)
    x_host = x.pin_memory()
    y_host = torch.full((T, wl.hidden), float("nan")).pin_memory()
    moe.moe_layer_forward_host(cfg, x_host, wr.cuda(), bias.cuda(), routed, shared, y_host, ws)
    torch.cuda.synchronize()
    assert torch.equal(y_host, y_dev.cpu())
