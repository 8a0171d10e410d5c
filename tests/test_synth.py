"""The seeded input generator: published SplitMix64 vectors, determinism, distributions."""
import numpy as np
import torch

import synth

# Outputs of Vigna's splitmix64.c seeded with 1234567 (the published test sequence).
SPLITMIX64_1234567 = [6457827717110365317, 3203168211198807973, 9817491932198370423,
                      4593380528125082431, 16408922859458223821]


def test_splitmix64_published_vectors():
    got = [v & synth.MASK64 for v in synth.stream(1234567, 5).tolist()]
    assert got == SPLITMIX64_1234567


def test_stream_matches_python_integers():
    key = synth.stream_key(3, synth.T_GATE_CODES, 17)
    got = [v & synth.MASK64 for v in synth.stream(key, 64, start=1000).tolist()]
    ref = [synth.mix64_int(key + (i + 1) * synth.GAMMA) for i in range(1000, 1064)]
    assert got == ref


def test_expert_regeneration_is_exact():
    wl = synth.WORKLOADS["tiny"]
    full = synth.gen_experts(wl)
    one = synth.gen_expert(wl, 5)
    for k, v in one.items():
        assert torch.equal(full[k][5], v)
    sub = synth.gen_experts(wl, experts=[5, 2])
    assert torch.equal(sub["w_down"][1], full["w_down"][2])
    shared = synth.gen_experts(wl, shared=True)
    assert not torch.equal(shared["w_gate"][0], full["w_gate"][0])


def test_distributions():
    wl = synth.WORKLOADS["a3b_decode"]
    ex = synth.gen_expert(wl, 3)
    codes = np.concatenate([ex["w_gate"].numpy().ravel() & 15, ex["w_gate"].numpy().ravel() >> 4])
    hist = np.bincount(codes, minlength=16) / codes.size
    assert np.all(np.abs(hist - 1 / 16) < 0.003)
    s = ex["s_up"].numpy()
    assert s.min() >= 0.005 and s.max() < 0.02 and abs(s.mean() - 0.0125) < 1e-4
    x = synth.gen_x(wl, 64).numpy()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    wr, bias = synth.gen_router(wl)
    assert abs(wr.numpy().std() * np.sqrt(wl.hidden) - 1) < 0.01
    assert abs(bias.numpy().std() - 0.5) < 0.1


def test_expert_size_matches_pages():
    """About 19 MB of int4 per GLM-style expert ("colibrì 深度拆解" §3.1, §8.4): 3 * 6144 * 2048 nibbles."""
    wl = synth.WORKLOADS["glm_decode"]
    nibble_bytes = 3 * wl.hidden * wl.d_ff // 2
    assert abs(nibble_bytes / 1e6 - 18.87) < 0.01
    assert wl.expert_bytes() == nibble_bytes + 3 * wl.hidden * wl.d_ff // 64 * 4


def test_zipf_bias_is_a_rank_permutation():
    wl = synth.WORKLOADS["prefill"]
    _, bias = synth.gen_router(wl)
    b = np.sort(bias.numpy())[::-1].astype(np.float64)
    r = np.arange(1, wl.n_experts + 1)
    np.testing.assert_allclose(b, -wl.zipf_beta * wl.zipf_s * np.log(r), rtol=1e-6, atol=1e-7)
