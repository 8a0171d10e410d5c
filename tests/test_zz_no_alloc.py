"""moe_route_noalloc: the router entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (a plugin inside an engine that owns all device memory,
or a decode loop that cannot take the synchronisation an allocation may cause).  For them
moe_route_noalloc keeps the router's scratch in a fixed array inside libmoe.so.  This test
calls it through the C ABI and checks it against moe_route (which takes a workspace) on two
calls in a row with different inputs, so a second call that reuses the array's previous
contents is covered too.  Kept in a file of its own, collected last.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import moe_cfg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_expert_ffn_route_gb300 as m
    m.load_library()
    return m


def _outputs(T, K):
    return (torch.full((T, K), -9, dtype=torch.int32, device="cuda"),
            torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda"),
            torch.full((T,), -9, dtype=torch.int32, device="cuda"))


# T <= 64 takes the cluster router (final logits [T][E] in the array); larger batches split
# the reduction over H ([S][T][E] partial logits), up to T = 4096 at E = 256
@pytest.mark.parametrize("name,T", [("glm_decode", 32), ("a3b_decode", 64), ("glm_decode", 512),
                                    ("prefill", 4096)])
def test_route_noalloc_matches_route_on_two_calls(moe, name, T):
    wl = synth.WORKLOADS[name]
    cfg = moe_cfg(wl)
    wr, bias = synth.gen_router(wl)
    wr, bias = wr.cuda(), bias.cuda()
    ws = moe.alloc_workspace(cfg, T)
    for batch in (0, 1):   # two calls in a row on different tokens
        x = synth.gen_x(wl, T, batch).cuda()
        ref = _outputs(T, wl.top_k)
        got = _outputs(T, wl.top_k)
        moe.moe_route(cfg, x, wr, bias, *ref, ws)
        moe.moe_route_noalloc(cfg, x, wr, bias, *got)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0])
        assert torch.equal(got[2], ref[2])
        np.testing.assert_allclose(got[1].cpu().numpy(), ref[1].cpu().numpy(), rtol=2e-5, atol=1e-7)


def test_route_noalloc_rejects_oversize(moe):
    wl = synth.WORKLOADS["wide"]
    cfg = moe_cfg(wl)
    T = 8192                     # needs more router scratch than the built-in array holds
    wr, bias = synth.gen_router(wl)
    x = torch.zeros(T, wl.hidden, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_noalloc(cfg, x, wr.cuda(), bias.cuda(), *_outputs(T, wl.top_k))
    assert ei.value.code == moe.MOE_ERR_SHAPE and "scratch" in str(ei.value)
