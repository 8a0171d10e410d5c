"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
include/moe.h declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import sparse_expert_ffn_route_gb300 as moe
from sparse_expert_ffn_route_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(moe.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def _cfg(**kw):
    base = dict(hidden=256, n_experts=8, top_k=2, d_ff=128, n_shared=1, d_ff_shared=128)
    base.update(kw)
    return moe.MoeConfig.make(**base)


def test_workspace_size(lib):
    cfg = _cfg()
    sizes = [moe.moe_workspace_size(cfg, t) for t in (0, 1, 16, 64, 65, 1000, 5000)]
    assert all(s > 0 for s in sizes) and sizes == sorted(sizes)
    for bad in (_cfg(hidden=250), _cfg(top_k=9), _cfg(n_experts=513, top_k=2), _cfg(d_ff=100),
                _cfg(group_size=32), _cfg(n_shared=2), _cfg(hidden=16384)):
        assert moe.moe_workspace_size(bad, 16) == 0
    assert moe.moe_workspace_size(cfg, -1) == 0


def test_ffn_path_query(lib):
    # the tensor-core grouped GEMM takes batches beyond the 64-token decode route when every
    # matrix of the layer has dimensions in multiples of 512
    # ... and, on wide matrices, at least 10 expected tokens per routed expert (GLM: T = 65,
    # 128 and 256 give 2.3, 4.1 and 8.0, T = 512 gives 16.0); narrow ones (d_ff 512) take it
    # at once
    glm = _cfg(hidden=6144, n_experts=256, top_k=8, d_ff=2048, d_ff_shared=2048)
    assert [moe.moe_ffn_uses_tensor_cores(glm, t) for t in (0, 1, 64, 65, 128, 256, 512, 4096)] == \
        [0, 0, 0, 0, 0, 0, 1, 1]
    a3b = _cfg(hidden=2048, n_experts=256, top_k=8, d_ff=512, d_ff_shared=512)
    assert [moe.moe_ffn_uses_tensor_cores(a3b, t) for t in (16, 31, 32, 64, 65, 128)] == [0, 0, 1, 1, 1, 1]
    tiny = _cfg()   # d_ff = 128: GEMV kernels at every batch size
    assert [moe.moe_ffn_uses_tensor_cores(tiny, t) for t in (1, 65, 5000)] == [0, 0, 0]
    assert moe.moe_ffn_uses_tensor_cores(_cfg(hidden=6144, d_ff=2048, d_ff_shared=640), 100) == 0
    assert moe.moe_ffn_uses_tensor_cores(glm, -1) == -1
    assert moe.moe_ffn_uses_tensor_cores(_cfg(top_k=9), 16) == -1
    # the kernel below the tensor path: the row GEMV when every reduction is a multiple of
    # 256 inputs and the batch has 3 tokens or more, the warp GEMV otherwise
    R, W, TC = moe.MOE_FFN_ROW_GEMV, moe.MOE_FFN_WARP_GEMV, moe.MOE_FFN_TENSOR
    assert [moe.moe_ffn_path(glm, t) for t in (1, 2, 3, 4, 8, 32, 256, 512)] == [W, W, R, R, R, R, R, TC]
    # the narrow A3B-style layer: in the decode route (T <= 64) gate/up on the row GEMV and
    # down on the tensor path from 32 tokens on; past it both on the tensor path
    assert [moe.moe_ffn_path(a3b, t) for t in (16, 31, 32, 64, 65)] == [R, R, R, R, TC]
    assert [moe.moe_ffn_path_down(a3b, t) for t in (16, 31, 32, 64, 65)] == [R, R, TC, TC, TC]
    assert [moe.moe_ffn_path_down(glm, t) for t in (1, 2, 3, 32, 512)] == [W, W, R, R, TC]
    assert moe.moe_ffn_path_down(glm, -1) == -1
    assert [moe.moe_ffn_path(tiny, t) for t in (1, 16, 65)] == [W, W, W]
    # reductions that are not multiples of 256 keep the warp GEMV at any decode batch
    assert moe.moe_ffn_path(_cfg(hidden=1088, d_ff=1088, n_shared=0, d_ff_shared=0), 8) == W
    assert moe.moe_ffn_path(_cfg(hidden=6144, d_ff=2048, d_ff_shared=640), 32) == W
    assert moe.moe_ffn_path(_cfg(hidden=6144, d_ff=2048, d_ff_shared=768), 32) == R
    assert moe.moe_ffn_path(glm, -1) == -1 and moe.moe_ffn_path(_cfg(top_k=9), 16) == -1


def test_lookahead_validation(lib):
    cfg = _cfg()
    args = lambda eps, norm=FAKE: (ctypes.byref(cfg), FAKE, norm, ctypes.c_float(eps), FAKE, FAKE, 4,
                                   FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert lib.moe_route_lookahead(*args(-1.0)) == moe.MOE_ERR_ARG
    assert lib.moe_route_lookahead(*args(float("nan"))) == moe.MOE_ERR_ARG
    assert lib.moe_route_lookahead(*args(float("inf"))) == moe.MOE_ERR_ARG
    assert lib.moe_route_lookahead(*args(1e-5, norm=None)) == moe.MOE_ERR_ARG
    assert lib.moe_route_lookahead(*args(1e-5, norm=FAKE + 4)) == moe.MOE_ERR_ALIGN
    assert lib.moe_topk_hits(ctypes.byref(cfg), FAKE, FAKE, None, FAKE, 4, FAKE, None) == moe.MOE_ERR_ARG
    assert lib.moe_topk_hits(ctypes.byref(_cfg(top_k=9)), FAKE, FAKE, FAKE, FAKE, 4, FAKE, None) \
        == moe.MOE_ERR_SHAPE


def test_selftest_validation(lib):
    st = lib.moe_selftest_wait_timeout
    assert st(None, 1 << 20, 16, None) == moe.MOE_ERR_WORKSPACE
    assert st(FAKE + 16, 1 << 20, 16, None) == moe.MOE_ERR_ALIGN
    assert st(FAKE, 128, 16, None) == moe.MOE_ERR_WORKSPACE
    assert st(FAKE, 1 << 20, 0, None) == moe.MOE_ERR_ARG
    assert st(FAKE, 1 << 20, (1 << 24) + 1, None) == moe.MOE_ERR_ARG


def test_quantize_validation(lib):
    q = lib.moe_quantize_int4_gs64
    assert q(FAKE, -1, 64, FAKE, FAKE, None) == moe.MOE_ERR_SHAPE
    assert q(FAKE, 4, 100, FAKE, FAKE, None) == moe.MOE_ERR_SHAPE
    assert q(FAKE, 4, 0, FAKE, FAKE, None) == moe.MOE_ERR_SHAPE
    assert q(None, 4, 64, FAKE, FAKE, None) == moe.MOE_ERR_ARG
    assert q(FAKE, 4, 64, FAKE + 8, FAKE, None) == moe.MOE_ERR_ALIGN
    assert q(FAKE, 0, 64, None, None, None) == moe.MOE_OK   # nothing to do
    q3 = lib.moe_quantize_int3_g64
    assert q3(FAKE, -1, 64, FAKE, FAKE, None) == moe.MOE_ERR_SHAPE
    assert q3(FAKE, 4, 96, FAKE, FAKE, None) == moe.MOE_ERR_SHAPE
    assert q3(None, 4, 64, FAKE, FAKE, None) == moe.MOE_ERR_ARG
    assert q3(FAKE + 4, 4, 64, FAKE, FAKE, None) == moe.MOE_ERR_ALIGN
    assert q3(FAKE, 4, 64, FAKE, FAKE + 2, None) == moe.MOE_ERR_ALIGN
    assert q3(FAKE, 0, 64, None, None, None) == moe.MOE_OK


FAKE = 1 << 20   # aligned, never dereferenced: validation fails before any use


def _route(lib, cfg, x=FAKE, wr=FAKE, b=FAKE, T=4, ids=FAKE, w=FAKE, keff=FAKE, ws=FAKE,
           nbytes=1 << 30):
    return lib.moe_route(ctypes.byref(cfg), x, wr, b, T, ids, w, keff, ws, nbytes, None)


def test_validation_codes(lib):
    cfg = _cfg()
    assert _route(lib, _cfg(hidden=100)) == moe.MOE_ERR_SHAPE
    assert _route(lib, cfg, T=-1) == moe.MOE_ERR_SHAPE
    assert _route(lib, cfg, x=None) == moe.MOE_ERR_ARG
    assert "x is NULL" in moe.last_error()
    assert _route(lib, cfg, x=FAKE + 4) == moe.MOE_ERR_ALIGN
    assert _route(lib, cfg, ws=None) == moe.MOE_ERR_WORKSPACE
    assert _route(lib, cfg, ws=FAKE + 16) == moe.MOE_ERR_ALIGN
    assert _route(lib, cfg, nbytes=100) == moe.MOE_ERR_WORKSPACE
    assert _route(lib, cfg, T=0) == moe.MOE_OK          # nothing to do, nothing enqueued
    assert lib.moe_route(None, FAKE, FAKE, FAKE, 4, FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == moe.MOE_ERR_ARG
    rw = moe.ExpertWeights(FAKE, FAKE, FAKE, FAKE, FAKE, None)
    rc = lib.moe_layer_forward(ctypes.byref(cfg), FAKE, 4, FAKE, FAKE, ctypes.byref(rw),
                               ctypes.byref(rw), FAKE, None, FAKE, 1 << 30, 0, None)
    assert rc == moe.MOE_ERR_ARG and "s_down" in moe.last_error()
    rw = moe.ExpertWeights(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    rc = lib.moe_layer_forward(ctypes.byref(cfg), FAKE, 4, FAKE, FAKE, ctypes.byref(rw), None,
                               FAKE, None, FAKE, 1 << 30, 0, None)
    assert rc == moe.MOE_ERR_ARG        # n_shared = 1 needs shared weights
    rc = lib.moe_layer_forward(ctypes.byref(cfg), FAKE, 4, FAKE, FAKE, ctypes.byref(rw),
                               ctypes.byref(rw), FAKE, None, FAKE, 1 << 30, 8, None)
    assert rc == moe.MOE_ERR_ARG        # unknown flag
    rc = lib.moe_permute(ctypes.byref(cfg), FAKE, FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2,
                         FAKE, 1 << 30, None)
    assert rc == moe.MOE_ERR_ALIGN


def test_no_device_is_reported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _route(lib, _cfg()) == moe.MOE_ERR_UNSUPPORTED


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from sparse_expert_ffn_route_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIBRARY_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        binding.load_library()
