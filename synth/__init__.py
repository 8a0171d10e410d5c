"""Seeded synthetic inputs for the sparse MoE FFN layer.

This module is the one thing the CUDA path and the CPU oracle share: it draws
the layer's inputs (activations, router weights and selection bias, int4 expert
codes and their group scales) and holds none of the layer's arithmetic.

Every value comes from a counter-based SplitMix64 stream (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014; the finaliser
constants are Vigna's published `splitmix64.c`).  Element ``i`` of a stream with
key ``k`` is ``mix64(k + (i + 1) * GAMMA)``, so any single expert of a 9.5 GB
layer can be regenerated on the host without producing the others.  Keys are
derived from ``(seed, tensor id, expert or batch index)``.

Integer draws (packed nibbles) and the affine uniform draws (scales) use only
64-bit integer operations and correctly rounded IEEE double multiply/add, so the
same call gives bit-identical tensors on the CPU and on a GPU.  Normal draws use
``log``/``cos`` and are therefore always made on the CPU and then moved.

Workload recipes mirror the shapes and distributions of the layer's benchmark
configurations; see ``WORKLOADS``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, Optional, Sequence, Tuple

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

# tensor ids used in key derivation
T_X = 1
T_ROUTER_W = 2
T_BIAS = 3
T_ZIPF_PERM = 4
T_RESID, T_RESID_SCALE, T_NORM_W = 5, 6, 7   # router look-ahead inputs
T_NEXT_ROUTER_W, T_NEXT_BIAS = 8, 9
T_DENSE_W, T_DENSE_ROW_SCALE = 20, 21        # fp32 weights for the offline quantiser
T_GATE_CODES, T_GATE_SCALES = 10, 11
T_UP_CODES, T_UP_SCALES = 12, 13
T_DOWN_CODES, T_DOWN_SCALES = 14, 15
SHARED_OFFSET = 10  # shared expert tensors use id + SHARED_OFFSET

GROUP = 64


def _signed(v: int) -> int:
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python integer (exact, mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor: int, index: int = 0) -> int:
    k = mix64_int(seed * GAMMA + tensor + 1)
    return mix64_int(k + (index + 1) * GAMMA)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    # logical right shift of an int64 tensor holding uint64 bits
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64_tensor(z: torch.Tensor) -> torch.Tensor:
    z = z ^ _lsr(z, 30)
    z = z * _signed(MIX1)
    z = z ^ _lsr(z, 27)
    z = z * _signed(MIX2)
    return z ^ _lsr(z, 31)


def stream(key: int, n: int, device="cpu", start: int = 0) -> torch.Tensor:
    """Elements ``start .. start+n-1`` of the stream with ``key`` as uint64 bits in int64."""
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    z = i * _signed(GAMMA) + _signed(key)
    return _mix64_tensor(z)


def uniform_bytes(key: int, nbytes: int, device="cpu") -> torch.Tensor:
    """``nbytes`` independent uniform bytes (two independent uniform nibbles each)."""
    n64 = (nbytes + 7) // 8
    return stream(key, n64, device).view(torch.uint8)[:nbytes]


def uniform01(key: int, n: int, device="cpu", start: int = 0) -> torch.Tensor:
    """float64 uniforms on [0, 1) with 53 random bits."""
    z = stream(key, n, device, start)
    return _lsr(z, 11).to(torch.float64) * (2.0 ** -53)


def uniform_range(key: int, n: int, lo: float, hi: float, device="cpu") -> torch.Tensor:
    u = uniform01(key, n, device)
    return (u * (hi - lo) + lo).to(torch.float32)


def normal(key: int, n: int, std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) draws as float32, Box-Muller (cosine branch) in float64 on the CPU.

    Element i uses stream elements 2i and 2i+1.
    """
    z = stream(key, 2 * n, "cpu")
    u = _lsr(z, 11).to(torch.float64) * (2.0 ** -53)
    u1 = 1.0 - u[0::2]          # (0, 1]
    u2 = u[1::2]
    r = torch.sqrt(-2.0 * torch.log(u1))
    return (r * torch.cos((2.0 * math.pi) * u2) * std).to(torch.float32)


# --------------------------------------------------------------------------
# workload recipes
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """Shapes, distributions and routing knobs of one synthetic MoE layer."""
    name: str
    hidden: int            # H
    n_experts: int         # E
    top_k: int             # K
    d_ff: int              # F
    n_shared: int          # 0 or 1
    d_ff_shared: int       # Fs
    tokens: Tuple[int, ...]  # batch sizes T this workload is run at
    norm_topk_prob: int = 1
    routed_scaling_factor: float = 1.0
    top_p: float = 0.0     # <= 0 or >= 1: off
    bias_std: float = 0.1  # N(0, bias_std) selection bias
    zipf_s: float = 0.0    # > 0: Zipf(s) selection bias instead of the normal one
    zipf_beta: float = 0.0
    scale_lo: float = 0.005
    scale_hi: float = 0.02
    seed: int = 0

    @property
    def x_std(self) -> float:
        return 1.0

    @property
    def router_std(self) -> float:
        # N(0, 1/sqrt(H)): logits x.W come out ~N(0, 1)
        return 1.0 / math.sqrt(self.hidden)

    def with_tokens(self, *t: int) -> "Workload":
        return replace(self, tokens=tuple(t))

    def expert_bytes(self, shared: bool = False) -> int:
        """Bytes of one expert: packed nibbles plus fp32 gs64 scales, gate+up+down."""
        F = self.d_ff_shared if shared else self.d_ff
        H = self.hidden
        return 3 * (H * F // 2 + (H * F // GROUP) * 4)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 256, 8, 2, 128, 1, 128, (16,), 1, 1.0, 0.0, 0.1),
    "glm_decode": Workload("glm_decode", 6144, 256, 8, 2048, 1, 2048,
                           (1, 2, 4, 8, 16, 32), 1, 2.5, 0.0, 0.1),
    "a3b_decode": Workload("a3b_decode", 2048, 256, 8, 512, 1, 512, (64,), 1, 1.0, 0.7, 0.5),
    # beta = 0.04: with seed 0 the busiest expert receives 970 of the 4096 tokens and the
    # least busy 24 (a Zipf(1.1) popularity profile realised through the selection bias)
    "prefill": Workload("prefill", 6144, 256, 8, 2048, 1, 2048, (4096,), 1, 2.5, 0.0, 0.1,
                        zipf_s=1.1, zipf_beta=0.04),
    "wide": Workload("wide", 7168, 384, 8, 2048, 1, 2048, (1, 8, 64, 512, 8192), 1, 1.0, 0.0, 0.1),
}


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------

def gen_x(wl: Workload, T: int, batch: int = 0) -> torch.Tensor:
    """Activations x ~ N(0, 1), float32 [T, H] on the CPU; ``batch`` selects an independent batch."""
    return normal(stream_key(wl.seed, T_X, batch), T * wl.hidden, wl.x_std).view(T, wl.hidden)


def gen_router(wl: Workload) -> Tuple[torch.Tensor, torch.Tensor]:
    """Router weights float32 [E, H] ~ N(0, 1/sqrt(H)) and selection bias float32 [E] (CPU)."""
    E, H = wl.n_experts, wl.hidden
    w = normal(stream_key(wl.seed, T_ROUTER_W), E * H, wl.router_std).view(E, H)
    if wl.zipf_s > 0:
        # Zipf(s) popularity by a seeded rank permutation: bias = -beta * s * ln(rank)
        order = torch.argsort(uniform01(stream_key(wl.seed, T_ZIPF_PERM), E), stable=True)
        rank = torch.empty(E, dtype=torch.float64)
        rank[order] = torch.arange(1, E + 1, dtype=torch.float64)
        bias = (-wl.zipf_beta * wl.zipf_s * torch.log(rank)).to(torch.float32)
    else:
        bias = normal(stream_key(wl.seed, T_BIAS), E, wl.bias_std)
    return w, bias


def gen_lookahead(wl: Workload, T: int, batch: int = 0):
    """Inputs of the router look-ahead: a residual state [T, H] (N(0, 1) rows times a per-token
    magnitude U(0.5, 20), as residual streams grow across layers), an RMSNorm weight [H] ~
    U(0.5, 1.5), and a later layer's router of the workload's shape (its own weights and bias,
    drawn like gen_router's).  All float32 on the CPU."""
    H, E = wl.hidden, wl.n_experts
    z = normal(stream_key(wl.seed, T_RESID, batch), T * H).view(T, H)
    mag = uniform_range(stream_key(wl.seed, T_RESID_SCALE, batch), T, 0.5, 20.0).view(T, 1)
    g = uniform_range(stream_key(wl.seed, T_NORM_W), H, 0.5, 1.5)
    w = normal(stream_key(wl.seed, T_NEXT_ROUTER_W), E * H, wl.router_std).view(E, H)
    bias = normal(stream_key(wl.seed, T_NEXT_BIAS), E, wl.bias_std if wl.bias_std > 0 else 0.1)
    return z * mag, g, w, bias


def gen_dense_weights(wl: Workload, rows: int, K: int, matrix: int = 0) -> torch.Tensor:
    """fp32 weights [rows, K] before quantisation: N(0, 1) entries times a per-row magnitude
    U(0.001, 0.05) (weight rows of trained layers differ in scale); ``matrix`` selects an
    independent matrix.  CPU."""
    z = normal(stream_key(wl.seed, T_DENSE_W, matrix), rows * K).view(rows, K)
    mag = uniform_range(stream_key(wl.seed, T_DENSE_ROW_SCALE, matrix), rows, 0.001, 0.05)
    return z * mag.view(rows, 1)


def _matrix_keys(shared: bool) -> Sequence[Tuple[str, int, int, bool]]:
    off = SHARED_OFFSET if shared else 0
    # (name, codes tensor id, scales tensor id, is_down)
    return (("gate", T_GATE_CODES + off, T_GATE_SCALES + off, False),
            ("up", T_UP_CODES + off, T_UP_SCALES + off, False),
            ("down", T_DOWN_CODES + off, T_DOWN_SCALES + off, True))


def gen_expert(wl: Workload, e: int, shared: bool = False, device="cpu") -> Dict[str, torch.Tensor]:
    """One expert's canonical tensors.

    ``w_gate``/``w_up``: uint8 [F, H/2]; ``s_gate``/``s_up``: float32 [F, H/64];
    ``w_down``: uint8 [H, F/2]; ``s_down``: float32 [H, F/64].  Byte j of a row
    holds element 2j in its low nibble and element 2j+1 in its high nibble; a
    code u in 0..15 stands for the value (u - 8) * scale.
    """
    H = wl.hidden
    F = wl.d_ff_shared if shared else wl.d_ff
    out = {}
    for name, tc, ts, is_down in _matrix_keys(shared):
        rows, cols = (H, F) if is_down else (F, H)
        codes = uniform_bytes(stream_key(wl.seed, tc, e), rows * cols // 2, device).view(rows, cols // 2)
        scales = uniform_range(stream_key(wl.seed, ts, e), rows * cols // GROUP,
                               wl.scale_lo, wl.scale_hi, device).view(rows, cols // GROUP)
        out["w_" + name] = codes
        out["s_" + name] = scales
    return out


def gen_experts(wl: Workload, shared: bool = False, device="cpu",
                experts: Optional[Sequence[int]] = None) -> Dict[str, torch.Tensor]:
    """Stacked tensors [E, ...] of every routed expert (or [1, ...] of the shared one).

    Filled one expert at a time so that temporaries stay at one expert's size.
    """
    H = wl.hidden
    F = wl.d_ff_shared if shared else wl.d_ff
    ids = [0] if shared else (list(range(wl.n_experts)) if experts is None else list(experts))
    n = len(ids)
    out = {
        "w_gate": torch.empty(n, F, H // 2, dtype=torch.uint8, device=device),
        "s_gate": torch.empty(n, F, H // GROUP, dtype=torch.float32, device=device),
        "w_up": torch.empty(n, F, H // 2, dtype=torch.uint8, device=device),
        "s_up": torch.empty(n, F, H // GROUP, dtype=torch.float32, device=device),
        "w_down": torch.empty(n, H, F // 2, dtype=torch.uint8, device=device),
        "s_down": torch.empty(n, H, F // GROUP, dtype=torch.float32, device=device),
    }
    for j, e in enumerate(ids):
        one = gen_expert(wl, e, shared, device)
        for k, v in one.items():
            out[k][j].copy_(v)
        del one
    return out
