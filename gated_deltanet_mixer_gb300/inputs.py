"""Seeded synthetic inputs for the mixer: shapes, value distributions, seeds.

This module only draws random numbers; it holds none of the mixer's
arithmetic.  The tests, the benchmark and the smoke check feed the same
arrays to the CUDA library and to the CPU oracle.

Every tensor has its own seed, ``seed = 1000 * case + tensor_id`` (decode
steps add ``100 * step``); large tensors are drawn in slabs of 2^24 values,
slab i from ``Generator(PCG64(SeedSequence([seed, i])))`` so that slabs can be
drawn in parallel and the values do not depend on the thread count.  Values
are drawn in float64, then rounded to the I/O dtype (round to nearest even).
Values come back as float32 arrays that hold exactly the rounded values, so a
bf16 copy made from them is exact.

Distributions (the workload recipe of the Qwen3.5 / Qwen3.8 shapes):
  qkv_pre, z, conv window ~ N(0, 1)      conv_w ~ N(0, 0.5^2)
  beta = sigmoid(N(0, 1))                g = log(sigmoid(N(mu_g, 1))), mu_g = 3 (5 for
                                         the long-horizon 27B prefill)
  norm_w = 1 + N(0, 0.1^2)               S0 = 0 (tiny case) or N(0, 0.02^2)
Raw gate projections (when the gates are prepared inside the library):
  a, b ~ N(0, 1) (io dtype)              A_log = log U(1, 16), dt_bias ~ U(-7, -2)
                                         per value head (fp32)
so that softplus(a + dt_bias) is mostly 1e-3 .. 0.1 and g spans about
-1e-3 .. -2 per token.
Packed (varlen) batches draw their token tensors as one [N, ...] run.
"""
import concurrent.futures as cf
import os
from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

TENSOR_IDS = {"qkv_pre": 1, "z": 2, "beta": 3, "g": 4, "conv_w": 5, "norm_w": 6,
              "S0": 7, "conv0": 8, "a": 9, "b": 10, "A_log": 11, "dt_bias": 12}

_SLAB = 1 << 24  # values drawn per call, to bound peak host memory


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (nearest, ties to even); return float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def _slab(seed, i, m, mean, std, io):
    gen = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, i])))
    x = gen.standard_normal(m) * std + mean
    return round_to_bf16(x) if io == "bf16" else x.astype(np.float32)


def _normal(seed: int, shape, mean=0.0, std=1.0, io="f32") -> np.ndarray:
    """N(mean, std^2) drawn in float64 slab by slab, rounded to ``io``."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    starts = list(range(0, n, _SLAB))

    def fill(j):
        s = starts[j]
        m = min(_SLAB, n - s)
        out[s:s + m] = _slab(seed, j, m, mean, std, io)

    if len(starts) > 1:
        with cf.ThreadPoolExecutor(max_workers=min(len(starts), _threads())) as ex:
            list(ex.map(fill, range(len(starts))))
    elif starts:
        fill(0)
    return out.reshape(shape)


def _threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _beta(seed, shape):
    gen = np.random.Generator(np.random.PCG64(seed))
    return _sigmoid(gen.standard_normal(shape)).astype(np.float32)


def _log_decay(seed, shape, mu):
    gen = np.random.Generator(np.random.PCG64(seed))
    x = gen.standard_normal(shape) + mu
    return (-np.logaddexp(0.0, -x)).astype(np.float32)  # log(sigmoid(x))


@dataclass
class Problem:
    """One mixer call's worth of inputs (host arrays, float32 values)."""
    B: int
    T: int
    Hk: int
    Hv: int
    io: str                      # "f32" or "bf16": dtype of qkv_pre, z, o, conv, weights
    Dk: int = 128
    Dv: int = 128
    arrays: Dict[str, Optional[np.ndarray]] = field(default_factory=dict)

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv

    def __getitem__(self, k):
        return self.arrays[k]


def prefill_problem(B, T, Hk, Hv, io="bf16", case=0, g_mu=3.0, s0_std=0.02,
                    conv0=True, Dk=128, Dv=128) -> Problem:
    """Inputs of one prefill call.  ``s0_std = 0`` gives S0 = None (zeros);
    ``conv0 = False`` gives no carried conv window (zeros)."""
    p = Problem(B, T, Hk, Hv, io, Dk, Dv)
    C = p.C
    base = 1000 * case
    a = p.arrays
    a["qkv_pre"] = _normal(base + 1, (B, T, C), io=io)
    a["z"] = _normal(base + 2, (B, T, Hv * Dv), io=io)
    a["beta"] = _beta(base + 3, (B, T, Hv))
    a["g"] = _log_decay(base + 4, (B, T, Hv), g_mu)
    a["conv_w"] = _normal(base + 5, (C, 4), std=0.5, io=io)
    a["norm_w"] = _normal(base + 6, (Dv,), mean=1.0, std=0.1, io=io)
    a["S0"] = _normal(base + 7, (B, Hv, Dv, Dk), std=s0_std) if s0_std > 0 else None
    a["conv0"] = _normal(base + 8, (B, 3, C), io=io) if conv0 else None
    return p


# The five workloads.  Sizes follow the model shapes: Qwen3.5-0.8B (16/16 heads),
# Qwen3.5-4B (16 key / 32 value heads), Qwen3.8-27B (16 key / 48 value heads),
# all with 128-wide heads; the tiny case is a 1-key / 2-value-head fp32 mixer.
CASES = {
    "tiny": dict(case=0, B=1, T=64, Hk=1, Hv=2, io="f32", s0_std=0.0, conv0=False),
    "0.8b_prefill": dict(case=1, B=1, T=4096, Hk=16, Hv=16, io="bf16"),
    "4b_prefill": dict(case=2, B=4, T=8192, Hk=16, Hv=32, io="bf16"),
    "27b_prefill": dict(case=3, B=1, T=65536, Hk=16, Hv=48, io="bf16", g_mu=5.0),
}
DECODE_CASE = dict(case=4, B=256, Hk=16, Hv=48, io="bf16", steps=64)


def case_problem(name: str, **override) -> Problem:
    kw = dict(CASES[name])
    kw.update(override)
    return prefill_problem(**kw)


@dataclass
class DecodeProblem:
    """Initial state plus ``steps`` fresh single-token inputs for B sequences."""
    B: int
    Hk: int
    Hv: int
    io: str
    steps: int
    Dk: int = 128
    Dv: int = 128
    S: Optional[np.ndarray] = None        # [B, Hv, Dv, Dk] float32
    conv: Optional[np.ndarray] = None     # [B, 3, C]
    conv_w: Optional[np.ndarray] = None   # [C, 4]
    norm_w: Optional[np.ndarray] = None   # [Dv]
    qkv_pre: Optional[np.ndarray] = None  # [steps, B, C]
    z: Optional[np.ndarray] = None        # [steps, B, Hv*Dv]
    g: Optional[np.ndarray] = None        # [steps, B, Hv]
    beta: Optional[np.ndarray] = None     # [steps, B, Hv]

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv


def decode_problem(B=256, Hk=16, Hv=48, io="bf16", steps=64, case=4, g_mu=3.0,
                   Dk=128, Dv=128) -> DecodeProblem:
    p = DecodeProblem(B, Hk, Hv, io, steps, Dk, Dv)
    C = p.C
    base = 1000 * case
    p.conv_w = _normal(base + 5, (C, 4), std=0.5, io=io)
    p.norm_w = _normal(base + 6, (Dv,), mean=1.0, std=0.1, io=io)
    p.S = _normal(base + 7, (B, Hv, Dv, Dk), std=0.02)
    p.conv = _normal(base + 8, (B, 3, C), io=io)
    with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
        p.qkv_pre = np.stack(list(ex.map(
            lambda s: _normal(base + 1 + 100 * s, (B, C), io=io), range(steps))))
        p.z = np.stack(list(ex.map(
            lambda s: _normal(base + 2 + 100 * s, (B, Hv * Dv), io=io), range(steps))))
    p.beta = np.stack([_beta(base + 3 + 100 * s, (B, Hv)) for s in range(steps)])
    p.g = np.stack([_log_decay(base + 4 + 100 * s, (B, Hv), g_mu) for s in range(steps)])
    return p


def raw_gate_arrays(case, lead, Hv, io="bf16"):
    """Raw gate projections a, b [*lead, Hv] (io-rounded) and the per-head
    parameters A_log, dt_bias [Hv] (fp32)."""
    base = 1000 * case
    gen = np.random.Generator(np.random.PCG64(base + 11))
    A_log = np.log(gen.uniform(1.0, 16.0, size=Hv)).astype(np.float32)
    gen = np.random.Generator(np.random.PCG64(base + 12))
    dt_bias = gen.uniform(-7.0, -2.0, size=Hv).astype(np.float32)
    return dict(a=_normal(base + 9, tuple(lead) + (Hv,), io=io),
                b=_normal(base + 10, tuple(lead) + (Hv,), io=io), A_log=A_log, dt_bias=dt_bias)


@dataclass
class PackedProblem:
    """Sequences of the given lengths packed back to back (cu_seqlens)."""
    lengths: tuple
    Hk: int
    Hv: int
    io: str
    Dk: int = 128
    Dv: int = 128
    arrays: Dict[str, Optional[np.ndarray]] = field(default_factory=dict)

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    @property
    def N(self) -> int:
        return int(sum(self.lengths))

    def __getitem__(self, k):
        return self.arrays[k]


def packed_problem(lengths, Hk, Hv, io="bf16", case=0, g_mu=3.0, state=True, raw_gates=False,
                   Dk=128, Dv=128) -> PackedProblem:
    """Inputs of one packed prefill call; with ``raw_gates`` the gates come as
    raw projections (arrays a, b, A_log, dt_bias) instead of g and beta."""
    p = PackedProblem(tuple(int(n) for n in lengths), Hk, Hv, io, Dk, Dv)
    B, N, C = len(p.lengths), p.N, p.C
    base = 1000 * case
    a = p.arrays
    a["qkv_pre"] = _normal(base + 1, (N, C), io=io)
    a["z"] = _normal(base + 2, (N, Hv * Dv), io=io)
    if raw_gates:
        a.update(raw_gate_arrays(case, (N,), Hv, io))
        a["g"] = a["beta"] = None
    else:
        a["beta"] = _beta(base + 3, (N, Hv))
        a["g"] = _log_decay(base + 4, (N, Hv), g_mu)
    a["conv_w"] = _normal(base + 5, (C, 4), std=0.5, io=io)
    a["norm_w"] = _normal(base + 6, (Dv,), mean=1.0, std=0.1, io=io)
    a["S0"] = _normal(base + 7, (B, Hv, Dv, Dk), std=0.02) if state else None
    a["conv0"] = _normal(base + 8, (B, 3, C), io=io) if state else None
    return p


def linear_problem(M, N, K, case=0, w_std=0.02):
    """Inputs of one projection: x ~ N(0, 1) [M, K] and w ~ N(0, w_std^2)
    [N, K], both bf16-rounded (tensor ids 13, 14)."""
    base = 1000 * case
    return _normal(base + 13, (M, K), io="bf16"), _normal(base + 14, (N, K), std=w_std, io="bf16")
