"""GPU parity on the method's edge cases, on every kernel that runs the
recurrence: the chunked prefill (fused, staged q^/k^, and the chunk-parallel
split form), the token-serial
prefill (fp32 io), the T-token decode and the single-token decode.

The cases:
  reset       g = -inf (alpha = e^g = 0: "How Qwen3.5 works" section 9.5
              keeps g <= 0, and the limit wipes the carried state) at a
              sequence's first token, at a chunk's first, middle and last
              token, and at the last token
  deep_decay  g far below the chunked kernel's clamp (-85, -200, -1e4) and a
              run of -30 per token (a chunk's total decay beyond e^-40)
  beta_runs   runs of beta = 0 (no write) and beta = 1 (full overwrite of the
              keyed slot, node gdn.core of the Qwen3.8-27B spec)
  frozen      beta = 0 and g = 0 everywhere: the state passes through
              unchanged, bit for bit, and o reads the initial state
  qkv_small / qkv_large   qkv_pre scaled by 1e-3 and by 30
  s0_small / s0_large     initial state drawn with std 1e-4 and 10
Each is compared with the fp64 oracle on the same values."""
import numpy as np
import pytest
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I
from oracle import oracle as O

from gpu_harness import check_o, check_S, dev, prefill_workspace, to_np, torch_io

pytestmark = pytest.mark.gpu
D = 128
KINDS = ["reset", "deep_decay", "beta_runs", "frozen", "qkv_small", "qkv_large", "s0_small", "s0_large"]
# path -> (io, tokens per sequence)
PATHS = {"fused": ("bf16", 200), "staged": ("bf16", 200), "split": ("bf16", 200), "serial": ("f32", 90),
         "decode": ("bf16", 16), "decode_step": ("bf16", 12)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_mixer_gb300 import build
    build.build()
    gdn.lib()
    assert torch.cuda.is_available()
    assert gdn.gdn_device_status(reset=True) == 0


def _rescale(x, f, io):
    y = x.astype(np.float64) * f
    return I.round_to_bf16(y) if io == "bf16" else y.astype(np.float32)


def edge_problem(kind, B, T, Hk, Hv, io, case):
    """A seeded problem (state and carried window given) with one edge case
    written into its gates, inputs or state."""
    p = I.prefill_problem(B, T, Hk, Hv, io=io, case=case, s0_std=0.02, conv0=True)
    a = p.arrays
    g, beta = a["g"], a["beta"]
    if kind == "reset":
        for b in range(B):
            for h in range(Hv):
                for t in {0, 64, 100, 127, T - 1, T // 2, (b + 3 * h) % T}:
                    if t < T and (t + b + h) % 2 == 0:
                        g[b, t, h] = -np.inf
        g[:, min(5, T - 1), :] = -np.inf  # every head at once
    elif kind == "deep_decay":
        g[:, min(3, T - 1), :] = -85.0
        g[:, T // 3, ::2] = -200.0
        g[:, T - 1, 1::2] = -1e4
        lo, hi = min(64, T // 2), min(96, T)
        g[:, lo:hi, 1::2] = -30.0
    elif kind == "beta_runs":
        beta[:, T // 20:(2 * T) // 5, :] = 0.0
        beta[:, (9 * T) // 20:(3 * T) // 4, :] = 1.0
    elif kind == "frozen":
        beta[:] = 0.0
        g[:] = 0.0
    elif kind == "qkv_small":
        a["qkv_pre"] = _rescale(a["qkv_pre"], 1e-3, io)
        a["conv0"] = _rescale(a["conv0"], 1e-3, io)
    elif kind == "qkv_large":
        a["qkv_pre"] = _rescale(a["qkv_pre"], 30.0, io)
        a["conv0"] = _rescale(a["conv0"], 30.0, io)
    elif kind == "s0_small":
        a["S0"] = (a["S0"].astype(np.float64) * (1e-4 / 0.02)).astype(np.float32)
    elif kind == "s0_large":
        a["S0"] = (a["S0"].astype(np.float64) * (10.0 / 0.02)).astype(np.float32)
    else:
        raise ValueError(kind)
    return p


def run_path(path, p):
    """o [B,T,Hv*D], S_T, conv_T of the problem on one GPU path (decode paths
    take the state and window as the cache and the T tokens as new ones)."""
    t = torch_io(p.io)
    a = p.arrays
    x = [dev(a["qkv_pre"], t), dev(a["z"], t), dev(a["g"]), dev(a["beta"]), dev(a["conv_w"], t),
         dev(a["norm_w"], t)]
    S0, conv0 = dev(a["S0"]), dev(a["conv0"], t)
    o, S_T, conv_T = gdn.alloc_prefill_outputs(p.B, p.T, p.Hk, p.Hv, t)
    if path in ("fused", "serial"):
        gdn.gdn_prefill(*x, S0, conv0, o, S_T, conv_T, Hk=p.Hk, Hv=p.Hv)
    elif path in ("staged", "split"):
        gdn.gdn_prefill_ex(*x, S0, conv0, o, S_T, conv_T, Hk=p.Hk, Hv=p.Hv,
                           workspace=prefill_workspace(p.B, p.T, p.Hk, p.Hv, form=path))
    elif path == "decode":
        S_T = S0.clone()
        gdn.gdn_decode_ex(*x, S_T, conv0, conv_T, o, Hk=p.Hk, Hv=p.Hv)
    elif path == "decode_step":
        S_T = S0.clone()
        win = [conv0.clone(), torch.empty_like(conv0)]
        ot = torch.empty(p.B, p.Hv * D, device="cuda", dtype=t)
        for s in range(p.T):
            gdn.gdn_decode_step(x[0][:, s].contiguous(), x[1][:, s].contiguous(), x[2][:, s].contiguous(),
                                x[3][:, s].contiguous(), x[4], x[5], S_T, win[s % 2], win[(s + 1) % 2], ot,
                                Hk=p.Hk, Hv=p.Hv)
            o[:, s] = ot
        conv_T = win[p.T % 2]
    else:
        raise ValueError(path)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    return o, S_T, conv_T


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("kind", KINDS)
def test_edge_case(kind, path):
    io, T = PATHS[path]
    B, Hk, Hv = 2, 2, 4
    p = edge_problem(kind, B, T, Hk, Hv, io, case=500 + KINDS.index(kind))
    o, S_T, conv_T = run_path(path, p)
    a = p.arrays
    ref = O.gdn_prefill(a["qkv_pre"], a["z"], a["g"], a["beta"], a["conv_w"], a["norm_w"], a["S0"], a["conv0"],
                        Hk=Hk, Hv=Hv, threads=O.default_threads())
    check_o(to_np(o), ref["o"], io, "o (%s, %s)" % (kind, path))
    check_S(to_np(S_T), ref["S_T"], "S_T (%s, %s)" % (kind, path))
    np.testing.assert_array_equal(to_np(conv_T), ref["conv_T"])
    if kind == "frozen":  # beta = 0, g = 0: every path passes the state through unchanged
        assert torch.equal(S_T, dev(a["S0"]))


@pytest.mark.parametrize("path", ["fused", "staged", "split"])
def test_reset_at_every_chunk_boundary_and_3_heads_per_key(path):
    """g = -inf on the first token of every chunk of one head and the last
    token of every chunk of another, with three value heads per key head."""
    B, T, Hk, Hv = 1, 260, 2, 6
    p = I.prefill_problem(B, T, Hk, Hv, io="bf16", case=520, s0_std=0.02, conv0=True)
    g = p.arrays["g"]
    g[:, 0::64, 1] = -np.inf
    g[:, 63::64, 4] = -np.inf
    g[:, 31::64, 5] = -np.inf
    o, S_T, conv_T = run_path(path, p)
    a = p.arrays
    ref = O.gdn_prefill(a["qkv_pre"], a["z"], a["g"], a["beta"], a["conv_w"], a["norm_w"], a["S0"], a["conv0"],
                        Hk=Hk, Hv=Hv, threads=O.default_threads())
    check_o(to_np(o), ref["o"], "bf16")
    check_S(to_np(S_T), ref["S_T"])
