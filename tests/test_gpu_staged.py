"""GPU parity of the staged q^ / k^ path of gdn_prefill_ex (a workspace is
given: the normalised q and k of each key head are formed once by their own
kernel and read back by TMA) against the fp64 oracle, on the shapes and
options of the fused path: ragged lengths, head ratios 1 to 3, raw gates,
packed sequences (with empty and short ones), and the 4B-shaped workload."""
import numpy as np
import pytest
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I
from oracle import oracle as O

from gpu_harness import (check_o, check_S, compare_prefill, dev, gpu_prefill, prefill_workspace, to_np,
                         torch_io)

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_mixer_gb300 import build
    build.build()
    gdn.lib()
    assert torch.cuda.is_available()
    assert gdn.gdn_device_status(reset=True) == 0


@pytest.mark.parametrize("B,T,Hk,Hv,state", [(1, 1, 1, 1, True), (2, 63, 1, 2, False), (1, 64, 2, 4, True),
                                             (2, 130, 2, 6, True), (3, 200, 1, 3, False), (1, 257, 4, 4, True)])
def test_staged_prefill(B, T, Hk, Hv, state):
    p = I.prefill_problem(B, T, Hk, Hv, io="bf16", case=400 + T, s0_std=0.02 if state else 0.0, conv0=state)
    compare_prefill(p, gpu_prefill(p, staged=True))


def test_staged_and_fused_share_the_window_and_agree():
    """Both paths carry the same raw window out; their outputs differ only by
    the rounding of Gamma k^ (formed from k^'s hi + lo pair in the staged
    path), far inside the tolerance."""
    p = I.prefill_problem(2, 300, 2, 4, io="bf16", case=430)
    x = None
    fo, fS, fc = gpu_prefill(p, inputs=x)
    so, sS, sc = gpu_prefill(p, staged=True)
    assert torch.equal(fc, sc)
    rms = fS.pow(2).mean().sqrt()
    assert (sS - fS).abs().max() <= 1e-3 * rms


def test_staged_raw_gates():
    B, T, Hk, Hv = 2, 150, 2, 4
    p = I.prefill_problem(B, T, Hk, Hv, io="bf16", case=431)
    rg = I.raw_gate_arrays(431, (B, T), Hv, "bf16")
    t = torch.bfloat16
    a = p.arrays
    o, S_T, conv_T = gdn.alloc_prefill_outputs(B, T, Hk, Hv, t)
    gdn.gdn_prefill_ex(dev(a["qkv_pre"], t), dev(a["z"], t), None, None, dev(a["conv_w"], t),
                       dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t), o, S_T, conv_T, Hk=Hk, Hv=Hv,
                       raw_gates=dict(a=dev(rg["a"], t), b=dev(rg["b"], t), A_log=dev(rg["A_log"]),
                                      dt_bias=dev(rg["dt_bias"])),
                       workspace=prefill_workspace(B, T, Hk, Hv, form="staged"))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    ref = O.gdn_prefill(a["qkv_pre"], a["z"], None, None, a["conv_w"], a["norm_w"], a["S0"], a["conv0"],
                        Hk=Hk, Hv=Hv, raw_gates={k: rg[k] for k in ("a", "b", "A_log", "dt_bias")},
                        threads=O.default_threads())
    check_o(to_np(o), ref["o"], "bf16")
    check_S(to_np(S_T), ref["S_T"])
    np.testing.assert_array_equal(to_np(conv_T), ref["conv_T"])


@pytest.mark.parametrize("lengths", [(1, 2, 3, 64, 65, 130, 63), (300, 0, 5, 129), tuple(range(1, 30))])
def test_staged_packed(lengths):
    """Packed sequences: every token's window stops at its own sequence start
    (rows before it come from that sequence's carried window)."""
    p = I.packed_problem(lengths, 2, 4, io="bf16", case=440 + len(lengths))
    a = p.arrays
    t = torch_io(p.io)
    B, N = len(p.lengths), p.N
    o = torch.full((N, p.Hv * D), 7.0, device="cuda", dtype=t)
    S_T = torch.empty(B, p.Hv, D, D, device="cuda")
    conv_T = torch.empty(B, 3, p.C, device="cuda", dtype=t)
    cu = torch.from_numpy(p.cu_seqlens).to("cuda")
    gdn.gdn_prefill_ex(dev(a["qkv_pre"], t), dev(a["z"], t), dev(a["g"]), dev(a["beta"]), dev(a["conv_w"], t),
                       dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t), o, S_T, conv_T, Hk=p.Hk, Hv=p.Hv,
                       cu_seqlens=cu, workspace=prefill_workspace(B, N, p.Hk, p.Hv, packed=True, form="staged"))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    keep = [s for s, n in enumerate(p.lengths) if n > 0]
    sub = I.PackedProblem(tuple(p.lengths[s] for s in keep), p.Hk, p.Hv, p.io)
    ref = O.gdn_prefill_varlen(a["qkv_pre"], a["z"], a["g"], a["beta"], a["conv_w"], a["norm_w"],
                               sub.cu_seqlens, a["S0"][keep], a["conv0"][keep], Hk=p.Hk, Hv=p.Hv,
                               threads=O.default_threads())
    check_o(to_np(o), ref["o"], p.io)
    check_S(to_np(S_T)[keep], ref["S_T"])
    np.testing.assert_array_equal(to_np(conv_T)[keep], ref["conv_T"])


def test_staged_4b_prefill_sampled():
    """The benchmark's workload through the staged path: Qwen3.5-4B-shaped,
    B=4, T=8192, 16/32 heads, full launch, units from every sequence and both
    value heads of a key head."""
    p = I.case_problem("4b_prefill")
    got = gpu_prefill(p, staged=True)
    assert torch.isfinite(got[0].float()).all()
    compare_prefill(p, got, units=[0, 1, 45, 70, 127])


def test_staged_27b_prefill_sampled():
    """The long 27B-shaped prefill (T=65536, 16/48 heads: three value heads
    per key head) through the staged path."""
    p = I.case_problem("27b_prefill")
    got = gpu_prefill(p, staged=True)
    compare_prefill(p, got, units=[0, 2, 25, 47])
