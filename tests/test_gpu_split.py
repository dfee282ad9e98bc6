"""GPU parity of the chunk-parallel form of gdn_prefill_ex (a workspace of
gdn_prefill_workspace_bytes: q^ / k^ staged once per key head, every chunk's
state-independent part -- T, U, W, the decayed Q K^T -- formed at once, then
one sequential pass per (sequence, value head) with the state in TMEM; for
few units of a fixed-length batch both parts share one cooperative launch)
against the fp64 oracle: ragged lengths, head ratios 1 to 3, raw gates,
packed sequences with empty and short ones, unusable offsets, in-place state,
continuation, and the model-shaped workloads."""
import numpy as np
import pytest
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I
from oracle import oracle as O

from gpu_harness import (check_o, check_S, compare_prefill, dev, gpu_prefill, oracle_prefill, prefill_workspace,
                         to_np, torch_io, upload_prefill)

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_mixer_gb300 import build
    build.build()
    gdn.lib()
    assert torch.cuda.is_available()
    assert gdn.gdn_device_status(reset=True) == 0


@pytest.mark.parametrize("B,T,Hk,Hv,state", [
    (1, 1, 1, 1, True), (2, 2, 1, 2, False), (1, 3, 1, 1, True), (2, 63, 1, 2, False), (1, 64, 2, 4, True),
    (1, 65, 1, 3, True), (2, 130, 2, 6, True), (3, 200, 1, 3, False), (1, 257, 4, 4, True), (2, 129, 4, 8, True)])
def test_split_prefill(B, T, Hk, Hv, state):
    p = I.prefill_problem(B, T, Hk, Hv, io="bf16", case=600 + T, s0_std=0.02 if state else 0.0, conv0=state)
    compare_prefill(p, gpu_prefill(p, split=True))


def test_split_many_units_two_launches():
    """More (sequence, value head) units than half the SMs: the two parts run
    as separate launches (with fewer, both run in one cooperative launch)."""
    p = I.prefill_problem(20, 130, 2, 4, io="bf16", case=629, s0_std=0.02, conv0=True)
    compare_prefill(p, gpu_prefill(p, split=True))


def test_split_and_staged_agree():
    """The split and staged forms compute the same chunked recurrence with the
    same operand roundings; they differ in summation order only, so a bf16
    output may round one unit apart."""
    p = I.prefill_problem(2, 300, 2, 4, io="bf16", case=630)
    so, sS, sc = gpu_prefill(p, staged=True)
    po, pS, pc = gpu_prefill(p, split=True)
    assert torch.equal(sc, pc)
    rms = sS.pow(2).mean().sqrt()
    assert (pS - sS).abs().max() <= 1e-3 * rms
    orms = so.float().pow(2).mean().sqrt()
    ulp = torch.exp2(torch.floor(torch.log2(so.float().abs().clamp_min(1e-30))) - 7)  # one bf16 unit of |so|
    assert ((po.float() - so.float()).abs() - ulp).max() <= 2e-2 * orms


def test_split_in_place_state_and_continuation():
    p = I.prefill_problem(2, 200, 2, 4, io="bf16", case=631)
    ref = oracle_prefill(p)
    x = upload_prefill(p)
    whole = gpu_prefill(p, x, in_place=True, split=True)
    assert whole[1].data_ptr() == x["S0"].data_ptr()
    check_o(to_np(whole[0]), ref["o"], "bf16")
    check_S(to_np(whole[1]), ref["S_T"])
    cut = 77
    seq = ("qkv_pre", "z", "g", "beta")
    pa = I.Problem(p.B, cut, p.Hk, p.Hv, p.io, arrays={k: (v[:, :cut] if k in seq else v) for k, v in p.arrays.items()})
    first = gpu_prefill(pa, split=True)
    pb = I.Problem(p.B, p.T - cut, p.Hk, p.Hv, p.io,
                   arrays={k: (v[:, cut:] if k in seq else v) for k, v in p.arrays.items()})
    xb = upload_prefill(pb)
    xb["S0"], xb["conv0"] = first[1], first[2]
    second = gpu_prefill(pb, xb, split=True)
    check_o(to_np(first[0]), ref["o"][:, :cut], "bf16")
    check_o(to_np(second[0]), ref["o"][:, cut:], "bf16")
    check_S(to_np(second[1]), ref["S_T"])


def test_split_raw_gates():
    B, T, Hk, Hv = 2, 150, 2, 4
    p = I.prefill_problem(B, T, Hk, Hv, io="bf16", case=632)
    rg = I.raw_gate_arrays(632, (B, T), Hv, "bf16")
    t = torch.bfloat16
    a = p.arrays
    o, S_T, conv_T = gdn.alloc_prefill_outputs(B, T, Hk, Hv, t)
    gdn.gdn_prefill_ex(dev(a["qkv_pre"], t), dev(a["z"], t), None, None, dev(a["conv_w"], t),
                       dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t), o, S_T, conv_T, Hk=Hk, Hv=Hv,
                       raw_gates=dict(a=dev(rg["a"], t), b=dev(rg["b"], t), A_log=dev(rg["A_log"]),
                                      dt_bias=dev(rg["dt_bias"])),
                       workspace=prefill_workspace(B, T, Hk, Hv))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    ref = O.gdn_prefill(a["qkv_pre"], a["z"], None, None, a["conv_w"], a["norm_w"], a["S0"], a["conv0"],
                        Hk=Hk, Hv=Hv, raw_gates={k: rg[k] for k in ("a", "b", "A_log", "dt_bias")},
                        threads=O.default_threads())
    check_o(to_np(o), ref["o"], "bf16")
    check_S(to_np(S_T), ref["S_T"])
    np.testing.assert_array_equal(to_np(conv_T), ref["conv_T"])


def _packed_run(p, cu):
    a = p.arrays
    t = torch_io(p.io)
    B, N = len(p.lengths), p.N
    o = torch.full((N, p.Hv * D), 7.0, device="cuda", dtype=t)
    S_T = torch.full((B, p.Hv, D, D), 3.0, device="cuda")
    conv_T = torch.full((B, 3, p.C), 5.0, device="cuda", dtype=t)
    gdn.gdn_prefill_ex(dev(a["qkv_pre"], t), dev(a["z"], t), dev(a["g"]), dev(a["beta"]), dev(a["conv_w"], t),
                       dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t), o, S_T, conv_T, Hk=p.Hk, Hv=p.Hv,
                       cu_seqlens=cu, workspace=prefill_workspace(B, N, p.Hk, p.Hv, packed=True))
    torch.cuda.synchronize()
    return o, S_T, conv_T


@pytest.mark.parametrize("lengths", [(1, 2, 3, 64, 65, 130, 63), (300, 0, 5, 129), tuple(range(1, 40)),
                                     (128, 64, 0, 0, 192)])
def test_split_packed(lengths):
    """Packed sequences: chunk slots of each sequence in the workspace, every
    token's window stopping at its own sequence's start."""
    p = I.packed_problem(lengths, 2, 4, io="bf16", case=640 + len(lengths))
    cu = torch.from_numpy(p.cu_seqlens).to("cuda")
    o, S_T, conv_T = _packed_run(p, cu)
    assert gdn.gdn_device_status() == 0
    a = p.arrays
    keep = [s for s, n in enumerate(p.lengths) if n > 0]
    sub = I.PackedProblem(tuple(p.lengths[s] for s in keep), p.Hk, p.Hv, p.io)
    ref = O.gdn_prefill_varlen(a["qkv_pre"], a["z"], a["g"], a["beta"], a["conv_w"], a["norm_w"],
                               sub.cu_seqlens, a["S0"][keep], a["conv0"][keep], Hk=p.Hk, Hv=p.Hv,
                               threads=O.default_threads())
    check_o(to_np(o), ref["o"], p.io)
    check_S(to_np(S_T)[keep], ref["S_T"])
    np.testing.assert_array_equal(to_np(conv_T)[keep], ref["conv_T"])
    empty = [s for s, n in enumerate(p.lengths) if n == 0]
    for s in empty:  # an empty sequence passes its state and window through
        assert torch.equal(S_T[s], dev(a["S0"][s]))


def test_split_packed_many_items_per_group():
    """A packed batch at the 4B head shape (about 8k tokens, 16/32 heads): each
    prep group walks a dozen work items or more across sequences of unequal
    length (the next item's loads, gates and chunk vectors prepared during the
    current one), then every output against the oracle."""
    lengths = (1500, 37, 2048, 700, 1000, 0, 2690)
    p = I.packed_problem(lengths, 16, 32, io="bf16", case=646)
    cu = torch.from_numpy(p.cu_seqlens).to("cuda")
    o, S_T, conv_T = _packed_run(p, cu)
    assert gdn.gdn_device_status() == 0
    a = p.arrays
    keep = [s for s, n in enumerate(p.lengths) if n > 0]
    sub = I.PackedProblem(tuple(p.lengths[s] for s in keep), p.Hk, p.Hv, p.io)
    ref = O.gdn_prefill_varlen(a["qkv_pre"], a["z"], a["g"], a["beta"], a["conv_w"], a["norm_w"],
                               sub.cu_seqlens, a["S0"][keep], a["conv0"][keep], Hk=p.Hk, Hv=p.Hv,
                               threads=O.default_threads())
    check_o(to_np(o), ref["o"], p.io)
    check_S(to_np(S_T)[keep], ref["S_T"])
    np.testing.assert_array_equal(to_np(conv_T)[keep], ref["conv_T"])


def test_split_packed_equal_lengths_match_fixed_length():
    """A packed batch of equal lengths uses other chunk slots than the
    fixed-length call but the same arithmetic: bit-identical outputs."""
    B, T, Hk, Hv = 3, 100, 2, 4
    p = I.prefill_problem(B, T, Hk, Hv, io="bf16", case=650)
    fo, fS, fc = gpu_prefill(p, split=True)
    a = p.arrays
    t = torch.bfloat16
    cu = torch.tensor([0, T, 2 * T, 3 * T], dtype=torch.int32, device="cuda")
    o = torch.empty(B * T, Hv * D, device="cuda", dtype=t)
    S_T = torch.empty(B, Hv, D, D, device="cuda")
    conv_T = torch.empty(B, 3, p.C, device="cuda", dtype=t)
    gdn.gdn_prefill_ex(dev(a["qkv_pre"].reshape(B * T, -1), t), dev(a["z"].reshape(B * T, -1), t),
                       dev(a["g"].reshape(B * T, -1)), dev(a["beta"].reshape(B * T, -1)), dev(a["conv_w"], t),
                       dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t), o, S_T, conv_T, Hk=Hk, Hv=Hv,
                       cu_seqlens=cu, workspace=prefill_workspace(B, B * T, Hk, Hv, packed=True))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    assert torch.equal(o.view(B, T, -1), fo)
    assert torch.equal(S_T, fS)
    assert torch.equal(conv_T, fc)


def test_split_unusable_offsets_are_reported_and_skipped():
    lengths = (40, 70, 30)
    p = I.packed_problem(lengths, 1, 2, io="bf16", case=655)
    bad = np.array([0, 90, 40, 140], dtype=np.int32)  # the second sequence's offsets decrease
    cu = torch.from_numpy(bad).to("cuda")
    o, S_T, conv_T = _packed_run(p, cu)
    assert gdn.gdn_device_status(reset=True) == gdn.GDN_ERR_INVALID_ARG
    assert bool((S_T[1] == 3.0).all())  # the skipped sequence's outputs stay untouched
    assert bool((conv_T[1].float() == 5.0).all())


def test_split_0p8b_prefill_full():
    """Qwen3.5-0.8B-shaped layer (B=1, T=4096, 16/16 heads): every output."""
    p = I.case_problem("0.8b_prefill")
    compare_prefill(p, gpu_prefill(p, split=True))


def test_split_4b_prefill_sampled():
    """The benchmark's workload: Qwen3.5-4B-shaped, B=4, T=8192, 16/32 heads,
    full launch; units from every sequence and both value heads of a key head."""
    p = I.case_problem("4b_prefill")
    got = gpu_prefill(p, split=True)
    assert torch.isfinite(got[0].float()).all()
    compare_prefill(p, got, units=[0, 1, 45, 70, 127])


def test_split_27b_prefill_sampled():
    """The long 27B-shaped prefill (T=65536, 16/48 heads, slow decay): 1024
    chunks per unit through the sequential pass."""
    p = I.case_problem("27b_prefill")
    got = gpu_prefill(p, split=True)
    assert got[1].numel() == 786432
    compare_prefill(p, got, units=[0, 2, 25, 47])
