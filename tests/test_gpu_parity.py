"""GPU parity: libgdn (through its C ABI) against the fp64 oracle on the same
seeded inputs.  Small cases are compared element by element on every output;
the full-size model shapes run in the benchmark's launch configuration and are
compared on sampled (sequence, head) units the oracle computes one by one."""
import numpy as np
import pytest
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I
from oracle import oracle as O

from gpu_harness import (check_o, check_S, compare_prefill, dev, gpu_prefill, oracle_prefill,
                         to_np, torch_io, upload_prefill)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_mixer_gb300 import build
    build.build()
    gdn.lib()
    assert torch.cuda.is_available()


def test_tiny_fp32_mixer():
    """The tiny full mixer: B=1, T=64, Hk=1, Hv=2, fp32 io, zero state."""
    p = I.case_problem("tiny")
    compare_prefill(p, gpu_prefill(p))


@pytest.mark.parametrize("B,T,Hk,Hv,state", [
    (2, 1, 1, 2, True), (2, 2, 2, 4, True), (1, 3, 1, 1, False), (1, 67, 2, 6, True),
    (2, 130, 1, 1, True), (1, 300, 2, 2, False), (3, 64, 2, 4, True), (1, 129, 4, 8, True)])
def test_small_bf16_prefill(B, T, Hk, Hv, state):
    p = I.prefill_problem(B, T, Hk, Hv, io="bf16", case=50 + T,
                          s0_std=0.02 if state else 0.0, conv0=state)
    compare_prefill(p, gpu_prefill(p))


def test_prefill_in_place_state():
    p = I.prefill_problem(2, 77, 2, 4, io="bf16", case=61)
    x = upload_prefill(p)
    got = gpu_prefill(p, x, in_place=True)
    assert got[1].data_ptr() == x["S0"].data_ptr()
    compare_prefill(p, got)


def test_prefill_continuation_on_gpu():
    """Prefill(a ++ b) and prefill(b) started from prefill(a)'s state and window
    (the carried cache of 'How Qwen3.5 works' section 13) both match the
    oracle's single pass; the carried windows agree bit for bit."""
    p = I.prefill_problem(2, 200, 2, 4, io="bf16", case=62)
    ref = oracle_prefill(p)
    whole = gpu_prefill(p)
    cut = 77
    seq = ("qkv_pre", "z", "g", "beta")
    pa = I.Problem(p.B, cut, p.Hk, p.Hv, p.io, arrays={k: (v[:, :cut] if k in seq else v)
                                                        for k, v in p.arrays.items()})
    first = gpu_prefill(pa)
    pb = I.Problem(p.B, p.T - cut, p.Hk, p.Hv, p.io,
                   arrays={k: (v[:, cut:] if k in seq else v) for k, v in p.arrays.items()})
    xb = upload_prefill(pb)
    xb["S0"], xb["conv0"] = first[1], first[2]
    second = gpu_prefill(pb, xb)
    check_o(to_np(whole[0]), ref["o"], "bf16")
    check_o(to_np(first[0]), ref["o"][:, :cut], "bf16")
    check_o(to_np(second[0]), ref["o"][:, cut:], "bf16")
    check_S(to_np(whole[1]), ref["S_T"])
    check_S(to_np(second[1]), ref["S_T"])
    np.testing.assert_array_equal(to_np(second[2]), to_np(whole[2]))


def test_head_map_bit_exact():
    """Value head h reads key head h // (Hv/Hk): with a one-hot key per key
    head, beta = 1, g = 0 and zero state, S_T[h] has its only non-zero column
    at that key head's index; the argmax must match exactly."""
    Hk, Hv, D = 4, 12, 128
    r = Hv // Hk
    C = (2 * Hk + Hv) * D
    x = np.zeros((1, 1, C), np.float32)
    for kh in range(Hk):
        x[0, 0, Hk * D + kh * D + kh] = 3.0
    x[0, 0, 2 * Hk * D:] = 1.0
    x[0, 0, :Hk * D] = 0.5
    w = np.zeros((C, 4), np.float32)
    w[:, 3] = 1.0
    t = torch.bfloat16
    o, S_T, conv_T = gdn.alloc_prefill_outputs(1, 1, Hk, Hv, t)
    ones = torch.ones(1, 1, Hv, device="cuda")
    gdn.gdn_prefill(dev(x, t), torch.ones(1, 1, Hv * D, device="cuda", dtype=t), 0 * ones, ones,
                    dev(w, t), torch.ones(D, device="cuda", dtype=t), None, None, o, S_T, conv_T,
                    Hk=Hk, Hv=Hv)
    S = to_np(S_T)[0]
    for h in range(Hv):
        col = np.abs(S[h]).sum(axis=0)
        assert int(np.argmax(col)) == h // r
        assert np.count_nonzero(col) == 1


def _decode_run(dp, seqs):
    """Run dp.steps decode steps on the GPU; return per-step o for `seqs`,
    the final state and window."""
    t = torch_io(dp.io)
    S = dev(dp.S)
    conv = [dev(dp.conv, t), torch.empty_like(dev(dp.conv, t))]
    cw, nw = dev(dp.conv_w, t), dev(dp.norm_w, t)
    o = torch.empty(dp.B, dp.Hv * 128, device="cuda", dtype=t)
    outs = []
    for s in range(dp.steps):
        gdn.gdn_decode_step(dev(dp.qkv_pre[s], t), dev(dp.z[s], t), dev(dp.g[s]),
                            dev(dp.beta[s]), cw, nw, S, conv[s % 2], conv[(s + 1) % 2], o,
                            Hk=dp.Hk, Hv=dp.Hv)
        outs.append(to_np(o[seqs]))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    return np.stack(outs, 1), to_np(S[seqs]), to_np(conv[dp.steps % 2][seqs])


def _decode_oracle(dp, seqs):
    """The same steps as one oracle prefill of dp.steps tokens per sequence
    (a decode step is a prefill of one token)."""
    q = np.ascontiguousarray(dp.qkv_pre[:, seqs].transpose(1, 0, 2))
    z = np.ascontiguousarray(dp.z[:, seqs].transpose(1, 0, 2))
    g = np.ascontiguousarray(dp.g[:, seqs].transpose(1, 0, 2))
    b = np.ascontiguousarray(dp.beta[:, seqs].transpose(1, 0, 2))
    return O.gdn_prefill(q, z, g, b, dp.conv_w, dp.norm_w, dp.S[seqs], dp.conv[seqs],
                         Hk=dp.Hk, Hv=dp.Hv, threads=O.default_threads())


def test_decode_small_64_steps():
    dp = I.decode_problem(B=3, Hk=1, Hv=2, io="bf16", steps=64, case=70)
    seqs = [0, 1, 2]
    o, S, conv = _decode_run(dp, seqs)
    ref = _decode_oracle(dp, seqs)
    check_o(o, ref["o"], "bf16")
    check_S(S, ref["S_T"])
    np.testing.assert_array_equal(conv, ref["conv_T"])


def test_decode_fp32_io():
    dp = I.decode_problem(B=2, Hk=2, Hv=4, io="f32", steps=5, case=71)
    o, S, conv = _decode_run(dp, [0, 1])
    ref = _decode_oracle(dp, [0, 1])
    check_o(o, ref["o"], "f32")
    check_S(S, ref["S_T"])
    np.testing.assert_array_equal(conv, ref["conv_T"])


def test_0p8b_prefill_full():
    """Qwen3.5-0.8B-shaped layer: B=1, T=4096, 16/16 heads, every output."""
    p = I.case_problem("0.8b_prefill")
    compare_prefill(p, gpu_prefill(p))


def test_4b_prefill_sampled():
    """Qwen3.5-4B-shaped layer: B=4, T=8192, 16/32 heads, full launch;
    sampled units cover every sequence and both value heads of a key head."""
    p = I.case_problem("4b_prefill")
    got = gpu_prefill(p)
    assert torch.isfinite(got[0].float()).all()
    compare_prefill(p, got, units=[0, 1, 45, 70, 127])


def test_27b_prefill_sampled():
    """Qwen3.8-27B-shaped long prefill: T=65536, 16/48 heads, slow decay."""
    p = I.case_problem("27b_prefill")
    got = gpu_prefill(p)
    assert got[1].numel() == 786432
    compare_prefill(p, got, units=[0, 2, 25, 47])


def test_27b_decode_sampled():
    """Qwen3.8-27B-shaped batched decode: B=256, 64 steps, full launches;
    three sequences are checked on all 64 outputs and the final state."""
    dp = I.decode_problem(**{k: v for k, v in I.DECODE_CASE.items()})
    seqs = [0, 129, 255]
    o, S, conv = _decode_run(dp, seqs)
    ref = _decode_oracle(dp, seqs)
    check_o(o, ref["o"], "bf16")
    check_S(S, ref["S_T"])
    np.testing.assert_array_equal(conv, ref["conv_T"])


def test_errors_leave_outputs_untouched():
    p = I.prefill_problem(1, 8, 1, 2, io="bf16", case=80)
    x = upload_prefill(p)
    o, S_T, conv_T = gdn.alloc_prefill_outputs(1, 8, 1, 2, torch.bfloat16)
    o.fill_(7.0)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill(x["qkv_pre"], x["z"], x["g"], x["beta"], x["conv_w"], x["norm_w"],
                        x["S0"], x["conv0"], o, S_T, x["conv0"], Hk=1, Hv=2)
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert bool((o.float() == 7.0).all())
    assert gdn.gdn_device_status() == 0
