"""GPU parity of the extended entry points against the fp64 oracle:
raw gate preparation (section 9.5 of "How Qwen3.5 works"), packed
variable-length prefill (cu_seqlens), per-token state snapshots and
multi-token decoding from the cache (section 13 of the same page)."""
import numpy as np
import pytest
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I
from oracle import oracle as O

from gpu_harness import check_o, check_S, dev, to_np, torch_io

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_mixer_gb300 import build
    build.build()
    gdn.lib()
    assert torch.cuda.is_available()
    assert gdn.gdn_device_status(reset=True) == 0


def _raw_dev(a, t):
    return dict(a=dev(a["a"], t), b=dev(a["b"], t), A_log=dev(a["A_log"]), dt_bias=dev(a["dt_bias"]))


def _raw_np(a):
    return {k: a[k] for k in ("a", "b", "A_log", "dt_bias")}


# ------------------------------------------------------------- raw gates ----
@pytest.mark.parametrize("io,T", [("bf16", 1), ("bf16", 130), ("f32", 70)])
def test_prefill_raw_gates(io, T):
    B, Hk, Hv = 2, 2, 4
    p = I.prefill_problem(B, T, Hk, Hv, io=io, case=100 + T)
    rg = I.raw_gate_arrays(100 + T, (B, T), Hv, io)
    t = torch_io(io)
    a = p.arrays
    o, S_T, conv_T = gdn.alloc_prefill_outputs(B, T, Hk, Hv, t)
    gdn.gdn_prefill_ex(dev(a["qkv_pre"], t), dev(a["z"], t), None, None, dev(a["conv_w"], t),
                       dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t), o, S_T, conv_T,
                       Hk=Hk, Hv=Hv, raw_gates=_raw_dev(rg, t))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    ref = O.gdn_prefill(a["qkv_pre"], a["z"], None, None, a["conv_w"], a["norm_w"], a["S0"],
                        a["conv0"], Hk=Hk, Hv=Hv, raw_gates=_raw_np(rg),
                        threads=O.default_threads())
    check_o(to_np(o), ref["o"], io)
    check_S(to_np(S_T), ref["S_T"])
    np.testing.assert_array_equal(to_np(conv_T), ref["conv_T"])


def test_decode_raw_gates():
    dp = I.decode_problem(B=4, Hk=2, Hv=6, io="bf16", steps=1, case=110)
    rg = I.raw_gate_arrays(110, (4, 1), 6, "bf16")
    t = torch.bfloat16
    S = dev(dp.S)
    conv_out = torch.empty(4, 3, dp.C, device="cuda", dtype=t)
    o = torch.empty(4, 1, 6 * D, device="cuda", dtype=t)
    gdn.gdn_decode_ex(dev(dp.qkv_pre[0][:, None], t), dev(dp.z[0][:, None], t), None, None,
                      dev(dp.conv_w, t), dev(dp.norm_w, t), S, dev(dp.conv, t), conv_out, o,
                      Hk=2, Hv=6, raw_gates=_raw_dev(rg, t))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    ref = O.gdn_decode_multi(dp.qkv_pre[0][:, None], dp.z[0][:, None], None, None, dp.conv_w,
                             dp.norm_w, dp.S, dp.conv, Hk=2, Hv=6, raw_gates=_raw_np(rg))
    check_o(to_np(o), ref["o"], "bf16")
    check_S(to_np(S), ref["S"])
    np.testing.assert_array_equal(to_np(conv_out), ref["conv_out"])


# ------------------------------------------------------------ varlen -------
def _run_packed(p, raw=False, snap=False):
    t = torch_io(p.io)
    a = p.arrays
    B, N = len(p.lengths), p.N
    o = torch.full((N, p.Hv * D), 7.0, device="cuda", dtype=t)
    S_T = torch.empty(B, p.Hv, D, D, device="cuda")
    conv_T = torch.empty(B, 3, p.C, device="cuda", dtype=t)
    S_snap = torch.empty(N, p.Hv, D, D, device="cuda") if snap else None
    cu = torch.from_numpy(p.cu_seqlens).to("cuda")
    gdn.gdn_prefill_ex(dev(a["qkv_pre"], t), dev(a["z"], t), dev(a["g"]), dev(a["beta"]),
                       dev(a["conv_w"], t), dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t),
                       o, S_T, conv_T, Hk=p.Hk, Hv=p.Hv, cu_seqlens=cu, S_snap=S_snap,
                       raw_gates=_raw_dev(a, t) if raw else None)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    return o, S_T, conv_T, S_snap


def _check_packed(p, got, raw=False):
    o, S_T, conv_T, _ = got
    a = p.arrays
    keep = [s for s, n in enumerate(p.lengths) if n > 0]
    cu = p.cu_seqlens
    sub = I.PackedProblem(tuple(p.lengths[s] for s in keep), p.Hk, p.Hv, p.io)
    ref = O.gdn_prefill_varlen(a["qkv_pre"], a["z"], a["g"], a["beta"], a["conv_w"], a["norm_w"],
                               sub.cu_seqlens, None if a["S0"] is None else a["S0"][keep],
                               None if a["conv0"] is None else a["conv0"][keep], Hk=p.Hk, Hv=p.Hv,
                               raw_gates=_raw_np(a) if raw else None, threads=O.default_threads())
    check_o(to_np(o), ref["o"], p.io)
    check_S(to_np(S_T)[keep], ref["S_T"])
    np.testing.assert_array_equal(to_np(conv_T)[keep], ref["conv_T"])
    for s, n in enumerate(p.lengths):  # empty sequences pass state and window through
        if n == 0:
            want_S = np.zeros((p.Hv, D, D)) if a["S0"] is None else a["S0"][s]
            np.testing.assert_array_equal(to_np(S_T)[s], want_S)
            want_c = np.zeros((3, p.C)) if a["conv0"] is None else a["conv0"][s]
            np.testing.assert_array_equal(to_np(conv_T)[s], want_c)
    assert cu[-1] == o.shape[0]


LENGTHS = [(1, 2, 3, 64, 65, 130, 63), (300, 0, 5, 129), (64,), tuple(range(1, 40))]


@pytest.mark.parametrize("lengths", LENGTHS)
def test_varlen_bf16(lengths):
    p = I.packed_problem(lengths, 2, 4, io="bf16", case=120 + len(lengths))
    _check_packed(p, _run_packed(p))


def test_varlen_bf16_no_state_raw_gates():
    p = I.packed_problem((70, 1, 200, 3), 1, 3, io="bf16", case=125, state=False, raw_gates=True)
    _check_packed(p, _run_packed(p, raw=True), raw=True)


def test_varlen_f32():
    p = I.packed_problem((5, 40, 0, 33), 2, 2, io="f32", case=126)
    _check_packed(p, _run_packed(p))


def test_varlen_equal_lengths_match_batched_kernel():
    """Equal-length packed sequences give the fixed-length call's outputs."""
    p = I.prefill_problem(3, 100, 2, 4, io="bf16", case=127)
    a = p.arrays
    t = torch.bfloat16
    o, S_T, conv_T = gdn.alloc_prefill_outputs(3, 100, 2, 4, t)
    gdn.gdn_prefill(dev(a["qkv_pre"], t), dev(a["z"], t), dev(a["g"]), dev(a["beta"]),
                    dev(a["conv_w"], t), dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t),
                    o, S_T, conv_T, Hk=2, Hv=4)
    q = I.PackedProblem((100, 100, 100), 2, 4, "bf16")
    q.arrays = dict(a, qkv_pre=a["qkv_pre"].reshape(300, -1), z=a["z"].reshape(300, -1),
                    g=a["g"].reshape(300, -1), beta=a["beta"].reshape(300, -1))
    po, pS, pc, _ = _run_packed(q)
    assert torch.equal(po, o.view(300, -1))
    assert torch.equal(pS, S_T)
    assert torch.equal(pc, conv_T)


def test_varlen_bad_offsets_are_reported_and_skipped():
    p = I.packed_problem((4, 4, 4), 1, 2, io="bf16", case=128)
    a = p.arrays
    t = torch.bfloat16
    o = torch.full((12, 2 * D), 7.0, device="cuda", dtype=t)
    S_T = torch.full((3, 2, D, D), 5.0, device="cuda")
    conv_T = torch.full((3, 3, p.C), 3.0, device="cuda", dtype=t)
    cu = torch.tensor([0, 8, 4, 1 << 20], dtype=torch.int32, device="cuda")  # seq 1 and 2 unusable
    gdn.gdn_prefill_ex(dev(a["qkv_pre"], t), dev(a["z"], t), dev(a["g"]), dev(a["beta"]),
                       dev(a["conv_w"], t), dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t),
                       o, S_T, conv_T, Hk=1, Hv=2, cu_seqlens=cu)
    assert gdn.gdn_device_status(reset=True) == gdn.GDN_ERR_INVALID_ARG
    assert gdn.gdn_device_status() == 0
    assert bool((S_T[1:] == 5.0).all()) and bool((conv_T[1:] == 3.0).all())
    assert bool((o[8:] == 7.0).all())
    ref = O.gdn_prefill_varlen(a["qkv_pre"][:8], a["z"][:8], a["g"][:8], a["beta"][:8],
                               a["conv_w"], a["norm_w"], [0, 8], a["S0"][:1], a["conv0"][:1],
                               Hk=1, Hv=2)
    check_o(to_np(o[:8]), ref["o"], "bf16")
    check_S(to_np(S_T[:1]), ref["S_T"])


# ------------------------------------------------- snapshots, multi-token ----
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_prefill_snapshots(io):
    p = I.packed_problem((9, 3), 1, 2, io=io, case=130)
    got = _run_packed(p, snap=True)
    a = p.arrays
    snap = to_np(got[3])
    for s, (lo, hi) in enumerate(zip(p.cu_seqlens[:-1], p.cu_seqlens[1:])):
        ref = O.gdn_prefill(a["qkv_pre"][None, lo:hi], a["z"][None, lo:hi], a["g"][None, lo:hi],
                            a["beta"][None, lo:hi], a["conv_w"], a["norm_w"], a["S0"][s:s + 1],
                            a["conv0"][s:s + 1], Hk=1, Hv=2, want_snap=True)
        for t in range(hi - lo):
            check_S(snap[lo + t], ref["S_snap"][0, t], "S_snap[%d]" % (lo + t))
        np.testing.assert_array_equal(snap[hi - 1], to_np(got[1])[s])


@pytest.mark.parametrize("io,T,raw", [("bf16", 2, False), ("bf16", 4, True), ("f32", 3, False),
                                      ("bf16", 1, False), ("bf16", 16, False), ("bf16", 20, True)])
def test_multi_token_decode(io, T, raw):
    B, Hk, Hv = 5, 2, 6
    dp = I.decode_problem(B=B, Hk=Hk, Hv=Hv, io=io, steps=T, case=140 + T)
    t = torch_io(io)
    qkv = np.ascontiguousarray(dp.qkv_pre.transpose(1, 0, 2))  # [B, T, C]
    z = np.ascontiguousarray(dp.z.transpose(1, 0, 2))
    g = np.ascontiguousarray(dp.g.transpose(1, 0, 2))
    beta = np.ascontiguousarray(dp.beta.transpose(1, 0, 2))
    rg = I.raw_gate_arrays(140 + T, (B, T), Hv, io) if raw else None
    S = dev(dp.S)
    snap = torch.empty(B, T, Hv, D, D, device="cuda")
    conv_out = torch.empty(B, 3, dp.C, device="cuda", dtype=t)
    o = torch.empty(B, T, Hv * D, device="cuda", dtype=t)
    gdn.gdn_decode_ex(dev(qkv, t), dev(z, t), None if raw else dev(g), None if raw else dev(beta),
                      dev(dp.conv_w, t), dev(dp.norm_w, t), S, dev(dp.conv, t), conv_out, o,
                      Hk=Hk, Hv=Hv, S_snap=snap, raw_gates=_raw_dev(rg, t) if raw else None)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    ref = O.gdn_decode_multi(qkv, z, None if raw else g, None if raw else beta, dp.conv_w,
                             dp.norm_w, dp.S, dp.conv, Hk=Hk, Hv=Hv,
                             raw_gates=_raw_np(rg) if raw else None)
    check_o(to_np(o), ref["o"], io)
    check_S(to_np(S), ref["S"])
    for k in range(T):
        check_S(to_np(snap[:, k]), ref["S_snap"][:, k], "S_snap[%d]" % k)
    assert torch.equal(snap[:, -1], S)
    np.testing.assert_array_equal(to_np(conv_out), ref["conv_out"])


@pytest.mark.parametrize("io,T,snap,raw", [("bf16", 2, False, False), ("bf16", 5, True, False),
                                           ("bf16", 8, False, True), ("bf16", 13, False, False),
                                           ("f32", 3, True, False)])
def test_multi_token_decode_many_units(io, T, snap, raw):
    """More (sequence, value head) pairs than the persistent T-token kernel has
    CTAs (768 against two per SM), so that each CTA walks two or three pairs
    and every pair after its first arrives by the prefetch (state, raw rows,
    window, conv weights and z by asynchronous copy with bf16 io, gates in
    registers; with fp32 io the state alone)."""
    B, Hk, Hv = 128, 2, 6
    dp = I.decode_problem(B=B, Hk=Hk, Hv=Hv, io=io, steps=T, case=160 + T)
    t = torch_io(io)
    qkv = np.ascontiguousarray(dp.qkv_pre.transpose(1, 0, 2))
    z = np.ascontiguousarray(dp.z.transpose(1, 0, 2))
    g = np.ascontiguousarray(dp.g.transpose(1, 0, 2))
    beta = np.ascontiguousarray(dp.beta.transpose(1, 0, 2))
    rg = I.raw_gate_arrays(160 + T, (B, T), Hv, io) if raw else None
    S = dev(dp.S)
    snaps = torch.empty(B, T, Hv, D, D, device="cuda") if snap else None
    conv_out = torch.empty(B, 3, dp.C, device="cuda", dtype=t)
    o = torch.empty(B, T, Hv * D, device="cuda", dtype=t)
    gdn.gdn_decode_ex(dev(qkv, t), dev(z, t), None if raw else dev(g), None if raw else dev(beta),
                      dev(dp.conv_w, t), dev(dp.norm_w, t), S, dev(dp.conv, t), conv_out, o,
                      Hk=Hk, Hv=Hv, S_snap=snaps, raw_gates=_raw_dev(rg, t) if raw else None)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    ref = O.gdn_decode_multi(qkv, z, None if raw else g, None if raw else beta, dp.conv_w,
                             dp.norm_w, dp.S, dp.conv, Hk=Hk, Hv=Hv,
                             raw_gates=_raw_np(rg) if raw else None)
    check_o(to_np(o), ref["o"], io)
    check_S(to_np(S), ref["S"])
    if snap:
        for k in range(T):
            check_S(to_np(snaps[:, k]), ref["S_snap"][:, k], "S_snap[%d]" % k)
    np.testing.assert_array_equal(to_np(conv_out), ref["conv_out"])


def test_decode_ex_single_token_matches_decode_step():
    dp = I.decode_problem(B=3, Hk=1, Hv=2, io="bf16", steps=1, case=150)
    t = torch.bfloat16
    S1, S2 = dev(dp.S), dev(dp.S)
    c1 = torch.empty(3, 3, dp.C, device="cuda", dtype=t)
    c2 = torch.empty_like(c1)
    o1 = torch.empty(3, 2 * D, device="cuda", dtype=t)
    o2 = torch.empty(3, 1, 2 * D, device="cuda", dtype=t)
    args = (dev(dp.conv_w, t), dev(dp.norm_w, t))
    gdn.gdn_decode_step(dev(dp.qkv_pre[0], t), dev(dp.z[0], t), dev(dp.g[0]), dev(dp.beta[0]),
                        *args, S1, dev(dp.conv, t), c1, o1, Hk=1, Hv=2)
    gdn.gdn_decode_ex(dev(dp.qkv_pre[0][:, None], t), dev(dp.z[0][:, None], t),
                      dev(dp.g[0][:, None]), dev(dp.beta[0][:, None]), *args, S2, dev(dp.conv, t),
                      c2, o2, Hk=1, Hv=2)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2) and torch.equal(c1, c2) and torch.equal(o1, o2[:, 0])


# ------------------------------ the bench's extended workloads, full size ----
def test_bench_packed_batch_sampled():
    """The benchmark's packed batch (24 sequences, log-uniform lengths
    100..4000, 4B head shape) in its launch configuration; sampled units of
    the longest, the shortest and a middle sequence against the oracle."""
    import bench
    lens = bench.varlen_lengths()
    p = I.packed_problem(lens, 16, 32, io="bf16", case=61)
    o, S_T, conv_T, _ = _run_packed(p)
    a = p.arrays
    cu = p.cu_seqlens
    order = np.argsort(lens)
    for s in (int(order[-1]), int(order[0]), int(order[len(lens) // 2])):
        lo, hi = int(cu[s]), int(cu[s + 1])
        units = [s * 32 + 0, s * 32 + 17]
        ref = O.gdn_prefill(a["qkv_pre"][None, lo:hi], a["z"][None, lo:hi], a["g"][None, lo:hi],
                            a["beta"][None, lo:hi], a["conv_w"], a["norm_w"], a["S0"][s:s + 1],
                            a["conv0"][s:s + 1], Hk=16, Hv=32, units=[u - s * 32 for u in units],
                            threads=O.default_threads())
        got_o = np.stack([to_np(o[lo:hi].view(hi - lo, 32, D)[:, u - s * 32]) for u in units])
        check_o(got_o, ref["o_units"], "bf16")
        check_S(np.stack([to_np(S_T[s, u - s * 32]) for u in units]), ref["S_T"])
        np.testing.assert_array_equal(to_np(conv_T[s]), ref["conv_T"][0])


def test_bench_multi_token_decode_sampled():
    """The benchmark's 4-token decode with snapshots at the 27B decode shape
    (B=256, Hv=48), three sequences checked on every output and snapshot."""
    B, Hk, Hv, T = 256, 16, 48, 4
    dp = I.decode_problem(B=B, Hk=Hk, Hv=Hv, io="bf16", steps=T, case=74)
    t = torch.bfloat16
    qkv = np.ascontiguousarray(dp.qkv_pre.transpose(1, 0, 2))
    z = np.ascontiguousarray(dp.z.transpose(1, 0, 2))
    g = np.ascontiguousarray(dp.g.transpose(1, 0, 2))
    beta = np.ascontiguousarray(dp.beta.transpose(1, 0, 2))
    S = dev(dp.S)
    snap = torch.empty(B, T, Hv, D, D, device="cuda")
    conv_out = torch.empty(B, 3, dp.C, device="cuda", dtype=t)
    o = torch.empty(B, T, Hv * D, device="cuda", dtype=t)
    gdn.gdn_decode_ex(dev(qkv, t), dev(z, t), dev(g), dev(beta), dev(dp.conv_w, t), dev(dp.norm_w, t), S,
                      dev(dp.conv, t), conv_out, o, Hk=Hk, Hv=Hv, S_snap=snap)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    seqs = [0, 131, 255]
    ref = O.gdn_decode_multi(qkv[seqs], z[seqs], g[seqs], beta[seqs], dp.conv_w, dp.norm_w, dp.S[seqs],
                             dp.conv[seqs], Hk=Hk, Hv=Hv, threads=O.default_threads())
    check_o(to_np(o[seqs]), ref["o"], "bf16")
    check_S(to_np(S[seqs]), ref["S"])
    for k in range(T):
        check_S(to_np(snap[seqs, k]), ref["S_snap"][:, k], "S_snap[%d]" % k)
    np.testing.assert_array_equal(to_np(conv_out[seqs]), ref["conv_out"])
