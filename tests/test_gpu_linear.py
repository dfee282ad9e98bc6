"""GPU parity of gdn_linear (the in_proj / out_proj projections of the page
"Qwen3.8-27B", y[t,n] = sum_k x[t,k] w[n,k]) against the fp64 oracle.

Tolerance: fp32 accumulation of exact bf16 products leaves errors far below
1e-3 of the output's rms; the stored bf16 output adds its own rounding, half
an ulp <= 2^-8 |y|.  So |y_gpu - y_ref| <= 2^-8 |y_ref| + 1e-3 rms(y_ref)."""
import numpy as np
import pytest
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I
from oracle import oracle as O

from gpu_harness import dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_mixer_gb300 import build
    build.build()
    gdn.lib()
    assert torch.cuda.is_available()
    assert gdn.gdn_device_status(reset=True) == 0


def check_linear(got, ref, what="y"):
    rms = float(np.sqrt(np.mean(ref * ref)))
    excess = np.abs(got - ref) - 2.0 ** -8 * np.abs(ref)
    worst = float(np.max(excess))
    assert np.all(np.isfinite(got)), what
    assert worst <= 1e-3 * rms, "%s: max excess %.3e > %.3e (rms %.3e)" % (what, worst, 1e-3 * rms, rms)


def run(x, w, outs):
    gdn.gdn_linear(x, w, outs)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (128, 256, 64), (200, 300, 136), (257, 520, 1000),
                                   (640, 1024, 5120)])
def test_linear_single_output(M, N, K):
    xa, wa = I.linear_problem(M, N, K, case=200 + M)
    x, w = dev(xa, torch.bfloat16), dev(wa, torch.bfloat16)
    y = torch.full((M, N), 7.0, device="cuda", dtype=torch.bfloat16)
    run(x, w, [(0, N, y)])
    check_linear(to_np(y), O.linear(xa, wa))


def test_linear_strided_inputs_and_split_outputs():
    """Row strides above K, four column blocks with unaligned boundaries, a
    column range left out."""
    M, N, K = 300, 700, 200
    xa, wa = I.linear_problem(M, N, K, case=210)
    xbig = torch.zeros(M, 264, device="cuda", dtype=torch.bfloat16)
    wbig = torch.zeros(N, 208, device="cuda", dtype=torch.bfloat16)
    xbig[:, :K] = dev(xa, torch.bfloat16)
    wbig[:, :K] = dev(wa, torch.bfloat16)
    edges = [(0, 100), (100, 333), (333, 517), (520, 700)]
    full = [torch.full((M, e - b + 5), 3.0, device="cuda", dtype=torch.bfloat16) for b, e in edges]
    outs = [(b, e, f[:, :e - b]) for (b, e), f in zip(edges, full)]
    run(xbig[:, :K], wbig[:, :K], outs)
    ref = O.linear(xa, wa)
    for (b, e, t), f in zip(outs, full):
        check_linear(to_np(t), ref[:, b:e], "cols %d-%d" % (b, e))
        assert bool(f[:, e - b:].eq(3.0).all())  # row padding untouched


def test_in_proj_27b_split_into_mixer_buffers():
    """The 27B in_proj (K=5120, N=16480) writes qkv_pre, z, b and a directly."""
    T = 384
    xa, wa = I.linear_problem(T, 16480, 5120, case=220)
    x, w = dev(xa, torch.bfloat16), dev(wa, torch.bfloat16)
    sp = O.in_proj_split(16, 48, 128)
    bufs = {k: torch.empty(T, hi - lo, device="cuda", dtype=torch.bfloat16) for k, (lo, hi) in sp.items()}
    run(x, w, [(sp[k][0], sp[k][1], bufs[k]) for k in ("qkv_pre", "z", "b", "a")])
    ref = O.linear(xa, wa)
    for k, (lo, hi) in sp.items():
        check_linear(to_np(bufs[k]), ref[:, lo:hi], k)


def test_out_proj_27b():
    T = 384
    xa, wa = I.linear_problem(T, 5120, 6144, case=230)
    y = torch.empty(T, 5120, device="cuda", dtype=torch.bfloat16)
    run(dev(xa, torch.bfloat16), dev(wa, torch.bfloat16), [(0, 5120, y)])
    check_linear(to_np(y), O.linear(xa, wa))


def test_linear_host_errors_leave_outputs_untouched():
    x = torch.zeros(4, 64, device="cuda", dtype=torch.bfloat16)
    w = torch.zeros(8, 64, device="cuda", dtype=torch.bfloat16)
    y = torch.full((4, 8), 5.0, device="cuda", dtype=torch.bfloat16)
    for outs in ([(0, 9, y)], [(0, 5, y), (4, 8, y)], [(3, 2, y)]):
        with pytest.raises(gdn.GdnError) as e:
            gdn.gdn_linear(x, w, outs)
        assert e.value.status in (1, 4)
    torch.cuda.synchronize()
    assert bool((y == 5.0).all())


def test_bench_in_proj_8192_tokens_sampled_rows():
    """The benchmark's 27B in_proj (8192 tokens, split outputs) in its launch
    configuration; 64 sampled rows against the oracle on every column."""
    T = 8192
    xa, wa = I.linear_problem(T, 16480, 5120, case=80)
    x, w = dev(xa, torch.bfloat16), dev(wa, torch.bfloat16)
    sp = O.in_proj_split(16, 48, 128)
    bufs = {k: torch.empty(T, hi - lo, device="cuda", dtype=torch.bfloat16) for k, (lo, hi) in sp.items()}
    run(x, w, [(sp[k][0], sp[k][1], bufs[k]) for k in ("qkv_pre", "z", "b", "a")])
    rows = np.random.default_rng(0).choice(T, size=64, replace=False)
    ref = O.linear(xa[rows], wa)
    for k, (lo, hi) in sp.items():
        check_linear(to_np(bufs[k][rows]), ref[:, lo:hi], k)
