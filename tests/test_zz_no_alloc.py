"""The allocation-free entry point gdn_prefill_static against gdn_prefill_ex
with a caller workspace: the same kernels, so two calls in a row through the
library's own scratch (the second one reusing what the first left there)
must give bit-identical outputs."""
import ctypes

import numpy as np
import pytest
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I

from gpu_harness import dev, prefill_workspace, torch_io

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_mixer_gb300 import build
    build.build()
    gdn.lib()
    assert torch.cuda.is_available()
    assert gdn.gdn_device_status(reset=True) == 0


def _inputs(p):
    t = torch_io(p.io)
    a = p.arrays
    return [dev(a["qkv_pre"], t), dev(a["z"], t), dev(a["g"]), dev(a["beta"]), dev(a["conv_w"], t),
            dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t)]


def _run(fn, p, x, **kw):
    o, S_T, conv_T = gdn.alloc_prefill_outputs(p.B, p.T, p.Hk, p.Hv, torch_io(p.io))
    fn(*x, o, S_T, conv_T, Hk=p.Hk, Hv=p.Hv, **kw)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
    return o, S_T, conv_T


def test_static_entry_matches_the_workspace_entry_over_two_calls():
    problems = [I.prefill_problem(2, 200, 2, 4, io="bf16", case=450),
                I.prefill_problem(3, 130, 1, 3, io="bf16", case=451)]
    inputs = [_inputs(p) for p in problems]
    got = [_run(gdn.gdn_prefill_static, p, x) for p, x in zip(problems, inputs)]  # back to back
    for p, x, g in zip(problems, inputs, got):
        want = _run(gdn.gdn_prefill_ex, p, x, workspace=prefill_workspace(p.B, p.T, p.Hk, p.Hv))
        for a, b in zip(g, want):
            assert torch.equal(a, b)


def test_static_entry_packed_matches_the_workspace_entry():
    """A packed batch (cu_seqlens, lengths 0 to 150) through the static scratch
    and through a caller workspace: bit-identical outputs."""
    lens = [37, 0, 150, 1, 64, 99]
    p = I.packed_problem(lens, 2, 4, io="bf16", case=453)
    a = p.arrays
    t = torch.bfloat16
    cu = torch.from_numpy(p.cu_seqlens).to("cuda")
    x = [dev(a["qkv_pre"], t), dev(a["z"], t), dev(a["g"]), dev(a["beta"]), dev(a["conv_w"], t),
         dev(a["norm_w"], t), dev(a["S0"]), dev(a["conv0"], t)]

    def run(fn, **kw):
        o = torch.empty(p.N, 4 * D, device="cuda", dtype=t)
        S_T = torch.empty(len(lens), 4, D, D, device="cuda")
        conv_T = torch.empty(len(lens), 3, p.C, device="cuda", dtype=t)
        fn(*x, o, S_T, conv_T, Hk=2, Hv=4, cu_seqlens=cu, **kw)
        torch.cuda.synchronize()
        assert gdn.gdn_device_status() == 0
        return o, S_T, conv_T

    got = [run(gdn.gdn_prefill_static) for _ in range(2)]
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(len(lens), p.N, 2, 4, packed=True), dtype=torch.uint8,
                     device="cuda")
    want = run(gdn.gdn_prefill_ex, workspace=ws)
    for g in got:
        for u, v in zip(g, want):
            assert torch.equal(u, v)


def _c_call(shape, workspace=None, workspace_bytes=0):
    """gdn_prefill_static called straight through the C ABI with small valid
    buffers (the checks under test return before any of them is read)."""
    L = gdn.lib()
    buf = torch.zeros(1 << 16, device="cuda", dtype=torch.float32)
    p = buf.data_ptr()
    io = gdn.gdn_prefill_io(p, p + 4096, p + 8192, p + 12288, None, p + 16384, p + 20480, None, None,
                            p + 24576, p + 32768, p + 40960, None, None,
                            None if workspace is None else workspace.data_ptr(), workspace_bytes)
    return L.gdn_prefill_static(ctypes.byref(shape), ctypes.byref(io), None)


def test_static_entry_rejects_a_workspace_and_oversize_shapes():
    p = I.prefill_problem(1, 64, 1, 1, io="bf16", case=452)
    x = _inputs(p)
    with pytest.raises(ValueError):
        _run(gdn.gdn_prefill_static, p, x, workspace=prefill_workspace(p.B, p.T, p.Hk, p.Hv))
    # through the C ABI: a workspace is an invalid argument
    ws = prefill_workspace(1, 64, 1, 1)
    sh = gdn.make_shape(1, 64, 1, 1, D, gdn.GDN_BF16)
    assert _c_call(sh, ws, ws.numel()) == gdn.GDN_ERR_INVALID_ARG
    # one token row more than the scratch holds at Hk=16: unsupported, before any launch
    rows = gdn.GDN_STATIC_SCRATCH_BYTES // (3 * 16 * D * 2) + 1
    assert gdn.gdn_prefill_workspace_bytes(1, rows, 16, 16) > gdn.GDN_STATIC_SCRATCH_BYTES
    assert _c_call(gdn.make_shape(1, rows, 16, 16, D, gdn.GDN_BF16)) == 2  # GDN_ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == 0
