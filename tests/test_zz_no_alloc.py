"""The allocation-free entry point gdn_prefill_static against gdn_prefill_ex
with a caller workspace: the same kernels, so two calls in a row through the
library's own scratch (the second one reusing what the first left there)
must give bit-identical outputs."""
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


def test_static_entry_rejects_a_workspace_and_oversize_shapes():
    p = I.prefill_problem(1, 64, 1, 1, io="bf16", case=452)
    x = _inputs(p)
    with pytest.raises(ValueError):
        _run(gdn.gdn_prefill_static, p, x, workspace=prefill_workspace(p.B, p.T, p.Hk, p.Hv))
    rows = gdn.GDN_STATIC_SCRATCH_BYTES // (3 * 16 * D * 2) + 1  # one token row more than fits at Hk=16
    assert gdn.gdn_prefill_workspace_bytes(1, rows, 16, 16) > gdn.GDN_STATIC_SCRATCH_BYTES
