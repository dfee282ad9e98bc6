"""Shared plumbing of the GPU parity tests: upload seeded inputs, call libgdn
through its C ABI, call the oracle on the same values, compare.

Tolerances (bf16 io, fp32 state):
  o   : max |o_gpu - o_ref| <= 2e-2 * rms(o_ref) + q(o_ref), where q is the
        rounding of the stored output (half a bf16 ulp, <= 2^-8 |o_ref|; zero
        for fp32 io) -- the arithmetic error bound plus the output's own
        quantisation, which no implementation can avoid.
  S_T : max |S_gpu - S_ref| <= 1e-2 * rms(S_ref)
  conv windows: bit-exact (they are raw copies).
"""
import numpy as np
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I
from oracle import oracle as O

O_TOL = 2e-2
S_TOL = 1e-2

# Every o comparison of the session, by yardstick (printed at the end of the
# run by conftest.py): the asserted excess over the output's rounding, the
# plain max |o_gpu - o_ref| / rms, the same against the oracle's output
# rounded to bf16 (round to nearest even), and that difference in bf16 ulps
# of the rounded reference where |o_ref| >= rms/16 (0 = every stored value is
# the correctly rounded one, 1 = off by one rounding step at most).
REPORT = []


def torch_io(io):
    return torch.bfloat16 if io == "bf16" else torch.float32


def dev(a, dtype=torch.float32):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype)


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def quantum(ref, io):
    return (2.0 ** -8) * np.abs(ref) if io == "bf16" else 0.0


def bf16_ulp(x):
    """The spacing of bf16 values at |x| (normals; 2^-133 below them)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def yardsticks(got, ref, io):
    """The o error measures of REPORT, relative to rms(ref)."""
    rms = float(np.sqrt(np.mean(ref * ref))) or 1.0
    out = {"excess": float(np.max(np.abs(got - ref) - quantum(ref, io))) / rms,
           "plain": float(np.max(np.abs(got - ref))) / rms}
    if io == "bf16":
        rne = I.round_to_bf16(ref).astype(np.float64)
        d = np.abs(got - rne)
        out["rne"] = float(np.max(d)) / rms
        big = np.abs(rne) >= rms / 16  # ulps are meaningful where |o| is not tiny against rms
        if np.any(big):
            out["rne_ulps"] = float(np.max(d[big] / bf16_ulp(rne[big])))
    return out


def check_o(got, ref, io, what="o"):
    rms = float(np.sqrt(np.mean(ref * ref)))
    excess = np.abs(got - ref) - quantum(ref, io)
    worst = float(np.max(excess)) if excess.size else 0.0
    if excess.size:
        REPORT.append(yardsticks(got, ref, io))
    assert np.all(np.isfinite(got)), "%s: non-finite values" % what
    assert worst <= O_TOL * rms, "%s: max excess error %.3e > %.3e (rms %.3e)" % (
        what, worst, O_TOL * rms, rms)
    return worst / rms if rms > 0 else 0.0


def check_S(got, ref, what="S_T"):
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.max(np.abs(got - ref)))
    assert np.all(np.isfinite(got)), "%s: non-finite values" % what
    assert err <= S_TOL * rms, "%s: max error %.3e > %.3e (rms %.3e)" % (what, err, S_TOL * rms, rms)
    return err / rms if rms > 0 else 0.0


def upload_prefill(p):
    """Device copies of a Problem's inputs."""
    t = torch_io(p.io)
    a = p.arrays
    return dict(qkv_pre=dev(a["qkv_pre"], t), z=dev(a["z"], t), g=dev(a["g"]),
                beta=dev(a["beta"]), conv_w=dev(a["conv_w"], t), norm_w=dev(a["norm_w"], t),
                S0=dev(a["S0"]), conv0=dev(a["conv0"], t))


def prefill_workspace(B, T, Hk, Hv, packed=False, form="split"):
    """A device workspace (256-byte aligned) sized for one form of the chunked
    prefill: "split" (the chunk-parallel form, gdn_prefill_workspace_bytes)
    or "staged" (q^ / k^ staged only, gdn_prefill_staged_bytes)."""
    size = gdn.gdn_prefill_staged_bytes if form == "staged" else gdn.gdn_prefill_workspace_bytes
    n = size(B, T, Hk, Hv, packed=packed)
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def gpu_prefill(p, inputs=None, in_place=False, staged=False, split=False):
    """The GPU prefill; staged: through gdn_prefill_ex with a workspace that
    holds the staged q^ / k^ only (two kernels); split: with a workspace for
    the chunk-parallel form (three kernels)."""
    x = inputs or upload_prefill(p)
    o, S_T, conv_T = gdn.alloc_prefill_outputs(p.B, p.T, p.Hk, p.Hv, torch_io(p.io))
    if in_place:
        assert x["S0"] is not None
        S_T = x["S0"]
    if staged or split:
        ws = prefill_workspace(p.B, p.T, p.Hk, p.Hv, form="staged" if staged else "split")
        gdn.gdn_prefill_ex(x["qkv_pre"], x["z"], x["g"], x["beta"], x["conv_w"], x["norm_w"],
                           x["S0"], x["conv0"], o, S_T, conv_T, Hk=p.Hk, Hv=p.Hv, workspace=ws)
    else:
        gdn.gdn_prefill(x["qkv_pre"], x["z"], x["g"], x["beta"], x["conv_w"], x["norm_w"],
                        x["S0"], x["conv0"], o, S_T, conv_T, Hk=p.Hk, Hv=p.Hv)
    torch.cuda.synchronize()
    st = gdn.gdn_device_status()
    assert st == 0, "device status %s" % gdn.STATUS_NAMES.get(st, st)
    return o, S_T, conv_T


def oracle_prefill(p, units=None, threads=0):
    a = p.arrays
    return O.gdn_prefill(a["qkv_pre"], a["z"], a["g"], a["beta"], a["conv_w"], a["norm_w"],
                         a["S0"], a["conv0"], Hk=p.Hk, Hv=p.Hv, units=units,
                         threads=threads or O.default_threads())


def compare_prefill(p, got, units=None):
    """Compare GPU outputs with the oracle on all units or on a sample."""
    o, S_T, conv_T = got
    ref = oracle_prefill(p, units)
    np.testing.assert_array_equal(to_np(conv_T), ref["conv_T"])
    if units is None:
        eo = check_o(to_np(o), ref["o"], p.io)
        es = check_S(to_np(S_T), ref["S_T"])
    else:
        D = 128
        o4 = o.view(p.B, p.T, p.Hv, D)
        got_o = np.stack([to_np(o4[u // p.Hv, :, u % p.Hv]) for u in units])
        got_S = np.stack([to_np(S_T[u // p.Hv, u % p.Hv]) for u in units])
        eo = check_o(got_o, ref["o_units"], p.io)
        es = check_S(got_S, ref["S_T"])
    return eo, es
