"""Small, self-contained launches of the libgdn kernels, for profilers.

    python -m gated_deltanet_mixer_gb300.profile_cases decode --B 48 --calls 3
    python -m gated_deltanet_mixer_gb300.profile_cases prefill --B 1 --T 2048 --calls 2
    python -m gated_deltanet_mixer_gb300.profile_cases prefill --B 4 --T 2048 --calls 2 --form split
    python -m gated_deltanet_mixer_gb300.profile_cases linear --T 2048 --K 5120 --N 16480 --calls 2
    python -m gated_deltanet_mixer_gb300.profile_cases decode_multi --B 64 --T 4 --calls 2 [--snap]
    python -m gated_deltanet_mixer_gb300.profile_cases serial --B 4 --T 1024 --Hv 32 --calls 2

Inputs are the seeded synthetic ones of ``inputs.py``; each case is sized so
that its working set is larger than L2 (129 MB) but only a few GB at most.
"""
import argparse

import numpy as np
import torch

from . import gdn
from . import inputs as I


def _dev(x, dt=torch.float32):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda().to(dt)


def decode(B, Hk, Hv, calls):
    dp = I.decode_problem(B=B, Hk=Hk, Hv=Hv, steps=1, case=200)
    t = torch.bfloat16
    S = _dev(dp.S)
    conv = [_dev(dp.conv, t), _dev(dp.conv, t)]
    q, z, g, b = _dev(dp.qkv_pre[0], t), _dev(dp.z[0], t), _dev(dp.g[0]), _dev(dp.beta[0])
    cw, nw = _dev(dp.conv_w, t), _dev(dp.norm_w, t)
    o = torch.empty(B, Hv * 128, device="cuda", dtype=t)
    for s in range(calls):
        gdn.gdn_decode_step(q, z, g, b, cw, nw, S, conv[s % 2], conv[(s + 1) % 2], o, Hk=Hk, Hv=Hv)


def prefill(B, T, Hk, Hv, calls, form="fused", g_mu=3.0):
    """form: "fused" (no workspace, one kernel), "staged" (q^ / k^ through a
    workspace, two kernels) or "split" (the chunk-parallel form, three)."""
    p = I.prefill_problem(B, T, Hk, Hv, io="bf16", case=201, g_mu=g_mu)
    t = torch.bfloat16
    a = p.arrays
    x = [_dev(a["qkv_pre"], t), _dev(a["z"], t), _dev(a["g"]), _dev(a["beta"]),
         _dev(a["conv_w"], t), _dev(a["norm_w"], t), _dev(a["S0"]), _dev(a["conv0"], t)]
    o, S_T, conv_T = gdn.alloc_prefill_outputs(B, T, Hk, Hv, t)
    ws = None
    if form != "fused":
        size = gdn.gdn_prefill_staged_bytes if form == "staged" else gdn.gdn_prefill_workspace_bytes
        ws = torch.empty(size(B, T, Hk, Hv), dtype=torch.uint8, device="cuda")
    for _ in range(calls):
        if ws is not None:
            gdn.gdn_prefill_ex(*x, o, S_T, conv_T, Hk=Hk, Hv=Hv, workspace=ws)
        else:
            gdn.gdn_prefill(*x, o, S_T, conv_T, Hk=Hk, Hv=Hv)


def decode_multi(B, T, Hk, Hv, calls, snap):
    """T tokens per sequence from the cache (the T-token decode kernel)."""
    dp = I.decode_problem(B=B, Hk=Hk, Hv=Hv, steps=T, case=203)
    t = torch.bfloat16
    S = _dev(dp.S)
    q = _dev(dp.qkv_pre.transpose(1, 0, 2), t)
    z = _dev(dp.z.transpose(1, 0, 2), t)
    g, b = _dev(dp.g.transpose(1, 0, 2)), _dev(dp.beta.transpose(1, 0, 2))
    cw, nw = _dev(dp.conv_w, t), _dev(dp.norm_w, t)
    conv_in = _dev(dp.conv, t)
    conv_out = torch.empty_like(conv_in)
    o = torch.empty(B, T, Hv * 128, device="cuda", dtype=t)
    S_snap = torch.empty(B, T, Hv, 128, 128, device="cuda") if snap else None
    for _ in range(calls):
        gdn.gdn_decode_ex(q, z, g, b, cw, nw, S, conv_in, conv_out, o, Hk=Hk, Hv=Hv, S_snap=S_snap)


def serial(B, T, Hk, Hv, calls):
    """fp32 io prefill: the token-serial kernel."""
    p = I.prefill_problem(B, T, Hk, Hv, io="f32", case=204)
    a = p.arrays
    x = [_dev(a[k]) for k in ("qkv_pre", "z", "g", "beta", "conv_w", "norm_w", "S0", "conv0")]
    o, S_T, conv_T = gdn.alloc_prefill_outputs(B, T, Hk, Hv, torch.float32)
    for _ in range(calls):
        gdn.gdn_prefill(*x, o, S_T, conv_T, Hk=Hk, Hv=Hv)


def linear(T, K, N, calls):
    xa, wa = I.linear_problem(T, N, K, case=202)
    x, w = _dev(xa, torch.bfloat16), _dev(wa, torch.bfloat16)
    y = torch.empty(T, N, device="cuda", dtype=torch.bfloat16)
    for _ in range(calls):
        gdn.gdn_linear(x, w, [(0, N, y)])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["decode", "prefill", "linear", "decode_multi", "serial"])
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--Hk", type=int, default=16)
    ap.add_argument("--Hv", type=int, default=None)
    ap.add_argument("--K", type=int, default=5120)
    ap.add_argument("--N", type=int, default=16480)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--form", choices=["fused", "staged", "split"], default="fused",
                    help="prefill: no workspace, the staged q^/k^ workspace, or the chunk-parallel workspace")
    ap.add_argument("--g-mu", type=float, default=3.0, help="prefill: mean of the log-decay logits")
    ap.add_argument("--snap", action="store_true", help="decode_multi: a state snapshot after every token")
    a = ap.parse_args()
    gdn.lib()
    if a.kernel == "decode":
        decode(a.B or 48, a.Hk, a.Hv or 48, a.calls)
    elif a.kernel == "linear":
        linear(a.T, a.K, a.N, a.calls)
    elif a.kernel == "decode_multi":
        decode_multi(a.B or 64, a.T, a.Hk, a.Hv or 48, a.calls, a.snap)
    elif a.kernel == "serial":
        serial(a.B or 4, a.T, a.Hk, a.Hv or 32, a.calls)
    else:
        prefill(a.B or 4, a.T, a.Hk, a.Hv or 32, a.calls, a.form, a.g_mu)
    torch.cuda.synchronize()
    st = gdn.gdn_device_status()
    if st != 0:
        raise SystemExit("device status %d" % st)
    print("ok")


if __name__ == "__main__":
    main()
