"""ctypes front end of the fp64 C oracle (``oracle/gdn_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Arrays are numpy; inputs are passed to C as float32 (bf16 values are exact in
float32) and every result comes back as float64.  The state layout is
[..., Dv, Dk]: row = value index, key index contiguous, as in the node
gdn.core of the page "Qwen3.8-27B" (docs.theformalera.com).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


class _RawGates(ctypes.Structure):
    _fields_ = [("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p)]


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int),
                ("Hv", ctypes.c_int), ("Dk", ctypes.c_int), ("Dv", ctypes.c_int),
                ("eps_l2", ctypes.c_double), ("eps_norm", ctypes.c_double),
                ("q_scale", ctypes.c_double)]


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        # GDN_ORACLE_LIB lets the mutation tests load a deliberately broken
        # build of this same source; normally the library is built in place.
        path = os.environ.get("GDN_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        L.oracle_silu.restype = ctypes.c_double
        L.oracle_silu.argtypes = [ctypes.c_double]
        L.oracle_conv_silu_one.restype = ctypes.c_double
        L.oracle_conv_silu_one.argtypes = [dp, dp]
        L.oracle_l2norm.restype = None
        L.oracle_l2norm.argtypes = [ctypes.c_int, dp, ctypes.c_double, ctypes.c_double, dp]
        L.oracle_core_step.restype = None
        L.oracle_core_step.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp, dp,
                                       ctypes.c_double, ctypes.c_double, dp]
        L.oracle_core_recurrent.restype = None
        L.oracle_core_recurrent.argtypes = [ctypes.c_int] * 3 + [dp] * 7
        L.oracle_gated_norm.restype = None
        L.oracle_gated_norm.argtypes = [ctypes.c_int, dp, dp, dp, ctypes.c_double, dp]
        L.oracle_sigmoid.restype = ctypes.c_double
        L.oracle_sigmoid.argtypes = [ctypes.c_double]
        L.oracle_softplus.restype = ctypes.c_double
        L.oracle_softplus.argtypes = [ctypes.c_double]
        L.oracle_gates.restype = None
        L.oracle_gates.argtypes = [ctypes.c_double] * 4 + [dp, dp]
        L.oracle_gdn_prefill_ex.restype = ctypes.c_int
        L.oracle_gdn_prefill_ex.argtypes = [ctypes.POINTER(_Shape)] + [ctypes.c_void_p] * 4 + [
            ctypes.POINTER(_RawGates)] + [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p] + [
            ctypes.c_void_p] * 5 + [ctypes.c_int]
        L.oracle_gdn_prefill.restype = ctypes.c_int
        L.oracle_gdn_prefill.argtypes = [ctypes.POINTER(_Shape)] + [ctypes.c_void_p] * 8 + [
            ctypes.c_int, ctypes.c_void_p] + [ctypes.c_void_p] * 4 + [ctypes.c_int]
        _lib = L
    return _lib


def _d(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- pieces
def silu(x):
    return lib().oracle_silu(float(x))


def conv_silu_one(window4, taps4):
    w, wp = _d(window4)
    t, tp = _d(taps4)
    return lib().oracle_conv_silu_one(wp, tp)


def l2norm(x, eps=1e-6, scale=1.0):
    x, xp = _d(x)
    y = np.empty_like(x)
    lib().oracle_l2norm(x.size, xp, eps, scale, y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return y


def sigmoid(x):
    return lib().oracle_sigmoid(float(x))


def softplus(x):
    return lib().oracle_softplus(float(x))


def gates(a, b, A_log, dt_bias):
    """Write gate and log decay of one token on one head (section 9.5 of
    "How Qwen3.5 works"): returns (g, beta) as floats."""
    g = ctypes.c_double()
    beta = ctypes.c_double()
    lib().oracle_gates(float(a), float(b), float(A_log), float(dt_bias), ctypes.byref(g),
                       ctypes.byref(beta))
    return g.value, beta.value


def gated_norm(x, z, w, eps=1e-6):
    x, xp = _d(x)
    z, zp = _d(z)
    w, wp = _d(w)
    y = np.empty_like(x)
    lib().oracle_gated_norm(x.size, xp, zp, wp, eps, y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return y


def core_recurrent(q, k, v, g, beta, S0=None):
    """The gated delta rule on one head.

    q, k: [T, Dk] (already normalised and scaled); v: [T, Dv]; g, beta: [T];
    S0: [Dv, Dk] or None (zeros).  Returns (o [T, Dv], S_T [Dv, Dk]).
    """
    q, qp = _d(q)
    k, kp = _d(k)
    v, vp = _d(v)
    g, gp = _d(np.atleast_1d(g))
    beta, bp = _d(np.atleast_1d(beta))
    T, Dk = k.shape
    Dv = v.shape[1]
    S = np.zeros((Dv, Dk)) if S0 is None else np.array(S0, dtype=np.float64, copy=True)
    S, Sp = _d(S)
    o = np.empty((T, Dv))
    lib().oracle_core_recurrent(T, Dk, Dv, qp, kp, vp, gp, bp, Sp,
                                o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return o, S


# ------------------------------------------------------------ full mixer
def conv_channels(Hk, Hv, Dk=128, Dv=128):
    return 2 * Hk * Dk + Hv * Dv


def gdn_prefill(qkv_pre, z, g, beta, conv_w, norm_w, S0=None, conv0=None, *, Hk, Hv,
                Dk=128, Dv=128, eps_l2=1e-6, eps_norm=1e-6, q_scale=None, units=None,
                threads=0, want_core=False, want_conv=True, raw_gates=None, want_snap=False):
    """The full mixer on the CPU in fp64.

    qkv_pre [B,T,C], z [B,T,Hv*Dv], g and beta [B,T,Hv], conv_w [C,4],
    norm_w [Dv], S0 [B,Hv,Dv,Dk] or None, conv0 [B,3,C] or None.
    With ``raw_gates`` = dict(a, b [B,T,Hv], A_log, dt_bias [Hv]), g and beta
    must be None and come from the raw projections (section 9.5).

    ``units`` (optional) lists b*Hv + h pairs to compute; the default is all.
    Returns a dict with ``o`` [B,T,Hv*Dv] (all units) or, when ``units`` is
    given, ``o_units`` [n,T,Dv]; ``S_T`` ([B,Hv,Dv,Dk] or [n,Dv,Dk]);
    ``conv_T`` [B,3,C]; ``core`` (pre-norm output) and ``S_snap`` (the state
    after every token, [B,T,Hv,Dv,Dk] or [n,T,Dv,Dk]) when asked.
    """
    qkv_pre = np.asarray(qkv_pre)
    B, T, C = qkv_pre.shape
    if C != conv_channels(Hk, Hv, Dk, Dv):
        raise ValueError("qkv_pre channel count %d does not match Hk/Hv/Dk/Dv" % C)
    sh = _Shape(B, T, Hk, Hv, Dk, Dv, eps_l2, eps_norm,
                (1.0 / np.sqrt(Dk)) if q_scale is None else q_scale)
    if (raw_gates is None) == (g is None or beta is None):
        raise ValueError("give either g and beta or raw_gates")
    arrs = [_f(qkv_pre), _f(z), _f(g), _f(beta), _f(conv_w), _f(norm_w), _f(S0), _f(conv0)]
    raw = None
    if raw_gates is not None:
        keep = [_f(raw_gates[k]) for k in ("a", "b", "A_log", "dt_bias")]
        raw = _RawGates(*[k[1] for k in keep])
    if units is None:
        n = B * Hv
        up = None
        uarr = None
    else:
        uarr = np.ascontiguousarray(units, dtype=np.int32)
        n = uarr.size
        up = uarr.ctypes.data_as(ctypes.c_void_p)
    y = np.empty((n, T, Dv))
    core = np.empty((n, T, Dv)) if want_core else None
    S_T = np.empty((n, Dv, Dk))
    conv_T = np.empty((B, 3, C)) if want_conv else None
    snap = np.empty((n, T, Dv, Dk)) if want_snap else None

    def ptr(x):
        return None if x is None else x.ctypes.data_as(ctypes.c_void_p)

    ins = [a[1] for a in arrs]
    rc = lib().oracle_gdn_prefill_ex(
        ctypes.byref(sh), *ins[:4], None if raw is None else ctypes.byref(raw), *ins[4:], n, up,
        ptr(y), ptr(core), ptr(S_T), ptr(snap), ptr(conv_T), int(threads))
    if rc != 0:
        raise ValueError("oracle_gdn_prefill rejected the problem (rc=%d)" % rc)
    out = {"conv_T": conv_T}
    if units is None:
        out["o"] = y.reshape(B, Hv, T, Dv).transpose(0, 2, 1, 3).reshape(B, T, Hv * Dv)
        out["S_T"] = S_T.reshape(B, Hv, Dv, Dk)
        if want_core:
            out["core"] = core.reshape(B, Hv, T, Dv).transpose(0, 2, 1, 3).reshape(B, T, Hv * Dv)
        if want_snap:
            out["S_snap"] = snap.reshape(B, Hv, T, Dv, Dk).transpose(0, 2, 1, 3, 4)
    else:
        out["o_units"] = y
        out["S_T"] = S_T
        if want_core:
            out["core_units"] = core
        if want_snap:
            out["S_snap"] = snap
    return out


def gdn_decode_step(qkv_pre, z, g, beta, conv_w, norm_w, S, conv_in, **kw):
    """One decode token for B sequences: the prefill above with T = 1.

    qkv_pre [B,C], z [B,Hv*Dv], g and beta [B,Hv], S [B,Hv,Dv,Dk],
    conv_in [B,3,C].  Returns dict(o [B,Hv*Dv], S [B,Hv,Dv,Dk], conv_out).
    """
    qkv_pre = np.asarray(qkv_pre)
    r = gdn_prefill(qkv_pre[:, None], np.asarray(z)[:, None], np.asarray(g)[:, None],
                    np.asarray(beta)[:, None], conv_w, norm_w, S, conv_in, **kw)
    return {"o": r["o"][:, 0], "S": r["S_T"], "conv_out": r["conv_T"]}


def gdn_decode_multi(qkv_pre, z, g, beta, conv_w, norm_w, S, conv_in, **kw):
    """T consecutive decode tokens for B sequences (speculative verification:
    "How Qwen3.5 works" section 13), with the state after every token kept
    for rollback.  qkv_pre [B,T,C], z [B,T,Hv*Dv], g and beta [B,T,Hv] (or
    raw_gates=...), S [B,Hv,Dv,Dk], conv_in [B,3,C].  The T tokens of a
    sequence are a prefill of T tokens from the cached state; returns
    dict(o [B,T,Hv*Dv], S [B,Hv,Dv,Dk], S_snap [B,T,Hv,Dv,Dk], conv_out)."""
    r = gdn_prefill(qkv_pre, z, g, beta, conv_w, norm_w, S, conv_in, want_snap=True, **kw)
    return {"o": r["o"], "S": r["S_T"], "S_snap": r["S_snap"], "conv_out": r["conv_T"]}


def gdn_prefill_varlen(qkv_pre, z, g, beta, conv_w, norm_w, cu_seqlens, S0=None, conv0=None, *,
                       Hk, Hv, raw_gates=None, **kw):
    """Packed variable-length prefill: sequence s owns the tokens
    cu_seqlens[s] .. cu_seqlens[s+1]-1 of qkv_pre [N,C], z [N,Hv*Dv], g and
    beta [N,Hv] (or raw_gates with a, b [N,Hv]); each starts from its own
    S0[s] / conv0[s] (zeros when None), and nothing flows between sequences.
    By definition that is one independent prefill per sequence, which is
    what this does.  Returns dict(o [N,Hv*Dv], S_T [nseq,Hv,Dv,Dk],
    conv_T [nseq,3,C])."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    nseq = cu.size - 1
    N, C = np.asarray(qkv_pre).shape
    if cu[0] != 0 or cu[-1] != N or np.any(np.diff(cu) < 1):
        raise ValueError("cu_seqlens must run from 0 to the token count in steps of >= 1")
    Dv = kw.get("Dv", 128)
    Dk = kw.get("Dk", 128)
    o = np.empty((N, Hv * Dv))
    S_T = np.empty((nseq, Hv, Dv, Dk))
    conv_T = np.empty((nseq, 3, C))
    for s in range(nseq):
        lo, hi = int(cu[s]), int(cu[s + 1])
        sl = slice(lo, hi)
        rg = None
        if raw_gates is not None:
            rg = dict(a=np.asarray(raw_gates["a"])[None, sl], b=np.asarray(raw_gates["b"])[None, sl],
                      A_log=raw_gates["A_log"], dt_bias=raw_gates["dt_bias"])
        r = gdn_prefill(np.asarray(qkv_pre)[None, sl], np.asarray(z)[None, sl],
                        None if g is None else np.asarray(g)[None, sl],
                        None if beta is None else np.asarray(beta)[None, sl], conv_w, norm_w,
                        None if S0 is None else np.asarray(S0)[s:s + 1],
                        None if conv0 is None else np.asarray(conv0)[s:s + 1],
                        Hk=Hk, Hv=Hv, raw_gates=rg, **kw)
        o[sl] = r["o"][0]
        S_T[s] = r["S_T"][0]
        conv_T[s] = r["conv_T"][0]
    return {"o": o, "S_T": S_T, "conv_T": conv_T}


def linear(x, w):
    """The projections gdn.in_proj and gdn.out_proj of the page "Qwen3.8-27B"
    (node table): y[t, n] = sum_k x[t, k] w[n, k], here in fp64 on the values
    given (the weight in nn.Linear layout [N, K]).  numpy's matmul is the one
    library step."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


# Columns of the in_proj output [T, 16480] at the 27B shape, in order:
# qkv_pre (the 10240 conv channels), z (48 x 128), b (48), a (48).
def in_proj_split(Hk=16, Hv=48, D=128):
    C = conv_channels(Hk, Hv, D, D)
    edges = np.cumsum([0, C, Hv * D, Hv, Hv])
    return {name: (int(lo), int(hi)) for name, lo, hi in zip(("qkv_pre", "z", "b", "a"), edges[:-1], edges[1:])}


def default_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
