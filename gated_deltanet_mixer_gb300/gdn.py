"""ctypes binding of libgdn (``include/gdn.h``): argument marshalling only.

Each function has the name of its C entry point and takes torch CUDA tensors
(device memory from PyTorch); all computation happens in libgdn's kernels.
There is no fallback: if ``libgdn.so`` is missing, loading it raises.
"""
import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# GDN_CHECKS=1: the bounds-checked build (python -m gated_deltanet_mixer_gb300.build --checks)
LIB_PATH = os.path.join(_HERE, "libgdn_checks.so" if os.environ.get("GDN_CHECKS", "0") not in ("", "0")
                        else "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_TIMEOUT = 6
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED_SHAPE",
                3: "GDN_ERR_ALIGNMENT", 4: "GDN_ERR_ALIAS", 5: "GDN_ERR_CUDA",
                6: "GDN_ERR_TIMEOUT", 7: "GDN_ERR_NO_DEVICE", 8: "GDN_ERR_BOUNDS"}
GDN_F32, GDN_BF16 = 0, 1
GDN_STATIC_SCRATCH_BYTES = 512 << 20  # include/gdn.h: the scratch of gdn_prefill_static


class GdnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (%s)" % (where, STATUS_NAMES.get(status, status),
                                          gdn_status_str(status)))


class gdn_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int),
                ("Hv", ctypes.c_int), ("Dk", ctypes.c_int), ("Dv", ctypes.c_int),
                ("io_dtype", ctypes.c_int), ("eps_l2", ctypes.c_float),
                ("eps_norm", ctypes.c_float), ("q_scale", ctypes.c_float)]


vp = ctypes.c_void_p


class gdn_raw_gates(ctypes.Structure):
    _fields_ = [("a", vp), ("b", vp), ("A_log", vp), ("dt_bias", vp)]


class gdn_prefill_io(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("qkv_pre", "z", "g", "beta", "raw_gates", "conv_w", "norm_w", "S0",
                                  "conv0", "o", "S_T", "conv_T", "cu_seqlens", "S_snap", "workspace")] + \
               [("workspace_bytes", ctypes.c_size_t)]


class gdn_linear_out(ctypes.Structure):
    _fields_ = [("col_begin", ctypes.c_int), ("col_end", ctypes.c_int), ("ptr", vp), ("ld", ctypes.c_longlong)]


class gdn_decode_io(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("qkv_pre", "z", "g", "beta", "raw_gates", "conv_w", "norm_w", "S",
                                  "S_snap", "conv_in", "conv_out", "o")]


_lib = None


def lib():
    """The loaded libgdn (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libgdn.so is not built (%s); run "
                               "`python -m gated_deltanet_mixer_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp = ctypes.c_void_p
        L.gdn_abi_version.restype = ctypes.c_int
        L.gdn_abi_version.argtypes = []
        L.gdn_status_str.restype = ctypes.c_char_p
        L.gdn_status_str.argtypes = [ctypes.c_int]
        L.gdn_prefill.restype = ctypes.c_int
        L.gdn_prefill.argtypes = [ctypes.POINTER(gdn_shape)] + [vp] * 12
        L.gdn_decode_step.restype = ctypes.c_int
        L.gdn_decode_step.argtypes = [ctypes.POINTER(gdn_shape)] + [vp] * 11
        L.gdn_device_status.restype = ctypes.c_int
        L.gdn_device_status.argtypes = [vp, ctypes.c_int]
        L.gdn_prefill_ex.restype = ctypes.c_int
        L.gdn_prefill_ex.argtypes = [ctypes.POINTER(gdn_shape), ctypes.POINTER(gdn_prefill_io), vp]
        L.gdn_decode_ex.restype = ctypes.c_int
        L.gdn_decode_ex.argtypes = [ctypes.POINTER(gdn_shape), ctypes.POINTER(gdn_decode_io), vp]
        L.gdn_linear.restype = ctypes.c_int
        L.gdn_linear.argtypes = [ctypes.c_int] * 3 + [vp, ctypes.c_longlong, vp, ctypes.c_longlong, ctypes.c_int,
                                                      ctypes.POINTER(gdn_linear_out), vp]
        L.gdn_selftest_wait_timeout.restype = ctypes.c_int
        L.gdn_selftest_wait_timeout.argtypes = [ctypes.c_int, vp]
        L.gdn_prefill_static.restype = ctypes.c_int
        L.gdn_prefill_static.argtypes = [ctypes.POINTER(gdn_shape), ctypes.POINTER(gdn_prefill_io), vp]
        L.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
        L.gdn_prefill_workspace_bytes.argtypes = [ctypes.POINTER(gdn_shape), ctypes.c_int]
        L.gdn_prefill_staged_bytes.restype = ctypes.c_size_t
        L.gdn_prefill_staged_bytes.argtypes = [ctypes.POINTER(gdn_shape), ctypes.c_int]
        _lib = L
    return _lib


def gdn_abi_version():
    return lib().gdn_abi_version()


def gdn_status_str(status):
    return lib().gdn_status_str(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _io_code(dtype):
    if dtype == torch.bfloat16:
        return GDN_BF16
    if dtype == torch.float32:
        return GDN_F32
    raise TypeError("io tensors must be bfloat16 or float32, not %s" % dtype)


def _head_width(C, Hk, Hv):
    D, rem = divmod(C, 2 * Hk + Hv)
    if rem:
        raise ValueError("channel count %d is not (2*Hk + Hv) * D" % C)
    return D


def make_shape(B, T, Hk, Hv, D, io_dtype, eps_l2=1e-6, eps_norm=1e-6, q_scale=0.0):
    return gdn_shape(B, T, Hk, Hv, D, D, io_dtype, eps_l2, eps_norm, q_scale)


def gdn_prefill(qkv_pre, z, g, beta, conv_w, norm_w, S0, conv0, o, S_T, conv_T, *, Hk, Hv,
                eps_l2=1e-6, eps_norm=1e-6, q_scale=0.0, stream=None):
    """Prefill T tokens of B sequences (layouts as in gdn.h).  S0 / conv0 may
    be None (zeros); S_T may be S0 itself.  Raises GdnError on a non-OK status."""
    B, T, C = qkv_pre.shape
    sh = make_shape(B, T, Hk, Hv, _head_width(C, Hk, Hv), _io_code(qkv_pre.dtype),
                    eps_l2, eps_norm, q_scale)
    st = lib().gdn_prefill(ctypes.byref(sh), _ptr(qkv_pre), _ptr(z), _ptr(g), _ptr(beta),
                           _ptr(conv_w), _ptr(norm_w), _ptr(S0), _ptr(conv0), _ptr(o),
                           _ptr(S_T), _ptr(conv_T), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_prefill")


def gdn_decode_step(qkv_pre, z, g, beta, conv_w, norm_w, S, conv_in, conv_out, o, *, Hk, Hv,
                    eps_l2=1e-6, eps_norm=1e-6, q_scale=0.0, stream=None):
    """One decode token for B sequences; S is updated in place, the new conv
    window goes to conv_out (distinct from conv_in)."""
    B, C = qkv_pre.shape
    sh = make_shape(B, 1, Hk, Hv, _head_width(C, Hk, Hv), _io_code(qkv_pre.dtype),
                    eps_l2, eps_norm, q_scale)
    st = lib().gdn_decode_step(ctypes.byref(sh), _ptr(qkv_pre), _ptr(z), _ptr(g), _ptr(beta),
                               _ptr(conv_w), _ptr(norm_w), _ptr(S), _ptr(conv_in),
                               _ptr(conv_out), _ptr(o), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_decode_step")


def _raw(raw_gates):
    """A gdn_raw_gates struct from dict(a, b, A_log, dt_bias) of tensors, or None."""
    if raw_gates is None:
        return None
    return gdn_raw_gates(*[_ptr(raw_gates[k]) for k in ("a", "b", "A_log", "dt_bias")])


def gdn_prefill_ex(qkv_pre, z, g, beta, conv_w, norm_w, S0, conv0, o, S_T, conv_T, *, Hk, Hv,
                   raw_gates=None, cu_seqlens=None, S_snap=None, workspace=None, eps_l2=1e-6,
                   eps_norm=1e-6, q_scale=0.0, stream=None, _entry="gdn_prefill_ex"):
    """Prefill with the options of gdn_prefill_ex: raw gate projections
    (raw_gates = dict(a, b, A_log, dt_bias), g = beta = None), packed
    sequences (qkv_pre [N, C], z and o [N, Hv*D], cu_seqlens int32 [B+1] on
    the device), per-token state snapshots S_snap [tokens, Hv, D, D], and a
    device workspace (any tensor of at least gdn_prefill_workspace_bytes()
    bytes) for the staged q^ / k^ path."""
    if cu_seqlens is not None:
        N, C = qkv_pre.shape
        B, T = cu_seqlens.numel() - 1, N
    else:
        B, T, C = qkv_pre.shape
    io_dtype = _io_code(qkv_pre.dtype)
    sh = make_shape(B, T, Hk, Hv, _head_width(C, Hk, Hv), io_dtype, eps_l2, eps_norm, q_scale)
    rg = _raw(raw_gates)
    io = gdn_prefill_io(_ptr(qkv_pre), _ptr(z), _ptr(g), _ptr(beta),
                        None if rg is None else ctypes.addressof(rg), _ptr(conv_w), _ptr(norm_w),
                        _ptr(S0), _ptr(conv0), _ptr(o), _ptr(S_T), _ptr(conv_T), _ptr(cu_seqlens),
                        _ptr(S_snap), _ptr(workspace),
                        0 if workspace is None else workspace.numel() * workspace.element_size())
    st = getattr(lib(), _entry)(ctypes.byref(sh), ctypes.byref(io), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, _entry)


def gdn_prefill_static(qkv_pre, z, g, beta, conv_w, norm_w, S0, conv0, o, S_T, conv_T, *, Hk, Hv, **kw):
    """gdn_prefill_ex in the library's own device scratch (gdn_prefill_static):
    no workspace argument, no allocation; calls that overlap in time race."""
    if kw.get("workspace") is not None:
        raise ValueError("gdn_prefill_static takes no workspace")
    gdn_prefill_ex(qkv_pre, z, g, beta, conv_w, norm_w, S0, conv0, o, S_T, conv_T, Hk=Hk, Hv=Hv,
                   _entry="gdn_prefill_static", **kw)


def gdn_prefill_workspace_bytes(B, T, Hk, Hv, packed=False, D=128, io_dtype=None):
    """Workspace bytes of the chunk-parallel prefill (gdn_prefill_workspace_bytes)."""
    sh = make_shape(B, T, Hk, Hv, D, GDN_BF16 if io_dtype is None else io_dtype)
    return lib().gdn_prefill_workspace_bytes(ctypes.byref(sh), 1 if packed else 0)


def gdn_prefill_staged_bytes(B, T, Hk, Hv, packed=False, D=128, io_dtype=None):
    """Workspace bytes of the staged q^ / k^ form alone (gdn_prefill_staged_bytes)."""
    sh = make_shape(B, T, Hk, Hv, D, GDN_BF16 if io_dtype is None else io_dtype)
    return lib().gdn_prefill_staged_bytes(ctypes.byref(sh), 1 if packed else 0)


def gdn_decode_ex(qkv_pre, z, g, beta, conv_w, norm_w, S, conv_in, conv_out, o, *, Hk, Hv,
                  raw_gates=None, S_snap=None, eps_l2=1e-6, eps_norm=1e-6, q_scale=0.0,
                  stream=None):
    """T new tokens per sequence from the cache (qkv_pre [B, T, C], z and o
    [B, T, Hv*D]); S is updated in place; S_snap [B, T, Hv, D, D] (optional)
    receives the state after every token; the window after the T tokens goes
    to conv_out."""
    B, T, C = qkv_pre.shape
    sh = make_shape(B, T, Hk, Hv, _head_width(C, Hk, Hv), _io_code(qkv_pre.dtype), eps_l2,
                    eps_norm, q_scale)
    rg = _raw(raw_gates)
    io = gdn_decode_io(_ptr(qkv_pre), _ptr(z), _ptr(g), _ptr(beta),
                       None if rg is None else ctypes.addressof(rg), _ptr(conv_w), _ptr(norm_w),
                       _ptr(S), _ptr(S_snap), _ptr(conv_in), _ptr(conv_out), _ptr(o))
    st = lib().gdn_decode_ex(ctypes.byref(sh), ctypes.byref(io), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_decode_ex")


def gdn_linear(x, w, outs, stream=None):
    """y = x w^T for bf16 x [M, K] and w [N, K] (row strides may exceed K);
    ``outs`` lists (col_begin, col_end, tensor) with tensor a bf16 [M, >=
    col_end - col_begin] view (row stride from the tensor) receiving those
    columns of y."""
    M, K = x.shape
    N, K2 = w.shape
    if K2 != K:
        raise ValueError("x and w disagree on K")
    arr = (gdn_linear_out * len(outs))(*[gdn_linear_out(int(b), int(e), _ptr(t), int(t.stride(0)))
                                         for b, e, t in outs])
    st = lib().gdn_linear(M, N, K, _ptr(x), int(x.stride(0)), _ptr(w), int(w.stride(0)), len(outs), arr,
                          _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_linear")


def gdn_device_status(stream=None, reset=False):
    """Synchronise and return the device-side status code (0 = OK)."""
    return lib().gdn_device_status(_stream(stream), int(bool(reset)))


def gdn_selftest_wait_timeout(wait_us, stream=None):
    """Enqueue the failure-detection self-test: a kernel whose bounded wait
    runs out after `wait_us` microseconds and records a timeout."""
    st = lib().gdn_selftest_wait_timeout(int(wait_us), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_selftest_wait_timeout")


# ---------------------------------------------------------------- helpers
def alloc_prefill_outputs(B, T, Hk, Hv, dtype, device="cuda", D=128):
    """Fresh (o, S_T, conv_T) buffers for a prefill call."""
    C = (2 * Hk + Hv) * D
    o = torch.empty(B, T, Hv * D, dtype=dtype, device=device)
    S_T = torch.empty(B, Hv, D, D, dtype=torch.float32, device=device)
    conv_T = torch.empty(B, 3, C, dtype=dtype, device=device)
    return o, S_T, conv_T


def default_q_scale(D=128):
    return 1.0 / math.sqrt(D)
