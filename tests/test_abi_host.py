"""libgdn host-side tests that need no GPU: the library loads, exports every
entry point declared in include/gdn.h, and rejects bad arguments on the host
before touching the device (fake, never dereferenced pointers)."""
import ctypes
import os
import re

import pytest

from gated_deltanet_mixer_gb300 import build as gdn_build
from gated_deltanet_mixer_gb300 import gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def L():
    gdn_build.build()
    return gdn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gdn_prefill", "gdn_decode_step", "gdn_status_str", "gdn_device_status",
              "gdn_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    out = os.popen("nm -D --defined-only %s" % gdn.LIB_PATH).read()
    for name in declared_functions():
        assert re.search(r"\bT %s\b" % name, out), name


def test_abi_version_and_status_strings(L):
    hdr = open(HEADER).read()
    ver = int(re.search(r"#define GDN_ABI_VERSION (\d+)", hdr).group(1))
    assert gdn.gdn_abi_version() == ver
    for code in range(8):
        assert gdn.gdn_status_str(code) != "unknown status"
    assert gdn.gdn_status_str(99) == "unknown status"


# Fake device addresses, 16-byte aligned and far apart; never dereferenced
# because every case below fails its host-side check first.
BASE = 0x7F0000000000
STEP = 1 << 36


def fake(i, offset=0):
    return BASE + i * STEP + offset


def prefill(L, shape, **over):
    args = dict(qkv=fake(0), z=fake(1), g=fake(2), beta=fake(3), conv_w=fake(4), norm_w=fake(5),
                S0=fake(6), conv0=fake(7), o=fake(8), S_T=fake(9), conv_T=fake(10))
    args.update(over)
    return L.gdn_prefill(None if shape is None else ctypes.byref(shape),
                         *[args[k] for k in ("qkv", "z", "g", "beta", "conv_w", "norm_w", "S0",
                                             "conv0", "o", "S_T", "conv_T")], None)


def decode(L, shape, **over):
    args = dict(qkv=fake(0), z=fake(1), g=fake(2), beta=fake(3), conv_w=fake(4), norm_w=fake(5),
                S=fake(6), conv_in=fake(7), conv_out=fake(8), o=fake(9))
    args.update(over)
    return L.gdn_decode_step(ctypes.byref(shape), *[args[k] for k in (
        "qkv", "z", "g", "beta", "conv_w", "norm_w", "S", "conv_in", "conv_out", "o")], None)


def shape(B=2, T=8, Hk=2, Hv=4, D=128, io=gdn.GDN_BF16, **kw):
    return gdn.make_shape(B, T, Hk, Hv, D, io, **kw)


def test_shape_errors(L):
    assert prefill(L, None) == 1
    assert prefill(L, shape(T=0)) == 1            # empty sequence is an error
    assert prefill(L, shape(B=0)) == 1
    assert prefill(L, shape(io=7)) == 1
    assert prefill(L, shape(eps_l2=-1.0)) == 1
    assert prefill(L, shape(q_scale=float("nan"))) == 1
    assert prefill(L, shape(D=64)) == 2           # only 128-wide heads on the GPU
    assert prefill(L, shape(Hk=3, Hv=4)) == 2     # Hv must be a multiple of Hk
    assert prefill(L, shape(Hv=5000, Hk=5000)) == 2
    assert decode(L, shape(T=2)) == 1             # decode is one token


def test_null_and_alignment_errors(L):
    assert prefill(L, shape(), qkv=None) == 1
    assert prefill(L, shape(), o=None) == 1
    assert prefill(L, shape(), z=fake(1, 8)) == 3
    assert prefill(L, shape(), S_T=fake(9, 4)) == 3
    assert decode(L, shape(T=1), S=None) == 1
    assert decode(L, shape(T=1), conv_out=fake(8, 2)) == 3


def test_alias_rules(L):
    # conv_T may never overlap conv0; o may never overlap an input.
    assert prefill(L, shape(), conv_T=fake(7)) == 4
    assert prefill(L, shape(), o=fake(0, 64)) == 4
    # S_T may be exactly S0 (in place) but not partly overlap it.
    assert prefill(L, shape(), S_T=fake(6, 4096)) == 4
    # decode: conv_out must differ from conv_in; S must not overlap o.
    assert decode(L, shape(T=1), conv_out=fake(7)) == 4
    assert decode(L, shape(T=1), o=fake(6, 1024)) == 4


def test_selftest_limit_checked_on_host(L):
    for us in (0, -1, 1000001):
        assert L.gdn_selftest_wait_timeout(us, None) == gdn.GDN_ERR_INVALID_ARG


def prefill_ex(L, sh, raw=None, **over):
    args = dict(qkv_pre=fake(0), z=fake(1), g=fake(2), beta=fake(3), raw_gates=None, conv_w=fake(4),
                norm_w=fake(5), S0=fake(6), conv0=fake(7), o=fake(8), S_T=fake(9), conv_T=fake(10),
                cu_seqlens=None, S_snap=None, workspace=None, workspace_bytes=0)
    args.update(over)
    if raw is not None:
        args["raw_gates"] = ctypes.addressof(raw)
    io = gdn.gdn_prefill_io(**args)
    return L.gdn_prefill_ex(ctypes.byref(sh), ctypes.byref(io), None)


def decode_ex(L, sh, raw=None, **over):
    args = dict(qkv_pre=fake(0), z=fake(1), g=fake(2), beta=fake(3), raw_gates=None, conv_w=fake(4),
                norm_w=fake(5), S=fake(6), S_snap=None, conv_in=fake(7), conv_out=fake(8), o=fake(9))
    args.update(over)
    if raw is not None:
        args["raw_gates"] = ctypes.addressof(raw)
    io = gdn.gdn_decode_io(**args)
    return L.gdn_decode_ex(ctypes.byref(sh), ctypes.byref(io), None)


def test_extended_entry_points_check_on_host(L):
    sh = shape()
    assert L.gdn_prefill_ex(ctypes.byref(sh), None, None) == 1
    assert L.gdn_decode_ex(ctypes.byref(sh), None, None) == 1
    raw = gdn.gdn_raw_gates(fake(11), fake(12), fake(13), fake(14))
    # exactly one gate source
    assert prefill_ex(L, sh, raw=raw) == 1
    assert prefill_ex(L, sh, g=None, beta=None) == 1
    assert decode_ex(L, shape(T=3), g=None, beta=None) == 1
    assert prefill_ex(L, sh, raw=gdn.gdn_raw_gates(fake(11), None, fake(13), fake(14)),
                      g=None, beta=None) == 1
    # raw gate tensors and offsets are aligned inputs; snapshots are outputs
    assert prefill_ex(L, sh, raw=gdn.gdn_raw_gates(fake(11, 2), fake(12), fake(13), fake(14)),
                      g=None, beta=None) == 3
    assert prefill_ex(L, sh, cu_seqlens=fake(11, 4)) == 3
    assert prefill_ex(L, sh, S_snap=fake(0)) == 4           # snapshots over an input
    assert prefill_ex(L, sh, S_snap=fake(9)) == 4           # snapshots over S_T
    assert prefill_ex(L, sh, o=fake(11), raw=raw, g=None, beta=None) == 4  # o over gate a
    assert decode_ex(L, shape(T=4), S_snap=fake(6, 256)) == 4  # snapshots over the state
    assert decode_ex(L, shape(T=4), conv_out=fake(7)) == 4
    assert prefill_ex(L, shape(T=1 << 29, B=4)) == 2        # token rows beyond 2^30


def test_workspace_checked_on_host(L):
    sh = shape(B=2, T=8, Hk=2, Hv=4)
    staged = L.gdn_prefill_staged_bytes(ctypes.byref(sh), 0)
    assert staged == 3 * 2 * 8 * 2 * 128 * 2
    assert L.gdn_prefill_staged_bytes(ctypes.byref(sh), 1) == 3 * 8 * 2 * 128 * 2   # packed: T rows
    item = 32768 + 16384 + 8192 + 512 + 4  # U^T, -W^T, M, vectors, flag of one (chunk slot, value head)
    need = L.gdn_prefill_workspace_bytes(ctypes.byref(sh), 0)
    assert need == staged + 2 * 1 * 4 * item                 # B * ceil(T/64) slots x Hv heads
    assert L.gdn_prefill_workspace_bytes(ctypes.byref(sh), 1) == 3 * 8 * 2 * 128 * 2 + (0 + 2 + 2) * 4 * item
    assert L.gdn_prefill_workspace_bytes(ctypes.byref(shape(io=gdn.GDN_F32)), 0) == 0  # no chunked kernel
    assert L.gdn_prefill_staged_bytes(ctypes.byref(shape(io=gdn.GDN_F32)), 0) == 0
    assert L.gdn_prefill_workspace_bytes(None, 0) == 0
    ws = fake(11)
    assert prefill_ex(L, sh, workspace=fake(11, 16), workspace_bytes=need) == 3     # not 256-byte aligned
    assert prefill_ex(L, sh, workspace=ws, workspace_bytes=staged - 1) == 1         # too small
    assert prefill_ex(L, sh, workspace=fake(0), workspace_bytes=need) == 4          # over qkv_pre
    assert prefill_ex(L, sh, workspace=fake(8), workspace_bytes=need) == 4          # over o


def test_static_entry_checked_on_host(L):
    sh = shape(B=2, T=8, Hk=2, Hv=4)
    io = gdn.gdn_prefill_io(*[fake(i) for i in range(4)], None, fake(4), fake(5), fake(6), fake(7), fake(8),
                            fake(9), fake(10), None, None, fake(11), 1 << 20)
    assert L.gdn_prefill_static(ctypes.byref(sh), ctypes.byref(io), None) == 1   # a workspace is given
    big = shape(B=1, T=1 << 20, Hk=2, Hv=4)   # 3 x 2^20 rows x 2 heads x 256 B = 1.5 GiB > the scratch
    io.workspace, io.workspace_bytes = None, 0
    assert L.gdn_prefill_static(ctypes.byref(big), ctypes.byref(io), None) == 2
    assert L.gdn_prefill_static(None, ctypes.byref(io), None) == 1


def test_linear_checked_on_host(L):
    out = (gdn.gdn_linear_out * 2)(gdn.gdn_linear_out(0, 8, fake(2), 8), gdn.gdn_linear_out(8, 16, fake(3), 8))
    assert L.gdn_linear(0, 16, 64, fake(0), 64, fake(1), 64, 2, out, None) == 1
    assert L.gdn_linear(4, 16, 64, fake(0), 32, fake(1), 64, 2, out, None) == 1   # ldx < K
    assert L.gdn_linear(4, 16, 64, fake(0), 68, fake(1), 64, 2, out, None) == 3   # row stride not 16 bytes
    assert L.gdn_linear(4, 16, 64, fake(0, 8), 64, fake(1), 64, 2, out, None) == 3
    assert L.gdn_linear(4, 12, 64, fake(0), 64, fake(1), 64, 2, out, None) == 1   # range past N
    assert L.gdn_linear(4, 16, 64, fake(0), 64, fake(1), 64, 5, out, None) == 1   # too many outputs
    bad = (gdn.gdn_linear_out * 1)(gdn.gdn_linear_out(0, 8, fake(0, 64), 8))
    assert L.gdn_linear(4, 16, 64, fake(0), 64, fake(1), 64, 1, bad, None) == 4  # output over x

