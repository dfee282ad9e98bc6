"""Canary guard bands around every buffer a libgdn call writes, for the GPU
tests (compute-sanitizer is not available; this is the out-of-bounds check).

While a GPU test runs, the binding's entry points are wrapped: each output
tensor (o, S_T, conv_T, S_snap, the decode state and window, the workspace,
the projection outputs) is replaced by an inner view of a buffer with
GUARD bytes of PATTERN before and after it, the call runs on those views,
and after a synchronize the guard bytes are checked and the results copied
back.  Tensors passed as two arguments (S_T == S0 in place) stay one buffer.
A damaged guard fails the test with the entry point and argument named."""
import torch

from gated_deltanet_mixer_gb300 import gdn

GUARD = 4096
PATTERN = 0xA5

# entry point -> (positional indices, keyword names) of the tensors it writes
WRITES = {
    "gdn_prefill": ((8, 9, 10), ()),
    "gdn_prefill_ex": ((8, 9, 10), ("S_snap", "workspace")),
    "gdn_prefill_static": ((8, 9, 10), ("S_snap",)),
    "gdn_decode_step": ((6, 8, 9), ()),
    "gdn_decode_ex": ((6, 8, 9), ("S_snap",)),
}
# inputs that may be the very same tensor as an output (in-place state)
MAY_ALIAS = {"gdn_prefill": (6,), "gdn_prefill_ex": (6,), "gdn_prefill_static": (6,)}

checked = {"calls": 0, "buffers": 0}


class Guarded:
    def __init__(self, t):
        self.orig = t
        self.n = t.numel() * t.element_size()
        self.raw = torch.empty(GUARD + self.n + GUARD, dtype=torch.uint8, device=t.device)
        self.raw[:GUARD].fill_(PATTERN)
        self.raw[GUARD + self.n:].fill_(PATTERN)
        self.inner = self.raw[GUARD:GUARD + self.n].view(t.dtype).view(t.shape)
        self.inner.copy_(t)

    def intact(self):
        return bool((self.raw[:GUARD] == PATTERN).all()) and bool((self.raw[GUARD + self.n:] == PATTERN).all())


def _guardable(t):
    return isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous() and t.numel() > 0


def wrap(name, fn):
    pos, kws = WRITES[name]
    alias = MAY_ALIAS.get(name, ())

    def wrapped(*args, **kw):
        args = list(args)
        by_ptr = {}
        slots = [("arg", i) for i in pos if i < len(args)] + [("kw", k) for k in kws if k in kw]

        def get(s):
            return args[s[1]] if s[0] == "arg" else kw[s[1]]

        def put(s, v):
            if s[0] == "arg":
                args[s[1]] = v
            else:
                kw[s[1]] = v

        # An output sharing memory with another argument (an aliasing error the
        # call must report, or an allowed in-place state) is not moved apart.
        others = [(a.data_ptr(), a.data_ptr() + a.numel() * a.element_size())
                  for j, a in enumerate(args) if isinstance(a, torch.Tensor) and j not in pos and j not in alias]
        others += [(a.data_ptr(), a.data_ptr() + a.numel() * a.element_size())
                   for k, a in kw.items() if isinstance(a, torch.Tensor) and k not in kws]
        outs = [get(s) for s in slots if _guardable(get(s))]
        for s in slots:
            t = get(s)
            if not _guardable(t):
                continue
            lo, hi = t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()
            if any(lo < b and a < hi for a, b in others):
                continue
            if sum(1 for u in outs if u.data_ptr() < hi and lo < u.data_ptr() + u.numel() * u.element_size()) > 1:
                continue  # two outputs overlapping each other: the call must reject it
            g = by_ptr.setdefault(lo, Guarded(t))
            put(s, g.inner)
        for i in alias:
            if i < len(args) and _guardable(args[i]) and args[i].data_ptr() in by_ptr:
                args[i] = by_ptr[args[i].data_ptr()].inner
        try:
            return fn(*args, **kw)
        finally:
            torch.cuda.synchronize()
            checked["calls"] += 1
            for g in by_ptr.values():
                checked["buffers"] += 1
                g.orig.copy_(g.inner)
                assert g.intact(), "%s wrote outside an output buffer (%d bytes, %s)" % (name, g.n, g.orig.dtype)

    wrapped.__wrapped__ = fn
    return wrapped


def wrap_linear(fn):
    def wrapped(x, w, outs, stream=None):
        gs, new = [], []
        for b, e, t in outs:
            if _guardable(t):
                g = Guarded(t)
                gs.append(g)
                new.append((b, e, g.inner))
            else:
                new.append((b, e, t))
        try:
            return fn(x, w, new, stream=stream)
        finally:
            torch.cuda.synchronize()
            checked["calls"] += 1
            for g in gs:
                checked["buffers"] += 1
                g.orig.copy_(g.inner)
                assert g.intact(), "gdn_linear wrote outside an output buffer (%d bytes)" % g.n

    wrapped.__wrapped__ = fn
    return wrapped


def install(monkeypatch):
    for name in WRITES:
        monkeypatch.setattr(gdn, name, wrap(name, getattr(gdn, name)))
    monkeypatch.setattr(gdn, "gdn_linear", wrap_linear(gdn.gdn_linear))
