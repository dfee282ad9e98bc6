"""Pins of the fp64 oracle to facts outside itself (CPU only, no GPU).

Each test ties one part of the oracle to a value printed on the pages, a
closed form, an invariant, a special case that reduces to a textbook result,
or a second independent formulation (the chunked WY form).  Non-square heads
(Dk != Dv) are used where a transposed operand would otherwise go unnoticed.
"""
import math

import numpy as np
import pytest
from scipy.special import expit

from oracle import oracle as O
from oracle.chunked import core_chunked

RTOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x)


# ------------------------------------------------------------------ core ----
def test_worked_2x2_example(golden):
    """'How Qwen3.5 works' section 9.8, every printed number."""
    G = golden("worked_2x2.txt")
    k1, v1, k2, v2 = (np.array(G[n]) for n in ("k1", "v1", "k2", "v2"))
    a1, b1, a2, b2 = G["alpha1"][0], G["beta1"][0], G["alpha2"][0], G["beta2"][0]
    q = np.array(G["query"]) / math.sqrt(G["query_scale_inv_sq"][0])
    qs, ks, vs = np.stack([q, q]), np.stack([k1, k2]), np.stack([v1, v2])
    g = np.log([a1, a2])
    o, S2 = O.core_recurrent(qs, ks, vs, g, [b1, b2])
    np.testing.assert_allclose(S2.T, np.reshape(G["S2_kv"], (2, 2)), rtol=RTOL, atol=1e-15)
    half_ulp = 0.5 * 10.0 ** -int(G["o2_decimals"][0])
    np.testing.assert_allclose(o[1], G["o2"], rtol=0, atol=half_ulp)
    _, S1 = O.core_recurrent(qs[:1], ks[:1], vs[:1], g[:1], [b1])
    np.testing.assert_allclose(S1.T, np.reshape(G["S1_kv"], (2, 2)), rtol=RTOL, atol=1e-15)
    # Decay alone (beta = 0) gives S-bar_2; reading it with k2 gives v-hat_2.
    vhat, Sbar = O.core_recurrent(k2[None], k2[None], v2[None], g[1:], [0.0], S0=S1)
    np.testing.assert_allclose(Sbar.T, np.reshape(G["Sbar2_kv"], (2, 2)), rtol=RTOL, atol=1e-15)
    np.testing.assert_allclose(vhat[0], G["vhat2"], rtol=RTOL, atol=1e-15)
    # The correction is written along k2: S2 - S-bar_2 = k2 delta_2^T (k x v).
    np.testing.assert_allclose((S2 - Sbar).T, np.outer(k2, G["delta2"]), rtol=RTOL, atol=1e-15)


def test_three_token_walkthrough(golden):
    """ayushdeva.com 'qwen35-architecture': [2,0] -> [5,0], slot B 3 -> 2.7."""
    G = golden("three_token_walkthrough.txt")
    ks = np.stack([G["k1"], G["k2"], G["k3"]])
    vs = np.stack([G["v1"], G["v2"], G["v3"]])
    g = np.log([G["alpha1"][0], G["alpha2"][0], G["alpha3"][0]])
    beta = [G["beta1"][0], G["beta2"][0], G["beta3"][0]]
    qA = np.array([1.0, 0.0])
    o, S3 = O.core_recurrent(np.stack([qA] * 3), ks, vs, g, beta)
    np.testing.assert_allclose(o[0], G["readA1"], rtol=RTOL, atol=1e-15)
    np.testing.assert_allclose(o[2], G["readA3"], rtol=RTOL, atol=1e-15)
    _, S2 = O.core_recurrent(np.stack([qA] * 2), ks[:2], vs[:2], g[:2], beta[:2])
    np.testing.assert_allclose(S2[:, 1], G["slotB_before"], rtol=RTOL, atol=1e-15)
    np.testing.assert_allclose(S3[:, 1], G["slotB_after"], rtol=RTOL, atol=1e-15)


@pytest.mark.parametrize("slot", [0, 2, 3])
def test_one_hot_key_rewrites_one_column(slot):
    """ayushdeva.com 'qwen35-architecture': a write at slot i turns column i
    into (1-beta) old + beta new; the decay tick scales the whole state."""
    rng = _rng(11 + slot)
    Dv, Dk = 3, 5
    S0 = rng.normal(size=(Dv, Dk))
    v = rng.normal(size=Dv)
    alpha, beta = 0.7, 0.35
    k = np.eye(Dk)[slot]
    _, S = O.core_recurrent(k[None], k[None], v[None], [math.log(alpha)], [beta], S0)
    want = alpha * S0
    want[:, slot] = (1 - beta) * alpha * S0[:, slot] + beta * v
    np.testing.assert_allclose(S, want, rtol=RTOL, atol=1e-15)


@pytest.mark.parametrize("T", [1, 2, 3])
def test_closed_form_product(T):
    """Node gdn.core of the 27B spec, unrolled by hand:
    S_t = e^g S_{t-1} (I - beta k k^T) + beta v k^T,  o_t = S_t q_t."""
    rng = _rng(100 + T)
    Dv, Dk = 2, 3
    S0 = rng.normal(size=(Dv, Dk))
    q, k, v = rng.normal(size=(T, Dk)), rng.normal(size=(T, Dk)), rng.normal(size=(T, Dv))
    g, beta = -rng.uniform(0.05, 1.0, size=T), rng.uniform(0.1, 0.9, size=T)
    o, S = O.core_recurrent(q, k, v, g, beta, S0)
    St = S0.copy()
    for t in range(T):
        St = math.exp(g[t]) * St @ (np.eye(Dk) - beta[t] * np.outer(k[t], k[t])) \
            + beta[t] * np.outer(v[t], k[t])
        np.testing.assert_allclose(o[t], St @ q[t], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(S, St, rtol=1e-11, atol=1e-14)


def test_beta0_g0_leaves_state_unchanged():
    rng = _rng(5)
    Dv, Dk, T = 4, 6, 9
    S0 = rng.normal(size=(Dv, Dk))
    q, k, v = rng.normal(size=(T, Dk)), rng.normal(size=(T, Dk)), rng.normal(size=(T, Dv))
    o, S = O.core_recurrent(q, k, v, np.zeros(T), np.zeros(T), S0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, q @ S0.T, rtol=RTOL, atol=1e-14)


def test_beta1_unit_key_stores_value_exactly():
    """'How Qwen3.5 works' section 9.7: with a unit key and beta = 1 the
    updated state returns the current value along that key."""
    rng = _rng(6)
    Dv, Dk, T = 3, 8, 7
    S = rng.normal(size=(Dv, Dk))
    for t in range(T):
        k = _unit(rng.normal(size=Dk))
        v = rng.normal(size=Dv)
        g = -rng.uniform(0, 2)
        _, S = O.core_recurrent(k[None], k[None], v[None], [g], [1.0], S)
        np.testing.assert_allclose(S @ k, v, rtol=1e-12, atol=1e-13)


def test_minus_infinity_gate_resets_state():
    rng = _rng(7)
    Dv, Dk = 3, 5
    S0 = rng.normal(size=(Dv, Dk)) * 100
    q, k, v = rng.normal(size=Dk), rng.normal(size=Dk), rng.normal(size=Dv)
    beta = 0.6
    o, S = O.core_recurrent(q[None], k[None], v[None], [-np.inf], [beta], S0)
    np.testing.assert_allclose(S, beta * np.outer(v, k), rtol=RTOL, atol=0)
    np.testing.assert_allclose(o[0], S @ q, rtol=RTOL, atol=0)


def test_orthogonal_keys_reduce_to_linear_attention():
    """alpha = beta = 1, S0 = 0, orthonormal keys: the delta rule writes each
    value untouched, so o_t = sum_{j<=t} (q_t . k_j) v_j ('How Qwen3.5 works'
    section 9.1.1; ayushdeva.com: attention with the softmax deleted)."""
    rng = _rng(8)
    T, Dk, Dv = 6, 8, 5
    Qm, _ = np.linalg.qr(rng.normal(size=(Dk, Dk)))
    k = Qm[:, :T].T
    q, v = rng.normal(size=(T, Dk)), rng.normal(size=(T, Dv))
    o, _ = O.core_recurrent(q, k, v, np.zeros(T), np.ones(T))
    want = np.stack([sum((q[t] @ k[j]) * v[j] for j in range(t + 1)) for t in range(T)])
    np.testing.assert_allclose(o, want, rtol=1e-11, atol=1e-13)


def test_delta_rule_is_a_gradient_step():
    """'How Qwen3.5 works' section 9.7: the correction is one gradient step of
    size beta on l(S) = 1/2 |S k - v|^2 at the decayed state.  The gradient is
    taken by central finite differences."""
    rng = _rng(9)
    Dv, Dk = 3, 4
    S0 = rng.normal(size=(Dv, Dk))
    k, v = rng.normal(size=Dk), rng.normal(size=Dv)
    alpha, beta = 0.8, 0.3
    _, S1 = O.core_recurrent(k[None], k[None], v[None], [math.log(alpha)], [beta], S0)
    Sbar = alpha * S0

    def loss(S):
        r = S @ k - v
        return 0.5 * float(r @ r)

    h = 1e-5
    grad = np.zeros_like(Sbar)
    for i in range(Dv):
        for j in range(Dk):
            E = np.zeros_like(Sbar)
            E[i, j] = h
            grad[i, j] = (loss(Sbar + E) - loss(Sbar - E)) / (2 * h)
    np.testing.assert_allclose(S1 - Sbar, -beta * grad, rtol=1e-7, atol=1e-9)


@pytest.mark.parametrize("chunk", [1, 2, 7, 64])
def test_chunked_form_equals_recurrence(chunk):
    """'How Qwen3.5 works' section 9.11: chunking reorganises the same
    recurrence.  T is not a multiple of the chunk; one token resets."""
    rng = _rng(20 + chunk)
    T, Dk, Dv = 150, 6, 4
    q, k, v = rng.normal(size=(T, Dk)), rng.normal(size=(T, Dk)), rng.normal(size=(T, Dv))
    k = k / np.linalg.norm(k, axis=1, keepdims=True)
    g = np.log(expit(rng.normal(3, 1, size=T)))
    g[77] = -np.inf
    beta = expit(rng.normal(size=T))
    S0 = rng.normal(size=(Dv, Dk)) * 0.1
    o_r, S_r = O.core_recurrent(q, k, v, g, beta, S0)
    o_c, S_c = core_chunked(q, k, v, g, beta, S0, chunk_size=chunk)
    np.testing.assert_allclose(o_c, o_r, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(S_c, S_r, rtol=1e-10, atol=1e-12)


def test_chunked_form_equals_recurrence_full_width():
    rng = _rng(31)
    T, D = 100, 128
    q = rng.normal(size=(T, D)) / math.sqrt(D)
    k = rng.normal(size=(T, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.normal(size=(T, D))
    g = np.log(expit(rng.normal(3, 1, size=T)))
    beta = expit(rng.normal(size=T))
    S0 = rng.normal(size=(D, D)) * 0.02
    o_r, S_r = O.core_recurrent(q, k, v, g, beta, S0)
    o_c, S_c = core_chunked(q, k, v, g, beta, S0, chunk_size=64)
    np.testing.assert_allclose(o_c, o_r, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S_c, S_r, rtol=1e-9, atol=1e-11)


# --------------------------------------------------------------- pieces ----
def test_silu_matches_library():
    for x in (-30.0, -3.5, -1e-3, 0.0, 0.7, 2.0, 25.0):
        assert O.silu(x) == pytest.approx(x * float(expit(x)), rel=1e-14, abs=1e-300)


def test_conv_taps_order_impulse():
    """Node gdn.conv of the 27B spec: y[t] = silu(sum_j w[j] x[t+j-3]), so tap
    3 multiplies the current token and tap 0 the token three back."""
    for j in range(4):
        for m in range(4):
            window = np.eye(4)[m]          # impulse at window position m
            taps = np.eye(4)[j]
            want = O.silu(1.0) if m == j else 0.0
            assert O.conv_silu_one(window, taps) == pytest.approx(want, abs=1e-15)


def test_l2norm_norm_and_direction():
    """'How Qwen3.5 works' section 9.4: x / sqrt(sum x^2 + eps), then a scale."""
    rng = _rng(12)
    for scale in (1.0, 1 / math.sqrt(128)):
        for mag in (1e-3, 1.0, 50.0):
            x = rng.normal(size=16) * mag
            y = O.l2norm(x, eps=1e-6, scale=scale)
            n = np.linalg.norm(x)
            assert np.linalg.norm(y) == pytest.approx(scale * n / math.sqrt(n * n + 1e-6), rel=1e-12)
            assert float(y @ x) / (np.linalg.norm(y) * n) == pytest.approx(1.0, rel=1e-12)


def test_gated_norm_properties():
    """Node gdn.norm of the 27B spec: y = w x / sqrt(mean x^2 + eps) silu(z)."""
    rng = _rng(13)
    n = 16
    w, z = 1 + 0.1 * rng.normal(size=n), rng.normal(size=n)
    c = 0.37
    y = O.gated_norm(np.full(n, c), z, w, eps=1e-6)
    sz = np.array([O.silu(t) for t in z])
    np.testing.assert_allclose(y, w * c / math.sqrt(c * c + 1e-6) * sz, rtol=1e-12)
    np.testing.assert_array_equal(O.gated_norm(rng.normal(size=n), np.zeros(n), w), np.zeros(n))
    x = rng.normal(size=n)
    np.testing.assert_allclose(O.gated_norm(7.5 * x, z, w, eps=0.0), O.gated_norm(x, z, w, eps=0.0),
                               rtol=1e-12)
    y = O.gated_norm(x, z, w, eps=1e-6)
    ms = float(np.mean(x * x))
    assert float(np.mean((y / (w * sz)) ** 2)) == pytest.approx(ms / (ms + 1e-6), rel=1e-12)


# ------------------------------------------------- the assembled mixer ----
def _identity_conv(C, tap=3):
    w = np.zeros((C, 4), np.float32)
    w[:, tap] = 1.0
    return w


def test_head_map_bit_exact():
    """Value head h reads key head floor(h / (Hv/Hk)) (repeat_interleave;
    the 27B spec: 'value head h reads key head h / 3').  With S0 = 0,
    beta = 1, g = 0 and a one-hot key per key head, S_T[h] has exactly one
    non-zero column, at that key head's index."""
    Hk, Hv, D = 4, 12, 8
    r = Hv // Hk
    C = O.conv_channels(Hk, Hv, D, D)
    x = np.zeros((1, 1, C), np.float32)
    for kh in range(Hk):
        x[0, 0, Hk * D + kh * D + kh] = 3.0            # k of key head kh = e_kh
    x[0, 0, 2 * Hk * D:] = 1.0                          # v: silu(1) everywhere
    x[0, 0, :Hk * D] = 0.5                              # q: irrelevant here
    one = np.ones((1, 1, Hv), np.float32)
    out = O.gdn_prefill(x, np.ones((1, 1, Hv * D), np.float32), 0 * one, one,
                        _identity_conv(C), np.ones(D, np.float32), Hk=Hk, Hv=Hv, Dk=D, Dv=D)
    S = out["S_T"][0]
    for h in range(Hv):
        col = np.abs(S[h]).sum(axis=0)
        assert int(np.argmax(col)) == h // r
        assert np.count_nonzero(col) == 1


def test_q_and_v_channel_blocks():
    """q channels come first, then k, then v ('How Qwen3.5 works' section 9.2;
    gdn.conv feeds q | k | v).  beta = 0 reads S0 with q; beta = 1 from zero
    state writes v along k."""
    rng = _rng(14)
    Hk, Hv, D = 2, 4, 8
    r = Hv // Hk
    C = O.conv_channels(Hk, Hv, D, D)
    eps = 1e-6
    s2 = O.silu(2.0)
    qn = s2 / math.sqrt(s2 * s2 + eps) / math.sqrt(D)
    # (a) q block: one-hot q at dim (kh + 1) % D per key head; state untouched.
    x = np.zeros((1, 1, C), np.float32)
    for kh in range(Hk):
        x[0, 0, kh * D + (kh + 1) % D] = 2.0
    S0 = rng.normal(size=(1, Hv, D, D)).astype(np.float32)
    zero = np.zeros((1, 1, Hv), np.float32)
    out = O.gdn_prefill(x, np.ones((1, 1, Hv * D), np.float32), zero, zero, _identity_conv(C),
                        np.ones(D, np.float32), S0=S0, Hk=Hk, Hv=Hv, Dk=D, Dv=D, want_core=True)
    core = out["core"][0, 0].reshape(Hv, D)
    for h in range(Hv):
        np.testing.assert_allclose(core[h], S0[0, h][:, (h // r + 1) % D].astype(np.float64) * qn,
                                   rtol=1e-12)
    # (b) v block: distinct values per v-head, one-hot k at dim 0.
    x = np.zeros((1, 1, C), np.float32)
    for kh in range(Hk):
        x[0, 0, Hk * D + kh * D] = 2.0
    vals = rng.normal(size=Hv * D).astype(np.float32)
    x[0, 0, 2 * Hk * D:] = vals
    one = np.ones((1, 1, Hv), np.float32)
    out = O.gdn_prefill(x, np.ones((1, 1, Hv * D), np.float32), zero, one, _identity_conv(C),
                        np.ones(D, np.float32), Hk=Hk, Hv=Hv, Dk=D, Dv=D)
    kn = s2 / math.sqrt(s2 * s2 + eps)
    for h in range(Hv):
        want = np.array([O.silu(float(t)) for t in vals[h * D:(h + 1) * D]]) * kn
        np.testing.assert_allclose(out["S_T"][0, h][:, 0], want, rtol=1e-12)


def _small_problem(seed, T=9, Hk=2, Hv=4, D=6, B=2, with_state=True):
    rng = _rng(seed)
    C = O.conv_channels(Hk, Hv, D, D)
    f = np.float32
    p = dict(qkv_pre=rng.normal(size=(B, T, C)).astype(f),
             z=rng.normal(size=(B, T, Hv * D)).astype(f),
             g=np.log(expit(rng.normal(3, 1, size=(B, T, Hv)))).astype(f),
             beta=expit(rng.normal(size=(B, T, Hv))).astype(f),
             conv_w=(0.5 * rng.normal(size=(C, 4))).astype(f),
             norm_w=(1 + 0.1 * rng.normal(size=D)).astype(f))
    p["S0"] = (0.02 * rng.normal(size=(B, Hv, D, D))).astype(f) if with_state else None
    p["conv0"] = rng.normal(size=(B, 3, C)).astype(f) if with_state else None
    return p, dict(Hk=Hk, Hv=Hv, Dk=D, Dv=D)


def test_conv_tap_order_through_the_mixer():
    """Tap 0 reads three tokens back: taps (1,0,0,0) on x equal taps
    (0,0,0,1) on x delayed by three tokens with zero left context; and with a
    carried window, tap 0 at t = 0 reads its oldest row."""
    p, sh = _small_problem(15, with_state=False)
    C = p["qkv_pre"].shape[2]
    x = p["qkv_pre"]
    delayed = np.zeros_like(x)
    delayed[:, 3:] = x[:, :-3]
    a = O.gdn_prefill(**dict(p, conv_w=_identity_conv(C, 0)), **sh)
    b = O.gdn_prefill(**dict(p, qkv_pre=delayed, conv_w=_identity_conv(C, 3)), **sh)
    np.testing.assert_allclose(a["o"], b["o"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(a["S_T"], b["S_T"], rtol=1e-13, atol=1e-15)
    # Carried window: with taps (1,0,0,0) and T = 1, the input is conv0[:, 0].
    p, sh = _small_problem(16, T=1)
    a = O.gdn_prefill(**dict(p, conv_w=_identity_conv(C, 0)), **sh)
    b = O.gdn_prefill(**dict(p, qkv_pre=p["conv0"][:, :1].copy(), conv_w=_identity_conv(C, 3)), **sh)
    np.testing.assert_allclose(a["o"], b["o"], rtol=1e-13, atol=1e-15)


def test_conv_window_carried_out():
    """The carried window is the last three raw rows of (window ++ tokens)."""
    p, sh = _small_problem(17, T=2)
    out = O.gdn_prefill(**p, **sh)
    np.testing.assert_array_equal(out["conv_T"][:, 0], p["conv0"][:, 2])
    np.testing.assert_array_equal(out["conv_T"][:, 1:], p["qkv_pre"])
    p, sh = _small_problem(18, T=5)
    out = O.gdn_prefill(**p, **sh)
    np.testing.assert_array_equal(out["conv_T"], p["qkv_pre"][:, 2:])


def test_prefill_continues_from_carried_state():
    """'How Qwen3.5 works' section 13: prefill keeps the final matrix and conv
    states, and continuing from them equals one longer prefill."""
    p, sh = _small_problem(19, T=11)
    full = O.gdn_prefill(**p, **sh)
    cut = 4
    first = O.gdn_prefill(**{k: (v[:, :cut] if k in ("qkv_pre", "z", "g", "beta") else v)
                             for k, v in p.items()}, **sh)
    rest = dict({k: (v[:, cut:] if k in ("qkv_pre", "z", "g", "beta") else v)
                 for k, v in p.items()}, S0=first["S_T"].astype(np.float32),
                conv0=first["conv_T"].astype(np.float32))
    # S_T of the first part is carried in float32 here, as a caller would.
    second = O.gdn_prefill(**rest, **sh)
    np.testing.assert_allclose(second["o"], full["o"][:, cut:], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(first["o"], full["o"][:, :cut], rtol=1e-13, atol=1e-15)


def test_prefill_equals_decode_steps():
    p, sh = _small_problem(21, T=5)
    full = O.gdn_prefill(**p, **sh)
    S, conv = p["S0"].astype(np.float64), p["conv0"]
    for t in range(5):
        d = O.gdn_decode_step(p["qkv_pre"][:, t], p["z"][:, t], p["g"][:, t], p["beta"][:, t],
                              p["conv_w"], p["norm_w"], S.astype(np.float32), conv, **sh)
        if t == 0:
            np.testing.assert_allclose(d["o"], full["o"][:, 0], rtol=1e-13, atol=1e-15)
        S, conv = d["S"], d["conv_out"].astype(np.float32)
    np.testing.assert_allclose(S, full["S_T"], rtol=1e-5, atol=1e-7)


def test_state_sizes(golden):
    """Sizes printed on the pages, from the oracle's own output shapes."""
    G = golden("state_sizes.txt")
    for key in ("qwen38_27b", "qwen35_9b"):
        row = G[key]
        fields = dict(zip(row[0::2], row[1::2]))
        Hv = int(fields["Hv"])
        p = dict(qkv_pre=np.zeros((1, 1, O.conv_channels(16, Hv)), np.float32),
                 z=np.zeros((1, 1, Hv * 128), np.float32), g=np.zeros((1, 1, Hv), np.float32),
                 beta=np.zeros((1, 1, Hv), np.float32),
                 conv_w=np.zeros((O.conv_channels(16, Hv), 4), np.float32),
                 norm_w=np.ones(128, np.float32))
        out = O.gdn_prefill(**p, Hk=16, Hv=Hv, units=[0], want_conv=False)
        per_layer = out["S_T"].size * Hv
        assert per_layer == fields["per_layer"]
        if "all_layers" in fields:
            assert per_layer * fields["layers"] == fields["all_layers"]
        if "bytes_fp32" in fields:
            assert per_layer * 4 == fields["bytes_fp32"]
    f = dict(zip(G["qwen35_08b"][0::2], G["qwen35_08b"][1::2]))
    Hk, Hv = int(f["Hk"]), int(f["Hv"])
    C = O.conv_channels(Hk, Hv)
    assert Hv * 128 * 128 == f["table_numel"] * f["tables"] / f["layers"]
    assert f["layers"] * (Hv * 128 * 128 + 3 * C) == f["all_numbers"]


def test_rejects_empty_and_bad_head_ratio():
    """'How Qwen3.5 works' section 9.10: an empty sequence is an error."""
    p, sh = _small_problem(22, T=1)
    with pytest.raises(ValueError):
        O.gdn_prefill(**{k: (v[:, :0] if k in ("qkv_pre", "z", "g", "beta") else v)
                         for k, v in p.items()}, **sh)
    p, sh = _small_problem(23, T=2, Hk=3, Hv=4)
    with pytest.raises(ValueError):
        O.gdn_prefill(**p, **sh)


# --------------------------------------------------------------- gates ----
def test_sigmoid_and_softplus():
    """Section 9.5 of "How Qwen3.5 works" uses the logistic sigmoid and
    softplus(x) = log(1 + e^x): library values, the reflection identities,
    and no overflow at large |x|."""
    assert O.sigmoid(0.0) == 0.5
    assert O.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    for x in (-30.0, -3.5, -0.25, 0.7, 4.0, 30.0):
        assert O.sigmoid(x) == pytest.approx(float(expit(x)), rel=1e-14)
        assert O.softplus(x) == pytest.approx(float(np.logaddexp(0.0, x)), rel=1e-14)
        assert O.sigmoid(x) + O.sigmoid(-x) == pytest.approx(1.0, rel=1e-15)
        assert O.softplus(x) - O.softplus(-x) == pytest.approx(x, rel=1e-13)
    assert O.softplus(800.0) == 800.0
    assert 0.0 <= O.softplus(-800.0) < 1e-300


def test_gates_closed_forms():
    """beta = sigmoid(b); g = -exp(A_log) softplus(a + dt_bias)."""
    g, beta = O.gates(0.4, 0.0, math.log(3.0), -0.4)  # a + dt_bias = 0
    assert g == pytest.approx(-3.0 * math.log(2.0), rel=1e-14)
    assert beta == 0.5
    g1, b1 = O.gates(1.0, -2.0, 0.5, 0.2)
    g2, b2 = O.gates(1.0, 3.0, 0.5, 0.2)
    assert g1 == g2 and b1 < 0.5 < b2  # b drives only the write gate
    g, _ = O.gates(40.0, 0.0, 0.0, 2.0)  # softplus(x) -> x for large x
    assert g == pytest.approx(-42.0, rel=1e-15)
    rng = _rng(40)
    for _ in range(20):
        a, b, A_log, dt = rng.normal(size=4) * (3.0, 2.0, 1.0, 2.0)
        g, beta = O.gates(a, b, A_log, dt)
        assert g <= 0.0
        assert g == pytest.approx(-math.exp(A_log) * float(np.logaddexp(0.0, a + dt)), rel=1e-13)
        assert beta == pytest.approx(float(expit(b)), rel=1e-14)


def _raw_gates(seed, B, T, Hv):
    rng = _rng(seed)
    f = np.float32
    return dict(a=rng.normal(size=(B, T, Hv)).astype(f), b=rng.normal(size=(B, T, Hv)).astype(f),
                A_log=np.log(rng.uniform(1.0, 16.0, size=Hv)).astype(f),
                dt_bias=rng.normal(-3.0, 1.0, size=Hv).astype(f))


def test_raw_gates_through_the_mixer():
    """The mixer fed the raw projections equals the mixer fed g and beta
    computed from them by library routines (per value head parameters)."""
    p, sh = _small_problem(41, T=6)
    rg = _raw_gates(42, 2, 6, sh["Hv"])
    want_g = -np.exp(rg["A_log"].astype(np.float64)) * np.logaddexp(
        0.0, rg["a"].astype(np.float64) + rg["dt_bias"].astype(np.float64))
    want_b = expit(rg["b"].astype(np.float64))
    plain = O.gdn_prefill(**dict(p, g=want_g, beta=want_b), **sh)
    raw = O.gdn_prefill(**dict(p, g=None, beta=None), raw_gates=rg, **sh)
    # the plain call carries g and beta in float32
    np.testing.assert_allclose(raw["o"], plain["o"], rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(raw["S_T"], plain["S_T"], rtol=2e-5, atol=1e-7)
    with pytest.raises(ValueError):
        O.gdn_prefill(**p, raw_gates=rg, **sh)


# ----------------------------------------------- snapshots and packing ----
def test_state_snapshots_are_prefix_states():
    """The state kept after token t equals the final state of a prefill of
    the first t + 1 tokens; the last one is S_T."""
    p, sh = _small_problem(43, T=4)
    full = O.gdn_prefill(**p, **sh, want_snap=True)
    np.testing.assert_array_equal(full["S_snap"][:, -1], full["S_T"])
    seq = ("qkv_pre", "z", "g", "beta")
    for t in range(1, 4):
        pre = O.gdn_prefill(**{k: (v[:, :t] if k in seq else v) for k, v in p.items()}, **sh)
        np.testing.assert_array_equal(full["S_snap"][:, t - 1], pre["S_T"])


def test_multi_token_decode_rollback():
    """Speculative verification: after T tokens, restoring the snapshot of
    token m and decoding token m + 1 again reproduces that token's output."""
    p, sh = _small_problem(44, T=3)
    r = O.gdn_decode_multi(p["qkv_pre"], p["z"], p["g"], p["beta"], p["conv_w"], p["norm_w"],
                           p["S0"], p["conv0"], **sh)
    np.testing.assert_array_equal(r["S_snap"][:, -1], r["S"])
    m = 0
    conv_m = np.concatenate([p["conv0"][:, 1:], p["qkv_pre"][:, :1]], axis=1)
    d = O.gdn_decode_step(p["qkv_pre"][:, 1], p["z"][:, 1], p["g"][:, 1], p["beta"][:, 1],
                          p["conv_w"], p["norm_w"], r["S_snap"][:, m], conv_m, **sh)
    np.testing.assert_allclose(d["o"], r["o"][:, 1], rtol=1e-5, atol=1e-7)


def _pack(p, keys=("qkv_pre", "z", "g", "beta")):
    return {k: (v.reshape(-1, v.shape[-1]) if k in keys else v) for k, v in p.items()}


def test_varlen_equal_lengths_equals_batched():
    """Packed sequences of equal length give the batched result exactly."""
    p, sh = _small_problem(45, T=7, B=3)
    batched = O.gdn_prefill(**p, **sh)
    q = _pack(p)
    packed = O.gdn_prefill_varlen(q["qkv_pre"], q["z"], q["g"], q["beta"], p["conv_w"],
                                  p["norm_w"], [0, 7, 14, 21], p["S0"], p["conv0"], **sh)
    np.testing.assert_array_equal(packed["o"], batched["o"].reshape(21, -1))
    np.testing.assert_array_equal(packed["S_T"], batched["S_T"])
    np.testing.assert_array_equal(packed["conv_T"], batched["conv_T"])


def test_varlen_sequences_do_not_interact():
    """Changing one packed sequence leaves the others untouched, and a
    sequence shorter than the conv window carries part of its old window."""
    p, sh = _small_problem(46, T=5, B=3)
    q = _pack(p)
    cu = [0, 5, 6, 15]
    base = O.gdn_prefill_varlen(q["qkv_pre"], q["z"], q["g"], q["beta"], p["conv_w"], p["norm_w"],
                                cu, p["S0"], p["conv0"], **sh)
    x2 = q["qkv_pre"].copy()
    x2[:5] += 1.0
    moved = O.gdn_prefill_varlen(x2, q["z"], q["g"], q["beta"], p["conv_w"], p["norm_w"], cu,
                                 p["S0"], p["conv0"], **sh)
    assert not np.allclose(moved["o"][:5], base["o"][:5])
    np.testing.assert_array_equal(moved["o"][5:], base["o"][5:])
    np.testing.assert_array_equal(moved["S_T"][1:], base["S_T"][1:])
    np.testing.assert_array_equal(base["conv_T"][1, :2], p["conv0"][1, 1:])
    np.testing.assert_array_equal(base["conv_T"][1, 2], q["qkv_pre"][5])


# ---------------------------------------------------------- projections ----
def test_linear_brute_force_and_special_cases():
    """y[t,n] = sum_k x[t,k] w[n,k]: a triple loop on a small case, the
    identity weight, and a rank-one product."""
    rng = _rng(50)
    x, w = rng.normal(size=(3, 7)), rng.normal(size=(5, 7))
    want = np.zeros((3, 5))
    for t in range(3):
        for n in range(5):
            for k in range(7):
                want[t, n] += x[t, k] * w[n, k]
    np.testing.assert_allclose(O.linear(x, w), want, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(O.linear(x, np.eye(7)), x)
    u, v = rng.normal(size=4), rng.normal(size=6)
    np.testing.assert_allclose(O.linear(u[:, None], v[:, None]), np.outer(u, v), rtol=1e-15)


def test_in_proj_split_matches_the_spec(golden):
    """The four column blocks of the 27B in_proj output fill N = 16480 and
    have the widths the spec's tensor table gives the next nodes."""
    G = golden("projection_shapes.txt")
    sp = O.in_proj_split(16, int(G["v_heads"][0]), int(G["head_dim"][0]))
    assert sp["qkv_pre"] == (0, int(G["conv_channels"][0]))
    assert sp["z"][1] - sp["z"][0] == G["v_heads"][0] * G["head_dim"][0]
    assert sp["b"][1] - sp["b"][0] == G["v_heads"][0] == sp["a"][1] - sp["a"][0]
    assert sp["a"][1] == G["in_proj"][3]
    assert G["out_proj"][1] == G["v_heads"][0] * G["head_dim"][0]
