"""The chunked (WY) form of the gated delta rule, written out in numpy, fp64.

TEST INFRASTRUCTURE ONLY.  It is a second, independent statement of the same
operation as the recurrent loop in ``gdn_oracle.c``: page "How Qwen3.5 works"
(azmle112.github.io), section 9.11, in that section's own k x v orientation
and notation.  The tests pin "chunked = recurrent" with it; nothing else uses
it.

Per chunk of n <= chunk_size tokens with incoming state S (k x v):

    d_i    = prod_{r<=i} alpha_r            R_ij = d_i / d_j  (j <= i), else 0
    A      = I + tril((B K K^T) o R, -1)    B = diag(beta), D = diag(d)
    U      = A^{-1} B V                      W = A^{-1} B D K
    Delta  = U - W S
    O      = D Q S + ((Q K^T) o R) Delta
    S_out  = d_n S + K^T diag(d_n / d_j) Delta

The ratios d_i / d_j are formed as products over the tokens between j and i,
never as a division, so a reset (alpha = 0) stays exact.
"""
import numpy as np


def _ratio(alpha, i, j):
    """prod_{r=j+1}^{i} alpha_r (0-based tokens within the chunk): d_i / d_j."""
    return float(np.prod(alpha[j + 1:i + 1]))


def core_chunked(q, k, v, g, beta, S0=None, chunk_size=64):
    """q, k [T, Dk] (normalised, q scaled); v [T, Dv]; g, beta [T];
    S0 [Dv, Dk] (value-major, as everywhere else in the oracle) or None.
    Returns (o [T, Dv], S_T [Dv, Dk])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, Dk = k.shape
    Dv = v.shape[1]
    # Section 9.11 keeps the state as k x v.
    S = np.zeros((Dk, Dv)) if S0 is None else np.asarray(S0, np.float64).T.copy()
    o = np.empty((T, Dv))
    for start in range(0, T, chunk_size):
        stop = min(start + chunk_size, T)
        n = stop - start
        K, Q, V = k[start:stop], q[start:stop], v[start:stop]
        alpha = np.exp(g[start:stop])
        d = np.array([float(np.prod(alpha[:i + 1])) for i in range(n)])
        R = np.zeros((n, n))
        for i in range(n):
            for j in range(i + 1):
                R[i, j] = _ratio(alpha, i, j)
        dn_over_d = np.array([_ratio(alpha, n - 1, j) for j in range(n)])
        Bm = np.diag(beta[start:stop])
        D = np.diag(d)
        A = np.eye(n) + np.tril((Bm @ K @ K.T) * R, -1)
        U = np.linalg.solve(A, Bm @ V)
        W = np.linalg.solve(A, Bm @ D @ K)
        Delta = U - W @ S
        o[start:stop] = D @ Q @ S + ((Q @ K.T) * R) @ Delta
        S = d[-1] * S + K.T @ np.diag(dn_over_d) @ Delta
    return o, S.T.copy()
