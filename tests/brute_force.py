"""Independent brute-force SSD forms used to pin the oracle (tests only).

Nothing here is shared with the oracle: it is the *quadratic* (attention-like)
form of the scan, materialised in full for one request and one head, written
straight from the state-space-duality reading of the recurrence:

  a_t   = softplus(dt_t + dt_bias) * A
  cs_t  = a_1 + ... + a_t                       (inclusive, from the request start)
  L     = lower-triangular, L[t,s] = exp(cs_t - cs_s) for s <= t, 0 above
  y     = (L o (C B^T)) (dt' * x)  +  exp(cs_t) * C_t . h0  +  D x,  then * silu(z)
  h_end = exp(cs_T) h0 + sum_s exp(cs_T - cs_s) dt'_s x_s (outer) B_s
"""
import numpy as np


def softplus(v):
    v = np.asarray(v, dtype=np.float64)
    return np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))


def quadratic_one(x, dt, dt_bias, A, B, C, D=None, z=None, h0=None):
    """x (L,P), dt (L,), B/C (L,N), h0 (P,N) -> y (L,P), h_end (P,N)."""
    L, P = x.shape
    N = B.shape[1]
    dtp = softplus(dt + dt_bias)
    a = dtp * A
    cs = np.cumsum(a)
    seg = cs[:, None] - cs[None, :]
    mask = np.tril(np.ones((L, L), dtype=bool))
    Lmat = np.where(mask, np.exp(np.where(mask, seg, 0.0)), 0.0)
    M = Lmat * (C @ B.T)
    y = M @ (dtp[:, None] * x)
    if h0 is None:
        h0 = np.zeros((P, N))
    y = y + np.exp(cs)[:, None] * (C @ h0.T)
    if D is not None:
        y = y + D * x
    if z is not None:
        y = y * (z / (1.0 + np.exp(-z)))
    w = np.exp(cs[-1] - cs) * dtp if L > 0 else np.zeros(0)
    h_end = (np.exp(cs[-1]) if L > 0 else 1.0) * h0 + (w[:, None] * x).T @ B
    return y, h_end
