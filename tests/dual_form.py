"""Brute-force O(T^2) "dual" (attention-like) form of the SSD scan, in NumPy.

A pin for the oracle, written independently of it: instead of walking the
recurrence token by token, it forms the full lower-triangular matrix of decayed
scores that the chunked kernels evaluate block by block ("bmm" + "chunk
scan", vLLM PR #61501 "Details"):

  y_t[p] = sum_{s<=t} (C_t . B_s) exp(A sum_{r=s+1..t} dt'_r) dt'_s x_s[p]
           + exp(A sum_{r<=t} dt'_r) sum_n C_t[n] h0[p,n] + D x_t[p]
  h_T[p,n] = exp(A sum_r dt'_r) h0[p,n]
           + sum_s exp(A sum_{r=s+1..T-1} dt'_r) dt'_s x_s[p] B_s[n]

softplus is NumPy's ``logaddexp(0, z)``.  Only for tiny inputs.
"""
import numpy as np


def dual_form_head(x, dt, A, B, C, D=0.0, h0=None, dt_bias=0.0, softplus=True):
    """One sequence, one head.  x [L,P], dt [L], B/C [L,N]; returns (y [L,P], h [P,N])."""
    x = np.asarray(x, np.float64)
    L, P = x.shape
    N = B.shape[1]
    z = np.asarray(dt, np.float64) + dt_bias
    d = np.logaddexp(0.0, z) if softplus else z
    seg = np.cumsum(d)                                   # sum_{r<=t} dt'_r
    diff = seg[:, None] - seg[None, :]                   # sum_{r=s+1..t} dt'_r
    tri = np.tril(np.ones((L, L), dtype=bool))
    decay = np.where(tri, np.exp(A * np.where(tri, diff, 0.0)), 0.0)
    scores = (C @ B.T) * decay * d[None, :]
    y = scores @ x + D * x
    h = (x * (np.exp(A * (seg[-1] - seg)) * d)[:, None]).T @ B if L else np.zeros((P, N))
    if h0 is not None:
        y = y + np.exp(A * seg)[:, None] * (C @ h0.T)
        h = h + np.exp(A * seg[-1] if L else 0.0) * h0
    return y, h
