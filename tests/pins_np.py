"""Independent numpy formulations that pin the oracle.

None of this shares code with ``oracle/``.  Each function states the method in
a different form from the oracle's: the conv as a library cross-correlation
over the explicit column sequence of a path, the recurrence as the literal
matrix product S_p (I - beta k k^T) of the gated delta rule, sigmoid and
softplus as scipy/numpy library routines.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

L2_EPS = 1e-6


def path_to(parents: np.ndarray, t: int) -> list:
    """Local nodes on the root-to-t path, root first."""
    out = []
    while t >= 0:
        out.append(t)
        t = int(parents[t])
    return out[::-1]


def conv_path(hist: np.ndarray, xs: np.ndarray, w: np.ndarray):
    """Conv over one path: hist [K-1][C], xs [L][C] (root first), w [C][K].

    Returns (y [L][C] pre-activation, silu(y), window of the last node).
    y[t, c] = sum_j seq[t + j, c] w[c, j] over seq = hist ++ xs, i.e. the
    'valid' cross-correlation of the column sequence with the taps.
    """
    seq = np.concatenate([hist.astype(np.float64), xs.astype(np.float64)], axis=0)
    C = seq.shape[1]
    y = np.stack([np.correlate(seq[:, c], w[c].astype(np.float64), mode="valid")
                  for c in range(C)], axis=1)
    K = w.shape[1]
    return y, y * expit(y), seq[-(K - 1):]


def l2n(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    return x / np.sqrt(np.dot(x, x) + L2_EPS)


def gates(b: float, a: float, dt_bias: float, A: float):
    beta = float(expit(np.float64(b)))
    decay = float(np.exp(np.float64(A) * np.logaddexp(0.0, np.float64(a) + np.float64(dt_bias))))
    return beta, decay


def decode_step(S: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray, beta: float,
                decay: float, q_scale: float = 1.0):
    """One token of the gated delta rule, literal matrix form:
    S_t = decay S (I - beta k k^T) + beta v k^T, o_t = S_t q."""
    d = S.shape[1]
    kn, qn = l2n(k), l2n(q)
    St = decay * S @ (np.eye(d) - beta * np.outer(kn, kn)) + beta * np.outer(v.astype(np.float64), kn)
    return St, q_scale * (St @ qn)


def head_slices(h_k: int, h_v: int, d: int, h: int):
    """(q, k, v) channel slices of value head h: q | k | v order, k-head h // (h_v // h_k)."""
    kh = h // (h_v // h_k)
    q = slice(kh * d, (kh + 1) * d)
    k = slice(h_k * d + kh * d, h_k * d + (kh + 1) * d)
    v = slice(2 * h_k * d + h * d, 2 * h_k * d + (h + 1) * d)
    return q, k, v


def decode_path(S0: np.ndarray, xc_rows: np.ndarray, ba_rows: np.ndarray, dt_bias: float,
                A: float, h_k: int, h_v: int, d: int, h: int, q_scale: float = 1.0):
    """Sequential decode of the tokens of one path for value head h.
    Returns (final state, outputs [L][d])."""
    qs, ks, vs = head_slices(h_k, h_v, d, h)
    S = S0.astype(np.float64)
    outs = []
    for row, bar in zip(xc_rows, ba_rows):
        beta, decay = gates(bar[h], bar[h_v + h], dt_bias, A)
        S, o = decode_step(S, row[qs], row[ks], row[vs], beta, decay, q_scale)
        outs.append(o)
    return S, np.array(outs)


def relerr(got: np.ndarray, ref: np.ndarray, floor_frac: float = 0.1) -> float:
    """max |got - ref| / max(|ref|, floor_frac * rms(ref)) over all elements."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), floor_frac * rms if rms > 0 else 1e-30)
    return float(np.max(np.abs(got - ref) / den))
