"""Offline rotation construction (fp64).

The MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同做法":

* Key error is measured in the attention logits, and
  ||Q K^T - Q Khat^T||_F^2 = tr((K - Khat) Q^T Q (K - Khat)^T), so the key
  rotation comes from the query covariance C_Q = (1/N) sum_n q_n^T q_n.
* Value error is measured in the attention output S V, so the value rotation
  comes from the score-weighted value covariance C_S = (1/N) V^T S^T S V.
* U_Q, U_S are the eigenvectors of C_Q, C_S; H_Had is the Walsh-Hadamard
  matrix (Lemma 1: every diagonal entry of H^T Lambda H equals tr(Lambda)/d);
  P_br is the bit-reversal permutation; R_K = U_Q H_Had P_br and
  R_V = U_S H_Had P_br.

The news article "超越 TurboQuant…", section "OSCAR 的设计思路", names the same three factors (U aligns the
attention-relevant directions, Hadamard spreads outliers, bit reversal
balances the INT2 groups) and says thresholds and rotations are fixed per layer
and head.

Conventions (readings where the pages are silent):

* Row vectors: a token x (shape [d]) is rotated as x R.
* U's columns are eigenvectors sorted by descending eigenvalue; each column's
  sign is chosen so that its entry of largest magnitude is positive.
* H_Had is the Sylvester-ordered Hadamard matrix scaled to be orthonormal,
  H[i, j] = (-1)^popcount(i & j) / sqrt(d).
* (x P_br)[j] = x[bitrev(j)], bitrev over log2(d) bits.
* S is the row softmax of sm_scale * Q_cal K_cal^T over the calibration tokens,
  with no causal mask.
* Clip thresholds: tau[j] = quantile_c(|X_cal R|[:, j]) per rotated channel,
  numpy's default (linear) interpolation; c = 0.96 for K, 0.92 for V
  (the MarkTechPost article "Together AI 开源 OSCAR…", visual guide step 4 table and "服务系统" section).
"""
from __future__ import annotations

import numpy as np


def bitrev(d: int) -> np.ndarray:
    """bitrev(j) for j in [0, d), d a power of two: the log2(d)-bit reversal of j."""
    nb = int(d).bit_length() - 1
    assert 1 << nb == d, "d must be a power of two"
    out = np.zeros(d, dtype=np.int64)
    for j in range(d):
        r = 0
        for b in range(nb):
            if (j >> b) & 1:
                r |= 1 << (nb - 1 - b)
        out[j] = r
    return out


def bitrev_matrix(d: int) -> np.ndarray:
    """P_br as a matrix acting on row vectors: (x P)[j] = x[bitrev(j)], i.e. P[bitrev(j), j] = 1."""
    p = np.zeros((d, d))
    br = bitrev(d)
    for j in range(d):
        p[br[j], j] = 1.0
    return p


def hadamard(d: int) -> np.ndarray:
    """Orthonormal Sylvester Hadamard matrix, H[i, j] = (-1)^popcount(i & j) / sqrt(d)."""
    h = np.empty((d, d))
    for i in range(d):
        for j in range(d):
            h[i, j] = -1.0 if bin(i & j).count("1") % 2 else 1.0
    return h / np.sqrt(d)


def query_covariance(q: np.ndarray) -> np.ndarray:
    """C_Q = (1/N) sum_n q_n^T q_n for row-vector queries q [N, d]."""
    q = np.asarray(q, dtype=np.float64)
    return q.T @ q / q.shape[0]


def softmax_rows(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def score_weighted_value_covariance(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float) -> np.ndarray:
    """C_S = (1/N) V^T S^T S V with S = softmax(sm_scale Q K^T), N = number of queries."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = softmax_rows(sm_scale * (q @ k.T))
    sv = s @ v
    return sv.T @ sv / q.shape[0]


def eigenbasis(c: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Eigen-decomposition of a symmetric matrix: (eigenvalues descending, U with eigenvector columns).

    Each column's sign is fixed so that its largest-magnitude entry is positive.
    """
    w, u = np.linalg.eigh(np.asarray(c, dtype=np.float64))
    order = np.argsort(w)[::-1]
    w = w[order]
    u = u[:, order].copy()
    for j in range(u.shape[1]):
        i = int(np.argmax(np.abs(u[:, j])))
        if u[i, j] < 0:
            u[:, j] = -u[:, j]
    return w, u


def composite_rotation(u: np.ndarray) -> np.ndarray:
    """R = U H_Had P_br."""
    d = u.shape[0]
    return np.asarray(u, dtype=np.float64) @ hadamard(d) @ bitrev_matrix(d)


def clip_thresholds(x_rot: np.ndarray, c: float) -> np.ndarray:
    """tau[j] = c-quantile of |x_rot[:, j]| over the calibration tokens (linear interpolation)."""
    return np.quantile(np.abs(np.asarray(x_rot, dtype=np.float64)), c, axis=0)


def calibrate(q_cal, k_cal, v_cal, sm_scale: float, c_k: float = 0.96, c_v: float = 0.92) -> dict:
    """Full offline calibration for one (layer, kv-head).

    Returns fp64 arrays: U_K, U_V (eigenvector columns), eigenvalues, R_K, R_V
    and the clip thresholds tau_K, tau_V in the rotated basis.
    """
    cq = query_covariance(q_cal)
    cs = score_weighted_value_covariance(q_cal, k_cal, v_cal, sm_scale)
    wq, uq = eigenbasis(cq)
    ws, us = eigenbasis(cs)
    rk = composite_rotation(uq)
    rv = composite_rotation(us)
    tau_k = clip_thresholds(np.asarray(k_cal, np.float64) @ rk, c_k)
    tau_v = clip_thresholds(np.asarray(v_cal, np.float64) @ rv, c_v)
    return {"C_Q": cq, "C_S": cs, "eig_Q": wq, "eig_S": ws, "U_K": uq, "U_V": us,
            "R_K": rk, "R_V": rv, "tau_K": tau_k, "tau_V": tau_v}


def rotate(x: np.ndarray, u: np.ndarray) -> np.ndarray:
    """x R for R = U H_Had P_br, row vectors x [..., d], in fp64."""
    return np.asarray(x, dtype=np.float64) @ composite_rotation(u)


def logit_error_direct(q: np.ndarray, k: np.ndarray, khat: np.ndarray) -> float:
    """||Q K^T - Q Khat^T||_F^2 computed directly."""
    q = np.asarray(q, np.float64)
    diff = q @ np.asarray(k, np.float64).T - q @ np.asarray(khat, np.float64).T
    return float(np.sum(diff * diff))


def logit_error_trace(q: np.ndarray, k: np.ndarray, khat: np.ndarray) -> float:
    """tr((K - Khat) Q^T Q (K - Khat)^T), the query-covariance-weighted form."""
    q = np.asarray(q, np.float64)
    e = np.asarray(k, np.float64) - np.asarray(khat, np.float64)
    return float(np.trace(e @ (q.T @ q) @ e.T))
