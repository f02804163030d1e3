"""Pins of ``oracle.rotation.calibrate`` against facts fixed outside it.

The MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同做法":
the key rotation comes from the query covariance C_Q and the value rotation from
the score-weighted value covariance C_S; section "服务系统：混合精度缓存布局" and the
visual guide's step-4 table: the clip thresholds are percentiles of the rotated
channels, c_K = 0.96 for keys and c_V = 0.92 for values.

Each check is computed here without the oracle's helpers (explicit sums,
torch's float64 attention, butterflies for the Hadamard transform, sorting for
the quantile), and each has a negative control showing that a plausible mistake
(the covariances swapped, the two quantiles swapped, thresholds taken on the
unrotated tokens) would fail it.
"""
import inspect
import json
import pathlib

import numpy as np
import pytest

import synth
from oracle import rotation

D = 128
GOLD = json.loads((pathlib.Path(__file__).parent / "golden" / "oscar_pages.json").read_text())
C_K = GOLD["clip_quantile_K"]["value"]
C_V = GOLD["clip_quantile_V"]["value"]


def _cq_explicit(q):
    acc = np.zeros((D, D))
    for qn in np.asarray(q, np.float64):
        acc += np.outer(qn, qn)
    return acc / len(q)


def _cs_sdpa(q, k, v, sm):
    torch = pytest.importorskip("torch")
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=sm)[0, 0].numpy()
    return o.T @ o / len(q)


def _rotate_butterflies(x, u):
    """x U, then an unnormalised in-place Walsh-Hadamard butterfly network, / sqrt(d), then the
    output position j takes element bitrev(j) (the bit reversal written with string reversal)."""
    z = np.asarray(x, np.float64) @ np.asarray(u, np.float64)
    w = z.copy()
    s = 1
    while s < D:
        blk = w.reshape(w.shape[0], D // (2 * s), 2, s)
        a, b = blk[:, :, 0, :].copy(), blk[:, :, 1, :].copy()
        blk[:, :, 0, :], blk[:, :, 1, :] = a + b, a - b
        s *= 2
    w /= np.sqrt(D)
    nb = D.bit_length() - 1
    perm = [int(format(j, f"0{nb}b")[::-1], 2) for j in range(D)]
    return w[:, perm]


def _quantile_sorted(col, c):
    a = np.sort(np.abs(col))
    pos = (len(a) - 1) * c
    lo = int(np.floor(pos))
    hi = min(lo + 1, len(a) - 1)
    return a[lo] + (pos - lo) * (a[hi] - a[lo])


def _offdiag(m):
    return np.abs(m - np.diag(np.diag(m))).max()


def test_calibrate_defaults_are_the_pages_clip_quantiles():
    p = inspect.signature(rotation.calibrate).parameters
    assert p["c_k"].default == C_K == 0.96
    assert p["c_v"].default == C_V == 0.92


@pytest.fixture(scope="module")
def cal_case():
    qc, kc, vc = synth.calibration(11, 3, 1)
    sm = synth.sm_scale()
    return qc, kc, vc, sm, rotation.calibrate(qc, kc, vc, sm)


def test_key_rotation_diagonalises_the_query_covariance(cal_case):
    qc, kc, vc, sm, cal = cal_case
    cq = _cq_explicit(qc)
    cs = _cs_sdpa(qc, kc, vc, sm)
    u = cal["U_K"]
    m = u.T @ cq @ u
    ev = np.sort(np.linalg.eigvalsh(cq))[::-1]
    assert _offdiag(m) <= 1e-11 * ev[0]
    assert np.abs(np.diag(m) - ev).max() <= 1e-11 * ev[0]
    # negative control: U_K is not an eigenbasis of C_S, so taking U_K from C_S would fail above
    assert _offdiag(u.T @ cs @ u) > 1e-3 * np.abs(cs).max()


def test_value_rotation_diagonalises_the_score_weighted_value_covariance(cal_case):
    qc, kc, vc, sm, cal = cal_case
    cq = _cq_explicit(qc)
    cs = _cs_sdpa(qc, kc, vc, sm)
    u = cal["U_V"]
    m = u.T @ cs @ u
    ev = np.sort(np.linalg.eigvalsh(cs))[::-1]
    assert _offdiag(m) <= 1e-10 * ev[0]
    assert np.abs(np.diag(m) - ev).max() <= 1e-10 * ev[0]
    assert _offdiag(u.T @ cq @ u) > 1e-3 * np.abs(cq).max()


def test_composite_rotations_are_u_hadamard_bitreversal(cal_case):
    qc, kc, vc, sm, cal = cal_case
    x = np.eye(D)
    assert np.abs(cal["R_K"] - _rotate_butterflies(x, cal["U_K"])).max() < 1e-13
    assert np.abs(cal["R_V"] - _rotate_butterflies(x, cal["U_V"])).max() < 1e-13


@pytest.mark.parametrize("kind", ["K", "V"])
def test_thresholds_are_the_pages_quantiles_of_rotated_calibration_tokens(cal_case, kind):
    qc, kc, vc, sm, cal = cal_case
    x, u, c, other = (kc, cal["U_K"], C_K, C_V) if kind == "K" else (vc, cal["U_V"], C_V, C_K)
    tau = cal["tau_" + kind]
    xr = _rotate_butterflies(x, u)
    ref = np.array([_quantile_sorted(xr[:, j], c) for j in range(D)])
    assert np.abs(tau - ref).max() <= 1e-12 * ref.max()
    # the fraction of |rotated values| at or below tau is the quantile, per channel
    frac = (np.abs(xr) <= tau[None] * (1 + 1e-15)).mean(axis=0)
    assert np.all(np.abs(frac - c) <= 1.0 / len(x))
    # negative controls: the other kind's quantile, and thresholds on the unrotated tokens
    swapped = np.array([_quantile_sorted(xr[:, j], other) for j in range(D)])
    assert np.abs(tau - swapped).max() > 1e-2 * ref.max()
    unrot = np.array([_quantile_sorted(np.asarray(x, np.float64)[:, j], c) for j in range(D)])
    assert np.abs(tau - unrot).max() > 1e-2 * ref.max()
