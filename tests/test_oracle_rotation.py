"""Pins of the oracle's rotation construction against facts fixed outside the oracle.

Each test checks a closed form, a theorem stated on the pages, or an
independent library computation, so that a dropped term, a wrong sign or a
transposed operand in ``oracle.rotation`` fails one of them.
"""
import numpy as np
import pytest

import synth
from oracle import rotation

D = 128


def test_hadamard_small_closed_form_and_recursion():
    # Sylvester construction: H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]] (unnormalised).
    h2 = rotation.hadamard(2) * np.sqrt(2)
    assert np.array_equal(h2, np.array([[1.0, 1.0], [1.0, -1.0]]))
    for n in (2, 4, 8, 16, 32, 64):
        hn = rotation.hadamard(n) * np.sqrt(n)
        h2n = rotation.hadamard(2 * n) * np.sqrt(2 * n)
        blk = np.block([[hn, hn], [hn, -hn]])
        assert np.array_equal(np.rint(h2n), blk)


def test_hadamard_orthonormal_symmetric():
    h = rotation.hadamard(D)
    assert np.allclose(h, h.T, atol=0)
    assert np.abs(h @ h.T - np.eye(D)).max() < 1e-13
    assert np.allclose(np.abs(h), 1 / np.sqrt(D))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lemma1_hadamard_equalises_diagonal(seed):
    # The MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同做法", Lemma 1: every diagonal entry of H^T Lambda H equals tr(Lambda)/d.
    rng = np.random.default_rng(seed)
    lam = np.diag(rng.exponential(size=D) * 10.0 ** rng.uniform(-3, 3, size=D))
    h = rotation.hadamard(D)
    dg = np.diag(h.T @ lam @ h)
    assert np.abs(dg - np.trace(lam) / D).max() <= 1e-12 * np.trace(lam)


def test_lemma1_on_calibration_spectrum():
    qc, kc, vc = synth.calibration(3, 0, 0)
    cq = rotation.query_covariance(qc)
    w, u = rotation.eigenbasis(cq)
    h = rotation.hadamard(D)
    dg = np.diag(h.T @ np.diag(w) @ h)
    assert np.abs(dg - w.sum() / D).max() <= 1e-12 * w.sum()
    # and the composite rotation therefore gives every channel the same query energy
    rk = rotation.composite_rotation(u)
    energy = np.diag(rk.T @ cq @ rk)
    assert np.abs(energy - np.trace(cq) / D).max() <= 1e-10 * np.trace(cq)


def test_bitrev_small_literal():
    assert list(rotation.bitrev(8)) == [0, 4, 2, 6, 1, 5, 3, 7]
    assert list(rotation.bitrev(4)) == [0, 2, 1, 3]
    br = rotation.bitrev(D)
    assert np.array_equal(br[br], np.arange(D))          # an involution
    assert sorted(br) == list(range(D))                  # a permutation


def test_bitrev_matrix_action():
    x = np.arange(D, dtype=np.float64)
    p = rotation.bitrev_matrix(D)
    assert np.array_equal(x @ p, x[rotation.bitrev(D)])
    assert np.array_equal(p, p.T)


@pytest.mark.parametrize("gsize", [2, 4, 8, 16, 32, 64, 128])
def test_bitrev_every_group_gets_every_tier(gsize):
    # The MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同做法": after P_br each power-of-two group holds one
    # representative of every level of the importance order. Source channel i
    # (sorted by importance) is in tier i // (d / gsize); output block b holds
    # positions [b*gsize, (b+1)*gsize).
    br = rotation.bitrev(D)
    ntier = gsize
    tier_width = D // ntier
    for b in range(D // gsize):
        src = br[b * gsize:(b + 1) * gsize]
        tiers = sorted(src // tier_width)
        assert tiers == list(range(ntier))


def test_query_covariance_against_outer_product_sum():
    qc, _, _ = synth.calibration(5, 1, 2)
    acc = np.zeros((D, D))
    for qn in qc.astype(np.float64):
        acc += np.outer(qn, qn)
    assert np.abs(rotation.query_covariance(qc) - acc / len(qc)).max() < 1e-12 * np.abs(acc).max()


def test_score_weighted_value_covariance_is_second_moment_of_attention_outputs():
    torch = pytest.importorskip("torch")
    qc, kc, vc = synth.calibration(6, 0, 1)
    sm = synth.sm_scale()
    q = torch.from_numpy(qc.astype(np.float64))[None, None]
    k = torch.from_numpy(kc.astype(np.float64))[None, None]
    v = torch.from_numpy(vc.astype(np.float64))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=sm)[0, 0].numpy()
    cs_ref = o.T @ o / len(qc)
    cs = rotation.score_weighted_value_covariance(qc, kc, vc, sm)
    assert np.abs(cs - cs_ref).max() < 1e-11 * np.abs(cs_ref).max()


def test_score_weighted_value_covariance_uniform_scores_closed_form():
    # All keys equal -> S is uniform 1/N -> S V has every row equal to mean(V) -> C_S = mu^T mu.
    rng = np.random.default_rng(0)
    q = rng.standard_normal((64, 16))
    k = np.tile(rng.standard_normal(16), (64, 1))
    v = rng.standard_normal((64, 16))
    mu = v.mean(axis=0)
    cs = rotation.score_weighted_value_covariance(q, k, v, 0.3)
    assert np.abs(cs - np.outer(mu, mu)).max() < 1e-13


def test_eigenbasis_diagonalises_descending_with_sign_convention():
    qc, kc, vc = synth.calibration(7, 2, 3)
    for c in (rotation.query_covariance(qc), rotation.score_weighted_value_covariance(qc, kc, vc, synth.sm_scale())):
        w, u = rotation.eigenbasis(c)
        assert np.all(np.diff(w) <= 0)
        assert np.abs(u.T @ u - np.eye(D)).max() < 1e-12
        assert np.abs(u.T @ c @ u - np.diag(w)).max() < 1e-12 * w[0]
        for j in range(D):
            i = np.argmax(np.abs(u[:, j]))
            assert u[i, j] > 0


def test_composite_rotation_orthogonal_and_preserves_logits():
    qc, kc, vc = synth.calibration(8, 0, 0)
    cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
    for r in (cal["R_K"], cal["R_V"]):
        assert np.abs(r.T @ r - np.eye(D)).max() <= 1e-12
    # (q R)(k R)^T = q k^T without quantisation.
    q = qc.astype(np.float64)[:32]
    k = kc.astype(np.float64)[:48]
    r = cal["R_K"]
    assert np.abs((q @ r) @ (k @ r).T - q @ k.T).max() <= 1e-12 * np.abs(q @ k.T).max()
    # R = U H P_br factor by factor: (x R)[j] = FWHT(x U)[bitrev(j)] / sqrt(d)
    x = kc[0].astype(np.float64)
    z = x @ cal["U_K"]
    w = z.copy()
    s = 1
    while s < D:                      # in-place butterflies, unnormalised
        for i in range(D):
            if i & s == 0:
                a, b = w[i], w[i + s]
                w[i], w[i + s] = a + b, a - b
        s *= 2
    w /= np.sqrt(D)
    assert np.abs(x @ cal["R_K"] - w[rotation.bitrev(D)]).max() < 1e-12 * np.abs(x).max()


def test_logit_error_identity():
    # The MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同做法": ||Q K^T - Q Khat^T||_F^2 = tr((K - Khat) Q^T Q (K - Khat)^T)
    rng = np.random.default_rng(1)
    q = rng.standard_normal((40, D))
    k = rng.standard_normal((70, D))
    khat = k + 0.1 * rng.standard_normal((70, D))
    a = rotation.logit_error_direct(q, k, khat)
    b = rotation.logit_error_trace(q, k, khat)
    assert abs(a - b) <= 1e-10 * a


def test_clip_threshold_quantile_brute_force():
    # Linear-interpolation quantile written out: position (n-1) c between sorted neighbours.
    rng = np.random.default_rng(2)
    x = rng.standard_normal((101, 5)) * np.arange(1, 6)
    for c in (0.96, 0.92, 0.5):
        tau = rotation.clip_thresholds(x, c)
        for j in range(5):
            a = np.sort(np.abs(x[:, j]))
            pos = (len(a) - 1) * c
            lo = int(np.floor(pos))
            ref = a[lo] + (pos - lo) * (a[min(lo + 1, len(a) - 1)] - a[lo])
            assert abs(tau[j] - ref) < 1e-12
            frac = np.mean(np.abs(x[:, j]) <= tau[j] + 1e-15)
            assert c - 1.0 / len(a) <= frac <= c + 1.0 / len(a)
