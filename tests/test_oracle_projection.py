"""Pins of the oracle's K / V projection (oracle/projection.py), independent of its code:

* exact rational dot products with a pure-Python round-to-nearest-even on 8 significant bits,
  on small random bf16 inputs (brute force);
* ties of the bf16 rounding, which go to the even neighbour, and the carry into the next binade;
* the layout: with W a selection matrix, output (head h, channel c) is the input column W picks
  for row 128 h + c (a transposed W or a swapped head / channel order fails);
* the composition with the write path: the pool after ``project_prefill`` equals the pool after
  ``pool.prefill`` of the rounded products written out by hand.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import pool as P
from oracle import projection as PR


def _bf16_values(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return ((x.view(np.uint32) & 0xFFFF0000).view(np.float32)).astype(np.float64)   # truncated to bf16


def _rne_bf16(fr: Fraction) -> Fraction:
    """round a positive or negative rational to 8 significant bits, ties to even (pure Python)"""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    scaled = a * 128                                   # 1.xxxxxxx: 7 fraction bits
    lo = scaled.numerator // scaled.denominator
    rem = scaled - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * Fraction(lo, 128) * Fraction(2) ** e


def test_brute_force_rational_dot_products():
    rng = np.random.default_rng(3)
    hkv, d, T = 2, 24, 5
    x = _bf16_values(rng, (T, d))
    w = _bf16_values(rng, (hkv * 128, d), 0.3)
    got = PR.project(x, w, hkv)
    for t in range(T):
        for j in range(0, hkv * 128, 7):
            s = sum(Fraction(float(x[t, i])) * Fraction(float(w[j, i])) for i in range(d))
            assert Fraction(float(got[t, j // 128, j % 128])) == _rne_bf16(s), (t, j)


def test_bf16_rounding_ties_go_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: to the even mantissa, 1; 1 + 3 2^-8 -> 1 + 2^-6
    vals = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2 - 2.0 ** -9, 1 + 2.0 ** -8 + 2.0 ** -30])
    want = np.array([1.0, 1 + 2.0 ** -6, -1.0, 2.0, 1 + 2.0 ** -7])
    assert np.array_equal(PR.round_to_bf16(vals), want)


def test_layout_head_channel_and_transpose():
    rng = np.random.default_rng(4)
    hkv, d = 3, 512
    perm = rng.permutation(d)[: hkv * 128]
    w = np.zeros((hkv * 128, d))
    w[np.arange(hkv * 128), perm] = 1.0                # output row j reads input column perm[j]
    x = _bf16_values(rng, (4, d))
    got = PR.project(x, w, hkv)
    for h in range(hkv):
        for c in range(0, 128, 5):
            assert np.array_equal(got[:, h, c], x[:, perm[128 * h + c]].astype(np.float32))


def test_project_prefill_writes_the_rounded_products():
    import synth
    from oracle import rotation
    rng = np.random.default_rng(5)
    hkv, d, L = 2, 256, 64 + 3 * 64 + 256 + 10
    prm = []
    for h in range(hkv):
        qc, kc, vc = synth.calibration(9, 0, h)
        cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
        prm.append(P.HeadParams(cal["U_K"].astype(np.float32), cal["U_V"].astype(np.float32),
                                cal["tau_K"].astype(np.float32), cal["tau_V"].astype(np.float32)))
    x = _bf16_values(rng, (L, d))
    wk = _bf16_values(rng, (hkv * 128, d), d ** -0.5)
    wv = _bf16_values(rng, (hkv * 128, d), d ** -0.5)
    geo = P.PoolGeometry(hkv=hkv)
    hist_pt, bf16_pt = np.arange(4), np.arange(5)
    a = P.PoolModel(geo, 4, 5)
    PR.project_prefill(a, x, wk, wv, hist_pt, bf16_pt, prm, True)
    # the composition by hand: products in float64 (exact for these 8-bit-mantissa inputs up to the
    # sum's rounding), rounded by the pinned rounding, then the write path
    k = PR.round_to_bf16(x @ wk.T).astype(np.float32).reshape(L, hkv, 128)
    v = PR.round_to_bf16(x @ wv.T).astype(np.float32).reshape(L, hkv, 128)
    b = P.PoolModel(geo, 4, 5)
    P.prefill(b, k, v, hist_pt, bf16_pt, prm, True)
    assert np.array_equal(a.int2, b.int2) and np.array_equal(a.bf16, b.bf16)
