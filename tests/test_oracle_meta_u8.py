"""Pins of the oracle's compact metadata format (16 bits per 64-channel group).

The pages budget the INT2 history at 2.25 bits per element, i.e. 16 bits of
metadata per group of 64; the format stores the group's minimum and maximum as
8-bit indices on a grid over [-T, T], T the group's largest clip threshold.
Checked against the pages' bit budgets, hand-worked groups, exact rational
floor / ceil, the containment and half-step error bounds of uniform
quantisation, nearest-level brute force, and the pool's byte layout.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import pool as P
from oracle import quant, rotation

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "oscar_pages.json")))
F32 = np.float32


def test_compact_format_meets_the_pages_bit_budget():
    u8 = P.PoolGeometry(hkv=1, meta_format="u8")
    f16 = P.PoolGeometry(hkv=1)
    bpe = lambda g: 8.0 * (g.codes_bytes + g.meta_bytes) / (g.page * g.d)
    assert bpe(u8) == GOLD["bits_per_element_rotation_baselines"]["value"] == 2.25
    assert bpe(f16) == 2.5
    assert u8.block_bytes == 4608 and f16.block_bytes == 5120
    # whole-cache averages with 320 BF16 tokens: the pages' 2.28 at 128K and 2.38 at 32K
    for key, L in (("bits_per_element_oscar_128k", 131072), ("bits_per_element_oscar_32k_aime", 32768)):
        avg = (bpe(u8) * (L - 320) + 16.0 * 320) / L
        assert round(avg, 2) == GOLD[key]["value"]


def test_hand_worked_groups():
    tau = np.concatenate([np.full(64, 1.5, F32), np.full(64, 3.0, F32)])
    x = np.zeros((1, 128), F32)
    x[0, :64] = np.tile(np.array([-1.5, -0.5, 0.5, 1.5], F32), 16)
    x[0, 64:] = F32(0.1)
    c, mn8, mx8 = quant.quantize_token_u8(x, tau, 64)
    # group 0 spans the whole grid [-T, T]: indices 0 and 255, zero' = -T, the four values are the levels
    assert (int(mn8[0, 0]), int(mx8[0, 0])) == (0, 255)
    assert np.array_equal(c[0, :64], np.tile(np.arange(4, dtype=np.uint8), 16))
    s, z = quant.u8_scale_zero(mn8, mx8, quant.group_bounds(tau, 64))
    assert float(z[0, 0]) == -1.5
    # group 1 is constant 0.1 with T = 3: (0.1 + 3) * 255 / 6 = 131.75 -> indices 131 and 132,
    # scale' = D / 3, (0.1 - zero') / scale' = 0.75 * 3 = 2.25 -> code 2
    assert (int(mn8[0, 1]), int(mx8[0, 1])) == (131, 132)
    assert np.all(c[0, 64:] == 2)
    D = 6.0 / 255.0
    assert abs(float(s[0, 1]) - D / 3) < 1e-7 and abs(float(z[0, 1]) - (131 * D - 3)) < 1e-6


def test_zero_threshold_group_stores_zeros():
    tau = np.concatenate([np.zeros(64, F32), np.ones(64, F32)])
    x = np.random.default_rng(1).standard_normal((5, 128)).astype(F32)
    c, mn8, mx8 = quant.quantize_token_u8(x, tau, 64)
    assert np.all(mn8[:, 0] == 0) and np.all(mx8[:, 0] == 0) and np.all(c[:, :64] == 0)
    s, z = quant.u8_scale_zero(mn8, mx8, quant.group_bounds(tau, 64))
    assert np.all(s[:, 0] == 0) and np.all(z[:, 0] == 0)
    assert np.all(quant.dequantize_sz(c, s, z)[:, :64] == 0.0)


def _random_case(seed, n=400):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n, 128)) * rng.uniform(0.05, 8, size=(n, 1))).astype(F32)
    tau = (rng.uniform(0.5, 4.0, size=128)).astype(F32)
    return x, tau


def test_indices_are_exact_floor_and_ceil():
    x, tau = _random_case(5)
    y = quant.clip(x, tau)
    c, mn8, mx8 = quant.quantize_token_u8(x, tau, 64)
    T = quant.group_bounds(tau, 64)
    yg = y.reshape(len(y), 2, 64)
    checked = 0
    for r in range(0, len(y), 7):
        for g in range(2):
            t = Fraction(float(T[g]))
            for val, got, rnd in ((yg[r, g].min(), mn8[r, g], "floor"), (yg[r, g].max(), mx8[r, g], "ceil")):
                q = (Fraction(float(val)) + t) * 255 / (2 * t)      # exact position on the grid
                want = q.numerator // q.denominator if rnd == "floor" else -((-q.numerator) // q.denominator)
                want = min(max(want, 0), 255)
                frac = abs(q - round(q))
                if frac > Fraction(1, 10000):
                    assert int(got) == want, (r, g, rnd)
                    checked += 1
                else:                      # float32 rounding may land on either side of an integer
                    assert abs(int(got) - want) <= 1
    assert checked > 100


def test_grid_contains_the_group_and_costs_at_most_two_steps():
    x, tau = _random_case(6)
    y = quant.clip(x, tau).astype(np.float64).reshape(-1, 2, 64)
    c, mn8, mx8 = quant.quantize_token_u8(x, tau, 64)
    T = quant.group_bounds(tau, 64).astype(np.float64)
    s, z = quant.u8_scale_zero(mn8, mx8, quant.group_bounds(tau, 64))
    s, z = s.astype(np.float64), z.astype(np.float64)
    mn, mx = y.min(-1), y.max(-1)
    eps = 1e-6 * T
    assert np.all(z <= mn + eps) and np.all(z + 3 * s >= mx - eps)
    D = 2 * T / 255
    assert np.all(3 * s <= (mx - mn) + 2 * D + eps)


def test_nearest_level_and_half_step_bound():
    x, tau = _random_case(7)
    y = quant.clip(x, tau).astype(np.float64)
    c, mn8, mx8 = quant.quantize_token_u8(x, tau, 64)
    s, z = quant.u8_scale_zero(mn8, mx8, quant.group_bounds(tau, 64))
    s64 = s.astype(np.float64).repeat(64, axis=1)
    z64 = z.astype(np.float64).repeat(64, axis=1)
    levels = z64[..., None] + s64[..., None] * np.arange(4)[None, None, :]
    dist = np.abs(y[..., None] - levels)
    mine = np.take_along_axis(dist, c[..., None].astype(np.int64), axis=-1)[..., 0]
    assert np.all(mine - dist.min(-1) <= 1e-5 * s64 + 1e-12)
    err = np.abs(y - quant.dequantize_sz(c, s, z))
    assert np.all(err <= 0.5 * s64 * (1 + 1e-5) + 1e-6 * np.abs(z64) + 1e-12)


def test_compact_block_layout_hand_built():
    geo = P.PoolGeometry(hkv=1, meta_format="u8")
    pm = P.PoolModel(geo, 1, 1)
    k0 = quant.pack_codes(np.full((1, 128), 3, np.uint8))
    v0 = quant.pack_codes(np.full((1, 128), 1, np.uint8))
    a = np.array([[7, 200]], np.uint8)
    b = np.array([[9, 255]], np.uint8)
    pm.write_history(0, [5], 0, k0, a, b, v0, b, a)
    blk = pm.int2[0, 0]
    assert blk.shape == (4608,)
    assert np.all(blk[5 * 32: 6 * 32] == 0xFF)
    assert list(blk[4096 + 5 * 4: 4096 + 6 * 4]) == [7, 9, 200, 255]     # K: mn8, mx8 per group
    assert list(blk[4352 + 5 * 4: 4352 + 6 * 4]) == [9, 7, 255, 200]     # V metadata region
    kc, ka, kb, vc, va, vb = pm.read_history(0, [5], 0)
    assert np.all(kc == 3) and np.all(vc == 1)
    assert list(ka[0]) == [7, 200] and list(kb[0]) == [9, 255] and list(va[0]) == [9, 255]


def _params(seed, hkv):
    out = []
    for h in range(hkv):
        qc, kc, vc = synth.calibration(seed, 0, h)
        cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
        out.append(P.HeadParams(cal["U_K"].astype(F32), cal["U_V"].astype(F32),
                                cal["tau_K"].astype(F32), cal["tau_V"].astype(F32)))
    return out


@pytest.mark.parametrize("v_absorbed", [False, True])
def test_compact_prefill_equals_incremental_append(v_absorbed):
    geo = P.PoolGeometry(hkv=2, meta_format="u8")
    prm = _params(21, 2)
    L0, L = 300, 64 + 256 + 140
    k = np.stack([synth.kv_tokens(21, 0, h, L)[0] for h in range(2)], axis=1)
    v = np.stack([synth.kv_tokens(21, 0, h, L)[1] for h in range(2)], axis=1)
    hist_pt, bf16_pt = np.array([3, 0, 5]), np.array([4, 1, 2, 0, 3])
    a = P.PoolModel(geo, 6, 5)
    P.prefill(a, k, v, hist_pt, bf16_pt, prm, v_absorbed)
    b = P.PoolModel(geo, 6, 5)
    P.prefill(b, k[:L0], v[:L0], hist_pt, bf16_pt, prm, v_absorbed)
    for pos in range(L0, L):
        P.append(b, k[pos], v[pos], pos, hist_pt, bf16_pt, prm, v_absorbed)
    assert np.array_equal(a.int2, b.int2) and np.array_equal(a.bf16, b.bf16)


def test_compact_gather_needs_thresholds_and_stays_within_half_a_step():
    geo = P.PoolGeometry(hkv=1, meta_format="u8")
    prm = _params(22, 1)
    L = 64 + 256 + 100
    k, v = synth.kv_tokens(22, 0, 0, L)
    hist_pt, bf16_pt = np.array([0, 1]), np.array([0, 1, 2, 3, 4])
    pm = P.PoolModel(geo, 2, 5)
    P.prefill(pm, k[:, None], v[:, None], hist_pt, bf16_pt, prm, True)
    with pytest.raises(ValueError):
        P.gather_request(pm, L, hist_pt, bf16_pt)
    seg, kk, vv = P.gather_request(pm, L, hist_pt, bf16_pt, params=prm)
    hist = np.array([s == "history" for s in seg])
    assert np.array_equal(kk[~hist, 0], k[~hist].astype(np.float64))
    for got, raw, u, tau in ((kk, k, prm[0].u_k, prm[0].tau_k), (vv, v, None, prm[0].tau_v)):
        xr = P.rotated_f32(raw[hist], u) if u is not None else raw[hist].astype(F32)
        y = quant.clip(xr, tau).astype(np.float64)
        _, mn8, mx8 = quant.quantize_token_u8(xr, tau, 64)
        s, z = quant.u8_scale_zero(mn8, mx8, quant.group_bounds(tau, 64))
        step = s.astype(np.float64).repeat(64, axis=1)
        assert np.all(np.abs(got[hist, 0] - y) <= 0.5 * step * (1 + 1e-5) + 1e-6)


def test_zero_point_is_the_once_rounded_exact_value():
    rng = np.random.default_rng(9)
    for _ in range(2000):
        T = F32(rng.uniform(1e-3, 50.0) * 10.0 ** int(rng.integers(-3, 3)))
        a = int(rng.integers(0, 256))
        b = int(rng.integers(a, 256))
        s, z = quant.u8_scale_zero(np.uint8(a), np.uint8(b), T)
        D, E = quant.u8_steps(T)
        exact = Fraction(a) * Fraction(float(D)) - Fraction(float(T))
        zf = float(z)
        ulp = float(np.spacing(np.abs(F32(zf)))) if zf != 0 else float(np.spacing(F32(0)))
        assert abs(Fraction(zf) - exact) <= Fraction(ulp) / 2
        assert float(s) == float(F32(F32(b - a) * E))
        assert float(E) == float(F32(D / F32(3)))
