"""Pins of the oracle's Lloyd-Max codebook variant.

Lloyd's iteration is pinned to the closed-form optimal 4-level quantisers of the
uniform distribution (levels 1/8, 3/8, 5/8, 7/8) and of the Gaussian (Max 1960:
levels +-0.4528, +-1.5104, thresholds 0, +-0.9816), to its fixed-point conditions
and its monotone descent from the uniform levels; the encoder to brute-force
nearest-level search, its tie rule and the half-gap error bound; the pool to the
bulk-prefill / token-by-token append equivalence.
"""
import numpy as np
import pytest
from scipy.stats import norm

import synth
from oracle import codebook as CB
from oracle import pool as P
from oracle import quant, rotation

F32 = np.float32


def test_lloyd_max_uniform_distribution_closed_form():
    n = 200000
    u = (np.arange(n) + 0.5) / n
    c = CB.lloyd_max(u)
    assert np.allclose(c, [1 / 8, 3 / 8, 5 / 8, 7 / 8], atol=1e-4)


def test_lloyd_max_gaussian_matches_max_1960():
    n = 400000
    x = norm.ppf((np.arange(n) + 0.5) / n)          # quantile grid of N(0, 1)
    u = np.clip(0.5 + x / 10.0, 0.0, 1.0)           # affine map into [0, 1]; Lloyd's iteration is equivariant
    c = CB.lloyd_max(u)
    lev = (c - 0.5) * 10.0
    assert np.allclose(lev, [-1.5104, -0.4528, 0.4528, 1.5104], atol=2e-3)
    th = 0.5 * (lev[:-1] + lev[1:])
    assert np.allclose(th, [-0.9816, 0.0, 0.9816], atol=2e-3)


def test_lloyd_fixed_point_and_descent():
    rng = np.random.default_rng(2)
    u = np.concatenate([rng.beta(2, 5, 30000), rng.beta(6, 2, 10000)])
    c = CB.lloyd_max(u)
    t = 0.5 * (c[:-1] + c[1:])
    cell = np.searchsorted(t, u, side="left")       # u <= t_0 -> 0, ...
    for i in range(4):
        assert abs(u[cell == i].mean() - c[i]) < 1e-9
    mse = lambda lv: np.mean(np.min((u[:, None] - np.asarray(lv)[None, :]) ** 2, axis=1))
    assert mse(c) <= mse([0, 1 / 3, 2 / 3, 1]) + 1e-15
    assert mse(c) < 0.8 * mse([0, 1 / 3, 2 / 3, 1])


def test_codebook_bytes_round_and_sort():
    assert list(CB.codebook_bytes([0.0, 1 / 3, 2 / 3, 1.0])) == [0, 85, 170, 255]
    assert list(CB.codebook_bytes([0.5, 0.1, 1.2, -0.1])) == [0, 26, 128, 255]


def test_encoder_is_nearest_level_brute_force():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((300, 128)) * rng.uniform(0.05, 6, size=(300, 1))).astype(F32)
    tau = rng.uniform(0.5, 4.0, 128).astype(F32)
    for kcb in (CB.UNIFORM, np.array([20, 70, 160, 240], np.uint8), np.array([0, 0, 200, 210], np.uint8)):
        y = quant.clip(x, tau)
        c, r16, z16 = CB.quantize_token(x, tau, kcb)
        t = (y.astype(np.float64).reshape(300, 2, 64) - z16.astype(np.float64)[..., None]) / \
            r16.astype(np.float64)[..., None]
        lev = kcb.astype(np.float64) / 255.0
        dist = np.abs(t[..., None] - lev)
        mine = np.take_along_axis(dist, c.reshape(300, 2, 64)[..., None].astype(np.int64), axis=-1)[..., 0]
        assert np.all(mine - dist.min(-1) <= 1e-6)
        assert c.max() <= 3


def test_encoder_tie_goes_to_the_lower_level():
    kcb = np.array([0, 100, 200, 255], np.uint8)
    th = CB.thresholds(kcb)
    y = np.zeros((1, 64), F32)
    y[0, 1] = 1.0                                   # min 0, max 1: range' = 1, zero' = 0, t = y
    y[0, 2] = th[0]
    y[0, 3] = np.nextafter(th[0], F32(1.0))
    y[0, 4] = th[2]
    c, r16, z16 = CB.quantize_groups(y, 64, kcb)
    assert float(r16[0, 0]) == 1.0 and float(z16[0, 0]) == 0.0
    assert c[0, 2] == 0 and c[0, 3] == 1 and c[0, 4] == 2 and c[0, 1] == 3 and c[0, 0] == 0


def test_constant_group_and_error_bound():
    kcb = np.array([30, 90, 150, 235], np.uint8)
    y = np.full((1, 64), 0.7, F32)
    c, r16, z16 = CB.quantize_groups(y, 64, kcb)
    assert np.all(c == 0) and float(r16[0, 0]) == 0.0
    assert np.all(CB.dequantize(c, r16, z16, kcb) == float(np.float16(0.7)))
    rng = np.random.default_rng(4)
    y = (rng.standard_normal((500, 128)) * 2).astype(F32)
    c, r16, z16 = CB.quantize_groups(y, 64, kcb)
    err = np.abs(y.astype(np.float64) - CB.dequantize(c, r16, z16, kcb))
    k = kcb.astype(np.float64)
    worst = max(k[0], 255 - k[3], *(np.diff(k) / 2)) / 255.0
    r = r16.astype(np.float64).repeat(64, axis=1)
    assert np.all(err <= worst * r * (1 + 1e-3) + 2e-3 * np.abs(y) + 1e-3)


def test_uniform_codebook_matches_uniform_quantiser_levels():
    # with (0, 85, 170, 255) the levels are min + range * {0, 1/3, 2/3, 1}: the codes agree with the
    # uniform quantiser's wherever neither sits within float rounding of a decision boundary
    rng = np.random.default_rng(5)
    y = (rng.standard_normal((400, 128)) * 3).astype(F32)
    c1, _, _ = CB.quantize_groups(y, 64, CB.UNIFORM)
    c2, s, z = quant.quantize_groups(y, 64)
    t = (y.astype(np.float64) - z.astype(np.float64).repeat(64, 1)) / np.maximum(s.astype(np.float64).repeat(64, 1),
                                                                              1e-30)
    near = np.abs(t - np.floor(t) - 0.5) < 1e-2
    assert np.array_equal(c1[~near], c2[~near])


def _params(seed, hkv):
    out = []
    for h in range(hkv):
        qc, kc, vc = synth.calibration(seed, 0, h)
        cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
        uk, uv = cal["U_K"].astype(F32), cal["U_V"].astype(F32)
        tk, tv = cal["tau_K"].astype(F32), cal["tau_V"].astype(F32)
        cbk = CB.calibrate_codebook(P.rotated_f32(kc, uk), tk)
        cbv = CB.calibrate_codebook(vc.astype(F32), tv)
        out.append(P.HeadParams(uk, uv, tk, tv, cbk, cbv))
    return out


def test_calibrated_codebook_beats_uniform_on_fresh_tokens():
    prm = _params(31, 1)[0]
    assert prm.cb_k[0] > 0 and prm.cb_k[3] < 255            # Lloyd pulls the end levels inwards
    k, v = synth.kv_tokens(31, 0, 0, 4000, extra=9)
    kr = P.rotated_f32(k, prm.u_k)
    y = quant.clip(kr, prm.tau_k).astype(np.float64)
    c, r, z = CB.quantize_token(kr, prm.tau_k, prm.cb_k)
    cu, ru, zu = CB.quantize_token(kr, prm.tau_k, CB.UNIFORM)
    e_cb = np.mean((y - CB.dequantize(c, r, z, prm.cb_k)) ** 2)
    e_un = np.mean((y - CB.dequantize(cu, ru, zu, CB.UNIFORM)) ** 2)
    assert e_cb < e_un


@pytest.mark.parametrize("v_absorbed", [False, True])
def test_codebook_prefill_equals_incremental_append(v_absorbed):
    geo = P.PoolGeometry(hkv=2, meta_format="cb")
    prm = _params(32, 2)
    L0, L = 300, 64 + 256 + 140
    k = np.stack([synth.kv_tokens(32, 0, h, L)[0] for h in range(2)], axis=1)
    v = np.stack([synth.kv_tokens(32, 0, h, L)[1] for h in range(2)], axis=1)
    hist_pt, bf16_pt = np.array([3, 0, 5]), np.array([4, 1, 2, 0, 3])
    a = P.PoolModel(geo, 6, 5)
    P.prefill(a, k, v, hist_pt, bf16_pt, prm, v_absorbed)
    b = P.PoolModel(geo, 6, 5)
    P.prefill(b, k[:L0], v[:L0], hist_pt, bf16_pt, prm, v_absorbed)
    for pos in range(L0, L):
        P.append(b, k[pos], v[pos], pos, hist_pt, bf16_pt, prm, v_absorbed)
    assert np.array_equal(a.int2, b.int2) and np.array_equal(a.bf16, b.bf16)
    seg, kk, vv = P.gather_request(a, L, hist_pt, bf16_pt, params=prm)
    hist = np.array([s == "history" for s in seg])
    xr = P.rotated_f32(k[hist, 0], prm[0].u_k)
    c, r, z = CB.quantize_token(xr, prm[0].tau_k, prm[0].cb_k)
    assert np.array_equal(kk[hist, 0], CB.dequantize(c, r, z, prm[0].cb_k))
