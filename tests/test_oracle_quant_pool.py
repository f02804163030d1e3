"""Pins of the oracle's quantiser, packing and pool model.

Checked against hand-worked cases, brute-force nearest-level search, the
packing rule (4 codes per byte), and the placement contract written out per
position; plus the equivalence of bulk prefill and token-by-token append.
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle import pool as P
from oracle import quant, rotation

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "oscar_pages.json")))


def test_page_constants_match_geometry_defaults():
    g = P.PoolGeometry(hkv=1)
    assert g.sink == GOLD["sink_tokens"]["value"]
    assert g.recent == GOLD["recent_tokens"]["value"]
    assert g.group == GOLD["group_channels"]["value"]
    # 4 codes per byte -> a 128-channel token is 32 bytes
    assert g.codes_bytes // g.page == g.d // GOLD["codes_per_byte"]["value"]
    share = 100.0 * (g.sink + g.recent) / GOLD["bf16_share_128k_percent"]["context_tokens"]
    assert round(share, 2) == GOLD["bf16_share_128k_percent"]["value"]


def test_quantizer_hand_worked_cases():
    # group of 64 with values 0,1,2,3 repeated: min 0, max 3, scale 1 -> codes are the values
    y = np.tile(np.array([0, 1, 2, 3], np.float32), 16)[None]
    c, s, z = quant.quantize_groups(y, 64)
    assert np.array_equal(c[0], y[0].astype(np.uint8))
    assert float(s[0, 0]) == 1.0 and float(z[0, 0]) == 0.0
    # -1.5 .. 1.5: scale 1, zero -1.5; y = 0 sits at 1.5 levels -> ties to even -> code 2
    y = np.full((1, 64), 0.0, np.float32)
    y[0, 0], y[0, 1] = -1.5, 1.5
    c, s, z = quant.quantize_groups(y, 64)
    assert c[0, 0] == 0 and c[0, 1] == 3 and np.all(c[0, 2:] == 2)
    # y = -1.0 -> 0.5 levels -> ties to even -> code 0 ; y = 1.0 -> 2.5 -> 2
    y[0, 2], y[0, 3] = -1.0, 1.0
    c, _, _ = quant.quantize_groups(y, 64)
    assert c[0, 2] == 0 and c[0, 3] == 2
    # constant group: scale 0, every code 0, dequantised value = fp16(constant)
    y = np.full((1, 64), 0.1, np.float32)
    c, s, z = quant.quantize_groups(y, 64)
    assert np.all(c == 0) and float(s[0, 0]) == 0.0
    assert np.all(quant.dequantize(c, s, z) == float(np.float16(0.1)))


def test_quantizer_fp16_metadata_saturates():
    y = np.zeros((1, 64), np.float32)
    y[0, 0], y[0, 1] = -1e6, 1e6
    c, s, z = quant.quantize_groups(y, 64)
    assert float(s[0, 0]) == 65504.0 and float(z[0, 0]) == -65504.0


def test_quantizer_nearest_level_brute_force():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((500, 128)) * rng.uniform(0.01, 20, size=(500, 1))).astype(np.float32)
    tau = np.full(128, 2.5, np.float32) * np.float32(np.abs(x).max(axis=0).mean() / 3)
    c, s, z = quant.quantize_token(x, tau, 64)
    y = quant.clip(x, tau).astype(np.float64)
    s64 = s.astype(np.float64).repeat(64, axis=1)
    z64 = z.astype(np.float64).repeat(64, axis=1)
    levels = z64[..., None] + s64[..., None] * np.arange(4)[None, None, :]
    dist = np.abs(y[..., None] - levels)
    best = dist.min(axis=-1)
    mine = np.take_along_axis(dist, c[..., None].astype(np.int64), axis=-1)[..., 0]
    # the chosen level is the nearest one, up to float32 rounding of (y - z)/s
    assert np.all(mine - best <= 1e-5 * s64 + 1e-12)
    assert c.max() <= 3
    # and the error bound of uniform quantisation: within half a step inside [z, z + 3 s]
    inside = (y >= z64) & (y <= z64 + 3 * s64)
    err = np.abs(y - quant.dequantize(c, s, z))
    assert np.all(err[inside] <= 0.5 * s64[inside] * (1 + 1e-5) + 1e-12)


def test_clip_is_elementwise_saturation():
    x = np.array([-5, -1, 0, 1, 5], np.float32)
    t = np.array([2, 2, 2, 0.5, 4], np.float32)
    assert np.array_equal(quant.clip(x, t), np.array([-2, -1, 0, 0.5, 4], np.float32))


def test_pack_unpack_roundtrip_and_bit_order():
    # every byte value round-trips
    allb = np.arange(256, dtype=np.uint8)
    assert np.array_equal(quant.pack_codes(quant.unpack_codes(allb[None]))[0], allb)
    # channel j -> byte j//4 at bits 2*(j%4)
    assert quant.pack_codes(np.array([[1, 2, 3, 0]], np.uint8))[0, 0] == 0b00111001
    rng = np.random.default_rng(4)
    c = rng.integers(0, 4, size=(7, 128)).astype(np.uint8)
    p = quant.pack_codes(c)
    assert p.shape == (7, 32)
    assert np.array_equal(quant.unpack_codes(p), c)


def test_int2_block_layout_hand_built():
    geo = P.PoolGeometry(hkv=1)
    pm = P.PoolModel(geo, 1, 1)
    z = np.zeros((1, 2), np.float16)
    k0 = quant.pack_codes(np.full((1, 128), 1, np.uint8))
    v0 = quant.pack_codes(np.full((1, 128), 1, np.uint8))
    v1 = quant.pack_codes(np.full((1, 128), 2, np.uint8))
    s = np.array([[0.5, 0.25]], np.float16)
    zz = np.array([[-1.0, 2.0]], np.float16)
    v3 = quant.pack_codes(np.full((1, 128), 3, np.uint8))
    pm.write_history(0, [5], 0, k0, z, z, v0, z, z)
    pm.write_history(0, [0], 0, k0, s, zz, v0, s, zz)
    pm.write_history(0, [1], 0, k0, z, z, v1, z, z)
    pm.write_history(0, [5], 0, k0, z, z, v3, z, z)      # rewriting row 5 replaces only its own bits
    blk = pm.int2[0, 0]
    assert geo.block_bytes == 5120
    assert np.all(blk[0:32] == 0x55) and np.all(blk[32:64] == 0x55)   # K rows 0, 1 token-major
    # V codes region, channel-major: channel c's 16 bytes in slot c ^ ((c >> 4) & 7). Row 0 (code 1) is word 0,
    # bits 0-1; row 1 (code 2) word 0, bits 16-17; row 5 (code 3) word 2 ((5 >> 1) & 3), bits 16-17.
    vreg = blk[2048:4096].reshape(128, 4, 4).view("<u4")[..., 0]       # [slot][word]
    for c in (0, 5, 17, 63, 100, 127):
        s = c ^ ((c >> 4) & 7)
        assert vreg[s, 0] == 1 | (2 << 16) and vreg[s, 1] == 0 and vreg[s, 2] == 3 << 16 and vreg[s, 3] == 0
    # K metadata of row 0: fp16 scale, zero per group
    meta = blk[4096:4104].view(np.float16)
    assert list(meta) == [0.5, -1.0, 0.25, 2.0]
    assert list(blk[4608:4616].view(np.float16)) == [0.5, -1.0, 0.25, 2.0]
    # round trip through the reader
    kc, ks, kz, vc, vs, vz = pm.read_history(0, [0, 1, 5, 2], 0)
    assert np.all(kc[:3] == 1) and np.all(vc[0] == 1) and np.all(vc[1] == 2) and np.all(vc[2] == 3)
    assert np.all(vc[3] == 0)
    assert list(ks[0]) == [0.5, 0.25] and list(vz[0]) == [-1.0, 2.0]


def test_segments_and_placement_contract():
    geo = P.PoolGeometry(hkv=1)
    L = 64 + 700 + 256
    segs = [P.segment_of(p, L, geo) for p in range(L)]
    assert segs[:64] == ["sink"] * 64
    assert segs[64:764] == ["history"] * 700
    assert segs[764:] == ["recent"] * 256
    assert P.history_len(L, geo) == 700
    for L2 in (1, 63, 64, 65, 320, 321):
        s = [P.segment_of(p, L2, geo) for p in range(L2)]
        assert s.count("history") == P.history_len(L2, geo)
        assert s.count("sink") == min(L2, 64)
    # recent ring slot of pos is (pos - S0) mod W: pos 764 -> slot (700 % 256) = 188 -> page 1 + 2, row 60
    assert P.bf16_location(764, "recent", [10, 11, 12, 13, 14], geo) == (13, 60)


def _params(seed, hkv):
    out = []
    for h in range(hkv):
        qc, kc, vc = synth.calibration(seed, 0, h)
        cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
        out.append(P.HeadParams(cal["U_K"].astype(np.float32), cal["U_V"].astype(np.float32),
                                cal["tau_K"].astype(np.float32), cal["tau_V"].astype(np.float32)))
    return out


@pytest.mark.parametrize("v_absorbed", [False, True])
def test_prefill_equals_incremental_append(v_absorbed):
    geo = P.PoolGeometry(hkv=2)
    prm = _params(11, 2)
    L0, L = 300, 64 + 256 + 140
    k = np.stack([synth.kv_tokens(11, 0, h, L)[0] for h in range(2)], axis=1)
    v = np.stack([synth.kv_tokens(11, 0, h, L)[1] for h in range(2)], axis=1)
    hist_pt = np.array([3, 0, 5])
    bf16_pt = np.array([4, 1, 2, 0, 3])
    a = P.PoolModel(geo, 6, 5)
    P.prefill(a, k, v, hist_pt, bf16_pt, prm, v_absorbed)
    b = P.PoolModel(geo, 6, 5)
    P.prefill(b, k[:L0], v[:L0], hist_pt, bf16_pt, prm, v_absorbed)
    for pos in range(L0, L):
        P.append(b, k[pos], v[pos], pos, hist_pt, bf16_pt, prm, v_absorbed)
    assert np.array_equal(a.int2, b.int2)
    assert np.array_equal(a.bf16, b.bf16)


def test_prefill_matches_per_token_placement():
    geo = P.PoolGeometry(hkv=1)
    prm = _params(12, 1)
    L = 64 + 256 + 70
    k, v = synth.kv_tokens(12, 0, 0, L)
    hist_pt, bf16_pt = np.array([1, 0]), np.array([0, 1, 2, 3, 4])
    a = P.PoolModel(geo, 2, 5)
    P.prefill(a, k[:, None], v[:, None], hist_pt, bf16_pt, prm, False)
    b = P.PoolModel(geo, 2, 5)
    for pos in range(L):
        P.place(b, pos, L, 0, k[pos], v[pos], prm[0], False, hist_pt, bf16_pt)
    assert np.array_equal(a.int2, b.int2) and np.array_equal(a.bf16, b.bf16)


def test_gather_dequantises_what_was_written():
    geo = P.PoolGeometry(hkv=1)
    prm = _params(13, 1)
    L = 64 + 256 + 100
    k, v = synth.kv_tokens(13, 0, 0, L)
    hist_pt, bf16_pt = np.array([0, 1]), np.array([0, 1, 2, 3, 4])
    pm = P.PoolModel(geo, 2, 5)
    P.prefill(pm, k[:, None], v[:, None], hist_pt, bf16_pt, prm, False)
    seg, kk, vv = P.gather_request(pm, L, hist_pt, bf16_pt)
    bf = np.array([s != "history" for s in seg])
    assert np.array_equal(kk[bf, 0], k[bf].astype(np.float64))
    # history rows: within half a quantisation step of the clipped rotated value
    kr = P.rotated_f32(k[~bf], prm[0].u_k)
    y = quant.clip(kr, prm[0].tau_k).astype(np.float64)
    c, s, z = quant.quantize_token(kr, prm[0].tau_k, 64)
    step = s.astype(np.float64).repeat(64, axis=1)
    assert np.all(np.abs(kk[~bf, 0] - y) <= 0.5 * step * (1 + 1e-5) + np.abs(y - np.clip(y, z.astype(np.float64).repeat(64, 1), None)) + 1e-3)
