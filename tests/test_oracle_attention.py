"""Pins of the oracle's attention: brute-force softmax, a library SDPA in float64,
the pages' read-path form (dequantise, inverse-rotate, attend), and the
method-level ordering of quantisation error the pages report."""
import itertools

import numpy as np
import pytest

import synth
from oracle import attention as A
from oracle import pool as P
from oracle import quant, rotation

torch = pytest.importorskip("torch")


def _sdpa(q, k, v, scale):
    qt = torch.from_numpy(np.asarray(q, np.float64))[None, None, None]
    kt = torch.from_numpy(np.asarray(k, np.float64))[None, None]
    vt = torch.from_numpy(np.asarray(v, np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, 0, 0].numpy()


def test_softmax_attention_brute_force():
    rng = np.random.default_rng(0)
    q, k, v = rng.standard_normal(8), rng.standard_normal((5, 8)), rng.standard_normal((5, 8))
    w = np.array([np.exp(0.7 * q @ k[i]) for i in range(5)])
    o_ref = sum(w[i] * v[i] for i in range(5)) / w.sum()
    o, lse = A.softmax_attention(q, k, v, 0.7)
    assert np.abs(o - o_ref).max() < 1e-14
    assert abs(lse - np.log(w.sum())) < 1e-13


@pytest.mark.parametrize("L", [1, 2, 5, 9, 16])
def test_segmented_merge_equals_full_softmax(L):
    rng = np.random.default_rng(L)
    q, k, v = rng.standard_normal(8) * 3, rng.standard_normal((L, 8)), rng.standard_normal((L, 8))
    logits = 0.5 * (k @ q)
    o_ref, lse_ref = A.softmax_attention(q, k, v, 0.5)
    # every split of [0, L) into up to 3 contiguous segments, empty segments allowed
    for a, b in itertools.combinations_with_replacement(range(L + 1), 2):
        parts = [A.segment_partial(logits[s], v[s]) for s in (slice(0, a), slice(a, b), slice(b, L))]
        parts.append(A.segment_partial(logits[:0], v[:0]))            # an explicitly empty one
        o, lse = A.merge_partials(parts)
        assert np.abs(o - o_ref).max() < 1e-13
        assert abs(lse - lse_ref) < 1e-13


def _params(seed, hkv):
    out = []
    for h in range(hkv):
        qc, kc, vc = synth.calibration(seed, 0, h)
        cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
        out.append(P.HeadParams(cal["U_K"].astype(np.float32), cal["U_V"].astype(np.float32),
                                cal["tau_K"].astype(np.float32), cal["tau_V"].astype(np.float32)))
    return out


def test_no_history_is_textbook_attention():
    geo = P.PoolGeometry(hkv=1)
    prm = _params(21, 1)
    for L in (1, 63, 64, 65, 200, 320):
        k, v = synth.kv_tokens(21, 0, 0, L)
        q = synth.queries(21, 0, 0, 4)
        pm = P.PoolModel(geo, 1, 5)
        P.prefill(pm, k[:, None], v[:, None], [0], [0, 1, 2, 3, 4], prm, False)
        o, lse = A.decode_request(q, L, pm, [0], [0, 1, 2, 3, 4], prm, False, synth.sm_scale())
        for i in range(4):
            ref = _sdpa(q[i], k, v, synth.sm_scale())
            assert np.abs(o[i] - ref).max() < 1e-12


@pytest.mark.parametrize("v_absorbed", [False, True])
def test_history_is_dequantise_inverse_rotate_attend(v_absorbed):
    # The MarkTechPost article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局": the INT2 read path unpacks, dequantises and
    # inverse-rotates before attention (V-absorbed mode skips V's inverse rotation).
    geo = P.PoolGeometry(hkv=2)
    prm = _params(22, 2)
    L = 64 + 256 + 150
    k = np.stack([synth.kv_tokens(22, 0, h, L)[0] for h in range(2)], axis=1)
    v = np.stack([synth.kv_tokens(22, 0, h, L)[1] for h in range(2)], axis=1)
    q = np.concatenate([synth.queries(22, 0, h, 3) for h in range(2)])
    hist_pt, bf16_pt = [2, 0, 1], [4, 3, 2, 1, 0]
    pm = P.PoolModel(geo, 3, 5)
    P.prefill(pm, k, v, hist_pt, bf16_pt, prm, v_absorbed)
    o, lse = A.decode_request(q, L, pm, hist_pt, bf16_pt, prm, v_absorbed, synth.sm_scale())
    seg, kk, vv = P.gather_request(pm, L, hist_pt, bf16_pt)
    hist = np.array([s == "history" for s in seg])
    for h in range(2):
        keff, veff = kk[:, h].copy(), vv[:, h].copy()
        rk = rotation.composite_rotation(prm[h].u_k.astype(np.float64))
        rv = rotation.composite_rotation(prm[h].u_v.astype(np.float64))
        keff[hist] = keff[hist] @ rk.T                 # inverse rotation of the dequantised key
        if not v_absorbed:
            veff[hist] = veff[hist] @ rv.T
        for i in range(3 * h, 3 * h + 3):
            ref = _sdpa(q[i], keff, veff, synth.sm_scale())
            assert np.abs(o[i] - ref).max() < 1e-11 * np.abs(ref).max()


def test_bf16_decode_reference_is_sdpa():
    rng = np.random.default_rng(5)
    L, hkv = 150, 2
    k = synth.bf16_round(rng.standard_normal((L, hkv, 128)))
    v = synth.bf16_round(rng.standard_normal((L, hkv, 128)))
    q = synth.bf16_round(rng.standard_normal((4, 128)))
    pt = np.array([2, 0, 1])
    pages = np.zeros((3, hkv, 2, 64, 128), np.uint16)
    for pos in range(L):
        pages[pt[pos // 64], :, 0, pos % 64] = synth.bf16_bits(k[pos])
        pages[pt[pos // 64], :, 1, pos % 64] = synth.bf16_bits(v[pos])
    o, lse = A.bf16_decode_request(q, L, pages, pt, 0.1)
    for i in range(4):
        ref = _sdpa(q[i], k[:, i // 2], v[:, i // 2], 0.1)
        assert np.abs(o[i] - ref).max() < 1e-12


def _logit_errors(model: str, seeds=range(3)):
    """Query-weighted logit error ||Q K^T - Q Khat^T||_F^2 summed over heads, per rotation."""
    d = 128
    errs = {"oscar": 0.0, "hadamard": 0.0, "naive": 0.0}
    for h in seeds:
        st = synth.head_stats(40, 0, h)
        rng = np.random.default_rng(100 + h)

        def gen_k(n):
            k = rng.standard_normal((n, d))
            if model == "aligned":       # large key energy along the queries' principal directions
                k += (rng.standard_normal((n, 4)) * 16) @ st.basis[:, :4].T
            else:                        # massive canonical channels (the configs' outlier recipe)
                k[:, st.outliers] *= 16
            return synth.bf16_round(k)

        qc = synth.queries(40, 0, h, 512, kind="calq")
        kc, vc = gen_k(512), gen_k(512)
        cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
        kt, qt = gen_k(512), synth.queries(40, 0, h, 256)
        rots = {"oscar": cal["R_K"], "hadamard": rotation.hadamard(d) @ rotation.bitrev_matrix(d), "naive": np.eye(d)}
        for name, r in rots.items():
            tau = rotation.clip_thresholds(kc.astype(np.float64) @ r, 0.96).astype(np.float32)
            kr = (kt.astype(np.float64) @ r).astype(np.float32)
            c, s, z = quant.quantize_token(kr, tau, 64)
            khat = quant.dequantize(c, s, z) @ r.T
            errs[name] += rotation.logit_error_trace(qt, kt, khat)
    return errs


def test_attention_aware_rotation_wins_when_keys_share_query_directions():
    # The MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同做法": the key rotation should come from the query
    # covariance, because the logit error is weighted by Q^T Q. When the keys'
    # large components lie along the queries' principal directions, U_Q maps
    # them onto a few channels that H_Had then spreads evenly, while a
    # data-independent Hadamard leaves them unevenly spread. Only the ordering is pinned.
    e = _logit_errors("aligned")
    assert e["oscar"] < 0.8 * e["hadamard"]
    assert e["oscar"] < 0.8 * e["naive"]


def test_any_rotation_beats_naive_on_massive_channels():
    # The MarkTechPost article "Together AI 开源 OSCAR…", section "为什么 INT2 KV 缓存量化很难": a few channels with huge values dominate
    # the per-group scale; rotations spread them (the news article "超越 TurboQuant…", section "OSCAR 的设计思路": Hadamard
    # disperses outliers). On axis-aligned outlier channels both rotations beat naive INT2.
    e = _logit_errors("axis")
    assert e["hadamard"] < 0.5 * e["naive"]
    assert e["oscar"] < 0.5 * e["naive"]
