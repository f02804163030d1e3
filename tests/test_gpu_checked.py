"""Status bits for inputs the method leaves undefined: non-finite values and fp16
metadata that does not fit.

The pages fix the quantiser (MarkTechPost article "Together AI 开源 OSCAR…",
section "服务系统：混合精度缓存布局": clip to per-channel thresholds, per-token
asymmetric INT2 over 64-channel groups) but not what a NaN or an infinity in a
query, key or value means, nor what happens when a group's scale or zero
exceeds fp16's range. The library stores such rows (clipping NaN and
infinities like any value, saturating the metadata at +-65504) and reports them
in the device status word: OSCAR_STATUS_NONFINITE and OSCAR_STATUS_SATURATED.
These tests plant NaN, infinity and 1e6 inputs on the host; none of them
faults the GPU."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import (DEV, build_decode_case, head_params, queries, to_dev_bf16, tokens, upload_params,
                           with_codebooks)
import synth

META = {"f16": 0, "u8": 1, "cb": 2}


def _cache(meta="f16", hkv=2, n_int2=8, n_bf16=10, max_batch=2):
    cfg = osc.CacheConfig(num_layers=1, num_kv_heads=hkv, num_q_heads=4 * hkv, num_int2_pages=n_int2,
                          num_bf16_pages=n_bf16, max_batch=max_batch, max_splits=32, meta_format=META[meta])
    cache = osc.OscarCache(cfg, device=DEV)
    prm = head_params(51, 0, hkv)
    if meta == "cb":
        prm = with_codebooks(51, 0, prm)
    upload_params(cache, 0, prm)
    return cache, prm


def test_nonfinite_query_is_flagged():
    lens = [1500, 700]
    cache, prm, hp, bp = build_decode_case(lens, 2, 4, 0, seed=52, algo=1)
    q = queries(52, 0, 2, 4, batch=2)
    cache.decode_attention(0, to_dev_bf16(q), np.array(lens, np.int32), hp, bp, synth.sm_scale())
    assert cache.get_status() == 0
    for bad in (np.nan, np.inf, -np.inf):
        q2 = q.copy()
        q2[1, 5, 77] = bad
        cache.decode_attention(0, to_dev_bf16(q2), np.array(lens, np.int32), hp, bp, synth.sm_scale())
        assert cache.get_status() == osc.STATUS_NONFINITE, bad


@pytest.mark.parametrize("where", ["sink", "history", "recent"])
def test_nonfinite_prefill_rows_are_flagged(where):
    L = 64 + 64 * 3 + 256
    cache, _ = _cache(n_int2=4, n_bf16=5, max_batch=1)
    k, v = tokens(53, 0, 2, L)
    pos = {"sink": 10, "history": 64 + 70, "recent": L - 5}[where]
    k[pos, 1, 3] = np.nan
    hist_pt = np.arange(4, dtype=np.int32)[None]
    bf16_pt = np.arange(5, dtype=np.int32)[None]
    cache.quantize_prefill(0, to_dev_bf16(k), to_dev_bf16(v), np.array([0, L], np.int32), hist_pt, bf16_pt)
    assert cache.get_status() == osc.STATUS_NONFINITE
    v[pos, 0, 100] = np.inf
    k[pos, 1, 3] = 0.5
    cache.quantize_prefill(0, to_dev_bf16(k), to_dev_bf16(v), np.array([0, L], np.int32), hist_pt, bf16_pt)
    assert cache.get_status() == osc.STATUS_NONFINITE
    v[pos, 0, 100] = 0.5
    cache.quantize_prefill(0, to_dev_bf16(k), to_dev_bf16(v), np.array([0, L], np.int32), hist_pt, bf16_pt)
    assert cache.get_status() == 0


def test_nonfinite_appended_token_is_flagged():
    L = 64 + 256 + 3                       # the recent window is full: every append demotes a row
    cache, _ = _cache(n_int2=4, n_bf16=5, max_batch=1)
    k, v = tokens(54, 0, 2, L + 2)
    hist_pt = np.arange(4, dtype=np.int32)[None]
    bf16_pt = np.arange(5, dtype=np.int32)[None]
    cache.quantize_prefill(0, to_dev_bf16(k[:L]), to_dev_bf16(v[:L]), np.array([0, L], np.int32), hist_pt, bf16_pt)
    assert cache.get_status() == 0
    kn, vn = k[L:L + 1].copy(), v[L:L + 1].copy()
    vn[0, 1, 0] = -np.inf
    cache.append_kv(0, to_dev_bf16(kn), to_dev_bf16(vn), np.array([L], np.int32), hist_pt, bf16_pt)
    assert cache.get_status() == osc.STATUS_NONFINITE
    cache.append_kv(0, to_dev_bf16(k[L + 1:L + 2]), to_dev_bf16(v[L + 1:L + 2]), np.array([L + 1], np.int32),
                    hist_pt, bf16_pt)
    assert cache.get_status() == 0


def test_nonfinite_pre_rotated_rows_are_flagged():
    cache, _ = _cache()
    x = np.random.default_rng(55).standard_normal((3, 2, 128)).astype(np.float32)
    pages, rows = np.array([0, 1, 2], np.int32), np.array([5, 6, 7], np.int32)
    cache.pack_rotated(0, osc.KIND_K, torch.from_numpy(x).to(DEV), pages, rows)
    assert cache.get_status() == 0
    x[2, 1, 64] = np.nan
    cache.pack_rotated(0, osc.KIND_V, torch.from_numpy(x).to(DEV), pages, rows)
    assert cache.get_status() == osc.STATUS_NONFINITE


@pytest.mark.parametrize("meta", ["f16", "u8", "cb"])
def test_fp16_metadata_saturation_is_flagged(meta):
    # clip thresholds of 1e6 let a group span [-1e6, 1e6]: scale (or range) and zero beyond +-65504 in fp16
    cache, prm = _cache(meta)
    hkv = 2
    tau = np.full((hkv, 128), 1e6, np.float32)
    cache.set_rotation(0, np.stack([p.u_k for p in prm]), np.stack([p.u_v for p in prm]), tau, tau)
    if meta == "cb":
        cache.set_codebook(0, np.stack([p.cb_k for p in prm]), np.stack([p.cb_v for p in prm]))
    x = np.random.default_rng(56).standard_normal((2, hkv, 128)).astype(np.float32)
    pages, rows = np.array([0, 1], np.int32), np.array([0, 1], np.int32)
    cache.pack_rotated(0, osc.KIND_K, torch.from_numpy(x).to(DEV), pages, rows)
    assert cache.get_status() == 0
    x[1, 0, :64] = np.where(np.arange(64) % 2 == 0, 1e6, -1e6)
    cache.pack_rotated(0, osc.KIND_K, torch.from_numpy(x).to(DEV), pages, rows)
    # the compact format stores grid indices, which cannot saturate
    assert cache.get_status() == (0 if meta == "u8" else osc.STATUS_SATURATED)
