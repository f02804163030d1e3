"""The allocation-free decode entry point (oscar_decode_attention_noalloc).

Callers that cannot call cudaMalloc (code running inside CUDA graph capture,
engines whose allocator owns all device memory, latency-critical hosts) use
this entry point: it keeps its scratch in a fixed device array inside the
library instead of a caller-allocated workspace. These tests call it through
the C ABI and check that it gives the same attention output as
oscar_decode_attention, within the decode tolerance (2e-3 of each row's
largest magnitude), on two calls in a row that reuse the shared scratch.
This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import DEV, head_params, queries, row_rel_err, to_dev_bf16, tokens, upload_params, with_codebooks
import synth

TOL = 2e-3


def _cache(lens, hkv, gq, v_mode, seed, meta=0):
    B = len(lens)
    nh = [max(0, (L - 320 + 63) // 64) for L in lens]
    mhp = max(1, max(nh))
    hist_pt = np.full((B, mhp), -1, np.int32)
    o = 0
    for r in range(B):
        hist_pt[r, :nh[r]] = np.arange(o, o + nh[r])
        o += nh[r]
    bf16_pt = np.arange(5 * B, dtype=np.int32).reshape(B, 5)
    cfg = osc.CacheConfig(num_layers=2, num_kv_heads=hkv, num_q_heads=hkv * gq, num_int2_pages=o + 1,
                          num_bf16_pages=5 * B, max_batch=B, max_splits=64, v_mode=v_mode, meta_format=meta)
    cache = osc.OscarCache(cfg, device=DEV)
    for layer in range(2):
        prm = head_params(seed + layer, layer, hkv)
        upload_params(cache, layer, with_codebooks(seed + layer, layer, prm) if meta == osc.META_CB else prm)
        ks, vs = zip(*[tokens(seed, layer, hkv, L, extra=r) for r, L in enumerate(lens)])
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        cache.quantize_prefill(layer, to_dev_bf16(np.concatenate(ks)), to_dev_bf16(np.concatenate(vs)), cu,
                               hist_pt, bf16_pt)
    assert cache.get_status() == 0
    return cache, hist_pt, bf16_pt


@pytest.mark.parametrize("meta", [0, 1, 2], ids=["meta_f16", "meta_u8", "meta_cb"])
@pytest.mark.parametrize("v_mode", [0, 1])
def test_noalloc_matches_decode_attention_on_two_calls(v_mode, meta):
    lens, hkv, gq = [1024, 5000, 300], 2, 4
    cache, hp, bp = _cache(lens, hkv, gq, v_mode, seed=41, meta=meta)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    hp_d, bp_d = torch.from_numpy(hp).to(DEV), torch.from_numpy(bp).to(DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    for call, layer in enumerate((1, 0)):            # two calls in a row, different layers and queries
        q = to_dev_bf16(queries(41 + call, layer, hkv, gq, batch=len(lens)))
        ref = cache.decode_attention(layer, q, seq, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32)
        lse = torch.zeros(len(lens), hkv * gq, dtype=torch.float32, device=DEV)
        got = osc.decode_attention_noalloc(cache.cfg, cache.pool, layer, q, seq, hp_d, bp_d, synth.sm_scale(),
                                           out_dtype=osc.OUT_FP32, lse=lse, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        r, g = ref.double().cpu().numpy(), got.double().cpu().numpy()
        for b in range(len(lens)):
            assert row_rel_err(g[b], r[b]).max() <= TOL, (call, b)
        assert torch.isfinite(lse).all()
    assert cache.get_status() == 0


def test_noalloc_rejects_work_beyond_its_scratch():
    # B * Hq query rows too many for the fixed scratch even with one split: rejected on the host
    cache, hp, bp = _cache([400], 1, 8, 0, seed=42)
    B = 4096
    q = torch.zeros(B, 8, 128, dtype=torch.bfloat16, device=DEV)
    seq = torch.full((B,), 400, dtype=torch.int32, device=DEV)
    hp_d = torch.zeros(B, hp.shape[1], dtype=torch.int32, device=DEV)
    bp_d = torch.zeros(B, 5, dtype=torch.int32, device=DEV)
    with pytest.raises(osc.OscarError) as e:
        osc.decode_attention_noalloc(cache.cfg, cache.pool, 0, q, seq, hp_d, bp_d, synth.sm_scale())
    assert e.value.code == osc.ERR_TOO_LARGE
