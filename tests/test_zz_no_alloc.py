"""The allocation-free decode entry point (oscar_decode_attention_noalloc).

Callers that cannot call cudaMalloc (serving engines whose allocator owns all
device memory, hosts that may not allocate on a latency-critical path) use
this entry point: it keeps its scratch in a fixed device array inside the
library instead of a caller-allocated workspace. These tests call it through
the C ABI and check, on two calls in a row that reuse the shared scratch, that
it gives the same attention output as oscar_decode_attention and as the
oracle's fp64 attention over the pool bytes the GPU wrote, within the decode
tolerance (2e-3 of each row's largest magnitude). One case has so many query
rows that the scratch holds fewer history splits than the split policy would
pick, so the history is split more coarsely than in oscar_decode_attention.
This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import (DEV, head_params, pool_from_device, queries, row_rel_err, to_dev_bf16, tokens,
                           upload_params, with_codebooks)
import synth
from oracle import attention as A

TOL = 2e-3


def _cache(lens, hkv, gq, v_mode, seed, meta=0, layers=2):
    B = len(lens)
    nh = [max(0, (L - 320 + 63) // 64) for L in lens]
    mhp = max(1, max(nh))
    hist_pt = np.full((B, mhp), -1, np.int32)
    o = 0
    for r in range(B):
        hist_pt[r, :nh[r]] = np.arange(o, o + nh[r])
        o += nh[r]
    bf16_pt = np.arange(5 * B, dtype=np.int32).reshape(B, 5)
    cfg = osc.CacheConfig(num_layers=layers, num_kv_heads=hkv, num_q_heads=hkv * gq, num_int2_pages=o + 1,
                          num_bf16_pages=5 * B, max_batch=B, max_splits=64, v_mode=v_mode, meta_format=meta)
    cache = osc.OscarCache(cfg, device=DEV)
    params = []
    for layer in range(layers):
        prm = head_params(seed + layer, layer, hkv)
        prm = with_codebooks(seed + layer, layer, prm) if meta == osc.META_CB else prm
        upload_params(cache, layer, prm)
        params.append(prm)
        ks, vs = zip(*[tokens(seed, layer, hkv, L, extra=r) for r, L in enumerate(lens)])
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        cache.quantize_prefill(layer, to_dev_bf16(np.concatenate(ks)), to_dev_bf16(np.concatenate(vs)), cu,
                               hist_pt, bf16_pt)
    assert cache.get_status() == 0
    return cache, hist_pt, bf16_pt, params


def _against_oracle(cache, layer, q, lens, hp, bp, prm, v_mode, got, requests):
    pm = pool_from_device(cache, layer)
    for b in requests:
        ref, _ = A.decode_request(q[b], lens[b], pm, hp[b], bp[b], prm, v_mode == osc.V_ABSORBED, synth.sm_scale())
        assert row_rel_err(got[b], ref).max() <= TOL, ("oracle", b)


@pytest.mark.parametrize("meta", [0, 1, 2], ids=["meta_f16", "meta_u8", "meta_cb"])
@pytest.mark.parametrize("v_mode", [0, 1])
def test_noalloc_matches_decode_attention_on_two_calls(v_mode, meta):
    lens, hkv, gq = [1024, 5000, 300], 2, 4
    cache, hp, bp, params = _cache(lens, hkv, gq, v_mode, seed=41, meta=meta)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    hp_d, bp_d = torch.from_numpy(hp).to(DEV), torch.from_numpy(bp).to(DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    for call, layer in enumerate((1, 0)):            # two calls in a row, different layers and queries
        qn = queries(41 + call, layer, hkv, gq, batch=len(lens))
        q = to_dev_bf16(qn)
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
        _against_oracle(cache, layer, qn, lens, hp, bp, params[layer], v_mode, g, range(len(lens)))
    assert cache.get_status() == 0


def test_noalloc_splits_coarsely_when_the_scratch_is_short():
    # 100 requests x 8 query heads of one kv head: 800 query rows leave the 4 MiB scratch room for
    # two history splits, where oscar_decode_attention's split policy takes more for these 64-page
    # histories; both calls must still agree with the existing entry point and with the oracle
    B, hkv, gq = 100, 1, 8
    lens = [64 + 64 * 60 + 13 * r + 256 for r in range(B)]
    cache, hp, bp, params = _cache(lens, hkv, gq, osc.V_ABSORBED, seed=43, layers=1)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    hp_d, bp_d = torch.from_numpy(hp).to(DEV), torch.from_numpy(bp).to(DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    for call in range(2):
        qn = queries(43 + call, 0, hkv, gq, batch=B)
        q = to_dev_bf16(qn)
        ref = cache.decode_attention(0, q, seq, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32)
        got = osc.decode_attention_noalloc(cache.cfg, cache.pool, 0, q, seq, hp_d, bp_d, synth.sm_scale(),
                                           out_dtype=osc.OUT_FP32, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        r, g = ref.double().cpu().numpy(), got.double().cpu().numpy()
        for b in range(B):
            assert row_rel_err(g[b], r[b]).max() <= TOL, (call, b)
        _against_oracle(cache, 0, qn, lens, hp, bp, params[0], osc.V_ABSORBED, g, (0, 37, 99))
    assert cache.get_status() == 0


def test_noalloc_rejects_work_beyond_its_scratch():
    # B * Hq query rows too many for the fixed scratch even with one split: rejected on the host
    cache, hp, bp, _ = _cache([400], 1, 8, 0, seed=42)
    B = 4096
    q = torch.zeros(B, 8, 128, dtype=torch.bfloat16, device=DEV)
    seq = torch.full((B,), 400, dtype=torch.int32, device=DEV)
    hp_d = torch.zeros(B, hp.shape[1], dtype=torch.int32, device=DEV)
    bp_d = torch.zeros(B, 5, dtype=torch.int32, device=DEV)
    with pytest.raises(osc.OscarError) as e:
        osc.decode_attention_noalloc(cache.cfg, cache.pool, 0, q, seq, hp_d, bp_d, synth.sm_scale())
    assert e.value.code == osc.ERR_TOO_LARGE
