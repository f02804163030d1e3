"""Failure detection on the GPU without a fault: a device wait that nothing
completes gives up after the library's wall-clock limit and reports
STATUS_TIMEOUT through the status word; the context stays usable and the next
decode matches the oracle."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import DEV, head_params, pool_from_device, queries, row_rel_err, to_dev_bf16, tokens, upload_params
import synth
from oracle import attention as A


def test_unfinished_wait_reports_timeout_and_context_survives():
    hkv, gq, L = 1, 4, 1024
    nh = (L - 320 + 63) // 64
    cfg = osc.CacheConfig(num_layers=1, num_kv_heads=hkv, num_q_heads=hkv * gq, num_int2_pages=nh,
                          num_bf16_pages=5, max_batch=1, max_splits=16)
    cache = osc.OscarCache(cfg, device=DEV)
    assert cache.get_status() == 0
    t0 = time.perf_counter()
    cache.check_wait_timeout()
    code = cache.get_status()
    waited = time.perf_counter() - t0
    assert code == osc.STATUS_TIMEOUT
    assert 1.5 < waited < 60.0, waited           # the wait ran out on its own clock (2 s), it did not hang
    assert cache.get_status() == 0               # reading the status cleared it
    # the context still works: a decode right after matches the oracle
    prm = head_params(5, 0, hkv)
    upload_params(cache, 0, prm)
    k, v = tokens(5, 0, hkv, L)
    hp, bp = np.arange(nh, dtype=np.int32)[None], np.arange(5, dtype=np.int32)[None]
    cache.quantize_prefill(0, to_dev_bf16(k), to_dev_bf16(v), np.array([0, L], np.int32), hp, bp)
    q = queries(5, 0, hkv, gq)
    out = cache.decode_attention(0, to_dev_bf16(q), np.array([L], np.int32), hp, bp, synth.sm_scale(),
                                 out_dtype=osc.OUT_FP32)
    assert cache.get_status() == 0
    ref, _ = A.decode_request(q[0], L, pool_from_device(cache, 0), hp[0], bp[0], prm, True, synth.sm_scale())
    assert row_rel_err(out[0].double().cpu().numpy(), ref).max() <= 2e-3
