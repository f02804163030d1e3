"""Multi-step decode on the GPU: oscar_decode_step against append + decode, and a
Qwen3-8B-shaped layer (32 query / 8 kv heads, 32,768-token prefill, then 256
steps of append, demotion and decode) against the oracle at steps 1, 64, 128,
192 and 256, with the final pool compared row by row."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import (DEV, compare_int2_pools, head_params, pool_from_device, queries, row_rel_err, to_dev_bf16,
                           tokens, upload_params, with_codebooks)
import synth
from oracle import attention as A
from oracle import pool as P

TOL = 2e-3


def _cache(hkv, gq, L_final, v_mode, algo, B=1, meta=0):
    nh = max(1, (L_final - 320 + 63) // 64)
    cfg = osc.CacheConfig(num_layers=1, num_kv_heads=hkv, num_q_heads=hkv * gq, num_int2_pages=B * nh,
                          num_bf16_pages=5 * B, max_batch=B, max_splits=256, v_mode=v_mode, meta_format=meta)
    cache = osc.OscarCache(cfg, device=DEV)
    cache.set_decode_algo(algo)
    hist_pt = np.arange(B * nh, dtype=np.int32).reshape(B, nh)[:, ::-1].copy()
    bf16_pt = np.arange(5 * B, dtype=np.int32).reshape(B, 5)
    return cache, hist_pt, bf16_pt


@pytest.mark.parametrize("algo", [pytest.param(0, id="simt"), pytest.param(1, id="mma")])
@pytest.mark.parametrize("v_mode", [0, 1])
def test_decode_step_equals_append_then_decode(algo, v_mode):
    hkv, gq, L0, steps = 2, 4, 64 + 256 + 500, 70
    prm = head_params(31, 0, hkv)
    k, v = tokens(31, 0, hkv, L0 + steps)
    caches = []
    for _ in range(2):
        c, hp, bp = _cache(hkv, gq, L0 + steps, v_mode, algo)
        upload_params(c, 0, prm)
        c.quantize_prefill(0, to_dev_bf16(k[:L0]), to_dev_bf16(v[:L0]), np.array([0, L0], np.int32), hp, bp)
        caches.append(c)
    hp_d, bp_d = torch.from_numpy(hp).to(DEV), torch.from_numpy(bp).to(DEV)
    for s in range(steps):
        q = to_dev_bf16(queries(31, 0, hkv, gq, extra=s))
        kn, vn = to_dev_bf16(k[L0 + s][None]), to_dev_bf16(v[L0 + s][None])
        lb = torch.tensor([L0 + s], dtype=torch.int32, device=DEV)
        o1 = caches[0].decode_step(0, q, kn, vn, lb, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32)
        caches[1].append_kv(0, kn, vn, lb, hp_d, bp_d)
        o2 = caches[1].decode_attention(0, q, lb + 1, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32)
        assert torch.equal(o1, o2), s
    assert caches[0].get_status() == 0 and caches[1].get_status() == 0
    assert torch.equal(caches[0].pool, caches[1].pool)


@pytest.mark.parametrize("meta", [pytest.param("u8", id="meta_u8"), pytest.param("cb", id="meta_cb")])
@pytest.mark.parametrize("v_mode", [0, 1])
def test_metadata_formats_8k_then_64_steps(v_mode, meta):
    # the 16-bit-per-group and the codebook formats through prefill, 64 fused append + demotion +
    # decode steps
    hkv, gq, L0, steps = 8, 4, 8192, 64
    cache, hp, bp = _cache(hkv, gq, L0 + steps, v_mode, 1, meta=osc.META_U8 if meta == "u8" else osc.META_CB)
    prm = head_params(33, 0, hkv)
    if meta == "cb":
        prm = with_codebooks(33, 0, prm)
    upload_params(cache, 0, prm)
    k, v = tokens(33, 0, hkv, L0 + steps)
    cache.quantize_prefill(0, to_dev_bf16(k[:L0]), to_dev_bf16(v[:L0]), np.array([0, L0], np.int32), hp, bp)
    hp_d, bp_d = torch.from_numpy(hp).to(DEV), torch.from_numpy(bp).to(DEV)
    for s in range(1, steps + 1):
        q = queries(33, 0, hkv, gq, extra=s)
        lb = torch.tensor([L0 + s - 1], dtype=torch.int32, device=DEV)
        out = cache.decode_step(0, to_dev_bf16(q), to_dev_bf16(k[L0 + s - 1][None]), to_dev_bf16(v[L0 + s - 1][None]),
                                lb, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32)
        if s in (1, steps):
            assert cache.get_status() == 0
            pm = pool_from_device(cache, 0)
            ref, _ = A.decode_request(q[0], L0 + s, pm, hp[0], bp[0], prm, v_mode == osc.V_ABSORBED,
                                      synth.sm_scale())
            err = row_rel_err(out[0].double().cpu().numpy(), ref)
            assert err.max() <= TOL, (s, err.max())
    ref_pool = P.PoolModel(P.PoolGeometry(hkv=hkv, meta_format=meta), cache.cfg.num_int2_pages,
                           cache.cfg.num_bf16_pages)
    P.prefill(ref_pool, k, v, hp[0], bp[0], prm, v_mode == osc.V_ABSORBED)
    got = pool_from_device(cache, 0)
    assert np.array_equal(got.bf16, ref_pool.bf16)
    compare_int2_pools(got, ref_pool, [(int(hp[0, h // 64]), h % 64) for h in range(L0 + steps - 320)], params=prm)


@pytest.mark.parametrize("algo", [pytest.param(0, id="simt"), pytest.param(1, id="mma")])
def test_qwen3_8b_layer_32k_then_256_steps(algo):
    hkv, gq, L0, steps = 8, 4, 32768, 256
    checks = {1, 64, 128, 192, 256}
    cache, hp, bp = _cache(hkv, gq, L0 + steps, osc.V_ABSORBED, algo)
    prm = head_params(32, 0, hkv)
    upload_params(cache, 0, prm)
    k, v = tokens(32, 0, hkv, L0 + steps)
    cache.quantize_prefill(0, to_dev_bf16(k[:L0]), to_dev_bf16(v[:L0]), np.array([0, L0], np.int32), hp, bp)
    hp_d, bp_d = torch.from_numpy(hp).to(DEV), torch.from_numpy(bp).to(DEV)
    worst = 0.0
    for s in range(1, steps + 1):
        q = queries(32, 0, hkv, gq, extra=s)
        lb = torch.tensor([L0 + s - 1], dtype=torch.int32, device=DEV)
        out = cache.decode_step(0, to_dev_bf16(q), to_dev_bf16(k[L0 + s - 1][None]), to_dev_bf16(v[L0 + s - 1][None]),
                                lb, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32)
        if s in checks:
            assert cache.get_status() == 0
            pm = pool_from_device(cache, 0)
            ref, _ = A.decode_request(q[0], L0 + s, pm, hp[0], bp[0], prm, True, synth.sm_scale())
            err = row_rel_err(out[0].double().cpu().numpy(), ref)
            worst = max(worst, float(err.max()))
            assert err.max() <= TOL, (s, err.max())
    # the pool after 256 demotions equals the oracle's bulk placement of all tokens
    ref_pool = P.PoolModel(P.PoolGeometry(hkv=hkv), cache.cfg.num_int2_pages, cache.cfg.num_bf16_pages)
    P.prefill(ref_pool, k, v, hp[0], bp[0], prm, True)
    got = pool_from_device(cache, 0)
    assert np.array_equal(got.bf16, ref_pool.bf16)
    rows = [(int(hp[0, h // 64]), h % 64) for h in range(L0 + steps - 320)]
    compare_int2_pools(got, ref_pool, rows)
    print(f"max row relative error over checks: {worst:.2e}")
