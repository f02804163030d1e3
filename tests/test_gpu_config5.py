"""Qwen3-32B-shaped mixed read/write workload at full size on the GPU: 64 query /
8 kv heads (GQA 8), 8 requests with lengths drawn uniformly from [98,304,
131,072], all prefilled by one oscar_quantize_prefill call, then 512 decode
steps (append with demotion + decode) through oscar_decode_step. Requests 0
and 7 are checked against the oracle: their pool bytes after the prefill, their
outputs at steps 1 and 512, and their pool bytes after the last step."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import DEV, compare_int2_pools, head_params, pool_from_device, row_rel_err, upload_params
import synth
from oracle import attention as A
from oracle import pool as P

SEED, HKV, GQ, B, STEPS = 55, 8, 8, 8, 512
CHECK = (0, 7)


def _tokens_dev(r: int, n: int, outl):
    g = torch.Generator(device=DEV)
    g.manual_seed(SEED * 1009 + r)
    return synth.torch_kv_tokens(n, HKV, outl, g, DEV)


def _rows(hp_row, L):
    return [(int(hp_row[h // 64]), h % 64) for h in range(max(0, L - 320))]


def test_qwen3_32b_mixed_prefill_then_512_steps():
    lens = synth.seq_lens_uniform(SEED, B, 98304, 131072).astype(np.int64)
    nh = [(int(L) + STEPS - 320 + 63) // 64 for L in lens]
    mhp = max(nh)
    hist_pt = np.zeros((B, mhp), np.int32)
    off = 0
    for r in range(B):
        hist_pt[r, :nh[r]] = off + np.arange(nh[r])
        off += nh[r]
    bf16_pt = np.arange(5 * B, dtype=np.int32).reshape(B, 5)
    cfg = osc.CacheConfig(num_layers=1, num_kv_heads=HKV, num_q_heads=HKV * GQ, num_int2_pages=off,
                          num_bf16_pages=5 * B, max_batch=B, max_splits=256, v_mode=osc.V_ABSORBED)
    cache = osc.OscarCache(cfg, device=DEV)
    prm = head_params(SEED, 0, HKV)
    upload_params(cache, 0, prm)
    outl = np.stack([synth.head_stats(SEED, 0, h).outliers for h in range(HKV)])

    # prefill: every request's tokens drawn on the device, one bulk call
    ks, vs, host = [], [], {}
    for r in range(B):
        k, v = _tokens_dev(r, int(lens[r]), outl)
        ks.append(k)
        vs.append(v)
        if r in CHECK:
            host[r] = (k.float().cpu().numpy(), v.float().cpu().numpy())
    k_all, v_all = torch.cat(ks), torch.cat(vs)
    del ks, vs
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    hp_d, bp_d = torch.from_numpy(hist_pt).to(DEV), torch.from_numpy(bf16_pt).to(DEV)
    cache.quantize_prefill(0, k_all, v_all, cu, hp_d, bp_d)
    del k_all, v_all
    assert cache.get_status() == 0
    got = pool_from_device(cache, 0)
    for r in CHECK:
        ref = P.PoolModel(P.PoolGeometry(hkv=HKV), off, 5 * B)
        P.prefill(ref, host[r][0], host[r][1], hist_pt[r], bf16_pt[r], prm, True)
        pages = bf16_pt[r]
        assert np.array_equal(got.bf16[pages], ref.bf16[pages]), r
        compare_int2_pools(got, ref, _rows(hist_pt[r], int(lens[r])))

    # decode steps
    rng = np.random.default_rng(SEED + 1)
    new_k = rng.standard_normal((STEPS, B, HKV, 128)).astype(np.float32)
    new_v = rng.standard_normal((STEPS, B, HKV, 128)).astype(np.float32)
    new_k = torch.from_numpy(new_k).to(torch.bfloat16)
    new_v = torch.from_numpy(new_v).to(torch.bfloat16)
    seq = torch.from_numpy(lens.astype(np.int32)).to(DEV)
    def step_queries(s):
        return np.stack([np.concatenate([synth.queries(SEED, 0, h, GQ, extra=1000 * r + s) for h in range(HKV)])
                         for r in range(B)]).astype(np.float32)

    q_mid = step_queries(2)                      # steps that are not checked reuse one query set
    for s in range(1, STEPS + 1):
        q = step_queries(s) if s in (1, STEPS) else q_mid
        out = cache.decode_step(0, torch.from_numpy(q).to(DEV).to(torch.bfloat16), new_k[s - 1].to(DEV),
                                new_v[s - 1].to(DEV), seq, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32)
        seq += 1
        if s in (1, STEPS):
            assert cache.get_status() == 0
            pm = pool_from_device(cache, 0)
            qb = torch.from_numpy(q).to(torch.bfloat16).float().numpy()
            for r in CHECK:
                L = int(lens[r]) + s
                ref, _ = A.decode_request(qb[r], L, pm, hist_pt[r], bf16_pt[r], prm, True, synth.sm_scale())
                err = row_rel_err(out[r].double().cpu().numpy(), ref)
                print("config5 err", s, r, float(err.max()))
                assert err.max() <= 2e-3, (s, r, err.max())

    # after 512 demotions: each checked request's pool equals the oracle's placement of all its tokens
    got = pool_from_device(cache, 0)
    nk, nv = new_k.float().numpy(), new_v.float().numpy()
    for r in CHECK:
        k = np.concatenate([host[r][0], nk[:, r]])
        v = np.concatenate([host[r][1], nv[:, r]])
        ref = P.PoolModel(P.PoolGeometry(hkv=HKV), off, 5 * B)
        P.prefill(ref, k, v, hist_pt[r], bf16_pt[r], prm, True)
        pages = bf16_pt[r]
        assert np.array_equal(got.bf16[pages], ref.bf16[pages]), r
        compare_int2_pools(got, ref, _rows(hist_pt[r], int(lens[r]) + STEPS))
