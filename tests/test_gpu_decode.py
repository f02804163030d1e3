"""GPU parity of decode attention against the oracle's fp64 attention over the
same dequantised cache (the pool bytes the GPU wrote, decoded by the oracle).

Tolerance: per (request, q-head) row, max_i |o_i - ref_i| / max_i |ref_i| <= 2e-3
on fp32 output. With bf16 output each element must also lie within one bf16
ulp of the reference plus the same 2e-3 slack (bf16 rounding alone reaches
2^-8 relative)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import (DEV, bf16_ulp, build_decode_case as _build, pool_from_device, queries, row_rel_err,
                           to_dev_bf16, tokens)
import synth
from oracle import attention as A
from oracle import pool as P
from oracle import rotation

TOL = 2e-3
ALGOS = [pytest.param(0, id="simt"), pytest.param(1, id="mma"), pytest.param(2, id="tc")]


def _check(cache, prm, hist_pt, bf16_pt, lens, gq, v_mode, seed, out_dtype=1, kv_heads=None, shared_pages=0):
    hkv = cache.cfg.num_kv_heads
    B = len(lens)
    q = queries(seed, 0, hkv, gq, batch=B)
    out = cache.decode_attention(0, to_dev_bf16(q), np.array(lens, np.int32), hist_pt, bf16_pt, synth.sm_scale(),
                                 out_dtype=out_dtype,
                                 lse=(lse_t := torch.zeros(B, hkv * gq, device=DEV, dtype=torch.float32)),
                                 shared_hist_pages=shared_pages)
    assert cache.get_status() == 0
    got = out.double().cpu().numpy()
    lse = lse_t.double().cpu().numpy()
    pm = pool_from_device(cache, 0)
    worst = 0.0
    for r, L in enumerate(lens):
        ref, ref_lse = A.decode_request(q[r], L, pm, hist_pt[r], bf16_pt[r], prm, v_mode == osc.V_ABSORBED,
                                        synth.sm_scale(), kv_heads=kv_heads)
        rows = ~np.isnan(ref[:, 0])
        err = row_rel_err(got[r][rows], ref[rows])
        worst = max(worst, float(err.max()))
        assert np.abs(lse[r][rows] - ref_lse[rows]).max() < 2e-3 * max(1.0, np.abs(ref_lse[rows]).max())
        if out_dtype == osc.OUT_FP32:
            assert err.max() <= TOL, (r, L, err.max())
        else:
            slack = TOL * np.abs(ref[rows]).max(axis=-1, keepdims=True)
            assert np.all(np.abs(got[r][rows] - ref[rows]) <= bf16_ulp(ref[rows]) + slack), (r, L)
    return worst


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("v_mode", [0, 1])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_tiny_config_decode(algo, v_mode, out_dtype):
    # one request, one kv head shared by 4 query heads, 64 sink + 704 history + 256 recent
    lens, gq = [1024], 4
    cache, prm, hp, bp = _build(lens, 1, gq, v_mode, seed=11, algo=algo)
    _check(cache, prm, hp, bp, lens, gq, v_mode, seed=11, out_dtype=out_dtype)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("v_mode", [0, 1])
def test_running_maximum_jumps(algo, v_mode):
    # One split (4 warps, each taking every fourth history page): keys aligned with the first query head of
    # each kv head on history pages 40 and 52 raise that head's logit maximum twice, each time by more than
    # 8 (log2 units) over everything before it, after the warp's first page. The tensor-core decode keeps
    # its softmax reference until a logit exceeds it by 2^8, then rescales and retakes the page's weights.
    lens, hkv, gq, seed = [4096], 2, 4, 17
    q = queries(seed, 0, hkv, gq, batch=1)[0]
    pos = [64 + 40 * 64 + 10, 64 + 52 * 64 + 33]

    def align(r, k, v):
        for j, p_ in enumerate(pos):
            for h in range(hkv):
                d = q[h * gq] / np.linalg.norm(q[h * gq])
                k[p_, h] = _bf16((1.0 + 3.0 * j) * np.linalg.norm(k[p_, h]) * d)

    cache, prm, hp, bp = _build(lens, hkv, gq, v_mode, seed=seed, algo=algo, max_splits=1, kv_hook=align)
    # the jumps, in the logits of the cache as stored (oracle decode of the pool the GPU wrote)
    pm = pool_from_device(cache, 0)
    seg, kk, _ = P.gather_request(pm, lens[0], hp[0], bp[0], heads=[0], params=prm)
    rk = rotation.composite_rotation(np.asarray(prm[0].u_k, np.float64))
    lg = synth.sm_scale() * 1.4426950408889634 * (kk[:, 0] @ (np.asarray(q[0], np.float64) @ rk))
    hist = np.array([s_ == "history" for s_ in seg])
    before = lg[hist & (np.arange(lens[0]) < pos[0])].max()
    assert lg[pos[0]] > before + 8 and lg[pos[1]] > lg[pos[0]] + 8, (before, lg[pos[0]], lg[pos[1]])
    _check(cache, prm, hp, bp, lens, gq, v_mode, seed=seed, out_dtype=osc.OUT_FP32)


def _bf16(x):
    """float32 -> nearest bf16 value (ties to even), as float32."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return b.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("algo", ALGOS)
def test_edge_lengths(algo):
    lens = [1, 2, 63, 64, 65, 319, 320, 321, 383, 384, 385, 448, 1000]
    cache, prm, hp, bp = _build(lens, 2, 4, 0, seed=12, algo=algo)
    _check(cache, prm, hp, bp, lens, 4, 0, seed=12)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("gq", [1, 2, 8])
def test_gqa_widths(algo, gq):
    lens = [900, 1500]
    cache, prm, hp, bp = _build(lens, 2, gq, 1, seed=13, algo=algo)
    _check(cache, prm, hp, bp, lens, gq, 1, seed=13)


@pytest.mark.parametrize("algo", ALGOS)
def test_shared_prefix_batch(algo):
    lens = [64 + 64 * 20 + 300, 64 + 64 * 20 + 700, 64 + 64 * 20 + 256]
    cache, prm, hp, bp = _build(lens, 2, 4, 0, seed=14, shared_prefix=64 + 64 * 20, algo=algo)
    assert (hp[0, :20] == hp[1, :20]).all() and (bp[:, 0] == bp[0, 0]).all()
    _check(cache, prm, hp, bp, lens, 4, 0, seed=14)


@pytest.mark.parametrize("v_mode", [0, 1])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_shared_prefix_kernel(v_mode, out_dtype):
    # 3 requests sharing 20 history pages read once for all 12 query rows per kv head; the third
    # request has no history pages of its own
    lens = [64 + 64 * 20 + 300, 64 + 64 * 20 + 700, 64 + 64 * 20 + 256]
    cache, prm, hp, bp = _build(lens, 2, 4, v_mode, seed=14, shared_prefix=64 + 64 * 20, algo=1)
    _check(cache, prm, hp, bp, lens, 4, v_mode, seed=14, out_dtype=out_dtype, shared_pages=20)


def test_shared_prefix_two_query_tiles():
    # 20 requests x 8 query heads = 160 rows of one kv head: a full 128-row tile and a partial one;
    # own history from 0 to 11 pages with ragged last pages
    lens = [64 + 64 * 10 + 256 + 37 * r for r in range(20)]
    cache, prm, hp, bp = _build(lens, 1, 8, 0, seed=16, shared_prefix=64 + 64 * 10, algo=1)
    _check(cache, prm, hp, bp, lens, 8, 0, seed=16, shared_pages=10)


def test_shared_prefix_steps():
    # decode_step with the shared-prefix kernel against the plain decode_step on an identical cache:
    # the same pools after 40 steps of append and demotion, outputs within the parity bound of each
    # other at every step and of the oracle at the last one
    B, hkv, gq, shp, S = 4, 2, 4, 12, 40
    lens = [64 + 64 * shp + 64 * r + 10 + 256 for r in range(B)]
    ca, prm, hp, bp = _build(lens, hkv, gq, 0, seed=17, shared_prefix=64 + 64 * shp, algo=1)
    cb, _, _, _ = _build(lens, hkv, gq, 0, seed=17, shared_prefix=64 + 64 * shp, algo=1)
    hp_d, bp_d = torch.from_numpy(hp).to(DEV), torch.from_numpy(bp).to(DEV)
    rng = np.random.default_rng(5)
    for s in range(S):
        q = to_dev_bf16(rng.standard_normal((B, hkv * gq, 128)).astype(np.float32))
        kn = to_dev_bf16(rng.standard_normal((B, hkv, 128)).astype(np.float32))
        vn = to_dev_bf16(rng.standard_normal((B, hkv, 128)).astype(np.float32))
        lb = torch.tensor([L + s for L in lens], dtype=torch.int32, device=DEV)
        oa = ca.decode_step(0, q, kn, vn, lb, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32,
                            shared_hist_pages=shp)
        ob = cb.decode_step(0, q, kn, vn, lb, hp_d, bp_d, synth.sm_scale(), out_dtype=osc.OUT_FP32)
        err = ((oa - ob).abs().amax(-1) / ob.abs().amax(-1)).max().item()
        assert err <= 2 * TOL, (s, err)
    assert ca.get_status() == 0 and cb.get_status() == 0
    assert torch.equal(ca.pool, cb.pool)
    pm = pool_from_device(ca, 0)
    qn = q.float().cpu().numpy().astype(np.float64)
    got = oa.double().cpu().numpy()
    for r in range(B):
        ref, _ = A.decode_request(qn[r], lens[r] + S, pm, hp[r], bp[r], prm, True, synth.sm_scale())
        assert row_rel_err(got[r], ref).max() <= TOL, r


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("v_mode", [0, 1])
@pytest.mark.parametrize("gq", [4, 8])
def test_compact_metadata_decode(algo, v_mode, gq):
    # the 16-bit-per-group metadata format: both decoders, both V modes, the one- and two-n-tile variants
    lens = [1024, 64 + 64 * 13 + 29 + 256, 300]
    cache, prm, hp, bp = _build(lens, 2, gq, v_mode, seed=18, algo=algo, meta="u8")
    assert cache.pool.numel() > 0 and cache.int2_pages(0).shape[-1] == 4608
    _check(cache, prm, hp, bp, lens, gq, v_mode, seed=18)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("v_mode", [0, 1])
@pytest.mark.parametrize("gq", [4, 8])
def test_codebook_decode(algo, v_mode, gq):
    # the Lloyd-Max codebook format: both decoders, both V modes, the one- and two-n-tile variants
    lens = [1024, 64 + 64 * 13 + 29 + 256, 300]
    cache, prm, hp, bp = _build(lens, 2, gq, v_mode, seed=21, algo=algo, meta="cb")
    _check(cache, prm, hp, bp, lens, gq, v_mode, seed=21)


@pytest.mark.parametrize("v_mode", [0, 1])
def test_codebook_shared_prefix_kernel(v_mode):
    lens = [64 + 64 * 20 + 300, 64 + 64 * 20 + 700, 64 + 64 * 20 + 256]
    cache, prm, hp, bp = _build(lens, 2, 4, v_mode, seed=22, shared_prefix=64 + 64 * 20, algo=1, meta="cb")
    _check(cache, prm, hp, bp, lens, 4, v_mode, seed=22, shared_pages=20)


@pytest.mark.parametrize("meta", ["f16", "u8", "cb"])
def test_many_waves_kernel_variant(meta):
    # 32 requests x 8 kv heads: a grid of more than two waves, where the split policy takes the
    # 4-CTAs-per-SM build of the tensor-core decode
    lens = [64 + 64 * 8 + 256 + 17 * r for r in range(32)]
    cache, prm, hp, bp = _build(lens, 8, 4, 0, seed=19, algo=1, meta=meta)
    _check(cache, prm, hp, bp, lens, 4, 0, seed=19)


@pytest.mark.parametrize("v_mode", [0, 1])
def test_compact_metadata_shared_prefix_kernel(v_mode):
    lens = [64 + 64 * 20 + 300, 64 + 64 * 20 + 700, 64 + 64 * 20 + 256]
    cache, prm, hp, bp = _build(lens, 2, 4, v_mode, seed=20, shared_prefix=64 + 64 * 20, algo=1, meta="u8")
    _check(cache, prm, hp, bp, lens, 4, v_mode, seed=20, shared_pages=20)


@pytest.mark.parametrize("algo", ALGOS)
def test_many_splits_ragged_tail(algo):
    # long enough for many splits and a partial last page
    lens = [64 + 64 * 150 + 37 + 256]
    cache, prm, hp, bp = _build(lens, 1, 4, 0, seed=15, algo=algo, max_splits=200)
    _check(cache, prm, hp, bp, lens, 4, 0, seed=15)


def test_bad_page_in_decode_reported():
    lens = [2000]
    cache, prm, hp, bp = _build(lens, 1, 4, 0, seed=16)
    hp_bad = hp.copy()
    hp_bad[0, 3] = -7
    q = queries(16, 0, 1, 4)
    cache.decode_attention(0, to_dev_bf16(q), np.array(lens, np.int32), hp_bad, bp, synth.sm_scale())
    assert cache.get_status() & osc.STATUS_BAD_PAGE
    # a sequence longer than its page table
    cache.decode_attention(0, to_dev_bf16(q), np.array([64 * 100], np.int32), hp, bp, synth.sm_scale())
    assert cache.get_status() & osc.STATUS_BAD_SEQLEN


def test_bf16_comparison_kernel():
    rng = np.random.default_rng(17)
    hkv, gq, B = 2, 4, 3
    lens = [1, 700, 3000]
    mp = (max(lens) + 63) // 64
    npages = sum((L + 63) // 64 for L in lens)
    perm = rng.permutation(npages).astype(np.int32)
    pt = np.zeros((B, mp), np.int32)
    pages = np.zeros((npages, hkv, 2, 64, 128), np.uint16)
    o = 0
    for r, L in enumerate(lens):
        n = (L + 63) // 64
        pt[r, :n] = perm[o:o + n]
        o += n
        k, v = tokens(17, 0, hkv, L, extra=r)
        for pos in range(L):
            pages[pt[r, pos // 64], :, 0, pos % 64] = synth.bf16_bits(k[pos])
            pages[pt[r, pos // 64], :, 1, pos % 64] = synth.bf16_bits(v[pos])
    q = queries(17, 0, hkv, gq, batch=B)
    ws = torch.zeros(osc.bf16_decode_workspace_bytes(B, hkv * gq, 32), dtype=torch.uint8, device=DEV)
    kv = torch.from_numpy(pages.view(np.int16)).to(DEV).view(torch.bfloat16)
    out = osc.bf16_decode(kv, to_dev_bf16(q), np.array(lens, np.int32), pt, synth.sm_scale(), hkv, ws, 32,
                          out_dtype=osc.OUT_FP32)
    got = out.double().cpu().numpy()
    for r, L in enumerate(lens):
        ref, _ = A.bf16_decode_request(q[r], L, pages, pt[r], synth.sm_scale())
        assert row_rel_err(got[r], ref).max() <= TOL
