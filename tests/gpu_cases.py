"""Helpers for the GPU parity tests: seeded caches built through the C ABI and
the oracle's view of the same inputs. Expected values always come from the
oracle; the device pool bytes are only ever the thing being checked (or, for
decode attention, the shared dequantised cache both sides attend over)."""
from __future__ import annotations

import numpy as np
import torch

import bit_kv_cache_decode_gb300 as osc
import synth
from oracle import codebook as CB
from oracle import pool as P
from oracle import rotation

DEV = torch.device("cuda:0")


def head_params(seed: int, layer: int, hkv: int) -> list[P.HeadParams]:
    out = []
    for h in range(hkv):
        qc, kc, vc = synth.calibration(seed, layer, h)
        cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
        out.append(P.HeadParams(cal["U_K"].astype(np.float32), cal["U_V"].astype(np.float32),
                                cal["tau_K"].astype(np.float32), cal["tau_V"].astype(np.float32)))
    return out


def with_codebooks(seed: int, layer: int, prm: list[P.HeadParams]) -> list[P.HeadParams]:
    """The heads' parameters with codebooks: K's from the oracle's Lloyd-Max calibration on the head's
    calibration keys, V's a fixed uneven one (so that a K / V mix-up shows)."""
    out = []
    for h, p in enumerate(prm):
        _, kc, _ = synth.calibration(seed, layer, h)
        cbk = CB.calibrate_codebook(P.rotated_f32(kc, p.u_k), p.tau_k)
        out.append(P.HeadParams(p.u_k, p.u_v, p.tau_k, p.tau_v, cbk, np.array([5, 90, 141, 240], np.uint8)))
    return out


def upload_params(cache: osc.OscarCache, layer: int, prm: list[P.HeadParams]):
    cache.set_rotation(layer, np.stack([p.u_k for p in prm]), np.stack([p.u_v for p in prm]),
                       np.stack([p.tau_k for p in prm]), np.stack([p.tau_v for p in prm]))
    if cache.cfg.meta_format == osc.META_CB:
        cache.set_codebook(layer, np.stack([p.cb_k for p in prm]), np.stack([p.cb_v for p in prm]))


META_NAMES = {osc.META_F16: "f16", osc.META_U8: "u8", osc.META_CB: "cb"}


def pool_from_device(cache: osc.OscarCache, layer: int) -> P.PoolModel:
    cfg = cache.cfg
    geo = P.PoolGeometry(hkv=cfg.num_kv_heads, meta_format=META_NAMES[cfg.meta_format])
    pm = P.PoolModel(geo, cfg.num_int2_pages, cfg.num_bf16_pages)
    torch.cuda.synchronize()
    pm.int2[:] = cache.int2_pages(layer).cpu().numpy()
    pm.bf16[:] = cache.bf16_pages(layer).cpu().numpy().view(np.uint16).reshape(pm.bf16.shape)
    return pm


def tokens(seed: int, layer: int, hkv: int, n: int, extra: int = 0):
    """K, V [n, hkv, 128] float32 holding bf16 values."""
    k = np.stack([synth.kv_tokens(seed, layer, h, n, extra=extra)[0] for h in range(hkv)], axis=1)
    v = np.stack([synth.kv_tokens(seed, layer, h, n, extra=extra)[1] for h in range(hkv)], axis=1)
    return k, v


def queries(seed: int, layer: int, hkv: int, gq: int, batch: int = 1, extra: int = 0):
    """q [batch, hkv*gq, 128] float32 of bf16 values; query head i belongs to kv head i // gq."""
    out = np.empty((batch, hkv * gq, 128), np.float32)
    for b in range(batch):
        for h in range(hkv):
            out[b, h * gq:(h + 1) * gq] = synth.queries(seed, layer, h, gq, extra=extra + 1000 * b)
    return out


def to_dev_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(DEV).to(torch.bfloat16)


# Write-path gates for a GPU path that rotates on the device (the rotation's float32
# result can differ from the oracle's fp64-then-float32 rotation in the last bits):
# * codes may differ only by one step, on at most CODE_FLIP_TOL of all codes: a value
#   within a rounding error of a rounding boundary;
# * the stored fp16 scale / zero (or compact-format index bytes) may differ by one unit
#   on at most META_FLIP_TOL of the stored fields: scale = fl32(max - min) / 3 and
#   zero = min are rounded to fp16's 11 significant bits, so an fp32 value carrying a
#   relative error of a few units of 2^-22 lands on the other side of an fp16 rounding
#   boundary with probability of a few times 2^-22 / 2^-11 = 2^-11 (about 5e-4) per
#   field; the gate allows 4e-3. The compact format's 8-bit index rounding flips less
#   often (a few times 2^-22 x 255 per field).
CODE_FLIP_TOL = 1e-4
META_FLIP_TOL = 4e-3
WRITE_PATH_RATES = []


def compare_int2_pools(got: P.PoolModel, ref: P.PoolModel, rows_written, code_tol: float = CODE_FLIP_TOL,
                       meta_tol: float = META_FLIP_TOL, params=None):
    """Compare history rows written by a GPU path that rotated on the device with
    the oracle's (fp64-rotated) rows.

    rows_written: iterable of (page, row). Codes and metadata must agree except
    where float32 rotation rounding moves a value across a rounding boundary:
    at most ``code_tol`` of the codes may differ and at most ``meta_tol`` of the
    stored scale / zero fields, and every dequantised value must stay within one
    quantisation step (plus a 1-ulp change of the fp16 scale/zero, or one grid step
    of the compact format's indices). ``params`` (HeadParams per kv head) is
    needed for the compact format. Returns (codes differing, codes, fields
    differing, fields) and records the rates in WRITE_PATH_RATES.
    """
    geo = ref.geo
    by_page = {}
    for page, row in rows_written:
        by_page.setdefault(int(page), []).append(int(row))
    n_codes = n_code_diff = n_meta = n_meta_diff = 0
    for page, rows in by_page.items():
        rows = np.array(sorted(set(rows)))
        for h in range(geo.hkv):
            a = got.read_history(page, rows, h)
            b = ref.read_history(page, rows, h)
            prm = params[h] if params is not None else None
            for kind, (ca, sa, za), (cb, sb, zb) in ((0, (a[0], a[1], a[2]), (b[0], b[1], b[2])),
                                                     (1, (a[3], a[4], a[5]), (b[3], b[4], b[5]))):
                n_codes += ca.size
                n_code_diff += int(np.count_nonzero(ca != cb))
                assert np.abs(ca.astype(np.int64) - cb.astype(np.int64)).max(initial=0) <= 1
                fa = np.stack([sa, za]).view(np.uint8).reshape(2, -1) if sa.dtype == np.uint8 else \
                    np.stack([sa, za]).view(np.uint16)
                fb = np.stack([sb, zb]).view(np.uint8).reshape(2, -1) if sb.dtype == np.uint8 else \
                    np.stack([sb, zb]).view(np.uint16)
                n_meta += fa.size
                n_meta_diff += int(np.count_nonzero(fa != fb))
                xa = P.dequant_rows(ca, sa, za, prm, kind, geo)
                xb = P.dequant_rows(cb, sb, zb, prm, kind, geo)
                if geo.meta_format == "cb":          # one step = the widest gap between neighbouring levels
                    lev = (prm.cb_k if kind == 0 else prm.cb_v).astype(np.float64)
                    sa = sa.astype(np.float64) * max(np.diff(lev).max(), lev[0], 255 - lev[3]) / 255.0
                    sb = sb.astype(np.float64) * max(np.diff(lev).max(), lev[0], 255 - lev[3]) / 255.0
                else:
                    tau = None if prm is None else (prm.tau_k if kind == 0 else prm.tau_v)
                    sa = P.dequant_params(sa, za, tau, geo)[0]
                    sb = P.dequant_params(sb, zb, tau, geo)[0]
                step = np.maximum(sa, sb).astype(np.float64).repeat(64, 1)
                d = np.abs(xa - xb)
                assert np.all(d <= 1.01 * step + 2e-3 * np.abs(xb) + 1e-6), (page, h, d.max())
    assert n_codes > 0
    WRITE_PATH_RATES.append((n_code_diff, n_codes, n_meta_diff, n_meta))
    print(f"write path vs oracle: {n_code_diff} of {n_codes} codes differ ({n_code_diff / n_codes:.2e}), "
          f"{n_meta_diff} of {n_meta} metadata fields differ ({n_meta_diff / n_meta:.2e})")
    assert n_code_diff <= code_tol * n_codes, f"{n_code_diff} of {n_codes} codes differ"
    assert n_meta_diff <= meta_tol * n_meta, f"{n_meta_diff} of {n_meta} metadata fields differ"
    return n_code_diff, n_codes, n_meta_diff, n_meta


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """max_i |o_i - ref_i| / max_i |ref_i| for each (request, q-head) row."""
    return np.abs(got - ref).max(axis=-1) / np.abs(ref).max(axis=-1)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 1e-38)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def build_decode_case(lens, hkv, gq, v_mode, seed, shared_prefix=0, algo=0, max_splits=64, meta="f16",
                      kv_hook=None):
    """Prefill B requests on the GPU. With shared_prefix > 0 all requests share their first
    `shared_prefix` tokens (sink page and the history pages covering them). kv_hook(r, k, v), if given,
    may edit request r's K and V [L, hkv, 128] (bf16 values) in place before the prefill."""
    B = len(lens)
    nh = [max(0, (L - 320 + 63) // 64) for L in lens]
    mhp = max(1, max(nh))
    shp = (shared_prefix - 64) // 64 if shared_prefix else 0           # shared history pages
    n_int2 = shp + sum(n - shp for n in nh) + 1
    n_bf16 = 1 + 4 * B if shared_prefix else 5 * B
    rng = np.random.default_rng(seed)
    perm_i, perm_b = rng.permutation(n_int2).astype(np.int32), rng.permutation(n_bf16).astype(np.int32)
    hist_pt = np.full((B, mhp), -1, np.int32)
    bf16_pt = np.zeros((B, 5), np.int32)
    oi, ob = shp, (1 if shared_prefix else 0)
    for r in range(B):
        hist_pt[r, :shp] = perm_i[:shp]
        hist_pt[r, shp:nh[r]] = perm_i[oi:oi + nh[r] - shp]
        oi += nh[r] - shp
        if shared_prefix:
            bf16_pt[r, 0] = perm_b[0]
            bf16_pt[r, 1:] = perm_b[ob:ob + 4]
            ob += 4
        else:
            bf16_pt[r] = perm_b[ob:ob + 5]
            ob += 5
    cfg = osc.CacheConfig(num_layers=1, num_kv_heads=hkv, num_q_heads=hkv * gq, num_int2_pages=n_int2,
                          num_bf16_pages=n_bf16, max_batch=B, max_splits=max_splits, v_mode=v_mode,
                          meta_format={"f16": 0, "u8": 1, "cb": 2}[meta])
    cache = osc.OscarCache(cfg, device=DEV)
    cache.set_decode_algo(algo)
    prm = head_params(seed, 0, hkv)
    if meta == "cb":
        prm = with_codebooks(seed, 0, prm)
    upload_params(cache, 0, prm)
    ks, vs = [], []
    for r, L in enumerate(lens):
        k, v = tokens(seed, 0, hkv, L, extra=r + 1)
        if shared_prefix:
            k0, v0 = tokens(seed, 0, hkv, shared_prefix, extra=0)
            k[:shared_prefix], v[:shared_prefix] = k0, v0
        if kv_hook is not None:
            kv_hook(r, k, v)
        ks.append(k)
        vs.append(v)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cache.quantize_prefill(0, to_dev_bf16(np.concatenate(ks)), to_dev_bf16(np.concatenate(vs)), cu, hist_pt, bf16_pt)
    assert cache.get_status() == 0
    return cache, prm, hist_pt, bf16_pt
