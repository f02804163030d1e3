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


def compare_int2_pools(got: P.PoolModel, ref: P.PoolModel, rows_written, tol_frac: float = 1e-3, params=None):
    """Compare history rows written by a GPU path that rotated on the device with
    the oracle's (fp64-rotated) rows.

    rows_written: iterable of (page, row). Codes and metadata must agree except
    where float32 rotation rounding moves a value across a rounding boundary: at
    most ``tol_frac`` of the dequantised values may differ, each by at most one
    quantisation step (plus a 1-ulp change of the fp16 scale/zero, or one grid step of
    the compact format's indices). ``params`` (HeadParams per kv head) is needed for
    the compact format.
    """
    geo = ref.geo
    by_page = {}
    for page, row in rows_written:
        by_page.setdefault(int(page), []).append(int(row))
    n_el = n_diff = 0
    for page, rows in by_page.items():
        rows = np.array(sorted(set(rows)))
        for h in range(geo.hkv):
            a = got.read_history(page, rows, h)
            b = ref.read_history(page, rows, h)
            prm = params[h] if params is not None else None
            for kind, (ca, sa, za), (cb, sb, zb) in ((0, (a[0], a[1], a[2]), (b[0], b[1], b[2])),
                                                     (1, (a[3], a[4], a[5]), (b[3], b[4], b[5]))):
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
                n_el += d.size
                n_diff += int(np.count_nonzero(d))
    assert n_el > 0
    assert n_diff <= tol_frac * n_el, f"{n_diff} of {n_el} dequantised values differ"
    return n_diff, n_el


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """max_i |o_i - ref_i| / max_i |ref_i| for each (request, q-head) row."""
    return np.abs(got - ref).max(axis=-1) / np.abs(ref).max(axis=-1)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 1e-38)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)
