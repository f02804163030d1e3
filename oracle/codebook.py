"""Lloyd-Max 4-level codebook variant of the INT2 history (test infrastructure: only the tests,
the smoke check and the bench's CPU baseline use this package).

Source: the news article "超越 TurboQuant…", section "总结与展望" (the project's latest code replaces the uniform 2-bit levels by a
stronger Lloyd-Max codebook inside the attention-aware rotation). The pages give no more than
that sentence, so everything below is this library's reading, stated in full:

* The 2-bit code still indexes 4 levels inside each group's [min, max] range, but the levels are
  a codebook c_0 <= c_1 <= c_2 <= c_3 on the normalised coordinate u = (y - min) / (max - min)
  in [0, 1] instead of the uniform {0, 1/3, 2/3, 1}. There is one codebook per (layer, kv head,
  K / V), shared by every token and group of that head.
* Calibration (Lloyd 1982 / Max 1960): the codebook minimises the mean squared error of u over
  the calibration rows' groups (rotated, clipped; groups with max = min are left out). Lloyd's
  iteration from the uniform levels: the thresholds are the midpoints between neighbouring
  levels, each level moves to the mean of the samples in its cell (u <= t_0 is cell 0,
  t_{i-1} < u <= t_i cell i, u > t_2 cell 3; an empty cell keeps its level), until no level
  moves by more than 1e-12 or after 1000 iterations.
* Storage: levels are stored as bytes k_i = rint(255 c_i) (sorted), so c_i = k_i / 255; the
  uniform quantiser is the codebook (0, 85, 170, 255). Per row and group the metadata are the
  fp16 range r' = fp16(max - min) and zero' = fp16(min) (RNE, saturating), in the same bytes as
  the fp16 scale / zero format.
* Encoding, float32 one operation at a time: t = (y - zero') / r'; thresholds
  theta_i = (k_i + k_{i+1}) / 510 (one float32 division); code = #{i : t > theta_i}, so a tie
  goes to the lower level; r' = 0 gives code 0.
* Decoding: xhat = zero' + r' * k_code / 255.
"""
from __future__ import annotations

import numpy as np

from .quant import F32, clip, to_fp16_saturating

UNIFORM = np.array([0, 85, 170, 255], dtype=np.uint8)


def normalised_samples(y: np.ndarray, group: int) -> np.ndarray:
    """u = (y - min) / (max - min) in fp64 for every value of every group with max > min."""
    y = np.asarray(y, dtype=np.float64)
    yg = y.reshape(-1, y.shape[-1] // group, group)
    mn = yg.min(axis=-1, keepdims=True)
    mx = yg.max(axis=-1, keepdims=True)
    keep = (mx > mn)[..., 0]
    u = (yg - mn) / np.where(mx > mn, mx - mn, 1.0)
    return u[keep].ravel()


def lloyd_max(u: np.ndarray, levels=None, max_iter: int = 1000, tol: float = 1e-12) -> np.ndarray:
    """Lloyd's iteration for a 4-level scalar quantiser of the samples u; returns fp64 levels."""
    u = np.sort(np.asarray(u, dtype=np.float64))
    c = np.array([0.0, 1 / 3, 2 / 3, 1.0]) if levels is None else np.asarray(levels, dtype=np.float64).copy()
    csum = np.concatenate([[0.0], np.cumsum(u)])
    for _ in range(max_iter):
        t = 0.5 * (c[:-1] + c[1:])
        # cell i holds u in (t_{i-1}, t_i]: boundaries by binary search on the sorted samples
        edges = np.concatenate([[0], np.searchsorted(u, t, side="right"), [len(u)]])
        new = c.copy()
        for i in range(4):
            a, b = edges[i], edges[i + 1]
            if b > a:
                new[i] = (csum[b] - csum[a]) / (b - a)
        done = np.max(np.abs(new - c)) <= tol
        c = new
        if done:
            break
    return c


def codebook_bytes(levels: np.ndarray) -> np.ndarray:
    """Stored codebook: k_i = rint(255 c_i) clamped to [0, 255], sorted."""
    k = np.clip(np.rint(255.0 * np.asarray(levels, dtype=np.float64)), 0, 255)
    return np.sort(k).astype(np.uint8)


def calibrate_codebook(x_rot: np.ndarray, tau: np.ndarray, group: int = 64) -> np.ndarray:
    """Codebook bytes of one (layer, kv head, kind) from rotated float32 calibration rows [n, d]."""
    return codebook_bytes(lloyd_max(normalised_samples(clip(x_rot, tau), group)))


def thresholds(kcb: np.ndarray) -> np.ndarray:
    """theta_i = (k_i + k_{i+1}) / 510 as float32 (one correctly rounded division)."""
    k = np.asarray(kcb).astype(F32)
    return ((k[:-1] + k[1:]).astype(F32) / F32(510.0)).astype(F32)


def quantize_groups(y: np.ndarray, group: int, kcb: np.ndarray):
    """Quantise clipped float32 values y [..., d] with codebook bytes kcb [4].

    Returns (codes uint8 [..., d], range fp16 [..., d/G], zero fp16 [..., d/G])."""
    y = np.asarray(y, dtype=F32)
    d = y.shape[-1]
    yg = y.reshape(y.shape[:-1] + (d // group, group))
    mn = yg.min(axis=-1)
    mx = yg.max(axis=-1)
    r16 = to_fp16_saturating((mx - mn).astype(F32))
    z16 = to_fp16_saturating(mn)
    r = r16.astype(F32)[..., None]
    z = z16.astype(F32)[..., None]
    diff = (yg - z).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (diff / r).astype(F32)
    th = thresholds(kcb)
    code = (t > th[0]).astype(np.uint8) + (t > th[1]) + (t > th[2])
    code = np.where(r == 0, 0, code).astype(np.uint8)
    return code.reshape(y.shape), r16, z16


def quantize_token(x_rot: np.ndarray, tau: np.ndarray, kcb: np.ndarray, group: int = 64):
    """Clip then quantise rotated float32 tokens x_rot [..., d] with the codebook."""
    return quantize_groups(clip(x_rot, tau), group, kcb)


def dequantize(codes: np.ndarray, r16: np.ndarray, z16: np.ndarray, kcb: np.ndarray, group: int = 64) -> np.ndarray:
    """xhat = zero' + range' * k_code / 255 in fp64, per group of ``group`` channels."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    lev = np.asarray(kcb).astype(np.float64)[codes.astype(np.int64)].reshape(codes.shape[:-1] + (d // group, group))
    r = np.asarray(r16, dtype=np.float16).astype(np.float64)[..., None]
    z = np.asarray(z16, dtype=np.float16).astype(np.float64)[..., None]
    return (z + r * lev / 255.0).reshape(codes.shape)
