"""Clip, per-token asymmetric INT2 quantiser, dequantiser and 2-bit packing.

Sources:
* Page B, "服务系统：混合精度缓存布局": on the write path every token is
  rotated, clipped to calibration-derived percentile thresholds, then quantised
  with per-token asymmetric INT2 over groups of G_K = 64 channels.
* Page A, "OSCAR 的设计思路": four 2-bit values are packed into one byte; the
  INT2 read path restores values from scale and zero point.

Readings taken where the pages are silent (each is listed in the design doc):
* Asymmetric INT2 with 4 levels: zero = group minimum (a float offset, not an
  integer zero point), scale = (max - min) / 3, code = round((y - zero)/scale)
  clamped to [0, 3], round half to even.
* Scale and zero are stored as IEEE fp16 (RNE, saturated to +-65504), and the
  codes are computed with the stored (fp16-rounded) scale and zero, so that the
  dequantised value is exactly zero' + scale' * code.
* A group whose stored scale is 0 gets all codes 0.
* The same per-token 64-channel grouping is used for V as for K.
* All of the above is evaluated in float32, one IEEE operation at a time,
  in the order written, so that a GPU implementation can reproduce the codes
  bit for bit.

Packing: channel j of a token goes to byte j // 4 at bits 2*(j % 4)
(little-endian within the byte). How tokens of one page are arranged in
memory is the pool's business (see ``oracle.pool``).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
FP16_MAX = 65504.0


def to_fp16_saturating(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 with round-to-nearest-even, finite values saturated to +-65504."""
    x = np.asarray(x, dtype=F32)
    sat = np.clip(x, F32(-FP16_MAX), F32(FP16_MAX))
    sat = np.where(np.isnan(x), x, sat)
    return sat.astype(np.float16)


def clip(x: np.ndarray, tau: np.ndarray) -> np.ndarray:
    """y = min(max(x, -tau), tau) in float32, tau per channel (broadcast over the last axis)."""
    x = np.asarray(x, dtype=F32)
    t = np.asarray(tau, dtype=F32)
    return np.minimum(np.maximum(x, -t), t)


def quantize_groups(y: np.ndarray, group: int):
    """Quantise clipped float32 values y [..., d] in groups of ``group`` consecutive channels.

    Returns (codes uint8 [..., d], scale fp16 [..., d/group], zero fp16 [..., d/group]).
    """
    y = np.asarray(y, dtype=F32)
    d = y.shape[-1]
    assert d % group == 0
    yg = y.reshape(y.shape[:-1] + (d // group, group))
    mn = yg.min(axis=-1)
    mx = yg.max(axis=-1)
    rng = (mx - mn).astype(F32)               # one fp32 subtraction
    s = (rng / F32(3.0)).astype(F32)          # one fp32 division
    s16 = to_fp16_saturating(s)
    z16 = to_fp16_saturating(mn)
    s32 = s16.astype(F32)[..., None]
    z32 = z16.astype(F32)[..., None]
    diff = (yg - z32).astype(F32)             # one fp32 subtraction
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (diff / s32).astype(F32)          # one fp32 division
    code = np.rint(t)                         # round half to even
    code = np.clip(code, 0.0, 3.0)
    code = np.where(s32 == 0, 0.0, code)
    code = np.nan_to_num(code, nan=0.0)
    return code.astype(np.uint8).reshape(y.shape), s16, z16


def quantize_token(x_rot: np.ndarray, tau: np.ndarray, group: int = 64):
    """Clip then quantise rotated float32 tokens x_rot [..., d]."""
    return quantize_groups(clip(x_rot, tau), group)


def dequantize(codes: np.ndarray, s16: np.ndarray, z16: np.ndarray, group: int = 64) -> np.ndarray:
    """xhat = zero' + scale' * code in fp64 (exact), per group of ``group`` channels."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    c = codes.astype(np.float64).reshape(codes.shape[:-1] + (d // group, group))
    s = np.asarray(s16, dtype=np.float16).astype(np.float64)[..., None]
    z = np.asarray(z16, dtype=np.float16).astype(np.float64)[..., None]
    return (z + s * c).reshape(codes.shape)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Pack 2-bit codes [..., d] into bytes [..., d/4]: channel j -> byte j//4, bits 2*(j%4)."""
    c = np.asarray(codes, dtype=np.uint8)
    d = c.shape[-1]
    c4 = c.reshape(c.shape[:-1] + (d // 4, 4)).astype(np.uint32)
    out = np.zeros(c4.shape[:-1], dtype=np.uint32)
    for i in range(4):
        out |= (c4[..., i] & 3) << (2 * i)
    return out.astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_codes`: bytes [..., d/4] -> codes [..., d]."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape + (4,), dtype=np.uint8)
    for i in range(4):
        out[..., i] = (p >> (2 * i)) & 3
    return out.reshape(p.shape[:-1] + (p.shape[-1] * 4,))
