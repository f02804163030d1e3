"""Clip, per-token asymmetric INT2 quantiser, dequantiser and 2-bit packing.

Sources:
* The MarkTechPost article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局": on the write path every token is
  rotated, clipped to calibration-derived percentile thresholds, then quantised
  with per-token asymmetric INT2 over groups of G_K = 64 channels.
* The news article "超越 TurboQuant…", section "OSCAR 的设计思路": four 2-bit values are packed into one byte; the
  INT2 read path restores values from scale and zero point.

Readings taken where the pages are silent:
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

Compact metadata (16 bits per group, the pages' 2.25 bits per history element; row f2 of the scope
table, a format of this library's choosing): the group's minimum and maximum are stored as 8-bit
indices on a fixed grid over [-T, T], T the group's largest clip threshold (every clipped value lies
within it). With step D = (2 T) / 255: mn8 = clamp(floor((mn + T) / D), 0, 255), mx8 = clamp(ceil((mx
+ T) / D), 0, 255), each operation of the two quotients rounded to float32 in the order written; the
dequantisation parameters are zero' = fl32(mn8 D - T) (one rounding of the exact value, a fused
multiply-add) and scale' = fl32((mx8 - mn8) E) with E = fl32(D / 3), and the codes are computed from
them exactly as in the fp16 format. Rounding mn down and mx up keeps [mn, mx] inside
[zero', zero' + 3 scale'] (up to float32 rounding), so |y - xhat| <= scale' / 2 still holds.

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


def _codes(yg: np.ndarray, s32: np.ndarray, z32: np.ndarray) -> np.ndarray:
    """code = clamp(rint((y - zero') / scale'), 0, 3), 0 where scale' == 0; float32 op by op."""
    diff = (yg - z32).astype(F32)             # one fp32 subtraction
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (diff / s32).astype(F32)          # one fp32 division
    code = np.clip(np.rint(t), 0.0, 3.0)      # round half to even
    code = np.where(s32 == 0, 0.0, code)
    return np.nan_to_num(code, nan=0.0)


def group_bounds(tau: np.ndarray, group: int) -> np.ndarray:
    """T per group of ``group`` consecutive channels: the largest clip threshold of the group (float32)."""
    t = np.asarray(tau, dtype=F32)
    return t.reshape(t.shape[:-1] + (t.shape[-1] // group, group)).max(axis=-1)


def u8_steps(T: np.ndarray):
    """(D, E) in float32 of the compact format: D = fl32(2T / 255), E = fl32(D / 3)."""
    T = np.asarray(T, dtype=F32)
    D = ((T + T).astype(F32) / F32(255.0)).astype(F32)
    return D, (D / F32(3.0)).astype(F32)


def u8_scale_zero(mn8: np.ndarray, mx8: np.ndarray, T: np.ndarray):
    """(scale', zero') in float32 of the compact format (T broadcast over leading axes):
    zero' = fl32(mn8 D - T), the exact value rounded once (mn8 D has at most 32 significant bits and
    lies within a factor 2 of T, so the fp64 difference is exact); scale' = fl32((mx8 - mn8) E)."""
    T = np.asarray(T, dtype=F32)
    D, E = u8_steps(T)
    a = np.asarray(mn8).astype(np.float64)
    b = np.asarray(mx8).astype(np.float64)
    z = (a * D.astype(np.float64) - T.astype(np.float64)).astype(F32)
    s = ((b - a).astype(F32) * E).astype(F32)
    return s, z


def quantize_groups_u8(y: np.ndarray, group: int, T: np.ndarray):
    """Quantise clipped float32 values y [..., d] with the compact (8 + 8 bit) metadata.

    T [d/group]: the groups' bounds (``group_bounds`` of the clip thresholds).
    Returns (codes uint8 [..., d], mn8 uint8 [..., d/group], mx8 uint8 [..., d/group]).
    """
    y = np.asarray(y, dtype=F32)
    d = y.shape[-1]
    assert d % group == 0
    yg = y.reshape(y.shape[:-1] + (d // group, group))
    mn = yg.min(axis=-1)
    mx = yg.max(axis=-1)
    T = np.broadcast_to(np.asarray(T, dtype=F32), mn.shape)
    D, _ = u8_steps(T)
    with np.errstate(divide="ignore", invalid="ignore"):
        lo = (((mn + T).astype(F32)) / D).astype(F32)
        hi = (((mx + T).astype(F32)) / D).astype(F32)
    mn8 = np.where(D > 0, np.clip(np.floor(np.nan_to_num(lo, nan=0.0)), 0, 255), 0).astype(np.uint8)
    mx8 = np.where(D > 0, np.clip(np.ceil(np.nan_to_num(hi, nan=0.0)), 0, 255), 0).astype(np.uint8)
    s, z = u8_scale_zero(mn8, mx8, T)
    code = _codes(yg, s[..., None], z[..., None])
    return code.astype(np.uint8).reshape(y.shape), mn8, mx8


def quantize_token(x_rot: np.ndarray, tau: np.ndarray, group: int = 64):
    """Clip then quantise rotated float32 tokens x_rot [..., d]."""
    return quantize_groups(clip(x_rot, tau), group)


def quantize_token_u8(x_rot: np.ndarray, tau: np.ndarray, group: int = 64):
    """Clip then quantise rotated float32 tokens x_rot [..., d] with the compact metadata."""
    return quantize_groups_u8(clip(x_rot, tau), group, group_bounds(tau, group))


def dequantize_sz(codes: np.ndarray, s: np.ndarray, z: np.ndarray, group: int = 64) -> np.ndarray:
    """xhat = zero + scale * code in fp64 for any float scale / zero per group of ``group`` channels."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    c = codes.astype(np.float64).reshape(codes.shape[:-1] + (d // group, group))
    sf = np.asarray(s).astype(np.float64)[..., None]
    zf = np.asarray(z).astype(np.float64)[..., None]
    return (zf + sf * c).reshape(codes.shape)


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
