"""K / V projection in front of the write path (test infrastructure only).

Source: the MarkTechPost article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局":
the write path (rotate, clip, quantise, pack) runs fused with the kernel that produces the tokens' K
and V, so the prompt's K and V need not be written out and read back before they are quantised. The
page names neither the projection's form nor its precision. Reading taken here: the
plainest one, a linear layer without bias, the way a transformer's K and V projections store their
weights:

    K = x W_k^T,  V = x W_v^T,   x [T, d_model],  W [Hkv * 128, d_model],

with output column j belonging to kv head j // 128, channel j % 128. The model emits K and V in
bf16, so each element of the product is rounded once, to nearest with ties to even, to bf16. The
write path then places and quantises those bf16 rows exactly as ``pool.prefill`` does with given
K and V.

The products of bf16 values are exact in float64 and the sums are taken in float64; a sum then
differs from the exact value by far less than half a bf16 ulp, except within about 2^-40 of a
rounding midpoint.
"""
from __future__ import annotations

import numpy as np

from . import pool as P


def round_to_bf16(y: np.ndarray) -> np.ndarray:
    """float64 -> the nearest bf16 value (8 significant bits, ties to even), as float64.

    Values beyond the largest finite bf16 become +-inf; the result of a value in the bf16 subnormal
    range is rounded on that range's fixed grid of 2^-133.
    """
    y = np.asarray(y, dtype=np.float64)
    out = np.zeros_like(y)
    nz = (y != 0) & np.isfinite(y)
    m, e = np.frexp(y[nz])                       # y = m 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                      # below 2^-126 the grid stops shrinking (subnormals)
    q = np.rint(np.ldexp(y[nz], 8 - e))          # 8 significant bits at exponent e; rint ties to even
    out[nz] = np.ldexp(q, e - 8)
    out[~np.isfinite(y)] = y[~np.isfinite(y)]
    big = np.abs(out) > 3.3895313892515355e38    # the largest finite bf16
    out[big] = np.sign(out[big]) * np.inf
    return out


def project(x: np.ndarray, w: np.ndarray, hkv: int) -> np.ndarray:
    """bf16(x W^T) as float32, shaped [T, hkv, 128]. x [T, d_model] and w [hkv*128, d_model] hold
    bf16 values (as any float dtype)."""
    x64 = np.asarray(x, dtype=np.float64)
    w64 = np.asarray(w, dtype=np.float64)
    y = x64 @ w64.T
    return round_to_bf16(y).astype(np.float32).reshape(x64.shape[0], hkv, 128)


def project_prefill(pool: P.PoolModel, x, w_k, w_v, hist_pt, bf16_pt, params, v_absorbed: bool):
    """One request's prompt from its hidden states: K and V by ``project``, then ``pool.prefill``."""
    hkv = pool.geo.hkv
    P.prefill(pool, project(x, w_k, hkv), project(x, w_v, hkv), hist_pt, bf16_pt, params, v_absorbed)
