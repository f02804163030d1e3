"""Exact decode attention over the mixed-precision cache, and the segmented merge (fp64).

Sources:
* The news article "超越 TurboQuant…", section "OSCAR 的设计思路": at decode time the cache is split into a BF16
  segment (sink and recent, handled by a BF16 kernel) and an INT2 segment
  (unpack, restore scale/zero, accumulate in floating point), and the two
  results are combined with an online-softmax merge.
* The MarkTechPost article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局": the INT2 read path dequantises and
  inverse-rotates before attention; the value rotation R_V may be absorbed
  offline into the projection weights so no online inverse rotation of V is
  needed.

What is computed here is the plain definition: one softmax over all L tokens
of the request, with

* BF16 tokens:    logit = sm_scale * q . k,           value = v as stored
* history tokens: logit = sm_scale * (q R_K) . khat,  value = vhat R_V^T (explicit
                  mode) or vhat (V-absorbed mode: the stored V, BF16 and INT2
                  alike, is already in the rotated basis, so is the output)

where khat, vhat are the dequantised history rows (rotated basis). Because R_K
is orthogonal, (q R_K) . khat = q . (khat R_K^T), which is the pages'
"inverse-rotate the key" form written on the query side.

GQA: query head i reads kv head i // (Hq / Hkv).
"""
from __future__ import annotations

import numpy as np

from . import pool as poolmod
from .rotation import composite_rotation


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float):
    """Textbook single-query attention: returns (o [d], lse) with lse = log sum exp(sm_scale q.k)."""
    logits = sm_scale * (np.asarray(k, np.float64) @ np.asarray(q, np.float64))
    m = logits.max()
    p = np.exp(logits - m)
    lsum = p.sum()
    return (p @ np.asarray(v, np.float64)) / lsum, m + np.log(lsum)


def segment_partial(logits: np.ndarray, v: np.ndarray):
    """Partial of one segment: (m, l, acc) with m = max logit, l = sum exp(logit - m),
    acc = sum exp(logit - m) v. An empty segment gives (-inf, 0, 0)."""
    v = np.asarray(v, np.float64)
    if logits.size == 0:
        return -np.inf, 0.0, np.zeros(v.shape[-1])
    m = float(np.max(logits))
    p = np.exp(logits - m)
    return m, float(p.sum()), p @ v


def merge_partials(parts):
    """Online-softmax (log-sum-exp) merge: M = max m_s, L = sum l_s e^(m_s - M),
    o = sum acc_s e^(m_s - M) / L; empty segments (m = -inf) contribute nothing.
    Returns (o, lse = M + log L)."""
    ms = [m for m, _, _ in parts if np.isfinite(m)]
    if not ms:
        raise ValueError("all segments empty")
    M = max(ms)
    lsum = 0.0
    acc = None
    for m, l, a in parts:
        if not np.isfinite(m):
            continue
        w = np.exp(m - M)
        lsum += l * w
        acc = a * w if acc is None else acc + a * w
    return acc / lsum, M + np.log(lsum)


def decode_request(q: np.ndarray, seq_len: int, pool: poolmod.PoolModel, hist_pt, bf16_pt, params,
                   v_absorbed: bool, sm_scale: float, kv_heads=None):
    """Decode attention of one request.

    q: [Hq, d] query (bf16 values as float); params: per-kv-head HeadParams with
    float32 U (R = U H P_br is formed in fp64 from them, i.e. the rotation as
    loaded). Returns (o [Hq, d], lse [Hq]) in fp64; rows of query heads whose kv
    head is not in ``kv_heads`` are left NaN.
    """
    geo = pool.geo
    hq = q.shape[0]
    gq = hq // geo.hkv
    kv_heads = list(range(geo.hkv)) if kv_heads is None else list(kv_heads)
    seg, kk, vv = poolmod.gather_request(pool, seq_len, hist_pt, bf16_pt, heads=kv_heads, params=params)
    hist = np.array([s == "history" for s in seg], dtype=bool)
    o = np.full((hq, geo.d), np.nan)
    lse = np.full(hq, np.nan)
    for j, hd in enumerate(kv_heads):
        rk = composite_rotation(np.asarray(params[hd].u_k, np.float64))
        vals = vv[:, j].copy()
        if not v_absorbed and hist.any():
            rv = composite_rotation(np.asarray(params[hd].u_v, np.float64))
            vals[hist] = vals[hist] @ rv.T
        for i in range(hd * gq, (hd + 1) * gq):
            qi = np.asarray(q[i], np.float64)
            logits = np.empty(seq_len)
            logits[~hist] = sm_scale * (kk[~hist, j] @ qi)
            logits[hist] = sm_scale * (kk[hist, j] @ (qi @ rk))
            m = logits.max()
            p = np.exp(logits - m)
            o[i] = (p @ vals) / p.sum()
            lse[i] = m + np.log(p.sum())
    return o, lse


def bf16_decode_request(q: np.ndarray, seq_len: int, kv_pages: np.ndarray, page_table, sm_scale: float,
                        page: int = 64):
    """Reference for the all-BF16 paged cache: kv_pages [n_pages, Hkv, 2, P, d] uint16 bf16 bits.

    Token pos lives in page ``page_table[pos // P]``, row ``pos % P``. Returns (o [Hq, d], lse [Hq]).
    """
    hkv = kv_pages.shape[1]
    hq = q.shape[0]
    gq = hq // hkv
    pos = np.arange(seq_len)
    pages = np.asarray(page_table)[pos // page]
    rows = pos % page
    o = np.empty((hq, kv_pages.shape[-1]))
    lse = np.empty(hq)
    for hd in range(hkv):
        k = poolmod.bits_to_f64(kv_pages[pages, hd, 0, rows])
        v = poolmod.bits_to_f64(kv_pages[pages, hd, 1, rows])
        for i in range(hd * gq, (hd + 1) * gq):
            o[i], lse[i] = softmax_attention(q[i], k, v, sm_scale)
    return o, lse
