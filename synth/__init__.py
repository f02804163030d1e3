"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers with fixed shapes and distributions. It
holds none of the method's arithmetic (no rotation, clipping, quantisation,
packing or attention), so both the CPU oracle and the CUDA library can be fed
from it without sharing any of the method's code.

The recipe follows the Qwen3-shaped workloads described for OSCAR:

* K and V tokens: i.i.d. N(0, 1) per channel, with ``n_outliers`` (default 4)
  fixed outlier channels scaled by 16, the channel indices drawn once per
  (layer, kv-head). Values are rounded to bfloat16 (round-to-nearest-even),
  which is the cache's storage type.
* Queries: q ~ N(0, Sigma_Q) with Sigma_Q = B diag(0.9**i) B^T, i = 0..d-1, B a
  random orthonormal basis (QR of a Gaussian with the sign of R's diagonal
  folded in) drawn per (layer, kv-head); the query heads of one GQA group share
  Sigma_Q. Queries are rounded to bfloat16.
* Calibration: 512 queries and 512 K/V tokens per (layer, kv-head), drawn from
  the same distributions but independently of the decode data.
* sm_scale = 1/sqrt(d).

Seeds: one base seed; ``numpy.random.SeedSequence(seed).spawn`` gives one child
per (layer, kv-head) and stream kind, so every (layer, head) is reproducible on
its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import functools

import numpy as np

HEAD_DIM = 128
N_OUTLIERS = 4
OUTLIER_SCALE = 16.0
QUERY_DECAY = 0.9
N_CALIB = 512

# stream kinds for SeedSequence children
_KIND = {"basis": 0, "outliers": 1, "kv": 2, "q": 3, "calq": 4, "calkv": 5, "lens": 6}


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32/float64 values to the nearest bfloat16 (ties to even); return float32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    out = rounded.astype(np.uint32).view(np.float32)
    nan = np.isnan(f)
    if nan.any():
        out = out.copy()
        out[nan] = np.nan
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bfloat16-representable."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _rng(seed: int, layer: int, head: int, kind: str, extra: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence([seed, layer, head, _KIND[kind], extra])
    return np.random.default_rng(ss)


@dataclass(frozen=True)
class HeadStats:
    """Per-(layer, kv-head) distribution parameters."""
    basis: np.ndarray          # [d, d] orthonormal, columns are directions
    sqrt_eig: np.ndarray       # [d] square roots of Sigma_Q's eigenvalues
    outliers: np.ndarray       # [N_OUTLIERS] channel indices


@functools.lru_cache(maxsize=4096)
def head_stats(seed: int, layer: int, head: int, d: int = HEAD_DIM) -> HeadStats:
    g = _rng(seed, layer, head, "basis").standard_normal((d, d))
    qm, rm = np.linalg.qr(g)
    qm = qm * np.sign(np.diag(rm))[None, :]
    sq = np.sqrt(QUERY_DECAY ** np.arange(d, dtype=np.float64))
    outl = _rng(seed, layer, head, "outliers").choice(d, size=N_OUTLIERS, replace=False)
    return HeadStats(basis=qm, sqrt_eig=sq, outliers=np.sort(outl))


def kv_tokens(seed: int, layer: int, head: int, n: int, kind: str = "kv", extra: int = 0,
              d: int = HEAD_DIM) -> tuple[np.ndarray, np.ndarray]:
    """K and V for ``n`` tokens of one (layer, kv-head): two float32 [n, d] arrays of bf16 values."""
    st = head_stats(seed, layer, head, d)
    r = _rng(seed, layer, head, kind, extra)
    k = r.standard_normal((n, d))
    v = r.standard_normal((n, d))
    k[:, st.outliers] *= OUTLIER_SCALE
    v[:, st.outliers] *= OUTLIER_SCALE
    return bf16_round(k), bf16_round(v)


def queries(seed: int, layer: int, head: int, n: int, kind: str = "q", extra: int = 0,
            d: int = HEAD_DIM) -> np.ndarray:
    """``n`` queries for one KV head's GQA group: float32 [n, d] of bf16 values."""
    st = head_stats(seed, layer, head, d)
    z = _rng(seed, layer, head, kind, extra).standard_normal((n, d))
    q = (z * st.sqrt_eig[None, :]) @ st.basis.T
    return bf16_round(q)


def calibration(seed: int, layer: int, head: int, d: int = HEAD_DIM, n: int = N_CALIB):
    """Calibration set for one (layer, kv-head): (Q [n,d], K [n,d], V [n,d]) float32 of bf16 values."""
    qc = queries(seed, layer, head, n, kind="calq", d=d)
    kc, vc = kv_tokens(seed, layer, head, n, kind="calkv", d=d)
    return qc, kc, vc


def sm_scale(d: int = HEAD_DIM) -> float:
    return 1.0 / math.sqrt(d)


def seq_lens_uniform(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """Sequence lengths drawn uniformly from [lo, hi] (inclusive), int64 [batch]."""
    return _rng(seed, 0, 0, "lens").integers(lo, hi + 1, size=batch)


def torch_kv_tokens(n: int, n_heads: int, outliers: np.ndarray, generator, device, d: int = HEAD_DIM):
    """Large-config K/V drawn on a torch device: two bf16 tensors [n, n_heads, d].

    ``outliers`` is an int array [n_heads, N_OUTLIERS] of channel indices per head
    (from :func:`head_stats`). ``generator`` is a seeded ``torch.Generator`` on
    ``device``. Only random draws and a per-channel scale happen here.
    """
    import torch
    scale = torch.ones(n_heads, d, device=device, dtype=torch.float32)
    idx = torch.as_tensor(np.asarray(outliers, dtype=np.int64), device=device)
    scale.scatter_(1, idx, OUTLIER_SCALE)
    k = torch.randn(n, n_heads, d, generator=generator, device=device, dtype=torch.float32)
    v = torch.randn(n, n_heads, d, generator=generator, device=device, dtype=torch.float32)
    k.mul_(scale)
    v.mul_(scale)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)
