"""Byte-exact model of the paged mixed-precision token pool.

Sources:
* The news article "超越 TurboQuant…", section "OSCAR 的设计思路": one token pool per request laid out as
  BF16 sink (64 tokens) | INT2 history | BF16 recent (256 tokens); a new token
  is written into the recent window and, as decoding proceeds, the oldest
  recent token is rotated, clipped, quantised, packed and demoted into the INT2
  history; the pool stays compatible with paged KV and prefix caching.
* The MarkTechPost article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局": sink = first S0 = 64 tokens, recent =
  the last W = 256 tokens before the current position, history = everything
  in between, stored as INT2 after rotation and clipping.

The placement contract and byte layout below are this library's own format
(the pages fix only the three regions, 4 codes per byte and the group size);
they are stated here independently of the CUDA sources.

Placement of the token at position ``pos`` of a request whose sequence length
is ``L`` (the token count after the newest append):

* sink,    pos < S0:                 bf16 page ``bf16_pt[pos // P]``, row ``pos % P``
* recent,  pos >= max(S0, L - W):    slot = (pos - S0) % W,
                                     bf16 page ``bf16_pt[S0 // P + slot // P]``, row ``slot % P``
* history, S0 <= pos < L - W:        h = pos - S0,
                                     INT2 page ``hist_pt[h // P]``, row ``h % P``

INT2 page block, one per (page, kv-head), ``block_bytes = P*d/2 + P*(d/G)*8``
bytes (5120 for P = 64, d = 128, G = 64), in this order:

1. K codes, token-major: row t occupies bytes [t*d/4, (t+1)*d/4), the token's
   codes packed with channel j in byte j//4 at bits 2*(j%4).
2. V codes, channel-major: channel c occupies the 16 bytes (P = 64) of slot
   c ^ ((c >> 4) & 7) of the region. Its 4 little-endian 32-bit words hold the
   64 rows: row t sits in word (t >> 1) & 3 at bit 16 (t & 1) + 4 (t >> 4) +
   2 ((t >> 3) & 1). So word w holds the rows t with t % 16 in
   {2w, 2w+1, 2w+8, 2w+9}, even rows in its low half and odd rows in its high
   half, each row next to its odd (even) partner.
3. K metadata: row t at t*(d/G)*m, m = 4 (fp16 format, the default): for each
   group g, fp16 scale then fp16 zero; m = 2 (compact u8 format): for each group
   g, the byte mn8 then the byte mx8 (see ``quant``: indices on the group's grid
   over [-T, T]); the block is then 4608 bytes.
4. V metadata: same layout.

BF16 page block, one per (page, kv-head): K [P][d] bf16 then V [P][d] bf16.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import codebook, quant


@dataclass(frozen=True)
class PoolGeometry:
    hkv: int
    d: int = 128
    group: int = 64
    page: int = 64
    sink: int = 64
    recent: int = 256
    # "f16": fp16 (scale, zero); "u8": 8-bit (mn8, mx8) on [-T, T]; "cb": fp16 (range, zero) with a
    # Lloyd-Max codebook per (kv head, kind) (see ``codebook``)
    meta_format: str = "f16"

    @property
    def meta_per_group(self) -> int:   # metadata bytes per group of one row
        return {"f16": 4, "u8": 2, "cb": 4}[self.meta_format]

    @property
    def codes_bytes(self) -> int:      # K (or V) codes per page block
        return self.page * self.d // 4

    @property
    def meta_bytes(self) -> int:       # K (or V) metadata per page block
        return self.page * (self.d // self.group) * self.meta_per_group

    @property
    def block_bytes(self) -> int:
        return 2 * self.codes_bytes + 2 * self.meta_bytes

    @property
    def bf16_pages_per_request(self) -> int:
        return (self.sink + self.recent) // self.page


def segment_of(pos: int, seq_len: int, geo: PoolGeometry) -> str:
    if pos < geo.sink:
        return "sink"
    if pos >= max(geo.sink, seq_len - geo.recent):
        return "recent"
    return "history"


def history_len(seq_len: int, geo: PoolGeometry) -> int:
    return max(0, seq_len - geo.sink - geo.recent)


class PoolModel:
    """Expected contents of one layer's INT2 and BF16 page pools."""

    def __init__(self, geo: PoolGeometry, n_int2_pages: int, n_bf16_pages: int):
        self.geo = geo
        self.int2 = np.zeros((n_int2_pages, geo.hkv, geo.block_bytes), dtype=np.uint8)
        self.bf16 = np.zeros((n_bf16_pages, geo.hkv, 2, geo.page, geo.d), dtype=np.uint16)

    # ---- INT2 page block accessors (vectorised over rows of one page) -------------
    def _k_byte_index(self, rows: np.ndarray) -> np.ndarray:
        """[n, d/4] byte offsets (within the block) of rows' packed K bytes."""
        g = self.geo
        return rows[:, None] * (g.d // 4) + np.arange(g.d // 4)[None, :]

    def _v_field(self, rows: np.ndarray):
        """([n, d] byte offsets within the block, [n, d] bit shifts within the byte) of rows' V codes."""
        g = self.geo
        assert g.page == 64, "the V word layout is defined for 64-row pages"
        c = np.arange(g.d)[None, :]
        t = rows[:, None].astype(np.int64)
        slot = c ^ ((c >> 4) & 7)
        word = (t >> 1) & 3
        bit = 16 * (t & 1) + 4 * (t >> 4) + 2 * ((t >> 3) & 1)
        return g.codes_bytes + slot * (g.page // 4) + 4 * word + bit // 8 + 0 * c, bit % 8 + 0 * c

    def _write_v_codes(self, blk: np.ndarray, rows: np.ndarray, codes: np.ndarray):
        """Set the 2-bit V fields of rows (codes [n, d] in 0..3), leaving the other rows' bits."""
        idx, sh = self._v_field(rows)
        for i in range(len(rows)):               # rows in order: a later write of a row wins
            keep = blk[idx[i]] & ~(np.uint8(3) << sh[i].astype(np.uint8))
            blk[idx[i]] = keep | (codes[i].astype(np.uint8) << sh[i].astype(np.uint8))

    def _read_v_codes(self, blk: np.ndarray, rows: np.ndarray) -> np.ndarray:
        idx, sh = self._v_field(rows)
        return ((blk[idx] >> sh.astype(np.uint8)) & 3).astype(np.uint8)

    def _meta_index(self, rows: np.ndarray, which: int) -> np.ndarray:
        """[n, (d/G)*m] byte offsets of rows' metadata; which = 0 for K, 1 for V."""
        g = self.geo
        per = (g.d // g.group) * g.meta_per_group
        base = 2 * g.codes_bytes + which * g.meta_bytes
        return base + rows[:, None] * per + np.arange(per)[None, :]

    def _meta_dtype(self):
        return np.uint8 if self.geo.meta_format == "u8" else np.float16

    def _meta_bytes(self, a, b) -> np.ndarray:
        """Interleave the two stored metadata fields of each group: (scale, zero) or (mn8, mx8)."""
        a = np.asarray(a, dtype=self._meta_dtype())
        b = np.asarray(b, dtype=self._meta_dtype())
        ab = np.empty(a.shape[:-1] + (2 * a.shape[-1],), dtype=a.dtype)
        ab[..., 0::2] = a
        ab[..., 1::2] = b
        return np.ascontiguousarray(ab).view(np.uint8)

    def write_history(self, page: int, rows, head: int, k_pack, k_s, k_z, v_pack, v_s, v_z):
        """Write rows (int array [n]) of one (page, head): packed codes [n, d/4] and the stored
        metadata [n, d/G]: fp16 scale / zero, or u8 mn8 / mx8 in the compact format."""
        rows = np.atleast_1d(np.asarray(rows, dtype=np.int64))
        blk = self.int2[page, head]
        blk[self._k_byte_index(rows)] = np.asarray(k_pack).reshape(len(rows), -1)
        self._write_v_codes(blk, rows, quant.unpack_codes(np.asarray(v_pack).reshape(len(rows), -1)))
        blk[self._meta_index(rows, 0)] = self._meta_bytes(np.reshape(k_s, (len(rows), -1)), np.reshape(k_z, (len(rows), -1)))
        blk[self._meta_index(rows, 1)] = self._meta_bytes(np.reshape(v_s, (len(rows), -1)), np.reshape(v_z, (len(rows), -1)))

    def read_history(self, page: int, rows, head: int):
        """(k_codes [n,d], k_s, k_z [n,d/G], v_codes, v_s, v_z) of rows of one (page, head); the
        metadata as stored (fp16 scale / zero, or u8 mn8 / mx8)."""
        rows = np.atleast_1d(np.asarray(rows, dtype=np.int64))
        blk = self.int2[page, head]
        kc = quant.unpack_codes(blk[self._k_byte_index(rows)])
        vc = self._read_v_codes(blk, rows)
        out = []
        for which in (0, 1):
            sz = np.ascontiguousarray(blk[self._meta_index(rows, which)]).view(self._meta_dtype())
            out.append((sz[:, 0::2].copy(), sz[:, 1::2].copy()))
        return kc, out[0][0], out[0][1], vc, out[1][0], out[1][1]

    # ---- BF16 page block accessors -------------------------------------------------
    def write_bf16(self, page: int, rows, head: int, k_bits, v_bits):
        self.bf16[page, head, 0, rows] = k_bits
        self.bf16[page, head, 1, rows] = v_bits

    def read_bf16(self, page: int, rows, head: int):
        return self.bf16[page, head, 0, rows].copy(), self.bf16[page, head, 1, rows].copy()


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16-representable float32 values -> their uint16 bit patterns (no rounding)."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@dataclass
class HeadParams:
    """Rotation and clip parameters of one (layer, kv-head), as loaded (float32)."""
    u_k: np.ndarray      # [d, d] float32, eigenvector columns
    u_v: np.ndarray      # [d, d] float32 (ignored when V is absorbed)
    tau_k: np.ndarray    # [d] float32, rotated basis
    tau_v: np.ndarray    # [d] float32
    cb_k: np.ndarray | None = None   # codebook bytes [4] (the "cb" metadata format)
    cb_v: np.ndarray | None = None


def rotated_f32(x: np.ndarray, u32: np.ndarray) -> np.ndarray:
    """The write path's rotated values: x (U H P_br) in fp64 from the float32 U, rounded to float32.

    x may be [d] or [n, d]."""
    from .rotation import composite_rotation
    r = composite_rotation(np.asarray(u32, dtype=np.float64))
    return (np.asarray(x, dtype=np.float64) @ r).astype(np.float32)


def quantize_history_tokens(k_f32, v_f32, prm: HeadParams, v_absorbed: bool, group: int,
                            meta_format: str = "f16"):
    """Rotate (K always; V unless absorbed), clip, quantise and pack tokens [n, d] of one head.

    Returns (k_pack, k_a, k_b, v_pack, v_a, v_b), (a, b) the stored metadata of the format."""
    kr = rotated_f32(k_f32, prm.u_k)
    vr = np.asarray(v_f32, dtype=np.float32) if v_absorbed else rotated_f32(v_f32, prm.u_v)
    if meta_format == "cb":
        kc, ks, kz = codebook.quantize_token(kr, prm.tau_k, prm.cb_k, group)
        vc, vs, vz = codebook.quantize_token(vr, prm.tau_v, prm.cb_v, group)
    else:
        qt = quant.quantize_token if meta_format == "f16" else quant.quantize_token_u8
        kc, ks, kz = qt(kr, prm.tau_k, group)
        vc, vs, vz = qt(vr, prm.tau_v, group)
    return quant.pack_codes(kc), ks, kz, quant.pack_codes(vc), vs, vz


def dequant_params(a, b, tau, geo: PoolGeometry):
    """Float (scale, zero) per group from the stored metadata (a, b) of the "f16" or "u8" format."""
    if geo.meta_format == "f16":
        return np.asarray(a, dtype=np.float16), np.asarray(b, dtype=np.float16)
    assert geo.meta_format == "u8"
    return quant.u8_scale_zero(a, b, quant.group_bounds(tau, geo.group))


def dequant_rows(codes, a, b, prm, kind: int, geo: PoolGeometry) -> np.ndarray:
    """Dequantised fp64 rows [n, d] of one kind (0 K, 1 V) from codes and stored metadata."""
    if geo.meta_format == "cb":
        return codebook.dequantize(codes, a, b, prm.cb_k if kind == 0 else prm.cb_v, geo.group)
    tau = None if prm is None else (prm.tau_k if kind == 0 else prm.tau_v)
    return quant.dequantize_sz(codes, *dequant_params(a, b, tau, geo), geo.group)


def bf16_location(pos: int, seg: str, bf16_pt, geo: PoolGeometry):
    """(page, row) of a sink or recent position under the placement contract."""
    if seg == "sink":
        return int(bf16_pt[pos // geo.page]), pos % geo.page
    slot = (pos - geo.sink) % geo.recent
    return int(bf16_pt[geo.sink // geo.page + slot // geo.page]), slot % geo.page


def place(pool: PoolModel, pos: int, seq_len: int, head: int, k_f32, v_f32, prm: HeadParams,
          v_absorbed: bool, hist_pt, bf16_pt):
    """Write token ``pos`` of a request with length ``seq_len`` where the contract puts it."""
    geo = pool.geo
    seg = segment_of(pos, seq_len, geo)
    if seg == "history":
        h = pos - geo.sink
        pk = quantize_history_tokens(np.asarray(k_f32)[None], np.asarray(v_f32)[None], prm, v_absorbed, geo.group,
                                     geo.meta_format)
        pool.write_history(int(hist_pt[h // geo.page]), [h % geo.page], head, *pk)
        return
    page, row = bf16_location(pos, seg, bf16_pt, geo)
    pool.write_bf16(page, row, head, f32_to_bf16_bits(k_f32), f32_to_bf16_bits(v_f32))


def prefill(pool: PoolModel, k, v, hist_pt, bf16_pt, params, v_absorbed: bool):
    """Bulk write of one request's tokens k, v [L, Hkv, d] (bf16 values as float32).

    Equivalent to calling :func:`place` for every position with seq_len = L;
    history tokens are quantised in one batch per head and written page by page.
    """
    geo = pool.geo
    L = k.shape[0]
    lh = history_len(L, geo)
    for hd in range(geo.hkv):
        if lh > 0:
            pk = quantize_history_tokens(k[geo.sink: geo.sink + lh, hd], v[geo.sink: geo.sink + lh, hd],
                                         params[hd], v_absorbed, geo.group, geo.meta_format)
            for i in range((lh + geo.page - 1) // geo.page):
                a, b = i * geo.page, min((i + 1) * geo.page, lh)
                pool.write_history(int(hist_pt[i]), np.arange(b - a), hd, *(x[a:b] for x in pk))
        for pos in list(range(min(L, geo.sink))) + list(range(max(geo.sink, L - geo.recent), L)):
            page, row = bf16_location(pos, segment_of(pos, L, geo), bf16_pt, geo)
            pool.write_bf16(page, row, hd, f32_to_bf16_bits(k[pos, hd]), f32_to_bf16_bits(v[pos, hd]))


def append(pool: PoolModel, k_new, v_new, seq_len_before: int, hist_pt, bf16_pt, params, v_absorbed: bool):
    """Append one token (k_new, v_new [Hkv, d]) at position ``seq_len_before``.

    If the recent window is full, the oldest recent token (position
    seq_len_before - W) is read back from its BF16 slot, quantised into the
    history, and only then is its slot overwritten by the new token.
    """
    geo = pool.geo
    L_old = seq_len_before
    if L_old >= geo.sink + geo.recent:
        old = L_old - geo.recent
        page, row = bf16_location(old, "recent", bf16_pt, geo)
        h = old - geo.sink
        for hd in range(geo.hkv):
            kb, vb = pool.read_bf16(page, row, hd)
            pk = quantize_history_tokens(bits_to_f64(kb)[None].astype(np.float32),
                                         bits_to_f64(vb)[None].astype(np.float32), params[hd], v_absorbed, geo.group,
                                         geo.meta_format)
            pool.write_history(int(hist_pt[h // geo.page]), [h % geo.page], hd, *pk)
    for hd in range(geo.hkv):
        place(pool, L_old, L_old + 1, hd, k_new[hd], v_new[hd], params[hd], v_absorbed, hist_pt, bf16_pt)


def gather_request(pool: PoolModel, seq_len: int, hist_pt, bf16_pt, heads=None, params=None):
    """Decode one request's cache from the pool bytes.

    Returns (seg, k, v): seg is a list of segment names per position; k, v are
    [L, n_heads, d] fp64 arrays where BF16 rows hold the stored bf16 values and
    history rows hold the dequantised values (rotated basis). ``heads`` selects
    kv heads (default: all). ``params`` (the heads' HeadParams, indexed by kv head) is required
    by the compact metadata format, whose grid depends on the clip thresholds.
    """
    geo = pool.geo
    heads = list(range(geo.hkv)) if heads is None else list(heads)
    if geo.meta_format != "f16" and params is None:
        raise ValueError("the compact and codebook metadata formats need the heads' parameters")
    L = seq_len
    kk = np.zeros((L, len(heads), geo.d))
    vv = np.zeros((L, len(heads), geo.d))
    seg = [segment_of(pos, L, geo) for pos in range(L)]
    lh = history_len(L, geo)
    for j, hd in enumerate(heads):
        for i in range((lh + geo.page - 1) // geo.page):
            a, b = i * geo.page, min((i + 1) * geo.page, lh)
            kc, ka, kb, vc, va, vb = pool.read_history(int(hist_pt[i]), np.arange(b - a), hd)
            prm = params[hd] if params is not None else None
            kk[geo.sink + a: geo.sink + b, j] = dequant_rows(kc, ka, kb, prm, 0, geo)
            vv[geo.sink + a: geo.sink + b, j] = dequant_rows(vc, va, vb, prm, 1, geo)
        for pos in range(L):
            if seg[pos] != "history":
                page, row = bf16_location(pos, seg[pos], bf16_pt, geo)
                kb, vb = pool.read_bf16(page, row, hd)
                kk[pos, j] = bits_to_f64(kb)
                vv[pos, j] = bits_to_f64(vb)
    return seg, kk, vv
