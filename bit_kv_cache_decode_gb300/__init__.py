"""Python binding of the OSCAR INT2 KV-cache library (liboscar.so, CUDA sm_103a).

Argument marshalling only: every step of the write and decode paths runs in
the library's CUDA kernels. PyTorch supplies device memory and the current
stream. If the compiled library is missing, importing the binding raises; there
is no fallback.

The C entry points, layouts and error behaviour are documented in
``include/oscar.h``; the names here follow them.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "liboscar.so")

OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_STATUS, ERR_TIMEOUT, ERR_NOT_ORTHOGONAL = -1, -2, -3, -4, -5, -6
ERR_TOO_LARGE = -7
STATUS_BAD_PAGE, STATUS_BAD_SEQLEN, STATUS_TIMEOUT, STATUS_NONFINITE, STATUS_SATURATED = 1, 2, 4, 8, 16
V_ABSORBED, V_EXPLICIT = 0, 1
OUT_BF16, OUT_FP32 = 0, 1
KIND_K, KIND_V = 0, 1
DECODE_SIMT, DECODE_MMA, DECODE_TC = 0, 1, 2
META_F16, META_U8, META_CB = 0, 1, 2

# every symbol include/oscar.h declares
EXPORTS = (
    "oscar_cache_bytes", "oscar_cache_create", "oscar_cache_destroy", "oscar_layer_offsets", "oscar_set_rotation",
    "oscar_quantize_prefill", "oscar_project_quantize_prefill", "oscar_append_kv", "oscar_decode_attention", "oscar_set_decode_algo",
    "oscar_get_status", "oscar_pack_rotated", "oscar_rotate", "oscar_bf16_decode_workspace_bytes",
    "oscar_bf16_decode", "oscar_calibrate", "oscar_profile_begin", "oscar_profile_read", "oscar_error_string",
    "oscar_decode_attention_noalloc", "oscar_trace_ctas", "oscar_decode_step",
    "oscar_decode_attention_shared", "oscar_decode_step_shared",
    "oscar_trace_timeline", "oscar_check_wait_timeout", "oscar_set_codebook", "oscar_calibrate_codebook",
)


class OscarError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_lib.oscar_error_string(code).decode()} ({code})")


class Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_layers", "num_kv_heads", "num_q_heads", "head_dim", "group", "page_size", "sink", "recent",
        "num_int2_pages", "num_bf16_pages", "v_mode", "max_batch", "max_splits", "meta_format")]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"OSCAR CUDA library not built ({LIB_PATH} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32p, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)
    c_int, c_float = ctypes.c_int, ctypes.c_float
    sig = {
        "oscar_cache_bytes": [ctypes.POINTER(Layout), sz, sz],
        "oscar_cache_create": [ctypes.POINTER(Layout), vp, vp, ctypes.POINTER(vp)],
        "oscar_cache_destroy": [vp],
        "oscar_layer_offsets": [vp, c_int, sz, sz, sz],
        "oscar_set_rotation": [vp, c_int, vp, vp, vp, vp, vp],
        "oscar_set_codebook": [vp, c_int, vp, vp, vp],
        "oscar_calibrate_codebook": [vp, c_int, vp, vp],
        "oscar_quantize_prefill": [vp, c_int, c_int, vp, vp, i32p, c_int, i32p, c_int, i32p, vp],
        "oscar_project_quantize_prefill": [vp, c_int, c_int, vp, c_int, vp, vp, i32p, c_int, i32p, c_int, i32p, vp],
        "oscar_append_kv": [vp, c_int, c_int, vp, vp, i32p, i32p, c_int, i32p, vp],
        "oscar_decode_attention": [vp, c_int, c_int, vp, i32p, i32p, c_int, i32p, c_float, vp, c_int, vp, vp],
        "oscar_set_decode_algo": [vp, c_int],
        "oscar_get_status": [vp, ctypes.POINTER(c_int)],
        "oscar_pack_rotated": [vp, c_int, c_int, vp, i32p, i32p, c_int, vp],
        "oscar_rotate": [vp, c_int, c_int, vp, vp, c_int, vp],
        "oscar_bf16_decode_workspace_bytes": [c_int, c_int, c_int, sz],
        "oscar_bf16_decode": [c_int, c_int, c_int, vp, c_int, vp, i32p, i32p, c_int, c_float, vp, c_int, vp, vp,
                              ctypes.c_size_t, c_int, vp],
        "oscar_calibrate": [vp, vp, vp, c_int, c_float, c_float, c_float, vp, vp, vp, vp, vp, vp],
        "oscar_profile_begin": [vp, c_int],
        "oscar_profile_read": [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_int)],
        "oscar_trace_ctas": [vp, vp, c_int],
        "oscar_trace_timeline": [vp, vp, c_int],
        "oscar_check_wait_timeout": [vp, vp],
        "oscar_decode_step": [vp, c_int, c_int, vp, vp, vp, i32p, i32p, c_int, i32p, c_float, vp, c_int, vp, vp],
        "oscar_decode_attention_shared": [vp, c_int, c_int, vp, i32p, i32p, c_int, c_int, i32p, c_float, vp, c_int,
                                          vp, vp],
        "oscar_decode_step_shared": [vp, c_int, c_int, vp, vp, vp, i32p, i32p, c_int, c_int, i32p, c_float, vp,
                                     c_int, vp, vp],
        "oscar_decode_attention_noalloc": [ctypes.POINTER(Layout), vp, c_int, c_int, vp, i32p, i32p, c_int, i32p,
                                           c_float, vp, c_int, vp, vp, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = c_int
    lib.oscar_error_string.argtypes = [c_int]
    lib.oscar_error_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def _check(rc: int, what: str):
    if rc != OK:
        raise OscarError(rc, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev_i32(x, device):
    import torch
    if isinstance(x, torch.Tensor):
        assert x.dtype == torch.int32 and x.is_cuda and x.is_contiguous()
        return x
    return torch.as_tensor(np.ascontiguousarray(x, dtype=np.int32), device=device)


@dataclass
class CacheConfig:
    num_layers: int
    num_kv_heads: int
    num_q_heads: int
    num_int2_pages: int
    num_bf16_pages: int
    max_batch: int = 1
    max_splits: int = 256
    v_mode: int = V_ABSORBED
    head_dim: int = 128
    group: int = 64
    page_size: int = 64
    sink: int = 64
    recent: int = 256
    meta_format: int = META_F16        # META_U8: 16-bit (mn8, mx8) group metadata, 4608-byte INT2 blocks;
    #                                    META_CB: Lloyd-Max codebook levels with fp16 (range, zero) metadata

    def layout(self) -> Layout:
        return Layout(self.num_layers, self.num_kv_heads, self.num_q_heads, self.head_dim, self.group,
                      self.page_size, self.sink, self.recent, self.num_int2_pages, self.num_bf16_pages, self.v_mode,
                      self.max_batch, self.max_splits, self.meta_format)


def cache_bytes(cfg: CacheConfig) -> tuple[int, int]:
    lay = cfg.layout()
    pb, wb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib.oscar_cache_bytes(ctypes.byref(lay), ctypes.byref(pb), ctypes.byref(wb)), "oscar_cache_bytes")
    return pb.value, wb.value


class OscarCache:
    """A mixed-precision KV cache: caller-owned pool and workspace (torch uint8 tensors) plus the library handle."""

    def __init__(self, cfg: CacheConfig, device="cuda", pool=None, workspace=None):
        import torch
        self.cfg = cfg
        self.device = torch.device(device)
        pb, wb = cache_bytes(cfg)
        self.pool = torch.zeros(pb, dtype=torch.uint8, device=self.device) if pool is None else pool
        self.workspace = torch.zeros(wb, dtype=torch.uint8, device=self.device) if workspace is None else workspace
        lay = cfg.layout()
        h = ctypes.c_void_p()
        _check(_lib.oscar_cache_create(ctypes.byref(lay), _ptr(self.pool), _ptr(self.workspace), ctypes.byref(h)),
               "oscar_cache_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.oscar_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # ---- layout views --------------------------------------------------------------
    def layer_offsets(self, layer: int) -> tuple[int, int, int]:
        a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
        _check(_lib.oscar_layer_offsets(self._h, layer, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
               "oscar_layer_offsets")
        return a.value, b.value, c.value

    def int2_pages(self, layer: int):
        """uint8 view [num_int2_pages, Hkv, block] of a layer's INT2 page blocks (block = 5120 bytes,
        or 4608 with the compact META_U8 metadata)."""
        o, _, _ = self.layer_offsets(layer)
        blk = 4608 if self.cfg.meta_format == META_U8 else 5120
        n = self.cfg.num_int2_pages * self.cfg.num_kv_heads * blk
        return self.pool[o:o + n].view(self.cfg.num_int2_pages, self.cfg.num_kv_heads, blk)

    def bf16_pages(self, layer: int):
        """uint8 view [num_bf16_pages, Hkv, 32768] of a layer's BF16 page blocks."""
        _, o, _ = self.layer_offsets(layer)
        n = self.cfg.num_bf16_pages * self.cfg.num_kv_heads * 32768
        return self.pool[o:o + n].view(self.cfg.num_bf16_pages, self.cfg.num_kv_heads, 32768)

    # ---- entry points ---------------------------------------------------------------
    def set_rotation(self, layer: int, U_K, U_V, tau_K, tau_V, stream=None):
        f32 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float32)
        uk, uv, tk, tv = f32(U_K), f32(U_V), f32(tau_K), f32(tau_V)
        _check(_lib.oscar_set_rotation(self._h, layer, _ptr(uk), _ptr(uv), _ptr(tk), _ptr(tv), _stream(stream)),
               "oscar_set_rotation")

    def set_codebook(self, layer: int, cb_K, cb_V, stream=None):
        """Codebook bytes uint8 [Hkv][4] of K and V (META_CB layouts); call after set_rotation."""
        ck = np.ascontiguousarray(cb_K, dtype=np.uint8)
        cv = np.ascontiguousarray(cb_V, dtype=np.uint8)
        _check(_lib.oscar_set_codebook(self._h, layer, _ptr(ck), _ptr(cv), _stream(stream)), "oscar_set_codebook")

    def quantize_prefill(self, layer: int, k, v, cu_seqlens, hist_pt, bf16_pt, total_tokens: int | None = None,
                         stream=None):
        cu = _dev_i32(cu_seqlens, self.device)
        hp = _dev_i32(hist_pt, self.device)
        bp = _dev_i32(bf16_pt, self.device)
        B = cu.numel() - 1
        total = int(k.shape[0]) if total_tokens is None else total_tokens
        mhp = hp.shape[1] if hp.dim() == 2 else 0
        _check(_lib.oscar_quantize_prefill(self._h, layer, B, _ptr(k), _ptr(v), _ptr(cu), total, _ptr(hp), mhp,
                                           _ptr(bp), _stream(stream)), "oscar_quantize_prefill")

    def project_quantize_prefill(self, layer: int, x, w_k, w_v, cu_seqlens, hist_pt, bf16_pt,
                                 total_tokens: int | None = None, stream=None):
        """quantize_prefill of K = bf16(x W_k^T), V = bf16(x W_v^T): x bf16 [T, d_model], w bf16 [Hkv*128, d_model]."""
        cu = _dev_i32(cu_seqlens, self.device)
        hp = _dev_i32(hist_pt, self.device)
        bp = _dev_i32(bf16_pt, self.device)
        B = cu.numel() - 1
        total = int(x.shape[0]) if total_tokens is None else total_tokens
        mhp = hp.shape[1] if hp.dim() == 2 else 0
        _check(_lib.oscar_project_quantize_prefill(self._h, layer, B, _ptr(x), int(x.shape[1]), _ptr(w_k), _ptr(w_v),
                                                   _ptr(cu), total, _ptr(hp), mhp, _ptr(bp), _stream(stream)),
               "oscar_project_quantize_prefill")

    def append_kv(self, layer: int, k, v, seq_lens_before, hist_pt, bf16_pt, stream=None):
        sl = _dev_i32(seq_lens_before, self.device)
        hp = _dev_i32(hist_pt, self.device)
        bp = _dev_i32(bf16_pt, self.device)
        _check(_lib.oscar_append_kv(self._h, layer, sl.numel(), _ptr(k), _ptr(v), _ptr(sl), _ptr(hp),
                                    hp.shape[1] if hp.dim() == 2 else 0, _ptr(bp), _stream(stream)),
               "oscar_append_kv")

    def decode_attention(self, layer: int, q, seq_lens, hist_pt, bf16_pt, sm_scale: float, out=None,
                         out_dtype: int = OUT_BF16, lse=None, stream=None, shared_hist_pages: int = 0):
        """Decode attention; shared_hist_pages > 0 states that history pages [0, shared_hist_pages) of every
        request are the same pages (oscar_decode_attention_shared)."""
        import torch
        sl = _dev_i32(seq_lens, self.device)
        hp = _dev_i32(hist_pt, self.device)
        bp = _dev_i32(bf16_pt, self.device)
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32 if out_dtype == OUT_FP32 else torch.bfloat16,
                              device=self.device)
        mhp = hp.shape[1] if hp.dim() == 2 else 0
        if shared_hist_pages:
            _check(_lib.oscar_decode_attention_shared(self._h, layer, sl.numel(), _ptr(q), _ptr(sl), _ptr(hp), mhp,
                                                      int(shared_hist_pages), _ptr(bp), float(sm_scale), _ptr(out),
                                                      out_dtype, _ptr(lse), _stream(stream)),
                   "oscar_decode_attention_shared")
        else:
            _check(_lib.oscar_decode_attention(self._h, layer, sl.numel(), _ptr(q), _ptr(sl), _ptr(hp), mhp,
                                               _ptr(bp), float(sm_scale), _ptr(out), out_dtype, _ptr(lse),
                                               _stream(stream)), "oscar_decode_attention")
        return out

    def decode_step(self, layer: int, q, k, v, seq_lens_before, hist_pt, bf16_pt, sm_scale: float, out=None,
                    out_dtype: int = OUT_BF16, lse=None, stream=None, shared_hist_pages: int = 0):
        """append_kv(k, v) then decode_attention(q) over seq_lens_before + 1 tokens, in one call
        (oscar_decode_step_shared when shared_hist_pages > 0)."""
        import torch
        sl = _dev_i32(seq_lens_before, self.device)
        hp = _dev_i32(hist_pt, self.device)
        bp = _dev_i32(bf16_pt, self.device)
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32 if out_dtype == OUT_FP32 else torch.bfloat16,
                              device=self.device)
        mhp = hp.shape[1] if hp.dim() == 2 else 0
        if shared_hist_pages:
            _check(_lib.oscar_decode_step_shared(self._h, layer, sl.numel(), _ptr(q), _ptr(k), _ptr(v), _ptr(sl),
                                                 _ptr(hp), mhp, int(shared_hist_pages), _ptr(bp), float(sm_scale),
                                                 _ptr(out), out_dtype, _ptr(lse), _stream(stream)),
                   "oscar_decode_step_shared")
        else:
            _check(_lib.oscar_decode_step(self._h, layer, sl.numel(), _ptr(q), _ptr(k), _ptr(v), _ptr(sl), _ptr(hp),
                                          mhp, _ptr(bp), float(sm_scale), _ptr(out), out_dtype, _ptr(lse),
                                          _stream(stream)), "oscar_decode_step")
        return out

    def set_decode_algo(self, algo: int):
        _check(_lib.oscar_set_decode_algo(self._h, algo), "oscar_set_decode_algo")

    def get_status(self) -> int:
        code = ctypes.c_int()
        rc = _lib.oscar_get_status(self._h, ctypes.byref(code))
        if rc not in (OK, ERR_DEVICE_STATUS):
            raise OscarError(rc, "oscar_get_status")
        return code.value

    def pack_rotated(self, layer: int, kind: int, xrot, page_ids, rows, stream=None):
        pi = _dev_i32(page_ids, self.device)
        ro = _dev_i32(rows, self.device)
        _check(_lib.oscar_pack_rotated(self._h, layer, kind, _ptr(xrot), _ptr(pi), _ptr(ro), pi.numel(),
                                       _stream(stream)), "oscar_pack_rotated")

    def rotate(self, layer: int, kind: int, x, stream=None):
        import torch
        y = torch.empty(x.shape, dtype=torch.float32, device=self.device)
        _check(_lib.oscar_rotate(self._h, layer, kind, _ptr(x), _ptr(y), int(x.shape[0]), _stream(stream)),
               "oscar_rotate")
        return y

    def trace_ctas(self, buf=None):
        """Record per-CTA timelines of following tensor-core decode launches into ``buf`` (an int64 device
        tensor of 8 * n elements, n records); None stops recording."""
        n = 0 if buf is None else buf.numel() // 8
        _check(_lib.oscar_trace_ctas(self._h, _ptr(buf), n), "oscar_trace_ctas")

    def check_wait_timeout(self, stream=None):
        """Run the bounded-wait self-check: a device wait that nothing completes must give up (about 2 s)
        and set the TIMEOUT bit of the status word."""
        _check(_lib.oscar_check_wait_timeout(self._h, _stream(stream)), "oscar_check_wait_timeout")

    def trace_timeline(self, buf=None):
        """Record a timeline of every CTA of the following kernel launches into ``buf`` (an int64 device tensor
        of 4 + 4 * n elements, n records, buf[0] zeroed by the caller); None stops recording."""
        n = 0 if buf is None else (buf.numel() - 4) // 4
        _check(_lib.oscar_trace_timeline(self._h, _ptr(buf), n), "oscar_trace_timeline")

    def profile_begin(self, capacity: int):
        _check(_lib.oscar_profile_begin(self._h, capacity), "oscar_profile_begin")

    def profile_read(self) -> tuple[float, int]:
        ms, n = ctypes.c_double(), ctypes.c_int()
        _check(_lib.oscar_profile_read(self._h, ctypes.byref(ms), ctypes.byref(n)), "oscar_profile_read")
        return ms.value, n.value


def bf16_decode_workspace_bytes(max_batch: int, num_q_heads: int, max_splits: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.oscar_bf16_decode_workspace_bytes(max_batch, num_q_heads, max_splits, ctypes.byref(n)),
           "oscar_bf16_decode_workspace_bytes")
    return n.value


def bf16_decode(kv_pages, q, seq_lens, page_table, sm_scale: float, num_kv_heads: int, workspace, max_splits: int,
                out=None, out_dtype: int = OUT_BF16, lse=None, stream=None):
    """Decode over an all-BF16 paged cache kv_pages [num_pages, Hkv, 2, 64, 128] bf16."""
    import torch
    B, hq = int(q.shape[0]), int(q.shape[1])
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32 if out_dtype == OUT_FP32 else torch.bfloat16, device=q.device)
    sl = _dev_i32(seq_lens, q.device)
    pt = _dev_i32(page_table, q.device)
    _check(_lib.oscar_bf16_decode(B, hq, num_kv_heads, _ptr(kv_pages), int(kv_pages.shape[0]), _ptr(q), _ptr(sl),
                                  _ptr(pt), int(pt.shape[1]), float(sm_scale), _ptr(out), out_dtype, _ptr(lse),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(), max_splits,
                                  _stream(stream)), "oscar_bf16_decode")
    return out


def calibrate_codebook(x_rot, tau) -> np.ndarray:
    """Host Lloyd-Max calibration of one codebook from rotated float32 rows x_rot [N, 128] and clip
    thresholds tau [128]: returns the codebook bytes uint8 [4]."""
    x = np.ascontiguousarray(x_rot, dtype=np.float32)
    t = np.ascontiguousarray(tau, dtype=np.float32)
    out = np.zeros(4, np.uint8)
    _check(_lib.oscar_calibrate_codebook(_ptr(x), x.shape[0], _ptr(t), _ptr(out)), "oscar_calibrate_codebook")
    return out


def calibrate(Q, K, V, sm_scale: float, c_K: float = 0.96, c_V: float = 0.92):
    """Host calibration of one (layer, kv head): returns dict with U_K, U_V [128,128], tau_K, tau_V [128] float32
    and eig_K, eig_V [128] float64."""
    q = np.ascontiguousarray(Q, dtype=np.float32)
    k = np.ascontiguousarray(K, dtype=np.float32)
    v = np.ascontiguousarray(V, dtype=np.float32)
    out = {n: np.zeros((128, 128), np.float32) for n in ("U_K", "U_V")}
    out.update({n: np.zeros(128, np.float32) for n in ("tau_K", "tau_V")})
    out.update({n: np.zeros(128, np.float64) for n in ("eig_K", "eig_V")})
    _check(_lib.oscar_calibrate(_ptr(q), _ptr(k), _ptr(v), q.shape[0], float(sm_scale), float(c_K), float(c_V),
                                _ptr(out["U_K"]), _ptr(out["U_V"]), _ptr(out["tau_K"]), _ptr(out["tau_V"]),
                                _ptr(out["eig_K"]), _ptr(out["eig_V"])), "oscar_calibrate")
    return out


def decode_attention_noalloc(cfg: CacheConfig, pool, layer: int, q, seq_lens, hist_pt, bf16_pt, sm_scale: float,
                             out=None, out_dtype: int = OUT_BF16, lse=None, status=None, stream=None):
    """Decode attention through the allocation-free entry point, for callers that cannot allocate device
    memory (for instance inside CUDA graph capture): same result as OscarCache.decode_attention, with the
    cache given by its config and pool tensor, scratch in the library's fixed device array, and the call's
    status bits written to ``status`` (an int32 device tensor of one element) when given. Calls that may
    overlap on the GPU share that scratch and must not be issued concurrently."""
    import torch
    dev = pool.device
    sl = _dev_i32(seq_lens, dev)
    hp = _dev_i32(hist_pt, dev)
    bp = _dev_i32(bf16_pt, dev)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32 if out_dtype == OUT_FP32 else torch.bfloat16, device=dev)
    lay = cfg.layout()
    _check(_lib.oscar_decode_attention_noalloc(ctypes.byref(lay), _ptr(pool), layer, sl.numel(), _ptr(q), _ptr(sl),
                                               _ptr(hp), hp.shape[1] if hp.dim() == 2 else 0, _ptr(bp),
                                               float(sm_scale), _ptr(out), out_dtype, _ptr(lse), _ptr(status),
                                               _stream(stream)), "oscar_decode_attention_noalloc")
    return out
