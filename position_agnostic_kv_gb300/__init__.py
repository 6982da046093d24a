"""position_agnostic_kv_gb300 -- LazyAttention's hot path on one GB300 (sm_103a).

A thin ctypes binding over ``liblazykv.so`` (C ABI declared in ``include/lazykv.h``).  Every
step of the path runs in the library's kernels; this module only marshals arguments: it checks
dtypes, shapes, contiguity and devices of PyTorch tensors and passes raw pointers and the
current CUDA stream.  There is no fallback of any kind: if the library is missing, importing
this package raises.

Functions mirror the C entry points: ``build_doc_meta`` (host), ``build_rope_table``,
``kv_write``, ``attn_decode``, ``attn_prefill``, ``workspace_size``, ``device_status``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = ["LIB_PATH", "lib", "PosCfg", "LazyError", "DocCache", "POS_ROPE", "POS_YARN", "POS_ALIBI",
           "POS_NONE", "PHASE_DECODE", "PHASE_PREFILL", "EXPORTED_SYMBOLS", "build_doc_meta",
           "build_rope_table", "kv_write", "attn_decode", "attn_decode_noalloc", "attn_prefill", "workspace_size",
           "device_status", "pos_cfg_from"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblazykv.so")
POS_ROPE, POS_YARN, POS_ALIBI, POS_NONE = 0, 1, 2, 3
PHASE_DECODE, PHASE_PREFILL = 0, 1
EXPORTED_SYMBOLS = ("lazy_build_doc_meta", "lazy_build_rope_table", "lazy_kv_write",
                    "lazy_attn_decode", "lazy_attn_decode_noalloc", "lazy_attn_prefill", "lazy_workspace_size",
                    "lazy_device_status", "lazy_last_error", "lazy_version", "lazy_doc_cache_create",
                    "lazy_doc_cache_destroy", "lazy_doc_cache_lookup", "lazy_doc_cache_acquire",
                    "lazy_doc_cache_release", "lazy_doc_cache_stats")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
lib = ctypes.CDLL(LIB_PATH)


class LazyError(RuntimeError):
    pass


class PosCfg(ctypes.Structure):
    """Mirror of ``lazy_pos_cfg``."""
    _fields_ = [("kind", ctypes.c_int32), ("rotary_dim", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("yarn_factor", ctypes.c_float),
                ("yarn_orig_ctx", ctypes.c_int32), ("yarn_beta_fast", ctypes.c_float),
                ("yarn_beta_slow", ctypes.c_float), ("alibi_slopes", ctypes.c_void_p),
                ("cos_sin", ctypes.c_void_p), ("max_pos", ctypes.c_int32),
                ("interleaved", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_sig = {
    "lazy_build_doc_meta": [_I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P],
    "lazy_build_rope_table": [ctypes.POINTER(PosCfg), _I, _P, _P],
    "lazy_kv_write": [_P, _P, _P, _P, _I, _I, _I, _P, _P, _I, ctypes.POINTER(PosCfg), _P],
    "lazy_attn_decode": [_P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, ctypes.c_float,
                         ctypes.POINTER(PosCfg), _P, _P, _P, _SZ, _P],
    "lazy_attn_decode_noalloc": [_P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I,
                                 ctypes.c_float, ctypes.POINTER(PosCfg), _P, _P, _P],
    "lazy_attn_prefill": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _I, _I,
                          ctypes.c_float, ctypes.POINTER(PosCfg), _P, _P, _P, _SZ, _P],
    "lazy_workspace_size": [_I, _I, _I, _I, _I, _I, _I],
    "lazy_device_status": [_P, ctypes.POINTER(ctypes.c_uint32)],
    "lazy_last_error": [],
    "lazy_version": [],
}
for _name, _args in _sig.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _I
lib.lazy_workspace_size.restype = _SZ
lib.lazy_last_error.restype = ctypes.c_char_p
_LL = ctypes.POINTER(ctypes.c_longlong)
_IP = ctypes.POINTER(ctypes.c_int)
lib.lazy_doc_cache_create.argtypes = [_I, _I]
lib.lazy_doc_cache_create.restype = _P
lib.lazy_doc_cache_destroy.argtypes = [_P]
lib.lazy_doc_cache_destroy.restype = None
lib.lazy_doc_cache_lookup.argtypes = [_P, _I, _I, _P, _I]
lib.lazy_doc_cache_lookup.restype = _I
lib.lazy_doc_cache_acquire.argtypes = [_P, _I, _I, _I, _P, _IP]
lib.lazy_doc_cache_acquire.restype = _I
lib.lazy_doc_cache_release.argtypes = [_P, _I, _I]
lib.lazy_doc_cache_release.restype = _I
lib.lazy_doc_cache_stats.argtypes = [_P, _LL, _LL, _LL, _IP, _IP]
lib.lazy_doc_cache_stats.restype = _I


def _check(rc: int, what: str):
    if rc != 0:
        msg = lib.lazy_last_error().decode(errors="replace")
        raise LazyError(f"{what} failed with code {rc}: {msg}")


# ------------------------------------------------------------------ tensor helpers
def _dev_ptr(t, dtype=None, name="tensor"):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def pos_cfg_from(kind: str, head_dim: int, rope_theta: float = 1e4, yarn_factor: float = 1.0,
                 yarn_orig_ctx: int = 0, yarn_beta_fast: float = 32.0,
                 yarn_beta_slow: float = 1.0, alibi_slopes=None, cos_sin=None,
                 rotary_dim: int | None = None, interleaved: bool = False) -> PosCfg:
    """Build a ``PosCfg`` (device tensors for slopes / table are referenced, not copied).
    ``rotary_dim`` defaults to ``head_dim``; ``interleaved`` selects (x_2i, x_2i+1) pairs."""
    import torch
    kinds = {"rope": POS_ROPE, "yarn": POS_YARN, "alibi": POS_ALIBI, "none": POS_NONE}
    c = PosCfg()
    c.kind = kinds[kind]
    c.rotary_dim = head_dim if rotary_dim is None else int(rotary_dim)
    c.interleaved = int(bool(interleaved))
    c.rope_theta = rope_theta
    c.yarn_factor = yarn_factor
    c.yarn_orig_ctx = yarn_orig_ctx
    c.yarn_beta_fast = yarn_beta_fast
    c.yarn_beta_slow = yarn_beta_slow
    c.alibi_slopes = _dev_ptr(alibi_slopes, torch.float32, "alibi_slopes")
    if cos_sin is not None:
        c.cos_sin = _dev_ptr(cos_sin, torch.float32, "cos_sin")
        c.max_pos = cos_sin.shape[0]
    return c


# ------------------------------------------------------------------ entry points
def build_doc_meta(req_doc_off, req_docs, doc_len, doc_page_off, doc_pages, q_len, q_page_off,
                   q_pages, max_blocks: int):
    """Host metadata builder.  Numpy int32 inputs; returns (block_table [B, max_blocks] int32,
    meta [B, max_blocks] uint64, seq_len, q_start, doc_blocks [B] int32)."""
    def a32(x):
        return np.ascontiguousarray(np.asarray(x, dtype=np.int32))
    req_doc_off, req_docs, doc_len = a32(req_doc_off), a32(req_docs), a32(doc_len)
    doc_page_off, doc_pages = a32(doc_page_off), a32(doc_pages)
    q_len, q_page_off, q_pages = a32(q_len), a32(q_page_off), a32(q_pages)
    B = len(req_doc_off) - 1
    bt = np.zeros((B, max_blocks), np.int32)
    meta = np.zeros((B, max_blocks), np.uint64)
    seq_len = np.zeros(B, np.int32)
    q_start = np.zeros(B, np.int32)
    doc_blocks = np.zeros(B, np.int32)
    p = lambda x: x.ctypes.data_as(ctypes.c_void_p)
    rc = lib.lazy_build_doc_meta(B, p(req_doc_off), p(req_docs), len(doc_len), p(doc_len),
                                 p(doc_page_off), p(doc_pages), p(q_len), p(q_page_off),
                                 p(q_pages), max_blocks, p(bt), p(meta), p(seq_len), p(q_start),
                                 p(doc_blocks))
    _check(rc, "lazy_build_doc_meta")
    return bt, meta, seq_len, q_start, doc_blocks


def build_rope_table(cfg: PosCfg, max_pos: int, out, stream=None):
    import torch
    if tuple(out.shape) != (max_pos, cfg.rotary_dim):
        raise ValueError("out must be [max_pos, rotary_dim]")
    _check(lib.lazy_build_rope_table(ctypes.byref(cfg), max_pos,
                                     _dev_ptr(out, torch.float32, "out"), _stream(stream)),
           "lazy_build_rope_table")


def kv_write(k, v, slot, local_pos, k_cache, v_cache, cfg: PosCfg, stream=None):
    """Write raw k/v [T, Hkv, D] into the paged caches [P, Hkv, 16, D] (bf16)."""
    import torch
    T, Hkv, D = k.shape
    if tuple(v.shape) != (T, Hkv, D) or k_cache.shape[1:] != (Hkv, 16, D) or \
            v_cache.shape != k_cache.shape or tuple(slot.shape) != (T,):
        raise ValueError("kv_write: inconsistent shapes")
    _check(lib.lazy_kv_write(_dev_ptr(k, torch.bfloat16, "k"), _dev_ptr(v, torch.bfloat16, "v"),
                             _dev_ptr(slot, torch.int32, "slot"),
                             _dev_ptr(local_pos, torch.int32, "local_pos"), T, Hkv, D,
                             _dev_ptr(k_cache, torch.bfloat16, "k_cache"),
                             _dev_ptr(v_cache, torch.bfloat16, "v_cache"), k_cache.shape[0],
                             ctypes.byref(cfg), _stream(stream)), "lazy_kv_write")


def workspace_size(phase: int, rows: int, B: int, max_blocks: int, Hq: int, Hkv: int, D: int) -> int:
    return int(lib.lazy_workspace_size(phase, rows, B, max_blocks, Hq, Hkv, D))


def attn_decode(q, seq_len, q_start, doc_blocks, meta, k_cache, v_cache, cfg: PosCfg, out,
                lse=None, ws=None, scale: float = 0.0, stream=None):
    """One decode step: q [B, Hq, D] raw at m = seq_len - 1; writes out [B, Hq, D] bf16."""
    import torch
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    max_blocks = meta.shape[1]
    if meta.dtype != torch.uint64 and meta.dtype != torch.int64:
        raise TypeError("meta must be uint64 (or int64 bits)")
    if tuple(out.shape) != (B, Hq, D) or meta.shape[0] != B:
        raise ValueError("attn_decode: inconsistent shapes")
    wsp, wsb = (None, 0) if ws is None else (_dev_ptr(ws, None, "ws"), ws.numel() * ws.element_size())
    _check(lib.lazy_attn_decode(_dev_ptr(q, torch.bfloat16, "q"),
                                _dev_ptr(seq_len, torch.int32, "seq_len"),
                                _dev_ptr(q_start, torch.int32, "q_start"),
                                _dev_ptr(doc_blocks, torch.int32, "doc_blocks"),
                                _dev_ptr(meta, None, "meta"), B, max_blocks,
                                _dev_ptr(k_cache, torch.bfloat16, "k_cache"),
                                _dev_ptr(v_cache, torch.bfloat16, "v_cache"), k_cache.shape[0],
                                Hq, Hkv, D, scale, ctypes.byref(cfg),
                                _dev_ptr(out, torch.bfloat16, "out"),
                                _dev_ptr(lse, torch.float32, "lse"), wsp, wsb, _stream(stream)),
           "lazy_attn_decode")


def attn_decode_noalloc(q, seq_len, q_start, doc_blocks, meta, k_cache, v_cache, cfg: PosCfg,
                        out, lse=None, scale: float = 0.0, stream=None):
    """``attn_decode`` without a workspace: for callers that cannot allocate device memory.
    The split scratch lives in a fixed 16 MiB array inside the library (one per GPU), shared by
    all calls on that device; calls that overlap on the GPU race on it.  The first call on a
    device looks up the array's address, so make it before any stream capture."""
    import torch
    B, Hq, D = q.shape
    if tuple(out.shape) != (B, Hq, D) or meta.shape[0] != B:
        raise ValueError("attn_decode_noalloc: inconsistent shapes")
    _check(lib.lazy_attn_decode_noalloc(_dev_ptr(q, torch.bfloat16, "q"),
                                        _dev_ptr(seq_len, torch.int32, "seq_len"),
                                        _dev_ptr(q_start, torch.int32, "q_start"),
                                        _dev_ptr(doc_blocks, torch.int32, "doc_blocks"),
                                        _dev_ptr(meta, None, "meta"), B, meta.shape[1],
                                        _dev_ptr(k_cache, torch.bfloat16, "k_cache"),
                                        _dev_ptr(v_cache, torch.bfloat16, "v_cache"),
                                        k_cache.shape[0], Hq, k_cache.shape[1], D, scale,
                                        ctypes.byref(cfg), _dev_ptr(out, torch.bfloat16, "out"),
                                        _dev_ptr(lse, torch.float32, "lse"), _stream(stream)),
           "lazy_attn_decode_noalloc")


def attn_prefill(q, cu_q, q_start, doc_blocks, meta, k_cache, v_cache, cfg: PosCfg, out,
                 max_q: int, lse=None, ws=None, scale: float = 0.0, stream=None):
    """Causal prefill: q [sum Lq, Hq, D] raw; writes out [sum Lq, Hq, D] bf16."""
    import torch
    total_q, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    B = cu_q.shape[0] - 1
    max_blocks = meta.shape[1]
    if tuple(out.shape) != (total_q, Hq, D) or meta.shape[0] != B:
        raise ValueError("attn_prefill: inconsistent shapes")
    wsp, wsb = (None, 0) if ws is None else (_dev_ptr(ws, None, "ws"), ws.numel() * ws.element_size())
    _check(lib.lazy_attn_prefill(_dev_ptr(q, torch.bfloat16, "q"),
                                 _dev_ptr(cu_q, torch.int32, "cu_q"),
                                 _dev_ptr(q_start, torch.int32, "q_start"),
                                 _dev_ptr(doc_blocks, torch.int32, "doc_blocks"),
                                 _dev_ptr(meta, None, "meta"), B, max_blocks, total_q, max_q,
                                 _dev_ptr(k_cache, torch.bfloat16, "k_cache"),
                                 _dev_ptr(v_cache, torch.bfloat16, "v_cache"), k_cache.shape[0],
                                 Hq, Hkv, D, scale, ctypes.byref(cfg),
                                 _dev_ptr(out, torch.bfloat16, "out"),
                                 _dev_ptr(lse, torch.float32, "lse"), wsp, wsb, _stream(stream)),
           "lazy_attn_prefill")


def device_status(stream=None) -> int:
    """Synchronise, then read and clear the device status word (LAZY_STATUS_* bits)."""
    v = ctypes.c_uint32(0)
    _check(lib.lazy_device_status(_stream(stream), ctypes.byref(v)), "lazy_device_status")
    return int(v.value)


# ------------------------------------------------------------------ document cache manager
class DocCache:
    """Host document cache manager over a pool of ``num_pages`` pages (``lazy_doc_cache_*``):
    one entry per document (position-agnostic, this library's cache) or, with
    ``position_aware=True``, one per (document, position) variant (for comparison)."""

    def __init__(self, num_pages: int, position_aware: bool = False):
        self._h = lib.lazy_doc_cache_create(int(num_pages), int(bool(position_aware)))
        if not self._h:
            raise LazyError(f"lazy_doc_cache_create failed: {lib.lazy_last_error().decode(errors='replace')}")
        self.num_pages = int(num_pages)
        self.position_aware = bool(position_aware)

    def close(self):
        if self._h:
            lib.lazy_doc_cache_destroy(self._h)
            self._h = None

    __del__ = close

    def lookup(self, doc: int, pos: int = 0):
        """Page ids of the resident entry (a numpy int32 array) or None; no recency change."""
        n = lib.lazy_doc_cache_lookup(self._h, int(doc), int(pos), None, 0)
        if n < 0:
            _check(n, "lazy_doc_cache_lookup")
        if n == 0:
            return None
        out = np.zeros(n, np.int32)
        _check(0 if lib.lazy_doc_cache_lookup(self._h, int(doc), int(pos), out.ctypes.data, n) == n else -1,
               "lazy_doc_cache_lookup")
        return out

    def acquire(self, doc: int, n_pages: int, pos: int = 0):
        """Hold the entry for a batch: (pages int32 array, hit bool).  On a miss the pages are
        newly assigned and the caller writes the document into them."""
        out = np.zeros(int(n_pages), np.int32)
        hit = ctypes.c_int(0)
        _check(lib.lazy_doc_cache_acquire(self._h, int(doc), int(pos), int(n_pages), out.ctypes.data,
                                          ctypes.byref(hit)), "lazy_doc_cache_acquire")
        return out, bool(hit.value)

    def release(self, doc: int, pos: int = 0):
        _check(lib.lazy_doc_cache_release(self._h, int(doc), int(pos)), "lazy_doc_cache_release")

    def stats(self) -> dict:
        h, m, e = ctypes.c_longlong(), ctypes.c_longlong(), ctypes.c_longlong()
        n, f = ctypes.c_int(), ctypes.c_int()
        _check(lib.lazy_doc_cache_stats(self._h, ctypes.byref(h), ctypes.byref(m), ctypes.byref(e),
                                        ctypes.byref(n), ctypes.byref(f)), "lazy_doc_cache_stats")
        return {"hits": h.value, "misses": m.value, "evictions": e.value, "entries": n.value,
                "free_pages": f.value}
