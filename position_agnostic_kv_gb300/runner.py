"""Device-resident driver for one batch of requests over a paged, position-free KV cache.

This is the call sequence a serving engine makes, expressed through the public binding only:
build the block words on the host (``lazy_build_doc_meta``), write each cached document's
keys and values once (``lazy_kv_write`` at local positions), then per batch write the query
tokens, run the causal prefill, and for every decode step write the new token and attend.

The batch description is duck-typed (any object with the attributes used below, e.g. a
``workloads.Workload``); values arrive as bf16 bit patterns (numpy uint16).
"""
from __future__ import annotations

import numpy as np
import torch

from . import (PHASE_DECODE, PHASE_PREFILL, attn_decode, attn_prefill, build_doc_meta,
               build_rope_table, kv_write, pos_cfg_from, workspace_size)

PAGE = 16


def bits_to_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """bf16 bit patterns (numpy uint16) -> bf16 tensor on ``device`` (exact)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def i32(x, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.int32))).to(device)


class PagedBatch:
    """Caches, block words and per-request metadata of one batch, resident on one GPU."""

    def __init__(self, w, device="cuda", use_table: bool = False, pos_kind: str | None = None):
        self.w = w
        self.device = torch.device(device)
        self.B, self.Hq, self.Hkv, self.D = w.B, w.Hq, w.Hkv, w.D
        (self.block_table, self.meta_h, self.seq_len0_h, self.q_start_h,
         self.doc_blocks_h) = build_doc_meta(w.req_inst_off, w.req_inst, w.inst_len,
                                             w.inst_page_off, w.inst_pages, w.q_len,
                                             w.q_page_off, w.q_pages, w.max_blocks)
        dev = self.device
        self.meta = torch.from_numpy(self.meta_h.view(np.int64)).to(dev)
        self.q_start = i32(self.q_start_h, dev)
        self.doc_blocks = i32(self.doc_blocks_h, dev)
        self.seq_len0 = i32(self.seq_len0_h, dev)
        self.cu_q = i32(w.cu_q, dev)
        self.max_q = int(np.max(w.q_len)) if len(w.q_len) else 0
        self.total_q = int(np.sum(w.q_len))
        shape = (w.num_pages, w.Hkv, PAGE, w.D)
        self.k_cache = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        self.v_cache = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        p = w.pos
        kind = pos_kind or p.kind
        self.slopes = None
        if p.alibi_slopes is not None:
            self.slopes = torch.from_numpy(np.asarray(p.alibi_slopes, np.float32)).to(dev)
        self.table = None
        rd = getattr(p, "rotary_dim", w.D) if kind in ("rope", "yarn") else w.D
        inter = bool(getattr(p, "interleaved", False))
        self.cfg = pos_cfg_from(kind, w.D, rope_theta=p.rope_theta, yarn_factor=p.yarn_factor,
                                yarn_orig_ctx=p.yarn_orig_ctx, yarn_beta_fast=p.yarn_beta_fast,
                                yarn_beta_slow=p.yarn_beta_slow, alibi_slopes=self.slopes,
                                rotary_dim=rd, interleaved=inter)
        if use_table and kind in ("rope", "yarn"):
            max_pos = int(self.q_start_h.max()) + int(np.max(w.q_len)) + w.n_decode + 1
            self.table = torch.empty((max_pos, rd), dtype=torch.float32, device=dev)
            build_rope_table(self.cfg, max_pos, self.table)
            self.cfg = pos_cfg_from(kind, w.D, rope_theta=p.rope_theta,
                                    yarn_factor=p.yarn_factor, yarn_orig_ctx=p.yarn_orig_ctx,
                                    yarn_beta_fast=p.yarn_beta_fast,
                                    yarn_beta_slow=p.yarn_beta_slow, alibi_slopes=self.slopes,
                                    cos_sin=self.table, rotary_dim=rd, interleaved=inter)
        self.max_blocks = w.max_blocks
        ws_dec = workspace_size(PHASE_DECODE, self.B, self.B, self.max_blocks, self.Hq, self.Hkv,
                                self.D)
        ws_pre = workspace_size(PHASE_PREFILL, max(self.total_q, 1), self.B, self.max_blocks,
                                self.Hq, self.Hkv, self.D)
        self.ws = torch.empty(max(ws_dec, ws_pre, 256), dtype=torch.uint8, device=dev)

    # ---------------------------------------------------------------- cache fill
    def fill_documents(self):
        """Write every document copy into the cache once (keys rotated by local position)."""
        w = self.w
        by_doc: dict[int, list[int]] = {}
        for i, d in enumerate(w.inst_doc):
            by_doc.setdefault(int(d), []).append(i)
        for d, insts in by_doc.items():
            k, v = w.doc_kv(d)
            kt, vt = bits_to_tensor(k, self.device), bits_to_tensor(v, self.device)
            for i in insts:
                slot, lp = w.inst_slots(i)
                kv_write(kt, vt, i32(slot, self.device), i32(lp, self.device), self.k_cache,
                         self.v_cache, self.cfg)

    # ---------------------------------------------------------------- prefill
    def upload_prefill(self):
        q, k, v, slot, lp = self.w.prefill_tokens()
        dev = self.device
        return dict(q=bits_to_tensor(q, dev), k=bits_to_tensor(k, dev), v=bits_to_tensor(v, dev),
                    slot=i32(slot, dev), lp=i32(lp, dev))

    def prefill(self, inp, out=None, lse=None):
        """Write the query tokens' keys/values, then the causal prefill of every query row."""
        if out is None:
            out = torch.empty((self.total_q, self.Hq, self.D), dtype=torch.bfloat16,
                              device=self.device)
        if self.total_q == 0:
            return out
        kv_write(inp["k"], inp["v"], inp["slot"], inp["lp"], self.k_cache, self.v_cache, self.cfg)
        attn_prefill(inp["q"], self.cu_q, self.q_start, self.doc_blocks, self.meta, self.k_cache,
                     self.v_cache, self.cfg, out, self.max_q, lse=lse, ws=self.ws)
        return out

    # ---------------------------------------------------------------- decode
    def upload_decode(self, t: int):
        q, k, v, slot, lp = self.w.decode_tokens(t)
        dev = self.device
        seq = self.seq_len0_h + t + 1
        return dict(q=bits_to_tensor(q, dev), k=bits_to_tensor(k, dev), v=bits_to_tensor(v, dev),
                    slot=i32(slot, dev), lp=i32(lp, dev), seq_len=i32(seq, dev))

    def decode_step(self, inp, out=None, lse=None):
        """Write step t's token (at p = m) then attend from it."""
        if out is None:
            out = torch.empty((self.B, self.Hq, self.D), dtype=torch.bfloat16, device=self.device)
        kv_write(inp["k"], inp["v"], inp["slot"], inp["lp"], self.k_cache, self.v_cache, self.cfg)
        attn_decode(inp["q"], inp["seq_len"], self.q_start, self.doc_blocks, self.meta,
                    self.k_cache, self.v_cache, self.cfg, out, lse=lse, ws=self.ws)
        return out


# -------------------------------------------------------------------- cold documents
def encode_document(q, k, v, pages, k_cache, v_cache, cfg, ws=None, out=None):
    """Cold-document processing: the first time a document is seen it is encoded alone, from
    local position 0 ([NOTE] 整体框架: each document's cache is built independently, indexed
    from 0).  Its keys (rotated by their local positions) and values are written into
    ``pages`` of the position-free cache, then the document's own causal attention runs as a
    request with no cached documents whose query segment is the document (Delta = 0).

    q, k, v: bf16 [L, Hq | Hkv, D] raw projections of the document's tokens; pages: int list
    of ceil(L / 16) physical page ids.  Returns the attention output [L, Hq, D] (bf16); the
    cached pages can then be reused by any later request at any document offset."""
    L, Hq, D = q.shape
    dev = q.device
    pages = np.asarray(pages, dtype=np.int32)
    if len(pages) * PAGE < L:
        raise ValueError("encode_document: fewer pages than the document needs")
    t = np.arange(L, dtype=np.int32)
    kv_write(k, v, i32(pages[t // PAGE] * PAGE + t % PAGE, dev), i32(t, dev), k_cache, v_cache, cfg)
    max_blocks = len(pages)
    _, meta_h, _, q_start_h, doc_blocks_h = build_doc_meta(
        [0, 0], [], [], [0], [], [L], [0, len(pages)], pages, max_blocks)
    meta = torch.from_numpy(meta_h.view(np.int64)).to(dev)
    if out is None:
        out = torch.empty((L, Hq, D), dtype=torch.bfloat16, device=dev)
    Hkv = k_cache.shape[1]
    if ws is None:
        n = workspace_size(PHASE_PREFILL, L, 1, max_blocks, Hq, Hkv, D)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    attn_prefill(q, i32([0, L], dev), i32(q_start_h, dev), i32(doc_blocks_h, dev), meta, k_cache,
                 v_cache, cfg, out, L, ws=ws)
    return out
