"""Test-side helpers that prepare oracle inputs from a seeded workload.

Test infrastructure: imports the oracle and the input generators, never the product.
"""
from __future__ import annotations

import numpy as np

import oracle
from workloads import Workload


def oracle_meta(w: Workload):
    """(block_table, meta, seq_len, q_start, doc_blocks) from the oracle's packer."""
    return oracle.build_meta(w.req_inst_off, w.req_inst, w.inst_len, w.inst_page_off,
                             w.inst_pages, w.q_len, w.q_page_off, w.q_pages, w.max_blocks)


def empty_caches(w: Workload):
    shape = (w.num_pages, w.Hkv, oracle.PAGE, w.D)
    return np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)


def oracle_fill_docs(w: Workload, kc, vc):
    """Write every document instance into the caches with the oracle's kv_write."""
    pos = w.pos.as_dict()
    for i in range(len(w.inst_doc)):
        k, v = w.doc_kv(int(w.inst_doc[i]))
        slot, lp = w.inst_slots(i)
        oracle.kv_write(k, v, slot, lp, pos, kc, vc)


def oracle_write_prefill(w: Workload, kc, vc):
    q, k, v, slot, lp = w.prefill_tokens()
    if len(slot):
        oracle.kv_write(k, v, slot, lp, w.pos.as_dict(), kc, vc)
    return q


def oracle_write_decode(w: Workload, t: int, kc, vc):
    q, k, v, slot, lp = w.decode_tokens(t)
    oracle.kv_write(k, v, slot, lp, w.pos.as_dict(), kc, vc)
    return q


def raw_segments(w: Workload, b: int, n_decode_written: int):
    """Request b's prompt as raw (pre-RoPE) fp64 segments: its documents in order, then its
    prefill tokens, then the decode tokens written so far."""
    segs = []
    for d in w.request_docs(b):
        k, v = w.doc_kv(int(d))
        segs.append((oracle.bf16_bits_to_f64(k), oracle.bf16_bits_to_f64(v)))
    q, k, v, _, _ = w.prefill_tokens()
    cu = w.cu_q
    if cu[b + 1] > cu[b]:
        segs.append((oracle.bf16_bits_to_f64(k[cu[b]:cu[b + 1]]),
                     oracle.bf16_bits_to_f64(v[cu[b]:cu[b + 1]])))
    for t in range(n_decode_written):
        _, kd, vd, _, _ = w.decode_tokens(t)
        segs.append((oracle.bf16_bits_to_f64(kd[b:b + 1]), oracle.bf16_bits_to_f64(vd[b:b + 1])))
    return segs


def error_stats(got: np.ndarray, ref: np.ndarray):
    d = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    rel = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300)
    return float(d.max()), float(d.mean()), float(rel)
