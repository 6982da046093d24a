"""Shared pieces of the GPU parity tests (test infrastructure)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests.oracle_setup import error_stats

# Tolerances: the attention outputs must match within max-abs 2e-2 and mean-abs 2e-3 (bf16
# inputs, fp32 accumulation); the relative Frobenius error bound 1e-2 is added because N(0,1)
# data over long contexts gives |O| ~ 1e-2, where max-abs alone would not separate a wrong
# kernel from a right one.
TOL_MAX, TOL_MEAN, TOL_REL = 2e-2, 2e-3, 1e-2


def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_gb300 as m
    return m


def assert_close(got, ref, what, tol_max=TOL_MAX, tol_mean=TOL_MEAN, tol_rel=TOL_REL):
    g = got.float().cpu().numpy().astype(np.float64) if hasattr(got, "cpu") else np.asarray(got)
    mx, mean, rel = error_stats(g, ref)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    assert mx <= tol_max and mean <= tol_mean and rel <= tol_rel, \
        f"{what}: max-abs {mx:.3e} mean-abs {mean:.3e} rel {rel:.3e}"
    return mx, mean, rel


def oracle_caches_for(w, instances=None, prefill=True, decode_steps=0):
    """Oracle-written caches holding the given document copies (all by default), the prefill
    tokens, and decode tokens 0..decode_steps-1."""
    shape = (w.num_pages, w.Hkv, oracle.PAGE, w.D)
    kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    pos = w.pos.as_dict()
    insts = range(len(w.inst_doc)) if instances is None else instances
    for i in insts:
        k, v = w.doc_kv(int(w.inst_doc[i]))
        slot, lp = w.inst_slots(i)
        oracle.kv_write(k, v, slot, lp, pos, kc, vc)
    if prefill:
        q, k, v, slot, lp = w.prefill_tokens()
        if len(slot):
            oracle.kv_write(k, v, slot, lp, pos, kc, vc)
    for t in range(decode_steps):
        _, k, v, slot, lp = w.decode_tokens(t)
        oracle.kv_write(k, v, slot, lp, pos, kc, vc)
    return kc, vc


def request_instances(w, reqs):
    return sorted({int(i) for b in reqs for i in w.req_inst[w.req_inst_off[b]:w.req_inst_off[b + 1]]})
