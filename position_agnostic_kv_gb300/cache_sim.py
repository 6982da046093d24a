"""Zipf trace-driven hit-ratio simulator for the document cache manager (``DocCache``).

[NOTE] 研究背景与动机 (核心矛盾): with Zipf document popularity p_i ~ i^-alpha, D possible
positions per document and a budget of C cache entries, a position-free cache can hold the C
most popular documents while a position-aware cache (one copy per (document, position)
variant) holds only floor(C / D) of them, so their hit ratios stand in the ratio
sum_{i<=C} i^-alpha / sum_{i<=floor(C/D)} i^-alpha.  [NOTE] 实验关键数据 (KV 缓存命中率)
reports trace-driven hit ratios under Zipf 1.1 / 1.5 / 2.1; its traces are not available, so
the traces here are synthetic Zipf draws.

Two policies run through the native cache manager:
  * ``static`` -- the cache is filled once with the most popular entries (top C documents, or
    the top floor(C/D) documents at every one of the D positions) and never changes: the
    setting of the formula above;
  * ``lru``    -- every request acquires its documents (misses are assigned pages, evicting the
    least recently used unheld entries) and releases them after the batch.

Usage: ``python -m position_agnostic_kv_gb300.cache_sim [--alpha 1.1] [--docs 500] ...``
"""
from __future__ import annotations

import argparse

import numpy as np

from . import DocCache


def zipf_probs(n_docs: int, alpha: float) -> np.ndarray:
    """Popularity of document rank i = 1..n_docs, proportional to i^-alpha."""
    w = np.arange(1, n_docs + 1, dtype=np.float64) ** -alpha
    return w / w.sum()


def formula_ratio(alpha: float, C: int, D: int) -> float:
    """The pages' hit-ratio ratio of a position-free over a position-aware cache."""
    i = np.arange(1, C + 1, dtype=np.float64)
    return float((i ** -alpha).sum() / (i[: C // D] ** -alpha).sum())


def make_trace(n_requests: int, n_docs: int, docs_per_request: int, alpha: float, seed: int = 0,
               positions: int | None = None):
    """Requests of `docs_per_request` distinct documents drawn by Zipf popularity (document id
    = popularity rank - 1).  By default they are placed in a random order (position = index in
    the request, D = docs_per_request); with `positions` = D each document's position is drawn
    uniformly from 0..D-1 instead (independent draws: with one document per request this is the
    independent-reference setting of the formula).  Returns int32 [n_requests, k, 2] of
    (document, position)."""
    rng = np.random.default_rng(seed)
    p = zipf_probs(n_docs, alpha)
    out = np.zeros((n_requests, docs_per_request, 2), np.int32)
    for r in range(n_requests):
        out[r, :, 0] = rng.choice(n_docs, size=docs_per_request, replace=False, p=p)
        out[r, :, 1] = (rng.permutation(docs_per_request) if positions is None
                        else rng.integers(0, positions, docs_per_request))
    return out


def simulate(trace: np.ndarray, capacity_entries: int, position_aware: bool, policy: str = "lru",
             pages_per_doc: int = 1, positions: int | None = None) -> float:
    """Hit ratio (hits / lookups) of the trace against a cache of `capacity_entries` documents'
    worth of pages."""
    cache = DocCache(capacity_entries * pages_per_doc, position_aware=position_aware)
    D = positions if positions is not None else trace.shape[1]
    if policy == "static":
        # fill with the most popular entries: ranks 0.. (every position for a position-aware
        # cache), then only look up
        n_docs = capacity_entries // (D if position_aware else 1)
        for d in range(n_docs):
            for p in (range(D) if position_aware else [0]):
                cache.acquire(d, pages_per_doc, pos=p)
        hits = sum(cache.lookup(int(d), int(p)) is not None for req in trace for d, p in req)
        cache.close()
        return hits / trace.shape[0] / trace.shape[1]
    if policy != "lru":
        raise ValueError(f"unknown policy {policy}")
    for req in trace:
        for d, p in req:
            cache.acquire(int(d), pages_per_doc, pos=int(p))
        for d, p in req:
            cache.release(int(d), pos=int(p))
    st = cache.stats()
    cache.close()
    return st["hits"] / (st["hits"] + st["misses"])


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--alpha", type=float, nargs="+", default=[1.1, 1.5, 2.1])
    ap.add_argument("--docs", type=int, default=500, help="document pool size")
    ap.add_argument("--per-request", type=int, default=20, help="documents per request (= positions D)")
    ap.add_argument("--budgets", type=int, nargs="+", default=[20, 100, 200], help="cache budgets in documents")
    ap.add_argument("--requests", type=int, default=2000)
    ap.add_argument("--seed", type=int, default=0)
    a = ap.parse_args()
    D = a.per_request
    print(f"D = {D} positions, pool of {a.docs} documents")
    print(f"{'alpha':>6} {'budget':>7} {'formula':>8} | independent draws, static: {'agn':>7} {'aware':>7} "
          f"{'ratio':>6} | RAG requests, LRU: {'agn':>7} {'aware':>7} {'ratio':>6}")
    for alpha in a.alpha:
        irm = make_trace(a.requests * D, a.docs, 1, alpha, a.seed, positions=D)
        rag = make_trace(a.requests, a.docs, D, alpha, a.seed)
        for C in a.budgets:
            sa = simulate(irm, C, False, "static", positions=D)
            sw = simulate(irm, C, True, "static", positions=D)
            la = simulate(rag, C, False, "lru")
            lw = simulate(rag, C, True, "lru")
            print(f"{alpha:6.2f} {C:7d} {formula_ratio(alpha, C, D):8.3f} | {'':26s}{sa:7.4f} {sw:7.4f} "
                  f"{sa / max(sw, 1e-12):6.3f} | {'':18s}{la:7.4f} {lw:7.4f} {la / max(lw, 1e-12):6.2f}")


if __name__ == "__main__":
    main()
