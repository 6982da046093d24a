"""Document cache manager (``lazy_doc_cache_*``) and the Zipf hit-ratio simulator (CPU only).

The pages' capacity argument ([NOTE] 研究背景与动机, 核心矛盾): under Zipf popularity with D
positions and C entries, a position-free cache holds the top C documents, a position-aware one
only floor(C/D), so hit ratios stand in the ratio sum_{i<=C} i^-a / sum_{i<=floor(C/D)} i^-a.
"""
from fractions import Fraction

import numpy as np
import pytest

lk = pytest.importorskip("position_agnostic_kv_gb300")
from position_agnostic_kv_gb300 import cache_sim  # noqa: E402


def test_hits_misses_and_lru_eviction():
    c = lk.DocCache(6)
    p0, hit = c.acquire(0, 2)
    assert not hit and len(set(p0)) == 2
    p1, hit = c.acquire(1, 2)
    assert not hit and not set(p0) & set(p1)
    p2, _ = c.acquire(2, 2)
    for d in (0, 1, 2):
        c.release(d)
    # a hit returns the same pages and refreshes recency: document 0 is now the most recent
    q0, hit = c.acquire(0, 2)
    assert hit and list(q0) == list(p0)
    c.release(0)
    # a fourth document evicts the least recently used one (document 1) and reuses its pages
    p3, hit = c.acquire(3, 2)
    assert not hit and sorted(p3) == sorted(p1)
    c.release(3)
    assert c.lookup(1) is None and list(c.lookup(0)) == list(p0) and list(c.lookup(2)) == list(p2)
    st = c.stats()
    assert (st["hits"], st["misses"], st["evictions"], st["entries"], st["free_pages"]) == (1, 4, 1, 3, 0)
    assert all(0 <= p < 6 for p in np.concatenate([p0, p2, p3]))


def test_pinned_entries_are_never_evicted():
    c = lk.DocCache(4)
    c.acquire(0, 2)
    c.acquire(1, 2)            # both held by a running batch
    with pytest.raises(lk.LazyError, match="code -2"):
        c.acquire(2, 1)        # no unheld entry to evict
    c.release(1)
    p, hit = c.acquire(2, 1)   # now document 1 goes
    assert not hit and c.lookup(1) is None and c.lookup(0) is not None
    with pytest.raises(lk.LazyError, match="code -1"):
        c.release(7)           # never held
    with pytest.raises(lk.LazyError, match="code -1"):
        c.acquire(0, 3)        # cached with 2 pages
    with pytest.raises(lk.LazyError, match="code -2"):
        c.acquire(9, 5)        # larger than the pool


def test_position_aware_keys_per_position():
    agn, aware = lk.DocCache(8), lk.DocCache(8, position_aware=True)
    for pos in range(3):
        _, hit_a = agn.acquire(5, 1, pos=pos)
        _, hit_w = aware.acquire(5, 1, pos=pos)
        agn.release(5, pos=pos)
        aware.release(5, pos=pos)
        assert hit_a == (pos > 0)   # one copy serves every position
        assert not hit_w            # one copy per (document, position)
    assert agn.stats()["entries"] == 1 and aware.stats()["entries"] == 3


def test_formula_against_exact_harmonic_numbers():
    """alpha = 1: the ratio is H_C / H_{floor(C/D)} with harmonic numbers, summed exactly."""
    H = lambda n: sum(Fraction(1, i) for i in range(1, n + 1))
    assert H(5) == Fraction(137, 60)
    exact = H(100) / H(5)
    assert abs(cache_sim.formula_ratio(1.0, 100, 20) - float(exact)) < 1e-12
    assert cache_sim.formula_ratio(1.3, 50, 1) == 1.0               # one position: no difference
    r = [cache_sim.formula_ratio(0.9, 100, D) for D in (2, 5, 10, 20)]
    assert all(x < y for x, y in zip(r, r[1:]))                     # more positions, larger gap


def test_static_simulation_reproduces_the_formula():
    """Independent Zipf draws at uniform positions, caches filled with the most popular entries:
    each simulated hit ratio is within 4 binomial standard deviations of its closed form, and
    their ratio follows the pages' formula."""
    D, C, n_docs, n = 10, 50, 400, 40000
    for alpha in (0.9, 1.5):
        tr = cache_sim.make_trace(n, n_docs, 1, alpha, seed=7, positions=D)
        p = cache_sim.zipf_probs(n_docs, alpha)
        for aware, expect in ((False, p[:C].sum()), (True, p[: C // D].sum())):
            got = cache_sim.simulate(tr, C, aware, "static", positions=D)
            sd = np.sqrt(expect * (1 - expect) / n)
            assert abs(got - expect) < 4 * sd, (alpha, aware, got, expect)
        ratio = (cache_sim.simulate(tr, C, False, "static", positions=D)
                 / cache_sim.simulate(tr, C, True, "static", positions=D))
        assert abs(ratio / cache_sim.formula_ratio(alpha, C, D) - 1) < 0.05


def test_lru_position_free_cache_hits_more():
    tr = cache_sim.make_trace(300, 200, 10, 1.1, seed=3)
    for C in (20, 60):
        agn = cache_sim.simulate(tr, C, False, "lru")
        aware = cache_sim.simulate(tr, C, True, "lru")
        assert 0 < aware < agn <= 1
