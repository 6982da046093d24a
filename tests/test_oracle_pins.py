"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties a part of ``oracle`` to a fact fixed by the pages or by mathematics: the
rotation formula the pages print, a complex-number restatement of RoPE, the RoPE relative
identity, brute force over tiny inputs with explicit loops, torch's fp64 scaled-dot-product
attention with an explicit mask, closed forms (ALiBi geometric weights, YaRN limits),
permutation invariants, and Example 3.1's sign convention.  The sources are the LazyAttention
pages: the papernotes.org reading note [NOTE] (sections 切入角度, 整体框架 with Example 3.1,
关键设计, 通用性) and the gist.science summary [GIST] (Equivalenza Matematica).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import lazy_oracle as lo
from workloads import PosCfg, make_custom, make_workload
from tests.oracle_setup import (empty_caches, oracle_fill_docs, oracle_meta,
                                oracle_write_decode, oracle_write_prefill, raw_segments)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(2024)


# ------------------------------------------------------------------ rotation
def test_rotation_formula_printed_on_the_pages():
    """[NOTE] 关键设计 prints k'1 = k1 cos D - k2 sin D, k'2 = k1 sin D + k2 cos D.
    With one pair (d = 2, theta_0 = 1) and unit vectors the result is read off directly."""
    inv = np.array([1.0])
    for delta in (0.0, 1.0, 2.5, -0.75):
        np.testing.assert_allclose(lo.rotate(np.array([1.0, 0.0]), delta, inv),
                                   [math.cos(delta), math.sin(delta)], atol=1e-15)
        np.testing.assert_allclose(lo.rotate(np.array([0.0, 1.0]), delta, inv),
                                   [-math.sin(delta), math.cos(delta)], atol=1e-15)
    # literal values for delta = 1 rad
    np.testing.assert_allclose(lo.rotate(np.array([1.0, 0.0]), 1.0, inv),
                               [0.5403023058681398, 0.8414709848078965], rtol=0, atol=1e-15)


def test_rotation_equals_complex_multiplication():
    """Half-split RoPE is z_i * exp(i p theta_i) on z_i = x_i + i x_{i+d/2}."""
    d = 64
    inv = lo.rope_inv_freq(d, 1e4)
    x = RNG.standard_normal((5, d))
    p = np.array([0, 1, 17, 1000, 123456])
    z = x[:, : d // 2] + 1j * x[:, d // 2:]
    zr = z * np.exp(1j * p[:, None] * inv[None, :])
    got = lo.rotate(x, p, inv)
    np.testing.assert_allclose(got[:, : d // 2], zr.real, atol=1e-9)
    np.testing.assert_allclose(got[:, d // 2:], zr.imag, atol=1e-9)


def test_interleaved_rotation_equals_complex_multiplication():
    """Interleaved (GPT-J) RoPE is z_i * exp(i p theta_i) on z_i = x_{2i} + i x_{2i+1}; with a
    partial rotary dimension d < D the dimensions from d on are untouched."""
    D, d = 64, 32
    inv = lo.rope_inv_freq(d, 1e4)
    x = RNG.standard_normal((5, D))
    p = np.array([0, 1, 17, 1000, 123456])
    z = x[:, 0:d:2] + 1j * x[:, 1:d:2]
    zr = z * np.exp(1j * p[:, None] * inv[None, :])
    got = lo.rotate(x, p, inv, interleaved=True)
    np.testing.assert_allclose(got[:, 0:d:2], zr.real, atol=1e-9)
    np.testing.assert_allclose(got[:, 1:d:2], zr.imag, atol=1e-9)
    np.testing.assert_array_equal(got[:, d:], x[:, d:])
    half = lo.rotate(x, p, inv)
    zh = x[:, : d // 2] + 1j * x[:, d // 2: d]
    np.testing.assert_allclose(half[:, : d // 2] + 1j * half[:, d // 2: d],
                               zh * np.exp(1j * p[:, None] * inv[None, :]), atol=1e-9)
    np.testing.assert_array_equal(half[:, d:], x[:, d:])


@pytest.mark.parametrize("inter", [False, True])
def test_relative_identity_partial_and_interleaved(inter):
    """(R_m q)^T (R_n k) = q^T R_{n-m} k also for interleaved pairs and partial rotary_dim (the
    unrotated tail contributes its plain dot product); theta_i uses the rotary dimension."""
    D, d = 128, 64
    inv = lo.rope_inv_freq(d, 5e5)
    assert abs(inv[d // 4] - 1.0 / math.sqrt(5e5)) < 1e-17
    for _ in range(20):
        q, k = RNG.standard_normal(D), RNG.standard_normal(D)
        m, n = RNG.integers(0, 200_000, size=2)
        lhs = lo.rotate(q, m, inv, inter) @ lo.rotate(k, n, inv, inter)
        rhs = q @ lo.rotate(k, n - m, inv, inter)
        assert abs(lhs - rhs) <= 1e-9 * (np.linalg.norm(q) * np.linalg.norm(k))
        np.testing.assert_allclose(lo.rotate(lo.rotate(k, m, inv, inter), n, inv, inter),
                                   lo.rotate(k, m + n, inv, inter), atol=1e-9)


def test_inv_freq_special_values():
    """theta_0 = 1 and theta_{d/4} = base^(-1/2); strictly decreasing."""
    t = lo.rope_inv_freq(64, 1e4)
    assert t[0] == 1.0
    assert abs(t[16] - 0.01) < 1e-16
    t = lo.rope_inv_freq(128, 5e5)
    assert abs(t[32] - 1.0 / math.sqrt(5e5)) < 1e-17
    assert np.all(np.diff(t) < 0)


def test_relative_identity():
    """[NOTE] 切入角度: (R_m q)^T (R_n k) = q^T R_{n-m} k, for m, n up to 2e5.

    Bound: each angle up to 2e5 rad carries ~2e5 * 2^-53 rad of rounding, so the dot product of
    128-dim N(0,1) vectors agrees to ~1e-9 relative (not 1e-12)."""
    d = 128
    inv = lo.rope_inv_freq(d, 5e5)
    for _ in range(50):
        q, k = RNG.standard_normal(d), RNG.standard_normal(d)
        m, n = RNG.integers(0, 200_000, size=2)
        lhs = lo.rotate(q, m, inv) @ lo.rotate(k, n, inv)
        rhs = q @ lo.rotate(k, n - m, inv)
        assert abs(lhs - rhs) <= 1e-9 * (np.linalg.norm(q) * np.linalg.norm(k))


def test_rotation_composition():
    """R_Delta R_j = R_{Delta + j}: one relative rotation of a locally rotated key lands at the
    absolute position ([NOTE] 关键设计: a single relative rotation, not un-rotate/re-rotate)."""
    d = 128
    inv = lo.rope_inv_freq(d, 1e4)
    k = RNG.standard_normal((20, d))
    j = RNG.integers(0, 2000, size=20)
    delta = RNG.integers(0, 40000, size=20)
    a = lo.rotate(lo.rotate(k, j, inv), delta, inv)
    b = lo.rotate(k, j + delta, inv)
    np.testing.assert_allclose(a, b, atol=1e-10)


def test_yarn_limits():
    """YaRN: s = 1 is plain RoPE; pairs with wavelength < L0/beta_fast keep theta; pairs with
    wavelength > L0/beta_slow get theta/s; mscale(1) = 1 and mscale(e^10) = 2."""
    d, base = 128, 5e5
    t = lo.rope_inv_freq(d, base)
    np.testing.assert_allclose(lo.yarn_inv_freq(d, base, 1.0, 8192), t, rtol=4e-16)
    y = lo.yarn_inv_freq(d, base, 8.0, 8192, 32.0, 1.0)
    lam = 2 * np.pi / t
    hi = lam < 8192 / 32.0
    lo_ = lam > 8192 / 1.0
    assert hi.any() and lo_.any()
    np.testing.assert_allclose(y[hi], t[hi], rtol=1e-15)
    np.testing.assert_allclose(y[lo_], t[lo_] / 8.0, rtol=1e-15)
    mid = ~(hi | lo_)
    assert np.all((y[mid] <= t[mid]) & (y[mid] >= t[mid] / 8.0))
    assert lo.yarn_mscale(1.0) == 1.0
    assert abs(lo.yarn_mscale(math.exp(10.0)) - 2.0) < 1e-15


@pytest.mark.parametrize("s", [8.0, 4.0, 2.5])
def test_yarn_ramp_interior_closed_form(s):
    """Inside the ramp the interpolated frequency is fixed by hand arithmetic.  With
    rotary_dim = 2 the only frequency is theta_0 = base^0 = 1 (wavelength 2 pi) for any base, so
    L0 = 33 pi gives r = L0 / lambda = 16.5 and gamma = (16.5 - 1) / (32 - 1) = 1/2, hence
    theta' = (1/s + 1) / 2; L0 = 17.5 pi gives r = 8.75, gamma = 1/4, theta' = 3/(4s) + 1/4.
    A ramp divided by beta_fast alone, one that forgets beta_slow, or one that interpolates
    wavelengths instead of frequencies gives other numbers at both points."""
    for base in (1e4, 5e5):
        y = lo.yarn_inv_freq(2, base, s, 33.0 * math.pi, 32.0, 1.0)
        assert y.shape == (1,)
        np.testing.assert_allclose(y[0], 0.5 * (1.0 / s + 1.0), rtol=1e-14)
        y = lo.yarn_inv_freq(2, base, s, 17.5 * math.pi, 32.0, 1.0)
        np.testing.assert_allclose(y[0], 0.75 / s + 0.25, rtol=1e-14)
    # rotary_dim = 4, base 4: theta = (1, 1/2), wavelengths (2 pi, 4 pi).  L0 = 66 pi puts pair 0
    # above beta_fast (r = 33: theta kept) and pair 1 mid-ramp (r = 16.5: gamma = 1/2).
    y = lo.yarn_inv_freq(4, 4.0, s, 66.0 * math.pi, 32.0, 1.0)
    np.testing.assert_allclose(y, [1.0, 0.5 * (0.5 / s + 0.5)], rtol=1e-14)
    # L0 = pi: r = 1/2 and 1/4, both below beta_slow: every frequency divided by s
    y = lo.yarn_inv_freq(4, 4.0, s, math.pi, 32.0, 1.0)
    np.testing.assert_allclose(y, [1.0 / s, 0.5 / s], rtol=1e-14)
    # other ramp bounds: beta (16, 2), r = 9 -> gamma = (9 - 2) / 14 = 1/2
    y = lo.yarn_inv_freq(2, 1e4, s, 18.0 * math.pi, 16.0, 2.0)
    np.testing.assert_allclose(y[0], 0.5 * (1.0 / s + 1.0), rtol=1e-14)


def test_yarn_ramp_pins_catch_plausible_slips():
    """Negative control for the pins above: the slips named there each miss the closed form."""
    s, theta, lam = 8.0, 1.0, 2.0 * math.pi
    r = 33.0 * math.pi / lam
    want = 0.5 * (1.0 / s + 1.0)
    slips = {
        "divide by beta_fast": np.clip((r - 1.0) / 32.0, 0, 1),
        "forget beta_slow": np.clip(r / 31.0, 0, 1),
    }
    for name, g in slips.items():
        assert abs((1 - g) * theta / s + g * theta - want) > 1e-3, name
    g = 0.5  # interpolating the wavelength instead of the frequency
    assert abs(2 * math.pi / ((1 - g) * lam * s + g * lam) - want) > 1e-3


def test_alibi_slopes_values():
    """2^(-8h/32): h = 1 gives 2^-0.25, h = 32 gives 1/256; the workload's input copy agrees."""
    s = lo.alibi_slopes(32)
    assert abs(s[0] - 0.8408964152537145) < 1e-15
    assert s[-1] == 1.0 / 256.0
    w = make_workload("mqa_alibi", batch=1)
    np.testing.assert_allclose(w.pos.alibi_slopes, s, rtol=1e-7)


# ------------------------------------------------------------------ bf16
def test_bf16_rounding_known_values():
    cases = [(1.0, 1.0), (1 + 2 ** -8, 1.0), (1 + 3 * 2 ** -8, 1 + 2 ** -6),
             (1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -7), (-2.5, -2.5), (3.14159, 3.140625),
             (0.0, 0.0), (-(1 + 2 ** -8), -1.0)]
    for x, want in cases:
        assert lo.round_to_bf16(np.array(x)) == want, x


def test_bf16_rounding_matches_torch():
    """For fp32-representable inputs torch's fp32 -> bf16 cast rounds to nearest-even too."""
    x = RNG.standard_normal(100000).astype(np.float32).astype(np.float64) * 7.3
    ours = lo.round_to_bf16(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)


# ------------------------------------------------------------------ block words
def test_meta_bit_layout_hand_values():
    assert lo.pack_meta(16, 0, 0, 0) == 16
    assert lo.pack_meta(1, 1, 1, 1) == 1 + 32 + 65536 + 2 ** 40
    assert lo.pack_meta(31, 2047, 2 ** 24 - 1, 2 ** 24 - 1) == 2 ** 64 - 1
    assert lo.pack_meta(8, 12, 2000, 77) == 8 | (12 << 5) | (2000 << 16) | (77 << 40)
    for _ in range(200):
        f = (int(RNG.integers(0, 32)), int(RNG.integers(0, 2048)),
             int(RNG.integers(0, 2 ** 24)), int(RNG.integers(0, 2 ** 24)))
        assert lo.unpack_meta(lo.pack_meta(*f)) == f
    for bad in [(32, 0, 0, 0), (0, 2048, 0, 0), (0, 0, 2 ** 24, 0), (0, 0, 0, 2 ** 24)]:
        with pytest.raises(OverflowError):
            lo.pack_meta(*bad)


def test_build_meta_hand_case():
    """Two documents (48 and 17 tokens) then a 20-token query capacity, written out by hand."""
    doc_len = np.array([48, 17])
    doc_page_off = np.array([0, 3, 5])
    doc_pages = np.array([9, 4, 7, 2, 11])
    bt, meta, seq_len, q_start, doc_blocks = lo.build_meta(
        np.array([0, 2]), np.array([0, 1]), doc_len, doc_page_off, doc_pages,
        np.array([5]), np.array([0, 2]), np.array([6, 3]), max_blocks=8)
    want = [(16, 0, 0, 9), (16, 1, 0, 4), (16, 2, 0, 7), (16, 0, 48, 2), (1, 1, 48, 11),
            (16, 0, 65, 6), (16, 1, 65, 3)]
    assert [lo.unpack_meta(w) for w in meta[0, :7]] == want
    assert meta[0, 7] == 0
    assert list(bt[0]) == [9, 4, 7, 2, 11, 6, 3, 0]
    assert (seq_len[0], q_start[0], doc_blocks[0]) == (70, 65, 5)


@pytest.mark.parametrize("name", ["tiny", "rag8b", "mqa_alibi"])
def test_build_meta_invariants(name):
    """Positions reached through the words are exactly 0 .. q_start-1 for the documents, then
    the query segment; Delta is constant within a document and non-decreasing; pg counts from
    0 within a document; the block table equals the page field."""
    w = make_workload(name)
    bt, meta, seq_len, q_start, doc_blocks = oracle_meta(w)
    for b in range(w.B):
        f = [lo.unpack_meta(x) for x in meta[b]]
        pos = []
        for j in range(doc_blocks[b]):
            nv, pg, dl, pg_id = f[j]
            pos.extend(dl + 16 * pg + t for t in range(nv))
            assert bt[b, j] == pg_id
        assert pos == list(range(q_start[b]))
        deltas = [x[2] for x in f[: doc_blocks[b]]]
        assert deltas == sorted(deltas)
        assert q_start[b] == int(w.doc_len[w.request_docs(b)].sum())
        assert seq_len[b] == q_start[b] + w.q_len[b]
        nq = w.q_page_off[b + 1] - w.q_page_off[b]
        for j in range(doc_blocks[b], doc_blocks[b] + nq):
            assert f[j][0] == 16 and f[j][2] == q_start[b]
        assert all(x == 0 for x in meta[b, doc_blocks[b] + nq:])


# ------------------------------------------------------------------ kv write
def test_kv_write_local_position_zero_is_identity_and_rounding():
    w = make_custom([20], [[0]], 4, 2, 64, PosCfg("rope", 1e4, 64), 0, 0)
    kc, vc = empty_caches(w)
    k, v = w.doc_kv(0)
    slot, lp = w.inst_slots(0)
    lo.kv_write(k, v, slot, lp, w.pos.as_dict(), kc, vc)
    page, row = slot // 16, slot % 16
    np.testing.assert_array_equal(kc[page[0], :, row[0]], k[0])       # R_0 k = k, bit-exact
    np.testing.assert_array_equal(vc[page, :, row], v)
    exact = lo.rotate(lo.bf16_bits_to_f64(k), lp[:, None], lo.rope_inv_freq(64, 1e4))
    stored = lo.bf16_bits_to_f64(kc[page, :, row])
    ulp = 2.0 ** (np.floor(np.log2(np.abs(exact) + 1e-300)) - 7)
    assert np.all(np.abs(stored - exact) <= 0.5 * ulp + 1e-300)


# ------------------------------------------------------------------ attention definitions
def _exact_caches(w):
    """Caches holding R_j k in exact fp64 (no bf16 rounding), for 1e-12 comparisons."""
    kc = np.zeros((w.num_pages, w.Hkv, 16, w.D))
    vc = np.zeros_like(kc)
    inv = lo.pos_inv_freq(w.pos.as_dict())
    def put(k, v, slot, lp):
        kk = lo.bf16_bits_to_f64(k)
        if inv is not None:
            kk = lo.rotate(kk, np.asarray(lp)[:, None], inv, w.pos.interleaved)
        kc[slot // 16, :, slot % 16] = kk
        vc[slot // 16, :, slot % 16] = lo.bf16_bits_to_f64(v)
    for i in range(len(w.inst_doc)):
        k, v = w.doc_kv(int(w.inst_doc[i]))
        put(k, v, *w.inst_slots(i))
    q, k, v, slot, lp = w.prefill_tokens()
    if len(slot):
        put(k, v, slot, lp)
    return kc, vc, q


EDGE_CASES = [
    ([1, 15, 17], [[0, 1, 2]], 4, 2, 8, 3, 2),
    ([17, 1, 16, 33], [[3, 1], [0, 2, 1]], 4, 2, 8, [2, 5], 3),
    ([5], [[0]], 2, 2, 8, 1, 4),
]


@pytest.mark.parametrize("kind", ["rope", "yarn", "alibi", "rope_partial", "rope_interleaved"])
@pytest.mark.parametrize("case", range(len(EDGE_CASES)))
def test_paged_oracle_equals_brute_force_loops(case, kind):
    """The paged route (block words, R_Delta on local-rotated K) equals an explicit-loop full
    recompute of the concatenated prompt at absolute positions ([NOTE] 整体框架;
    [GIST] Equivalenza Matematica), for prefill rows and for the decode rows."""
    doc_len, req_docs, Hq, Hkv, D, q_len, n_dec = EDGE_CASES[case]
    pos = {"rope": PosCfg("rope", 1e4, D),
           "rope_partial": PosCfg("rope", 1e4, D // 2),
           "rope_interleaved": PosCfg("yarn", 1e4, D, yarn_factor=4.0, yarn_orig_ctx=32, interleaved=True),
           "yarn": PosCfg("yarn", 5e5, D, yarn_factor=8.0, yarn_orig_ctx=64),
           "alibi": PosCfg("alibi", rotary_dim=D,
                           alibi_slopes=lo.alibi_slopes(Hq).astype(np.float32))}[kind]
    w = make_custom(doc_len, req_docs, Hq, Hkv, D, pos, q_len, n_dec, seed=7 + case)
    kc, vc, q = _exact_caches(w)
    bt, meta, seq_len, q_start, doc_blocks = oracle_meta(w)
    out, _ = lo.prefill(q, w.cu_q, q_start, doc_blocks, meta, kc, vc, w.pos.as_dict())
    cu = w.cu_q
    for b in range(w.B):
        if cu[b + 1] == cu[b]:
            continue
        m = q_start[b] + np.arange(cu[b + 1] - cu[b])
        ref = lo.full_recompute_loops(raw_segments(w, b, 0), lo.bf16_bits_to_f64(q[cu[b]:cu[b + 1]]),
                                      m, w.pos.as_dict())
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ref, atol=1e-12, rtol=0)
    # decode steps
    inv = lo.pos_inv_freq(w.pos.as_dict())
    for t in range(n_dec):
        qd, kd, vd, slot, lp = w.decode_tokens(t)
        kk = lo.bf16_bits_to_f64(kd)
        if inv is not None:
            kk = lo.rotate(kk, lp[:, None], inv, w.pos.interleaved)
        kc[slot // 16, :, slot % 16] = kk
        vc[slot // 16, :, slot % 16] = lo.bf16_bits_to_f64(vd)
        sl = q_start + w.q_len + t + 1
        od, _ = lo.decode(qd, sl, q_start, doc_blocks, meta, kc, vc, w.pos.as_dict())
        for b in range(w.B):
            ref = lo.full_recompute_loops(raw_segments(w, b, t + 1),
                                          lo.bf16_bits_to_f64(qd[b:b + 1]), [sl[b] - 1],
                                          w.pos.as_dict())
            np.testing.assert_allclose(od[b:b + 1], ref, atol=1e-12, rtol=0)


def test_against_torch_sdpa_bottom_right_mask():
    """Textbook attention equals torch's fp64 scaled_dot_product_attention given an explicit
    bottom-right-aligned causal mask (query rows are the LAST rows of the key sequence)."""
    M, N, Hq, Hkv, D = 7, 40, 6, 2, 16
    q = RNG.standard_normal((M, Hq, D))
    k = RNG.standard_normal((N, Hkv, D))
    v = RNG.standard_normal((N, Hkv, D))
    qp = np.arange(N - M, N)
    kp = np.arange(N)
    out, lse = lo.softmax_attention(q, qp, k, v, kp, 0.3)
    G = Hq // Hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(np.repeat(k, G, axis=1)).permute(1, 0, 2)
    tv = torch.from_numpy(np.repeat(v, G, axis=1)).permute(1, 0, 2)
    mask = torch.from_numpy(kp[None, :] <= qp[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.3)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-13)
    logits = 0.3 * np.einsum("hmd,hnd->hmn", tq.numpy(), tk.numpy())
    logits = np.where(mask.numpy()[None], logits, -np.inf)
    ref_lse = np.log(np.exp(logits).sum(-1)).T
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_alibi_geometric_closed_form():
    """q = 0 leaves only the ALiBi bias -slope (m - p); with v[p] = p the output is the mean of
    p under weights r^(m-p), r = e^-slope, a ratio of two geometric sums in closed form."""
    m, D = 37, 4
    slopes = np.array([0.5, 0.125])
    q = np.zeros((1, 2, D))
    k = RNG.standard_normal((m + 1, 1, D))
    v = np.repeat(np.arange(m + 1, dtype=np.float64)[:, None, None], D, axis=2)
    out, _ = lo.softmax_attention(q, [m], k, v, np.arange(m + 1), 1.0, slopes)
    for h, s in enumerate(slopes):
        r = math.exp(-s)
        S0 = (1 - r ** (m + 1)) / (1 - r)
        S1 = r * (1 - (m + 1) * r ** m + m * r ** (m + 1)) / (1 - r) ** 2
        np.testing.assert_allclose(out[0, h], (m * S0 - S1) / S0, rtol=1e-13)


def test_special_cases():
    """One document at Delta = 0 is standard RoPE attention; ALiBi with zero slopes is plain
    attention; V = c gives O = c; MHA with replicated KV heads equals GQA."""
    D = 16
    w = make_custom([40], [[0]], 4, 2, D, PosCfg("rope", 1e4, D), 9, 0, seed=3)
    kc, vc, q = _exact_caches(w)
    bt, meta, sl, qs, db = oracle_meta(w)
    out, _ = lo.prefill(q, w.cu_q, qs, db, meta, kc, vc, w.pos.as_dict())
    segs = raw_segments(w, 0, 0)
    kraw = np.concatenate([s[0] for s in segs])
    vraw = np.concatenate([s[1] for s in segs])
    inv = lo.rope_inv_freq(D, 1e4)
    p = np.arange(kraw.shape[0])
    m = 40 + np.arange(9)
    ref, _ = lo.softmax_attention(lo.rotate(lo.bf16_bits_to_f64(q), m[:, None], inv), m,
                                  lo.rotate(kraw, p[:, None], inv), vraw, p, 1 / 4.0)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    # ALiBi with zero slopes == no positional term at all
    qq = RNG.standard_normal((3, 4, D))
    kk = RNG.standard_normal((10, 2, D))
    vv = RNG.standard_normal((10, 2, D))
    a, _ = lo.softmax_attention(qq, [7, 8, 9], kk, vv, np.arange(10), 0.25, np.zeros(4))
    b_, _ = lo.softmax_attention(qq, [7, 8, 9], kk, vv, np.arange(10), 0.25)
    np.testing.assert_array_equal(a, b_)
    # V constant
    c, _ = lo.softmax_attention(qq, [7, 8, 9], kk, np.full_like(vv, 2.5), np.arange(10), 0.25)
    np.testing.assert_allclose(c, 2.5, atol=1e-14)
    # MHA with replicated heads
    mha, _ = lo.softmax_attention(qq, [7, 8, 9], np.repeat(kk, 2, axis=1),
                                  np.repeat(vv, 2, axis=1), np.arange(10), 0.25)
    np.testing.assert_allclose(mha, b_, atol=1e-14)


def test_yarn_factor_one_is_plain_rope():
    D = 16
    wr = make_custom([23, 9], [[0, 1]], 4, 2, D, PosCfg("rope", 5e5, D), 4, 0, seed=11)
    wy = make_custom([23, 9], [[0, 1]], 4, 2, D,
                     PosCfg("yarn", 5e5, D, yarn_factor=1.0, yarn_orig_ctx=64), 4, 0, seed=11)
    outs = []
    for w in (wr, wy):
        kc, vc, q = _exact_caches(w)
        bt, meta, sl, qs, db = oracle_meta(w)
        outs.append(lo.prefill(q, w.cu_q, qs, db, meta, kc, vc, w.pos.as_dict())[0])
    np.testing.assert_allclose(outs[0], outs[1], atol=1e-12)


# ------------------------------------------------------------------ invariants
def test_permutation_invariance_pages_and_docs():
    """(i) Moving pages physically and reordering the block list while each block keeps its
    (Delta, pg) leaves the output unchanged.  (ii) Reordering the documents changes the output
    only through Delta: it equals a full recompute of the reordered prompt."""
    D = 16
    pos = PosCfg("rope", 1e4, D)
    w = make_custom([30, 17, 9], [[0, 1, 2]], 4, 2, D, pos, 5, 0, seed=5)
    kc, vc, q = _exact_caches(w)
    bt, meta, sl, qs, db = oracle_meta(w)
    base, _ = lo.prefill(q, w.cu_q, qs, db, meta, kc, vc, pos.as_dict())
    # (i) permute physical pages and the order of the block words
    perm = RNG.permutation(w.num_pages)
    kc2, vc2 = np.zeros_like(kc), np.zeros_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    nb = lo.visible_blocks(db[0], qs[0], qs[0] + 4)
    words = []
    for x in meta[0, :nb]:
        nv, pg, dl, page = lo.unpack_meta(x)
        words.append(lo.pack_meta(nv, pg, dl, int(perm[page])))
    order = RNG.permutation(nb)
    meta2 = np.zeros_like(meta)
    meta2[0, :nb] = np.array(words, dtype=np.uint64)[order]
    m = qs[0] + np.arange(5)
    got, _ = lo.attend_paged(lo.as_f64(q), m, meta2[0], nb, kc2, vc2, pos.as_dict())
    np.testing.assert_allclose(got, base, atol=1e-12)
    # (ii) reorder documents: same cache, new Delta from the packer
    w2 = make_custom([30, 17, 9], [[2, 0, 1]], 4, 2, D, pos, 5, 0, seed=5)
    kcb, vcb, qb = _exact_caches(w2)
    _, meta_b, _, qs_b, db_b = oracle_meta(w2)
    out_b, _ = lo.prefill(qb, w2.cu_q, qs_b, db_b, meta_b, kcb, vcb, pos.as_dict())
    ref_b, _ = lo.materialized_attention(raw_segments(w2, 0, 0), lo.as_f64(qb), m, pos.as_dict())
    np.testing.assert_allclose(out_b, ref_b, atol=1e-12)
    assert np.abs(out_b - base).max() > 1e-3


def test_example_3_1_sign_convention():
    """Example 3.1: for d1 || d2 || Q, using d2's cache C2 (indexed from 0) means rotating Q
    BACKWARDS by |d1|: (R_{m-|d1|} q) . (R_j k) equals the full-recompute score
    (R_m q) . (R_{|d1|+j} k); rotating forwards does not."""
    with open(os.path.join(GOLDEN, "example_3_1.json")) as f:
        ex = json.load(f)
    L1, L2, D = ex["d1_len"], ex["d2_len"], ex["head_dim"]
    inv = lo.rope_inv_freq(D, ex["rope_theta"])
    k2 = RNG.standard_normal((L2, D))
    q = RNG.standard_normal(D)
    m = L1 + L2 + ex["query_offset"]
    c2 = lo.rotate(k2, np.arange(L2), inv)                  # cache of d2, from 0
    full = lo.rotate(k2, L1 + np.arange(L2), inv) @ lo.rotate(q, m, inv)
    back = c2 @ lo.rotate(q, m - L1, inv)
    fwd = c2 @ lo.rotate(q, m + L1, inv)
    np.testing.assert_allclose(back, full, atol=1e-10)
    assert np.abs(fwd - full).max() > 1e-2


def test_negative_controls_are_separated():
    """Wrong metadata must move the output well beyond the GPU tolerance (max-abs 2e-2), so a
    kernel that ignored Delta, was off by one, or rotated twice cannot pass the parity tests
    (checked with queries sharpened x4, as the parity tests also do)."""
    w = make_workload("tiny")
    kc, vc = empty_caches(w)
    oracle_fill_docs(w, kc, vc)
    q = oracle_write_prefill(w, kc, vc)
    q4 = lo.f64_to_bf16_bits(4.0 * lo.bf16_bits_to_f64(q))
    bt, meta, sl, qs, db = oracle_meta(w)
    pos = w.pos.as_dict()
    good, _ = lo.prefill(q4, w.cu_q, qs, db, meta, kc, vc, pos)

    def with_delta(fn):
        m2 = meta.copy()
        for j in range(meta.shape[1]):
            nv, pg, dl, page = lo.unpack_meta(meta[0, j])
            if nv:
                m2[0, j] = lo.pack_meta(nv, pg, fn(dl), page)
        return lo.prefill(q4, w.cu_q, qs, db, m2, kc, vc, pos)[0]
    for fn in (lambda d: 0, lambda d: d + 1, lambda d: 2 * d):
        assert np.abs(with_delta(fn) - good).max() > 2e-2


def test_lse_and_row_sums():
    qq = RNG.standard_normal((4, 2, 8))
    kk = RNG.standard_normal((12, 1, 8))
    vv = np.ones((12, 1, 8))
    o, lse = lo.softmax_attention(qq, [8, 9, 10, 11], kk, vv, np.arange(12), 0.5)
    np.testing.assert_allclose(o, 1.0, atol=1e-14)        # rows of the softmax sum to one
    s = 0.5 * np.einsum("mhd,nd->mhn", qq, kk[:, 0])
    for r, mm in enumerate([8, 9, 10, 11]):
        ref = np.log(np.exp(s[r, :, : mm + 1]).sum(-1))
        np.testing.assert_allclose(lse[r], ref, atol=1e-13)


def test_decode_oracle_on_tiny_matches_materialized():
    """End-to-end definition on the tiny workload: caches written by the oracle's kv_write
    (bf16 rounding of R_j k) versus the materialised fp64 recompute from raw keys; agreement is
    limited only by bf16 rounding of the stored keys."""
    w = make_workload("tiny")
    kc, vc = empty_caches(w)
    oracle_fill_docs(w, kc, vc)
    oracle_write_prefill(w, kc, vc)
    bt, meta, sl, qs, db = oracle_meta(w)
    for t in range(w.n_decode):
        qd = oracle_write_decode(w, t, kc, vc)
        cur = sl + t + 1
        od, _ = lo.decode(qd, cur, qs, db, meta, kc, vc, w.pos.as_dict())
        ref, _ = lo.materialized_attention(raw_segments(w, 0, t + 1), lo.as_f64(qd),
                                           [cur[0] - 1], w.pos.as_dict())
        assert np.abs(od - ref).max() < 2e-2


def test_softmax_scale_special_values():
    """1/sqrt(D) for RoPE and ALiBi; YaRN multiplies the logits by mscale^2 (YaRN applies
    mscale to both q and k), so s = e^10 (mscale 2) gives 4/sqrt(D)."""
    assert lo.softmax_scale({"kind": "rope"}, 64) == 0.125
    assert lo.softmax_scale({"kind": "alibi"}, 16) == 0.25
    got = lo.softmax_scale({"kind": "yarn", "yarn_factor": math.exp(10.0)}, 16)
    assert abs(got - 1.0) < 1e-15
