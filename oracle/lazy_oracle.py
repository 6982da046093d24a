"""Plain fp64 CPU oracle for LazyAttention's hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module.  The product path (the CUDA library under
``position_agnostic_kv_gb300/`` and its Python binding) never imports, calls or links it, and
this module imports nothing from the product.  The two share no code: the only common module
is ``workloads/``, which draws seeded inputs and holds none of the method's arithmetic.

Sources (four web pages about one paper, "LazyAttention: Efficient Retrieval-Augmented
Generation with Deferred Positional Encoding", ICML 2026, arXiv 2606.04302):

* [NOTE]   papernotes.org reading note on the paper (Chinese).  Sections cited by name:
           "研究背景与动机 / 切入角度" (the RoPE relative identity), "方法详解 / 整体框架"
           (position-free cache, Example 3.1), "关键设计" with its three items
           "Deferred Positional Encoding", "Tiling 感知的 Q/K 旋转分派",
           "融合 Triton kernel + bit-packed 元数据", and "通用性" (variants).
* [GIST]   gist.science technical summary (Italian): "Concetto Core",
           "Implementazione Tecnica" (1. Prefilling, 2. Decoding), "Equivalenza Matematica".
* [README] illinoisdata/lazy-attention README mirror (shadowgraph.io), "Variants".

What the oracle computes.  The pages state that deferred positional encoding is
mathematically identical to attention over K rotated to its absolute position
([NOTE] 整体框架; [GIST] Equivalenza Matematica).  So the oracle's definition of the result is
that plain thing: rotate every key to its absolute position p and every query to its absolute
position m, then run textbook causal softmax attention in fp64.  The paged functions below
reach the keys the way the method does (walk the per-request block list, read each block's
document offset Delta from its packed word, apply one relative rotation R_Delta to the
position-free stored key) and then call the same textbook attention; tests check that both
routes agree and pin both against brute force, closed forms and invariants.

Readings taken where the pages are silent (each is listed in the design notes):

* RoPE is half-split (pairs (i, i + d/2)): [NOTE] "Tiling 感知" / "融合 Triton kernel" split a
  K tile into two halves and rotate per half-dimension.  theta_i = base^(-2i/d).
* The cache stores R_j k for the token's local position j inside its document (each document
  indexed from local position 0, [NOTE] 整体框架); the attention side applies R_Delta with
  Delta the document's start position in the request, so R_Delta R_j = R_{Delta+j}.
* Q enters raw (pre-RoPE) with its absolute position m.
* GQA maps query head h to KV head floor(h / G), G = Hq / Hkv.
* Softmax scale 1/sqrt(D); under YaRN multiplied by mscale^2, mscale = 0.1 ln(s) + 1.
* YaRN frequencies follow the YaRN paper's ramp (the pages name YaRN only as "metadata",
  [NOTE] 通用性): gamma_i = clamp((L0/lambda_i - beta_slow)/(beta_fast - beta_slow), 0, 1),
  lambda_i = 2 pi / theta_i, theta'_i = (1 - gamma_i) theta_i / s + gamma_i theta_i.
* ALiBi (score-space, [NOTE] 通用性): logit += -slope_h * (m - p); no rotation anywhere.
* The 64-bit block word ([NOTE] "融合 Triton kernel + bit-packed 元数据"; [GIST] Decoding
  bullet on bit-packing) has no published layout; this oracle uses
  bits [4:0] n_valid, [15:5] page-within-document pg, [39:16] Delta, [63:40] physical page.
  The key position of row t of a block is p = Delta + 16 * pg + t.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py`` against
something other than itself (closed forms, a complex-number restatement of RoPE, brute-force
loops over tiny inputs, torch's fp64 scaled-dot-product attention with an explicit mask,
geometric-series closed forms for ALiBi, and permutation invariants).
"""
from __future__ import annotations

import math

import numpy as np

PAGE = 16  # tokens per physical page ("PagedAttention default N=16", [NOTE] Tiling 感知)

# 64-bit block word fields (LSB first).
NVALID_BITS, PG_BITS, DELTA_BITS, PAGE_BITS = 5, 11, 24, 24
PG_SHIFT = NVALID_BITS
DELTA_SHIFT = NVALID_BITS + PG_BITS
PAGE_SHIFT = NVALID_BITS + PG_BITS + DELTA_BITS


# ----------------------------------------------------------------------------------------
# bf16 helpers (the inputs are bf16; the oracle computes in fp64)
# ----------------------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), returned as fp64.

    bf16 keeps 8 significant bits.  Written from the definition: x = m * 2^e with
    0.5 <= |m| < 1, so m * 2^8 rounded half-to-even is the bf16 significand.  Only the normal
    range is supported (|x| >= 2^-126, which N(0,1) data never leaves except for 0).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    tiny = (x != 0) & (np.abs(x) < 2.0 ** -126)
    if np.any(tiny):
        raise ValueError("round_to_bf16: subnormal bf16 range not supported")
    return np.ldexp(np.rint(m * 256.0), e - 8)


def as_f64(a) -> np.ndarray:
    """bf16 bit arrays (uint16) are widened exactly; anything else is taken as fp64 values."""
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of values that are already exactly representable in bf16."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32)
    if np.any(u & np.uint32(0xFFFF)):
        raise ValueError("value is not exactly a bf16")
    return (u >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------------------
# Positional encodings
# ----------------------------------------------------------------------------------------
def rope_inv_freq(rotary_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/d), i < d/2 (standard RoPE frequencies)."""
    i = np.arange(rotary_dim // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * i / rotary_dim)


def yarn_inv_freq(rotary_dim: int, base: float, factor: float, orig_ctx: int,
                  beta_fast: float = 32.0, beta_slow: float = 1.0) -> np.ndarray:
    """YaRN "NTK-by-parts" frequencies: interpolate by 1/s only the long-wavelength pairs.

    The pages say only that NTK/YaRN-scaled RoPE changes nothing but metadata ([NOTE] 通用性);
    the ramp is the YaRN paper's: r_i = L0 / lambda_i, gamma_i = clamp((r_i - beta_slow) /
    (beta_fast - beta_slow), 0, 1), theta'_i = (1 - gamma_i) theta_i / s + gamma_i theta_i.
    """
    theta = rope_inv_freq(rotary_dim, base)
    wavelen = 2.0 * np.pi / theta
    r = orig_ctx / wavelen
    gamma = np.clip((r - beta_slow) / (beta_fast - beta_slow), 0.0, 1.0)
    return (1.0 - gamma) * theta / factor + gamma * theta


def yarn_mscale(factor: float) -> float:
    """YaRN attention temperature factor sqrt(1/t) = 0.1 ln(s) + 1 (1 for s <= 1)."""
    return 1.0 if factor <= 1.0 else 0.1 * math.log(factor) + 1.0


def pos_inv_freq(pos: dict) -> np.ndarray | None:
    """Frequencies for a positional config dict; None for ALiBi (no rotation)."""
    kind = pos["kind"]
    if kind == "rope":
        return rope_inv_freq(pos["rotary_dim"], pos["rope_theta"])
    if kind == "yarn":
        return yarn_inv_freq(pos["rotary_dim"], pos["rope_theta"], pos["yarn_factor"],
                             pos["yarn_orig_ctx"], pos.get("yarn_beta_fast", 32.0),
                             pos.get("yarn_beta_slow", 1.0))
    if kind == "alibi":
        return None
    raise ValueError(kind)


def softmax_scale(pos: dict, head_dim: int) -> float:
    """1/sqrt(D); YaRN multiplies the logits by mscale^2 (mscale applied to both q and k)."""
    s = 1.0 / math.sqrt(head_dim)
    if pos["kind"] == "yarn":
        s *= yarn_mscale(pos["yarn_factor"]) ** 2
    return s


def rotate(x: np.ndarray, pos, inv_freq: np.ndarray, interleaved: bool = False) -> np.ndarray:
    """R_pos x for RoPE over the first d = 2 * len(inv_freq) dimensions, fp64.

    x has shape [..., D]; pos broadcasts against x[..., 0].  Pair i is (x_i, x_{i+d/2})
    (half-split, the form the pages use) or (x_{2i}, x_{2i+1}) (interleaved, GPT-J style; the
    pages list the other RoPE variants as metadata-only changes, [NOTE] 通用性), with angle
    pos * theta_i, and the rotation is the one the pages print for the deferred step
    ([NOTE] 关键设计 / Deferred Positional Encoding): x'_1 = x_1 cos - x_2 sin,
    x'_2 = x_1 sin + x_2 cos.  Dimensions beyond d pass through (partial rotary_dim).
    """
    x = np.asarray(x, dtype=np.float64)
    half = inv_freq.shape[0]
    rd = 2 * half
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    if interleaved:
        i1, i2 = np.arange(0, rd, 2), np.arange(1, rd, 2)
    else:
        i1, i2 = np.arange(half), np.arange(half, rd)
    x1, x2 = x[..., i1], x[..., i2]
    out = x.copy()
    out[..., i1] = x1 * c - x2 * s
    out[..., i2] = x1 * s + x2 * c
    return out


def alibi_slopes(n_heads: int) -> np.ndarray:
    """ALiBi head slopes 2^(-8 h / H), h = 1..H (ALiBi's 1-based head index)."""
    h = np.arange(1, n_heads + 1, dtype=np.float64)
    return np.power(2.0, -8.0 * h / n_heads)


# ----------------------------------------------------------------------------------------
# The 64-bit block word and the per-request metadata ([NOTE] 融合 Triton kernel + bit-packed
# 元数据; [README] Variants: the scheduler builds the per-request rotation metadata)
# ----------------------------------------------------------------------------------------
def pack_meta(n_valid: int, pg: int, delta: int, page: int) -> int:
    """Pack (n_valid, page-within-document, Delta, physical page) into one 64-bit word."""
    if not (0 <= n_valid < (1 << NVALID_BITS) and 0 <= pg < (1 << PG_BITS)
            and 0 <= delta < (1 << DELTA_BITS) and 0 <= page < (1 << PAGE_BITS)):
        raise OverflowError("field out of range for the 64-bit block word")
    return n_valid | (pg << PG_SHIFT) | (delta << DELTA_SHIFT) | (page << PAGE_SHIFT)


def unpack_meta(word: int):
    """Inverse of pack_meta: (n_valid, pg, Delta, page)."""
    word = int(word)
    return (word & ((1 << NVALID_BITS) - 1),
            (word >> PG_SHIFT) & ((1 << PG_BITS) - 1),
            (word >> DELTA_SHIFT) & ((1 << DELTA_BITS) - 1),
            (word >> PAGE_SHIFT) & ((1 << PAGE_BITS) - 1))


def build_meta(req_doc_off, req_docs, doc_len, doc_page_off, doc_pages,
               q_len, q_page_off, q_pages, max_blocks: int):
    """Per-request block list: documents in request order, then the query segment.

    Walk each request's documents in order.  A document of length L occupies ceil(L/16)
    blocks; block pg holds min(16, L - 16 pg) valid tokens, and every block of the document
    carries the same Delta = total length of the documents before it.  The query segment
    (prefill tokens, then decode tokens) is one more document at Delta_q = sum of document
    lengths, with all of its capacity pages listed as full (causality masks the unwritten
    slots).  Returns block_table [B, max_blocks] int32, meta [B, max_blocks] uint64,
    seq_len [B] (keys after the prefill tokens are written), q_start [B] (= Delta_q) and
    doc_blocks [B] (number of document blocks before the query segment).
    """
    B = len(req_doc_off) - 1
    block_table = np.zeros((B, max_blocks), dtype=np.int32)
    meta = np.zeros((B, max_blocks), dtype=np.uint64)
    seq_len = np.zeros(B, dtype=np.int32)
    q_start = np.zeros(B, dtype=np.int32)
    doc_blocks = np.zeros(B, dtype=np.int32)
    for b in range(B):
        j = 0
        delta = 0
        for d in req_docs[req_doc_off[b]:req_doc_off[b + 1]]:
            L = int(doc_len[d])
            pages = doc_pages[doc_page_off[d]:doc_page_off[d + 1]]
            npg = -(-L // PAGE)
            if len(pages) < npg:
                raise ValueError("document has fewer pages than its length needs")
            for pg in range(npg):
                if j >= max_blocks:
                    raise OverflowError("max_blocks too small")
                n_valid = min(PAGE, L - PAGE * pg)
                meta[b, j] = pack_meta(n_valid, pg, delta, int(pages[pg]))
                block_table[b, j] = int(pages[pg])
                j += 1
            delta += L
        doc_blocks[b] = j
        q_start[b] = delta
        for pg, page in enumerate(q_pages[q_page_off[b]:q_page_off[b + 1]]):
            if j >= max_blocks:
                raise OverflowError("max_blocks too small")
            meta[b, j] = pack_meta(PAGE, pg, delta, int(page))
            block_table[b, j] = int(page)
            j += 1
        seq_len[b] = delta + int(q_len[b])
    return block_table, meta, seq_len, q_start, doc_blocks


# ----------------------------------------------------------------------------------------
# KV write: the cache holds keys rotated only by their local position ([NOTE] 整体框架)
# ----------------------------------------------------------------------------------------
def kv_write(k_raw_bits, v_bits, slot, local_pos, pos: dict, k_cache_bits, v_cache_bits):
    """Scatter one batch of tokens into the paged caches (in place, bf16 bit arrays).

    Stored K = bf16_RNE(R_j k_raw) with j the token's local position in its document (no
    rotation at all for ALiBi); stored V = v.  Caches are [P, Hkv, 16, D] bf16 bits; token t
    goes to page slot[t] // 16, row slot[t] % 16.
    """
    inv = pos_inv_freq(pos)
    k = bf16_bits_to_f64(k_raw_bits)
    if inv is not None:
        k = rotate(k, np.asarray(local_pos)[:, None], inv, pos.get("interleaved", False))
    kb = f64_to_bf16_bits(round_to_bf16(k))
    slot = np.asarray(slot, dtype=np.int64)
    page, row = slot // PAGE, slot % PAGE
    k_cache_bits[page, :, row, :] = kb
    v_cache_bits[page, :, row, :] = np.asarray(v_bits, dtype=np.uint16)


# ----------------------------------------------------------------------------------------
# Textbook attention
# ----------------------------------------------------------------------------------------
def softmax_attention(q_abs, q_pos, k_abs, v, k_pos, scale, slopes=None):
    """Causal softmax attention, fp64, written as its definition.

    O[i, h] = sum_{p <= m_i} softmax_p(scale * q_abs[i, h] . k_abs[p, g] + bias) v[p, g],
    g = floor(h / G); bias = -slope_h (m_i - p) for ALiBi, else 0.  Also returns the
    natural-log log-sum-exp of the (biased, scaled) logits per (row, head).
    """
    q_abs = np.asarray(q_abs, np.float64)
    k_abs = np.asarray(k_abs, np.float64)
    v = np.asarray(v, np.float64)
    q_pos = np.asarray(q_pos, np.float64)
    k_pos = np.asarray(k_pos, np.float64)
    M, Hq, D = q_abs.shape
    Hkv = k_abs.shape[1]
    G = Hq // Hkv
    out = np.zeros((M, Hq, v.shape[2]))
    lse = np.zeros((M, Hq))
    visible = k_pos[None, :] <= q_pos[:, None]
    for h in range(Hq):
        g = h // G
        s = scale * (q_abs[:, h, :] @ k_abs[:, g, :].T)
        if slopes is not None:
            s = s - slopes[h] * (q_pos[:, None] - k_pos[None, :])
        s = np.where(visible, s, -np.inf)
        mx = s.max(axis=1, keepdims=True)
        e = np.exp(s - mx)
        den = e.sum(axis=1, keepdims=True)
        out[:, h, :] = (e @ v[:, g, :]) / den
        lse[:, h] = mx[:, 0] + np.log(den[:, 0])
    return out, lse


# ----------------------------------------------------------------------------------------
# Paged attention the way the method reaches the keys
# ----------------------------------------------------------------------------------------
def gather_request(meta_row, n_blocks: int, k_cache_bits, v_cache_bits):
    """Walk a request's first n_blocks block words; return the valid keys in block order.

    Returns stored K and V (fp64, [N, Hkv, D]), each key's document offset Delta and
    absolute position p = Delta + 16 pg + t.
    """
    ks, vs, dl, ps = [], [], [], []
    for w in meta_row[:n_blocks]:
        n_valid, pg, delta, page = unpack_meta(int(w))
        if n_valid == 0:
            continue
        ks.append(k_cache_bits[page, :, :n_valid, :].transpose(1, 0, 2))
        vs.append(v_cache_bits[page, :, :n_valid, :].transpose(1, 0, 2))
        dl.append(np.full(n_valid, delta, dtype=np.int64))
        ps.append(delta + PAGE * pg + np.arange(n_valid, dtype=np.int64))
    k = as_f64(np.concatenate(ks))
    v = as_f64(np.concatenate(vs))
    return k, v, np.concatenate(dl), np.concatenate(ps)


def visible_blocks(doc_blocks: int, q_start: int, m_max: int) -> int:
    """Blocks a query at absolute position m_max can see: all document blocks plus the query
    segment's blocks up to the one holding position m_max."""
    return int(doc_blocks) + (int(m_max) - int(q_start)) // PAGE + 1


def _pos_args(pos: dict, n_heads: int, head_dim: int, scale):
    inv = pos_inv_freq(pos)
    slopes = None
    if pos["kind"] == "alibi":
        slopes = np.asarray(pos["alibi_slopes"], dtype=np.float64)
        assert slopes.shape == (n_heads,)
    if scale is None:
        scale = softmax_scale(pos, head_dim)
    return inv, slopes, scale


def attend_paged(q_raw, m, meta_row, n_blocks, k_cache_bits, v_cache_bits, pos: dict,
                 scale=None):
    """Attention of raw queries at absolute positions m over one request's paged keys.

    K_abs = R_Delta(stored K): the single relative rotation of the deferred step
    ([NOTE] 关键设计 / Deferred Positional Encoding; [GIST] Prefilling), applied here in
    fp64 to every key; Q_abs = R_m q_raw.  Then textbook attention.
    """
    q = np.asarray(q_raw, np.float64)
    inv, slopes, scale = _pos_args(pos, q.shape[1], q.shape[2], scale)
    k, v, delta, p = gather_request(meta_row, n_blocks, k_cache_bits, v_cache_bits)
    m = np.asarray(m, dtype=np.int64)
    if inv is not None:
        k = rotate(k, delta[:, None], inv, pos.get("interleaved", False))
        q = rotate(q, m[:, None], inv, pos.get("interleaved", False))
    return softmax_attention(q, m, k, v, p, scale, slopes)


def prefill(q_bits, cu_q, q_start, doc_blocks, meta, k_cache_bits, v_cache_bits, pos: dict,
            scale=None, requests=None):
    """Prefill of every request's query rows (q rows cu_q[b]:cu_q[b+1] sit at absolute
    positions q_start[b] + i).  Returns (O [sum Lq, Hq, D], LSE [sum Lq, Hq]) in fp64;
    ``requests`` restricts the work to a subset (rows of other requests stay zero)."""
    q_all = as_f64(q_bits)
    out = np.zeros(q_all.shape)
    lse = np.zeros(q_all.shape[:2])
    B = len(cu_q) - 1
    for b in (range(B) if requests is None else requests):
        r0, r1 = int(cu_q[b]), int(cu_q[b + 1])
        if r1 == r0:
            continue
        m = int(q_start[b]) + np.arange(r1 - r0)
        nb = visible_blocks(doc_blocks[b], q_start[b], m[-1])
        o, l = attend_paged(q_all[r0:r1], m, meta[b], nb, k_cache_bits, v_cache_bits, pos,
                            scale)
        out[r0:r1], lse[r0:r1] = o, l
    return out, lse


def decode(q_bits, seq_len, q_start, doc_blocks, meta, k_cache_bits, v_cache_bits, pos: dict,
           scale=None, requests=None):
    """One decode step: request b's single query sits at m = seq_len[b] - 1 (its own key and
    value were written at p = m before the call).  Returns (O [B, Hq, D], LSE [B, Hq])."""
    q_all = as_f64(q_bits)
    B = q_all.shape[0]
    out = np.zeros(q_all.shape)
    lse = np.zeros(q_all.shape[:2])
    for b in (range(B) if requests is None else requests):
        m = int(seq_len[b]) - 1
        nb = visible_blocks(doc_blocks[b], q_start[b], m)
        o, l = attend_paged(q_all[b:b + 1], np.array([m]), meta[b], nb, k_cache_bits,
                            v_cache_bits, pos, scale)
        out[b], lse[b] = o[0], l[0]
    return out, lse


# ----------------------------------------------------------------------------------------
# Materialised reference: the concatenated prompt at absolute positions
# ----------------------------------------------------------------------------------------
def materialized_attention(segments, q_raw, m, pos: dict, scale=None):
    """Attention over the concatenated prompt with keys rotated straight to their absolute
    positions from the RAW keys (no position-free cache, no rounding of stored K).

    segments: list of (k_raw, v) fp64 arrays [L, Hkv, D] in prompt order (documents, then the
    query segment's written tokens).  Token j of a segment starting at absolute position s
    sits at p = s + j.  This is the "materialise position-adjusted KV" computation the pages
    say the method equals ([NOTE] 整体框架; [GIST] Equivalenza Matematica).
    """
    q = np.asarray(q_raw, np.float64)
    inv, slopes, scale = _pos_args(pos, q.shape[1], q.shape[2], scale)
    k = np.concatenate([np.asarray(s[0], np.float64) for s in segments])
    v = np.concatenate([np.asarray(s[1], np.float64) for s in segments])
    p = np.arange(k.shape[0], dtype=np.int64)
    m = np.asarray(m, dtype=np.int64)
    if inv is not None:
        k = rotate(k, p[:, None], inv, pos.get("interleaved", False))
        q = rotate(q, m[:, None], inv, pos.get("interleaved", False))
    return softmax_attention(q, m, k, v, p, scale, slopes)


def full_recompute_loops(segments, q_raw, m, pos: dict, scale=None):
    """Brute force with explicit Python loops (tiny inputs only): every score, max, exponent,
    sum and weighted sum is written out element by element.  Rotation uses the pages' pair
    formula directly on each (k_i, k_{i+d/2}) pair at the absolute position."""
    q = np.asarray(q_raw, np.float64)
    M, Hq, D = q.shape
    inv, slopes, scale = _pos_args(pos, Hq, D, scale)
    keys = []
    p = 0
    for k_seg, v_seg in segments:
        for j in range(k_seg.shape[0]):
            keys.append((p, np.asarray(k_seg[j], np.float64), np.asarray(v_seg[j], np.float64)))
            p += 1
    Hkv = keys[0][1].shape[0]
    G = Hq // Hkv

    inter = pos.get("interleaved", False)

    def rot(vec, position):
        if inv is None:
            return vec.copy()
        out = vec.copy()
        half = inv.shape[0]
        for i in range(half):
            a = position * inv[i]
            c, s = math.cos(a), math.sin(a)
            j1, j2 = (2 * i, 2 * i + 1) if inter else (i, i + half)
            out[j1] = vec[j1] * c - vec[j2] * s
            out[j2] = vec[j1] * s + vec[j2] * c
        return out

    out = np.zeros((M, Hq, D))
    for r in range(M):
        mr = int(m[r])
        for h in range(Hq):
            g = h // G
            qa = rot(q[r, h], mr)
            logits = []
            for (pk, kv, _vv) in keys:
                if pk > mr:
                    continue
                ka = rot(kv[g], pk)
                s = 0.0
                for i in range(D):
                    s += qa[i] * ka[i]
                s *= scale
                if slopes is not None:
                    s -= slopes[h] * (mr - pk)
                logits.append((pk, s))
            mx = max(s for _, s in logits)
            den = 0.0
            acc = np.zeros(D)
            for (pk, s) in logits:
                w = math.exp(s - mx)
                den += w
                acc += w * keys[pk][2][g]
            out[r, h] = acc / den
    return out
