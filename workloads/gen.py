"""Seeded synthetic inputs for LazyAttention's hot path.

This module is shared by the tests, the bench and the smoke check, and it is the ONLY code the
CPU oracle and the CUDA path have in common.  It holds none of the method's arithmetic: it
draws N(0, 1) values and rounds them to bf16, picks documents by Zipf popularity, assigns
physical pages and lists the cache slot every token is written to.  Rotations, offsets,
block words, masks and softmax live on either side of it, never here.

Workloads (the paper's RAG QA workloads -- 2WikiMQA, HotpotQA, TriviaQA, NarrativeQA with Zipf
document popularity -- are not available; these seeded inputs take their shapes instead):

  tiny        1 request, 4/2 heads, D 64, RoPE theta 1e4; docs of 48 and 80 tokens; 16 query
              tokens then 8 decode steps.
  rag8b       Llama-3.1-8B attention shape (32/8/128, theta 5e5); 16 requests of 10 distinct
              200-token docs drawn from a 200-doc pool by Zipf alpha 1.1, shuffled; 32-token
              query prefill then 64 decode steps.
  decode32k   8B shape; 64 requests of 20 distinct 1600-token docs from a 500-doc pool by Zipf
              alpha 2.1, random order (32 000-token context); 128 decode steps, no query
              prefill (decode tokens follow the documents directly).
  prefill70b  Llama-3.1-70B attention shape (64/8/128, theta 5e5); 8 requests of 20 distinct
              512-token docs from a 200-doc pool by Zipf alpha 1.5, shuffled; 64-token causal
              query prefill, no decode.
  mqa_alibi   MQA 32/1/128 with ALiBi slopes 2^(-8h/32), h = 1..32; 32 requests over the same
              12 docs of 1000 tokens in a per-request shuffled order; 32-token query, then 64
              decode steps.
  yarn8b      As mqa_alibi but the 8B shape 32/8/128 with YaRN-scaled RoPE (factor 8, original
              context 8192, theta 5e5).

Sharing: ``sharing="shared"`` gives every document ONE physical copy that all requests point
at (the method's position-agnostic cache); ``sharing="private"`` gives every (request,
document) pair its own pages holding identical contents (no cross-request reuse, so logical
bytes equal the bytes that must come from HBM).

Values: float32 N(0, 1) from numpy's PCG64, rounded to bf16 (ties to even) here so that both
sides see the same bits.  Document d's keys/values come from the stream seeded [seed, 1, d];
request b's prefill tokens from [seed, 2, b]; decode step t from [seed, 3, t]; structure
(Zipf draws, order, page permutation) from [seed, 0].
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PAGE = 16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the bit patterns (uint16)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def zipf_distinct(rng: np.random.Generator, n_pool: int, k: int, alpha: float) -> np.ndarray:
    """Draw k DISTINCT documents, P(rank i) proportional to i^-alpha over the pool (rank 1 =
    doc 0), by sequential draws that reject repeats; returned in draw order."""
    w = np.arange(1, n_pool + 1, dtype=np.float64) ** (-alpha)
    w /= w.sum()
    cdf = np.cumsum(w)
    cdf[-1] = 1.0
    chosen: list[int] = []
    seen = set()
    while len(chosen) < k:
        draws = np.searchsorted(cdf, rng.random(64), side="right")
        for d in draws:
            d = int(d)
            if d not in seen:
                seen.add(d)
                chosen.append(d)
                if len(chosen) == k:
                    break
    return np.array(chosen, dtype=np.int32)


@dataclass
class PosCfg:
    kind: str                     # "rope" | "yarn" | "alibi"
    rope_theta: float = 1e4
    rotary_dim: int = 128
    yarn_factor: float = 1.0
    yarn_orig_ctx: int = 0
    yarn_beta_fast: float = 32.0
    yarn_beta_slow: float = 1.0
    alibi_slopes: np.ndarray | None = None   # float32 [Hq], ALiBi only
    interleaved: bool = False                # pairs (x_2i, x_2i+1) instead of (x_i, x_i+d/2)

    def as_dict(self) -> dict:
        return dict(kind=self.kind, rope_theta=self.rope_theta, rotary_dim=self.rotary_dim,
                    yarn_factor=self.yarn_factor, yarn_orig_ctx=self.yarn_orig_ctx,
                    yarn_beta_fast=self.yarn_beta_fast, yarn_beta_slow=self.yarn_beta_slow,
                    alibi_slopes=self.alibi_slopes, interleaved=self.interleaved)


@dataclass
class Workload:
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    pos: PosCfg
    sharing: str
    # document pool contents: doc_len[d]
    doc_len: np.ndarray
    # physical copies ("instances"): inst_doc[i] = content doc, pages in CSR
    inst_doc: np.ndarray
    inst_page_off: np.ndarray
    inst_pages: np.ndarray
    # requests: ordered instance lists (CSR)
    req_inst_off: np.ndarray
    req_inst: np.ndarray
    # query segment: Lq per request, decode steps, capacity pages per request (CSR)
    q_len: np.ndarray
    n_decode: int
    q_page_off: np.ndarray
    q_pages: np.ndarray
    num_pages: int
    max_blocks: int
    _doc_cache: dict = field(default_factory=dict, repr=False)

    # ---------------- sizes ----------------
    @property
    def inst_len(self) -> np.ndarray:
        return self.doc_len[self.inst_doc].astype(np.int32)

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_len)]).astype(np.int32)

    def request_docs(self, b: int) -> np.ndarray:
        """Content-doc ids of request b in prompt order."""
        return self.inst_doc[self.req_inst[self.req_inst_off[b]:self.req_inst_off[b + 1]]]

    # ---------------- values ----------------
    def doc_kv(self, d: int):
        """Raw (pre-RoPE) keys and values of content doc d: bf16 bits [L, Hkv, D] each."""
        if d in self._doc_cache:
            return self._doc_cache[d]
        rng = np.random.default_rng([self.seed, 1, int(d)])
        L = int(self.doc_len[d])
        k = _normal_bf16(rng, (L, self.Hkv, self.D))
        v = _normal_bf16(rng, (L, self.Hkv, self.D))
        if len(self._doc_cache) < 64:
            self._doc_cache[d] = (k, v)
        return k, v

    def used_docs(self) -> np.ndarray:
        return np.unique(self.inst_doc[self.req_inst])

    def inst_slots(self, i: int):
        """Cache slot (page * 16 + row) and local position of every token of instance i."""
        L = int(self.doc_len[self.inst_doc[i]])
        pages = self.inst_pages[self.inst_page_off[i]:self.inst_page_off[i + 1]]
        j = np.arange(L, dtype=np.int32)
        return (pages[j // PAGE] * PAGE + j % PAGE).astype(np.int32), j

    def prefill_tokens(self):
        """Prefill inputs: q [sum Lq, Hq, D], k/v [sum Lq, Hkv, D] (bf16 bits), each token's
        cache slot and local position inside the query segment."""
        qs, ks, vs, slots, lps = [], [], [], [], []
        for b in range(self.B):
            L = int(self.q_len[b])
            rng = np.random.default_rng([self.seed, 2, b])
            qs.append(_normal_bf16(rng, (L, self.Hq, self.D)))
            ks.append(_normal_bf16(rng, (L, self.Hkv, self.D)))
            vs.append(_normal_bf16(rng, (L, self.Hkv, self.D)))
            pages = self.q_pages[self.q_page_off[b]:self.q_page_off[b + 1]]
            j = np.arange(L, dtype=np.int32)
            slots.append(pages[j // PAGE] * PAGE + j % PAGE)
            lps.append(j)
        cat = lambda xs, dt: np.concatenate(xs).astype(dt) if xs else np.zeros(0, dt)
        return (np.concatenate(qs), np.concatenate(ks), np.concatenate(vs),
                cat(slots, np.int32), cat(lps, np.int32))

    def decode_tokens(self, t: int):
        """Decode step t inputs: q [B, Hq, D], k/v [B, Hkv, D] (bf16 bits), slot, local pos."""
        rng = np.random.default_rng([self.seed, 3, int(t)])
        q = _normal_bf16(rng, (self.B, self.Hq, self.D))
        k = _normal_bf16(rng, (self.B, self.Hkv, self.D))
        v = _normal_bf16(rng, (self.B, self.Hkv, self.D))
        slots = np.empty(self.B, np.int32)
        lps = np.empty(self.B, np.int32)
        for b in range(self.B):
            j = int(self.q_len[b]) + t
            pages = self.q_pages[self.q_page_off[b]:self.q_page_off[b + 1]]
            slots[b] = pages[j // PAGE] * PAGE + j % PAGE
            lps[b] = j
        return q, k, v, slots, lps

    # ---------------- accounting (sizes only) ----------------
    def logical_doc_tokens(self) -> np.ndarray:
        """Document tokens per request (sum of its documents' lengths)."""
        return np.array([int(self.doc_len[self.request_docs(b)].sum()) for b in range(self.B)])

    def cache_bytes(self) -> int:
        return 2 * self.num_pages * self.Hkv * PAGE * self.D * 2


def _build(name, seed, B, Hq, Hkv, D, pos, doc_len, req_docs, q_len, n_decode, sharing,
           rng) -> Workload:
    """Lay out pages: instances in order, then every request's query-segment capacity pages;
    then permute all physical page ids (a fragmented pool)."""
    doc_len = np.asarray(doc_len, dtype=np.int32)
    if sharing == "shared":
        used = sorted({int(d) for docs in req_docs for d in docs})
        inst_of = {d: i for i, d in enumerate(used)}
        inst_doc = np.array(used, dtype=np.int32)
        req_inst = [[inst_of[int(d)] for d in docs] for docs in req_docs]
    elif sharing == "private":
        inst_doc_l, req_inst = [], []
        for docs in req_docs:
            row = []
            for d in docs:
                row.append(len(inst_doc_l))
                inst_doc_l.append(int(d))
            req_inst.append(row)
        inst_doc = np.array(inst_doc_l, dtype=np.int32)
    else:
        raise ValueError(sharing)
    npages_inst = -(-doc_len[inst_doc] // PAGE)
    inst_page_off = np.concatenate([[0], np.cumsum(npages_inst)]).astype(np.int32)
    q_len = np.broadcast_to(np.asarray(q_len, dtype=np.int32), (B,)).copy()
    q_cap = q_len + n_decode
    npages_q = -(-q_cap // PAGE)
    q_page_off = np.concatenate([[0], np.cumsum(npages_q)]).astype(np.int32)
    n_inst_pages = int(inst_page_off[-1])
    num_pages = n_inst_pages + int(q_page_off[-1])
    perm = rng.permutation(num_pages).astype(np.int32)
    inst_pages = perm[:n_inst_pages]
    q_pages = perm[n_inst_pages:]
    req_inst_off = np.concatenate([[0], np.cumsum([len(r) for r in req_inst])]).astype(np.int32)
    req_inst_flat = np.array([i for r in req_inst for i in r], dtype=np.int32)
    max_blocks = 0
    for b in range(B):
        ii = req_inst_flat[req_inst_off[b]:req_inst_off[b + 1]]
        max_blocks = max(max_blocks, int(npages_inst[ii].sum()) + int(npages_q[b]))
    return Workload(name=name, seed=seed, B=B, Hq=Hq, Hkv=Hkv, D=D, pos=pos, sharing=sharing,
                    doc_len=doc_len, inst_doc=inst_doc, inst_page_off=inst_page_off,
                    inst_pages=inst_pages, req_inst_off=req_inst_off, req_inst=req_inst_flat,
                    q_len=q_len, n_decode=int(n_decode), q_page_off=q_page_off,
                    q_pages=q_pages, num_pages=num_pages, max_blocks=max_blocks)


def alibi_slopes_input(n_heads: int) -> np.ndarray:
    """The ALiBi slopes the mqa_alibi workload states, 2^(-8h/32) for h = 1..32, as float32
    input data (the oracle derives its own copy)."""
    return np.array([2.0 ** (-8.0 * h / n_heads) for h in range(1, n_heads + 1)],
                    dtype=np.float32)


WORKLOADS = ("tiny", "rag8b", "decode32k", "prefill70b", "mqa_alibi", "yarn8b")
SEEDS = {"tiny": 0, "rag8b": 1, "decode32k": 2, "prefill70b": 3, "mqa_alibi": 4, "yarn8b": 4}


def make_workload(name: str, sharing: str = "shared", seed: int | None = None,
                  batch: int | None = None) -> Workload:
    """Build one of the named workloads.  ``batch`` (optional) keeps only the first requests,
    for bounded CPU samples of the same workload."""
    seed = SEEDS[name] if seed is None else seed
    rng = np.random.default_rng([seed, 0])
    if name == "tiny":
        B, Hq, Hkv, D = 1, 4, 2, 64
        pos = PosCfg("rope", 1e4, D)
        doc_len = [48, 80]
        req_docs = [[0, 1]]
        q_len, n_dec = 16, 8
    elif name in ("rag8b", "decode32k", "prefill70b"):
        spec = {"rag8b": (16, 32, 8, 200, 200, 10, 1.1, 32, 64),
                "decode32k": (64, 32, 8, 500, 1600, 20, 2.1, 0, 128),
                "prefill70b": (8, 64, 8, 200, 512, 20, 1.5, 64, 0)}[name]
        B, Hq, Hkv, n_pool, L, k, alpha, q_len, n_dec = spec
        D = 128
        pos = PosCfg("rope", 5e5, D)
        doc_len = [L] * n_pool
        req_docs = []
        for _ in range(B):
            docs = zipf_distinct(rng, n_pool, k, alpha)
            rng.shuffle(docs)
            req_docs.append(docs)
    elif name in ("mqa_alibi", "yarn8b"):
        B, Hq, D = 32, 32, 128
        if name == "mqa_alibi":
            Hkv = 1
            pos = PosCfg("alibi", rotary_dim=D, alibi_slopes=alibi_slopes_input(Hq))
        else:
            Hkv = 8
            pos = PosCfg("yarn", 5e5, D, yarn_factor=8.0, yarn_orig_ctx=8192)
        doc_len = [1000] * 12
        req_docs = [rng.permutation(12) for _ in range(B)]
        q_len, n_dec = 32, 64
    else:
        raise ValueError(name)
    if batch is not None:
        B = min(B, batch)
        req_docs = req_docs[:B]
    return _build(name, seed, B, Hq, Hkv, D, pos, doc_len, req_docs, q_len, n_dec, sharing, rng)


def make_custom(doc_len, req_docs, Hq, Hkv, D, pos: PosCfg, q_len, n_decode, seed=123,
                sharing="shared", name="custom") -> Workload:
    """A workload with explicit document lengths and per-request document order (edge cases:
    1-, 15- and 17-token documents, empty queries, ...)."""
    rng = np.random.default_rng([seed, 0])
    return _build(name, seed, len(req_docs), Hq, Hkv, D, pos, doc_len,
                  [np.asarray(r, dtype=np.int32) for r in req_docs], q_len, n_decode,
                  sharing, rng)
