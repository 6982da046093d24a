"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Inputs are the seeded workloads; the oracle computes from the same bf16 bits with its own KV
write (fp64 rotation, one rounding to bf16) and its own block words.  Attention outputs must
meet max-abs 2e-2, mean-abs 2e-3 and relative 1e-2 (see tests/gpu_common.py); the stored K must
be within one bf16 unit in the last place of the oracle's and the stored V bit-exact.
"""
import numpy as np
import pytest

import oracle
from oracle import lazy_oracle as lo
from tests.gpu_common import (assert_close, lib, oracle_caches_for, request_instances)
from tests.oracle_setup import oracle_meta, raw_segments
from workloads import PosCfg, alibi_slopes_input, f32_to_bf16_bits, make_custom, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lk():
    return lib()


NAN_BITS = 0x7FC0  # a quiet-NaN bf16 pattern


def _batch(w, poison=False, **kw):
    """A PagedBatch; with poison=True every cache row starts as NaN bits, so any row the kernels
    read without a key written there (past a document's end, past the causal frontier, or a
    page slot past the last block) would turn the output into NaN."""
    from position_agnostic_kv_gb300.runner import PagedBatch
    pb = PagedBatch(w, device="cuda", **kw)
    if poison:
        pb.k_cache.view(torch_int16()).fill_(NAN_BITS)
        pb.v_cache.view(torch_int16()).fill_(NAN_BITS)
    return pb


def torch_int16():
    import torch
    return torch.int16


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _status_clean(lk):
    assert lk.device_status() == 0


# ------------------------------------------------------------------ cos/sin table
@pytest.mark.parametrize("kind,D", [("rope", 128), ("yarn", 128), ("rope", 48), ("yarn", 32)])
def test_rope_table_matches_fp64(lk, kind, D):
    """Table rows for full and partial rotary dimensions (D here is the rotary dimension)."""
    import torch
    max_pos = 40000
    if kind == "rope":
        cfg = lk.pos_cfg_from("rope", D, rope_theta=5e5)
        inv = lo.rope_inv_freq(D, 5e5)
    else:
        cfg = lk.pos_cfg_from("yarn", D, rope_theta=5e5, yarn_factor=8.0, yarn_orig_ctx=8192)
        inv = lo.yarn_inv_freq(D, 5e5, 8.0, 8192)
    out = torch.empty((max_pos, D), dtype=torch.float32, device="cuda")
    lk.build_rope_table(cfg, max_pos, out)
    got = out.cpu().numpy().astype(np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    # exact angle reduction: error ~2^-25 turn plus one ulp of sin/cos
    np.testing.assert_allclose(got[:, : D // 2], np.cos(ang), atol=1e-6, rtol=0)
    np.testing.assert_allclose(got[:, D // 2:], np.sin(ang), atol=1e-6, rtol=0)
    _status_clean(lk)


# ------------------------------------------------------------------ kv write
@pytest.mark.parametrize("name", ["tiny", "rag8b", "yarn8b", "mqa_alibi"])
def test_kv_write_parity(lk, name):
    import torch
    w = make_workload(name, batch=4)
    pb = _batch(w)
    pb.fill_documents()
    pb.prefill(pb.upload_prefill())
    torch.cuda.synchronize()
    _status_clean(lk)
    kc, vc = oracle_caches_for(w)
    np.testing.assert_array_equal(_bits(pb.v_cache), vc)
    gk = lo.bf16_bits_to_f64(_bits(pb.k_cache))
    rk = lo.bf16_bits_to_f64(kc)
    # The kernel rotates in fp32 with cos/sin good to ~5e-7 absolute, so before its single
    # rounding the value is within 5e-7 * (|k1| + |k2|) + 2^-23 |y| of the exact one; after
    # rounding it is within one bf16 ulp of the oracle's plus that absolute term, which only
    # matters where the two products nearly cancel (|y| << |k|).  |k| <= 6 for these inputs.
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(rk), 2.0 ** -126))) - 7)
    bad = np.abs(gk - rk) > ulp + 6e-6
    assert not bad.any(), f"{bad.sum()} stored K values beyond one bf16 ulp + 6e-6"
    frac = np.mean(gk != rk)
    assert frac < 0.01, f"{frac:.4f} of stored K differ from the oracle's rounding"


# ------------------------------------------------------------------ attention
def _run_and_check(lk, w, reqs, n_steps, check_steps, use_table=False, sharpen=1.0, poison=False,
                   outputs=None):
    """Run fill -> prefill -> n_steps decode steps on the GPU; compare prefill rows of `reqs`
    and the decode outputs of `reqs` at `check_steps` against the oracle.  `outputs`, a dict,
    receives the GPU outputs ('prefill' and 'decode<t>' for t in check_steps)."""
    import torch
    pb = _batch(w, use_table=use_table, poison=poison)
    pb.fill_documents()
    inp = pb.upload_prefill()
    if sharpen != 1.0:
        inp["q"] = (inp["q"].float() * sharpen).to(torch.bfloat16)
    out_p = pb.prefill(inp)
    outs_d = {}
    for t in range(n_steps):
        o = pb.decode_step(pb.upload_decode(t))
        if t in check_steps:
            outs_d[t] = o.clone()
    torch.cuda.synchronize()
    _status_clean(lk)
    if outputs is not None:
        outputs["prefill"] = out_p.clone()
        outputs.update({f"decode{t}": o for t, o in outs_d.items()})

    bt, meta, seq_len, q_start, doc_blocks = oracle_meta(w)
    np.testing.assert_array_equal(meta, pb.meta_h)
    pos = w.pos.as_dict()
    kc, vc = oracle_caches_for(w, request_instances(w, reqs), prefill=True)
    q = w.prefill_tokens()[0]
    if sharpen != 1.0:
        q = _bits(inp["q"])
    results = {}
    if w.q_len.sum():
        ref_p, _ = lo.prefill(q, w.cu_q, q_start, doc_blocks, meta, kc, vc, pos, requests=reqs)
        rows = np.concatenate([np.arange(w.cu_q[b], w.cu_q[b + 1]) for b in reqs])
        results["prefill"] = assert_close(out_p[rows], ref_p[rows], f"{w.name} prefill")
    done = 0
    for t in sorted(check_steps):
        while done <= t:
            _, k, v, slot, lp = w.decode_tokens(done)
            oracle.kv_write(k, v, slot, lp, pos, kc, vc)
            done += 1
        qd = w.decode_tokens(t)[0]
        ref_d, _ = lo.decode(qd, seq_len + t + 1, q_start, doc_blocks, meta, kc, vc, pos,
                             requests=reqs)
        results[f"decode{t}"] = assert_close(outs_d[t][reqs], ref_d[reqs], f"{w.name} decode step {t}")
    return results


def test_tiny_all_steps(lk):
    w = make_workload("tiny")
    _run_and_check(lk, w, [0], w.n_decode, set(range(w.n_decode)))


def test_tiny_matches_materialized_definition(lk):
    """End to end against the definition itself: keys rotated straight to absolute positions
    from the raw bf16 inputs (no position-free cache anywhere on the oracle side)."""
    import torch
    w = make_workload("tiny")
    pb = _batch(w)
    pb.fill_documents()
    out_p = pb.prefill(pb.upload_prefill())
    q = w.prefill_tokens()[0]
    _, _, sl, qs, _ = oracle_meta(w)
    m = qs[0] + np.arange(w.q_len[0])
    ref, _ = lo.materialized_attention(raw_segments(w, 0, 0), lo.as_f64(q), m, w.pos.as_dict())
    assert_close(out_p, ref, "tiny prefill vs materialised")
    for t in range(w.n_decode):
        o = pb.decode_step(pb.upload_decode(t))
        qd = w.decode_tokens(t)[0]
        ref, _ = lo.materialized_attention(raw_segments(w, 0, t + 1), lo.as_f64(qd),
                                           [sl[0] + t], w.pos.as_dict())
        assert_close(o, ref, f"tiny decode {t} vs materialised")
    torch.cuda.synchronize()
    _status_clean(lk)


@pytest.mark.parametrize("sharing", ["shared", "private"])
def test_rag8b(lk, sharing):
    w = make_workload("rag8b", sharing=sharing)
    _run_and_check(lk, w, [0, 5, 15], 4, {0, 3})


def test_rag8b_table_mode(lk):
    w = make_workload("rag8b")
    _run_and_check(lk, w, [1, 7], 3, {2}, use_table=True)


def test_yarn8b(lk):
    w = make_workload("yarn8b")
    _run_and_check(lk, w, [0, 31], 3, {0, 2})


def test_mqa_alibi(lk):
    w = make_workload("mqa_alibi")
    _run_and_check(lk, w, [0, 13], 3, {0, 2})


def test_prefill70b(lk):
    w = make_workload("prefill70b")
    _run_and_check(lk, w, list(range(w.B)), 0, set())


def test_decode32k(lk):
    """Full decode-bound workload (64 requests, 32 000-token contexts, 128 steps) on the GPU;
    the oracle checks four requests at steps 0, 63 and 127."""
    w = make_workload("decode32k")
    _run_and_check(lk, w, [0, 21, 42, 63], 128, {0, 63, 127})


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 4), (64, 8, 2), (128, 8, 1), (128, 16, 2), (64, 16, 2),
                                      (128, 24, 1), (64, 48, 2)])
def test_edge_shapes(lk, D, Hq, Hkv):
    """Documents of 1, 15, 16, 17 and 33 tokens, uneven query lengths (one request without a
    query segment), MHA / GQA / MQA groupings and both head dims.  Head groups of 24 do not
    divide the tensor-core kernel's 128 rows, so their prefill runs one CUDA-core CTA per query
    row (the decode kernel's row mode) and their decode takes 8 heads per CTA."""
    w = make_custom([1, 15, 16, 17, 33], [[4, 0, 2], [1, 3], [2, 4, 1, 0]], Hq, Hkv, D,
                    PosCfg("rope", 1e4, D), [3, 0, 17], 5, seed=D + Hq)
    _run_and_check(lk, w, [0, 1, 2], 5, {0, 4})


@pytest.mark.parametrize("D,Hq,Hkv,kind", [(128, 32, 1, "rope"), (64, 16, 1, "alibi"), (128, 32, 2, "yarn")])
def test_wide_group_decode(lk, D, Hq, Hkv, kind):
    """Head groups of 16 and 32 (MQA-like) decode on the tensor-core kernel with the key range
    split over CTAs: one long request (several splits), a 1-token one (empty splits), ragged
    documents, rotary and ALiBi variants."""
    if kind == "yarn":
        pos = PosCfg(kind, 5e5, D, yarn_factor=8.0, yarn_orig_ctx=8192)
    elif kind == "alibi":
        pos = PosCfg(kind, 1e4, D, alibi_slopes=alibi_slopes_input(Hq))
    else:
        pos = PosCfg(kind, 1e4, D)
    w = make_custom([2900, 700, 17, 1], [[0, 1, 2], [3], [2, 3, 1]], Hq, Hkv, D, pos, [5, 1, 0], 3,
                    seed=D + Hq + Hkv)
    _run_and_check(lk, w, [0, 1, 2], 3, {0, 2})


def test_long_context_128k(lk):
    """Long context: a 32 768-token document (the page-in-document field's maximum, pg 2047),
    six of 16 384 tokens and one of 5 000, shuffled into one 136 072-token prompt; the query and
    decode tokens sit at absolute positions ~1.36e5 (exact-turn angles, 24-bit Delta)."""
    w = make_custom([32768, 16384, 16384, 16384, 16384, 16384, 16384, 5000],
                    [[3, 0, 7, 1, 6, 2, 5, 4]], 8, 2, 128, PosCfg("rope", 5e5, 128), [16], 2,
                    seed=1280)
    assert int(oracle_meta(w)[2][0]) == 136072 + 16
    _run_and_check(lk, w, [0], 2, {0, 1})


@pytest.mark.parametrize("D,Hq,Hkv,L", [(128, 8, 2, 200), (64, 4, 4, 33), (128, 32, 1, 130)])
def test_cold_document_encode_then_reuse(lk, D, Hq, Hkv, L):
    """A document seen for the first time is encoded alone from local position 0 (keys written
    at local positions, its own causal attention at Delta = 0); the written pages are then the
    document's cache, which a later request reuses at a non-zero offset."""
    import torch
    from position_agnostic_kv_gb300.runner import bits_to_tensor, encode_document
    rng = np.random.default_rng([L, D, Hq])
    bf = lambda *shape: f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    pos = PosCfg("rope", 1e4, D)
    q, k, v = bf(L, Hq, D), bf(L, Hkv, D), bf(L, Hkv, D)
    n_pages = (L + 15) // 16
    pages = rng.permutation(3 * n_pages)[:n_pages].astype(np.int32)
    dev = torch.device("cuda")
    kc = torch.zeros((3 * n_pages, Hkv, 16, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    cfg = lk.pos_cfg_from("rope", D, rope_theta=1e4)
    out = encode_document(bits_to_tensor(q, dev), bits_to_tensor(k, dev), bits_to_tensor(v, dev),
                          pages, kc, vc, cfg)
    torch.cuda.synchronize()
    _status_clean(lk)
    ref, _ = lo.materialized_attention([(lo.bf16_bits_to_f64(k), lo.bf16_bits_to_f64(v))],
                                       lo.bf16_bits_to_f64(q), np.arange(L), pos.as_dict())
    assert_close(out, ref, "cold document self-attention")
    # the written pages are the document's cache: what the oracle writes for the same tokens
    okc = np.zeros((3 * n_pages, Hkv, 16, D), np.uint16)
    ovc = np.zeros_like(okc)
    t = np.arange(L)
    oracle.kv_write(k, v, pages[t // 16] * 16 + t % 16, t, pos.as_dict(), okc, ovc)
    np.testing.assert_array_equal(_bits(vc), ovc)
    gk, rk = lo.bf16_bits_to_f64(_bits(kc)), lo.bf16_bits_to_f64(okc)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(rk), 2.0 ** -126))) - 7)
    assert not (np.abs(gk - rk) > ulp + 6e-6).any()
    # reuse: a request [another document of 37 tokens, this document] + a 5-token query
    pre_len, ql = 37, 5
    kp, vp, qq, kq, vq = bf(pre_len, Hkv, D), bf(pre_len, Hkv, D), bf(ql, Hq, D), bf(ql, Hkv, D), bf(ql, Hkv, D)
    kc2 = torch.zeros((3 * n_pages + 8, Hkv, 16, D), dtype=torch.bfloat16, device=dev)
    vc2 = torch.zeros_like(kc2)
    kc2[: 3 * n_pages], vc2[: 3 * n_pages] = kc, vc
    pre_pages = np.array([3 * n_pages, 3 * n_pages + 1, 3 * n_pages + 2], np.int32)
    q_pages = np.array([3 * n_pages + 3], np.int32)
    tp = np.arange(pre_len)
    lk.kv_write(bits_to_tensor(kp, dev), bits_to_tensor(vp, dev),
                torch.from_numpy((pre_pages[tp // 16] * 16 + tp % 16).astype(np.int32)).to(dev),
                torch.from_numpy(tp.astype(np.int32)).to(dev), kc2, vc2, cfg)
    doc_len = [pre_len, L]
    doc_page_off = [0, len(pre_pages), len(pre_pages) + n_pages]
    max_blocks = len(pre_pages) + n_pages + 1
    bt, meta_h, seq_len, q_start, doc_blocks = lk.build_doc_meta(
        [0, 2], [0, 1], doc_len, doc_page_off, np.concatenate([pre_pages, pages]), [ql], [0, 1],
        q_pages, max_blocks)
    tq = np.arange(ql)
    lk.kv_write(bits_to_tensor(kq, dev), bits_to_tensor(vq, dev),
                torch.from_numpy((q_pages[0] * 16 + tq).astype(np.int32)).to(dev),
                torch.from_numpy(tq.astype(np.int32)).to(dev), kc2, vc2, cfg)
    out2 = torch.empty((ql, Hq, D), dtype=torch.bfloat16, device=dev)
    i32 = lambda x: torch.from_numpy(np.asarray(x, np.int32)).to(dev)
    ws = torch.empty(max(lk.workspace_size(lk.PHASE_PREFILL, ql, 1, max_blocks, Hq, Hkv, D), 256),
                     dtype=torch.uint8, device=dev)
    lk.attn_prefill(bits_to_tensor(qq, dev), i32([0, ql]), i32(q_start), i32(doc_blocks),
                    torch.from_numpy(meta_h.view(np.int64)).to(dev), kc2, vc2, cfg, out2, ql, ws=ws)
    torch.cuda.synchronize()
    _status_clean(lk)
    segs = [(lo.bf16_bits_to_f64(kp), lo.bf16_bits_to_f64(vp)), (lo.bf16_bits_to_f64(k), lo.bf16_bits_to_f64(v)),
            (lo.bf16_bits_to_f64(kq), lo.bf16_bits_to_f64(vq))]
    ref2, _ = lo.materialized_attention(segs, lo.bf16_bits_to_f64(qq), pre_len + L + tq, pos.as_dict())
    assert_close(out2, ref2, "reuse of the cold-encoded document at offset 37")


ROPE_VARIANTS = [  # D, Hq, Hkv, rotary_dim, interleaved, kind, table
    (128, 8, 2, 64, False, "rope", False),
    (128, 8, 2, 128, True, "rope", True),
    (64, 4, 4, 32, True, "yarn", False),
    (64, 16, 2, 48, False, "rope", True),
    (128, 32, 1, 32, True, "rope", False),
    (128, 32, 1, 96, False, "yarn", False),
]


@pytest.mark.parametrize("D,Hq,Hkv,rd,inter,kind,table", ROPE_VARIANTS)
def test_rope_variants(lk, D, Hq, Hkv, rd, inter, kind, table):
    """Interleaved (GPT-J) pairs and partial rotary_dim through every kernel: the written K
    cache (one bf16 ulp of the oracle), the tensor-core prefill, the CUDA-core decode (G <= 8)
    or the tensor-core decode (G >= 16), cos/sin on the fly or from the table."""
    import torch
    extra = dict(yarn_factor=8.0, yarn_orig_ctx=512) if kind == "yarn" else {}
    pos = PosCfg(kind, 1e4, rd, interleaved=inter, **extra)
    w = make_custom([1, 15, 16, 17, 333], [[4, 0, 2], [1, 3], [2, 4, 1, 0]], Hq, Hkv, D, pos,
                    [3, 0, 17], 4, seed=D + Hq + rd)
    _run_and_check(lk, w, [0, 1, 2], 4, {0, 3}, use_table=table)
    pb = _batch(w, use_table=table)
    pb.fill_documents()
    torch.cuda.synchronize()
    _status_clean(lk)
    kc, _ = oracle_caches_for(w, prefill=False)
    gk, rk = lo.bf16_bits_to_f64(_bits(pb.k_cache)), lo.bf16_bits_to_f64(kc)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(rk), 2.0 ** -126))) - 7)
    assert not (np.abs(gk - rk) > ulp + 6e-6).any()
    # the dimensions beyond rotary_dim are stored unrotated (bit-exact copies)
    np.testing.assert_array_equal(_bits(pb.k_cache)[..., rd:], kc[..., rd:])


@pytest.mark.parametrize("name,batch", [("rag8b", 2), ("prefill70b", 1)])
def test_one_key_far_above_the_running_max(lk, name, batch):
    """The key of each request's first query token replaced by one large component (1024 in
    the lowest-frequency dimension 63, zeros elsewhere): every query row sees it, and where q's
    dimension 63 is positive its logit lies up to hundreds of log2 units above the running max
    taken on the document tiles, so the lazy softmax rescales O and l by a factor that
    underflows to zero and the row's output becomes that key's value.  A single component
    keeps the logit's rounding error proportional to the logit (a random key scaled up would
    carry every component's rounding, scaled, into rows where it only half dominates).  Key
    halves (rag8b, one Q tile per CTA) and two Q tiles per CTA (prefill70b)."""
    import torch
    from position_agnostic_kv_gb300.runner import bits_to_tensor
    w = make_workload(name, batch=batch)
    pb = _batch(w)
    pb.fill_documents()
    q, k, v, slot, lp = w.prefill_tokens()
    k64 = k.copy()
    first = w.cu_q[:-1][w.q_len > 0]
    k64[first] = 0
    k64[first, :, 63] = f32_to_bf16_bits(np.full((len(first), w.Hkv), 1024.0, np.float32))
    inp = pb.upload_prefill()
    inp["k"] = bits_to_tensor(k64, inp["k"].device)
    out = pb.prefill(inp)
    torch.cuda.synchronize()
    _status_clean(lk)
    _, meta, _, qs, db = oracle_meta(w)
    pos = w.pos.as_dict()
    kc, vc = oracle_caches_for(w, prefill=False)
    oracle.kv_write(k64, v, slot, lp, pos, kc, vc)
    ref, _ = lo.prefill(q, w.cu_q, qs, db, meta, kc, vc, pos)
    assert_close(out, ref, f"{name} prefill, one key far above the running max")


def test_sharpened_queries_separate_negative_controls(lk):
    """With queries x4 the softmax is sharp: the GPU output must match the oracle, while the
    oracle run with wrong offsets (Delta = 0 everywhere, Delta + 1, the naive double rotation
    2*Delta) misses the GPU output by more than the tolerance."""
    import torch
    w = make_workload("rag8b", batch=2)
    pb = _batch(w)
    pb.fill_documents()
    inp = pb.upload_prefill()
    inp["q"] = (inp["q"].float() * 4.0).to(torch.bfloat16)
    out = pb.prefill(inp)
    torch.cuda.synchronize()
    _status_clean(lk)
    q4 = _bits(inp["q"])
    _, meta, _, qs, db = oracle_meta(w)
    kc, vc = oracle_caches_for(w)
    pos = w.pos.as_dict()
    ref, _ = lo.prefill(q4, w.cu_q, qs, db, meta, kc, vc, pos)
    assert_close(out, ref, "sharpened prefill")
    for fn in (lambda d: 0, lambda d: d + 1, lambda d: 2 * d):
        bad = meta.copy()
        for b in range(w.B):
            for j in range(meta.shape[1]):
                nv, pg, dl, page = lo.unpack_meta(int(meta[b, j]))
                if nv:
                    bad[b, j] = lo.pack_meta(nv, pg, fn(dl), page)
        wrong, _ = lo.prefill(q4, w.cu_q, qs, db, bad, kc, vc, pos)
        err = np.abs(out.float().cpu().numpy() - wrong).max()
        assert err > 2e-2, f"negative control not separated: {err:.3e}"


# ------------------------------------------------------------------ log-sum-exp output
@pytest.mark.parametrize("Hq,Hkv,q_len,path", [
    (8, 2, [20, 7, 32], "one Q tile per CTA: key halves"),
    (8, 2, [70, 33, 100], "two Q tiles per CTA"),
    (24, 1, [20, 7, 32], "row mode (head group of 24)"),
])
def test_prefill_lse_matches_oracle(lk, Hq, Hkv, q_len, path):
    """The optional log-sum-exp output of the prefill (natural log of the row's softmax
    denominator over the scaled logits) on each prefill path, against the oracle's."""
    import torch
    w = make_custom([200, 37, 1000, 15, 1], [[0, 1, 2], [3, 4, 0], [2]], Hq, Hkv, 128,
                    PosCfg("rope", 5e5, 128), q_len, 0, seed=61)
    pb = _batch(w)
    pb.fill_documents()
    inp = pb.upload_prefill()
    lse = torch.full((pb.total_q, Hq), float("nan"), dtype=torch.float32, device="cuda")
    out = pb.prefill(inp, lse=lse)
    torch.cuda.synchronize()
    _status_clean(lk)
    _, meta, _, q_start, doc_blocks = oracle_meta(w)
    reqs = [0, 1, 2]
    kc, vc = oracle_caches_for(w, request_instances(w, reqs), prefill=True)
    ref_o, ref_l = lo.prefill(w.prefill_tokens()[0], w.cu_q, q_start, doc_blocks, meta, kc, vc, w.pos.as_dict(),
                              requests=reqs)
    assert_close(out, ref_o, f"prefill output ({path})")
    err = np.abs(lse.cpu().numpy() - ref_l)
    assert np.isfinite(err).all(), f"{path}: non-finite log-sum-exp"
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, f"{path}: lse max-abs {err.max():.3e} mean {err.mean():.3e}"


# ------------------------------------------------------------------ poisoned caches
POISON_CASES = {  # name -> (workload, requests checked, decode steps, steps checked)
    # 32-token queries of a 4-head group: one live Q tile per CTA; 200-token documents end
    # mid-page; 16 requests x 8 head groups = 128 units: the decode's 12-warp CTAs
    "rag8b_one_q_tile": (lambda: make_workload("rag8b"), [0, 3, 15], 2, {1}),
    # longer ragged queries: two live Q tiles per CTA, a partial second tile, documents of 1..1000
    "two_q_tiles": (lambda: make_custom([200, 37, 1000, 15, 1], [[0, 1, 2], [3, 4, 0], [2]], 8, 2, 128,
                                        PosCfg("rope", 5e5, 128), [70, 33, 100], 2, seed=77), [0, 1, 2], 2, {1}),
    "prefill70b": (lambda: make_workload("prefill70b", batch=2), [0, 1], 0, set()),
    # MQA: prefill and the tensor-core decode mode (key range split over CTAs, merged)
    "mqa_alibi": (lambda: make_workload("mqa_alibi", batch=4), [0, 2], 3, {0, 2}),
}


@pytest.mark.parametrize("case", sorted(POISON_CASES))
def test_poisoned_cache_rows_never_reach_the_output(lk, case):
    """Caches filled with NaN bits before the documents and query tokens are written: only the
    written rows may influence the result.  The output must match the oracle and be bit-identical
    to the same launches over zero-filled caches."""
    import torch
    make, reqs, n_steps, check = POISON_CASES[case]
    got_nan, got_zero = {}, {}
    _run_and_check(lk, make(), reqs, n_steps, check, poison=True, outputs=got_nan)
    _run_and_check(lk, make(), reqs, n_steps, check, poison=False, outputs=got_zero)
    for key in got_zero:
        assert torch.equal(got_nan[key].view(torch.int16), got_zero[key].view(torch.int16)), \
            f"{case} {key}: poisoned cache rows changed the output"


def test_poisoned_cache_no_rotation_twin(lk):
    """The kernels built without positional work (the Delta = 0 twin) over poisoned caches give
    the same bits as over zero-filled ones."""
    import torch
    outs = []
    for poison in (True, False):
        w = make_workload("rag8b", batch=4)
        pb = _batch(w, poison=poison, pos_kind="none")
        pb.fill_documents()
        o_p = pb.prefill(pb.upload_prefill())
        o_d = pb.decode_step(pb.upload_decode(0))
        torch.cuda.synchronize()
        _status_clean(lk)
        assert torch.isfinite(o_p.float()).all() and torch.isfinite(o_d.float()).all()
        outs.append((o_p.view(torch.int16).clone(), o_d.view(torch.int16).clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_poisoned_cache_cold_document_encode(lk):
    """Cold encode of a 130-token document (last page 2 rows) into pages full of NaN bits."""
    import torch
    from position_agnostic_kv_gb300.runner import bits_to_tensor, encode_document
    L, Hq, Hkv, D = 130, 32, 1, 128
    rng = np.random.default_rng([L, D, Hq, 1])
    bf = lambda *shape: f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    q, k, v = bf(L, Hq, D), bf(L, Hkv, D), bf(L, Hkv, D)
    pages = rng.permutation(20)[:9].astype(np.int32)
    dev = torch.device("cuda")
    kc = torch.full((20, Hkv, 16, D), 0, dtype=torch.int16, device=dev).fill_(NAN_BITS).view(torch.bfloat16)
    vc = kc.clone()
    cfg = lk.pos_cfg_from("rope", D, rope_theta=1e4)
    out = encode_document(bits_to_tensor(q, dev), bits_to_tensor(k, dev), bits_to_tensor(v, dev), pages, kc, vc, cfg)
    torch.cuda.synchronize()
    _status_clean(lk)
    ref, _ = lo.materialized_attention([(lo.bf16_bits_to_f64(k), lo.bf16_bits_to_f64(v))], lo.bf16_bits_to_f64(q),
                                       np.arange(L), PosCfg("rope", 1e4, D).as_dict())
    assert_close(out, ref, "cold document over poisoned pages")


def test_no_rotation_twin(lk):
    """The 'Delta = 0' twin (POS_NONE) computes plain attention with no positional term: it
    equals the oracle's ALiBi path with zero slopes (which rotates nothing)."""
    import torch
    w = make_workload("rag8b", batch=3)
    pb = _batch(w, pos_kind="none")
    pb.fill_documents()
    out_p = pb.prefill(pb.upload_prefill())
    out_d = pb.decode_step(pb.upload_decode(0))
    torch.cuda.synchronize()
    _status_clean(lk)
    pos = dict(kind="alibi", alibi_slopes=np.zeros(w.Hq))
    shape = (w.num_pages, w.Hkv, 16, w.D)
    kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    for i in range(len(w.inst_doc)):
        k, v = w.doc_kv(int(w.inst_doc[i]))
        slot, lp = w.inst_slots(i)
        lo.kv_write(k, v, slot, lp, pos, kc, vc)
    q, k, v, slot, lp = w.prefill_tokens()
    lo.kv_write(k, v, slot, lp, pos, kc, vc)
    _, meta, sl, qs, db = oracle_meta(w)
    ref_p, _ = lo.prefill(q, w.cu_q, qs, db, meta, kc, vc, pos, scale=1 / np.sqrt(w.D))
    assert_close(out_p, ref_p, "no-rotation prefill")
    qd, kd, vd, sd, lpd = w.decode_tokens(0)
    lo.kv_write(kd, vd, sd, lpd, pos, kc, vc)
    ref_d, _ = lo.decode(qd, sl + 1, qs, db, meta, kc, vc, pos, scale=1 / np.sqrt(w.D))
    assert_close(out_d, ref_d, "no-rotation decode")


def test_bad_page_sets_status_and_skips(lk):
    """A block word naming a page beyond the cache is caught by the kernel's bounds check:
    the status word gets LAZY_STATUS_BAD_PAGE and the page is skipped (no access)."""
    import torch
    w = make_workload("tiny")
    pb = _batch(w)
    pb.fill_documents()
    bad = pb.meta_h.copy()
    nv, pg, dl, _ = lo.unpack_meta(int(bad[0, 1]))
    bad[0, 1] = lo.pack_meta(nv, pg, dl, w.num_pages + 5)
    pb.meta = torch.from_numpy(bad.view(np.int64)).cuda()
    pb.prefill(pb.upload_prefill())
    st = lk.device_status()
    assert st & 1, st
    assert lk.device_status() == 0  # cleared by the read


def test_workspace_too_small_is_rejected(lk):
    """A batch whose decode splits the key range needs a workspace; 256 bytes is refused."""
    import torch
    w = make_workload("yarn8b", batch=20)
    pb = _batch(w)
    pb.ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lk.LazyError, match="workspace"):
        pb.decode_step(pb.upload_decode(0))


# ------------------------------------------------------------------ CUDA graph replay
@pytest.mark.parametrize("name", ["rag8b", "mqa_alibi"])
def test_graph_replay_matches_eager(lk, name):
    """A whole step (kv_write + prefill, then kv_write + decode for 4 tokens) captured as one
    CUDA graph and replayed gives bit-identical outputs to the same launches made eagerly.
    Every kernel is launched with programmatic dependent launch, so this checks that stream
    order survives graph capture (the kernels are deterministic: no atomics on the data path).
    rag8b decodes on the CUDA-core kernel with a split merge, mqa_alibi on the tensor cores."""
    import torch
    w = make_workload(name, batch=4)
    pb = _batch(w)
    pb.fill_documents()
    pre = pb.upload_prefill()
    decs = [pb.upload_decode(t) for t in range(4)]
    stream = torch.cuda.Stream()

    def step(out_p, outs):
        lk.kv_write(pre["k"], pre["v"], pre["slot"], pre["lp"], pb.k_cache, pb.v_cache, pb.cfg, stream=stream)
        lk.attn_prefill(pre["q"], pb.cu_q, pb.q_start, pb.doc_blocks, pb.meta, pb.k_cache, pb.v_cache,
                        pb.cfg, out_p, pb.max_q, ws=pb.ws, stream=stream)
        for d, o in zip(decs, outs):
            lk.kv_write(d["k"], d["v"], d["slot"], d["lp"], pb.k_cache, pb.v_cache, pb.cfg, stream=stream)
            lk.attn_decode(d["q"], d["seq_len"], pb.q_start, pb.doc_blocks, pb.meta, pb.k_cache,
                           pb.v_cache, pb.cfg, o, ws=pb.ws, stream=stream)

    def buffers():
        return (torch.full((pb.total_q, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda"),
                [torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
                 for _ in decs])

    eager_p, eager_d = buffers()
    with torch.cuda.stream(stream):
        step(eager_p, eager_d)
    stream.synchronize()
    graph_p, graph_d = buffers()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step(graph_p, graph_d)
    for _ in range(2):
        with torch.cuda.stream(stream):
            g.replay()
    stream.synchronize()
    _status_clean(lk)
    assert torch.equal(graph_p.view(torch.int16), eager_p.view(torch.int16)), "prefill differs under graph replay"
    for t, (a, b) in enumerate(zip(graph_d, eager_d)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"decode step {t} differs under graph replay"
    # and the replayed decode of the last token against the oracle
    bt, meta, seq_len, q_start, doc_blocks = oracle_meta(w)
    pos = w.pos.as_dict()
    kc, vc = oracle_caches_for(w, prefill=True, decode_steps=4)
    ref, _ = lo.decode(w.decode_tokens(3)[0], seq_len + 4, q_start, doc_blocks, meta, kc, vc, pos,
                       requests=list(range(w.B)))
    assert_close(graph_d[3], ref, f"{name} decode step 3 under graph replay")
