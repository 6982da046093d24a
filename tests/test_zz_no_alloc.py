"""Decode for callers that cannot allocate device memory.

Some users of this library cannot call cudaMalloc: an engine that reserves all of HBM for its
own KV pool at start-up and gives plugins no allocator, or a latency-bound decode loop that
must never allocate (cudaMalloc can synchronise the device).  They cannot pass the split-KV
workspace that lazy_attn_decode needs, so the library offers lazy_attn_decode_noalloc, whose
scratch is a fixed 16 MiB array compiled into the library.

This test calls that entry point through the C ABI and checks it against lazy_attn_decode
(with a caller workspace) on the same inputs, on two calls in a row: the second call reuses
the array the first one left behind.  Both calls run the same kernels on the same inputs, so
their outputs must be bit-identical.  Two head groupings: 4 heads per KV head (the CUDA-core
decode split over the key range, 20 requests of the YaRN workload, and its merge) and 32 (MQA: the tensor-core decode, its key range split over CTAs
and merged).  It lives in a file of its own, collected last, so that a run stopping at the
first failure has run every other test first; it needs nothing from them.
"""
import ctypes

import numpy as np
import pytest

from tests.gpu_common import assert_close, lib
from workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,batch", [("yarn8b", 20), ("mqa_alibi", 4)])
def test_noalloc_decode_matches_workspace_decode_on_two_calls(name, batch):
    import torch
    lk = lib()
    from position_agnostic_kv_gb300.runner import PagedBatch

    w = make_workload(name, batch=batch)  # every request over ~12 000 keys
    pb = PagedBatch(w, device="cuda")
    need = lk.workspace_size(lk.PHASE_DECODE, w.B, w.B, pb.max_blocks, w.Hq, w.Hkv, w.D)
    assert need > 0, "this batch must use split scratch for the test to mean anything"
    pb.fill_documents()
    pb.prefill(pb.upload_prefill())
    stream = torch.cuda.current_stream()
    for t in (0, 1):  # two calls in a row
        inp = pb.upload_decode(t)
        lk.kv_write(inp["k"], inp["v"], inp["slot"], inp["lp"], pb.k_cache, pb.v_cache, pb.cfg)
        ref = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lk.attn_decode(inp["q"], inp["seq_len"], pb.q_start, pb.doc_blocks, pb.meta, pb.k_cache,
                       pb.v_cache, pb.cfg, ref, ws=pb.ws)
        got = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lk.lib.lazy_attn_decode_noalloc(
            ctypes.c_void_p(inp["q"].data_ptr()), ctypes.c_void_p(inp["seq_len"].data_ptr()),
            ctypes.c_void_p(pb.q_start.data_ptr()), ctypes.c_void_p(pb.doc_blocks.data_ptr()),
            ctypes.c_void_p(pb.meta.data_ptr()), w.B, pb.max_blocks,
            ctypes.c_void_p(pb.k_cache.data_ptr()), ctypes.c_void_p(pb.v_cache.data_ptr()),
            w.num_pages, w.Hq, w.Hkv, w.D, ctypes.c_float(0.0), ctypes.byref(pb.cfg),
            ctypes.c_void_p(got.data_ptr()), None, ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, lk.lib.lazy_last_error()
        torch.cuda.synchronize()
        assert lk.device_status() == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), \
            f"{name}: no-alloc decode call {t + 1} differs from the workspace decode"
        assert_close(got, ref.float().cpu().numpy().astype(np.float64), f"{name} no-alloc decode call {t + 1}")
