"""The bench's multi-rank host logic on CPU: two gloo ranks (127.0.0.1), no GPU.

The path shards with no exchange (replicas only), so what N > 1 adds is host-side: the barrier,
the max over ranks of the step time, the whole-job throughput, and rank 0 alone printing.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        # rank r times steps of (r + 1) ms: the job's step time is the slowest rank's
        value, ms = bench.job_throughput(d, 100, [float(rank + 1)] * 4)
        q.put((rank, d.world, ms, value))
    finally:
        d.close()


def test_two_gloo_ranks_take_the_slowest_step():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, world, ms, value in got:
        assert world == 2
        assert ms == pytest.approx(2.0)                 # max over ranks of the mean step time
        assert value == pytest.approx(2 * 100 / 2e-3)   # all ranks' tokens / slowest step


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_prefill_roof_by_arithmetic_intensity():
    """The bench names the roof of a prefill launch by its FLOPs per unique HBM byte against
    the ridge of the measured peaks: the 70B shape's two 128-row Q tiles per KV head sit above
    it (tensor-bound), the 32-token RAG and YaRN queries over long contexts below (HBM-bound)."""
    import types
    sys.path.insert(0, ROOT)
    import bench
    from workloads import make_workload
    peaks = {"bf16_tflops": 1932.3, "hbm_gbs": 6784.5}
    bounds = {}
    for name in ("prefill70b", "rag8b", "yarn8b", "mqa_alibi"):
        w = make_workload(name, sharing="private")
        q_start = [int(w.inst_len[w.req_inst[w.req_inst_off[b]:w.req_inst_off[b + 1]]].sum()) for b in range(w.B)]
        pb = types.SimpleNamespace(q_start_h=q_start, total_q=int(w.q_len.sum()))
        flops, nbytes = bench.prefill_flops(w, pb), bench.prefill_bytes(w, pb)
        roof = bench.prefill_roof(flops, nbytes, 100.0, peaks)
        assert abs(roof["ridge_flop_per_byte"] - 1932.3e12 / 6784.5e9) < 1e-9
        assert abs(roof["hbm_gbs"] - nbytes / 100e-6 / 1e9) < 1e-6 * roof["hbm_gbs"]
        bounds[name] = roof["bound"]
    assert bounds == {"prefill70b": "tensor", "rag8b": "hbm", "yarn8b": "hbm", "mqa_alibi": "tensor"}
