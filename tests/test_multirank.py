"""The N > 1 benchmark path on the CPU: two gloo ranks on 127.0.0.1.

Covers the parts of `bench.py` that differ from the single-GPU run: process-group set-up from
the launcher's environment, the barrier, the max-over-ranks reduction of the timed region, the
whole-job (weak-scaling) tokens/s, and the reference arm's rule that only rank 0 runs and prints.
No GPU and no collective on a data path are involved (sequences are independent)."""

import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code: str, world: int = 2, timeout: float = 180.0):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(world), LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), PYTHONPATH=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_barrier_max_and_job_value():
    code = textwrap.dedent("""
        import json
        import bench
        dist, rank, world, local = bench._dist_setup()
        assert dist is not None and world == 2 and local == rank
        dist.barrier()
        mx = bench._barrier_max(dist, 10.0 + 5.0 * rank)   # rank 1 is the slow one: 15 ms
        value = bench._job_value(world, 8192, 100, mx)
        print(json.dumps({"rank": rank, "max": mx, "value": value}))
        dist.barrier()
        dist.destroy_process_group()
    """)
    outs = [json.loads(o.strip().splitlines()[-1]) for o in _run_ranks(code)]
    assert [o["rank"] for o in outs] == [0, 1]
    for o in outs:
        assert o["max"] == 15.0                                # every rank sees the slowest rank's time
        assert abs(o["value"] - 2 * 8192 * 100 / 0.015) < 1e-6 * o["value"]  # both ranks' tokens


def test_job_value_is_weak_scaling():
    import bench

    one = bench._job_value(1, 8192, 100, 10.0)
    assert bench._job_value(2, 8192, 100, 10.0) == 2 * one   # same per-rank work, same time: twice the job
    assert bench._job_value(2, 8192, 100, 20.0) == one       # the slowest rank sets the job's time


def test_reference_arm_runs_on_rank_zero_only():
    code = textwrap.dedent("""
        import types
        import bench
        from weight_linear_attention_gb300 import inputs as I
        w = I.WORKLOADS["f1_tiny_fp32"]
        args = types.SimpleNamespace(steps=1, warmup=1, ref_batch=1, gpus=2)
        bench.run_reference(args, w)
    """)
    outs = _run_ranks(code)
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    assert len(lines0) == 1
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert not [l for l in outs[1].splitlines() if l.startswith("{")]  # rank 1: no work, no line


def test_backward_reference_arm_runs_on_rank_zero_only():
    code = textwrap.dedent("""
        import types
        import bench
        from weight_linear_attention_gb300 import inputs as I
        w = I.WORKLOADS["f1_bwd_b8h12t1024_bf16"].with_(seqlen=64)
        args = types.SimpleNamespace(steps=1, warmup=1, gpus=2)
        bench.run_reference_bwd(args, w)
    """)
    outs = _run_ranks(code)
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    assert len(lines0) == 1
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["metric"] == "falcon_bwd_tokens_per_s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["d2h_bytes_per_step"] == 0
    assert not [l for l in outs[1].splitlines() if l.startswith("{")]
