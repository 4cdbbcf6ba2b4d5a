"""Host-side accounting of the benchmark, without a GPU: the algorithmic bytes and flops
its roofline fractions divide by, the reference arm's output line (the oracle timed on
the host cores) on the tiny workload, and the replica path's timing over two gloo ranks."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from diffusion_lookahead_decoding_gb300 import synth  # noqa: E402


def test_weight_bytes_are_the_qwen25_7b_parameter_count():
    """The verification step reads every weight once except the input embedding (only its
    gathered rows): 2 bytes x (7,615,283,200 - 152064 x 3584), the published size of the
    Qwen2.5-7B architecture that Dream-7B shares, less its embedding table."""
    shape, _ = synth.WORKLOADS["dream7b"]
    total_params = 7_615_283_200
    embed = 152064 * 3584
    by0, _ = bench.verify_bytes_flops(shape, T=256, P=0, B=32)
    kv_block = 256 * 28 * 2 * 4 * 128 * 2  # the 256 rows' K and V, bf16
    assert by0 - kv_block == 2 * (total_params - embed)


def test_verification_bytes_and_flops_hand_count():
    shape, _ = synth.WORKLOADS["dream7b"]
    by, fl = bench.verify_bytes_flops(shape, T=256, P=640, B=32)
    per_layer = 3584 * (28 * 128 + 2 * 4 * 128) + 28 * 128 * 3584 + 3 * 3584 * 18944
    params = 28 * per_layer + 152064 * 3584
    kv_row = 28 * 2 * 4 * 128 * 2  # bytes of one position's K and V over all layers
    assert by == 2 * params + (640 + 256) * kv_row
    # 2 flops per weight per row; q.k and p.v: 2 x 2 flops per (query head, key, dim).
    assert fl == 2 * params * 256 + 28 * 4 * 28 * 128 * 256 * (640 + 32)


def test_prefill_flops_hand_count():
    shape, _ = synth.WORKLOADS["dream7b"]
    proj = 3584 * (4608 + 3584 + 2 * 18944) + 18944 * 3584  # weights of one layer
    attn = 4 * 28 * 128 * 512 * 512  # q.k and p.v over the 512 x 512 prompt block
    assert bench.prefill_flops(shape, 512) == 28 * (2 * proj * 512 + attn)


def test_gemm_bytes_per_kind():
    shape, _ = synth.WORKLOADS["dream7b"]
    T = 256
    assert bench.gemm_bytes(shape, T, 2) == 2 * 2 * 18944 * 3584 + 2 * T * 3584 + 2 * T * 18944
    assert bench.gemm_flops(shape, T, 3) == 2 * 3584 * 18944 * T


def _run_bench(args, env_extra=None, timeout=600):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny"


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                   env_extra={"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"}, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def _replica(rank, world, port, seconds, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.replica_barrier(world)
        t = bench.max_over_ranks(seconds[rank], world)
        out.put((rank, t, bench.job_throughput(256, world, t)))
    finally:
        dist.destroy_process_group()


def test_replicas_report_the_slowest_rank_over_gloo():
    """Two CPU ranks (gloo, world size 2): both see the slower rank's time, and the job's
    tokens/s counts both replicas' tokens over it."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    seconds = [0.5, 0.8]
    procs = [ctx.Process(target=_replica, args=(r, 2, port, seconds, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [0.8, 0.8]
    assert all(abs(g[2] - 2 * 256 / 0.8) < 1e-9 for g in got)


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(0.25, 1) == 0.25
    bench.replica_barrier(1)
    assert bench.job_throughput(256, 1, 0.5) == 512.0
