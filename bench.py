"""Benchmark of the LoPA branch-verification path on one GB300.

A step is one whole single-sample decode of the workload: gen_len tokens in 32-token
blocks, each block = one block-start forward + LoPA iterations (decide, 8-branch
isolated verification forward, select, Commit-Winner), all inside the library's CUDA
graphs.  Inputs (weights, prompt K/V) are resident in HBM before the timed region; each
step rewinds the decoder to the end of the prompt and decodes again (nothing cached:
every forward re-streams the 15 GB of weights, far larger than L2).

Prints one JSON line (see the keys below).  --impl reference times the CPU oracle on
the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes as C
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decoded tokens/s per sample (Dream-7B-shaped, 8 branches)"
UNIT = "tokens/s"
# ASSUMED tokens per forward of the 7B workloads, used only by the reference arm to turn
# the oracle's measured seconds per verification forward into tokens/s: the oracle cannot
# finish a 7B decode within a bounded sample.  The value is the unmerged count (tokens /
# (iterations + blocks), the oracle's own way of counting) that the CUDA path measured on
# this workload, 8.0 to 8.8 across runs (the random-weight model's greedy decisions move
# with summation order).  The reference arm's line labels it as assumed.  The oracle's own
# TPF is measured on the tiny and small workloads (oracle_decodes in the default run).
ASSUMED_TPF = {"dream7b": 8.4, "dream7b_scaling": 8.4}
# DRAM bytes (read + write) of one gemm_kernel<SWIGLU> launch at the 7B step shape (256 rows),
# from ncu on the one-layer slice (profiles/gemm_swiglu_dream7b_layer.md: 273.47 MB read,
# 1.73 MB written on average over two launches).  It describes the kernel as it was
# profiled and must be re-taken (or set to None) when the kernel changes.
SWIGLU_TRAFFIC_BYTES = 275.20e6


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def replica_barrier(world: int):
    """Barrier over the replicas (gloo), a no-op for one process."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(seconds: float, world: int) -> float:
    """The job's time: the slowest replica's (every rank gets the same value)."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job tokens/s: every replica decodes the same workload (weak scaling), and the
    job ends with the slowest one."""
    return world * tokens_per_rank / seconds


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # nvidia-smi's start-up (NVML initialisation) briefly stalls this process's GPU
        # work; let it finish before the timed region opens.
        t0 = time.perf_counter()
        while not self.rows and self.proc.poll() is None and time.perf_counter() - t0 < 10.0:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows if len(r) >= 9
                          for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def oracle_seconds_per_forward(shape, dshape, weights, budget_s: float):
    """Oracle (float64, bf16 storage) time of one nb x B verification forward, timed on
    1 and 2 layers plus the LM head and extrapolated linearly to all layers."""
    import dataclasses
    from oracle import lopa_oracle as O
    nb, B, P = dshape.k + 1, dshape.block, dshape.prompt_len
    rng = np.random.default_rng(0)
    br = rng.integers(1, shape.vocab, (nb, B))
    br[rng.random((nb, B)) < 0.5] = shape.mask_id
    times = {}
    for n_l in (1, 2):
        sh = dataclasses.replace(shape, n_layers=n_l)
        m = O.OracleModel(sh, weights, act="bf16", cache_weights=False)
        cache = O.KVCache.empty(sh, P + B)
        for l in range(n_l):
            cache.k[l][:P] = rng.standard_normal(cache.k[l][:P].shape)
            cache.v[l][:P] = rng.standard_normal(cache.v[l][:P].shape)
        t0 = time.perf_counter()
        O.forward(m, cache, P, br)
        times[n_l] = time.perf_counter() - t0
    per_layer = max(times[2] - times[1], 1e-9)
    fixed = max(times[1] - per_layer, 0.0)
    return fixed + per_layer * shape.n_layers, times


def bench_config(args, shape, dshape, world):
    """The `config` object of both arms' output lines."""
    return {"workload": args.workload,
            "model": f"Qwen2.5-7B-architecture diffusion LM shape ({shape.n_layers} layers, "
                     f"d {shape.d_model}, vocab {shape.vocab}), random init",
            "prompt": dshape.prompt_len, "gen_len": dshape.gen_len, "block": dshape.block,
            "branches": dshape.k + 1, "tau": dshape.tau,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "inputs larger than L2 (15 GB weights re-streamed per forward)",
            "weights": getattr(args, "weight_format", "bf16")}


def oracle_decode_run(name, threads, max_blocks=None):
    """The oracle's full decode of a workload (prompt, then LoPA blocks), timed in this
    process; returns tokens, forwards (its own unmerged count), iterations and seconds."""
    from oracle import lopa_oracle as O
    from diffusion_lookahead_decoding_gb300 import synth
    shape, dshape = synth.WORKLOADS[name]
    w = synth.make_weights(shape, 0, threads=1)
    m = O.OracleModel(shape, w, act="bf16")
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    gen = dshape.gen_len if max_blocks is None else min(dshape.gen_len, max_blocks * dshape.block)
    O.forward(m, O.KVCache.empty(shape, dshape.prompt_len), 0, prompt[None, :8])  # warm caches
    t0 = time.perf_counter()
    toks, fw, _, log = O.decode(m, prompt, dshape.block, dshape.k, dshape.tau, gen, record=True)
    sec = time.perf_counter() - t0
    return {"tokens": int(len(toks)), "forwards": int(fw), "iterations": len(log),
            "seconds": sec, "threads": threads}


def oracle_decode_subprocess(name, threads, max_blocks=None, timeout=600):
    """oracle_decode_run in a fresh interpreter limited to `threads` BLAS / torch threads
    (the thread count has to be fixed before numpy loads)."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-decode", name,
           "--threads", str(threads)] + (["--max-blocks", str(max_blocks)] if max_blocks else [])
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=timeout)
    line = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode or not line:
        return {"error": (r.stderr or r.stdout)[-300:]}
    d = json.loads(line[-1])
    d["tok_per_s"] = d["tokens"] / d["seconds"]
    d["tpf"] = d["tokens"] / d["forwards"]
    d["ms_per_forward"] = d["seconds"] * 1e3 / max(1, d["forwards"])
    return d


def oracle_decodes():
    """Full oracle decodes of the tiny and small workloads on 1 core and on all cores (the
    small one on 1 core only for its first block, labelled), beside the GPU numbers."""
    cores = os.cpu_count() or 1
    out = {"cores": cores}
    out["tiny"] = {"1_core": oracle_decode_subprocess("tiny", 1),
                   "all_cores": oracle_decode_subprocess("tiny", cores)}
    out["small"] = {"1_core_first_block": oracle_decode_subprocess("small", 1, max_blocks=1),
                    "all_cores": oracle_decode_subprocess("small", cores)}
    return out


def run_reference_decode(args, shape, dshape, world):
    """Reference arm on a workload the oracle decodes in seconds: every step is one whole
    oracle decode (prompt + all blocks), so tokens/s and TPF are both measured."""
    for _ in range(args.warmup):
        oracle_decode_run(args.workload, os.cpu_count())
    runs = [oracle_decode_run(args.workload, os.cpu_count()) for _ in range(max(1, args.steps))]
    sec = sum(r["seconds"] for r in runs)
    tok = sum(r["tokens"] for r in runs)
    value = tok / sec
    tpf = runs[0]["tokens"] / runs[0]["forwards"]
    sample = (f"oracle (numpy float64, bf16 storage) full decode of the workload, "
              f"{len(runs)} step(s) of {runs[0]['tokens']} tokens, measured TPF {tpf:.2f}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3 / len(runs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(args, shape, dshape, world),
        "tpf": tpf, "tpf_source": "measured by this run",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from diffusion_lookahead_decoding_gb300 import synth
    shape, dshape = synth.WORKLOADS[args.workload]
    if args.workload not in ASSUMED_TPF:
        return run_reference_decode(args, shape, dshape, world)
    weights = synth.make_weights(shape, 0)
    tpf = ASSUMED_TPF[args.workload]
    for _ in range(args.warmup):
        oracle_seconds_per_forward(shape, dshape, weights, 0)
    t0 = time.perf_counter()
    per_fwd = []
    for _ in range(args.steps):
        s, _ = oracle_seconds_per_forward(shape, dshape, weights, 0)
        per_fwd.append(s)
    wall = time.perf_counter() - t0
    spf = statistics.mean(per_fwd)
    value = tpf / spf
    cores = os.cpu_count()
    sample = (f"oracle (numpy float64, bf16 storage) {dshape.k + 1}x{dshape.block}-token "
              f"verification forward timed at 1 and 2 layers + LM head, extrapolated to "
              f"{shape.n_layers} layers ({spf:.1f} s/forward); tokens/s = ASSUMED TPF {tpf} "
              f"(the CUDA path's measured unmerged TPF on this workload) / that")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(args, shape, dshape, world),
        "tpf": tpf, "tpf_source": "assumed (the CUDA path's measured unmerged TPF on this "
                                  "workload); the oracle's seconds per forward are measured",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def gemm_bytes(shape, T, kind, wb=2):
    """Algorithmic HBM bytes of one launch: weights once (wb bytes per weight: 2 for bf16,
    1 for E4M3 codes, plus 4 bytes of scale per weight row), activations in, outputs out."""
    d, F, V = shape.d_model, shape.ffn, shape.vocab
    sc = 4 if wb == 1 else 0
    if kind == 0:
        return (wb * d + sc) * shape.qkv_rows + 2 * T * d + 4 * T * shape.qkv_rows
    if kind == 1:
        return (wb * shape.n_heads * shape.head_dim + sc) * d + 2 * T * shape.n_heads * shape.head_dim + 4 * T * d
    if kind == 2:
        return (wb * d + sc) * 2 * F + 2 * T * d + 2 * T * F
    if kind == 3:
        return (wb * F + sc) * d + 2 * T * F + 4 * T * d
    return (wb * d + sc) * V + 2 * T * d + 12 * T * ((V + 255) // 256)


def gemm_flops(shape, T, kind):
    d, F, V = shape.d_model, shape.ffn, shape.vocab
    n = {0: shape.qkv_rows * d, 1: d * shape.n_heads * shape.head_dim, 2: 2 * F * d, 3: d * F,
         4: V * d}[kind]
    return 2 * n * T


def verify_bytes_flops(shape, T, P, B, wb=2):
    """Algorithmic bytes and flops of one verification forward over T token rows (blocks
    of B) at prefix P: every weight read once (projections and LM head; wb bytes per weight,
    2 for bf16, 1 for E4M3 codes plus 4 bytes of scale per row), the prefix K/V read once and
    the block K/V written once (bf16); 2 flops per weight per row plus the attention's q.k
    and p.v (4 per query, key and dimension, P + B keys per query)."""
    L, d, H, Hk, dh, F, V = (shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                             shape.head_dim, shape.ffn, shape.vocab)
    params = L * (d * H * dh + 2 * d * Hk * dh + H * dh * d + 3 * d * F) + V * d
    rows = L * (H * dh + 2 * Hk * dh + d + 2 * F + d) + V
    kv = L * 2 * Hk * dh * 2
    by = wb * params + (4 * rows if wb == 1 else 0) + P * kv + T * kv
    fl = 2 * params * T + 4 * L * H * dh * T * (P + B)
    return by, fl


def prefill_flops(shape, P):
    """Flops of the prompt forward over P tokens: 2 per projection weight per token (no LM
    head) plus q.k and p.v over the P x P bidirectional prompt block."""
    L = shape.n_layers
    proj = sum(gemm_flops(shape, P, kind) for kind in range(4))
    return L * (proj + 4 * shape.n_heads * shape.head_dim * P * P)


def e4m3_summary(api, shape, dshape, dev_w, prompt, peak_bw, peak_tc, steps):
    """The same workload with the E4M3 weight stream (a second context quantising the same
    device weights): decode tokens/s and TPF over `steps` decodes after one warm-up, the
    verification forward against its roofline on the halved weight bytes, the block-start
    forward, and the gate/up GEMM and LM head."""
    import torch
    B, P0, gen = dshape.block, dshape.prompt_len, dshape.gen_len
    dec = api.LopaDecoder(shape, dev_w, B, dshape.k, dshape.tau, P0, P0 + gen, weight_format="e4m3")
    dec.prefill(prompt)
    dec.rewind(P0)
    dec.decode(gen)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(dec.stream)
    toks = fw = 0
    for _ in range(steps):
        dec.rewind(P0)
        _, st = dec.decode(gen)
        toks += st["tokens"]
        fw += st["forwards"]
    ev1.record(dec.stream)
    torch.cuda.synchronize()
    sec = ev0.elapsed_time(ev1) / 1e3
    T = (dshape.k + 1) * B
    Pv = P0 + (gen // 2 // B) * B
    dec.rewind(Pv)
    v_med, _ = dec.time_forward(1, 50)
    s_med, _ = dec.time_forward(0, 50)
    vb, vf = verify_bytes_flops(shape, T, Pv, B, 1)
    gu = dec.time_gemm(2, 2 * shape.n_layers)
    lm = dec.time_gemm(4, 8)
    dec.close()
    gb = gemm_bytes(shape, T, 2, 1)
    lb = gemm_bytes(shape, T, 4, 1)
    return {"tokens_per_s": toks / sec, "tpf": toks / fw, "ms_per_forward": sec * 1e3 / fw,
            "decodes": steps,
            "verify_step": {"ms_median": v_med, "prefix": Pv, "rows": T, "bytes": vb,
                            "hbm_roofline_ms": vb / peak_bw / 1e6,
                            "tensor_roofline_ms": vf / peak_tc / 1e9,
                            "frac_hbm_roofline": vb / peak_bw / 1e6 / v_med,
                            "block_start_forward_ms_median": s_med},
            "gate_up_swiglu": {"ms": gu, "GB/s": gb / gu / 1e6, "frac_hbm": gb / gu / 1e6 / peak_bw,
                               "TFLOP/s": gemm_flops(shape, T, 2) / gu / 1e9},
            "lm_head": {"ms": lm, "GB/s": lb / lm / 1e6, "TFLOP/s": gemm_flops(shape, T, 4) / lm / 1e9}}


def kernel_table(args):
    """Per-kernel CUDA-event times of the five projection GEMMs (layers cycled) and the
    verification-forward latency for bf16 and E4M3 weights at k in {0, 3, 7} (32, 128 and
    256 token rows) on the 7B shape, with each GEMM's fraction of the measured HBM peak on its
    own algorithmic bytes."""
    import torch
    from diffusion_lookahead_decoding_gb300 import api, build, synth
    build.build()
    shape, dshape = synth.WORKLOADS["dream7b"]
    w = synth.make_weights(shape, 0)
    dw = api.upload_weights(shape, w)
    del w
    bw, _, _, src = _peaks()
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    B, P0, gen = dshape.block, dshape.prompt_len, dshape.gen_len
    rows = []
    for fmt in ("bf16", "e4m3"):
        for k in (0, 3, 7):
            dec = api.LopaDecoder(shape, dw, B, k, dshape.tau, P0, P0 + gen, weight_format=fmt)
            dec.prefill(prompt)
            T, wb = (k + 1) * B, 1 if fmt == "e4m3" else 2
            row = {"weights": fmt, "k": k, "rows": T}
            for kind, name in enumerate(["qkv", "o_proj", "gate_up_swiglu", "down", "lm_head"]):
                ms = dec.time_gemm(kind, 2 * shape.n_layers if kind < 4 else 8)
                row[name] = {"us": ms * 1e3, "frac_hbm": gemm_bytes(shape, T, kind, wb) / ms / 1e6 / bw}
            dec.decode(gen)
            dec.rewind(P0 + (gen // 2 // B) * B)
            row["verify_ms"] = dec.time_forward(1, 30)[0]
            row["block_start_ms"] = dec.time_forward(0, 30)[0]
            dec.close()
            rows.append(row)
            print(json.dumps(row), flush=True)
    print(json.dumps({"kernel_table": rows, "peaks": {"hbm_gbs": bw, "source": src}}), flush=True)


def _peaks():
    try:
        p = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops_sustained", 1700.0)), \
            float(p.get("bf16_tflops", 1900.0)), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1700.0, 1900.0, "fallback"


def sweep_branches(args):
    """Branch scaling on the 7B shape with a 2048-token prompt and 512 generated tokens:
    for k in {0, 1, 3, 7, 15} (1 to 16 branches) a whole decode (tokens/s, TPF) and the
    verification-forward latency at a mid-decode prefix against its HBM and tensor
    rooflines (k = 0 is plain confidence-driven threshold decoding)."""
    import dataclasses
    import torch
    from diffusion_lookahead_decoding_gb300 import api, build, synth
    build.build()
    shape, dshape = synth.WORKLOADS["dream7b_scaling"]
    w = synth.make_weights(shape, 0)
    dw = api.upload_weights(shape, w)
    del w
    bw, tc_s, _, src = _peaks()
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    rows = []
    for k in (0, 1, 3, 7, 15):
        ds = dataclasses.replace(dshape, k=k)
        B, P0, gen = ds.block, ds.prompt_len, ds.gen_len
        dec = api.LopaDecoder(shape, dw, B, k, ds.tau, P0, P0 + gen, weight_format=args.weight_format)
        dec.prefill(prompt)
        dec.decode(gen)  # warm-up
        times, stats = [], None
        for _ in range(max(1, args.steps)):
            dec.rewind(P0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(dec.stream)
            _, stats = dec.decode(gen)
            e1.record(dec.stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / 1e3)
        sec = statistics.median(times)
        Pv = P0 + (gen // 2 // B) * B
        dec.rewind(Pv)
        v_med, _ = dec.time_forward(1, 30)
        T = (k + 1) * B
        vb, vf = verify_bytes_flops(shape, T, Pv, B, 1 if args.weight_format == "e4m3" else 2)
        t_hbm, t_tc = vb / bw / 1e6, vf / tc_s / 1e9
        rows.append({"k": k, "branches": k + 1, "tok_per_s": gen / sec,
                     "tpf": stats["tokens"] / stats["forwards"],
                     "tpf_unmerged": stats["tokens"] / (stats["steps"] + stats["blocks"]),
                     "forwards": stats["forwards"], "iterations": stats["steps"],
                     "verify_ms": v_med, "verify_prefix": Pv, "verify_rows": T,
                     "frac_hbm_roofline": t_hbm / v_med, "frac_tensor_roofline": t_tc / v_med,
                     "bound": "hbm" if t_hbm >= t_tc else "tensor"})
        dec.close()
        print(json.dumps(rows[-1]), flush=True)
    print(json.dumps({"sweep_branches": rows, "workload": "dream7b_scaling", "prompt": dshape.prompt_len,
                      "weights": args.weight_format,
                      "gen_len": dshape.gen_len, "peaks": {"hbm_gbs": bw, "bf16_tflops_sustained": tc_s,
                                                           "source": src}}), flush=True)


def microbench(args):
    """Branch-isolated attention and the fused LM head on the 7B layer dims over branches
    {1,2,4,8,16} x block {16,32,64} x committed prefix {256,1024,4096,8192}: CUDA-event time
    per launch, algorithmic GB/s and TFLOP/s against the measured peaks.  The LM head runs
    over the masked rows only (mask fraction of each block uniform in [0.25, 1], seed 2)."""
    import torch
    from diffusion_lookahead_decoding_gb300 import api, build, synth
    build.build()
    bw, tc_s, tc_b, src = _peaks()
    H, Hk, dh, d, V = 28, 4, 128, 3584, 152064

    def timed(fn, n=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n * 1e3  # us

    attn = []
    for nb in (1, 2, 4, 8, 16):
        for B in (16, 32, 64):
            for P in (256, 1024, 4096, 8192):
                T = nb * B
                ins = [x.cuda() for x in synth.make_attention_inputs(nb, B, P, H, Hk, dh, seed=7)]
                pack = api.attention_layouts(*ins)
                us = timed(lambda: api.branch_attention_call(pack))
                by = 2 * (2 * T * H * dh + 2 * P * Hk * dh + 2 * T * Hk * dh)
                fl = 4 * H * dh * T * (P + B)
                attn.append({"branches": nb, "block": B, "prefix": P, "us": us,
                             "GB/s": by / us / 1e3, "TFLOP/s": fl / us / 1e6,
                             "frac_tensor_burst": fl / us / 1e6 / tc_b})
                del ins, pack
    api.kernel_status()
    g = torch.Generator().manual_seed(2)
    wl = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16).cuda()
    lm = []
    for nb in (1, 2, 4, 8, 16):
        for B in (16, 32, 64):
            frac = torch.rand(nb, generator=g) * 0.75 + 0.25
            rows = int(sum(max(1, round(float(f) * B)) for f in frac))
            h = torch.randn(rows, d, generator=g).to(torch.bfloat16).cuda()
            us = timed(lambda: api.lmhead_argmax(h, wl, 20.0, 0))
            by = 2 * V * d + 2 * rows * d + 12 * rows * ((V + 255) // 256)
            fl = 2 * rows * d * V
            lm.append({"branches": nb, "block": B, "rows": rows, "us": us,
                       "GB/s": by / us / 1e3, "frac_hbm": by / us / 1e3 / bw,
                       "TFLOP/s": fl / us / 1e6, "frac_tensor_burst": fl / us / 1e6 / tc_b})
    api.kernel_status()
    print(json.dumps({"microbench": {"attention": attn, "lm_head": lm,
                                     "dims": {"H": H, "Hk": Hk, "head_dim": dh, "d_model": d, "vocab": V},
                                     "peaks": {"hbm_gbs": bw, "bf16_tflops_burst": tc_b, "source": src}}}),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dream7b")
    ap.add_argument("--k", type=int, default=None, help="override the lookahead branch count")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--profile-gemm", type=int, default=None,
                    help="only launch this projection GEMM kind 3 times (for ncu captures)")
    ap.add_argument("--profile-decode", action="store_true",
                    help="prefill + warmup decodes + steps decodes, no timing (for ncu launch lists)")
    ap.add_argument("--oracle-decode", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--threads", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--max-blocks", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--sweep-branches", action="store_true",
                    help="branch-scaling table on the 2048-token-prompt workload, k in 0,1,3,7,15")
    ap.add_argument("--kernel-table", action="store_true",
                    help="per-GEMM times and verification latency, bf16 vs E4M3 weights, k in 0,3,7")
    ap.add_argument("--microbench", action="store_true",
                    help="attention + LM-head grid: branches x block x prefix")
    ap.add_argument("--weight-format", default="bf16", choices=["bf16", "e4m3"],
                    help="weights the GEMMs stream: bf16, or per-row-scaled E4M3 codes")
    ap.add_argument("--profile-attention", type=int, default=None, metavar="PREFIX",
                    help="only the branch attention of the workload's verification step over a "
                         "PREFIX-key prefix: 3 + 20 launches, CUDA-event time (small ncu case)")
    args = ap.parse_args()
    if args.oracle_decode:
        import torch
        torch.set_num_threads(args.threads)
        print(json.dumps(oracle_decode_run(args.oracle_decode, args.threads, args.max_blocks)),
              flush=True)
        return
    if args.sweep_branches:
        return sweep_branches(args)
    if args.microbench:
        return microbench(args)
    if args.kernel_table:
        return kernel_table(args)
    profiling = args.profile_decode or args.profile_gemm is not None or args.profile_attention is not None
    if args.warmup < 3 and args.impl == "ours" and not profiling:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    from diffusion_lookahead_decoding_gb300 import api, build, synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")  # replicas only: used for the barrier and the max
    build.build()
    shape, dshape = synth.WORKLOADS[args.workload]
    if args.k is not None:
        import dataclasses
        dshape = dataclasses.replace(dshape, k=args.k)
    B, P0, gen = dshape.block, dshape.prompt_len, dshape.gen_len
    if args.profile_attention is not None:
        nb = dshape.k + 1
        ins = [x.cuda() for x in synth.make_attention_inputs(
            nb, B, args.profile_attention, shape.n_heads, shape.n_kv_heads, shape.head_dim, seed=7)]
        pack = api.attention_layouts(*ins)
        for _ in range(3):
            api.branch_attention_call(pack)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(20):
            api.branch_attention_call(pack)
        e1.record()
        torch.cuda.synchronize()
        print(json.dumps({"profile_attention": {"prefix": args.profile_attention, "rows": nb * B,
                                                "us": e0.elapsed_time(e1) / 20 * 1e3}}), flush=True)
        return
    t_gen = time.perf_counter()
    weights = synth.make_weights(shape, 0)
    dev_w = api.upload_weights(shape, weights)
    if args.no_cpu_baseline or rank != 0 or args.profile_decode or args.profile_gemm is not None:
        del weights
        weights = None
    t_gen = time.perf_counter() - t_gen
    dec = api.LopaDecoder(shape, dev_w, B, dshape.k, dshape.tau, P0, P0 + gen,
                          weight_format=args.weight_format)
    wb = 1 if args.weight_format == "e4m3" else 2
    if args.profile_gemm is not None:
        ms = dec.time_gemm(args.profile_gemm, 3)
        print(json.dumps({"profile_gemm": args.profile_gemm, "ms": ms}), flush=True)
        dec.close()
        return
    prompt = synth.make_prompt(shape, P0, seed=1 + rank)
    dec.prefill(prompt)
    if args.profile_decode:
        for _ in range(args.warmup + args.steps):
            dec.rewind(P0)
            _, st = dec.decode(gen)
        torch.cuda.synchronize()
        print(json.dumps({"profile_decode": st}), flush=True)
        dec.close()
        return

    def one_step():
        dec.rewind(P0)
        return dec.decode(gen)

    for _ in range(args.warmup):
        one_step()
    stats = []

    with ClockSampler(local) as clocks:
        replica_barrier(world)
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(dec.stream)
        for _ in range(args.steps):
            toks, st = one_step()
            stats.append(st)
        ev1.record(dec.stream)
        torch.cuda.synchronize()
        replica_barrier(world)
    elapsed = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world)
    forwards = sum(s["forwards"] for s in stats)
    iters = sum(s["steps"] for s in stats)
    blocks = sum(s["blocks"] for s in stats)
    tokens = sum(s["tokens"] for s in stats)
    value = job_throughput(tokens, world, elapsed)
    tpf = tokens / forwards
    ms_per_forward = elapsed * 1e3 / forwards
    # per layer: q/k/v, attention, O, residual+norm, gate/up, down, residual+norm; then
    # embedding, LM head, merge
    launches_per_forward = 7 * shape.n_layers + 3
    # per iteration: decide, select, commit, finalize; per block-start graph: decide
    gpu_launches = forwards * launches_per_forward + iters * 4 + (forwards - iters)

    # Per-kernel timing of the projection GEMMs in the step's launch configuration.
    T = (dshape.k + 1) * B
    kern = {}
    for kind, name in enumerate(["qkv", "o_proj", "gate_up_swiglu", "down", "lm_head"]):
        iters_k = 2 * shape.n_layers if kind < 4 else 8
        ms = dec.time_gemm(kind, iters_k)
        by, fl = gemm_bytes(shape, T, kind, wb), gemm_flops(shape, T, kind)
        kern[name] = {"ms": ms, "GB/s": by / ms / 1e6, "TFLOP/s": fl / ms / 1e9}
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak_bw, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        peak_bw, peak_src = 6800.0, "fallback"
    dom = kern["gate_up_swiglu"]
    roofline = {"kernel": "gemm_kernel<SWIGLU> (gate/up + SwiGLU)", "bound": "hbm",
                "achieved": dom["GB/s"], "peak": peak_bw, "unit": "GB/s",
                "frac": dom["GB/s"] / peak_bw,
                "traffic": SWIGLU_TRAFFIC_BYTES if wb == 2 else None,
                "traffic_source": "ncu on the one-layer 7B slice at the step shape: "
                                  "dram__bytes_read.sum + dram__bytes_write.sum per launch",
                "peak_source": peak_src}

    # Verification-step latency: the forward-only graph of the 8-branch verification (and
    # of the block-start forward), median of 50 back-to-back launches, at a mid-decode
    # prefix; against the step's algorithmic bytes (every weight once, the prefix K/V
    # once, the block K/V written once) and flops.
    Pv = P0 + (gen // 2 // B) * B
    dec.rewind(Pv)
    v_med, v_mean = dec.time_forward(1, 50)
    s_med, _ = dec.time_forward(0, 50)
    vb, vf = verify_bytes_flops(shape, T, Pv, B, wb)
    peak_tc = float(peaks.get("bf16_tflops_sustained", 1700.0)) if peaks else 1700.0
    t_hbm, t_tc = vb / peak_bw / 1e6, vf / peak_tc / 1e9
    verify = {"ms_median": v_med, "ms_mean": v_mean, "prefix": Pv, "rows": T,
              "bytes": vb, "flops": vf, "hbm_roofline_ms": t_hbm, "tensor_roofline_ms": t_tc,
              "frac_hbm_roofline": t_hbm / v_med, "frac_roofline": max(t_hbm, t_tc) / v_med,
              "block_start_forward_ms_median": s_med,
              "peaks": {"hbm_gbs": peak_bw, "bf16_tflops_sustained": peak_tc, "source": peak_src}}

    # Prompt forward (the step before the decode): CUDA-event time of lopa_prefill
    # (synchronous, so the events bracket it), median of 3, against the tensor roofline.
    pre_ms = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(dec.stream)
        dec.prefill(prompt)
        e1.record(dec.stream)
        torch.cuda.synchronize()
        pre_ms.append(e0.elapsed_time(e1))
    pf = prefill_flops(shape, P0)
    prefill = {"ms_median": statistics.median(pre_ms), "tokens": P0, "flops": pf,
               "tensor_roofline_ms": pf / peak_tc / 1e9,
               "frac_tensor_roofline": pf / peak_tc / 1e9 / statistics.median(pre_ms)}

    # End to end through the public API with host buffers: prompt H2D, tokens D2H.
    import torch as _t
    pin_prompt = _t.from_numpy(prompt.astype(np.int32)).pin_memory()
    e2e_times = []
    replica_barrier(world)
    for _ in range(max(1, args.e2e_steps)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dec.prefill(pin_prompt.numpy())
        toks_e, st_e = dec.decode(gen)
        e2e_times.append(time.perf_counter() - t0)
    from diffusion_lookahead_decoding_gb300 import _lib as L
    d2h = gen * 4 + int(st_e["steps"]) * C.sizeof(L.StepResult)
    e2e_s = max_over_ranks(statistics.mean(e2e_times), world)
    e2e = {"value": job_throughput(gen, world, e2e_s), "unit": UNIT,
           "h2d_bytes_per_step": P0 * 4, "d2h_bytes_per_step": d2h,
           "includes": "prefill of the prompt + full decode per step"}

    cpu = None
    if rank == 0 and weights is not None:
        spf, times = oracle_seconds_per_forward(shape, dshape, weights, 20.0)
        cpu = {"value": tpf / spf, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": (f"oracle {dshape.k + 1}x{B}-token verification forward timed at 1 "
                          f"layer ({times[1]:.1f} s) and 2 layers ({times[2]:.1f} s) incl. LM "
                          f"head, extrapolated to {shape.n_layers} layers = {spf:.1f} s/forward; "
                          f"tokens/s at the measured TPF {tpf:.2f}")}
    dec.close()
    e4m3 = None
    if args.weight_format == "bf16" and rank == 0:
        e4m3 = e4m3_summary(api, shape, dshape, dev_w, prompt, peak_bw, peak_tc, max(1, args.steps // 2))
    odec = oracle_decodes() if (rank == 0 and not args.no_cpu_baseline) else None
    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": bench_config(args, shape, dshape, world),
            "tpf": tpf, "tpf_unmerged": tokens / (iters + blocks),
            "ms_per_forward": ms_per_forward,
            "lopa_iterations": iters, "blocks": blocks, "forwards": forwards,
            "verify_step": verify, "prefill": prefill,
            "kernels": kern, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "oracle_decodes": odec, "e4m3_weights": e4m3,
            "gpu_launches": gpu_launches, "clocks": clocks.summary(),
            "weight_gen_s": t_gen,
        }
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
