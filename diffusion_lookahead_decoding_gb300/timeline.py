"""Per-CTA device timeline of a verification forward (profiling tool).

Builds a variant of the library with -DLOPA_TIMELINE (every kernel records, per CTA, the
%globaltimer at entry, when its dependent work can start and at exit; see
csrc/timeline.cuh) into its own directory, runs the captured verification-forward graph of
a workload with recording on, and prints the per-layer critical path: for each kernel of a
layer, how far its last CTA ends after the previous kernel's last CTA, and for one layer
the distribution of start / ready / end times.  Kernels overlap under programmatic
dependent launch; a profiler that serialises them cannot show this.

    python -m diffusion_lookahead_decoding_gb300.timeline [--workload dream7b] [--prefix 640]
    python -m diffusion_lookahead_decoding_gb300.timeline --prefill   # the prompt forward
    python -m diffusion_lookahead_decoding_gb300.timeline --decode    # idle gaps of a decode
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import ctypes as C
import os
import subprocess

import numpy as np

from . import build as B

OUT = os.path.join(B.HERE, "_build_timeline")
LIB = os.path.join(OUT, "liblopa_timeline.so")
TAGS = {10: "redadd", 11: "swiglu", 12: "lmstats", 13: "qkv", 20: "attn", 21: "attn_mma",
        30: "resnorm", 31: "embed", 32: "merge", 40: "decide", 41: "select", 42: "commit",
        43: "finalize"}
SLOTS = ["qkv", "attn", "o", "rn1", "gu", "dn", "rn2"]


def build_timeline_lib() -> str:
    os.makedirs(OUT, exist_ok=True)
    cc = B.nvcc()

    def one(src):
        obj = os.path.join(OUT, src.replace(".cu", ".o"))
        r = subprocess.run([cc, *B.ARCH, *B.FLAGS, "-DLOPA_TIMELINE", "-c",
                            os.path.join(B.CSRC, src), "-o", obj], capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError(r.stderr[-4000:])
        return obj

    with cf.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(one, B.SOURCES))
    r = subprocess.run([cc, *B.ARCH, "-shared", "-o", LIB, *objs], capture_output=True, text=True)
    if r.returncode:
        raise RuntimeError(r.stderr)
    return LIB


def _records(buf):
    n = int(buf[0].item())
    raw = buf[4:4 + n * 10].cpu().numpy().view(np.uint32).reshape(n, 10)
    t = raw[:, 4:].view(np.uint64).reshape(n, 3).astype(np.int64)
    ready = np.where((t[:, 1] >= t[:, 0]) & (t[:, 1] <= t[:, 2]), t[:, 1], 0)
    return np.stack([raw[:, 0].astype(np.int64), t[:, 0], ready, t[:, 2],
                     raw[:, 1].astype(np.int64), raw[:, 2].astype(np.int64)], axis=1)


def record_prefill(workload: str):
    """Runs the prompt forward (lopa_prefill; one warm-up call) with recording on; returns
    the records, the shape and the CUDA-event time of the recorded call in ms."""
    import torch
    from . import _lib as L, api, synth
    lib = L.load(build_timeline_lib())
    lib.lopa_timeline_set_buffer.argtypes = [C.c_void_p]
    lib.lopa_timeline_set_buffer.restype = C.c_int
    shape, dshape = synth.WORKLOADS[workload]
    dw = api.upload_weights(shape, synth.make_weights(shape, 0))
    P0, Bk = dshape.prompt_len, dshape.block
    dec = api.LopaDecoder(shape, dw, Bk, dshape.k, dshape.tau, P0, P0 + dshape.gen_len)
    prompt = synth.make_prompt(shape, P0, seed=1)
    dec.prefill(prompt)
    buf = torch.zeros(4 + 400000 * 10, dtype=torch.int32, device="cuda")
    buf[1] = 400000
    torch.cuda.synchronize()
    if lib.lopa_timeline_set_buffer(C.c_void_p(buf.data_ptr())) != 0:
        raise RuntimeError("timeline buffer")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(dec.stream)
    dec.prefill(prompt)
    e1.record(dec.stream)
    torch.cuda.synchronize()
    lib.lopa_timeline_set_buffer(None)
    recs = _records(buf)
    dec.close()
    return recs, shape, e0.elapsed_time(e1)


def record_decode(workload: str):
    """Records one whole decode (after a warm-up decode); returns the records, the shape and
    the CUDA-event time of the decode in ms."""
    import torch
    from . import _lib as L, api, synth
    lib = L.load(build_timeline_lib())
    lib.lopa_timeline_set_buffer.argtypes = [C.c_void_p]
    lib.lopa_timeline_set_buffer.restype = C.c_int
    shape, dshape = synth.WORKLOADS[workload]
    dw = api.upload_weights(shape, synth.make_weights(shape, 0))
    P0, Bk = dshape.prompt_len, dshape.block
    dec = api.LopaDecoder(shape, dw, Bk, dshape.k, dshape.tau, P0, P0 + dshape.gen_len)
    dec.prefill(synth.make_prompt(shape, P0, seed=1))
    dec.decode(dshape.gen_len)
    dec.rewind(P0)
    cap = 2000000
    buf = torch.zeros(4 + cap * 10, dtype=torch.int32, device="cuda")
    buf[1] = cap
    torch.cuda.synchronize()
    if lib.lopa_timeline_set_buffer(C.c_void_p(buf.data_ptr())) != 0:
        raise RuntimeError("timeline buffer")
    _, st = dec.decode(dshape.gen_len)
    torch.cuda.synchronize()
    lib.lopa_timeline_set_buffer(None)
    recs = _records(buf)
    dec.close()
    return recs, shape, st["seconds"] * 1e3


def gaps(recs, min_ns: int = 2000):
    """Intervals in which no CTA of any kernel was resident: (total busy span, idle time in
    gaps of at least min_ns, the number of such gaps)."""
    iv = recs[np.argsort(recs[:, 1])][:, [1, 3]]
    idle, n, end = 0, 0, iv[0, 1]
    for t0, t1 in iv[1:]:
        if t0 > end:
            g = t0 - end
            if g >= min_ns:
                idle += g
                n += 1
        end = max(end, t1)
    return int(iv[:, 1].max() - iv[0, 0]), int(idle), n


def record(workload: str, prefix: int, forwards: int = 2):
    """Runs the verification-forward graph (one warm-up + `forwards` launches) with
    recording on; returns records (tag, t0, t_ready, t1, cta, sm) as an int64 array."""
    import torch
    from . import _lib as L, api, synth
    lib = L.load(build_timeline_lib())
    lib.lopa_timeline_set_buffer.argtypes = [C.c_void_p]
    lib.lopa_timeline_set_buffer.restype = C.c_int
    shape, dshape = synth.WORKLOADS[workload]
    dw = api.upload_weights(shape, synth.make_weights(shape, 0))
    P0, Bk = dshape.prompt_len, dshape.block
    dec = api.LopaDecoder(shape, dw, Bk, dshape.k, dshape.tau, P0, P0 + dshape.gen_len)
    dec.prefill(synth.make_prompt(shape, P0, seed=1))
    dec.decode(dshape.gen_len)
    dec.rewind(P0 + max(0, prefix - P0) // Bk * Bk)
    med, _ = dec.time_forward(1, 20)
    cap = 400000
    buf = torch.zeros(4 + cap * 10, dtype=torch.int32, device="cuda")
    buf[1] = cap
    torch.cuda.synchronize()
    if lib.lopa_timeline_set_buffer(C.c_void_p(buf.data_ptr())) != 0:
        raise RuntimeError("timeline buffer")
    dec.time_forward(1, forwards)
    torch.cuda.synchronize()
    lib.lopa_timeline_set_buffer(None)
    recs = _records(buf)
    dec.close()
    return recs, shape, med


def launches(recs):
    """Groups the records of each kernel into launches (time-disjoint groups of CTAs),
    ordered by their first start."""
    out = []
    for tg in np.unique(recs[:, 0]):
        r = recs[recs[:, 0] == tg]
        r = r[np.argsort(r[:, 1])]
        start, mx = 0, -1
        for i in range(len(r)):
            if i > start and r[i, 1] > mx + 1000:
                out.append((int(r[start:i, 1].min()), int(tg), r[start:i]))
                start, mx = i, -1
            mx = max(mx, int(r[i, 3]))
        out.append((int(r[start:, 1].min()), int(tg), r[start:]))
    out.sort(key=lambda x: x[0])
    return out


def report(recs, n_layers: int, layer: int = 10) -> str:
    ls = launches(recs)
    names = [TAGS.get(tg, str(tg)) for _, tg, _ in ls]
    starts = [i for i, nm in enumerate(names) if nm == "embed"]
    fw = ls[starts[-1]:]
    lines = [f"forward: {len(fw)} launches, {(max(c[:, 3].max() for _, _, c in fw) - fw[0][0]) / 1e3:.1f} us"]
    body = fw[1:1 + 7 * n_layers]
    inc = {s: [] for s in SLOTS}
    prev = fw[0][2][:, 3].max()
    for i, (_, _, c) in enumerate(body):
        inc[SLOTS[i % 7]].append(c[:, 3].max() - prev)
        prev = c[:, 3].max()
    lines.append("critical-path increment per layer (mean over layers, us):")
    for s in SLOTS:
        lines.append(f"  {s:5s} {np.mean(inc[s]) / 1e3:7.2f}")
    lines.append(f"  layer {sum(np.mean(inc[s]) for s in SLOTS) / 1e3:.2f}")
    for _, tg, c in fw[1 + 7 * n_layers:]:
        lines.append(f"  {TAGS.get(tg, tg)}: +{(c[:, 3].max() - prev) / 1e3:.2f}")
        prev = c[:, 3].max()
    base = 1 + 7 * layer
    prev = fw[base - 1][2][:, 3].max()
    lines.append(f"layer {layer}, relative to the previous kernel's last CTA end (us):")
    lines.append("  kernel ctas   start min/med/max     ready min/med/max       end min/med/max")
    for j in range(7):
        _, tg, c = fw[base + j]
        q = lambda v: np.percentile(v, [0, 50, 100]) / 1e3
        st, en = q(c[:, 1] - prev), q(c[:, 3] - prev)
        rd = q(c[c[:, 2] > 0, 2] - prev) if (c[:, 2] > 0).any() else np.zeros(3)
        lines.append(f"  {SLOTS[j]:5s} {len(c):4d}  {st[0]:6.1f} {st[1]:6.1f} {st[2]:6.1f}   "
                     f"{rd[0]:6.1f} {rd[1]:6.1f} {rd[2]:6.1f}   {en[0]:6.1f} {en[1]:6.1f} {en[2]:6.1f}")
        prev = c[:, 3].max()
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="dream7b")
    ap.add_argument("--prefix", type=int, default=640)
    ap.add_argument("--layer", type=int, default=10)
    ap.add_argument("--prefill", action="store_true", help="record the prompt forward instead")
    ap.add_argument("--decode", action="store_true", help="record a whole decode: idle gaps")
    args = ap.parse_args()
    if args.decode:
        recs, shape, ms = record_decode(args.workload)
        span, idle, n = gaps(recs)
        print(f"decode: {ms:.3f} ms (CUDA events), {len(recs)} CTA records, GPU span "
              f"{span / 1e6:.3f} ms, idle {idle / 1e6:.3f} ms in {n} gaps of >= 2 us "
              f"({100.0 * idle / span:.1f} % of the span)")
        return
    if args.prefill:
        recs, shape, ms = record_prefill(args.workload)
        print(f"prompt forward (recorded call, CUDA events around lopa_prefill): {ms:.3f} ms; "
              f"{len(recs)} CTA records")
        print(report(recs, shape.n_layers, min(args.layer, shape.n_layers - 1)))
        return
    recs, shape, med = record(args.workload, args.prefix)
    print(f"verification forward (no recording): {med:.3f} ms median; {len(recs)} CTA records")
    print(report(recs, shape.n_layers, min(args.layer, shape.n_layers - 1)))


if __name__ == "__main__":
    main()
