"""Shared helpers for the GPU parity tests (the CUDA path vs the CPU oracle).

Every oracle input comes from the seeded generators in ``synth``; nothing read back
from the GPU is ever fed to the oracle.
"""
from __future__ import annotations

import functools

import numpy as np

from diffusion_lookahead_decoding_gb300 import synth
from oracle import lopa_oracle as O

# Bounds stated for the path: maxp within 2e-2 absolute, final hidden state within 3e-2
# relative L2, integer decisions exact except where the oracle's competing confidences
# differ by less than 1e-3.
NEAR_TIE = 1e-3
MP_ABS = 2e-2
HIDDEN_REL_L2 = 3e-2


def build_lib():
    from diffusion_lookahead_decoding_gb300 import build
    build.build()


@functools.lru_cache(maxsize=4)
def workload_weights(name: str, seed: int = 0):
    shape, dshape = synth.WORKLOADS[name]
    return shape, dshape, synth.make_weights(shape, seed)


@functools.lru_cache(maxsize=2)
def device_weights(name: str, seed: int = 0):
    from diffusion_lookahead_decoding_gb300 import api
    shape, _, w = workload_weights(name, seed)
    return api.upload_weights(shape, w)


def make_decoder(name: str, k: int | None = None, max_seq: int | None = None,
                 weight_format: str = "bf16"):
    from diffusion_lookahead_decoding_gb300 import api
    build_lib()
    shape, dshape, _ = workload_weights(name)
    dw = device_weights(name)
    k = dshape.k if k is None else k
    max_seq = max_seq or dshape.prompt_len + dshape.gen_len
    return api.LopaDecoder(shape, dw, dshape.block, k, dshape.tau, dshape.prompt_len, max_seq,
                           weight_format=weight_format)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def f32(x):
    """Values as float32 (the precision in which the kernels hold and compare them)."""
    return np.asarray(x, dtype=np.float32).astype(np.float64)


class Conditioning:
    """How much the oracle itself moves when only its accumulation precision changes
    (float64 -> float32 sums, same bf16 storage): a report printed beside the GPU-oracle
    differences, never a tolerance.  It shows how far from the oracle any correct
    implementation with another summation order lands on these random-weight models."""

    def __init__(self, ref, alt):
        self.mp = float(np.abs(alt.mp - ref.mp).max())
        self.mp_pos = np.abs(alt.mp - ref.mp)
        self.hidden = rel_l2(alt.x_final, ref.x_final)

    def __repr__(self):
        return f"oracle float32-vs-float64 movement: maxp {self.mp:.2e}, hidden {self.hidden:.2e}"


def oracle_forward_pair(shape, w, prompt, branches, capacity, cache_weights=None,
                        weight_format="bf16"):
    """Oracle forward of `branches` after prefilling `prompt`, with float64 and with
    float32 accumulation.  Returns (model, cache, out, conditioning) of the float64 run
    (its logits included)."""
    P = len(prompt)
    m = O.OracleModel(shape, w, act="bf16", cache_weights=cache_weights,
                      weight_format=weight_format)
    cache = O.prefill(m, prompt, capacity)
    out = O.forward(m, cache, P, branches, want_logits=True)
    m32 = O.OracleModel(shape, w, act="bf16", cache_weights=cache_weights, accum="fp32",
                        weight_format=weight_format)
    c32 = O.prefill(m32, prompt, capacity)
    alt = O.forward(m32, c32, P, branches)
    return m, cache, out, Conditioning(out, alt)


def softmax_rows(z):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def token_flips(gpu_am, gpu_mp, out, mask_id=0, gpu_hidden=None, shape=None, weights=None,
                weight_format="bf16"):
    """Greedy-token differences between the GPU and the oracle: (all, beyond the window).

    At a position where the GPU picks token a and the oracle token b, the oracle's
    probabilities (its full logits, [MASK] excluded) give the gap p(b) - p(a) between
    exactly those two tokens; the GPU's max-probability is its probability of a, so
    e_a = |mp_gpu - p_oracle(a)| is measured.  With the GPU's final hidden state (and the
    model's final-norm gain and LM head), the GPU's logits of a and b are recomputed from
    it, which measures e_b as well: the flip is allowed where the gap is below
    max(1e-3, e_a + e_b) - by the triangle inequality that holds whenever the GPU's own
    logits rank a over b, so a position beyond it means the fused LM head's argmax
    disagrees with its own input.  Without the hidden state the error on b is taken equal
    to the one measured on a (window 2 e_a): a report, not a bound.  With E4M3 weights the
    two LM-head rows are their quantised values (the quantisation is per row)."""
    am = np.asarray(gpu_am).reshape(-1)
    mp = np.asarray(gpu_mp, np.float64).reshape(-1)
    oam = np.asarray(out.am).reshape(-1)
    z = np.array(out.logits, np.float64).reshape(len(oam), -1)
    z[:, mask_id] = -np.inf
    hid = None if gpu_hidden is None else np.asarray(gpu_hidden, np.float64).reshape(len(oam), -1)
    flips = np.nonzero(am != oam)[0]
    bad = 0
    for i in flips:
        p = softmax_rows(z[i])
        a, b = int(am[i]), int(oam[i])
        gap = p[b] - p[a]
        e_a = abs(mp[i] - p[a])
        window = 2.0 * e_a
        if hid is not None:
            import torch
            x = hid[i]
            g = weights["final_norm"].to(torch.float64).numpy()
            n = x / np.sqrt(np.mean(x * x) + shape.rms_eps) * g
            n = torch.from_numpy(n).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
            W = weights["lm_head"][[a, b]].to(torch.float64).numpy()
            if weight_format == "e4m3":
                codes, s = O.quantize_e4m3_rows(W)
                W = codes * s[:, None]
            zg = shape.logit_scale * (W @ n)
            p_b_gpu = mp[i] * np.exp(zg[1] - zg[0])
            window = e_a + abs(p_b_gpu - p[b])
        if gap >= max(NEAR_TIE, window):
            bad += 1
    return int(len(flips)), bad


def seeded_branches(shape, nb, B, seed, masked=0.6):
    rng = np.random.default_rng(seed)
    br = rng.integers(1, shape.vocab, (nb, B))
    br[rng.random((nb, B)) < masked] = shape.mask_id
    br[:, 0] = shape.mask_id
    return br.astype(np.int32)
