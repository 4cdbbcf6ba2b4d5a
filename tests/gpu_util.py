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


def make_decoder(name: str, k: int | None = None, max_seq: int | None = None):
    from diffusion_lookahead_decoding_gb300 import api
    build_lib()
    shape, dshape, _ = workload_weights(name)
    dw = device_weights(name)
    k = dshape.k if k is None else k
    max_seq = max_seq or dshape.prompt_len + dshape.gen_len
    return api.LopaDecoder(shape, dw, dshape.block, k, dshape.tau, dshape.prompt_len, max_seq)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def f32(x):
    """Values as float32 (the precision in which the kernels hold and compare them)."""
    return np.asarray(x, dtype=np.float32).astype(np.float64)


class Conditioning:
    """How much the oracle itself moves when only its accumulation precision changes
    (float64 -> float32 sums, same bf16 storage).  A correct implementation with a
    different summation order cannot be expected to agree more closely than this, so
    the tolerances below never go under it (times 2)."""

    def __init__(self, ref, alt):
        self.mp = float(np.abs(alt.mp - ref.mp).max())
        self.hidden = rel_l2(alt.x_final, ref.x_final)

    @property
    def mp_bound(self):
        return max(MP_ABS, 2.0 * self.mp)

    @property
    def hidden_bound(self):
        return max(HIDDEN_REL_L2, 2.0 * self.hidden)

    @property
    def tie(self):
        return max(NEAR_TIE, 2.0 * self.mp)

    def __repr__(self):
        return f"oracle sensitivity: maxp {self.mp:.2e}, hidden {self.hidden:.2e}"


def oracle_forward_pair(shape, w, prompt, branches, capacity, cache_weights=None):
    """Oracle forward of `branches` after prefilling `prompt`, with float64 and with
    float32 accumulation.  Returns (model, cache, out, conditioning) of the float64 run."""
    P = len(prompt)
    m = O.OracleModel(shape, w, act="bf16", cache_weights=cache_weights)
    cache = O.prefill(m, prompt, capacity)
    out = O.forward(m, cache, P, branches)
    m32 = O.OracleModel(shape, w, act="bf16", cache_weights=cache_weights, accum="fp32")
    c32 = O.prefill(m32, prompt, capacity)
    alt = O.forward(m32, c32, P, branches)
    return m, cache, out, Conditioning(out, alt)


def tokens_ok(gpu_am, out, tie):
    """Greedy tokens must match except where the oracle's top-2 probabilities differ by
    less than `tie`.  Returns (ok, number of disallowed mismatches)."""
    bad = (np.asarray(gpu_am) != np.asarray(out.am)) & ((out.mp - out.p2) >= tie)
    return not bad.any(), int(bad.sum())


def seeded_branches(shape, nb, B, seed, masked=0.6):
    rng = np.random.default_rng(seed)
    br = rng.integers(1, shape.vocab, (nb, B))
    br[rng.random((nb, B)) < masked] = shape.mask_id
    br[:, 0] = shape.mask_id
    return br.astype(np.int32)
