"""Seeded synthetic inputs: model shapes, random-init weights and prompts.

This module is the one piece shared by the CUDA path's callers (tests, bench) and the
CPU oracle's callers.  It holds no arithmetic of the decoding method: it only draws
random numbers and names shapes.

Shapes follow the workloads of the LoPA announcement ("LoPA: 7B diffusion LM, single
sample 1000+ tokens/s", section on results): D2F-Dream is a Qwen2.5-7B-architecture
diffusion LM decoded in 32-token blocks.  No trained weights exist here, so every weight
is drawn N(0, 0.02) and every prompt id uniformly from [1, vocab) (id 0 is [MASK]).

Generation recipe (fixed, documented so both sides see identical values):
  * each tensor gets its own ``torch.Generator('cpu')`` seeded with
    ``seed * 1_000_003 + index`` where ``index`` is the tensor's position in
    ``weight_names(shape)``; values are ``randn * 0.02`` in fp32 and then rounded to
    bf16 (round-to-nearest-even, torch's conversion);
  * norm gains are ones (stored bf16);
  * prompt ids come from ``torch.Generator('cpu').manual_seed(prompt_seed)`` via
    ``randint(1, vocab)``.
Per-tensor generators let the 7B-shaped draw run on a thread pool.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np
import torch

MASK_ID = 0


@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_base: float
    rms_eps: float = 1e-6
    logit_scale: float = 20.0
    mask_id: int = MASK_ID

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    def streamed_params(self) -> int:
        """Parameters read once per forward (all projections and the LM head)."""
        d, hd = self.d_model, self.head_dim
        per_layer = d * self.qkv_rows + self.n_heads * hd * d + 3 * d * self.ffn
        return self.n_layers * per_layer + self.vocab * d


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    block: int
    k: int
    tau: float
    prompt_len: int
    gen_len: int

    @property
    def n_branches(self) -> int:
        return self.k + 1


# Workloads (names describe what they are; sizes as in the pages' D2F-Dream setting).
TINY = (ModelShape(2, 128, 4, 4, 32, 512, 1024, 10000.0),
        DecodeShape(block=16, k=3, tau=0.9, prompt_len=32, gen_len=64))
SMALL = (ModelShape(4, 1024, 16, 4, 64, 2816, 32768, 10000.0),
         DecodeShape(block=32, k=4, tau=0.9, prompt_len=256, gen_len=256))
DREAM7B = (ModelShape(28, 3584, 28, 4, 128, 18944, 152064, 1e6),
           DecodeShape(block=32, k=7, tau=0.9, prompt_len=512, gen_len=256))
DREAM7B_SCALING = (DREAM7B[0], DecodeShape(block=32, k=7, tau=0.9, prompt_len=2048, gen_len=512))

# Dream-7B's head geometry (head_dim 128, 7 query heads per KV head) in a 2-layer model the
# oracle decodes in seconds: the decode-level parity case of the tensor-core attention.
HEADS128 = (ModelShape(2, 896, 7, 1, 128, 2048, 8192, 1e6),
            DecodeShape(block=32, k=7, tau=0.9, prompt_len=96, gen_len=128))

# One layer with the Dream-7B layer and vocabulary sizes: a few GB on the device, used to
# profile single kernels in isolation.
DREAM7B_LAYER = (ModelShape(1, 3584, 28, 4, 128, 18944, 152064, 1e6), DREAM7B[1])

WORKLOADS = {"tiny": TINY, "small": SMALL, "heads128": HEADS128, "dream7b": DREAM7B,
             "dream7b_scaling": DREAM7B_SCALING, "dream7b_layer": DREAM7B_LAYER}

LAYER_TENSORS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def weight_names(shape: ModelShape) -> list[str]:
    names = ["embed"]
    for l in range(shape.n_layers):
        names += [f"{t}.{l}" for t in LAYER_TENSORS]
    names.append("lm_head")
    return names


def weight_shape(shape: ModelShape, name: str) -> tuple[int, int]:
    d, hd, H, Hk, F, V = (shape.d_model, shape.head_dim, shape.n_heads, shape.n_kv_heads,
                          shape.ffn, shape.vocab)
    base = name.split(".")[0]
    return {"embed": (V, d), "lm_head": (V, d), "wq": (H * hd, d), "wk": (Hk * hd, d),
            "wv": (Hk * hd, d), "wo": (d, H * hd), "wg": (F, d), "wu": (F, d),
            "wd": (d, F)}[base]


def _draw(shape: ModelShape, seed: int, idx: int, name: str) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(seed * 1_000_003 + idx)
    t = torch.randn(weight_shape(shape, name), generator=g, dtype=torch.float32)
    return t.mul_(0.02).to(torch.bfloat16)


def make_weights(shape: ModelShape, seed: int = 0, threads: int | None = None) -> dict:
    """All weights as CPU bf16 torch tensors, keyed by ``weight_names`` plus norm gains.

    Linear weights use the [out_features, in_features] layout.  Norm gains
    ``attn_norm.l``, ``mlp_norm.l`` and ``final_norm`` are ones.
    """
    names = weight_names(shape)
    threads = threads or min(16, os.cpu_count() or 1)
    out: dict[str, torch.Tensor] = {}
    if threads > 1 and len(names) > 4:
        with _cf.ThreadPoolExecutor(threads) as ex:
            futs = {n: ex.submit(_draw, shape, seed, i, n) for i, n in enumerate(names)}
            for n, f in futs.items():
                out[n] = f.result()
    else:
        for i, n in enumerate(names):
            out[n] = _draw(shape, seed, i, n)
    ones = torch.ones(shape.d_model, dtype=torch.bfloat16)
    for l in range(shape.n_layers):
        out[f"attn_norm.{l}"] = ones
        out[f"mlp_norm.{l}"] = ones
    out["final_norm"] = ones
    return out


def make_prompt(shape: ModelShape, n: int, seed: int = 1) -> np.ndarray:
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(1, shape.vocab, (n,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def make_block_state(shape: ModelShape, block: int, seed: int, masked_frac: float | None = None):
    """A mid-block decoding state: tokens with some [MASK] positions, plus per-position
    (argmax, max-probability) summaries.  Used by the decision-logic and step tests."""
    rng = np.random.default_rng(seed)
    frac = rng.uniform(0.25, 1.0) if masked_frac is None else masked_frac
    tok = rng.integers(1, shape.vocab, size=block).astype(np.int32)
    masked = rng.random(block) < frac
    if not masked.any():
        masked[rng.integers(block)] = True
    tok[masked] = shape.mask_id
    am = rng.integers(1, shape.vocab, size=block).astype(np.int32)
    mp = rng.uniform(0.3, 1.0, size=block).astype(np.float32)
    return tok, am, mp


def make_attention_inputs(nb: int, block: int, prefix: int, n_heads: int, n_kv_heads: int,
                          head_dim: int, seed: int = 2):
    """Random q [nb*block, H, dh], prefix K/V [prefix, Hk, dh] and per-branch block K/V
    [nb, block, Hk, dh], all N(0,1) rounded to bf16 (as torch CPU tensors)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    bf = torch.bfloat16
    q = torch.randn(nb * block, n_heads, head_dim, generator=g).to(bf)
    kp = torch.randn(max(prefix, 0), n_kv_heads, head_dim, generator=g).to(bf)
    vp = torch.randn(max(prefix, 0), n_kv_heads, head_dim, generator=g).to(bf)
    kb = torch.randn(nb, block, n_kv_heads, head_dim, generator=g).to(bf)
    vb = torch.randn(nb, block, n_kv_heads, head_dim, generator=g).to(bf)
    return q, kp, vp, kb, vb


def make_hidden(rows: int, d: int, seed: int = 2) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(rows, d, generator=g).to(torch.bfloat16)
