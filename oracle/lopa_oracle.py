"""CPU oracle for the LoPA branch-verification step.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import or call this module.  The product (the CUDA library and its binding) never
does, and this module never imports the product.  It is plain, slow, and written to be
checked against the pages by eye: numpy float64 throughout, one loop per branch and
per head, no blocking, fusion or reordering.

Sources (titles of the pages; all describe arXiv 2512.16229, "LoPA: Lookahead
Parallel Decoding"):
  [ANN]  "SJTU x Huawei Xiaoyi release LoPA: 7B diffusion LM, 1000+ tokens/s single
          sample" (developer-community re-post of the official announcement).
          Sections: "Problem: the filling order limits parallelism" (confidence-driven
          sampling fills the most confident positions greedily), "Core design of LoPA"
          (anchor branch + k lookahead branches from the k most confident positions;
          branch confidence = mean predicted confidence of the still-unfilled
          positions; all branches verified in one forward with attention isolated per
          branch; the winner's logits are reused for the next fill), "LoPA-Dist"
          (static KV cache, Pre-Write then Commit-Winner-Cache).
  [BLOG] "Decoding-efficiency revolution: how LoPA breaks the parallel bottleneck of
          dLLMs", section 3.3 (attention isolation: a branch sees the prompt and its
          own tokens only; all branch forwards share one matmul).

What the pages leave open is fixed by the workload definitions (blocks decoded
causally by block and bidirectionally inside a block; threshold tau with at least one
fill per step; each lookahead branch = anchor fills + one more of the top-k masked
positions filled with its argmax; greedy argmax with ties to the lowest index) and by
these readings: [MASK] is never a prediction; a threshold is met at mp >= tau; an
empty confidence mean is 1.0; weights are bf16 and activations are bf16 at every
tensor the path stores, arithmetic otherwise float64 here.

Pins (tests/test_oracle_*.py): bf16 rounding vs torch and hand cases; RMSNorm,
RoPE and softmax closed forms; attention vs brute-force loops; the whole forward vs an
independent torch-fp64 implementation that isolates branches by an attention mask;
decision rules vs hand-worked cases and brute force; k=0 vs a separately written
threshold decoder; logit reuse; KV-cache consistency vs a full-sequence block-causal
pass; exhaustive one-extra-position replay on tiny blocks.  Every function here is
pinned by at least one of them.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "bf16_round", "e4m3_round", "quantize_e4m3_rows", "QUANTIZED_WEIGHTS", "rmsnorm", "rope", "silu", "linear", "isolated_attention", "logit_summary", "OracleModel", "prefill",
    "forward", "anchor_fill", "lookahead_candidates", "build_branches",
    "branch_confidence", "select_winner", "decision_margins", "lopa_step", "decode",
    "StepRecord",
]

# ----------------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------------
_BF16_MAX = float.fromhex("0x1.fe00000000000p+127")  # largest finite bf16 (0x7F7F)


def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value (ties to even), returned as
    float64.  bfloat16 = 1 sign, 8 exponent, 7 fraction bits (same exponent range as
    IEEE binary32).  Normal numbers: drop the low 45 of the 52 fraction bits of the
    binary64 encoding with round-half-even; below 2**-126 the bf16 grid is the fixed
    spacing 2**-133; results beyond the largest finite value become infinities."""
    x = np.asarray(x, dtype=np.float64)
    bits = np.ascontiguousarray(x).view(np.uint64)
    keep_lsb = (bits >> np.uint64(45)) & np.uint64(1)
    half_minus_one = np.uint64((1 << 44) - 1)
    mask = np.uint64(0xFFFFFFFFFFFFFFFF ^ ((1 << 45) - 1))
    rounded = ((bits + half_minus_one + keep_lsb) & mask).view(np.float64)
    rounded = np.where(np.abs(rounded) > _BF16_MAX, np.copysign(np.inf, x), rounded)
    sub = np.round(x / 2.0 ** -133) * 2.0 ** -133  # np.round: half to even
    out = np.where(np.abs(x) < 2.0 ** -126, sub, rounded)
    return out.reshape(x.shape)


def _identity(x):
    return np.asarray(x, dtype=np.float64)


# E4M3: the 8-bit float with 1 sign, 4 exponent (bias 7) and 3 fraction bits.  It has no
# infinities; the pattern S.1111.111 is NaN, so the largest finite magnitude is
# 2^8 * 1.75 = 448.  Exponent field 0 holds the subnormals m/8 * 2^-6.
E4M3_MAX = 448.0


def e4m3_round(x):
    """Round float64 values to the nearest E4M3 value, ties to even; magnitudes beyond
    448 saturate to 448 (a finite-saturating conversion: a quantised weight is never
    NaN).  Within the binade [2^e, 2^(e+1)), e >= -6, the E4M3 grid has spacing
    2^(e-3); below 2^-6 it is the subnormal spacing 2^-9."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                      # a = f * 2^ex, 0.5 <= f < 1: binade e = ex - 1
    e = np.maximum(ex.astype(np.int64) - 1, -6)
    spacing = np.ldexp(1.0, e - 3)
    q = np.round(a / spacing) * spacing      # exact scaling by a power of two; half to even
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, x).reshape(x.shape)


def quantize_e4m3_rows(W):
    """Per-output-channel E4M3 quantisation of a weight [out_features][in_features].

    Reading (the pages name FP16/INT8 switching for the NVIDIA system and a quantisation
    mechanism without a format): each row r gets the scale s_r = max|W_r| / 448 and the
    codes c = E4M3(W_r / s_r); the row is used as c * s_r.  The scale and the quotient
    are both formed in float32 (the precision in which the codes are decided); an
    all-zero row gets s_r = 1.  Returns (codes as float64 values, scales as float64
    holding the float32 values)."""
    W32 = np.asarray(W, dtype=np.float32)
    amax = np.max(np.abs(W32), axis=1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    codes = e4m3_round((W32 / s[:, None]).astype(np.float64))
    return codes, s.astype(np.float64)


# Weights that the E4M3 weight stream quantises (per layer and the LM head); the
# embedding table and the norm gains stay bf16.
QUANTIZED_WEIGHTS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "lm_head")


# ----------------------------------------------------------------------------------
# Transformer pieces (standard pre-norm decoder of the Qwen2.5 family that D2F-Dream
# uses; the pages name the models, the workload fixes the architecture)
# ----------------------------------------------------------------------------------
def rmsnorm(x, g, eps):
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope(x, pos, base):
    """Rotary position embedding, rotate-half convention: for j < dh/2 the pair
    (x_j, x_{j+dh/2}) is rotated by the angle pos * base**(-2j/dh).
    x: [..., n_pos, n_heads, dh]; pos: [n_pos] absolute positions."""
    dh = x.shape[-1]
    half = dh // 2
    j = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * j / dh)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]  # [n_pos, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def linear(x, W, accum="fp64"):
    """x @ W^T for a weight stored [out_features, in_features].  accum='fp32' forms the
    same sum with float32 arithmetic; it exists only to measure how strongly the result
    depends on the accumulation precision (the problem's conditioning)."""
    if accum == "fp32":
        return (np.asarray(x, dtype=np.float32) @ np.asarray(W, dtype=np.float32).T).astype(np.float64)
    return np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def isolated_attention(q, prefix_k, prefix_v, block_k, block_v):
    """Attention of every branch over the shared prefix and its own block only.

    q: [nb, B, H, dh]; prefix_k/v: [P, Hk, dh]; block_k/v: [nb, B, Hk, dh].
    Query head h reads KV head h // (H / Hk) (grouped-query attention); softmax scale
    1/sqrt(dh); no mask inside the block (bidirectional).  Each branch is a separate
    loop iteration: branch b never sees another branch's keys."""
    nb, B, H, dh = q.shape
    Hk = block_k.shape[2]
    group = H // Hk
    out = np.zeros((nb, B, H, dh))
    for b in range(nb):
        keys = np.concatenate([prefix_k, block_k[b]], axis=0)  # [P+B, Hk, dh]
        vals = np.concatenate([prefix_v, block_v[b]], axis=0)
        for h in range(H):
            g = h // group
            s = q[b, :, h, :] @ keys[:, g, :].T / math.sqrt(dh)  # [B, P+B]
            s = s - s.max(axis=-1, keepdims=True)
            a = np.exp(s)
            a /= a.sum(axis=-1, keepdims=True)
            out[b, :, h, :] = a @ vals[:, g, :]
    return out


def logit_summary(z, mask_id):
    """Per row of logits z[..., V]: the greedy token (argmax, lowest id on ties), its
    softmax probability maxp = 1 / sum(exp(z - max z)), and the second-largest
    probability (only used to report near-ties).  [MASK] is never a prediction: its
    logit is -inf before both the argmax and the softmax."""
    z = np.array(z, dtype=np.float64, copy=True)
    z[..., mask_id] = -np.inf
    am = np.argmax(z, axis=-1)  # first occurrence = lowest id
    zmax = np.take_along_axis(z, am[..., None], axis=-1)
    e = np.exp(z - zmax)
    denom = e.sum(axis=-1)
    mp = 1.0 / denom
    e_wo = e.copy()
    np.put_along_axis(e_wo, am[..., None], -1.0, axis=-1)
    p2 = e_wo.max(axis=-1) / denom
    return am.astype(np.int64), mp, p2


# ----------------------------------------------------------------------------------
# Model container
# ----------------------------------------------------------------------------------
class OracleModel:
    """Holds the shape, the weights (bf16 values, read as float64) and the activation
    format.  ``act='bf16'`` rounds every tensor that the decoding path stores (GEMM
    inputs, q/k/v and the KV cache, attention output, MLP hidden, final normed
    hidden) to bf16, as the workload's "bf16 weights/activations" states; arithmetic
    stays float64.  ``act='fp64'`` keeps everything float64.  ``weights='e4m3'`` uses
    every projection matrix and the LM head as its per-row E4M3 quantisation
    (quantize_e4m3_rows: codes times scale, exact in float64)."""

    def __init__(self, shape, weights, act="bf16", cache_weights=None, accum="fp64",
                 weight_format="bf16"):
        if weight_format not in ("bf16", "e4m3"):
            raise ValueError(weight_format)
        self.shape = shape
        self._w = weights  # name -> torch bf16 CPU tensor or numpy array
        self.act = act
        self.accum = accum
        self.weight_format = weight_format
        self.rnd = bf16_round if act == "bf16" else _identity
        if cache_weights is None:
            cache_weights = shape.streamed_params() < 400_000_000
        self._cache = {} if cache_weights else None

    def W(self, name):
        if self._cache is not None and name in self._cache:
            return self._cache[name]
        t = self._w[name]
        if hasattr(t, "numpy"):
            import torch  # plain CPU tensor conversion of the given weights
            a = t.to(torch.float64).numpy()
        else:
            a = np.asarray(t, dtype=np.float64)
        if self.weight_format == "e4m3" and name.split(".")[0] in QUANTIZED_WEIGHTS:
            codes, s = quantize_e4m3_rows(a)
            a = codes * s[:, None]
        if self._cache is not None:
            self._cache[name] = a
        return a


@dataclasses.dataclass
class KVCache:
    """Static KV cache: per layer K and V of shape [capacity, Hk, dh] (float64 holding
    the stored values), valid up to ``length``."""
    k: list
    v: list
    length: int

    @staticmethod
    def empty(shape, capacity):
        z = lambda: np.zeros((capacity, shape.n_kv_heads, shape.head_dim))
        return KVCache([z() for _ in range(shape.n_layers)],
                       [z() for _ in range(shape.n_layers)], 0)


@dataclasses.dataclass
class ForwardOut:
    am: np.ndarray       # [nb, B] greedy token per position
    mp: np.ndarray       # [nb, B] its probability
    p2: np.ndarray       # [nb, B] second-largest probability
    x_final: np.ndarray  # [nb, B, d] residual stream after the last layer
    block_k: list        # per layer [nb, B, Hk, dh]
    block_v: list


def forward(model, cache, P, branches, want_logits=False):
    """One forward of ``nb`` branches of a block that starts at absolute position P.

    Every branch sees the committed prefix cache[0:P] and its own block only
    (bidirectionally inside the block); branches never see each other ([ANN] "Core
    design": isolated attention, all branches in one forward; [BLOG] 3.3).
    branches: int array [nb, B].  Returns per-branch greedy tokens and max-probs."""
    sh = model.shape
    rnd = model.rnd
    branches = np.asarray(branches, dtype=np.int64)
    nb, B = branches.shape
    H, Hk, dh = sh.n_heads, sh.n_kv_heads, sh.head_dim
    pos = P + np.arange(B)
    x = model.W("embed")[branches]  # [nb, B, d]
    block_k, block_v = [], []
    for l in range(sh.n_layers):
        n = rnd(rmsnorm(x, model.W(f"attn_norm.{l}"), sh.rms_eps))
        lin = lambda a, name: linear(a, model.W(name), model.accum)
        q = lin(n, f"wq.{l}").reshape(nb, B, H, dh)
        k = lin(n, f"wk.{l}").reshape(nb, B, Hk, dh)
        v = lin(n, f"wv.{l}").reshape(nb, B, Hk, dh)
        q = rnd(np.stack([rope(q[b], pos, sh.rope_base) for b in range(nb)]))
        k = rnd(np.stack([rope(k[b], pos, sh.rope_base) for b in range(nb)]))
        v = rnd(v)
        block_k.append(k)
        block_v.append(v)
        attn = isolated_attention(q, cache.k[l][:P], cache.v[l][:P], k, v)
        o = rnd(attn.reshape(nb, B, H * dh))
        x = x + lin(o, f"wo.{l}")
        n2 = rnd(rmsnorm(x, model.W(f"mlp_norm.{l}"), sh.rms_eps))
        hm = rnd(silu(lin(n2, f"wg.{l}")) * lin(n2, f"wu.{l}"))
        x = x + lin(hm, f"wd.{l}")
    hf = rnd(rmsnorm(x, model.W("final_norm"), sh.rms_eps))
    z = sh.logit_scale * linear(hf, model.W("lm_head"), model.accum)
    am, mp, p2 = logit_summary(z, sh.mask_id)
    out = ForwardOut(am, mp, p2, x, block_k, block_v)
    if want_logits:
        out.logits = z
    return out


def prefill(model, prompt, capacity):
    """Run the prompt as one block (bidirectional inside itself, no prefix) and store
    its K/V as cache[0:len(prompt)]."""
    cache = KVCache.empty(model.shape, capacity)
    prompt = np.asarray(prompt, dtype=np.int64)
    out = forward(model, cache, 0, prompt[None, :])
    n = len(prompt)
    for l in range(model.shape.n_layers):
        cache.k[l][:n] = out.block_k[l][0]
        cache.v[l][:n] = out.block_v[l][0]
    cache.length = n
    return cache


# ----------------------------------------------------------------------------------
# Decision rules of one LoPA iteration ([ANN] "Core design of LoPA")
# ----------------------------------------------------------------------------------
def anchor_fill(tok, am, mp, tau, mask_id):
    """Anchor branch = the standard confidence-driven greedy policy: every masked
    position whose max-probability reaches tau is filled with its greedy token; if none
    does, the single most confident masked position is filled (ties: lowest position).
    Returns (anchor tokens, sorted list of filled positions)."""
    tok = np.asarray(tok)
    masked = [i for i in range(len(tok)) if tok[i] == mask_id]
    S = [i for i in masked if mp[i] >= tau]
    if not S and masked:
        best = masked[0]
        for i in masked[1:]:
            if mp[i] > mp[best]:
                best = i
        S = [best]
    anchor = np.array(tok, copy=True)
    for i in S:
        anchor[i] = am[i]
    return anchor, S


def lookahead_candidates(anchor, mp, k, mask_id):
    """The k most confident positions still masked after the anchor fill, most
    confident first (ties: lowest position).  Fewer if fewer remain."""
    R = [i for i in range(len(anchor)) if anchor[i] == mask_id]
    R.sort(key=lambda i: (-float(mp[i]), i))
    return R[:k]


def build_branches(anchor, am, candidates):
    """Branch 0 is the anchor; branch i is the anchor with candidate c_i additionally
    filled with its greedy token."""
    out = [np.array(anchor, copy=True)]
    for c in candidates:
        b = np.array(anchor, copy=True)
        b[c] = am[c]
        out.append(b)
    return np.stack(out)


def branch_confidence(branch, mp_branch, mask_id):
    """Mean predicted confidence (max-probability from this branch's own logits) over
    the branch's still-unfilled positions.  A branch with none left scores 1.0."""
    rem = [i for i in range(len(branch)) if branch[i] == mask_id]
    if not rem:
        return 1.0
    return float(sum(float(mp_branch[i]) for i in rem) / len(rem))


def select_winner(conf):
    """Highest branch confidence wins; ties go to the lowest branch index (so the
    anchor wins a tie)."""
    w = 0
    for b in range(1, len(conf)):
        if conf[b] > conf[w]:
            w = b
    return w


@dataclasses.dataclass
class StepRecord:
    filled: list            # positions filled by the anchor rule
    candidates: list        # lookahead positions, branch i+1 fills candidates[i]
    branches: np.ndarray    # [nb, B]
    conf: list
    winner: int
    am: np.ndarray          # winner's greedy tokens (reused for the next fill)
    mp: np.ndarray
    p2: np.ndarray
    out: ForwardOut
    margins: dict


def decision_margins(tok, mp, p2, tau, k, mask_id, conf, winner):
    """How close each decision of one iteration came to going the other way.  Only the
    quantities the iteration's outcome (the positions it fills and their tokens) depends
    on are measured; a value under a tolerance marks that decision as a near-tie.

      tau      : min over masked positions of |mp - tau| (each one's threshold test).
      fallback : when no masked position reaches tau, the gap between the two highest
                 masked mp (which single position the anchor fills); else inf.
      rank     : when more positions remain masked after the anchor fill than there are
                 lookahead branches (k >= 1), the gap between the k-th and (k+1)-th
                 highest remaining mp (which positions become candidates); else inf.
                 The order among the chosen k only permutes the branches.
      conf     : the winner's confidence minus the best other branch's; inf for one branch.
      token    : min over the positions this iteration fills (anchor fills and the
                 winner's extra position) of mp - p2, the top-2 probability gap of the
                 logits that chose their tokens; inf when p2 is not given.
    """
    masked = [i for i in range(len(tok)) if tok[i] == mask_id]
    m_tau = min((abs(float(mp[i]) - tau) for i in masked), default=math.inf)
    m_fb = math.inf
    if masked and not any(float(mp[i]) >= tau for i in masked) and len(masked) >= 2:
        top = sorted((float(mp[i]) for i in masked), reverse=True)
        m_fb = top[0] - top[1]
    anchor, S = anchor_fill(tok, np.zeros(len(tok), dtype=np.int64) + (mask_id + 1), mp, tau,
                            mask_id)
    R = sorted((float(mp[i]) for i in range(len(tok)) if anchor[i] == mask_id), reverse=True)
    m_rank = R[k - 1] - R[k] if 1 <= k < len(R) else math.inf
    others = [c for b, c in enumerate(conf) if b != winner]
    m_conf = conf[winner] - max(others) if others else math.inf
    m_tok = math.inf
    if p2 is not None:
        C = lookahead_candidates(anchor, mp, k, mask_id)
        filled = list(S) + ([C[winner - 1]] if winner >= 1 else [])
        m_tok = min(float(mp[i]) - float(p2[i]) for i in filled)
    return {"tau": m_tau, "fallback": m_fb, "rank": m_rank, "conf": m_conf, "token": m_tok}


def lopa_step(model, cache, P, tok, am, mp, k, tau, p2=None):
    """One LoPA iteration on the current block state (tok, and the (am, mp) summary of
    the logits that produced it; p2, their second-largest probabilities, only feeds the
    reported margins): anchor fill, k lookahead branches, one isolated forward over all
    branches, branch confidences, winner.  The winner's (am, mp) are returned for reuse
    by the next iteration ([ANN]: no extra forward)."""
    sh = model.shape
    anchor, S = anchor_fill(tok, am, mp, tau, sh.mask_id)
    C = lookahead_candidates(anchor, mp, k, sh.mask_id)
    branches = build_branches(anchor, am, C)
    out = forward(model, cache, P, branches)
    conf = [branch_confidence(branches[b], out.mp[b], sh.mask_id) for b in range(len(branches))]
    w = select_winner(conf)
    margins = decision_margins(tok, mp, p2, tau, k, sh.mask_id, conf, w)
    return StepRecord(S, C, branches, conf, w, out.am[w], out.mp[w], out.p2[w], out, margins)


def decode(model, prompt, block, k, tau, gen_len, record=False):
    """Semi-autoregressive block decoding with LoPA.  The prompt is prefilled as one
    block; each output block starts all-[MASK], gets one forward (its first logits),
    then LoPA iterations run until no [MASK] is left.  After each iteration the
    winner's block K/V is committed to the static cache (Pre-Write of all branches,
    Commit-Winner).  Returns generated tokens, the forward count (block-start forwards
    plus one per iteration; prefill excluded), the cache and optionally the step log."""
    sh = model.shape
    assert gen_len % block == 0
    prompt = np.asarray(prompt, dtype=np.int64)
    P = len(prompt)
    cache = prefill(model, prompt, P + gen_len)
    generated, forwards, log = [], 0, []
    for _ in range(gen_len // block):
        tok = np.full(block, sh.mask_id, dtype=np.int64)
        first = forward(model, cache, P, tok[None, :])
        forwards += 1
        am, mp, p2 = first.am[0], first.mp[0], first.p2[0]
        while (tok == sh.mask_id).any():
            st = lopa_step(model, cache, P, tok, am, mp, k, tau, p2)
            forwards += 1
            w = st.winner
            tok, am, mp, p2 = st.branches[w], st.am, st.mp, st.p2
            for l in range(sh.n_layers):
                cache.k[l][P:P + block] = st.out.block_k[l][w]
                cache.v[l][P:P + block] = st.out.block_v[l][w]
            if record:
                log.append((P, st))
        generated.extend(int(t) for t in tok)
        P += block
        cache.length = P
    return np.array(generated, dtype=np.int64), forwards, cache, log
