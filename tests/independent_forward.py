"""A second, independent forward used to pin the oracle (torch CPU, float64).

It shares nothing with the oracle: whole-sequence computation with library primitives
(F.rms_norm, F.linear, F.scaled_dot_product_attention with a boolean visibility mask,
complex-number RoPE) instead of the oracle's per-branch, per-head loops.  Branch
isolation ('SJTU x Huawei Xiaoyi release LoPA', section 'Core design of LoPA': all
branches verified in one forward with isolated attention) is expressed here as a
block-diagonal attention mask rather than as separate loops.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def rope_complex(x, pos, base):
    """x: [S, heads, dh]; treats (x_j, x_{j+dh/2}) as the complex number
    x_j + i x_{j+dh/2} and multiplies it by exp(i * pos * theta_j)."""
    dh = x.shape[-1]
    half = dh // 2
    inv_freq = 1.0 / (base ** (torch.arange(0, dh, 2, dtype=torch.float64) / dh))
    ang = torch.outer(pos.to(torch.float64), inv_freq)  # [S, half]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    c = torch.complex(x[..., :half], x[..., half:]) * rot
    return torch.cat([c.real, c.imag], dim=-1)


def torch_forward(weights, shape, tokens, positions, visible, act=None):
    """tokens, positions: [S]; visible: [S, S] bool, True where query i may attend key j.
    act='bf16' rounds the stored tensors through torch's bfloat16 conversion.
    Returns (logits [S, V] with [MASK] at -inf, x_final [S, d], per-layer K, V)."""
    W = lambda n: weights[n].to(torch.float64)
    r = (lambda t: t.to(torch.bfloat16).to(torch.float64)) if act == "bf16" else (lambda t: t)
    tokens = torch.as_tensor(np.asarray(tokens), dtype=torch.long)
    positions = torch.as_tensor(np.asarray(positions), dtype=torch.long)
    mask = torch.as_tensor(np.asarray(visible), dtype=torch.bool)
    S = tokens.shape[0]
    H, Hk, dh, d = shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.d_model
    x = F.embedding(tokens, W("embed"))
    ks, vs = [], []
    for l in range(shape.n_layers):
        n = r(F.rms_norm(x, (d,), weight=W(f"attn_norm.{l}"), eps=shape.rms_eps))
        q = F.linear(n, W(f"wq.{l}")).view(S, H, dh)
        k = F.linear(n, W(f"wk.{l}")).view(S, Hk, dh)
        v = r(F.linear(n, W(f"wv.{l}")).view(S, Hk, dh))
        q = r(rope_complex(q, positions, shape.rope_base))
        k = r(rope_complex(k, positions, shape.rope_base))
        ks.append(k)
        vs.append(v)
        kk = k.repeat_interleave(H // Hk, dim=1)
        vv = v.repeat_interleave(H // Hk, dim=1)
        o = F.scaled_dot_product_attention(q.transpose(0, 1), kk.transpose(0, 1),
                                           vv.transpose(0, 1), attn_mask=mask)
        o = r(o.transpose(0, 1).reshape(S, H * dh))
        x = x + F.linear(o, W(f"wo.{l}"))
        n2 = r(F.rms_norm(x, (d,), weight=W(f"mlp_norm.{l}"), eps=shape.rms_eps))
        hm = r(F.silu(F.linear(n2, W(f"wg.{l}"))) * F.linear(n2, W(f"wu.{l}")))
        x = x + F.linear(hm, W(f"wd.{l}"))
    hf = r(F.rms_norm(x, (d,), weight=W("final_norm"), eps=shape.rms_eps))
    z = shape.logit_scale * F.linear(hf, W("lm_head"))
    z[:, shape.mask_id] = -torch.inf
    return z, x, ks, vs


def block_layout(prompt_len, committed_blocks, block, n_branches):
    """Sequence layout [prompt | committed block 1..m | branch 0 .. branch nb-1] with
    its positions and visibility: the prompt is one bidirectional block, every later
    block sees all earlier blocks and itself (causal by block, bidirectional within),
    and each branch sees the prompt, the committed blocks and itself only."""
    P = prompt_len + committed_blocks * block
    groups = [0] * prompt_len
    for j in range(committed_blocks):
        groups += [j + 1] * block
    n_committed_groups = committed_blocks + 1
    for b in range(n_branches):
        groups += [n_committed_groups + b] * block
    groups = np.array(groups)
    positions = np.concatenate([np.arange(P)] + [np.arange(P, P + block)] * n_branches)
    gq = groups[:, None]
    gk = groups[None, :]
    committed_key = gk < n_committed_groups
    committed_query = gq < n_committed_groups
    visible = np.where(committed_query, committed_key & (gk <= gq),
                       committed_key | (gk == gq))
    return positions, visible
