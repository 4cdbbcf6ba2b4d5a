"""Pins for the CPU oracle: each check compares it with something other than itself
(hand-worked values, closed forms, library routines, an independent torch forward,
brute force).  All CPU, no GPU."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import lopa_oracle as O
OL = O
from diffusion_lookahead_decoding_gb300 import synth
from tests.independent_forward import block_layout, rope_complex, torch_forward

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
# A micro model with grouped-query attention (2 query heads per KV head).
MICRO = synth.ModelShape(2, 64, 4, 2, 16, 128, 97, 10000.0)


@pytest.fixture(scope="module")
def micro_w():
    return synth.make_weights(MICRO, seed=3, threads=1)


# ----------------------------------------------------------------------------- formats
def test_bf16_round_hand_cases():
    cases = {
        1.0: 1.0,
        1 + 2 ** -8: 1.0,                 # exact midpoint, ties to even (fraction 0)
        1 + 3 * 2 ** -8: 1 + 2 ** -6,     # midpoint between 1+2^-7 and 1+2^-6 -> even
        1 + 2 ** -8 + 2 ** -30: 1 + 2 ** -7,  # just above the midpoint rounds up
        -(1 + 2 ** -8 + 2 ** -30): -(1 + 2 ** -7),
        3.0e38: (1 + 98 / 128) * 2.0 ** 127,  # 3e38/2^127 = 1.7632..; 0.7632*128 = 97.69 -> 98
        3.4e38: math.inf,                 # beyond the largest finite bf16 + half ulp
        2.0 ** -130: 2.0 ** -130,         # subnormal grid point
        2.0 ** -134: 0.0,                 # half of the smallest subnormal -> even (0)
        3 * 2.0 ** -134: 2.0 ** -132,     # 1.5 * 2^-133 -> 2 * 2^-133
        0.0: 0.0,
    }
    xs = np.array(list(cases.keys()))
    got = O.bf16_round(xs)
    for x, g in zip(cases, got):
        assert g == cases[x], (x, g, cases[x])


def test_bf16_round_matches_torch_on_float32_inputs():
    # torch rounds binary32 -> bf16 directly; on binary32 inputs both must agree.
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.randn(200000, generator=g) * s for s in (1e-3, 1.0, 1e3, 1e30)])
    x = torch.cat([x, torch.tensor([2.0 ** -127, -(2.0 ** -140), 1.5 * 2 ** -133])])
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(x.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------------------- transformer pieces
def test_rmsnorm_closed_form():
    d = 10
    for c in (3.0, -0.02, 1e-4):
        g = np.arange(1, d + 1, dtype=np.float64)
        y = O.rmsnorm(np.full(d, c), g, 1e-6)
        np.testing.assert_allclose(y, c / math.sqrt(c * c + 1e-6) * g, rtol=1e-14)
    # scale invariance without eps
    x = np.random.default_rng(0).standard_normal((3, d))
    np.testing.assert_allclose(O.rmsnorm(7.5 * x, 1.0, 0.0), O.rmsnorm(x, 1.0, 0.0), rtol=1e-13)


def test_rope_equals_complex_rotation_and_is_relative():
    rng = np.random.default_rng(1)
    dh, base = 16, 10000.0
    x = rng.standard_normal((5, 3, dh))
    pos = np.array([0, 1, 7, 100, 4095])
    ours = O.rope(x, pos, base)
    ref = rope_complex(torch.from_numpy(x), torch.from_numpy(pos), base).numpy()
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(O.rope(x[:1], np.array([0]), base), x[:1])  # identity at 0
    np.testing.assert_allclose(np.linalg.norm(ours, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    # <rope(q, m), rope(k, n)> depends only on m - n
    q, k = rng.standard_normal((1, 1, dh)), rng.standard_normal((1, 1, dh))
    dots = [np.sum(O.rope(q, np.array([m + s]), base) * O.rope(k, np.array([n + s]), base))
            for (m, n) in [(5, 2)] for s in (0, 13, 999)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)
    # first pair rotates by exactly pos radians (theta_0 = 1)
    e = np.zeros((1, 1, dh)); e[..., 0] = 1.0
    r = O.rope(e, np.array([2]), base)
    assert abs(r[0, 0, 0] - math.cos(2)) < 1e-15 and abs(r[0, 0, dh // 2] - math.sin(2)) < 1e-15


def test_silu_matches_logistic():
    from scipy.special import expit
    x = np.linspace(-30, 30, 101)
    np.testing.assert_allclose(O.silu(x), x * expit(x), rtol=1e-13, atol=1e-300)


def test_logit_summary_special_cases():
    V = 11
    am, mp, p2 = O.logit_summary(np.zeros((1, V)), mask_id=0)
    assert am[0] == 1 and abs(mp[0] - 1.0 / (V - 1)) < 1e-15  # [MASK] excluded, ties -> lowest
    z = np.full(V, -1e9); z[0] = 50.0; z[3] = 2.0; z[7] = 0.5
    am, mp, p2 = O.logit_summary(z, mask_id=0)
    assert am == 3
    assert abs(mp - 1.0 / (1.0 + math.exp(-1.5))) < 1e-15       # two-way softmax closed form
    assert abs(p2 - math.exp(-1.5) / (1.0 + math.exp(-1.5))) < 1e-15
    z = np.array([0.0, 5.0, 5.0, 1.0])
    assert O.logit_summary(z, 0)[0] == 1
    from scipy.special import softmax
    z = np.random.default_rng(2).standard_normal((4, 50)) * 20
    am, mp, _ = O.logit_summary(z, 0)
    zz = z.copy(); zz[:, 0] = -np.inf
    sm = softmax(zz, axis=-1)
    np.testing.assert_array_equal(am, sm.argmax(-1))
    np.testing.assert_allclose(mp, sm.max(-1), rtol=1e-13)


# --------------------------------------------------------------------------- forward
def _oracle_branch_pass(w, shape, act, prompt, branches):
    m = O.OracleModel(shape, w, act=act)
    cache = O.prefill(m, prompt, len(prompt) + branches.shape[1])
    return m, cache, O.forward(m, cache, len(prompt), branches, want_logits=True)


@pytest.mark.parametrize("act", ["fp64", "bf16"])
def test_forward_matches_independent_torch_forward(micro_w, act):
    """Oracle (cache + per-branch loops) vs torch (one masked whole-sequence pass)."""
    rng = np.random.default_rng(4)
    B, nb, Pn = 6, 3, 9
    prompt = rng.integers(1, MICRO.vocab, Pn)
    branches = rng.integers(0, MICRO.vocab, (nb, B))
    branches[rng.random((nb, B)) < 0.5] = MICRO.mask_id
    _, cache, out = _oracle_branch_pass(micro_w, MICRO, act, prompt, branches)
    positions, visible = block_layout(Pn, 0, B, nb)
    toks = np.concatenate([prompt, branches.reshape(-1)])
    z, x, ks, _ = torch_forward(micro_w, MICRO, toks, positions, visible,
                                act="bf16" if act == "bf16" else None)
    z = z[Pn:].numpy().reshape(nb, B, -1)
    x = x[Pn:].numpy().reshape(nb, B, -1)
    tol = 1e-10 if act == "fp64" else 1e-6
    np.testing.assert_allclose(out.logits[..., 1:], z[..., 1:], rtol=tol, atol=tol)
    np.testing.assert_allclose(out.x_final, x, rtol=tol, atol=tol)
    np.testing.assert_allclose(cache.k[1][:Pn], ks[1][:Pn].numpy(), rtol=tol, atol=tol)
    zz = z.copy(); zz[..., 0] = -np.inf
    np.testing.assert_array_equal(out.am, zz.argmax(-1))


def test_isolation_batched_equals_separate(micro_w):
    rng = np.random.default_rng(5)
    B, nb = 8, 4
    prompt = rng.integers(1, MICRO.vocab, 12)
    branches = rng.integers(1, MICRO.vocab, (nb, B))
    branches[rng.random((nb, B)) < 0.6] = MICRO.mask_id
    m, cache, out = _oracle_branch_pass(micro_w, MICRO, "fp64", prompt, branches)
    for b in range(nb):
        one = O.forward(m, cache, len(prompt), branches[b:b + 1], want_logits=True)
        np.testing.assert_allclose(one.logits[0], out.logits[b], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(one.am[0], out.am[b])


def test_forward_without_attention_and_mlp_is_embedding_readout(micro_w):
    """With Wo = Wd = 0 the residual stream is the embedding: logits are
    scale * rmsnorm(E[tok]) @ Wlm^T (a closed form that skips every layer)."""
    w = dict(micro_w)
    for l in range(MICRO.n_layers):
        w[f"wo.{l}"] = torch.zeros_like(w[f"wo.{l}"])
        w[f"wd.{l}"] = torch.zeros_like(w[f"wd.{l}"])
    tok = np.array([[5, 0, 17, 96]])
    m = O.OracleModel(MICRO, w, act="fp64")
    out = O.forward(m, O.KVCache.empty(MICRO, 8), 0, tok, want_logits=True)
    E = w["embed"].double().numpy()[tok[0]]
    h = E / np.sqrt((E ** 2).mean(-1, keepdims=True) + MICRO.rms_eps)
    z = 20.0 * h @ w["lm_head"].double().numpy().T
    np.testing.assert_allclose(out.logits[0], z, rtol=1e-12)


# ---------------------------------------------------------------------- decision rules
def _golden_cases():
    with open(os.path.join(GOLDEN, "decision_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_decision_rules_hand_worked(case):
    mask = 0
    anchor, S = O.anchor_fill(np.array(case["tok"]), case["am"], case["mp"], case["tau"], mask)
    assert S == case["expect_filled"]
    C = O.lookahead_candidates(anchor, case["mp"], case["k"], mask)
    assert C == case["expect_candidates"]
    br = O.build_branches(anchor, case["am"], C)
    assert br.tolist() == case["expect_branches"]
    conf = [O.branch_confidence(br[b], case["verify_mp"][b], mask) for b in range(len(br))]
    np.testing.assert_allclose(conf, case["expect_conf"], rtol=0, atol=1e-15)
    assert O.select_winner(conf) == case["expect_winner"]
    m = O.decision_margins(np.array(case["tok"]), case["mp"], case["p2"], case["tau"], case["k"],
                           mask, case["expect_conf"], case["expect_winner"])
    for key, want in case["expect_margins"].items():
        if want is None:
            assert m[key] == math.inf, (key, m[key])
        else:
            assert abs(m[key] - want) < 1e-12, (key, m[key], want)


def test_candidates_match_counting_definition():
    """Candidate set = remaining positions with fewer than k others ranked above them
    (above = strictly more confident, or equally confident and lower position)."""
    rng = np.random.default_rng(6)
    for _ in range(300):
        B = int(rng.integers(1, 12))
        tok = np.where(rng.random(B) < 0.7, 0, 5)
        mp = np.round(rng.random(B), 1)  # coarse values force ties
        am = rng.integers(1, 9, B)
        k = int(rng.integers(0, 6))
        anchor, S = O.anchor_fill(tok, am, mp, 0.9, 0)
        masked = [i for i in range(B) if tok[i] == 0]
        if masked:
            assert S, "at least one fill per step"
        for i in masked:
            assert (i in S) == (mp[i] >= 0.9) or (len(S) == 1 and all(mp[j] < 0.9 for j in masked))
        R = [i for i in range(B) if anchor[i] == 0]
        above = {i: sum(1 for j in R if mp[j] > mp[i] or (mp[j] == mp[i] and j < i)) for i in R}
        want = sorted((i for i in R if above[i] < k), key=lambda i: above[i])
        assert O.lookahead_candidates(anchor, mp, k, 0) == want


# ------------------------------------------------------------------ whole-method pins
def _threshold_decode(m, prompt, block, tau, gen_len):
    """Plain confidence-driven threshold decoding, written independently of
    lopa_step: fill all masked positions with confidence >= tau (at least the single
    most confident one), one forward per fill round."""
    mask = m.shape.mask_id
    cache = O.prefill(m, prompt, len(prompt) + gen_len)
    P, out, fw = len(prompt), [], 0
    for _ in range(gen_len // block):
        tok = [mask] * block
        res = O.forward(m, cache, P, np.array([tok])); fw += 1
        while mask in tok:
            masked = [i for i, t in enumerate(tok) if t == mask]
            conf, pred = res.mp[0], res.am[0]
            fill = [i for i in masked if conf[i] >= tau]
            if not fill:
                fill = [max(masked, key=lambda i: (conf[i], -i))]
            for i in fill:
                tok[i] = int(pred[i])
            res = O.forward(m, cache, P, np.array([tok])); fw += 1
        for l in range(m.shape.n_layers):
            cache.k[l][P:P + block] = res.block_k[l][0]
            cache.v[l][P:P + block] = res.block_v[l][0]
        out += tok
        P += block
    return np.array(out), fw


def test_k0_reduces_to_threshold_decoding(micro_w):
    m = O.OracleModel(MICRO, micro_w, act="fp64")
    prompt = synth.make_prompt(MICRO, 10, seed=1)
    want, fw_want = _threshold_decode(m, prompt, 8, 0.9, 24)
    got, fw, _, _ = O.decode(m, prompt, 8, 0, 0.9, 24)
    np.testing.assert_array_equal(got, want)
    assert fw == fw_want


def test_logit_reuse_and_kv_consistency(micro_w):
    m = O.OracleModel(MICRO, micro_w, act="fp64")
    prompt = synth.make_prompt(MICRO, 10, seed=1)
    block, gen = 6, 18
    toks, fw, cache, log = O.decode(m, prompt, block, 3, 0.9, gen, record=True)
    assert len(log) > 0
    for P, st in log:
        w = st.winner
        fresh = O.forward(m, cache, P, st.branches[w:w + 1])  # cache[0:P] is final
        np.testing.assert_array_equal(fresh.am[0], st.am)
        np.testing.assert_allclose(fresh.mp[0], st.mp, rtol=1e-12)
        conf = [O.branch_confidence(st.branches[b], st.out.mp[b], 0) for b in range(len(st.branches))]
        assert conf == st.conf
    # KV cache after decoding == K/V of one block-causal pass over prompt + output
    n_blocks = gen // block
    positions, visible = block_layout(len(prompt), n_blocks, block, 0)
    seq = np.concatenate([prompt, toks])
    _, _, ks, vs = torch_forward(micro_w, MICRO, seq, positions, visible)
    for l in range(MICRO.n_layers):
        np.testing.assert_allclose(cache.k[l][:len(seq)], ks[l].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(cache.v[l][:len(seq)], vs[l].numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("block", [4, 6])
def test_exhaustive_one_extra_position_replay(micro_w, block):
    """With k >= block every remaining position is a lookahead candidate.  At every
    iteration, score the anchor and every one-extra-position branch with its own
    separate forward; LoPA's winner must reach the brute-force maximum confidence."""
    m = O.OracleModel(MICRO, micro_w, act="fp64")
    prompt = synth.make_prompt(MICRO, 7, seed=9)
    _, _, cache, log = O.decode(m, prompt, block, block, 0.9, 2 * block, record=True)
    for P, st in log:
        anchor = st.branches[0]
        cands = [i for i in range(block) if anchor[i] == 0]
        best = -1.0
        for c in [None] + cands:
            br = anchor.copy()
            if c is not None:
                br[c] = _greedy_token_of_step(st, c)
            one = O.forward(m, cache, P, br[None, :])
            rem = [i for i in range(block) if br[i] == 0]
            conf = 1.0 if not rem else float(np.mean([one.mp[0][i] for i in rem]))
            best = max(best, conf)
        assert abs(st.conf[st.winner] - best) < 1e-12
        assert sorted(st.candidates) == cands


def _greedy_token_of_step(st, c):
    # the lookahead branch that fills c carries the greedy token of the step's input
    # summary at c; read it back from that branch
    b = 1 + st.candidates.index(c)
    return st.branches[b][c]


# ------------------------------------------------ the completing iteration (merged start)
def _completing_states(block, k, mask, seed):
    """Block states whose next iteration completes the block: every masked position
    reaches tau (the anchor completes it), or exactly one stays below tau after the anchor
    fill (lookahead branch 1 completes it, when k >= 1)."""
    rng = np.random.default_rng(seed)
    for case in range(12):
        tok = rng.integers(1, MICRO.vocab, block)
        tok[tok == mask] = 1
        am = rng.integers(1, MICRO.vocab, block)
        am[am == mask] = 1
        mp = rng.uniform(0.2, 0.99, block)
        masked = rng.choice(block, size=1 + case % 3, replace=False)
        tok[masked] = mask
        mp[masked] = 0.95
        via = "anchor"
        if case % 2 and k >= 1:
            free = np.setdiff1d(np.arange(block), masked)
            j = int(rng.choice(free))
            tok[j], mp[j] = mask, 0.5
            via = "lookahead"
        yield tok, am, mp, via


@pytest.mark.parametrize("k", [0, 1, 3])
def test_completing_iteration_winner_is_known_before_the_forward(micro_w, k):
    """When the anchor fill leaves nothing masked, or leaves one position that lookahead
    branch 1 fills, that branch scores exactly 1.0 and every other branch less, whatever
    the forward returns: the oracle's full iteration picks it (anchor, else branch 1)."""
    m = O.OracleModel(MICRO, micro_w, act="fp64")
    prompt = synth.make_prompt(MICRO, 10, seed=4)
    block, tau, mask = 6, 0.9, MICRO.mask_id
    cache = O.prefill(m, prompt, len(prompt) + block)
    n = 0
    for tok, am, mp, via in _completing_states(block, k, mask, seed=21 + k):
        st = O.lopa_step(m, cache, len(prompt), tok, am, mp, k, tau)
        want = 0 if via == "anchor" else 1
        assert st.winner == want
        assert st.conf[want] == 1.0
        assert all(c < 1.0 for b, c in enumerate(st.conf) if b != want)
        assert not (st.branches[want] == mask).any()
        n += 1
    assert n == 12


def test_merged_block_start_equals_commit_then_start(micro_w):
    """The next block's first logits computed in the completing iteration's pass - the
    finished block and the all-[MASK] next block in one block-causal forward, positions
    running on - equal the oracle's order: commit the finished block, then the next
    block's block-start forward.  The joint pass is the independent torch forward with
    a block-causal mask; both in float64."""
    m = O.OracleModel(MICRO, micro_w, act="fp64")
    prompt = synth.make_prompt(MICRO, 10, seed=5)
    P, block, mask = len(prompt), 6, MICRO.mask_id
    finished = synth.make_prompt(MICRO, block, seed=6)
    finished[finished == mask] = 1
    blank = np.full(block, mask)
    cache = O.prefill(m, prompt, P + 2 * block)
    out1 = O.forward(m, cache, P, finished[None, :])
    for l in range(MICRO.n_layers):
        cache.k[l][P:P + block] = out1.block_k[l][0]
        cache.v[l][P:P + block] = out1.block_v[l][0]
    out2 = O.forward(m, cache, P + block, blank[None, :])
    positions, visible = block_layout(P, 2, block, 0)
    seq = np.concatenate([prompt, finished, blank])
    z, _, _, _ = torch_forward(micro_w, MICRO, seq, positions, visible)
    for rows, ref in ((slice(P, P + block), out1), (slice(P + block, P + 2 * block), out2)):
        p = torch.softmax(z[rows], dim=-1)
        np.testing.assert_array_equal(torch.argmax(z[rows], dim=-1).numpy(), ref.am[0])
        np.testing.assert_allclose(p.max(dim=-1).values.numpy(), ref.mp[0], rtol=1e-10)


# ------------------------------------------------------------- planted mistakes
def _planted(monkeypatch, name, fn):
    monkeypatch.setattr(OL, name, fn)


@pytest.mark.parametrize("plant", ["rope_sign", "silu_identity", "rms_no_eps"])
def test_pins_catch_planted_mistakes(micro_w, monkeypatch, plant):
    real_rope, real_rms = OL.rope, OL.rmsnorm
    if plant == "rope_sign":
        _planted(monkeypatch, "rope", lambda x, pos, base: real_rope(x, -np.asarray(pos), base))
    elif plant == "silu_identity":
        _planted(monkeypatch, "silu", lambda x: x)
    else:
        _planted(monkeypatch, "rmsnorm", lambda x, g, eps: real_rms(x, g, 0.0))
    with pytest.raises(AssertionError):
        test_forward_matches_independent_torch_forward(micro_w, "fp64")


def test_pins_catch_planted_decision_mistakes(monkeypatch):
    cases = _golden_cases()
    monkeypatch.setattr(OL, "select_winner", lambda conf: int(len(conf) - 1 - np.argmax(conf[::-1])))
    with pytest.raises(AssertionError):
        for c in cases:
            test_decision_rules_hand_worked(c)
    monkeypatch.undo()
    monkeypatch.setattr(OL, "branch_confidence",
                        lambda br, mp, mask: float(sum(mp[i] for i in range(len(br)) if br[i] == mask)))
    with pytest.raises(AssertionError):
        for c in cases:
            test_decision_rules_hand_worked(c)


def _margins_all_positions_token(tok, mp, p2, tau, k, mask_id, conf, winner):
    m = REAL_MARGINS(tok, mp, p2, tau, k, mask_id, conf, winner)
    m["token"] = min(float(mp[i]) - float(p2[i]) for i in range(len(tok)))
    return m


def _margins_adjacent_rank(tok, mp, p2, tau, k, mask_id, conf, winner):
    m = REAL_MARGINS(tok, mp, p2, tau, k, mask_id, conf, winner)
    vals = sorted(float(mp[i]) for i in range(len(tok)) if tok[i] == mask_id)
    m["rank"] = min((b - a for a, b in zip(vals, vals[1:])), default=math.inf)
    return m


def _margins_tau_over_all(tok, mp, p2, tau, k, mask_id, conf, winner):
    m = REAL_MARGINS(tok, mp, p2, tau, k, mask_id, conf, winner)
    m["tau"] = min(abs(float(v) - tau) for v in mp)
    return m


def _margins_conf_vs_lowest(tok, mp, p2, tau, k, mask_id, conf, winner):
    m = REAL_MARGINS(tok, mp, p2, tau, k, mask_id, conf, winner)
    others = [c for b, c in enumerate(conf) if b != winner]
    m["conf"] = conf[winner] - min(others) if others else math.inf
    return m


REAL_MARGINS = O.decision_margins


@pytest.mark.parametrize("plant", [_margins_all_positions_token, _margins_adjacent_rank,
                                   _margins_tau_over_all, _margins_conf_vs_lowest])
def test_pins_catch_planted_margin_mistakes(monkeypatch, plant):
    """Each over-broad or wrong margin (the token gap over every position, the rank gap
    between any two masked positions, the threshold distance over unmasked positions, the
    confidence gap to the weakest branch) fails a hand-worked case."""
    monkeypatch.setattr(OL, "decision_margins", plant)
    with pytest.raises(AssertionError):
        for c in _golden_cases():
            test_decision_rules_hand_worked(c)


# ------------------------------------------------------ exhaustive fill-order replay
# "SJTU x Huawei Xiaoyi release LoPA", section "Problem: the token filling order limits
# parallelism": the order in which a block's positions are filled (TFO) decides what the
# model can fill in parallel, and confidence-driven decoding picks it greedily.  On tiny
# blocks every one of the B! single-token fill orders is replayed with separate forwards.
TFO_PROMPT = 9


def _state_summary(m, cache, P, state, memo):
    key = tuple(int(t) for t in state)
    if key not in memo:
        out = O.forward(m, cache, P, np.array(state)[None, :])
        memo[key] = (out.am[0], out.mp[0])
    return memo[key]


def _consistent_orders(m, cache, P, block, mask, memo):
    """All single-token fill orders (each fill takes the greedy token of a fresh forward of
    the state before it) whose every step fills the most confident masked position (lowest
    position on ties): the exhaustive replay walks every order and keeps those."""
    kept, prefixes = [], set()
    import itertools
    for order in itertools.permutations(range(block)):
        state = [mask] * block
        ok = True
        for j, pos in enumerate(order):
            prefixes.add(order[:j])
            am, mp = _state_summary(m, cache, P, state, memo)
            masked = [i for i in range(block) if state[i] == mask]
            best = max(masked, key=lambda i: (mp[i], -i))
            ok = ok and pos == best
            state[pos] = int(am[pos])
        if ok:
            kept.append((list(order), state))
    return kept, len(prefixes)


@pytest.fixture(scope="module")
def tiny_w():
    return synth.make_weights(synth.TINY[0], seed=0, threads=1)


@pytest.mark.parametrize("block", [4, 6])
def test_exhaustive_fill_order_replay_reproduces_the_chosen_order(tiny_w, block):
    """k = 0 with a threshold no probability reaches: the anchor fills one position per
    iteration, so the decode's TFO is a single-token order.  Among all block! orders,
    replayed exhaustively with a separate forward per state, exactly one is consistent with
    the per-step argmax choices, and it is the TFO the oracle recorded, with the same
    tokens and one forward per fill plus the block start."""
    shape = synth.TINY[0]
    m = O.OracleModel(shape, tiny_w, act="fp64")
    prompt = synth.make_prompt(shape, TFO_PROMPT, seed=3)
    toks, fw, cache, log = O.decode(m, prompt, block, 0, 1.5, block, record=True)
    tfo = [p for _, st in log for p in st.filled]
    assert all(len(st.filled) == 1 for _, st in log)
    memo = {}
    kept, n_prefix = _consistent_orders(m, cache, TFO_PROMPT, block, shape.mask_id, memo)
    assert n_prefix == sum(math.perm(block, j) for j in range(block))  # every order, every step
    assert len(kept) == 1
    order, state = kept[0]
    assert order == tfo
    np.testing.assert_array_equal(state, toks)
    assert fw == block + 1


@pytest.mark.parametrize("block", [4, 6])
def test_exhaustive_replay_with_lookahead_branches(tiny_w, block):
    """k >= block (every remaining position is a candidate), threshold never reached: each
    iteration fills the most confident position (the anchor) and, when a lookahead branch
    wins, one more.  Replaying all block! single-token orders, the recorded TFO (anchor
    position first within an iteration) is the only order whose groups are the iterations'
    fills, whose first fill per group is the argmax of a fresh forward of the state, and
    whose second fill is the position of the best one-extra branch, every branch scored by
    its own separate forward."""
    import itertools
    shape = synth.TINY[0]
    mask = shape.mask_id
    m = O.OracleModel(shape, tiny_w, act="fp64")
    prompt = synth.make_prompt(shape, TFO_PROMPT, seed=4)
    toks, fw, cache, log = O.decode(m, prompt, block, block, 1.5, block, record=True)
    P = TFO_PROMPT
    groups = []
    state = [mask] * block
    memo = {}
    for _, st in log:
        am, mp = _state_summary(m, cache, P, state, memo)  # fresh forward of the state
        masked = [i for i in range(block) if state[i] == mask]
        a_t = max(masked, key=lambda i: (mp[i], -i))
        anchor = list(state)
        anchor[a_t] = int(am[a_t])
        best, best_c = -1.0, None
        for c in [None] + [i for i in masked if i != a_t]:
            br = list(anchor)
            if c is not None:
                br[c] = int(am[c])
            _, mp_b = _state_summary(m, cache, P, br, memo)
            rem = [i for i in range(block) if br[i] == mask]
            conf = 1.0 if not rem else float(np.mean([mp_b[i] for i in rem]))
            if conf > best:
                best, best_c = conf, c
        group = [a_t] + ([best_c] if best_c is not None else [])
        groups.append(group)
        assert st.filled == [a_t]
        filled = sorted(i for i in range(block) if st.branches[st.winner][i] != mask and state[i] == mask)
        assert filled == sorted(group)
        state = list(st.branches[st.winner])
    np.testing.assert_array_equal(state, toks)
    tfo = [p for g in groups for p in g]
    sizes = [len(g) for g in groups]
    consistent = []
    for order in itertools.permutations(range(block)):
        i, ok = 0, True
        for g in groups:
            if list(order[i:i + len(g)]) != g:
                ok = False
                break
            i += len(g)
        if ok:
            consistent.append(list(order))
    assert consistent == [tfo] and sum(sizes) == block
    assert fw == len(log) + 1


def test_fill_order_replay_catches_planted_mistakes(tiny_w, monkeypatch):
    """An anchor fallback that fills the least confident position, or a winner rule that
    takes the lowest confidence, makes the replays fail."""
    real_fill = OL.anchor_fill

    def least_confident(tok, am, mp, tau, mask_id):
        masked = [i for i in range(len(tok)) if tok[i] == mask_id]
        if not any(mp[i] >= tau for i in masked) and masked:
            worst = min(masked, key=lambda i: (mp[i], i))
            anchor = np.array(tok, copy=True)
            anchor[worst] = am[worst]
            return anchor, [worst]
        return real_fill(tok, am, mp, tau, mask_id)

    monkeypatch.setattr(OL, "anchor_fill", least_confident)
    with pytest.raises(AssertionError):
        test_exhaustive_fill_order_replay_reproduces_the_chosen_order(tiny_w, 4)
    monkeypatch.undo()
    monkeypatch.setattr(OL, "select_winner", lambda conf: int(np.argmin(conf)))
    with pytest.raises(AssertionError):
        test_exhaustive_replay_with_lookahead_branches(tiny_w, 4)


# ------------------------------------------------------------- isolated attention
def test_isolated_attention_bruteforce_and_special_cases():
    rng = np.random.default_rng(11)
    nb, B, H, Hk, dh, P = 2, 3, 4, 2, 4, 5
    q = rng.standard_normal((nb, B, H, dh))
    kp, vp = rng.standard_normal((P, Hk, dh)), rng.standard_normal((P, Hk, dh))
    kb, vb = rng.standard_normal((nb, B, Hk, dh)), rng.standard_normal((nb, B, Hk, dh))
    got = O.isolated_attention(q, kp, vp, kb, vb)
    for b in range(nb):
        for i in range(B):
            for h in range(H):
                g = h // (H // Hk)
                keys = [kp[j, g] for j in range(P)] + [kb[b, j, g] for j in range(B)]
                vals = [vp[j, g] for j in range(P)] + [vb[b, j, g] for j in range(B)]
                sc = [sum(q[b, i, h, e] * kk[e] for e in range(dh)) / math.sqrt(dh) for kk in keys]
                mx = max(sc)
                w = [math.exp(s - mx) for s in sc]
                tot = sum(w)
                ref = [sum(w[j] * vals[j][e] for j in range(len(vals))) / tot for e in range(dh)]
                np.testing.assert_allclose(got[b, i, h], ref, rtol=1e-12, atol=1e-12)
    # one key only -> its value; identical keys -> mean of the values
    one = O.isolated_attention(q[:, :1], kp[:0], vp[:0], kb[:, :1], vb[:, :1])
    np.testing.assert_allclose(one[:, 0], np.repeat(vb[:, 0], H // Hk, axis=1), rtol=1e-14)
    same_k = np.ones((nb, B, Hk, dh))
    mean = O.isolated_attention(q, kp[:0], vp[:0], same_k, vb)
    np.testing.assert_allclose(mean[0, 1, 3], vb[0, :, 1].mean(0), rtol=1e-12)
    # another branch's block never leaks in
    vb2 = vb.copy(); vb2[1] += 100.0
    np.testing.assert_array_equal(O.isolated_attention(q, kp, vp, kb, vb2)[0], got[0])
