"""Step-local decision parity of the CUDA decode against the oracle.

The GPU decodes with lopa_step.  Before every iteration the harness reads the GPU's block
state (its tokens, and the greedy tokens / max-probabilities of the reused logits) and:

1. Decision kernels, exactly: the oracle's decision rules applied to the GPU's own
   inputs (tokens, reused (argmax, maxp) as float32, tau as float32) and to the GPU's own
   branch confidences must give the GPU's branch count, winner and filled positions and
   tokens bit for bit.  No excuse applies here.
2. Forward: the oracle runs its own forward of the same block state (its own cache, built
   from the prompt and the blocks the GPU committed) and the GPU's reused (argmax, maxp)
   are compared with it position by position.
3. Decisions against the oracle: the oracle runs its own iteration from that state with
   its own logits.  The positions filled and their tokens must equal the GPU's, except
   where a decision the difference traces back to is a near-tie at that step: its margin
   (oracle.decision_margins) is below max(1e-3, the measured GPU-oracle difference of the
   quantities it compares at that step).  Every excused step is recorded.
   Greedy-token differences at masked positions the iteration does not fill decide
   nothing; they are counted (flips, and those whose two-token gap exceeds twice the
   error measured on the GPU's token) as a report.

Only integer tokens of the GPU's decode reach the oracle (to replay the GPU's trajectory,
as step-local parity requires); every float the oracle uses is its own.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth

NEAR_TIE = 1e-3


def f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


@dataclasses.dataclass
class StepReport:
    P: int
    exact: bool
    excused_by: str | None
    margin: float
    window: float
    d_mp: float          # max |GPU - oracle| maxp over the masked positions of the state
    flips: int           # greedy-token differences at masked positions
    flips_beyond: int    # ... beyond the per-position window (tests/gpu_util.token_flips)


@dataclasses.dataclass
class Summary:
    steps: list
    blocks: int
    tokens: np.ndarray
    forwards: int

    @property
    def n(self):
        return len(self.steps)

    @property
    def excused(self):
        return [s for s in self.steps if not s.exact]

    def table_row(self, name):
        ex = self.excused
        big = max((s.margin for s in ex), default=float("nan"))
        return (f"{name}: {self.n} iterations compared, {self.n - len(ex)} identical, "
                f"{len(ex)} excused ({', '.join(sorted(set(s.excused_by for s in ex))) or '-'}), "
                f"largest excused margin {big:.2e}, max |d maxp| {max(s.d_mp for s in self.steps):.2e}, "
                f"token flips beyond the window {sum(s.flips_beyond for s in self.steps)}")


def _filled(before, after, mask):
    pos = [i for i in range(len(before)) if before[i] == mask and after[i] != mask]
    return pos, [int(after[i]) for i in pos]


def _gpu_branches(tok, am, mp, k, tau, mask):
    """The branches the decision rules build from the GPU's inputs (float32 values)."""
    anchor, S = O.anchor_fill(tok, am, f32(mp), float(np.float32(tau)), mask)
    C = O.lookahead_candidates(anchor, f32(mp), k, mask)
    return O.build_branches(anchor, am, C), S, C


def _excuse(st, res, tok, mp_g, mp_o, z, S_g, C_g, pos_g, fill_g, pos_o, fill_o, w_g, tau,
            mask):
    """The decision a GPU/oracle difference traces back to, its margin at this step and
    the window: (name, margin, window)."""
    tau32 = float(np.float32(tau))
    d = np.abs(mp_g - mp_o)
    masked = [i for i in range(len(tok)) if tok[i] == mask]
    if sorted(st.filled) != sorted(S_g):
        reach_o = any(mp_o[i] >= tau for i in masked)
        reach_g = any(f32(mp_g)[i] >= tau32 for i in masked)
        if not reach_o and not reach_g:  # both fell back to the single best position
            return "fallback", st.margins["fallback"], max(NEAR_TIE, 2.0 * float(d[masked].max()))
        diff = sorted(set(st.filled) ^ set(S_g))
        return ("tau", min(abs(float(mp_o[i]) - tau) for i in diff),
                max(NEAR_TIE, float(d[diff].max())))
    if sorted(st.candidates) != sorted(C_g):
        diff = sorted(set(st.candidates) ^ set(C_g))
        return "rank", st.margins["rank"], max(NEAR_TIE, 2.0 * float(d[diff].max()))
    # Same branches (the candidate order may differ): map GPU branch b to the oracle's.
    to_o = lambda b: 0 if b == 0 else 1 + st.candidates.index(C_g[b - 1])
    to_g = lambda b: 0 if b == 0 else 1 + C_g.index(st.candidates[b - 1])
    if set(pos_o) != set(pos_g):
        w_o = st.winner
        d_conf = abs(float(res.conf[w_g]) - st.conf[to_o(w_g)]) + \
            abs(float(res.conf[to_g(w_o)]) - st.conf[w_o])
        return "conf", st.conf[w_o] - st.conf[to_o(w_g)], max(NEAR_TIE, d_conf)
    # The same positions with another token: per position, the oracle's probability gap
    # between its token and the GPU's against twice the measured error on the GPU's token;
    # the position closest to failing is reported.
    worst = None
    for p, a, b in zip(pos_g, fill_g, fill_o):
        if a == b:
            continue
        pr = np.exp(z[p] - z[p].max())
        pr /= pr.sum()
        g_ab = float(pr[b] - pr[a])
        win = max(NEAR_TIE, 2.0 * abs(float(mp_g[p]) - float(pr[a])))
        if worst is None or g_ab / win > worst[0] / worst[1]:
            worst = (g_ab, win)
    return "token", worst[0], worst[1]


def run(dec, model, shape, dshape, prompt, k, max_steps=None, oracle_prompt_cache=None):
    """Decodes dshape.gen_len tokens (or max_steps iterations) with dec.step(), checking every
    iteration as described above.  Returns a Summary; raises AssertionError on a failure."""
    B, tau, mask = dshape.block, dshape.tau, shape.mask_id
    P0 = len(prompt)
    cap = P0 + dshape.gen_len
    cache = oracle_prompt_cache or O.prefill(model, prompt, cap)
    P = P0
    steps, out_tokens, forwards = [], [], 0
    first = True
    while P < cap and (max_steps is None or len(steps) < max_steps):
        tok_g, am_g, mp_g, Pg = dec.get_block_state()
        assert Pg == P, (Pg, P)
        if first:  # a fresh block: its logits come from the block-start forward in step()
            am_s, mp_s, _ = dec.verify_forward(tok_g[None, :])
            am_g, mp_g = am_s[0], mp_s[0]
            first = False
        ref = O.forward(model, cache, P, tok_g[None, :], want_logits=True)
        am_o, mp_o, p2_o = ref.am[0], ref.mp[0], ref.p2[0]
        masked = tok_g == mask
        d_mp = float(np.abs(mp_g - mp_o)[masked].max())
        flip = masked & (am_g != am_o)
        gap = (mp_o - p2_o)
        # per flipped position: the oracle's gap between its token and the GPU's, against
        # twice the measured error on the GPU's token (tests/gpu_util.token_flips)
        z = np.array(ref.logits[0], np.float64)
        z[:, mask] = -np.inf
        n_beyond = 0
        for i in np.nonzero(flip)[0]:
            p = np.exp(z[i] - z[i].max())
            p /= p.sum()
            g_ab = p[am_o[i]] - p[am_g[i]]
            n_beyond += int(g_ab >= max(NEAR_TIE, 2.0 * abs(float(mp_g[i]) - p[am_g[i]])))

        # (1) the decision kernels on the GPU's own inputs, exactly
        br_g, S_g, C_g = _gpu_branches(tok_g, am_g, mp_g, k, tau, mask)
        res = dec.step()
        forwards += res.forwards
        nrem = int((br_g[0] == mask).sum())
        final = 0 if nrem == 0 else (1 if nrem == 1 and len(C_g) >= 1 else -1)
        assert res.n_valid_branches == len(br_g), (res.n_valid_branches, len(br_g))
        if final >= 0:
            assert res.block_done and res.winner == final, (res.winner, final)
            assert res.conf[final] == 1.0
        else:
            assert res.winner == O.select_winner(list(res.conf[:len(br_g)])), res.conf
        w_g = res.winner
        pos_g, tok_fill_g = _filled(tok_g, br_g[w_g], mask)
        assert list(res.filled_pos) == pos_g, (res.filled_pos, pos_g)
        assert list(res.filled_tok) == tok_fill_g
        assert res.block_done == (not (br_g[w_g] == mask).any())

        # (3) against the oracle's own iteration from the same state
        st = O.lopa_step(model, cache, P, tok_g, am_o, mp_o, k, tau, p2_o)
        pos_o, tok_fill_o = _filled(tok_g, st.branches[st.winner], mask)
        exact = pos_o == pos_g and tok_fill_o == tok_fill_g
        excused_by, margin, window = None, math.nan, math.nan
        if not exact:
            key, margin, window = _excuse(st, res, tok_g, mp_g, mp_o, z, S_g, C_g, pos_g,
                                          tok_fill_g, pos_o, tok_fill_o, w_g, tau, mask)
            assert margin < window, (f"P={P}: GPU filled {pos_g} {tok_fill_g}, oracle {pos_o} "
                                     f"{tok_fill_o}; {key} margin {margin:.3e} >= window {window:.3e}")
            excused_by = key
        steps.append(StepReport(P, exact, excused_by, margin, window, d_mp, int(flip.sum()),
                                n_beyond))

        if res.block_done:
            block = br_g[w_g]
            out_tokens.extend(int(t) for t in block)
            done = O.forward(model, cache, P, block[None, :])
            for l in range(shape.n_layers):
                cache.k[l][P:P + B] = done.block_k[l][0]
                cache.v[l][P:P + B] = done.block_v[l][0]
            P += B
            if P >= cap:
                break
    return Summary(steps, (P - P0) // B, np.array(out_tokens, dtype=np.int64), forwards)
