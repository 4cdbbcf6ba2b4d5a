"""Full-size check on the Dream-7B-shaped workload (Qwen2.5-7B architecture, prompt
512, block 32, k=7).  The GPU runs the block-start forward, the 8-branch verification
forward (the launch configuration the benchmark times) on seeded branches, and one LoPA
iteration from a seeded block state; the oracle recomputes sampled outputs (the
block-start rows and two branches) in float64 with bf16 storage."""
import numpy as np
import pytest

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth
from tests.gpu_util import (f32, make_decoder, oracle_forward_pair, rel_l2, seeded_branches,
                            tokens_ok, workload_weights)

pytestmark = pytest.mark.gpu


def test_dream7b_verification_sampled_parity():
    shape, dshape, w = workload_weights("dream7b")
    B, k, tau, mask, P = dshape.block, dshape.k, dshape.tau, shape.mask_id, dshape.prompt_len
    dec = make_decoder("dream7b", max_seq=P + 4 * B)
    prompt = synth.make_prompt(shape, P, seed=1)
    dec.prefill(prompt)
    blank = np.full((1, B), mask, np.int32)
    am0, mp0, hid0 = dec.verify_forward(blank, want_hidden=True)
    br = seeded_branches(shape, k + 1, B, seed=5)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    tok, sam, smp = synth.make_block_state(shape, B, seed=7)
    dec.set_block_state(tok, sam, smp)
    res = dec.step()

    sample = [0, k]
    rows = np.concatenate([blank, br[sample]])
    m, cache, out, cond = oracle_forward_pair(shape, w, prompt, rows, P + B, cache_weights=False)
    print(cond)
    for j, (g_am, g_mp, g_h) in enumerate([(am0[0], mp0[0], hid0[0]),
                                           (am[0], mp[0], hid[0]), (am[k], mp[k], hid[k])]):
        e_h = rel_l2(g_h, out.x_final[j])
        e_mp = float(np.abs(g_mp - out.mp[j]).max())
        # When every probability is within e_mp of the oracle's, the greedy token can only
        # differ where the oracle's top-2 margin is below 2 * e_mp; a flip at a wider
        # margin would be an argmax inconsistency.  (e_mp itself is bounded below.)
        tie = max(cond.tie, 2.0 * e_mp)
        ok, nbad = tokens_ok(g_am[None], type("o", (), {"am": out.am[j:j + 1], "mp": out.mp[j:j + 1],
                                                         "p2": out.p2[j:j + 1]}), tie)
        print(f"row-set {j}: hidden relL2 {e_h:.2e} (bound {cond.hidden_bound:.1e}) maxp max|d| "
              f"{e_mp:.2e} (bound {cond.mp_bound:.1e}) token flips beyond ties {nbad}")
        assert e_h <= cond.hidden_bound and e_mp <= cond.mp_bound and ok

    anchor, S = O.anchor_fill(tok, sam, f32(smp), float(np.float32(tau)), mask)
    C = O.lookahead_candidates(anchor, f32(smp), k, mask)
    sb = O.build_branches(anchor, sam, C)
    assert res.n_valid_branches == len(sb)
    assert set(S) <= set(res.filled_pos)
    pick = [0, len(sb) - 1]
    o2 = O.forward(m, cache, P, sb[pick])
    for j, b in enumerate(pick):
        conf_o = O.branch_confidence(sb[b], o2.mp[j], mask)
        print(f"branch {b}: conf GPU {res.conf[b]:.4f} oracle {conf_o:.4f}")
        if not np.isfinite(res.conf[b]):  # a completing iteration evaluates only its winner
            assert res.block_done and b != res.winner
            continue
        assert abs(res.conf[b] - conf_o) <= cond.mp_bound
