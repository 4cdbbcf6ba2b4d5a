"""Parity on the Dream-7B-shaped workload (Qwen2.5-7B architecture, prompt 512, block 32,
k = 7): the configuration the benchmark times.

* One layer (the 7B layer and vocabulary sizes, 1 layer): all 256 rows of the 8 x 32
  verification forward through one full layer plus the LM head against the oracle.
* All 28 layers: the block-start rows and two branches of the 8-branch verification
  forward, sampled (the oracle's float64 forward of 28 layers takes seconds per row set).
  The final hidden state is held to its stated bound; the per-position max-probabilities
  and greedy tokens are printed beside the oracle's own float32-vs-float64 movement, the
  conditioning of these random-weight logits at depth.
* Four consecutive LoPA iterations from the first block, step-local (tests/steplocal.py).
"""
import copy

import numpy as np
import pytest

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth
from tests import steplocal
from tests.gpu_util import (HIDDEN_REL_L2, MP_ABS, make_decoder, oracle_forward_pair, rel_l2,
                            seeded_branches, token_flips, workload_weights)

pytestmark = pytest.mark.gpu


def _report(tag, hid, mp, am, out, cond, shape, w):
    e_h = rel_l2(hid, out.x_final)
    d = np.abs(mp - out.mp)
    nflip, nbad = token_flips(am, mp, out, 0, hid, shape, w)
    well = cond.mp_pos < 0.1 * MP_ABS
    print(f"{tag}: hidden relL2 {e_h:.2e} (bound {HIDDEN_REL_L2}); maxp |d| max {d.max():.2e}, "
          f"mean {d.mean():.2e}, positions over {MP_ABS}: {(d > MP_ABS).sum()} of {d.size}; at the "
          f"{well.sum()} positions the oracle's own float32 twin moves by < {0.1 * MP_ABS:.0e}: "
          f"max {d[well].max() if well.any() else 0:.2e}; greedy-token flips {nflip}, beyond the "
          f"per-position window {nbad}; {cond}")
    return e_h, d, nbad


def test_dream7b_one_layer_all_rows():
    """All 256 rows of the 8 x 32 step through one 7B-sized layer and the LM head."""
    shape, dshape, w = workload_weights("dream7b_layer")
    B, k, P = dshape.block, dshape.k, dshape.prompt_len
    dec = make_decoder("dream7b_layer", max_seq=P + B)
    prompt = synth.make_prompt(shape, P, seed=1)
    dec.prefill(prompt)
    br = seeded_branches(shape, k + 1, B, seed=5)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    _, _, out, cond = oracle_forward_pair(shape, w, prompt, br, P + B)
    e_h, d, nbad = _report("7B one layer, 256 rows", hid, mp, am, out, cond, shape, w)
    dec.close()
    assert e_h <= HIDDEN_REL_L2
    assert nbad == 0


@pytest.fixture(scope="module")
def dream7b_oracle():
    shape, dshape, w = workload_weights("dream7b")
    P = dshape.prompt_len
    prompt = synth.make_prompt(shape, P, seed=1)
    m = O.OracleModel(shape, w, act="bf16", cache_weights=False)
    cache = O.prefill(m, prompt, P + dshape.gen_len)
    return shape, dshape, w, prompt, m, cache


def test_dream7b_verification_sampled(dream7b_oracle):
    shape, dshape, w, prompt, m, cache = dream7b_oracle
    B, k, mask, P = dshape.block, dshape.k, shape.mask_id, dshape.prompt_len
    dec = make_decoder("dream7b", max_seq=P + 4 * B)
    dec.prefill(prompt)
    blank = np.full((1, B), mask, np.int32)
    am0, mp0, hid0 = dec.verify_forward(blank, want_hidden=True)
    br = seeded_branches(shape, k + 1, B, seed=5)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    dec.close()
    sample = [0, k]
    rows = np.concatenate([blank, br[sample]])
    out = O.forward(m, cache, P, rows, want_logits=True)
    m32 = O.OracleModel(shape, w, act="bf16", cache_weights=False, accum="fp32")
    alt = O.forward(m32, O.prefill(m32, prompt, P + B), P, rows)
    from tests.gpu_util import Conditioning
    cond = Conditioning(out, alt)
    g_am = np.stack([am0[0], am[0], am[k]])
    g_mp = np.stack([mp0[0], mp[0], mp[k]])
    g_h = np.stack([hid0[0], hid[0], hid[k]])
    e_h, _, nbad = _report("7B 28 layers, block-start rows + branches 0 and 7", g_h, g_mp, g_am,
                           out, cond, shape, w)
    assert e_h <= HIDDEN_REL_L2
    assert nbad == 0


def test_dream7b_four_iterations_step_local(dream7b_oracle):
    """The first four LoPA iterations of a 7B decode, checked step by step: the decision
    kernels exactly on the GPU's own inputs; every filled position and token against the
    oracle's own iteration from the same state, excused only by a near-tie at that step
    under the measured per-position window."""
    shape, dshape, w, prompt, m, cache = dream7b_oracle
    dec = make_decoder("dream7b")
    dec.prefill(prompt)
    summ = steplocal.run(dec, m, shape, dshape, prompt, dshape.k, max_steps=4,
                         oracle_prompt_cache=copy.deepcopy(cache))
    dec.close()
    print(summ.table_row("7B k=7, first 4 iterations"))
    for s in summ.steps:
        print(f"  P={s.P} identical={s.exact} excused_by={s.excused_by} margin={s.margin:.2e} "
              f"window={s.window:.2e} |d maxp|={s.d_mp:.2e} flips={s.flips}/{s.flips_beyond}")
    assert summ.n == 4
