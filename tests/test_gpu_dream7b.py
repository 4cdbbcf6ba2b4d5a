"""Full-size check on the Dream-7B-shaped workload (Qwen2.5-7B architecture, prompt
512, block 32, k=7): the GPU runs the block-start forward and the 8-branch verification
forward in the configuration the benchmark times; the oracle recomputes sampled outputs
(the block-start rows and two of the eight branches) in float64 with bf16 storage."""
import numpy as np
import pytest

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth
from tests.gpu_util import (MP_ABS, NEAR_TIE, f32, make_decoder, rel_l2, token_mismatch_ok,
                            workload_weights)

pytestmark = pytest.mark.gpu


def test_dream7b_verification_step_sampled_parity():
    name = "dream7b"
    shape, dshape, w = workload_weights(name)
    B, k, tau, mask = dshape.block, dshape.k, dshape.tau, shape.mask_id
    dec = make_decoder(name, max_seq=dshape.prompt_len + 4 * B)
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    dec.prefill(prompt)
    blank = np.full((1, B), mask, np.int32)
    am0, mp0, hid0 = dec.verify_forward(blank, want_hidden=True)
    dec.set_block_state(blank[0], am0[0], mp0[0])
    anchor, S = O.anchor_fill(blank[0], am0[0], f32(mp0[0]), float(np.float32(tau)), mask)
    C = O.lookahead_candidates(anchor, f32(mp0[0]), k, mask)
    br = O.build_branches(anchor, am0[0], C)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)  # the 8-branch launch config
    res = dec.step()
    assert res.n_valid_branches == len(br)

    m = O.OracleModel(shape, w, act="bf16", cache_weights=False)
    cache = O.prefill(m, prompt, dshape.prompt_len + B)
    P = dshape.prompt_len
    o0 = O.forward(m, cache, P, blank)
    print(f"start: hidden relL2 {rel_l2(hid0[0], o0.x_final[0]):.2e} "
          f"maxp max|d| {np.abs(mp0[0] - o0.mp[0]).max():.2e}")
    assert rel_l2(hid0[0], o0.x_final[0]) <= 3e-2
    assert np.abs(mp0[0] - o0.mp[0]).max() <= MP_ABS
    assert token_mismatch_ok(am0[0], o0.am[0], o0.mp[0], o0.p2[0])[0]
    sample = [0, len(br) - 1]
    ob = O.forward(m, cache, P, br[sample])
    for j, b in enumerate(sample):
        e_h = rel_l2(hid[b], ob.x_final[j])
        e_mp = float(np.abs(mp[b] - ob.mp[j]).max())
        print(f"branch {b}: hidden relL2 {e_h:.2e} maxp max|d| {e_mp:.2e}")
        assert e_h <= 3e-2 and e_mp <= MP_ABS
        ok, nbad = token_mismatch_ok(am[b], ob.am[j], ob.mp[j], ob.p2[j])
        assert ok, nbad
        conf_o = O.branch_confidence(br[b], ob.mp[j], mask)
        assert abs(res.conf[b] - conf_o) <= MP_ABS
