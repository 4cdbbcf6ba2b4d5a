"""Decode-level parity of the CUDA path against the CPU oracle (tiny and small
workloads): the verification forward, branch isolation, step-local decisions along the
GPU trajectory, whole-decode trajectories, the k=0 reduction and KV-cache consistency.
Integer outputs must match exactly except at oracle near-ties (< 1e-3)."""
import math

import numpy as np
import pytest

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth
from tests.gpu_util import (HIDDEN_REL_L2, MP_ABS, NEAR_TIE, f32, make_decoder, rel_l2,
                            token_mismatch_ok, workload_weights)

pytestmark = pytest.mark.gpu
WORKLOADS = ["tiny", "small"]


def _setup(name, k=None):
    shape, dshape, w = workload_weights(name)
    dec = make_decoder(name, k=k)
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    dec.prefill(prompt)
    return shape, dshape, w, dec, prompt


def _random_branches(shape, nb, B, seed):
    rng = np.random.default_rng(seed)
    br = rng.integers(1, shape.vocab, (nb, B))
    br[rng.random((nb, B)) < 0.6] = shape.mask_id
    br[:, 0] = shape.mask_id
    return br


@pytest.mark.parametrize("name", WORKLOADS)
def test_verify_forward_matches_oracle(name):
    shape, dshape, w, dec, prompt = _setup(name)
    B, P, nb = dshape.block, dshape.prompt_len, dshape.k + 1
    br = _random_branches(shape, nb, B, seed=5)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    for act, hid_tol, mp_tol in (("bf16", 1e-2, 5e-3), ("fp64", HIDDEN_REL_L2, MP_ABS)):
        m = O.OracleModel(shape, w, act=act)
        cache = O.prefill(m, prompt, P + B)
        out = O.forward(m, cache, P, br)
        e_h = rel_l2(hid, out.x_final)
        e_mp = float(np.abs(mp - out.mp).max())
        ok, nbad = token_mismatch_ok(am, out.am, out.mp, out.p2)
        print(f"{name} act={act}: hidden relL2 {e_h:.2e}  maxp max|d| {e_mp:.2e}  token flips {nbad}")
        assert e_h <= hid_tol and e_mp <= mp_tol
        if act == "bf16":
            assert ok, f"{nbad} greedy tokens differ away from near-ties"


@pytest.mark.parametrize("name", WORKLOADS)
def test_branches_are_isolated_on_gpu(name):
    shape, dshape, w, dec, prompt = _setup(name)
    B, nb = dshape.block, dshape.k + 1
    br = _random_branches(shape, nb, B, seed=6)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    for b in range(nb):
        am1, mp1, hid1 = dec.verify_forward(br[b:b + 1], want_hidden=True)
        assert rel_l2(hid1[0], hid[b]) < 1e-3
        assert np.abs(mp1[0] - mp[b]).max() < 2e-3
        assert (am1[0] == am[b]).mean() > 0.9


def _start_state(dec, shape, B):
    blank = np.full((1, B), shape.mask_id, np.int32)
    am0, mp0, _ = dec.verify_forward(blank)
    dec.set_block_state(blank[0], am0[0], mp0[0])
    return blank[0], am0[0], mp0[0]


@pytest.mark.parametrize("name", WORKLOADS)
def test_step_local_parity_along_gpu_trajectory(name):
    """Before every GPU iteration read the GPU state; the oracle takes the same
    decisions from it (in fp32, the kernels' precision), runs its own verification
    forward and scores the branches.  Branch count, filled positions and tokens must
    match exactly; confidences within 2e-2; the winner except at confidence near-ties."""
    shape, dshape, w, dec, prompt = _setup(name)
    B, k, tau, mask = dshape.block, dshape.k, dshape.tau, shape.mask_id
    m = O.OracleModel(shape, w, act="bf16")
    cache = O.prefill(m, prompt, dshape.prompt_len + 2 * B)
    P = dshape.prompt_len
    n_iter, n_ties, worst_conf = 0, 0, 0.0
    for blk in range(2):
        _start_state(dec, shape, B)
        for _ in range(B + 1):
            tok, am, mp, Pg = dec.get_block_state()
            assert Pg == P
            res = dec.step()
            n_iter += 1
            anchor, S = O.anchor_fill(tok, am, f32(mp), float(np.float32(tau)), mask)
            C = O.lookahead_candidates(anchor, f32(mp), k, mask)
            br = O.build_branches(anchor, am, C)
            assert res.n_valid_branches == len(br)
            out = O.forward(m, cache, P, br)
            conf_o = [O.branch_confidence(br[b], out.mp[b], mask) for b in range(len(br))]
            conf_g = res.conf[:len(br)]
            worst_conf = max(worst_conf, float(np.abs(conf_g - conf_o).max()))
            assert np.abs(conf_g - conf_o).max() <= MP_ABS
            assert np.isneginf(res.conf[len(br):k + 1]).all()
            w_o = O.select_winner(conf_o)
            wg = res.winner
            if wg != w_o:
                n_ties += 1
                assert abs(conf_o[wg] - conf_o[w_o]) < NEAR_TIE, (conf_o, conf_g, wg, w_o)
            exp_pos = [i for i in range(B) if tok[i] == mask and br[wg][i] != mask]
            assert list(res.filled_pos) == exp_pos
            assert list(res.filled_tok) == [int(br[wg][i]) for i in exp_pos]
            assert res.block_done == (not (br[wg] == mask).any())
            if res.block_done:
                for l in range(shape.n_layers):
                    cache.k[l][P:P + B] = out.block_k[l][wg]
                    cache.v[l][P:P + B] = out.block_v[l][wg]
                P += B
                break
            tok2, am2, mp2, _ = dec.get_block_state()
            np.testing.assert_array_equal(tok2, br[wg])
            assert np.abs(mp2 - out.mp[wg]).max() <= MP_ABS
            ok, nbad = token_mismatch_ok(am2, out.am[wg], out.mp[wg], out.p2[wg])
            assert ok, nbad
        else:
            pytest.fail("block did not finish within B iterations")
    print(f"{name}: {n_iter} iterations, {n_ties} winner near-ties, max |conf diff| {worst_conf:.2e}")


def _first_divergence(a, b):
    d = np.nonzero(np.asarray(a) != np.asarray(b))[0]
    return int(d[0]) if len(d) else None


@pytest.mark.parametrize("name,k", [("tiny", None), ("small", None), ("tiny", 0), ("small", 0)])
def test_decode_trajectory_matches_oracle(name, k):
    """Whole decode on the GPU vs the oracle's decode.  Identical unless the oracle met
    a near-tie (< 1e-3) in the block where they first diverge; k=0 is plain
    confidence-driven threshold decoding."""
    shape, dshape, w, dec, prompt = _setup(name, k=k)
    kk = dshape.k if k is None else k
    toks, stats = dec.decode(dshape.gen_len)
    m = O.OracleModel(shape, w, act="bf16")
    otoks, ofw, _, log = O.decode(m, prompt, dshape.block, kk, dshape.tau, dshape.gen_len,
                                  record=True)
    tpf = stats["tokens"] / stats["forwards"]
    print(f"{name} k={kk}: GPU TPF {tpf:.2f} ({stats['forwards']} fwd), oracle TPF "
          f"{len(otoks) / ofw:.2f} ({ofw} fwd)")
    assert stats["tokens"] == dshape.gen_len and stats["blocks"] == dshape.gen_len // dshape.block
    div = _first_divergence(toks, otoks)
    if div is None:
        assert stats["forwards"] == ofw
        return
    blk_start = dshape.prompt_len + (div // dshape.block) * dshape.block
    margins = [min(st.margins.values()) for (P, st) in log if P <= blk_start]
    print(f"diverged at token {div}; smallest oracle margin up to that block {min(margins):.2e}")
    assert min(margins) < NEAR_TIE, "diverged without an oracle near-tie"


@pytest.mark.parametrize("name", WORKLOADS)
def test_kv_cache_matches_oracle_recompute(name):
    """Two-phase update: after decoding, the static cache must hold the K/V that a
    from-scratch pass over [prompt + generated tokens] produces."""
    shape, dshape, w, dec, prompt = _setup(name)
    B = dshape.block
    gen = 2 * B
    toks, _ = dec.decode(gen)
    m = O.OracleModel(shape, w, act="bf16")
    cache = O.prefill(m, prompt, dshape.prompt_len + gen)
    P = dshape.prompt_len
    for j in range(gen // B):
        blk = toks[j * B:(j + 1) * B]
        out = O.forward(m, cache, P, blk[None, :])
        for l in range(shape.n_layers):
            cache.k[l][P:P + B] = out.block_k[l][0]
            cache.v[l][P:P + B] = out.block_v[l][0]
        P += B
    for l in range(shape.n_layers):
        kg, vg = dec.read_kv(l, 0, P)
        for got, ref in ((kg, cache.k[l][:P]), (vg, cache.v[l][:P])):
            err = np.abs(got - ref)
            assert err.max() <= 2e-2 * max(1.0, np.abs(ref).max()), (l, err.max())
            assert err.mean() <= 2e-3 * max(1.0, np.abs(ref).mean()), (l, err.mean())


def test_state_errors_leave_state_unchanged():
    from diffusion_lookahead_decoding_gb300 import _lib as L
    shape, dshape, w = workload_weights("tiny")
    dec = make_decoder("tiny")
    with pytest.raises(L.LopaError) as e:
        dec.step()
    assert e.value.code == L.ERR_BAD_STATE
    dec.prefill(synth.make_prompt(shape, dshape.prompt_len, seed=1))
    with pytest.raises(L.LopaError) as e:
        dec.decode(dshape.block + 1)
    assert e.value.code == L.ERR_INVALID_ARG
    with pytest.raises(L.LopaError) as e:
        dec.decode(dshape.gen_len + dshape.block)  # beyond max_seq
    assert e.value.code == L.ERR_BAD_STATE
    tok, am, mp, P = dec.get_block_state()
    assert P == dshape.prompt_len and (tok == shape.mask_id).all()
    toks, st = dec.decode(dshape.gen_len)
    assert st["tokens"] == dshape.gen_len and (toks != shape.mask_id).all()
    with pytest.raises(L.LopaError) as e:
        dec.step()  # cache full
    assert e.value.code == L.ERR_BAD_STATE
