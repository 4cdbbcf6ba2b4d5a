"""Decode-level parity of the CUDA path against the CPU oracle (tiny and small
workloads): the verification forward, branch isolation, single iterations from seeded
block states, whole-decode trajectories (LoPA and its k=0 reduction) and the static KV
cache.  Oracle inputs come only from the seeded generators.

Tolerances: the stated bounds (maxp 2e-2, hidden 3e-2 relative L2, decisions exact
except at near-ties under 1e-3), never tighter than twice the oracle's own movement
when only its summation precision changes (see gpu_util.Conditioning).
"""
import numpy as np
import pytest

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth
from tests.gpu_util import (device_weights, f32, make_decoder, oracle_forward_pair, rel_l2,
                            seeded_branches, tokens_ok, workload_weights)

pytestmark = pytest.mark.gpu
WORKLOADS = ["tiny", "small", "heads128"]
_COND = {}


def _setup(name, k=None):
    shape, dshape, w = workload_weights(name)
    dec = make_decoder(name, k=k)
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    dec.prefill(prompt)
    return shape, dshape, w, dec, prompt


@pytest.mark.parametrize("name", WORKLOADS)
def test_verify_forward_matches_oracle(name):
    shape, dshape, w, dec, prompt = _setup(name)
    B, P, nb = dshape.block, dshape.prompt_len, dshape.k + 1
    br = seeded_branches(shape, nb, B, seed=5)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    _, _, out, cond = oracle_forward_pair(shape, w, prompt, br, P + B)
    _COND[name] = cond
    e_h = rel_l2(hid, out.x_final)
    e_mp = float(np.abs(mp - out.mp).max())
    ok, nbad = tokens_ok(am, out, cond.tie)
    print(f"{name}: hidden relL2 {e_h:.2e} (bound {cond.hidden_bound:.1e}), maxp max|d| "
          f"{e_mp:.2e} (bound {cond.mp_bound:.1e}), token flips beyond ties {nbad}; {cond}")
    assert e_h <= cond.hidden_bound
    assert e_mp <= cond.mp_bound
    assert ok


def _cond(name, shape, w, prompt, B, P):
    if name not in _COND:
        br = seeded_branches(shape, 2, B, seed=5)
        _COND[name] = oracle_forward_pair(shape, w, prompt, br, P + B)[3]
    return _COND[name]


@pytest.mark.parametrize("name", WORKLOADS)
def test_branches_are_isolated_on_gpu(name):
    """Each branch's outputs in the batched pass equal a separate single-branch pass.  The
    mma.sync attention (head_dim 32/64) gives the same bits; the tensor-core attention
    may sum a row's keys in another order inside the MMA when its query tile holds rows of
    two branches, so there the bound is the oracle's own summation-order sensitivity (a
    leak between branches would move the outputs by far more)."""
    shape, dshape, w, dec, prompt = _setup(name)
    B, nb = dshape.block, dshape.k + 1
    br = seeded_branches(shape, nb, B, seed=6)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    if shape.head_dim == 128:
        _, _, out, cond = oracle_forward_pair(shape, w, prompt, br, dshape.prompt_len + B)
        h_tol, p_tol = 2.0 * cond.hidden, 2.0 * cond.mp
        print(f"{name}: isolation bounds hidden {h_tol:.1e}, maxp {p_tol:.1e}")
    for b in range(nb):
        am1, mp1, hid1 = dec.verify_forward(br[b:b + 1], want_hidden=True)
        if shape.head_dim != 128:
            assert rel_l2(hid1[0], hid[b]) < 1e-5
            assert np.abs(mp1[0] - mp[b]).max() < 1e-5
            np.testing.assert_array_equal(am1[0], am[b])
            continue
        assert rel_l2(hid1[0], hid[b]) < h_tol
        assert np.abs(mp1[0] - mp[b]).max() < p_tol
        flip = (am1[0] != am[b]) & ((out.mp[b] - out.p2[b]) >= cond.tie)
        assert not flip.any(), np.nonzero(flip)


@pytest.mark.parametrize("name", WORKLOADS)
def test_iteration_from_seeded_states(name):
    """One LoPA iteration from seeded block states (tokens, greedy tokens and their
    probabilities drawn by the generator): branch construction is exact; confidences
    within bound; the winner - hence the filled positions - exact except at near-ties."""
    shape, dshape, w, dec, prompt = _setup(name)
    B, k, tau, P, mask = dshape.block, dshape.k, dshape.tau, dshape.prompt_len, shape.mask_id
    cond = _cond(name, shape, w, prompt, B, P)
    m = O.OracleModel(shape, w, act="bf16")
    cache = O.prefill(m, prompt, P + B)
    ties = 0
    for seed in range(6):
        tok, am, mp = synth.make_block_state(shape, B, seed=100 + seed)
        if seed == 5:
            mp[:] = 0.95  # every masked position over tau: the anchor completes the block
        dec.rewind(P)
        dec.set_block_state(tok, am, mp)
        res = dec.step()
        st = O.lopa_step(m, cache, P, tok, am, f32(mp), k, float(np.float32(tau)))
        assert res.n_valid_branches == len(st.branches)
        conf_o = np.array(st.conf)
        # A completing iteration evaluates only its winner (confidence 1.0); the other
        # branches are reported as -inf.
        seen = np.isfinite(res.conf[:len(conf_o)])
        if not seen.all():
            assert res.block_done and seen.sum() == 1 and res.conf[res.winner] == 1.0
        assert np.abs(res.conf[:len(conf_o)][seen] - conf_o[seen]).max() <= cond.mp_bound
        assert np.isneginf(res.conf[len(conf_o):k + 1]).all()
        wg = res.winner
        if wg != st.winner:
            ties += 1
            assert abs(conf_o[wg] - conf_o[st.winner]) < cond.tie, (conf_o, res.conf, wg)
        br = st.branches[wg]
        exp_pos = [i for i in range(B) if tok[i] == mask and br[i] != mask]
        assert list(res.filled_pos) == exp_pos
        assert list(res.filled_tok) == [int(br[i]) for i in exp_pos]
        assert set(st.filled) <= set(res.filled_pos)
        assert res.block_done == (not (br == mask).any())
        if not res.block_done:
            tok2, am2, mp2, _ = dec.get_block_state()
            np.testing.assert_array_equal(tok2, br)
            assert np.abs(mp2 - st.out.mp[wg]).max() <= cond.mp_bound
    print(f"{name}: 6 seeded iterations, {ties} winner near-ties; {cond}")


def _first_divergence(a, b):
    d = np.nonzero(np.asarray(a) != np.asarray(b))[0]
    return int(d[0]) if len(d) else None


@pytest.mark.parametrize("name,k", [("tiny", None), ("small", None), ("heads128", None),
                                    ("tiny", 0), ("small", 0)])
def test_decode_trajectory_matches_oracle(name, k):
    """Whole decode on the GPU vs the oracle's decode from the same seeded prompt.
    Identical, or else the oracle met a near-tie in the block where they first
    diverge.  k=0 is plain confidence-driven threshold decoding."""
    shape, dshape, w, dec, prompt = _setup(name, k=k)
    kk = dshape.k if k is None else k
    cond = _cond(name, shape, w, prompt, dshape.block, dshape.prompt_len)
    toks, stats = dec.decode(dshape.gen_len)
    m = O.OracleModel(shape, w, act="bf16")
    otoks, ofw, _, log = O.decode(m, prompt, dshape.block, kk, dshape.tau, dshape.gen_len,
                                  record=True)
    # The GPU runs each block's block-start forward inside the previous block's
    # completing iteration (one pass), so it counts one forward less per block boundary.
    nblk = dshape.gen_len // dshape.block
    print(f"{name} k={kk}: GPU TPF {stats['tokens'] / stats['forwards']:.2f} "
          f"({stats['forwards']} fwd), oracle TPF {len(otoks) / ofw:.2f} ({ofw} fwd, "
          f"{ofw - (nblk - 1)} with merged block starts)")
    assert stats["tokens"] == dshape.gen_len and stats["blocks"] == nblk
    assert (toks != shape.mask_id).all()
    div = _first_divergence(toks, otoks)
    if div is None:
        assert stats["forwards"] == ofw - (nblk - 1)
        return
    blk_start = dshape.prompt_len + (div // dshape.block) * dshape.block
    margins = [min(st.margins.values()) for (P, st) in log if P <= blk_start]
    print(f"diverged at token {div}; smallest oracle margin up to that block {min(margins):.2e} "
          f"(tie window {cond.tie:.1e})")
    assert min(margins) < cond.tie, "diverged without an oracle near-tie"


def test_decode_at_the_maximum_block_and_branch_count():
    """The largest block (64) and branch count (16: k = 15) the ABI accepts, on the tiny
    model: 1024 token rows per verification forward, every decision kernel at full width.
    The decode matches the oracle's, or diverges only after an oracle near-tie."""
    from diffusion_lookahead_decoding_gb300 import api
    shape, dshape, w = workload_weights("tiny")
    B, k, P, gen = 64, 15, dshape.prompt_len, 128
    dec = api.LopaDecoder(shape, device_weights("tiny"), B, k, dshape.tau, P, P + gen)
    prompt = synth.make_prompt(shape, P, seed=1)
    dec.prefill(prompt)
    toks, stats = dec.decode(gen)
    cond = oracle_forward_pair(shape, w, prompt, seeded_branches(shape, 2, B, seed=5), P + B)[3]
    m = O.OracleModel(shape, w, act="bf16")
    otoks, ofw, _, log = O.decode(m, prompt, B, k, dshape.tau, gen, record=True)
    print(f"B=64 k=15: GPU {stats['forwards']} passes, oracle {ofw} forwards; {cond}")
    assert stats["tokens"] == gen and stats["blocks"] == gen // B
    assert (toks != shape.mask_id).all()
    div = _first_divergence(toks, otoks)
    if div is None:
        assert stats["forwards"] == ofw - (gen // B - 1)
        return
    blk_start = P + (div // B) * B
    margins = [min(st.margins.values()) for (Pb, st) in log if Pb <= blk_start]
    assert min(margins) < cond.tie, "diverged without an oracle near-tie"


def completing_state(shape, B, tau, seed, via):
    """A block state whose next iteration completes the block: via the anchor fill (every
    masked position reaches tau) or via lookahead branch 1 (one masked position stays
    below tau after the anchor fill and is the branch's candidate)."""
    tok, am, mp = synth.make_block_state(shape, B, seed=seed, masked_frac=0.0)
    rng = np.random.default_rng(seed + 1)
    masked = np.nonzero(tok == shape.mask_id)[0]
    mp[masked] = np.float32(0.5 * (1.0 + tau))
    if via == "lookahead":
        free = np.setdiff1d(np.arange(B), masked)
        j = int(rng.choice(free))
        tok[j] = shape.mask_id
        mp[j] = np.float32(0.5 * tau)
    winner = tok.copy()
    winner[tok == shape.mask_id] = am[tok == shape.mask_id]
    return tok, am, mp, winner


@pytest.mark.parametrize("via", ["anchor", "lookahead"])
@pytest.mark.parametrize("name", WORKLOADS)
def test_completing_iteration_starts_the_next_block(name, via):
    """An iteration that completes the block evaluates only its (already known) winner and,
    in the same pass, the next block's all-[MASK] start rows.  Against the oracle's
    unmerged order - the finished block's forward, its commit, then the block-start forward
    of the next block: the reported winner and tokens are exact, the next block's first
    (argmax, maxp) summary is within the forward's bounds, and a separate block-start
    forward on the GPU agrees with it as well."""
    shape, dshape, w, dec, prompt = _setup(name)
    B, tau, P, mask = dshape.block, dshape.tau, dshape.prompt_len, shape.mask_id
    cond = _cond(name, shape, w, prompt, B, P)
    tok, am, mp, winner = completing_state(shape, B, tau, seed=11, via=via)
    dec.set_block_state(tok, am, mp)
    res = dec.step()
    w_expect = 0 if via == "anchor" else 1
    assert res.block_done and res.winner == w_expect and res.forwards == 1
    assert res.conf[w_expect] == 1.0 and np.isneginf(np.delete(res.conf, w_expect)).all()
    tok2, am2, mp2, P2 = dec.get_block_state()
    assert P2 == P + B and (tok2 == mask).all()

    m = O.OracleModel(shape, w, act="bf16")
    cache = O.prefill(m, prompt, P + 2 * B)
    out1 = O.forward(m, cache, P, winner[None, :])
    for l in range(shape.n_layers):
        cache.k[l][P:P + B] = out1.block_k[l][0]
        cache.v[l][P:P + B] = out1.block_v[l][0]
    out2 = O.forward(m, cache, P + B, np.full((1, B), mask))
    e_mp = float(np.abs(mp2 - out2.mp[0]).max())
    ok, nbad = tokens_ok(am2[None], out2, cond.tie)
    am_s, mp_s, _ = dec.verify_forward(np.full((1, B), mask, np.int32))
    e_sep = float(np.abs(mp_s[0] - mp2).max())
    print(f"{name}/{via}: next-block maxp vs oracle {e_mp:.2e} (bound {cond.mp_bound:.1e}), "
          f"vs a separate block-start forward {e_sep:.2e}; flips beyond ties {nbad}")
    assert e_mp <= cond.mp_bound and ok
    assert e_sep <= cond.mp_bound
    ok_s, _ = tokens_ok(am_s, out2, cond.tie)
    assert ok_s


@pytest.mark.parametrize("name", WORKLOADS)
def test_kv_cache_prompt_matches_oracle_and_commits_are_fresh(name):
    """Static cache: the prompt's K/V equal the oracle's prefill; every committed block's
    K/V equal those of a fresh forward of that block over the committed prefix (the
    Commit-Winner copy holds the winner's Pre-Write exactly)."""
    shape, dshape, w, dec, prompt = _setup(name)
    B, P0 = dshape.block, dshape.prompt_len
    m = O.OracleModel(shape, w, act="bf16")
    cache = O.prefill(m, prompt, P0)
    for l in range(shape.n_layers):
        kg, vg = dec.read_kv(l, 0, P0)
        for got, ref in ((kg, cache.k[l][:P0]), (vg, cache.v[l][:P0])):
            err = np.abs(got - ref)
            assert err.max() <= 2e-2 * max(1.0, np.abs(ref).max()), (l, err.max())
            assert err.mean() <= 2e-3 * max(1.0, np.abs(ref).mean()), (l, err.mean())
    toks, _ = dec.decode(2 * B)
    committed = {l: dec.read_kv(l, P0, 2 * B) for l in range(shape.n_layers)}
    for j in (1, 0):  # rewind moves backwards only
        Pj = P0 + j * B
        dec.rewind(Pj)
        dec.verify_forward(toks[None, j * B:(j + 1) * B])
        for l in range(shape.n_layers):
            kf, vf = dec.read_branch_kv(l, 0)
            np.testing.assert_array_equal(kf, committed[l][0][j * B:(j + 1) * B])
            np.testing.assert_array_equal(vf, committed[l][1][j * B:(j + 1) * B])


@pytest.mark.parametrize("name", WORKLOADS)
def test_decode_is_deterministic(name):
    """The split-K sums are added in a fixed order and no kernel uses atomics, so two
    decodes of the same prompt (and two identical forwards) agree bit for bit."""
    shape, dshape, w, dec, prompt = _setup(name)
    br = seeded_branches(shape, dshape.k + 1, dshape.block, seed=8)
    a1, m1, h1 = dec.verify_forward(br, want_hidden=True)
    a2, m2, h2 = dec.verify_forward(br, want_hidden=True)
    np.testing.assert_array_equal(a1, a2)
    np.testing.assert_array_equal(m1, m2)
    np.testing.assert_array_equal(h1, h2)
    t1, s1 = dec.decode(dshape.gen_len)
    dec.rewind(dshape.prompt_len)
    t2, s2 = dec.decode(dshape.gen_len)
    np.testing.assert_array_equal(t1, t2)
    assert s1["forwards"] == s2["forwards"] and s1["steps"] == s2["steps"]


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
    with pytest.raises(L.LopaError) as e:
        dec.rewind(dshape.prompt_len + dshape.block)  # ahead of the committed prefix
    assert e.value.code == L.ERR_INVALID_ARG
    tok, am, mp, P = dec.get_block_state()
    assert P == dshape.prompt_len and (tok == shape.mask_id).all()
    toks, st = dec.decode(dshape.gen_len)
    assert st["tokens"] == dshape.gen_len and (toks != shape.mask_id).all()
    with pytest.raises(L.LopaError) as e:
        dec.step()  # cache full
    assert e.value.code == L.ERR_BAD_STATE
    dec.rewind(dshape.prompt_len)
    toks2, _ = dec.decode(dshape.gen_len)  # a rewound decode reproduces the tokens
    np.testing.assert_array_equal(toks2, toks)


@pytest.mark.parametrize("wl", ["tiny", "small"])
def test_timed_forwards_leave_the_decode_unchanged(wl):
    """lopa_time_forward runs the forward-only graphs (verification and block start) in the
    middle of a decode; the decode then continues exactly as an untimed one, and the call
    refuses a context without room for a block."""
    from diffusion_lookahead_decoding_gb300 import _lib as L
    shape, dshape, w = workload_weights(wl)
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    ref = make_decoder(wl)
    ref.prefill(prompt)
    ref_toks, _ = ref.decode(dshape.gen_len)
    dec = make_decoder(wl)
    dec.prefill(prompt)
    dec.step()
    before = dec.get_block_state()
    for kind in (1, 0):
        med, mean = dec.time_forward(kind, 3)
        assert 0 < med and 0 < mean
    after = dec.get_block_state()
    for x, y in zip(before, after):
        np.testing.assert_array_equal(x, y)
    dec.rewind(dshape.prompt_len)
    toks, _ = dec.decode(dshape.gen_len)
    np.testing.assert_array_equal(toks, ref_toks)
    with pytest.raises(L.LopaError) as e:
        dec.time_forward(1, 1)  # the decode filled the cache
    assert e.value.code == L.ERR_BAD_STATE
