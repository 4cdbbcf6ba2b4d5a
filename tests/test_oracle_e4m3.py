"""Pins for the oracle's E4M3 weight format (the quantised weight stream).  CPU only.

The format is fixed by its bit fields (1 sign, 4 exponent with bias 7, 3 fraction bits,
no infinities, S.1111.111 = NaN); the checks compare the oracle's rounding with a decoder
of those fields written here, with torch's float32 -> float8_e4m3fn conversion (an
independent library routine), and the per-row quantisation and the quantised forward
with the same steps written in torch."""
import numpy as np
import pytest
import torch

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth
from tests.independent_forward import block_layout, torch_forward

MICRO = synth.ModelShape(2, 64, 4, 2, 16, 128, 97, 10000.0)


def decode_e4m3_bits(code):
    """Value of an 8-bit pattern by the field definition (None for the NaN patterns)."""
    s, e, m = code >> 7, (code >> 3) & 0xF, code & 7
    if e == 15 and m == 7:
        return None
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def grid():
    vals = sorted({v for v in (decode_e4m3_bits(c) for c in range(256)) if v is not None})
    return np.array(vals)


def test_e4m3_grid_from_bit_fields_is_fixed_by_rounding():
    g = grid()
    assert len(g) == 253                      # 254 finite patterns, +0 and -0 equal
    assert g.max() == 448.0 and g.min() == -448.0
    assert g[g > 0].min() == 2.0 ** -9        # smallest subnormal
    np.testing.assert_array_equal(O.e4m3_round(g), g)


def test_e4m3_round_hand_cases():
    cases = {
        1.0625: 1.0,                 # midpoint of 1 and 1.125: ties to even (fraction 0)
        1.1875: 1.25,                # midpoint of 1.125 and 1.25: to the even fraction 2
        1.0625 + 2.0 ** -20: 1.125,  # just above a midpoint rounds up
        -3.3: -3.25,
        2.0 ** -10: 0.0,             # half the smallest subnormal -> 0 (even)
        3 * 2.0 ** -10: 2.0 ** -8,   # 1.5 subnormal steps -> 2 steps
        2.0 ** -6 - 2.0 ** -11: 2.0 ** -6,  # top of the subnormal range rounds to the first normal
        448.0: 448.0,
        464.0: 448.0,                # midpoint of 448 and (unrepresentable) 480: even, and finite
        465.0: 448.0,                # saturates
        1.0e9: 448.0,
        -1.0e9: -448.0,
        0.0: 0.0,
    }
    xs = np.array(list(cases))
    got = O.e4m3_round(xs)
    for x, g in zip(cases, got):
        assert g == cases[x], (x, g, cases[x])


def _torch_e4m3(x):
    return torch.tensor(np.asarray(x), dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_round_matches_torch_float8():
    g = grid()
    pos = g[g >= 0]
    mids = (pos[1:] + pos[:-1]) / 2                       # every tie
    ulp = lambda v, d: np.nextafter(v.astype(np.float32), np.float32(d)).astype(np.float64)
    near = np.concatenate([ulp(mids, np.inf), ulp(mids, 0)])
    rng = np.random.default_rng(0)
    rand = np.exp2(rng.uniform(-12, np.log2(448), 200000)).astype(np.float32).astype(np.float64)
    x = np.concatenate([pos, mids, near, rand])
    x = np.concatenate([x, -x])
    np.testing.assert_array_equal(O.e4m3_round(x), _torch_e4m3(x))


def _torch_quantize_rows(W):
    """The per-row quantisation written with torch tensor ops."""
    w = torch.as_tensor(np.asarray(W), dtype=torch.float32)
    amax = w.abs().amax(dim=1)
    s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    c = (w / s[:, None]).to(torch.float8_e4m3fn).to(torch.float64)
    return c.numpy(), s.to(torch.float64).numpy()


def test_quantize_rows_matches_torch_and_invariants():
    rng = np.random.default_rng(1)
    W = (rng.standard_normal((64, 96)) * np.exp2(rng.uniform(-20, 4, (64, 1))))
    W = torch.tensor(W, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    W[5] = 0.0
    W[7, :] = 2.0 ** -130  # subnormal-sized row: the scale itself is tiny
    codes, s = O.quantize_e4m3_rows(W)
    c_ref, s_ref = _torch_quantize_rows(W)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(codes, c_ref)
    assert s[5] == 1.0 and not codes[5].any()
    nz = np.abs(W).max(axis=1) > 0
    np.testing.assert_array_equal(np.abs(codes[nz]).max(axis=1), 448.0)  # the row maximum maps to 448
    np.testing.assert_array_equal(O.e4m3_round(codes), codes)            # codes on the grid
    np.testing.assert_array_equal(s.astype(np.float32).astype(np.float64), s)
    # Error of each element at most half the grid spacing at its magnitude, times the scale.
    q = W / s[:, None]
    _, ex = np.frexp(np.abs(q))
    half_step = np.ldexp(0.5, np.maximum(ex - 1, -6) - 3)
    assert np.all(np.abs(codes - q) <= half_step * (1 + 1e-6))


@pytest.fixture(scope="module")
def micro_w():
    return synth.make_weights(MICRO, seed=3, threads=1)


def test_e4m3_forward_matches_independent_torch_forward(micro_w):
    """The oracle's E4M3-weight forward against the independent torch forward fed with
    weights that torch quantised itself (every projection and the LM head)."""
    rng = np.random.default_rng(4)
    B, nb, Pn = 6, 3, 9
    prompt = rng.integers(1, MICRO.vocab, Pn)
    branches = rng.integers(0, MICRO.vocab, (nb, B))
    branches[rng.random((nb, B)) < 0.5] = MICRO.mask_id
    m = O.OracleModel(MICRO, micro_w, act="bf16", weight_format="e4m3")
    cache = O.prefill(m, prompt, Pn + B)
    out = O.forward(m, cache, Pn, branches, want_logits=True)
    wq = {}
    for name, t in micro_w.items():
        if name.split(".")[0] in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "lm_head"):
            c, s = _torch_quantize_rows(t.to(torch.float64).numpy())
            wq[name] = torch.tensor(c * s[:, None])
        else:
            wq[name] = t
    positions, visible = block_layout(Pn, 0, B, nb)
    toks = np.concatenate([prompt, branches.reshape(-1)])
    z, x, _, _ = torch_forward(wq, MICRO, toks, positions, visible, act="bf16")
    z = z[Pn:].numpy().reshape(nb, B, -1)
    x = x[Pn:].numpy().reshape(nb, B, -1)
    np.testing.assert_allclose(out.logits[..., 1:], z[..., 1:], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(out.x_final, x, rtol=1e-6, atol=1e-6)
    # The quantised model is a different model: its logits move visibly from the bf16 one.
    ref = O.forward(O.OracleModel(MICRO, micro_w, act="bf16"), O.prefill(
        O.OracleModel(MICRO, micro_w, act="bf16"), prompt, Pn + B), Pn, branches, want_logits=True)
    assert np.abs(ref.logits[..., 1:] - out.logits[..., 1:]).max() > 1e-3


@pytest.mark.parametrize("plant", ["no_subnormal_floor", "half_away_from_zero", "scale_256", "lm_head_unquantised"])
def test_e4m3_pins_catch_planted_mistakes(micro_w, monkeypatch, plant):
    if plant == "no_subnormal_floor":
        def bad(x):
            x = np.asarray(x, dtype=np.float64)
            _, ex = np.frexp(np.abs(x))
            sp = np.ldexp(1.0, ex.astype(np.int64) - 4)
            return np.copysign(np.minimum(np.round(np.abs(x) / sp) * sp, 448.0), x)
        monkeypatch.setattr(O, "e4m3_round", bad)
        check = test_e4m3_round_matches_torch_float8
    elif plant == "half_away_from_zero":
        def bad(x):
            x = np.asarray(x, dtype=np.float64)
            _, ex = np.frexp(np.abs(x))
            sp = np.ldexp(1.0, np.maximum(ex.astype(np.int64) - 1, -6) - 3)
            return np.copysign(np.minimum(np.floor(np.abs(x) / sp + 0.5) * sp, 448.0), x)
        monkeypatch.setattr(O, "e4m3_round", bad)
        check = test_e4m3_round_matches_torch_float8
    elif plant == "scale_256":
        monkeypatch.setattr(O, "E4M3_MAX", 256.0)
        check = test_quantize_rows_matches_torch_and_invariants
    else:
        monkeypatch.setattr(O, "QUANTIZED_WEIGHTS", ("wq", "wk", "wv", "wo", "wg", "wu", "wd"))
        check = lambda: test_e4m3_forward_matches_independent_torch_forward(micro_w)
    with pytest.raises(AssertionError):
        check()
