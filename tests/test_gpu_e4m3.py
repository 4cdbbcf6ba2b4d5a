"""Parity of the E4M3 weight stream (per-output-channel E4M3 weights, bf16 activations)
against the oracle's e4m3 weight mode.

* The quantiser: codes and scales byte-exact against the oracle's quantize_e4m3_rows (the
  codes are decided in float32 on both sides).
* The GEMM with E4M3 weights: every one of the 254 finite codes, through one-hot
  activations, comes back exactly (the on-chip widening to bf16, the swizzled layout and
  the per-row scale); random shapes against the oracle's float64 product.
* The verification forward and whole decodes (step-local) on the tiny, small and heads128
  (head_dim 128: the tensor-core attention) workloads, and all 256 rows of the 7B layer
  slice, against the oracle with the same quantised weights, under the bounds of the bf16
  path.
"""
import numpy as np
import pytest
import torch

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth
from tests import steplocal
from tests.gpu_util import (HIDDEN_REL_L2, MP_ABS, build_lib, make_decoder, oracle_forward_pair,
                            rel_l2, seeded_branches, token_flips, workload_weights)

pytestmark = pytest.mark.gpu


def e4m3_values(codes):
    """Values of E4M3 bytes by the field definition (1 sign, 4 exponent bits with bias 7,
    3 fraction bits; exponent field 0 = subnormal)."""
    b = np.asarray(codes, dtype=np.int64)
    s = np.where(b >> 7, -1.0, 1.0)
    e, m = (b >> 3) & 15, b & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * np.exp2(e - 7.0))
    return s * mag


@pytest.fixture(scope="module")
def api():
    build_lib()
    from diffusion_lookahead_decoding_gb300 import api as A
    return A


@pytest.mark.parametrize("rows,K", [(384, 3584), (130, 192), (1, 64)])
def test_quantizer_is_byte_exact(api, rows, K):
    rng = np.random.default_rng(rows + K)
    W = rng.standard_normal((rows, K)) * np.exp2(rng.uniform(-20, 4, (rows, 1)))
    W[rng.random((rows, K)) < 0.01] = 0.0
    if rows > 3:
        W[1] = 0.0                      # zero row: scale 1
        W[2] = 2.0 ** -130              # bf16-subnormal row
        W[3, : K // 2] *= 2.0 ** -12    # codes down in the E4M3 subnormal range
    wt = torch.tensor(W, dtype=torch.float32).to(torch.bfloat16)
    codes, scales = api.quantize_e4m3(wt.cuda())
    torch.cuda.synchronize()
    c_ref, s_ref = O.quantize_e4m3_rows(wt.to(torch.float64).numpy())
    np.testing.assert_array_equal(scales.cpu().numpy().astype(np.float64), s_ref)
    got = e4m3_values(codes.cpu().numpy())
    np.testing.assert_array_equal(got, c_ref)
    b = codes.cpu().numpy()
    assert not ((b & 0x7F) == 0x7F).any()  # never the NaN pattern


def test_e4m3_gemm_returns_every_code_exactly(api):
    """x = one-hot rows, so y[t][n] = codes[n][t] * scale[n] with a single nonzero term: the
    on-chip widening, the swizzled operand layout and the scale are checked exactly."""
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)  # 254 codes
    N, K = 384, 1024
    rng = np.random.default_rng(7)
    codes = np.stack([rng.permutation(np.resize(finite, K)) for _ in range(N)]).astype(np.uint8)
    scales = np.exp2(rng.integers(-6, 6, N)).astype(np.float32)
    T = K
    x = torch.eye(K, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((T, N), dtype=torch.float32, device="cuda")
    api.linear_accumulate_e4m3(x, torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), y)
    api.kernel_status()
    want = (e4m3_values(codes) * scales[:, None].astype(np.float64)).T
    np.testing.assert_array_equal(y.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("T,N,K", [(256, 3584, 3584), (300, 384, 18944), (77, 4608, 3584), (16, 128, 64)])
def test_e4m3_gemm_matches_oracle(api, T, N, K):
    rng = np.random.default_rng(T + N + K)
    x = torch.tensor(rng.standard_normal((T, K)), dtype=torch.float32).to(torch.bfloat16)
    w = torch.tensor(rng.standard_normal((N, K)) * 0.02, dtype=torch.float32).to(torch.bfloat16)
    codes, scales = api.quantize_e4m3(w.cuda())
    y = torch.zeros((T, N), dtype=torch.float32, device="cuda")
    api.linear_accumulate_e4m3(x.cuda(), codes, scales, y)
    api.kernel_status()
    c_ref, s_ref = O.quantize_e4m3_rows(w.to(torch.float64).numpy())
    xd, wq = x.to(torch.float64).numpy(), c_ref * s_ref[:, None]
    ref = O.linear(xd, wq)
    err = np.abs(y.cpu().numpy() - ref)
    bound = 1e-4 * (np.abs(xd) @ np.abs(wq).T) + 1e-6
    print(f"T={T} N={N} K={K}: max |y - oracle| = {err.max():.2e}")
    assert (err <= bound).all()


@pytest.mark.parametrize("name", ["tiny", "small", "heads128"])
def test_verify_forward_e4m3_matches_oracle(name):
    shape, dshape, w = workload_weights(name)
    dec = make_decoder(name, weight_format="e4m3")
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    dec.prefill(prompt)
    B, P, nb = dshape.block, dshape.prompt_len, dshape.k + 1
    br = seeded_branches(shape, nb, B, seed=5)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    dec.close()
    _, _, out, cond = oracle_forward_pair(shape, w, prompt, br, P + B, weight_format="e4m3")
    e_h = rel_l2(hid, out.x_final)
    e_mp = float(np.abs(mp - out.mp).max())
    nflip, nbad = token_flips(am, mp, out, shape.mask_id, hid, shape, w, weight_format="e4m3")
    print(f"{name} (E4M3 weights): hidden relL2 {e_h:.2e} (bound {HIDDEN_REL_L2}), maxp max|d| "
          f"{e_mp:.2e}, greedy-token flips {nflip}, beyond their window {nbad}; {cond}")
    assert e_h <= HIDDEN_REL_L2
    if name == "tiny":
        assert e_mp <= MP_ABS
    assert nbad == 0


@pytest.mark.parametrize("name", ["tiny", "small", "heads128"])
def test_decode_e4m3_step_local(name):
    shape, dshape, w = workload_weights(name)
    dec = make_decoder(name, weight_format="e4m3")
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    dec.prefill(prompt)
    m = O.OracleModel(shape, w, act="bf16", weight_format="e4m3")
    summ = steplocal.run(dec, m, shape, dshape, prompt, dshape.k)
    dec.close()
    print(summ.table_row(f"{name} E4M3 weights"))
    assert summ.n > 0


def test_dream7b_layer_e4m3_all_rows():
    """All 256 rows of the 8 x 32 step through one 7B-sized layer and the LM head, with
    E4M3 weights."""
    shape, dshape, w = workload_weights("dream7b_layer")
    B, k, P = dshape.block, dshape.k, dshape.prompt_len
    dec = make_decoder("dream7b_layer", max_seq=P + B, weight_format="e4m3")
    prompt = synth.make_prompt(shape, P, seed=1)
    dec.prefill(prompt)
    br = seeded_branches(shape, k + 1, B, seed=5)
    am, mp, hid = dec.verify_forward(br, want_hidden=True)
    dec.close()
    _, _, out, cond = oracle_forward_pair(shape, w, prompt, br, P + B, weight_format="e4m3")
    e_h = rel_l2(hid, out.x_final)
    nflip, nbad = token_flips(am, mp, out, 0, hid, shape, w, weight_format="e4m3")
    print(f"7B layer (E4M3 weights), 256 rows: hidden relL2 {e_h:.2e}, maxp max|d| "
          f"{np.abs(mp - out.mp).max():.2e}, flips {nflip} (beyond window {nbad}); {cond}")
    assert e_h <= HIDDEN_REL_L2
    assert nbad == 0
