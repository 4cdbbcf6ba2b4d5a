"""Kernel-level parity: tcgen05 projection GEMM, fused LM head + online softmax, and
branch-isolated attention, each against the CPU oracle on seeded inputs (several tiles
plus ragged tails), through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import lopa_oracle as O
from diffusion_lookahead_decoding_gb300 import synth
from tests.gpu_util import NEAR_TIE, build_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("T,N,K", [(64, 384, 128), (160, 1536, 1024), (256, 4608, 512),
                                   (37, 256, 64), (300, 384, 192), (1, 128, 64),
                                   (256, 3584, 3584), (256, 3584, 18944), (77, 384, 18944)])
def test_linear_accumulate_matches_oracle(T, N, K):
    from diffusion_lookahead_decoding_gb300 import api
    x = _bf16((T, K), 1)
    w = _bf16((N, K), 2, 0.02)
    y0 = torch.randn(T, N, generator=torch.Generator().manual_seed(3))
    y = y0.cuda()
    api.linear_accumulate(x.cuda(), w.cuda(), y)
    got = y.cpu().double().numpy()
    xd, wd = x.double().numpy(), w.double().numpy()
    ref = y0.double().numpy() + O.linear(xd, wd)
    bound = 1e-4 * (np.abs(xd) @ np.abs(wd).T) + 1e-6 * np.abs(y0.double().numpy()) + 1e-6
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"max err {err.max()} (bound {bound[err > bound][:3]})"


@pytest.mark.parametrize("T,F,K", [(64, 128, 128), (37, 256, 64), (300, 384, 192), (1, 128, 1024),
                                   (160, 1536, 1024), (256, 18944, 3584)])
def test_swiglu_matches_oracle(T, F, K):
    """Gate/up GEMM with the SwiGLU epilogue (the last case is the 7B layer's, 256 rows)
    against the oracle's silu(x Wg^T) * (x Wu^T) rounded to bf16."""
    from diffusion_lookahead_decoding_gb300 import api
    x = _bf16((T, K), 11)
    w = _bf16((2 * F, K), 12, 0.02)
    h = api.swiglu(x.cuda(), w.cuda())
    api.kernel_status()
    got = h.cpu().double().numpy()
    xd, wd = x.double().numpy(), w.double().numpy()
    g, u = O.linear(xd, wd[:F]), O.linear(xd, wd[F:])
    ref = O.silu(g) * u
    # fp32 sums (within 1e-4 of the absolute sum, as above), then one bf16 rounding
    eg = 1e-4 * (np.abs(xd) @ np.abs(wd[:F]).T) + 1e-6
    eu = 1e-4 * (np.abs(xd) @ np.abs(wd[F:]).T) + 1e-6
    bound = 2.0 ** -8 * np.abs(ref) + 1.1 * np.abs(u) * eg + np.abs(O.silu(g)) * eu + 1e-6
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"max err {err.max()}"
    # The oracle's bf16 value exactly, except where the fp32 sums land on the other side of a
    # rounding boundary: then one bf16 step apart.  Checked where |ref| >= 1e-2, so that the
    # bf16 step (>= 2^-14) is far above the fp32 error of the sums (a few 1e-6); a wrong
    # formula (no silu, gate and up swapped) disagrees almost everywhere.
    exact = O.bf16_round(ref)
    big = np.abs(ref) >= 1e-2
    diff = (got != exact) & big
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    print(f"T={T} F={F} K={K}: {int(diff.sum())} of {int(big.sum())} outputs one bf16 step from "
          f"the oracle's rounding")
    assert diff.sum() <= 1e-2 * big.sum()
    assert (np.abs(got - exact)[diff] <= step[diff] * 1.0001).all()


@pytest.mark.parametrize("rows,d,V,mask", [(64, 128, 1024, 0), (160, 1024, 32768, 0),
                                           (37, 256, 1000, 5), (256, 512, 4096, 0),
                                           (300, 512, 4096, 3), (200, 3584, 152064, 0)])
def test_lmhead_argmax_matches_oracle(rows, d, V, mask):
    from diffusion_lookahead_decoding_gb300 import api
    h = _bf16((rows, d), 4)
    w = _bf16((V, d), 5, 0.02)
    am, mp = api.lmhead_argmax(h.cuda(), w.cuda(), 20.0, mask)
    am, mp = am.cpu().numpy(), mp.cpu().numpy()
    z = 20.0 * O.linear(h.double().numpy(), w.double().numpy())
    ram, rmp, rp2 = O.logit_summary(z, mask)
    assert (am != mask).all()
    tie = (rmp - rp2) < NEAR_TIE
    assert ((am == ram) | tie).all(), np.nonzero((am != ram) & ~tie)
    np.testing.assert_allclose(mp, rmp, atol=1e-3, rtol=0)


@pytest.mark.parametrize("nb,B,P,H,Hk,dh", [
    (1, 16, 0, 4, 4, 32), (4, 16, 32, 4, 4, 32), (5, 32, 256, 16, 4, 64),
    (8, 32, 100, 28, 4, 128), (8, 32, 1024, 28, 4, 128), (2, 64, 4096, 28, 4, 128),
    (16, 16, 257, 16, 4, 64), (1, 512, 0, 28, 4, 128),
    # head_dim 128 with the keys split over a CTA pair (prefix of 4 or more key tiles): an odd
    # tile count with a ragged last prefix tile, and a long ragged prefix; the threshold
    # itself (4 tiles), the 7B step's prefix (5 tiles), and just below it (3 tiles, one CTA)
    (3, 32, 1100, 28, 4, 128), (8, 32, 2000, 28, 4, 128), (8, 32, 512, 28, 4, 128),
    (8, 32, 640, 28, 4, 128), (8, 32, 383, 28, 4, 128)])
def test_branch_attention_matches_oracle(nb, B, P, H, Hk, dh):
    from diffusion_lookahead_decoding_gb300 import api
    q, kp, vp, kb, vb = synth.make_attention_inputs(nb, B, P, H, Hk, dh, seed=7)
    out = api.branch_attention(q.cuda(), kp.cuda(), vp.cuda(), kb.cuda(), vb.cuda())
    got = out.cpu().double().numpy().reshape(nb, B, H, dh)
    ref = O.isolated_attention(q.double().numpy().reshape(nb, B, H, dh), kp.double().numpy(),
                               vp.double().numpy(), kb.double().numpy(), vb.double().numpy())
    err = np.abs(got - ref)
    # bf16 output rounding (2^-9 relative) plus bf16 attention weights inside P.V
    assert err.max() <= 2e-2 + 8e-3 * np.abs(ref).max(), err.max()
    assert err.mean() <= 3e-3, err.mean()
