"""The device-error path, exercised without faulting the GPU.

(a) A failure planted on the host: the context's device error word is set as a bounded
    device-side wait that gave up would set it.  lopa_step must report
    LOPA_ERR_DEVICE_TIMEOUT, and after lopa_rewind the decode must reproduce the tokens of
    an undisturbed decode.
(b) A wait that really runs out: with a test-only wait limit of 100 ns the standalone LM
    head's pipeline waits give up; the kernel drains its own copies and MMAs, frees its
    tensor memory and returns, and lopa_kernel_status reports the timeout.  With the
    default limit restored the same call is correct again, so the context stays usable.
    The same with the E4M3 weight stream's GEMM (its converter warps wait too) and the
    gate/up GEMM with its SwiGLU epilogue.
"""
import numpy as np
import pytest
import torch

from diffusion_lookahead_decoding_gb300 import _lib as L
from diffusion_lookahead_decoding_gb300 import synth
from tests.gpu_util import build_lib, make_decoder, workload_weights

pytestmark = pytest.mark.gpu


def test_planted_device_error_is_reported_and_rewind_recovers():
    from diffusion_lookahead_decoding_gb300 import api
    shape, dshape, _ = workload_weights("tiny")
    dec = make_decoder("tiny")
    prompt = synth.make_prompt(shape, dshape.prompt_len, seed=1)
    dec.prefill(prompt)
    ref, _ = dec.decode(dshape.gen_len)
    dec.rewind(dshape.prompt_len)
    dec.debug_set_device_error(1)
    with pytest.raises(L.LopaError) as e:
        dec.step()
    assert e.value.code == L.ERR_DEVICE_TIMEOUT
    dec.rewind(dshape.prompt_len)
    toks, st = dec.decode(dshape.gen_len)
    np.testing.assert_array_equal(toks, ref)
    # A decode that meets the planted error stops with the same status.
    dec.rewind(dshape.prompt_len)
    dec.debug_set_device_error(3)
    with pytest.raises(L.LopaError) as e:
        dec.decode(dshape.gen_len)
    assert e.value.code == L.ERR_DEVICE_TIMEOUT
    dec.rewind(dshape.prompt_len)
    toks, _ = dec.decode(dshape.gen_len)
    np.testing.assert_array_equal(toks, ref)
    dec.close()


@pytest.mark.parametrize("static", [False, True])
def test_short_wait_limit_reports_timeout_and_the_call_recovers(static):
    from diffusion_lookahead_decoding_gb300 import api
    build_lib()
    lib = L.load()
    rows, d, V = 256, 3584, 152064
    g = torch.Generator().manual_seed(13)
    h = torch.randn(rows, d, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16).cuda()

    def call():
        if not static:
            return api.lmhead_argmax(h, w, 20.0, 0)
        am = torch.empty(rows, dtype=torch.int32, device="cuda")
        mp = torch.empty(rows, dtype=torch.float32, device="cuda")
        L.check(lib.lopa_lmhead_argmax_static(h.data_ptr(), w.data_ptr(), rows, d, V, 20.0, 0,
                                              am.data_ptr(), mp.data_ptr(), api._stream_ptr()))
        return am, mp

    api.kernel_status()  # nothing pending
    am_ref, mp_ref = call()
    api.kernel_status()
    am_ref, mp_ref = am_ref.cpu().numpy(), mp_ref.cpu().numpy()
    try:
        api.set_wait_limit_ns(100)
        call()
        with pytest.raises(L.LopaError) as e:
            api.kernel_status()
        assert e.value.code == L.ERR_DEVICE_TIMEOUT
    finally:
        api.set_wait_limit_ns(0)
    api.kernel_status()  # the record was cleared
    am, mp = call()
    api.kernel_status()
    np.testing.assert_array_equal(am.cpu().numpy(), am_ref)
    np.testing.assert_array_equal(mp.cpu().numpy(), mp_ref)


def test_short_wait_limit_in_the_e4m3_gemm_reports_timeout_and_recovers():
    """The same for the E4M3 weight stream, whose converter warps add their own bounded
    waits (staging ring of codes, converted slots): a wait that gives up stops the kernel
    cleanly (the codes' copies and the MMAs it started are drained) and is reported; the
    next call with the default limit is correct."""
    from diffusion_lookahead_decoding_gb300 import api
    from oracle import lopa_oracle as O
    build_lib()
    T, N, K = 256, 3584, 18944
    g = torch.Generator().manual_seed(17)
    x = torch.randn(T, K, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    codes, scales = api.quantize_e4m3(w)
    api.kernel_status()
    try:
        api.set_wait_limit_ns(100)
        y = torch.zeros(T, N, dtype=torch.float32, device="cuda")
        api.linear_accumulate_e4m3(x, codes, scales, y)
        with pytest.raises(L.LopaError) as e:
            api.kernel_status()
        assert e.value.code == L.ERR_DEVICE_TIMEOUT
    finally:
        api.set_wait_limit_ns(0)
    api.kernel_status()
    y = torch.zeros(T, N, dtype=torch.float32, device="cuda")
    api.linear_accumulate_e4m3(x, codes, scales, y)
    api.kernel_status()
    c_ref, s_ref = O.quantize_e4m3_rows(w.cpu().to(torch.float64).numpy())
    xd, wq = x.cpu().to(torch.float64).numpy(), c_ref * s_ref[:, None]
    err = np.abs(y.cpu().numpy() - O.linear(xd, wq))
    assert (err <= 1e-4 * (np.abs(xd) @ np.abs(wq).T) + 1e-6).all()


def test_short_wait_limit_in_the_swiglu_gemm_reports_timeout_and_recovers():
    """The same for the gate/up GEMM with its SwiGLU epilogue (`lopa_swiglu`): a wait that
    gives up is reported, and the next call with the default limit matches the oracle."""
    from diffusion_lookahead_decoding_gb300 import api
    from oracle import lopa_oracle as O
    build_lib()
    T, F, K = 256, 1536, 3584
    g = torch.Generator().manual_seed(19)
    x = torch.randn(T, K, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(2 * F, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    api.kernel_status()
    try:
        api.set_wait_limit_ns(100)
        api.swiglu(x, w)
        with pytest.raises(L.LopaError) as e:
            api.kernel_status()
        assert e.value.code == L.ERR_DEVICE_TIMEOUT
    finally:
        api.set_wait_limit_ns(0)
    api.kernel_status()
    h = api.swiglu(x, w)
    api.kernel_status()
    xd, wd = x.cpu().to(torch.float64).numpy(), w.cpu().to(torch.float64).numpy()
    g_, u = O.linear(xd, wd[:F]), O.linear(xd, wd[F:])
    ref = O.silu(g_) * u
    eg = 1e-4 * (np.abs(xd) @ np.abs(wd[:F]).T) + 1e-6
    eu = 1e-4 * (np.abs(xd) @ np.abs(wd[F:]).T) + 1e-6
    bound = 2.0 ** -8 * np.abs(ref) + 1.1 * np.abs(u) * eg + np.abs(O.silu(g_)) * eu + 1e-6
    assert (np.abs(h.cpu().to(torch.float64).numpy() - ref) <= bound).all()
