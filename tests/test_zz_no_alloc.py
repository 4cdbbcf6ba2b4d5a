"""The allocation-free LM-head entry point (lopa_lmhead_argmax_static).

Callers that cannot allocate device memory - code under a caller-owned memory pool, a
loop that must never enter an allocator, or a host that only hands out fixed buffers -
use this variant, whose workspace is a fixed array inside the library.  It must give the
same greedy tokens and max-probabilities as lopa_lmhead_argmax (which takes a workspace
from the caller), call after call, and refuse requests that do not fit its array.

This file is collected last on purpose, so a run that stops at the first failure has
already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from diffusion_lookahead_decoding_gb300 import _lib as L
from tests.gpu_util import build_lib

pytestmark = pytest.mark.gpu


def _static_call(lib, h, w, scale, mask):
    rows, d = h.shape
    am = torch.empty(rows, dtype=torch.int32, device=h.device)
    mp = torch.empty(rows, dtype=torch.float32, device=h.device)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.lopa_lmhead_argmax_static(h.data_ptr(), w.data_ptr(), rows, d, w.shape[0], scale,
                                       mask, am.data_ptr(), mp.data_ptr(), stream)
    L.check(rc)
    torch.cuda.synchronize()
    return am.cpu().numpy(), mp.cpu().numpy()


@pytest.mark.parametrize("rows,d,V", [(256, 3584, 152064), (37, 1024, 32768)])
def test_static_scratch_lmhead_matches_workspace_version(rows, d, V):
    from diffusion_lookahead_decoding_gb300 import api
    build_lib()
    lib = L.load()
    g = torch.Generator().manual_seed(11)
    h = torch.randn(rows, d, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16).cuda()
    am_ref, mp_ref = api.lmhead_argmax(h, w, 20.0, 0)
    am_ref, mp_ref = am_ref.cpu().numpy(), mp_ref.cpu().numpy()
    for _ in range(2):  # two calls in a row share the array
        am, mp = _static_call(lib, h, w, 20.0, 0)
        np.testing.assert_array_equal(am, am_ref)
        np.testing.assert_allclose(mp, mp_ref, rtol=0, atol=1e-6)


def test_static_scratch_rejects_requests_beyond_its_size():
    build_lib()
    lib = L.load()
    rows, d, V = 1024, 64, 152064  # 1024 * 594 * 12 bytes > 4 MiB
    h = torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(V, d, dtype=torch.bfloat16, device="cuda")
    am = torch.empty(rows, dtype=torch.int32, device="cuda")
    mp = torch.empty(rows, dtype=torch.float32, device="cuda")
    rc = lib.lopa_lmhead_argmax_static(h.data_ptr(), w.data_ptr(), rows, d, V, 20.0, 0,
                                       am.data_ptr(), mp.data_ptr(), None)
    assert rc == L.ERR_INVALID_ARG
    assert b"exceeds" in lib.lopa_last_error(None)
