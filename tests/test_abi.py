"""The C-ABI library loads, exports every symbol its header declares, and rejects bad
arguments on the host before touching a GPU.  Runs without a GPU."""
import ctypes as C
import os
import re

import pytest

from diffusion_lookahead_decoding_gb300 import _lib as L
from diffusion_lookahead_decoding_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "lopa.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lopa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("lopa_init_model", "lopa_prefill", "lopa_step", "lopa_decode",
                 "lopa_last_error", "lopa_free"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.SIGNATURES, f"binding lacks {n}"
    assert lib.lopa_version() >= 100


def test_struct_layouts_match_header_sizes(lib):
    # lopa_step_result: 7 ints + 16 floats + 2*64 ints
    assert C.sizeof(L.StepResult) == 4 * (7 + 16 + 128)
    assert C.sizeof(L.ModelConfig) == 4 * 12
    assert C.sizeof(L.DecodeConfig) == 16


def test_host_side_argument_errors_without_gpu(lib):
    out = C.c_void_p()
    rc = lib.lopa_init_model(None, None, None, None, C.byref(out))
    assert rc == L.ERR_INVALID_ARG and not out.value
    assert b"null" in lib.lopa_last_error(None)
    mc = L.ModelConfig(2, 128, 4, 4, 48, 512, 1024, 0, 128, 1e4, 1e-6, 20.0)  # head_dim 48
    dc = L.DecodeConfig(16, 3, 0.9, 32)
    w = L.Weights()
    rc = lib.lopa_init_model(C.byref(mc), C.byref(w), C.byref(dc), None, C.byref(out))
    assert rc == L.ERR_UNSUPPORTED
    mc.head_dim = 32
    dc.block = 24  # not a multiple of 16
    rc = lib.lopa_init_model(C.byref(mc), C.byref(w), C.byref(dc), None, C.byref(out))
    assert rc == L.ERR_UNSUPPORTED
    dc.block, dc.k = 16, 16  # too many branches
    assert lib.lopa_init_model(C.byref(mc), C.byref(w), C.byref(dc), None, C.byref(out)) == L.ERR_INVALID_ARG
    dc.k, dc.max_prompt = 3, 200  # prompt + block beyond max_seq
    assert lib.lopa_init_model(C.byref(mc), C.byref(w), C.byref(dc), None, C.byref(out)) == L.ERR_INVALID_ARG
    assert lib.lopa_linear_accumulate(None, None, None, 1, 128, 64, None) == L.ERR_INVALID_ARG
    assert lib.lopa_prefill(None, None, 0) == L.ERR_INVALID_ARG
    assert lib.lopa_step(None, None) == L.ERR_INVALID_ARG
    assert lib.lopa_lmhead_workspace_bytes(256, 152064) == 594 * 256 * 12 + 256
    assert lib.lopa_lmhead_workspace_bytes(0, 10) == 0
