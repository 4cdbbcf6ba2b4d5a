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
    assert C.sizeof(L.ModelConfig) == 4 * 13
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
    assert lib.lopa_swiglu(None, None, None, 1, 128, 64, None) == L.ERR_INVALID_ARG
    assert lib.lopa_swiglu(4096, 4096, 4096, 1, 100, 64, None) == L.ERR_UNSUPPORTED  # F % 128
    assert lib.lopa_linear_accumulate_e4m3(None, None, None, None, 1, 128, 64, None) == L.ERR_INVALID_ARG
    assert lib.lopa_quantize_e4m3(None, 1, 64, None, None, None) == L.ERR_INVALID_ARG
    assert lib.lopa_quantize_e4m3(4096, 1, 60, 4096, 4096, None) == L.ERR_INVALID_ARG  # K % 64
    assert lib.lopa_prefill(None, None, 0) == L.ERR_INVALID_ARG
    assert lib.lopa_step(None, None) == L.ERR_INVALID_ARG
    assert lib.lopa_lmhead_workspace_bytes(256, 152064) == 594 * 256 * 12 + 256
    assert lib.lopa_lmhead_workspace_bytes(0, 10) == 0


def _cfgs():
    mc = L.ModelConfig(2, 128, 4, 4, 32, 512, 1024, 0, 128, 1e4, 1e-6, 20.0)
    dc = L.DecodeConfig(16, 3, 0.9, 32)
    return mc, dc


@pytest.mark.parametrize("field,value,code", [
    ("d_model", 4224, "UNSUPPORTED"),      # above the 4096 the fused kernels hold
    ("ffn", 576, "UNSUPPORTED"),           # not a multiple of 128
    ("n_heads", 6, "INVALID_ARG"),         # not a multiple of n_kv_heads (4)
    ("n_layers", 0, "INVALID_ARG"),
    ("mask_id", 1024, "INVALID_ARG"),      # outside the vocabulary
    ("rms_eps", -1e-6, "INVALID_ARG"),
    ("rope_base", 0.0, "INVALID_ARG"),
    ("logit_scale", float("inf"), "INVALID_ARG"),
    ("block", 80, "UNSUPPORTED"),          # above the 64 of a block's state
    ("k", -1, "INVALID_ARG"),
    ("max_prompt", 0, "INVALID_ARG"),
    ("tau", float("nan"), "INVALID_ARG"),
    ("weight_format", 2, "INVALID_ARG"),   # neither bf16 (0) nor E4M3 (1)
])
def test_config_validation_without_gpu(lib, field, value, code):
    """Every configuration the kernels do not implement is refused on the host, before
    any CUDA call, with a message and no context."""
    mc, dc = _cfgs()
    setattr(mc if hasattr(mc, field) else dc, field, value)
    out = C.c_void_p()
    w = L.Weights()
    rc = lib.lopa_init_model(C.byref(mc), C.byref(w), C.byref(dc), None, C.byref(out))
    assert rc == getattr(L, "ERR_" + code), (field, rc)
    assert not out.value
    assert lib.lopa_last_error(None)


@pytest.mark.parametrize("case", ["null_q", "head_dim", "block", "prefix_ld", "heads"])
def test_branch_attention_host_checks_without_gpu(lib, case):
    """The standalone attention refuses bad pointers and shapes before launching."""
    p = 4096  # a 16-byte aligned stand-in address: every case below is refused first
    args = dict(q=p, kp=p, vtp=p, P=64, ld=64, kb=p, vtb=p, nb=2, B=32, H=8, Hk=2, dh=128, out=p)
    want = L.ERR_INVALID_ARG
    if case == "null_q":
        args["q"] = None
    elif case == "head_dim":
        args["dh"], want = 96, L.ERR_UNSUPPORTED
    elif case == "block":
        args["B"] = 24
    elif case == "prefix_ld":
        args["ld"] = 60  # below the prefix length
    else:
        args["H"] = 7  # not a multiple of Hk
    rc = lib.lopa_branch_attention(args["q"], args["kp"], args["vtp"], args["P"], args["ld"],
                                   args["kb"], args["vtb"], args["nb"], args["B"], args["H"],
                                   args["Hk"], args["dh"], args["out"], None)
    assert rc == want, (case, rc)
