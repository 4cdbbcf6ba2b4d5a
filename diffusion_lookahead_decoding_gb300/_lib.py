"""ctypes binding of liblopa.so (declarations mirror include/lopa.h).

Argument marshalling only: every step of the decoding path runs in the library's
CUDA kernels.  Importing this module fails loudly when the library is not built.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblopa.so")

MAX_BRANCHES = 16
MAX_BLOCK = 64

OK, ERR_INVALID_ARG, ERR_BAD_STATE, ERR_CUDA, ERR_OOM, ERR_DEVICE_TIMEOUT, ERR_UNSUPPORTED = (
    0, -1, -2, -3, -4, -5, -6)
ERROR_NAMES = {ERR_INVALID_ARG: "INVALID_ARG", ERR_BAD_STATE: "BAD_STATE", ERR_CUDA: "CUDA",
               ERR_OOM: "OOM", ERR_DEVICE_TIMEOUT: "DEVICE_TIMEOUT",
               ERR_UNSUPPORTED: "UNSUPPORTED"}


class ModelConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("d_model", C.c_int), ("n_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("mask_id", C.c_int), ("max_seq", C.c_int),
                ("rope_base", C.c_float), ("rms_eps", C.c_float), ("logit_scale", C.c_float),
                ("weight_format", C.c_int)]


WEIGHTS_BF16, WEIGHTS_E4M3 = 0, 1
WEIGHT_FORMATS = {"bf16": WEIGHTS_BF16, "e4m3": WEIGHTS_E4M3}


LAYER_WEIGHTS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p)] + [
        (name, C.POINTER(C.c_void_p)) for name in LAYER_WEIGHTS]


class DecodeConfig(C.Structure):
    _fields_ = [("block", C.c_int), ("k", C.c_int), ("tau", C.c_float), ("max_prompt", C.c_int)]


class StepResult(C.Structure):
    _fields_ = [("winner", C.c_int), ("n_filled", C.c_int), ("block_done", C.c_int),
                ("n_valid_branches", C.c_int), ("forwards", C.c_int), ("prefix_len", C.c_int),
                ("device_error", C.c_int), ("conf", C.c_float * MAX_BRANCHES),
                ("filled_pos", C.c_int * MAX_BLOCK), ("filled_tok", C.c_int * MAX_BLOCK)]


class Stats(C.Structure):
    _fields_ = [("tokens", C.c_longlong), ("forwards", C.c_longlong), ("steps", C.c_longlong),
                ("blocks", C.c_longlong), ("seconds", C.c_double)]


# name -> (restype, argtypes); every symbol declared in include/lopa.h
SIGNATURES = {
    "lopa_version": (C.c_int, []),
    "lopa_last_error": (C.c_char_p, [C.c_void_p]),
    "lopa_init_model": (C.c_int, [C.POINTER(ModelConfig), C.POINTER(Weights),
                                  C.POINTER(DecodeConfig), C.c_void_p, C.POINTER(C.c_void_p)]),
    "lopa_prefill": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.c_int]),
    "lopa_step": (C.c_int, [C.c_void_p, C.POINTER(StepResult)]),
    "lopa_decode": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(C.c_int32), C.POINTER(Stats)]),
    "lopa_free": (None, [C.c_void_p]),
    "lopa_get_block_state": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32),
                                       C.POINTER(C.c_float), C.POINTER(C.c_int)]),
    "lopa_set_block_state": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32),
                                       C.POINTER(C.c_float)]),
    "lopa_verify_forward": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.c_int,
                                      C.POINTER(C.c_int32), C.POINTER(C.c_float),
                                      C.POINTER(C.c_float)]),
    "lopa_read_kv": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.POINTER(C.c_uint16),
                               C.POINTER(C.c_uint16)]),
    "lopa_rewind": (C.c_int, [C.c_void_p, C.c_int]),
    "lopa_read_branch_kv": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.POINTER(C.c_uint16),
                                      C.POINTER(C.c_uint16)]),
    "lopa_time_gemm": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.POINTER(C.c_float)]),
    "lopa_time_forward": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.POINTER(C.c_float),
                                    C.POINTER(C.c_float)]),
    "lopa_linear_accumulate": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                         C.c_int, C.c_void_p]),
    "lopa_swiglu": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                              C.c_void_p]),
    "lopa_quantize_e4m3": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                                     C.c_void_p]),
    "lopa_linear_accumulate_e4m3": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                              C.c_int, C.c_int, C.c_int, C.c_void_p]),
    "lopa_lmhead_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int]),
    "lopa_lmhead_argmax": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                     C.c_float, C.c_int, C.c_void_p, C.c_size_t, C.c_void_p,
                                     C.c_void_p, C.c_void_p]),
    "lopa_lmhead_argmax_static": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                            C.c_float, C.c_int, C.c_void_p, C.c_void_p,
                                            C.c_void_p]),
    "lopa_branch_attention": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                        C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                        C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "lopa_kernel_status": (C.c_int, [C.c_void_p]),
    "lopa_set_wait_limit_ns": (C.c_int, [C.c_ulonglong]),
    "lopa_debug_set_device_error": (C.c_int, [C.c_void_p, C.c_int]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Loads liblopa.so and declares its signatures.  Raises if it is missing: there
    is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"LoPA CUDA library not found at {path}; build it with "
                           "diffusion_lookahead_decoding_gb300.build.build()")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


class LopaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def check(rc: int, ctx=None):
    if rc != OK:
        msg = load().lopa_last_error(ctx)
        raise LopaError(rc, msg.decode() if msg else "")
