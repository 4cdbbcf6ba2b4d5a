"""Python face of the LoPA library: device memory and streams come from torch, every
computation runs in liblopa.so (see include/lopa.h for the contract of each call)."""
from __future__ import annotations

import ctypes as C
import dataclasses

import numpy as np
import torch

from . import _lib as L


def _i32p(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


def _f32p(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_float))


@dataclasses.dataclass
class StepOutcome:
    winner: int
    n_filled: int
    block_done: bool
    n_valid_branches: int
    forwards: int
    prefix_len: int
    conf: np.ndarray
    filled_pos: np.ndarray
    filled_tok: np.ndarray


def upload_weights(shape, weights: dict, device="cuda") -> dict:
    """Moves generated CPU weights (bf16, nn.Linear layout) to the device, one tensor per
    matrix as lopa_weights takes them."""
    bf = torch.bfloat16
    names = ["embed", "lm_head", "final_norm"] + [f"{n}.{l}" for l in range(shape.n_layers)
                                                  for n in L.LAYER_WEIGHTS]
    return {n: weights[n].to(device=device, dtype=bf).contiguous() for n in names}


class LopaDecoder:
    """One decoding context: static KV cache, branch scratch, state, captured graphs."""

    def __init__(self, shape, dev_weights: dict, block: int, k: int, tau: float,
                 max_prompt: int, max_seq: int, stream: torch.cuda.Stream | None = None,
                 weight_format: str = "bf16"):
        self.lib = L.load()
        self.shape = shape
        self.block = block
        self.k = k
        self.w = dev_weights  # keep the borrowed tensors alive
        self.stream = stream or torch.cuda.Stream()
        mc = L.ModelConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                           shape.head_dim, shape.ffn, shape.vocab, shape.mask_id, max_seq,
                           shape.rope_base, shape.rms_eps, shape.logit_scale,
                           L.WEIGHT_FORMATS[weight_format])
        self.weight_format = weight_format
        n = shape.n_layers
        arr = lambda key: (C.c_void_p * n)(*[dev_weights[f"{key}.{l}"].data_ptr() for l in range(n)])
        self._arrays = {k_: arr(k_) for k_ in L.LAYER_WEIGHTS}
        cast = lambda a: C.cast(a, C.POINTER(C.c_void_p))
        w = L.Weights(dev_weights["embed"].data_ptr(), dev_weights["lm_head"].data_ptr(),
                      dev_weights["final_norm"].data_ptr(),
                      *[cast(self._arrays[k_]) for k_ in L.LAYER_WEIGHTS])
        dc = L.DecodeConfig(block, k, tau, max_prompt)
        ctx = C.c_void_p()
        torch.cuda.synchronize()
        L.check(self.lib.lopa_init_model(C.byref(mc), C.byref(w), C.byref(dc),
                                         C.c_void_p(self.stream.cuda_stream), C.byref(ctx)))
        self.ctx = ctx

    # -- decoding -------------------------------------------------------------------
    def prefill(self, prompt: np.ndarray):
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        L.check(self.lib.lopa_prefill(self.ctx, _i32p(p), len(p)), self.ctx)

    def step(self) -> StepOutcome:
        r = L.StepResult()
        L.check(self.lib.lopa_step(self.ctx, C.byref(r)), self.ctx)
        nf = r.n_filled
        return StepOutcome(r.winner, nf, bool(r.block_done), r.n_valid_branches, r.forwards,
                           r.prefix_len, np.array(r.conf[:]), np.array(r.filled_pos[:nf]),
                           np.array(r.filled_tok[:nf]))

    def decode(self, gen_len: int):
        out = np.zeros(gen_len, dtype=np.int32)
        st = L.Stats()
        L.check(self.lib.lopa_decode(self.ctx, gen_len, _i32p(out), C.byref(st)), self.ctx)
        return out, {"tokens": st.tokens, "forwards": st.forwards, "steps": st.steps,
                     "blocks": st.blocks, "seconds": st.seconds}

    def rewind(self, pos: int):
        L.check(self.lib.lopa_rewind(self.ctx, pos), self.ctx)

    def time_gemm(self, kind: int, iters: int) -> float:
        ms = C.c_float()
        L.check(self.lib.lopa_time_gemm(self.ctx, kind, iters, C.byref(ms)), self.ctx)
        return ms.value

    def time_forward(self, kind: int, iters: int):
        """(median, mean) ms per launch of the forward-only graph: kind 1 = verification
        forward of all branches, 0 = block-start forward."""
        med, mean = C.c_float(), C.c_float()
        L.check(self.lib.lopa_time_forward(self.ctx, kind, iters, C.byref(med), C.byref(mean)),
                self.ctx)
        return med.value, mean.value

    # -- inspection -----------------------------------------------------------------
    def get_block_state(self):
        B = self.block
        tok = np.zeros(B, np.int32)
        am = np.zeros(B, np.int32)
        mp = np.zeros(B, np.float32)
        P = C.c_int()
        L.check(self.lib.lopa_get_block_state(self.ctx, _i32p(tok), _i32p(am), _f32p(mp),
                                              C.byref(P)), self.ctx)
        return tok, am, mp, P.value

    def set_block_state(self, tok, am, mp):
        tok = np.ascontiguousarray(tok, np.int32)
        am = np.ascontiguousarray(am, np.int32)
        mp = np.ascontiguousarray(mp, np.float32)
        L.check(self.lib.lopa_set_block_state(self.ctx, _i32p(tok), _i32p(am), _f32p(mp)),
                self.ctx)

    def verify_forward(self, branches: np.ndarray, want_hidden=False):
        br = np.ascontiguousarray(branches, np.int32)
        nb = br.shape[0]
        am = np.zeros(br.shape, np.int32)
        mp = np.zeros(br.shape, np.float32)
        hid = np.zeros((nb, self.block, self.shape.d_model), np.float32) if want_hidden else None
        L.check(self.lib.lopa_verify_forward(
            self.ctx, _i32p(br), nb, _i32p(am), _f32p(mp),
            _f32p(hid) if want_hidden else None), self.ctx)
        return am, mp, hid

    def read_kv(self, layer: int, pos0: int, n: int):
        shp = (n, self.shape.n_kv_heads, self.shape.head_dim)
        k = np.zeros(shp, np.uint16)
        v = np.zeros(shp, np.uint16)
        L.check(self.lib.lopa_read_kv(self.ctx, layer, pos0, n,
                                      k.ctypes.data_as(C.POINTER(C.c_uint16)),
                                      v.ctypes.data_as(C.POINTER(C.c_uint16))), self.ctx)
        return bf16_words_to_f64(k), bf16_words_to_f64(v)

    def read_branch_kv(self, layer: int, branch: int):
        shp = (self.block, self.shape.n_kv_heads, self.shape.head_dim)
        k = np.zeros(shp, np.uint16)
        v = np.zeros(shp, np.uint16)
        L.check(self.lib.lopa_read_branch_kv(self.ctx, layer, branch,
                                             k.ctypes.data_as(C.POINTER(C.c_uint16)),
                                             v.ctypes.data_as(C.POINTER(C.c_uint16))), self.ctx)
        return bf16_words_to_f64(k), bf16_words_to_f64(v)

    def debug_set_device_error(self, code: int):
        """Test hook: plants `code` in the context's device error word."""
        L.check(self.lib.lopa_debug_set_device_error(self.ctx, code), self.ctx)

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.lopa_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bf16_words_to_f64(words: np.ndarray) -> np.ndarray:
    return (words.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# -- kernel-level calls (device tensors, current torch stream) ---------------------------
def _stream_ptr():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def kernel_status():
    """Synchronizes the current stream; raises LopaError(DEVICE_TIMEOUT) when a device-side
    wait of a kernel-level call gave up since the last check."""
    L.check(L.load().lopa_kernel_status(_stream_ptr()))


def set_wait_limit_ns(ns: int):
    """Test hook: device-side wait limit of later kernel-level calls (0 = default)."""
    L.check(L.load().lopa_set_wait_limit_ns(int(ns)))


def linear_accumulate(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor):
    """y += x @ w.T  (x [T,K] bf16, w [N,K] bf16, y [T,N] fp32, all contiguous on cuda)."""
    T, K = x.shape
    N = w.shape[0]
    assert y.shape == (T, N) and y.dtype == torch.float32
    L.check(L.load().lopa_linear_accumulate(x.data_ptr(), w.data_ptr(), y.data_ptr(), T, N, K,
                                            _stream_ptr()))
    return y


def swiglu(x: torch.Tensor, w: torch.Tensor, h: torch.Tensor = None):
    """h = bf16(silu(x @ w[:F].T) * (x @ w[F:].T))  (x [T,K] bf16, w [2F,K] bf16 with the gate
    rows first, h [T,F] bf16; all contiguous on cuda)."""
    T, K = x.shape
    F = w.shape[0] // 2
    if h is None:
        h = torch.empty((T, F), dtype=torch.bfloat16, device=x.device)
    assert h.shape == (T, F) and h.dtype == torch.bfloat16 and w.shape == (2 * F, K)
    L.check(L.load().lopa_swiglu(x.data_ptr(), w.data_ptr(), h.data_ptr(), T, F, K, _stream_ptr()))
    return h


def quantize_e4m3(w: torch.Tensor):
    """Per-row E4M3 codes [N,K] (uint8) and float32 scales [N] of a bf16 weight [N,K]."""
    N, K = w.shape
    codes = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    scales = torch.empty(N, dtype=torch.float32, device=w.device)
    L.check(L.load().lopa_quantize_e4m3(w.data_ptr(), N, K, codes.data_ptr(), scales.data_ptr(),
                                        _stream_ptr()))
    return codes, scales


def linear_accumulate_e4m3(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                           y: torch.Tensor):
    """y += x @ (scales[:, None] * codes).T with E4M3 codes [N,K] (uint8) from quantize_e4m3."""
    T, K = x.shape
    N = codes.shape[0]
    assert y.shape == (T, N) and y.dtype == torch.float32 and codes.dtype == torch.uint8
    L.check(L.load().lopa_linear_accumulate_e4m3(x.data_ptr(), codes.data_ptr(), scales.data_ptr(),
                                                 y.data_ptr(), T, N, K, _stream_ptr()))
    return y


def lmhead_argmax(hidden: torch.Tensor, lm_head: torch.Tensor, logit_scale: float, mask_id: int):
    rows, d = hidden.shape
    V = lm_head.shape[0]
    lib = L.load()
    ws = torch.empty(lib.lopa_lmhead_workspace_bytes(rows, V), dtype=torch.uint8,
                     device=hidden.device)
    am = torch.empty(rows, dtype=torch.int32, device=hidden.device)
    mp = torch.empty(rows, dtype=torch.float32, device=hidden.device)
    L.check(lib.lopa_lmhead_argmax(hidden.data_ptr(), lm_head.data_ptr(), rows, d, V,
                                   logit_scale, mask_id, ws.data_ptr(), ws.numel(),
                                   am.data_ptr(), mp.data_ptr(), _stream_ptr()))
    return am, mp


def attention_layouts(q, k_prefix, v_prefix, k_block, v_block):
    """Rearranges natural-layout attention inputs - q [nb*B, H, dh], k/v_prefix [P, Hk, dh],
    k/v_block [nb, B, Hk, dh] (bf16, cuda) - into the library's layouts (group-major q,
    values transposed; torch copies only) and allocates the output.  Returns the argument
    pack for branch_attention_call."""
    nb, B, Hk, dh = k_block.shape
    H = q.shape[1]
    G = H // Hk
    P = k_prefix.shape[0]
    qg = q.reshape(nb * B, Hk, G, dh).permute(1, 0, 2, 3).contiguous()
    ld = max(8, (P + 7) // 8 * 8)
    vtp = torch.zeros(Hk * dh, ld, dtype=torch.bfloat16, device=q.device)
    if P:
        vtp[:, :P] = v_prefix.reshape(P, Hk * dh).t()
    vtb = v_block.reshape(nb * B, Hk * dh).t().contiguous()
    kp, kb = k_prefix.contiguous(), k_block.contiguous()
    out = torch.empty(nb * B, H * dh, dtype=torch.bfloat16, device=q.device)
    return dict(q=qg, kp=kp, vtp=vtp, P=P, ld=ld, kb=kb, vtb=vtb, nb=nb, B=B, H=H, Hk=Hk,
                dh=dh, out=out)


def branch_attention_call(a: dict):
    """One lopa_branch_attention launch on an argument pack from attention_layouts;
    returns its output tensor [nb*B, H*dh]."""
    P = a["P"]
    L.check(L.load().lopa_branch_attention(
        a["q"].data_ptr(), a["kp"].data_ptr() if P else None, a["vtp"].data_ptr() if P else None,
        P, a["ld"], a["kb"].data_ptr(), a["vtb"].data_ptr(), a["nb"], a["B"], a["H"], a["Hk"],
        a["dh"], a["out"].data_ptr(), _stream_ptr()))
    return a["out"]


def branch_attention(q, k_prefix, v_prefix, k_block, v_block):
    """Branch-isolated attention on natural layouts (see attention_layouts).  Returns out
    [nb*B, H*dh]."""
    return branch_attention_call(attention_layouts(q, k_prefix, v_prefix, k_block, v_block))
