"""Python binding of libdg.so -- argument marshalling only.

Every function here forwards to the C ABI declared in include/dg.h with
ctypes: tensors are passed as device pointers (``tensor.data_ptr()``), the
stream as the raw cudaStream_t of the current torch stream.  No step of the
denoising path runs in Python or PyTorch; if the library is missing, the
first call raises (there is no fallback).

PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdg.so")

DG_OK = 0
STATUS_NAMES = {0: "DG_OK", 1: "DG_ERR_INVALID_ARG", 2: "DG_ERR_UNSUPPORTED",
                3: "DG_ERR_ALIGNMENT", 4: "DG_ERR_WORKSPACE", 5: "DG_ERR_CUDA",
                6: "DG_ERR_TIMEOUT", 7: "DG_ERR_DEVICE"}

# Functions include/dg.h declares (checked by the CPU test-suite).
EXPORTED = ["dg_status_string", "dg_version", "dg_set_device_checks", "dg_device_checks",
            "dg_read_device_status",
            "dg_canvas_attn_workspace", "dg_canvas_attn",
            "dg_encoder_append_workspace", "dg_encoder_append",
            "dg_denoise_step_workspace", "dg_denoise_step", "dg_denoise_step_noalloc",
            "dg_noalloc_read_device_status",
            "dg_generate_block_workspace", "dg_generate_block",
            "dg_sampler_workspace", "dg_sampler_from_logits", "dg_accept_renoise",
            "dg_lm_head_fold", "dg_kernel_launches", "dg_lm_head_plan", "dg_gumbel_fill",
            "dg_logf_eval", "dg_quantize_rows_e4m3", "dg_quantize_weight_e4m3",
            "dg_denoise_step_fp8_workspace", "dg_denoise_step_fp8", "dg_lm_head_fold_fp8",
            "dg_wait_timeout_probe", "dg_denoise_step_sc_workspace", "dg_denoise_step_sc",
            "dg_lm_head_fold_sc", "dg_moe_ffn_workspace", "dg_moe_ffn",
            "dg_generate_block_fn", "dg_hidden_from_steps", "dg_hidden_embed_add",
            "dg_canvas_step_workspace", "dg_canvas_step",
            "dg_lm_weight_packed_bytes", "dg_pack_lm_weight",
            "dg_canvas_step_fp8_workspace", "dg_canvas_step_fp8",
            "dg_canvas_step_sc_workspace", "dg_canvas_step_sc", "dg_canvas_step_plan"]


class DgError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%s)" % (what, STATUS_NAMES.get(code, code),
                                                 _lib().dg_status_string(code).decode()))


class StepParams(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("L", ctypes.c_int), ("d", ctypes.c_int), ("V", ctypes.c_int),
                ("temperature", ctypes.c_double), ("entropy_bound", ctypes.c_float),
                ("stop_threshold", ctypes.c_float), ("step", ctypes.c_int),
                ("seed", ctypes.c_uint64), ("w_layout", ctypes.c_int)]

W_ROWMAJOR = 0   # the LM-head weight as [d, V]
W_PACKED = 1     # as pack_lm_weight writes it


class StepIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("canvas", "prev_argmax", "argmax", "sample", "entropy", "accepted",
                 "n_accepted", "mean_entropy", "stop")]


class MoeParams(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("d", ctypes.c_int), ("f", ctypes.c_int),
                ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int)]


class BlockParams(ctypes.Structure):
    _fields_ = [("max_steps", ctypes.c_int), ("t_start", ctypes.c_double),
                ("t_end", ctypes.c_double), ("hidden_step_stride", ctypes.c_int64)]


class BlockIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("canvas", "argmax", "steps_taken", "mean_entropy", "n_accepted_hist")]


class CanvasStepPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("attn_reserved_sms", "attn_pair", "attn_ctas", "attn_splits", "attn_key_tiles",
                 "attn_key_tile", "lm_kind", "lm_bn", "lm_ctas", "lm_tiles",
                 "lm_epilogue_warps", "lm_sms")]


_L = None


def _lib():
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libdg.so is not built: run __graft_entry__.build() "
                               "(block_diffusion_decoding_gb300/build.py)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u32, u64, sz, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32,
                                      ctypes.c_uint64, ctypes.c_size_t, ctypes.c_float)
        sp, si, bp, bi = (ctypes.POINTER(StepParams), ctypes.POINTER(StepIO),
                          ctypes.POINTER(BlockParams), ctypes.POINTER(BlockIO))
        ip = ctypes.POINTER(ctypes.c_int)
        sig = {
            "dg_status_string": ([i32], ctypes.c_char_p),
            "dg_version": ([], i32),
            "dg_set_device_checks": ([i32], i32),
            "dg_device_checks": ([], i32),
            "dg_read_device_status": ([vp, ctypes.POINTER(ctypes.c_int), i32, vp], i32),
            "dg_canvas_attn_workspace": ([i32] * 6, sz),
            "dg_canvas_attn": ([vp] * 6 + [i32] * 6 + [f32, vp, sz, vp], i32),
            "dg_encoder_append_workspace": ([i32] * 6, sz),
            "dg_encoder_append": ([vp, vp, vp, i32, i32, vp, vp, vp] + [i32] * 5
                                  + [f32, vp, sz, vp], i32),
            "dg_denoise_step_workspace": ([sp], sz),
            "dg_denoise_step": ([vp, vp, sp, si, vp, sz, vp], i32),
            "dg_denoise_step_noalloc": ([vp, vp, sp, si, vp], i32),
            "dg_noalloc_read_device_status": ([ctypes.POINTER(ctypes.c_int), i32, vp], i32),
            "dg_generate_block_workspace": ([sp, bp], sz),
            "dg_generate_block": ([vp, vp, sp, bp, bi, vp, sz, vp], i32),
            "dg_sampler_workspace": ([sp], sz),
            "dg_sampler_from_logits": ([vp, sp, si, vp, sz, vp], i32),
            "dg_accept_renoise": ([vp, vp, vp, sp, si, vp, sz, vp], i32),
            "dg_lm_head_fold": ([vp, vp, sp, vp, sz, vp], i32),
            "dg_kernel_launches": ([], u64),
            "dg_lm_head_plan": ([i32, i32, i32, ip, ip, ip, ip], i32),
            "dg_gumbel_fill": ([u64, u32, u32, u32, i32, vp, vp], i32),
            "dg_logf_eval": ([vp, vp, i32, vp], i32),
            "dg_quantize_rows_e4m3": ([vp, ctypes.c_int64, i32, vp, vp, vp], i32),
            "dg_quantize_weight_e4m3": ([vp, i32, i32, vp, vp, vp], i32),
            "dg_lm_weight_packed_bytes": ([i32, i32], sz),
            "dg_pack_lm_weight": ([vp, i32, i32, vp, vp], i32),
            "dg_denoise_step_fp8_workspace": ([sp], sz),
            "dg_denoise_step_fp8": ([vp, vp, vp, sp, si, vp, sz, vp], i32),
            "dg_lm_head_fold_fp8": ([vp, vp, vp, sp, vp, sz, vp], i32),
            "dg_wait_timeout_probe": ([vp, sz, u64, vp], i32),
            "dg_denoise_step_sc_workspace": ([sp], sz),
            "dg_denoise_step_sc": ([vp, vp, vp, sp, si, vp, vp, sz, vp], i32),
            "dg_lm_head_fold_sc": ([vp, vp, vp, sp, vp, sz, vp], i32),
            "dg_moe_ffn_workspace": ([ctypes.POINTER(MoeParams)], sz),
            "dg_moe_ffn": ([vp] * 8 + [ctypes.POINTER(MoeParams), vp, sz, vp], i32),
            "dg_generate_block_fn": ([vp, vp, vp, vp, sp, bp, bi, vp, sz, vp], i32),
            "dg_hidden_from_steps": ([vp] * 5, i32),
            "dg_hidden_embed_add": ([vp] * 5, i32),
            "dg_canvas_step_workspace": ([sp, i32, i32, i32, i32], sz),
            "dg_canvas_step": ([vp] * 6 + [i32] * 4 + [f32, vp, vp, sp, si, vp, sz, vp], i32),
            "dg_canvas_step_fp8_workspace": ([sp, i32, i32, i32, i32], sz),
            "dg_canvas_step_fp8": ([vp] * 6 + [i32] * 4 + [f32, vp, vp, vp, sp, si, vp, sz, vp],
                                   i32),
            "dg_canvas_step_sc_workspace": ([sp, i32, i32, i32, i32], sz),
            "dg_canvas_step_sc": ([vp] * 6 + [i32] * 4 + [f32, vp, vp, vp, sp, si, vp, vp, sz, vp],
                                  i32),
            "dg_canvas_step_plan": ([sp] + [i32] * 5 + [ctypes.POINTER(CanvasStepPlan)], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _L = L
    return _L


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    return _lib()


# Every entry point has its argtypes set, so device pointers and streams go
# through as plain integers (no ctypes object per argument).
def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(rc: int, what: str):
    if rc != DG_OK:
        raise DgError(rc, what)


# ---------------------------------------------------------------- attention
def canvas_attn_workspace(B, L, P, Hq, Hkv, D) -> int:
    return int(_lib().dg_canvas_attn_workspace(B, L, P, Hq, Hkv, D))


def canvas_attn(q, k_prefix, v_prefix, k_canvas, v_canvas, out, scale, workspace, stream=None):
    """dg_canvas_attn on bf16 tensors q/out [B,L,Hq,D], k/v prefix [B,P,Hkv,D], canvas [B,L,Hkv,D]."""
    B, L, Hq, D = q.shape
    if k_prefix is not None and k_prefix.shape[1] > 0:
        P = k_prefix.shape[1]
    else:
        P = 0
    Hkv = k_canvas.shape[2]
    rc = _lib().dg_canvas_attn(_p(q), _p(k_prefix) if P else None, _p(v_prefix) if P else None,
                               _p(k_canvas), _p(v_canvas), _p(out), B, L, P, Hq, Hkv, D,
                               float(scale), _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "dg_canvas_attn")


def encoder_append_workspace(B, L, P, Hq, Hkv, D) -> int:
    return int(_lib().dg_encoder_append_workspace(B, L, P, Hq, Hkv, D))


def encoder_append(q, k_cache, v_cache, P, k_new, v_new, out, scale, workspace, stream=None):
    """dg_encoder_append: the caches [B, P_max, Hkv, D] hold P tokens; the block's
    k_new/v_new [B, L, Hkv, D] are appended and q [B, L, Hq, D] attends causally."""
    B, L, Hq, D = q.shape
    P_max, Hkv = k_cache.shape[1], k_cache.shape[2]
    rc = _lib().dg_encoder_append(_p(q), _p(k_cache), _p(v_cache), int(P), int(P_max),
                                  _p(k_new), _p(v_new), _p(out), B, L, Hq, Hkv, D, float(scale),
                                  _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "dg_encoder_append")


# ---------------------------------------------------------------- step
def step_params(B, L, d, V, temperature, entropy_bound=0.1, stop_threshold=0.005, step=0,
                seed=0, w_layout=W_ROWMAJOR) -> StepParams:
    return StepParams(B, L, d, V, temperature, entropy_bound, stop_threshold, step, seed, w_layout)


class StepBuffers:
    """Device outputs of one step (dg_step_io) for B canvases of length L."""

    def __init__(self, B: int, L: int, device="cuda"):
        M = B * L
        i32 = dict(dtype=torch.int32, device=device)
        # what a caller reads back after a step -- canvas, argmax, stop -- is
        # one contiguous int32 block (`readback`), so one copy fetches it
        self.readback = torch.zeros(2 * M + B, **i32)
        self.canvas = self.readback[:M]
        self.argmax = self.readback[M:2 * M]
        self.stop = self.readback[2 * M:]
        self.prev_argmax = torch.full((M,), -1, **i32)
        self.sample = torch.zeros(M, **i32)
        self.entropy = torch.zeros(M, dtype=torch.float32, device=device)
        self.accepted = torch.zeros(M, dtype=torch.uint8, device=device)
        self.n_accepted = torch.zeros(B, **i32)
        self.mean_entropy = torch.zeros(B, dtype=torch.float32, device=device)

    def __setattr__(self, name, value):
        # a replaced tensor invalidates the cached dg_step_io
        object.__setattr__(self, name, value)
        if name != "_io":
            object.__setattr__(self, "_io", None)

    def io(self) -> StepIO:
        if self._io is None:
            self._io = StepIO(*[ctypes.c_void_p(getattr(self, n).data_ptr())
                                for n, _ in StepIO._fields_])
        return self._io


def denoise_step_workspace(p: StepParams) -> int:
    return int(_lib().dg_denoise_step_workspace(ctypes.byref(p)))


def denoise_step(hidden, w, p: StepParams, bufs: StepBuffers, workspace, stream=None):
    io = bufs.io()
    rc = _lib().dg_denoise_step(_p(hidden), _p(w), ctypes.byref(p), ctypes.byref(io),
                                _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "dg_denoise_step")


def canvas_step_workspace(p: StepParams, P, Hq, Hkv, D) -> int:
    return int(_lib().dg_canvas_step_workspace(ctypes.byref(p), P, Hq, Hkv, D))


def canvas_step(q, k_prefix, v_prefix, k_canvas, v_canvas, attn_out, scale, hidden, w,
                p: StepParams, bufs: StepBuffers, workspace, stream=None):
    """dg_canvas_step: the canvas attention and the denoising step in one call."""
    B, L, Hq, D = q.shape
    P = k_prefix.shape[1] if k_prefix is not None else 0
    Hkv = k_canvas.shape[2]
    io = bufs.io()
    rc = _lib().dg_canvas_step(_p(q), _p(k_prefix) if P else None, _p(v_prefix) if P else None,
                               _p(k_canvas), _p(v_canvas), _p(attn_out), P, Hq, Hkv, D,
                               float(scale), _p(hidden), _p(w), ctypes.byref(p), ctypes.byref(io),
                               _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "dg_canvas_step")


def canvas_step_fp8_workspace(p: StepParams, P, Hq, Hkv, D) -> int:
    return int(_lib().dg_canvas_step_fp8_workspace(ctypes.byref(p), P, Hq, Hkv, D))


def canvas_step_fp8(q, k_prefix, v_prefix, k_canvas, v_canvas, attn_out, scale, hidden, w8t,
                    w_scale, p: StepParams, bufs: StepBuffers, workspace, stream=None):
    """dg_canvas_step_fp8: the canvas attention beside the E4M3 denoising step."""
    B, L, Hq, D = q.shape
    P = k_prefix.shape[1] if k_prefix is not None else 0
    Hkv = k_canvas.shape[2]
    io = bufs.io()
    rc = _lib().dg_canvas_step_fp8(_p(q), _p(k_prefix) if P else None,
                                   _p(v_prefix) if P else None, _p(k_canvas), _p(v_canvas),
                                   _p(attn_out), P, Hq, Hkv, D, float(scale), _p(hidden), _p(w8t),
                                   _p(w_scale), ctypes.byref(p), ctypes.byref(io), _p(workspace),
                                   workspace.numel(), _stream(stream))
    _check(rc, "dg_canvas_step_fp8")


def canvas_step_sc_workspace(p: StepParams, P, Hq, Hkv, D) -> int:
    return int(_lib().dg_canvas_step_sc_workspace(ctypes.byref(p), P, Hq, Hkv, D))


def canvas_step_sc(q, k_prefix, v_prefix, k_canvas, v_canvas, attn_out, scale, hidden, w,
                   sc_table, p: StepParams, bufs: StepBuffers, sc_out, workspace, stream=None):
    """dg_canvas_step_sc: the canvas attention beside the self-conditioning step."""
    B, L, Hq, D = q.shape
    P = k_prefix.shape[1] if k_prefix is not None else 0
    Hkv = k_canvas.shape[2]
    io = bufs.io()
    rc = _lib().dg_canvas_step_sc(_p(q), _p(k_prefix) if P else None,
                                  _p(v_prefix) if P else None, _p(k_canvas), _p(v_canvas),
                                  _p(attn_out), P, Hq, Hkv, D, float(scale), _p(hidden), _p(w),
                                  _p(sc_table), ctypes.byref(p), ctypes.byref(io), _p(sc_out),
                                  _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "dg_canvas_step_sc")


def lm_head_fold(hidden, w, p: StepParams, workspace, stream=None):
    """The LM-head kernel of the step alone (partial states into the workspace)."""
    rc = _lib().dg_lm_head_fold(_p(hidden), _p(w), ctypes.byref(p), _p(workspace),
                                workspace.numel(), _stream(stream))
    _check(rc, "dg_lm_head_fold")


def canvas_step_plan(p: StepParams, P: int, Hq: int, Hkv: int, D: int, sms: int = 0) -> dict:
    """The launches canvas_step would make on a GPU with `sms` SMs (0: the
    current device's); with sms > 0 no device is touched."""
    out = CanvasStepPlan()
    rc = _lib().dg_canvas_step_plan(ctypes.byref(p), P, Hq, Hkv, D, sms, ctypes.byref(out))
    _check(rc, "dg_canvas_step_plan")
    return {name: getattr(out, name) for name, _ in CanvasStepPlan._fields_}


def lm_head_plan(rows: int, d: int, V: int) -> dict:
    """The LM-head launch the step would make on the current device."""
    kind, bn, ctas, epi = (ctypes.c_int(0) for _ in range(4))
    rc = _lib().dg_lm_head_plan(rows, d, V, ctypes.byref(kind), ctypes.byref(bn),
                                ctypes.byref(ctas), ctypes.byref(epi))
    _check(rc, "dg_lm_head_plan")
    # kinds 2 and 3: the 2-SM kernel (3: adjacent BN-column schedule tiles
    # fused), with 8 epilogue warps or, in lm_head_duo_wide_kernel, 16
    if kind.value >= 2:
        name = "lm_head_duo_wide_kernel" if epi.value == 16 else "lm_head_duo_kernel"
    else:
        name = "lm_head_kernel"
    return {"kernel": name, "kind": kind.value, "BN": bn.value, "ctas": ctas.value,
            "fused": kind.value == 3, "epilogue_warps": epi.value}


# ---------------------------------------------------------------- self-conditioning step
SC_DIM = 32


def denoise_step_sc_workspace(p: StepParams) -> int:
    return int(_lib().dg_denoise_step_sc_workspace(ctypes.byref(p)))


def denoise_step_sc(hidden, w, sc_table, p: StepParams, bufs: StepBuffers, sc_out, workspace,
                    stream=None):
    """dg_denoise_step_sc: sc_table [V, 32] bf16, sc_out [B*L, 32] fp32."""
    io = bufs.io()
    rc = _lib().dg_denoise_step_sc(_p(hidden), _p(w), _p(sc_table), ctypes.byref(p),
                                   ctypes.byref(io), _p(sc_out), _p(workspace), workspace.numel(),
                                   _stream(stream))
    _check(rc, "dg_denoise_step_sc")


def lm_head_fold_sc(hidden, w, sc_table, p: StepParams, workspace, stream=None):
    rc = _lib().dg_lm_head_fold_sc(_p(hidden), _p(w), _p(sc_table), ctypes.byref(p),
                                   _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "dg_lm_head_fold_sc")


# ---------------------------------------------------------------- MoE FFN
def moe_params(M, d, f, n_experts, top_k) -> MoeParams:
    return MoeParams(M, d, f, n_experts, top_k)


def moe_ffn_workspace(p: MoeParams) -> int:
    return int(_lib().dg_moe_ffn_workspace(ctypes.byref(p)))


def moe_ffn(x, w_router, w_gate, w_up, w_down, out, p: MoeParams, workspace, experts=None,
            gates=None, stream=None):
    """dg_moe_ffn: x [M, d] bf16, w_router [E, d], w_gate / w_up [E+1, f, d],
    w_down [E+1, d, f] bf16 -> out [M, d] fp32 (+ routing when given)."""
    rc = _lib().dg_moe_ffn(_p(x), _p(w_router), _p(w_gate), _p(w_up), _p(w_down), _p(out),
                           _p(experts), _p(gates), ctypes.byref(p), _p(workspace),
                           workspace.numel(), _stream(stream))
    _check(rc, "dg_moe_ffn")


# ---------------------------------------------------------------- FP8 LM head
def quantize_rows_e4m3(x, codes, scale, stream=None):
    """x [rows, cols] bf16 -> E4M3 codes (uint8, same shape) and fp32 row scales."""
    rows, cols = x.shape
    rc = _lib().dg_quantize_rows_e4m3(_p(x), rows, cols, _p(codes), _p(scale), _stream(stream))
    _check(rc, "dg_quantize_rows_e4m3")


def lm_weight_packed_bytes(d, V) -> int:
    return int(_lib().dg_lm_weight_packed_bytes(d, V))


def pack_lm_weight(w, out=None, stream=None):
    """W [d, V] bf16 -> the packed LM-head weight (a 1-D bf16 tensor of
    lm_weight_packed_bytes(d, V) bytes), for steps with w_layout=W_PACKED."""
    import torch
    if w.dim() != 2 or w.dtype != torch.bfloat16 or not w.is_contiguous():
        raise ValueError("pack_lm_weight: w must be a contiguous bf16 [d, V] tensor")
    d, V = w.shape
    if out is None:
        out = torch.empty(lm_weight_packed_bytes(d, V) // 2, dtype=w.dtype, device=w.device)
    rc = _lib().dg_pack_lm_weight(_p(w), d, V, _p(out), _stream(stream))
    _check(rc, "dg_pack_lm_weight")
    return out


def quantize_weight_e4m3(w, w8t, scale, stream=None):
    """W [d, V] bf16 -> W8t [V, d] E4M3 codes and fp32 column scales [V]."""
    d, V = w.shape
    rc = _lib().dg_quantize_weight_e4m3(_p(w), d, V, _p(w8t), _p(scale), _stream(stream))
    _check(rc, "dg_quantize_weight_e4m3")


def denoise_step_fp8_workspace(p: StepParams) -> int:
    return int(_lib().dg_denoise_step_fp8_workspace(ctypes.byref(p)))


def denoise_step_fp8(hidden, w8t, w_scale, p: StepParams, bufs: StepBuffers, workspace,
                     stream=None):
    io = bufs.io()
    rc = _lib().dg_denoise_step_fp8(_p(hidden), _p(w8t), _p(w_scale), ctypes.byref(p),
                                    ctypes.byref(io), _p(workspace), workspace.numel(),
                                    _stream(stream))
    _check(rc, "dg_denoise_step_fp8")


def lm_head_fold_fp8(hidden, w8t, w_scale, p: StepParams, workspace, stream=None):
    """Row quantisation + the FP8 LM-head kernel of the step alone."""
    rc = _lib().dg_lm_head_fold_fp8(_p(hidden), _p(w8t), _p(w_scale), ctypes.byref(p),
                                    _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "dg_lm_head_fold_fp8")


def kernel_launches() -> int:
    """Kernels this library has launched (or enqueued into a capture) so far."""
    return int(_lib().dg_kernel_launches())


def sampler_workspace(p: StepParams) -> int:
    return int(_lib().dg_sampler_workspace(ctypes.byref(p)))


def sampler_from_logits(logits, p: StepParams, bufs: StepBuffers, workspace, stream=None):
    io = bufs.io()
    rc = _lib().dg_sampler_from_logits(_p(logits), ctypes.byref(p), ctypes.byref(io),
                                       _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "dg_sampler_from_logits")


def accept_renoise(entropy, sample, argmax, p: StepParams, bufs: StepBuffers, workspace,
                   stream=None):
    io = bufs.io()
    rc = _lib().dg_accept_renoise(_p(entropy), _p(sample), _p(argmax), ctypes.byref(p),
                                  ctypes.byref(io), _p(workspace), workspace.numel(),
                                  _stream(stream))
    _check(rc, "dg_accept_renoise")


# ---------------------------------------------------------------- block loop
class BlockBuffers:
    def __init__(self, B: int, L: int, max_steps: int, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        self.canvas = torch.zeros(B * L, **i32)
        self.argmax = torch.zeros(B * L, **i32)
        self.steps_taken = torch.zeros(B, **i32)
        self.mean_entropy = torch.zeros(B, dtype=torch.float32, device=device)
        self.n_accepted_hist = torch.zeros(max_steps * B, **i32)

    def __setattr__(self, name, value):
        # a replaced tensor invalidates the cached dg_block_io
        object.__setattr__(self, name, value)
        if name != "_io":
            object.__setattr__(self, "_io", None)

    def io(self) -> BlockIO:
        if self._io is None:
            self._io = BlockIO(*[ctypes.c_void_p(getattr(self, n).data_ptr())
                                 for n, _ in BlockIO._fields_])
        return self._io


class HiddenSteps(ctypes.Structure):
    """dg_hidden_steps: the user data of dg_hidden_from_steps."""
    _fields_ = [("hidden_steps", ctypes.c_void_p), ("step_stride", ctypes.c_int64),
                ("n", ctypes.c_int64)]


class HiddenEmbed(ctypes.Structure):
    """dg_hidden_embed: the user data of dg_hidden_embed_add."""
    _fields_ = [("base", ctypes.c_void_p), ("base_step_stride", ctypes.c_int64),
                ("table", ctypes.c_void_p), ("rows", ctypes.c_int), ("d", ctypes.c_int),
                ("V", ctypes.c_int)]


# A producer written in Python: f(step_ptr, canvas_ptr, hidden_out_ptr, stream_ptr, user_ptr) -> int
HIDDEN_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                             ctypes.c_void_p, ctypes.c_void_p)


def hidden_producer(name: str) -> ctypes.c_void_p:
    """Address of a built-in producer: "from_steps" or "embed_add"."""
    fn = {"from_steps": _lib().dg_hidden_from_steps,
          "embed_add": _lib().dg_hidden_embed_add}[name]
    return ctypes.cast(fn, ctypes.c_void_p)


def generate_block_fn(producer, user, hidden_buf, w, p: StepParams, bp: BlockParams,
                      bufs: "BlockBuffers", workspace, stream=None):
    """dg_generate_block_fn: producer is hidden_producer(name) or a HIDDEN_FN
    object; user a ctypes structure (kept alive by the caller while the loop's
    graph may be rebuilt for the same arguments)."""
    io = bufs.io()
    fn = producer if isinstance(producer, ctypes.c_void_p) else ctypes.cast(producer,
                                                                             ctypes.c_void_p)
    rc = _lib().dg_generate_block_fn(fn, ctypes.cast(ctypes.byref(user), ctypes.c_void_p),
                                     _p(hidden_buf), _p(w), ctypes.byref(p), ctypes.byref(bp),
                                     ctypes.byref(io), _p(workspace), workspace.numel(),
                                     _stream(stream))
    _check(rc, "dg_generate_block_fn")


def block_params(max_steps=48, t_start=0.8, t_end=0.4, hidden_step_stride=0) -> BlockParams:
    return BlockParams(max_steps, t_start, t_end, hidden_step_stride)


def generate_block_workspace(p: StepParams, bp: BlockParams) -> int:
    return int(_lib().dg_generate_block_workspace(ctypes.byref(p), ctypes.byref(bp)))


def generate_block(hidden_steps, w, p: StepParams, bp: BlockParams, bufs: BlockBuffers,
                   workspace, stream=None):
    io = bufs.io()
    rc = _lib().dg_generate_block(_p(hidden_steps), _p(w), ctypes.byref(p), ctypes.byref(bp),
                                  ctypes.byref(io), _p(workspace), workspace.numel(),
                                  _stream(stream))
    _check(rc, "dg_generate_block")


# ---------------------------------------------------------------- checks / status
def gumbel_fill(seed, row, step, v0, n, out, stream=None):
    _check(_lib().dg_gumbel_fill(seed, row, step, v0, n, _p(out), _stream(stream)),
           "dg_gumbel_fill")


def logf_eval(x, y, stream=None):
    _check(_lib().dg_logf_eval(_p(x), _p(y), x.numel(), _stream(stream)), "dg_logf_eval")


def wait_timeout_probe(workspace, limit_ns: int, stream=None):
    """dg_wait_timeout_probe: a bounded wait that nothing completes, on purpose."""
    _check(_lib().dg_wait_timeout_probe(_p(workspace), workspace.numel(), int(limit_ns),
                                        _stream(stream)), "dg_wait_timeout_probe")


def set_device_checks(on: bool) -> None:
    """dg_set_device_checks: device-side index and finiteness checks (off by
    default); a failed check reads back as DG_ERR_DEVICE."""
    _check(_lib().dg_set_device_checks(1 if on else 0), "dg_set_device_checks")


def device_checks() -> bool:
    return bool(_lib().dg_device_checks())


def read_device_status(workspace, clear=False, stream=None) -> int:
    v = ctypes.c_int(0)
    _check(_lib().dg_read_device_status(_p(workspace), ctypes.byref(v), 1 if clear else 0,
                                        _stream(stream)), "dg_read_device_status")
    return v.value


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed byte tensor usable as a workspace."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def bf16_from_bits(bits, device="cuda") -> torch.Tensor:
    """A bf16 tensor holding the given uint16 bit patterns (numpy array)."""
    import numpy as np
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if str(device) != "cpu" else t
