"""The C ABI without a GPU: the library loads, exports every function that
include/dg.h declares, answers workspace queries, and rejects bad arguments
on the host before anything is launched."""
import ctypes
import os
import re

import pytest

import block_diffusion_decoding_gb300 as dg
from block_diffusion_decoding_gb300 import build as dgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dgbuild.build()
    return dg.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "dg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_function(lib):
    declared = _declared_functions()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(dg.EXPORTED) == declared


def test_status_strings(lib):
    for code in range(8):
        assert isinstance(lib.dg_status_string(code), bytes)
    assert lib.dg_status_string(99) == b"unknown status"
    assert lib.dg_version() >= 100


def test_struct_layouts_match_header(lib):
    # int B, L, d, V; double T; float b, thr; int step; (pad) uint64 seed; int w_layout (pad)
    assert ctypes.sizeof(dg.StepParams) == 56
    assert dg.StepParams.seed.offset == 40
    assert dg.StepParams.w_layout.offset == 48
    assert ctypes.sizeof(dg.StepIO) == 9 * 8
    assert ctypes.sizeof(dg.BlockParams) == 32
    assert ctypes.sizeof(dg.BlockIO) == 5 * 8


def test_workspace_queries(lib):
    p = dg.step_params(1, 256, 2816, 262144, 0.8)
    ws = dg.denoise_step_workspace(p)
    assert ws >= 256 + 7 * 4 * 256 * 152
    assert dg.generate_block_workspace(p, dg.block_params()) > ws
    assert dg.sampler_workspace(p) > 0
    # a long cache needs split-KV scratch
    assert dg.canvas_attn_workspace(1, 256, 32768, 4, 1, 128) > 1 << 20
    assert dg.canvas_attn_workspace(1, 16, 0, 4, 1, 128) >= 256
    # unsupported shapes answer 0
    assert dg.canvas_attn_workspace(1, 256, 256, 4, 1, 64) == 0
    assert dg.canvas_attn_workspace(1, 256, 256, 3, 2, 128) == 0
    assert dg.denoise_step_workspace(dg.step_params(1, 256, 1024, 1001, 0.8)) == 0


def _vp(x):
    return ctypes.c_void_p(x)


def test_host_validation_rejects_before_launch(lib):
    good = 1 << 20   # aligned fake addresses: never dereferenced, validation fails first
    p = dg.step_params(1, 256, 1024, 16384, 0.8)
    io = dg.StepIO(*[_vp(good + 64 * i) for i in range(9)])
    ws_sz = dg.denoise_step_workspace(p)

    def call(h, w, p_, io_, ws, n):
        return lib.dg_denoise_step(h, w, ctypes.byref(p_), ctypes.byref(io_), ws, n, None)

    assert call(None, _vp(good), p, io, _vp(good), ws_sz) == 1            # null hidden
    assert call(_vp(good + 2), _vp(good), p, io, _vp(good), ws_sz) == 3   # misaligned
    assert call(_vp(good), _vp(good), p, io, _vp(good), ws_sz - 1) == 4   # workspace too small
    assert call(_vp(good), _vp(good), p, io, None, ws_sz) == 4            # no workspace
    bad = dg.step_params(1, 256, 1000, 16384, 0.8)                         # d % 64 != 0
    assert call(_vp(good), _vp(good), bad, io, _vp(good), 1 << 30) == 2
    bad = dg.step_params(1, 256, 1024, 16384, -1.0)                        # T <= 0
    assert call(_vp(good), _vp(good), bad, io, _vp(good), 1 << 30) == 1
    bad = dg.step_params(1, 2048, 1024, 16384, 0.8)                        # L > 1024
    assert call(_vp(good), _vp(good), bad, io, _vp(good), 1 << 30) == 2
    io_missing = dg.StepIO(*([None] + [_vp(good)] * 8))
    assert call(_vp(good), _vp(good), p, io_missing, _vp(good), ws_sz) == 1

    def attn(D, Hq, Hkv, q=good, n=1 << 30):
        return lib.dg_canvas_attn(_vp(q), _vp(good), _vp(good), _vp(good), _vp(good), _vp(good),
                                  1, 256, 256, Hq, Hkv, D, 0.1, _vp(good), n, None)

    assert attn(64, 4, 1) == 2          # head dim
    assert attn(128, 6, 4) == 2         # Hq % Hkv
    assert attn(128, 12, 4) == 2        # G = 3 not a power of two
    assert attn(128, 4, 1, q=good + 8) == 3
    assert attn(128, 4, 1, n=0) == 4
    # block loop
    bio = dg.BlockIO(*[_vp(good + 64 * i) for i in range(5)])
    for bp, code in ((dg.block_params(max_steps=0), 2), (dg.block_params(t_start=0.0), 1),
                     (dg.block_params(hidden_step_stride=-1), 1)):
        assert lib.dg_generate_block(_vp(good), _vp(good), ctypes.byref(p), ctypes.byref(bp),
                                     ctypes.byref(bio), _vp(good), 1 << 30, None) == code
    # check entries
    assert lib.dg_logf_eval(None, None, -1, None) == 1
    assert lib.dg_gumbel_fill(0, 0, 0, 0, 0, None, None) == 0
    # encoder cache append: the cache must have room for the block
    def enc(P, P_max, D=128, kc=good):
        return lib.dg_encoder_append(_vp(good), _vp(kc), _vp(good), P, P_max, _vp(good), _vp(good),
                                     _vp(good), 1, 256, 4, 1, D, 0.1, _vp(good), 1 << 30, None)

    assert enc(100, 300) == 1           # P + L > P_max
    assert enc(0, 256, D=64) == 2       # head dim
    assert enc(0, 256, kc=good + 4) == 3
    # LM-head plan query: shapes the step rejects are rejected before any device call
    assert lib.dg_lm_head_plan(0, 1024, 16384, None, None, None, None) == 1
    assert lib.dg_lm_head_plan(256, 1000, 16384, None, None, None, None) == 2
    assert lib.dg_lm_head_plan(256, 1024, 16380, None, None, None, None) == 2


def test_fp8_entry_points_validate_before_launch(lib):
    good = 1 << 20
    p = dg.step_params(1, 256, 1024, 16384, 0.8)
    io = dg.StepIO(*[_vp(good + 64 * i) for i in range(9)])
    ws_sz = dg.denoise_step_fp8_workspace(p)
    # the step's workspace plus the quantised hidden block and its row scales
    assert ws_sz >= dg.denoise_step_workspace(p) + 256 * 1024 + 256 * 4

    def step(h=good, w8=good, sw=good, p_=p, n=ws_sz, io_=io):
        return lib.dg_denoise_step_fp8(_vp(h) if h else None, _vp(w8) if w8 else None,
                                       _vp(sw) if sw else None, ctypes.byref(p_),
                                       ctypes.byref(io_), _vp(good), n, None)

    assert step(sw=0) == 1                                               # null scales
    assert step(w8=good + 8) == 3                                        # misaligned codes
    assert step(n=ws_sz - 1) == 4                                        # workspace too small
    assert step(p_=dg.step_params(1, 256, 1088, 16384, 0.8), n=1 << 30) == 2   # d % 128 != 0
    assert step(io_=dg.StepIO(*([None] + [_vp(good)] * 8))) == 1
    assert lib.dg_lm_head_fold_fp8(_vp(good), None, _vp(good), ctypes.byref(p), _vp(good),
                                   ws_sz, None) == 1
    assert dg.denoise_step_fp8_workspace(dg.step_params(1, 256, 1024, 1001, 0.8)) == 0
    assert lib.dg_quantize_rows_e4m3(None, 4, 4, _vp(good), _vp(good), None) == 1
    assert lib.dg_quantize_rows_e4m3(_vp(good), 0, 4, _vp(good), _vp(good), None) == 1
    assert lib.dg_quantize_weight_e4m3(_vp(good), 0, 64, _vp(good), _vp(good), None) == 1


def test_wait_probe_rejects_bad_arguments_before_launch(lib):
    buf = ctypes.create_string_buffer(512)
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.dg_wait_timeout_probe(None, 256, 1000000, None) == 4          # no workspace
    assert lib.dg_wait_timeout_probe(ctypes.c_void_p(addr), 128, 1000000, None) == 4
    assert lib.dg_wait_timeout_probe(ctypes.c_void_p(addr), 256, 10, None) == 1
    assert lib.dg_wait_timeout_probe(ctypes.c_void_p(addr), 256, 2 * 10**9, None) == 1
    assert lib.dg_wait_timeout_probe(ctypes.c_void_p(addr + 4), 256, 1000000, None) == 3


def test_moe_rejects_bad_arguments_before_launch(lib):
    p = dg.moe_params(256, 2816, 768, 128, 8)
    assert dg.moe_ffn_workspace(p) > 256 * 9 * 2816 * 4
    assert dg.moe_ffn_workspace(dg.moe_params(256, 2816, 700, 128, 8)) == 0    # f % 128
    assert dg.moe_ffn_workspace(dg.moe_params(256, 320, 768, 128, 8)) == 0     # d % 128
    assert dg.moe_ffn_workspace(dg.moe_params(4096, 2816, 768, 128, 8)) == 0   # M > 2048
    assert dg.moe_ffn_workspace(dg.moe_params(256, 2816, 768, 4, 8)) == 0      # top_k > E
    bad = dg.moe_params(256, 2816, 768, 256, 8)                                 # E > 128
    rc = lib.dg_moe_ffn(*([None] * 8), ctypes.byref(bad), None, 0, None)
    assert rc == 2
    rc = lib.dg_moe_ffn(*([None] * 8), ctypes.byref(p), None, 0, None)
    assert rc == 1


def test_packed_weight_size_and_argument_checks(lib):
    """dg_pack_lm_weight: [ceil(V / 128)][d][128] bf16; the argument checks
    answer before any device work."""
    assert lib.dg_lm_weight_packed_bytes(2816, 262144) == 2048 * 2816 * 128 * 2
    assert lib.dg_lm_weight_packed_bytes(64, 1000) == 8 * 64 * 128 * 2
    assert lib.dg_lm_weight_packed_bytes(0, 1000) == 0
    a, b = 1 << 20, 1 << 40
    assert lib.dg_pack_lm_weight(None, 64, 1024, _vp(b), None) == 1
    assert lib.dg_pack_lm_weight(_vp(a), 64, 1024, None, None) == 1
    assert lib.dg_pack_lm_weight(_vp(a), 100, 1024, _vp(b), None) == 1    # d % 64
    assert lib.dg_pack_lm_weight(_vp(a), 64, 1001, _vp(b), None) == 1     # V % 8
    assert lib.dg_pack_lm_weight(_vp(a + 8), 64, 1024, _vp(b), None) == 3  # alignment
    # the packed copy may not overlap the weight
    assert lib.dg_pack_lm_weight(_vp(a), 64, 1024, _vp(a + 4096), None) == 1
    # a step's layout is 0 (row-major) or 1 (packed)
    assert dg.denoise_step_workspace(dg.step_params(1, 256, 1024, 16384, 0.8, w_layout=1)) > 0
    assert dg.denoise_step_workspace(dg.step_params(1, 256, 1024, 16384, 0.8, w_layout=2)) == 0


def test_pack_lm_weight_binding_rejects_bad_tensors(lib):
    """The binding packs only a contiguous bf16 [d, V] tensor (checked before
    any call into the library)."""
    import torch
    w = torch.zeros(64, 256, dtype=torch.bfloat16)
    for bad in (w.t(), w.float(), w.view(-1)):
        with pytest.raises(ValueError):
            dg.pack_lm_weight(bad)


def test_whole_step_fp8_and_sc_validate_before_launch(lib):
    """dg_canvas_step_fp8 / dg_canvas_step_sc: the step's checks and the
    workspace size are answered before anything is forked or launched."""
    good = 1 << 20
    p = dg.step_params(1, 256, 1024, 16384, 0.8)
    io = dg.StepIO(*[_vp(good + 64 * i) for i in range(9)])
    P, Hq, Hkv, D = 256, 4, 1, 128
    a = dg.canvas_attn_workspace(1, 256, P, Hq, Hkv, D)
    n8 = dg.canvas_step_fp8_workspace(p, P, Hq, Hkv, D)
    nsc = dg.canvas_step_sc_workspace(p, P, Hq, Hkv, D)
    # the step's workspace (rounded to 256 B), then the attention's
    assert n8 == (dg.denoise_step_fp8_workspace(p) + 255) // 256 * 256 + a
    assert nsc == (dg.denoise_step_sc_workspace(p) + 255) // 256 * 256 + a
    assert dg.canvas_step_fp8_workspace(p, P, Hq, Hkv, 64) == 0          # head dim
    assert dg.canvas_step_sc_workspace(dg.step_params(1, 256, 1024, 1001, 0.8), P, Hq, Hkv, D) == 0

    def fp8(h=good, w8=good, sw=good, n=n8, ws=good):
        return lib.dg_canvas_step_fp8(*[_vp(good)] * 6, P, Hq, Hkv, D, 0.1,
                                      _vp(h) if h else None, _vp(w8) if w8 else None,
                                      _vp(sw) if sw else None, ctypes.byref(p), ctypes.byref(io),
                                      _vp(ws) if ws else None, n, None)

    assert fp8(h=0) == 1                 # null hidden
    assert fp8(sw=good + 4) == 3         # misaligned scales
    assert fp8(n=n8 - 1) == 4            # workspace too small
    assert fp8(ws=0) == 4                # no workspace

    def sc(h=good, w=good, tab=good, out=good, n=nsc):
        return lib.dg_canvas_step_sc(*[_vp(good)] * 6, P, Hq, Hkv, D, 0.1,
                                     _vp(h) if h else None, _vp(w) if w else None,
                                     _vp(tab) if tab else None, ctypes.byref(p),
                                     ctypes.byref(io), _vp(out) if out else None, _vp(good), n,
                                     None)

    assert sc(tab=0) == 1                # null table
    assert sc(out=0) == 1                # null read-out
    assert sc(w=good + 2) == 3           # misaligned weight
    assert sc(n=nsc - 1) == 4            # workspace too small
