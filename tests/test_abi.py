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


# ------------------------------------------------------------------ canvas step plan
_SMALL = dict(B=1, L=256, d=1024, V=16384, P=256, Hq=4, Hkv=1, D=128)
_FULL = dict(B=1, L=256, d=2816, V=262144, P=4096, Hq=16, Hkv=8, D=256)


@pytest.fixture
def planner_defaults(monkeypatch):
    """No planner override from the caller's environment."""
    for v in ("DG_ATTN_KERNEL", "DG_ATTN_SPLITS", "DG_ATTN_RESERVE", "DG_LM_KERNEL", "DG_LM_BN",
              "DG_LM_EPI"):
        monkeypatch.delenv(v, raising=False)


def _plan(sms=152, w_layout=dg.W_ROWMAJOR, **kw):
    c = dict(_SMALL, **kw)
    p = dg.step_params(c["B"], c["L"], c["d"], c["V"], 0.8, w_layout=w_layout)
    return dg.canvas_step_plan(p, c["P"], c["Hq"], c["Hkv"], c["D"], sms)


def test_canvas_step_plan_of_the_measured_shapes(lib, planner_defaults):
    """The plans the measured canvas steps run on a 152-SM GB300, computed on
    the host: the small step sets 4 SMs aside for its 8 attention CTAs and
    runs the single-CTA LM head as 147 tiles of 112 columns on the other 148;
    with 2048 cached keys the attention keeps 24 SMs (3 key splits of at most
    6 tiles) and the LM head runs 128 tiles of 128 columns; the full-width
    step reserves nothing: the 2-SM attention on 128 CTAs (4 splits) shares
    the GPU with the fused 2-SM LM head on all 152 SMs."""
    assert _plan() == dict(attn_reserved_sms=4, attn_pair=0, attn_ctas=8, attn_splits=1,
                           attn_key_tiles=4, attn_key_tile=128, lm_kind=0, lm_bn=112,
                           lm_ctas=147, lm_tiles=147, lm_epilogue_warps=0, lm_sms=148)
    b1 = _plan(P=2048)
    assert (b1["attn_reserved_sms"], b1["attn_ctas"], b1["attn_splits"], b1["attn_key_tiles"]) \
        == (24, 24, 3, 6)
    assert (b1["lm_kind"], b1["lm_bn"], b1["lm_ctas"], b1["lm_sms"]) == (0, 128, 128, 128)
    for layout in (dg.W_ROWMAJOR, dg.W_PACKED):
        full = _plan(w_layout=layout, **_FULL)
        assert full == dict(attn_reserved_sms=0, attn_pair=1, attn_ctas=128, attn_splits=4,
                            attn_key_tiles=9, attn_key_tile=128, lm_kind=3, lm_bn=128,
                            lm_ctas=152, lm_tiles=2048, lm_epilogue_warps=8, lm_sms=152)
    # four canvases with 2048 cached keys: no reservation, the fused 2-SM LM
    # head with 16 epilogue warps (four 256-row blocks)
    b4 = _plan(B=4, P=2048)
    assert (b4["attn_reserved_sms"], b4["lm_kind"], b4["lm_epilogue_warps"]) == (0, 3, 16)


def test_canvas_step_plan_reservation_override(lib, planner_defaults, monkeypatch):
    """DG_ATTN_RESERVE=n forces n SMs (rounded down to even; 0: none) and
    skips the search for a smaller reservation."""
    monkeypatch.setenv("DG_ATTN_RESERVE", "0")
    p0 = _plan()
    assert p0["attn_reserved_sms"] == 0 and p0["lm_sms"] == 152
    monkeypatch.setenv("DG_ATTN_RESERVE", "9")
    p8 = _plan()
    assert p8["attn_reserved_sms"] == 8 and p8["lm_sms"] == 144
    # one wave of 128-column tiles on 144 SMs
    assert (p8["lm_kind"], p8["lm_bn"], p8["lm_ctas"]) == (0, 128, 128)


def _ceil(a, b):
    return -(-a // b)


@pytest.mark.parametrize("sms", [16, 60, 132, 148, 152, 256])
def test_canvas_step_plan_invariants(lib, planner_defaults, sms):
    """Over a sweep of shapes and SM counts: the LM-head tiles cover the
    vocabulary and rows once, its grid fits the SMs left to it, the key
    splits cover every key tile, a reservation is even and leaves the LM head
    the rest, and a packed W keeps the LM head on the 2-SM kernels."""
    for B, L, P, Hq, Hkv, D, d, V in [
            (1, 256, 256, 4, 1, 128, 1024, 16384), (1, 256, 2048, 4, 1, 128, 1024, 16384),
            (4, 256, 2048, 4, 1, 128, 1024, 16384), (16, 256, 2048, 4, 1, 128, 1024, 16384),
            (1, 256, 32768, 4, 1, 128, 1024, 16384), (1, 256, 4096, 16, 8, 256, 2816, 262144),
            (2, 100, 0, 8, 2, 128, 512, 1000), (1, 17, 777, 16, 1, 256, 64, 64),
            (3, 256, 130, 8, 8, 256, 2048, 50000), (1, 64, 1, 2, 1, 128, 128, 262144)]:
        for layout in (dg.W_ROWMAJOR, dg.W_PACKED):
            pl = _plan(sms, layout, B=B, L=L, P=P, Hq=Hq, Hkv=Hkv, D=D, d=d, V=V)
            r = pl["attn_reserved_sms"]
            assert r % 2 == 0 and 0 <= r <= sms // 6 + 1
            assert pl["lm_sms"] == sms - r
            # attention: every key tile of [cache ; canvas] in some split
            bkv = pl["attn_key_tile"]
            nkt = _ceil(P, bkv) + _ceil(L, bkv)
            ns, tps = pl["attn_splits"], pl["attn_key_tiles"]
            assert ns * tps >= nkt and (ns - 1) * tps < nkt
            G = Hq // Hkv
            mtiles = _ceil(L * G, 128)
            if pl["attn_pair"]:
                mtiles += mtiles & 1
            assert pl["attn_ctas"] == mtiles * Hkv * B * ns
            assert pl["attn_pair"] == (1 if D == 256 else 0)
            if r > 0 and ns > 1:
                assert pl["attn_ctas"] <= r
            # LM head
            kind, bn = pl["lm_kind"], pl["lm_bn"]
            mblocks = _ceil(B * L, 256)
            assert pl["lm_tiles"] == _ceil(V, bn) * mblocks
            if layout == dg.W_PACKED:
                assert kind in (2, 3)
            if kind == 0:
                assert bn % 16 == 0 and 64 <= bn <= 128
                assert pl["lm_ctas"] <= min(pl["lm_sms"], pl["lm_tiles"])
                assert pl["lm_epilogue_warps"] == 0
            else:
                assert kind in (2, 3) and bn in ((128, 256) if kind == 2 else (128,))
                assert pl["lm_ctas"] % 2 == 0
                assert pl["lm_ctas"] <= max(2, pl["lm_sms"] // 2 * 2)
                assert pl["lm_ctas"] // 2 <= pl["lm_tiles"]
                assert pl["lm_epilogue_warps"] == (8 if mblocks == 1 else 16)
            assert pl["lm_ctas"] <= 256


def test_canvas_step_plan_rejects_before_planning(lib, planner_defaults):
    """Bad arguments are answered without touching a device, and the output
    is left as it was."""
    p = dg.step_params(1, 256, 1024, 16384, 0.8)
    out = dg.CanvasStepPlan(*([-7] * len(dg.CanvasStepPlan._fields_)))

    def call(pp=p, P=256, Hq=4, Hkv=1, D=128, sms=152, o=out):
        return lib.dg_canvas_step_plan(ctypes.byref(pp) if pp is not None else None, P, Hq, Hkv,
                                       D, sms, ctypes.byref(o) if o is not None else None)

    assert call(pp=None) == 1
    assert call(o=None) == 1
    assert call(sms=257) == 1
    assert call(pp=dg.step_params(1, 256, 1024, 16384, -1.0)) == 1     # temperature
    assert call(D=64) == 2                                            # head dim
    assert call(Hq=3, Hkv=2) == 2                                     # GQA group
    assert call(pp=dg.step_params(1, 256, 1000, 16384, 0.8)) == 2     # d % 64
    assert call(pp=dg.step_params(1, 256, 1024, 1001, 0.8)) == 2      # V % 8
    assert [getattr(out, n) for n, _ in dg.CanvasStepPlan._fields_] == [-7] * 12
    assert call() == 0 and out.lm_ctas == 147
    import torch
    if not torch.cuda.is_available():
        assert call(sms=0) == 5                                       # no device


def _r256(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("env", [{}, {"DG_ATTN_SPLITS": "1"}, {"DG_ATTN_SPLITS": "3"},
                                 {"DG_ATTN_SPLITS": "64"}, {"DG_ATTN_KERNEL": "single"},
                                 {"DG_ATTN_KERNEL": "pair"}, {"DG_LM_KERNEL": "single"},
                                 {"DG_LM_KERNEL": "duo", "DG_LM_BN": "128"},
                                 {"DG_LM_KERNEL": "fused"}, {"DG_LM_BN": "64"},
                                 {"DG_ATTN_RESERVE": "40"}])
def test_canvas_step_plans_fit_the_queried_workspace(lib, planner_defaults, monkeypatch, env):
    """Whatever the SM count or a forced planner choice, the plan's partial
    states fit the workspace the queries answered without knowing either:
    the attention's key-split partials (bf16 outputs and fp32 max / sum per
    split and query row, after a 256-byte header) and the LM head's per-unit
    partial states (7 words per row and unit, at most one unit per 64-column
    tile or 256 units)."""
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    for B, L, P, Hq, Hkv, D, d, V in [
            (1, 256, 256, 4, 1, 128, 1024, 16384), (1, 256, 32768, 4, 1, 128, 1024, 16384),
            (16, 256, 2048, 4, 1, 128, 1024, 16384), (1, 256, 4096, 16, 8, 256, 2816, 262144),
            (1, 200, 3000, 16, 8, 256, 512, 4096), (1, 1, 100000, 2, 1, 256, 64, 64),
            (3, 37, 129, 8, 1, 128, 128, 1000)]:
        p = dg.step_params(B, L, d, V, 0.8)
        attn_ws = dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D)
        step_ws = dg.denoise_step_workspace(p)
        assert dg.canvas_step_workspace(p, P, Hq, Hkv, D) == _r256(step_ws) + attn_ws
        M = B * L
        for sms in (8, 24, 76, 148, 152, 200, 256):
            pl = dg.canvas_step_plan(p, P, Hq, Hkv, D, sms)
            ns = pl["attn_splits"]
            need = 256 if ns == 1 else 256 + _r256(ns * M * Hq * D * 2) + _r256(ns * M * Hq * 8)
            assert need <= attn_ws, (B, L, P, Hq, Hkv, D, sms, pl)
            units = pl["lm_ctas"] // (1 if pl["lm_kind"] == 0 else 2)
            assert units <= min(_ceil(M, 256) * _ceil(V, 64), 256)
            assert 256 + _r256(7 * units * M * 4) + _r256(B * 4) + _r256(M * 4) <= step_ws
