"""The packed LM-head weight (dg_pack_lm_weight, w_layout = DG_W_PACKED).

The packed weight holds W [d, V] as [ceil(V / 128)][d][128] (zero past V),
so the 2-SM LM-head kernels read one contiguous 16 KB stretch per 128 columns
and 64 hidden dimensions.  Checked here: the layout itself against its
definition (a zero-padded reshape and transpose of W); and that every entry
point taking W -- the step, the whole step with the attention beside it, the
block loop and the allocation-free step -- gives the same outputs bit for bit
with either layout on the same kernel plan, with the packed step also against
the fp64 oracle on a ragged vocabulary, including tiles that reach past the
last packed column tile.
"""
import ctypes
import math
import os

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import (DEV, check_step_against_oracle, force_lm_kernel, np_i32, status_ok,
                            to_dev)

pytestmark = pytest.mark.gpu

WORKERS = os.cpu_count() or 1
OUTS = ("canvas", "argmax", "sample", "n_accepted", "stop", "prev_argmax")


def _expected_packed(w):
    d, V = w.shape
    T = (V + 127) // 128
    wp = torch.zeros(d, T * 128, dtype=w.dtype, device=w.device)
    wp[:, :V] = w
    return wp.view(d, T, 128).permute(1, 0, 2).contiguous()


@pytest.mark.parametrize("d,V", [(64, 1000), (128, 4096), (192, 264), (2816, 262144)])
def test_pack_layout(d, V):
    g = torch.Generator(device=DEV).manual_seed(d + V)
    w = torch.randn(d, V, device=DEV, generator=g).to(torch.bfloat16)
    wp = dg.pack_lm_weight(w)
    torch.cuda.synchronize()
    T = (V + 127) // 128
    assert wp.numel() * 2 == dg.lm_weight_packed_bytes(d, V) == T * d * 256
    assert torch.equal(wp.view(T, d, 128), _expected_packed(w))


def _same_outputs(a, b):
    for name in OUTS:
        assert np.array_equal(np_i32(getattr(a, name)), np_i32(getattr(b, name))), name
    assert torch.equal(a.entropy, b.entropy)
    assert torch.equal(a.accepted, b.accepted)
    assert torch.equal(a.mean_entropy, b.mean_entropy)


def _two_layouts(x, w, B, L, d, V, T, k, seed, canvas0, prev):
    wp = dg.pack_lm_weight(w)
    out = []
    for layout, ww in ((dg.W_ROWMAJOR, w), (dg.W_PACKED, wp)):
        p = dg.step_params(B, L, d, V, T, 0.1, 0.005, step=k, seed=seed, w_layout=layout)
        ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
        bufs = dg.StepBuffers(B, L, DEV)
        bufs.canvas.copy_(torch.from_numpy(canvas0))
        bufs.prev_argmax.copy_(torch.from_numpy(prev))
        dg.denoise_step(x, ww, p, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        out.append(bufs)
    return out


def test_full_width_step_packed_equals_rowmajor_and_oracle():
    """2816 x 262144 (the planned 2-SM kernel on either layout): identical
    outputs, and the packed step against the oracle on every row."""
    cfg = dg_synth.CONFIGS["step_full"]
    B, L, d, V = cfg.B, cfg.L, cfg.d, cfg.V
    assert dg.lm_head_plan(B * L, d, V)["kind"] >= 2
    wb, xb = dg_synth.lm_weight(cfg), dg_synth.lm_hidden(cfg)
    k, seed = 2, 4
    T = oracle.temperature(k, cfg.max_steps)
    rng = np.random.default_rng(3)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    row, packed = _two_layouts(to_dev(xb), to_dev(wb), B, L, d, V, T, k, seed, canvas0, prev)
    _same_outputs(packed, row)
    ref = oracle.step(xb, wb, canvas0, prev, B, L, T, cfg.entropy_bound, seed, k,
                      cfg.stop_threshold, workers=WORKERS)
    assert check_step_against_oracle(packed, ref, B, L, exact_tokens=False) == 1


@pytest.mark.parametrize("kernel,bn", [("fused", None), ("duo", "256"), ("duo", "128")])
@pytest.mark.parametrize("B,L,d,V", [(1, 100, 128, 1000), (1, 64, 64, 264), (2, 200, 256, 4104)])
def test_ragged_packed_step_matches_oracle(kernel, bn, B, L, d, V, monkeypatch):
    """Ragged vocabularies (V % 128 != 0; with 256-column tiles the last tile
    reaches past the last packed column tile) and ragged row counts, on each
    2-SM kernel form: packed equals row-major bit for bit and matches the
    oracle (tokens outside the near-tie margins)."""
    force_lm_kernel(monkeypatch, kernel)
    if bn:
        monkeypatch.setenv("DG_LM_BN", bn)
    cfg = dg_synth.StepConfig("packed", B=B, L=L, d=d, V=V, w_std=0.05, seed=B + d)
    wb, xb = dg_synth.lm_weight(cfg), dg_synth.lm_hidden(cfg)
    rng = np.random.default_rng(V)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    T, k, seed = 0.7, 1, 6
    row, packed = _two_layouts(to_dev(xb), to_dev(wb), B, L, d, V, T, k, seed, canvas0, prev)
    _same_outputs(packed, row)
    ref = oracle.step(xb, wb, canvas0, prev, B, L, T, 0.1, seed, k, 0.005, workers=WORKERS)
    check_step_against_oracle(packed, ref, B, L, exact_tokens=False)


def test_canvas_step_packed_equals_rowmajor():
    """The whole full-width step (attention beside the LM head) on the packed
    weight: the same attention output and step outputs as on W [d, V]."""
    cfg = dg_synth.CONFIGS["step_full"]
    B, L, P, Hq, Hkv, D, d, V = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D, cfg.d, cfg.V
    t = {k: to_dev(v) for k, v in dg_synth.attention_inputs(cfg).items()}
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(dg_synth.lm_weight(cfg))
    wp = dg.pack_lm_weight(w)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    canvas0 = torch.from_numpy(np.random.default_rng(2).integers(0, V, B * L).astype(np.int32))
    res = []
    for layout, ww in ((dg.W_ROWMAJOR, w), (dg.W_PACKED, wp)):
        p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=4, seed=3, w_layout=layout)
        bufs = dg.StepBuffers(B, L, DEV)
        bufs.canvas.copy_(canvas0)
        out = torch.empty_like(t["q"])
        ws = dg.workspace(dg.canvas_step_workspace(p, P, Hq, Hkv, D), DEV)
        dg.canvas_step(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out, scale, x, ww, p, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        res.append((out, bufs))
    assert torch.equal(res[0][0], res[1][0])
    _same_outputs(res[1][1], res[0][1])


def test_block_loop_packed_equals_rowmajor(monkeypatch):
    """The block loop (one CUDA graph, a conditional while node) on the
    packed weight: steps taken, final canvas, argmax and per-step commits
    equal those on W [d, V] (both on the 2-SM kernel)."""
    force_lm_kernel(monkeypatch, "fused")
    B, L, d, V, steps = 2, 256, 256, 8192, 8
    cfg = dg_synth.StepConfig("packed_block", B=B, L=L, d=d, V=V, w_std=0.05, seed=12)
    w = to_dev(dg_synth.lm_weight(cfg))
    wp = dg.pack_lm_weight(w)
    g = torch.Generator(device=DEV).manual_seed(5)
    hs = (torch.randn(steps, B * L, d, device=DEV, generator=g) *
          torch.linspace(0.5, 4.0, steps, device=DEV).view(steps, 1, 1)).to(torch.bfloat16)
    res = []
    for layout, ww in ((dg.W_ROWMAJOR, w), (dg.W_PACKED, wp)):
        p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=0, seed=7, w_layout=layout)
        bp = dg.block_params(steps, 0.8, 0.4, B * L * d)
        bufs = dg.BlockBuffers(B, L, steps, DEV)
        ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
        dg.generate_block(hs, ww, p, bp, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        res.append(bufs)
    a, b = res
    for name in ("canvas", "argmax", "steps_taken", "mean_entropy", "n_accepted_hist"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert int(a.steps_taken.min()) >= 1


def test_noalloc_step_packed_equals_rowmajor(monkeypatch):
    """The allocation-free entry point reads the packed weight too."""
    force_lm_kernel(monkeypatch, "fused")
    B, L, d, V = 1, 256, 512, 32768
    cfg = dg_synth.StepConfig("packed_na", B=B, L=L, d=d, V=V, w_std=0.05, seed=33)
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(dg_synth.lm_weight(cfg))
    wp = dg.pack_lm_weight(w)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    canvas0 = torch.from_numpy(np.random.default_rng(1).integers(0, V, B * L).astype(np.int32))
    res = []
    for layout, ww in ((dg.W_ROWMAJOR, w), (dg.W_PACKED, wp)):
        p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=1, seed=2, w_layout=layout)
        bufs = dg.StepBuffers(B, L, DEV)
        bufs.canvas.copy_(canvas0)
        io = bufs.io()
        rc = dg.lib().dg_denoise_step_noalloc(ctypes.c_void_p(x.data_ptr()),
                                              ctypes.c_void_p(ww.data_ptr()), ctypes.byref(p),
                                              ctypes.byref(io), stream)
        assert rc == 0, dg.STATUS_NAMES.get(rc, rc)
        torch.cuda.synchronize()
        res.append(bufs)
    _same_outputs(res[1], res[0])


@pytest.mark.parametrize("B,L,d,V", [(1, 256, 256, 8200), (2, 130, 128, 4096)])
def test_self_conditioning_step_packed_equals_rowmajor(B, L, d, V):
    """The self-conditioning step (its own 2-SM instance, which also stages
    the table rows of each tile) on the packed weight: the same step outputs
    and the same read-out, bit for bit."""
    cfg = dg_synth.StepConfig("packed_sc", B=B, L=L, d=d, V=V, w_std=0.05, seed=40 + B)
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(dg_synth.lm_weight(cfg))
    wp = dg.pack_lm_weight(w)
    g = torch.Generator(device=DEV).manual_seed(V)
    table = (torch.randn(V, dg.SC_DIM, device=DEV, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    canvas0 = torch.from_numpy(np.random.default_rng(9).integers(0, V, B * L).astype(np.int32))
    res = []
    for layout, ww in ((dg.W_ROWMAJOR, w), (dg.W_PACKED, wp)):
        p = dg.step_params(B, L, d, V, 0.75, 0.1, 0.005, step=2, seed=5, w_layout=layout)
        ws = dg.workspace(dg.denoise_step_sc_workspace(p), DEV)
        bufs = dg.StepBuffers(B, L, DEV)
        bufs.canvas.copy_(canvas0)
        sc = torch.full((B * L, dg.SC_DIM), float("nan"), device=DEV)
        dg.denoise_step_sc(x, ww, table, p, bufs, sc, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        res.append((bufs, sc))
    _same_outputs(res[1][0], res[0][0])
    assert torch.equal(res[0][1], res[1][1])
    assert bool(torch.isfinite(res[1][1]).all())


def test_block_loop_with_producer_packed_equals_rowmajor(monkeypatch):
    """The loop with the decoder body captured into it (the built-in
    canvas-dependent producer, hidden_k = bf16(base_k + E[canvas])) on the
    packed weight: the same run as on W [d, V] (both on the 2-SM kernel)."""
    force_lm_kernel(monkeypatch, "fused")
    B, L, d, V, steps = 1, 128, 256, 4096, 10
    cfg = dg_synth.StepConfig("packed_fn", B=B, L=L, d=d, V=V, w_std=0.05, seed=14)
    w = to_dev(dg_synth.lm_weight(cfg))
    wp = dg.pack_lm_weight(w)
    g = torch.Generator(device=DEV).manual_seed(8)
    base = (torch.randn(steps, L, d, device=DEV, generator=g) * 2.0).to(torch.bfloat16)
    table = (torch.randn(V, d, device=DEV, generator=g) * 0.05).to(torch.bfloat16)
    user = dg.HiddenEmbed(base.data_ptr(), L * d, table.data_ptr(), L, d, V)
    res = []
    for layout, ww in ((dg.W_ROWMAJOR, w), (dg.W_PACKED, wp)):
        p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=0, seed=6, w_layout=layout)
        bp = dg.block_params(steps, 0.8, 0.4, 0)
        bufs = dg.BlockBuffers(B, L, steps, DEV)
        ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
        buf = torch.empty(L, d, dtype=torch.bfloat16, device=DEV)
        dg.generate_block_fn(dg.hidden_producer("embed_add"), user, buf, ww, p, bp, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        res.append(bufs)
    a, b = res
    for name in ("canvas", "argmax", "steps_taken", "mean_entropy", "n_accepted_hist"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
