"""dg_denoise_step_noalloc: the denoising step for callers that cannot allocate.

Callers such as an engine that owns all device memory through its own pool,
or code that runs where cudaMalloc is not allowed, have no workspace to pass.
The allocation-free entry point runs the same kernels with a fixed scratch
array inside the library.  Here it is called through the C ABI twice in a
row (two consecutive steps, so the second call reuses the scratch the first
one left behind) and each result is compared with dg_denoise_step run on the
same inputs with a caller workspace; the scratch's device status word is read
with dg_noalloc_read_device_status after every call.  Shapes: the small LM
head at one and two canvases, the full-width LM head (2816 x 262144, the 2-SM
kernel), and the largest step the 8 MiB scratch holds on this device; the
first step beyond it is rejected.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
from tests._helpers import DEV, H_TOL, np_f, np_i32, to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


def _ru(x, a=256):
    return (x + a - 1) // a * a


def _scratch_need(B, L, d, V):
    """Bytes of scratch a step needs (the formula include/dg.h states)."""
    M = B * L
    plan = dg.lm_head_plan(M, d, V)
    units = plan["ctas"] // 2 if plan["kind"] >= 2 else plan["ctas"]
    return 256 + _ru(7 * 4 * units * M) + _ru(4 * B) + _ru(4 * M)


def _noalloc_status(clear=False):
    v = ctypes.c_int(-1)
    rc = dg.lib().dg_noalloc_read_device_status(ctypes.byref(v), 1 if clear else 0, None)
    assert rc == 0, dg.STATUS_NAMES.get(rc, rc)
    return v.value


def _two_calls_match(x, w, B, L, d, V, seed=9):
    lib = dg.lib()
    M = B * L
    rng = np.random.default_rng(5)
    canvas0 = torch.from_numpy(rng.integers(0, V, M).astype(np.int32))
    ref, got = dg.StepBuffers(B, L, DEV), dg.StepBuffers(B, L, DEV)
    ref.canvas.copy_(canvas0)
    got.canvas.copy_(canvas0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for k in (0, 1):   # two calls in a row; the second sees the first call's scratch
        p = dg.step_params(B, L, d, V, 0.8 - 0.05 * k, 0.1, 0.005, step=k, seed=seed)
        ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
        dg.denoise_step(x, w, p, ref, ws)
        io = got.io()
        rc = lib.dg_denoise_step_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                         ctypes.byref(p), ctypes.byref(io), stream)
        assert rc == 0, dg.STATUS_NAMES.get(rc, rc)
        torch.cuda.synchronize()
        assert dg.read_device_status(ws) == 0
        assert _noalloc_status() == 0
        assert np.abs(np_f(got.entropy) - np_f(ref.entropy)).max() <= H_TOL
        for name in ("argmax", "sample", "canvas", "prev_argmax", "n_accepted", "stop"):
            assert np.array_equal(np_i32(getattr(got, name)), np_i32(getattr(ref, name))), name
        assert np.array_equal(got.accepted.cpu().numpy(), ref.accepted.cpu().numpy())
        assert np.abs(np_f(got.mean_entropy) - np_f(ref.mean_entropy)).max() <= H_TOL


@pytest.mark.parametrize("B", [1, 2])   # one row block / two (the LM head's two epilogue widths)
def test_noalloc_step_matches_workspace_step_on_two_consecutive_calls(B):
    cfg = dg_synth.StepConfig("noalloc", B=B, L=256, d=1024, V=16384, w_std=0.05, seed=21)
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(dg_synth.lm_weight(cfg))
    _two_calls_match(x, w, cfg.B, cfg.L, cfg.d, cfg.V)


def test_noalloc_full_width_step_matches_workspace_step():
    """The full-width LM head (2816 x 262144): the 2-SM kernel on the fused
    schedule, with its per-row Gumbel bounds shared between units."""
    B, L, d, V = 1, 256, 2816, 262144
    g = torch.Generator(device=DEV).manual_seed(31)
    x = (torch.randn(B * L, d, device=DEV, generator=g)
         * (torch.rand(B * L, 1, device=DEV, generator=g) * 7.5 + 0.5)).to(torch.bfloat16)
    w = (torch.randn(d, V, device=DEV, generator=g) * 0.02).to(torch.bfloat16)
    assert dg.lm_head_plan(B * L, d, V)["kind"] >= 2
    _two_calls_match(x, w, B, L, d, V)


def _capacity_cases(d, V):
    """(B, L) of the largest step that fits the scratch and of the smallest one
    that does not, over B <= 16 and L <= 1024."""
    fit, over = None, None
    for B in range(1, 17):
        lo, hi = 0, 1024             # need grows with L: largest L that fits
        while lo < hi:
            mid = (lo + hi + 1) // 2
            if _scratch_need(B, mid, d, V) <= SCRATCH_BYTES:
                lo = mid
            else:
                hi = mid - 1
        if lo >= 1 and (fit is None or B * lo > fit[0] * fit[1]):
            fit = (B, lo)
        if lo < 1024 and (over is None or B * (lo + 1) < over[0] * over[1]):
            over = (B, lo + 1)
    return fit, over


def test_noalloc_largest_step_that_fits_and_first_rejected():
    d, V = 1024, 16384
    fit, over = _capacity_cases(d, V)
    assert fit is not None and over is not None
    assert fit[0] * fit[1] >= 1968 or torch.cuda.get_device_properties(0).multi_processor_count != 152
    B, L = fit
    g = torch.Generator(device=DEV).manual_seed(41)
    x = torch.randn(B * L, d, device=DEV, generator=g).to(torch.bfloat16)
    w = (torch.randn(d, V, device=DEV, generator=g) * 0.05).to(torch.bfloat16)
    _two_calls_match(x, w, B, L, d, V)
    # the first step beyond the scratch is rejected before anything is launched
    B, L = over
    p = dg.step_params(B, L, d, V, 0.8)
    bufs = dg.StepBuffers(1, 8, DEV)          # never touched: the call is rejected first
    io = bufs.io()
    rc = dg.lib().dg_denoise_step_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                          ctypes.byref(p), ctypes.byref(io), None)
    assert rc == 2   # DG_ERR_UNSUPPORTED
    assert _noalloc_status() == 0


def test_noalloc_rejects_steps_beyond_its_scratch():
    lib = dg.lib()
    # 16 canvases of 1024 positions need far more than the 8 MiB scratch
    p = dg.step_params(16, 1024, 1024, 16384, 0.8)
    bufs = dg.StepBuffers(1, 8, DEV)          # never touched: the call is rejected first
    x = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    io = bufs.io()
    rc = lib.dg_denoise_step_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                                     ctypes.byref(p), ctypes.byref(io), None)
    assert rc == 2   # DG_ERR_UNSUPPORTED
