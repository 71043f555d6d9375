"""dg_denoise_step_noalloc: the denoising step for callers that cannot allocate.

Callers such as an engine that owns all device memory through its own pool,
or code that runs where cudaMalloc is not allowed, have no workspace to pass.
The allocation-free entry point runs the same kernels with a fixed scratch
array inside the library.  Here it is called through the C ABI twice in a
row (two consecutive steps, so the second call reuses the scratch the first
one left behind) and each result is compared with dg_denoise_step run on the
same inputs with a caller workspace.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
from tests._helpers import DEV, H_TOL, np_f, np_i32, to_dev

pytestmark = pytest.mark.gpu


def _state(bufs):
    return {n: getattr(bufs, n).detach().cpu().numpy().copy() for n, _ in dg.StepIO._fields_}


@pytest.mark.parametrize("B", [1, 2])   # one row block / two (the LM head's two epilogue widths)
def test_noalloc_step_matches_workspace_step_on_two_consecutive_calls(B):
    lib = dg.lib()
    cfg = dg_synth.StepConfig("noalloc", B=B, L=256, d=1024, V=16384, w_std=0.05, seed=21)
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(dg_synth.lm_weight(cfg))
    rng = np.random.default_rng(5)
    canvas0 = torch.from_numpy(rng.integers(0, cfg.V, cfg.M).astype(np.int32))

    ref, got = dg.StepBuffers(cfg.B, cfg.L, DEV), dg.StepBuffers(cfg.B, cfg.L, DEV)
    ref.canvas.copy_(canvas0)
    got.canvas.copy_(canvas0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for k in (0, 1):   # two calls in a row; the second sees the first call's scratch
        p = dg.step_params(cfg.B, cfg.L, cfg.d, cfg.V, 0.8 - 0.05 * k, 0.1, 0.005, step=k, seed=9)
        ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
        dg.denoise_step(x, w, p, ref, ws)
        io = got.io()
        rc = lib.dg_denoise_step_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                         ctypes.byref(p), ctypes.byref(io), stream)
        assert rc == 0, dg.STATUS_NAMES.get(rc, rc)
        torch.cuda.synchronize()
        assert dg.read_device_status(ws) == 0
        assert np.abs(np_f(got.entropy) - np_f(ref.entropy)).max() <= H_TOL
        for name in ("argmax", "sample", "canvas", "prev_argmax", "n_accepted", "stop"):
            assert np.array_equal(np_i32(getattr(got, name)), np_i32(getattr(ref, name))), name
        assert np.array_equal(got.accepted.cpu().numpy(), ref.accepted.cpu().numpy())
        assert np.abs(np_f(got.mean_entropy) - np_f(ref.mean_entropy)).max() <= H_TOL


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
