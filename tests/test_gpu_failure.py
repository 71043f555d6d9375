"""The failure path of the library's bounded device waits, on a GPU, without
a fault: a wait that nothing completes gives up after its limit, records
DG_ERR_TIMEOUT in the workspace's status word, frees its TMEM and returns;
the context and the workspace stay usable (after the status is cleared, a
denoising step on the same workspace runs and matches the oracle)."""
import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import DEV, H_TOL, np_f, to_dev

pytestmark = pytest.mark.gpu

DG_ERR_TIMEOUT = 6


def test_bounded_wait_times_out_and_the_context_stays_usable():
    cfg = dg_synth.StepConfig("fail", L=64, d=128, V=1024, w_std=0.05, seed=2)
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    p = dg.step_params(1, cfg.L, cfg.d, cfg.V, 0.8, 0.1, 0.005, step=1, seed=4)
    ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
    for limit_ns in (1_000_000, 20_000_000):        # 1 ms, 20 ms
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        dg.wait_timeout_probe(ws, limit_ns)
        e.record()
        torch.cuda.synchronize()
        # the wait really waited for its limit, then gave up
        assert s.elapsed_time(e) * 1e6 >= 0.9 * limit_ns
        assert dg.read_device_status(ws, clear=True) == DG_ERR_TIMEOUT
        assert dg.read_device_status(ws) == 0
    # the same workspace (status cleared) serves a normal step afterwards
    bufs = dg.StepBuffers(1, cfg.L, DEV)
    canvas0 = oracle.init_canvas(cfg.L, cfg.V, 4)
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    dg.denoise_step(to_dev(xb), to_dev(wb), p, bufs, ws)
    torch.cuda.synchronize()
    assert dg.read_device_status(ws) == 0
    ref = oracle.step(xb, wb, canvas0, np.full(cfg.L, -1, np.int32), 1, cfg.L, 0.8, 0.1, 4, 1)
    assert np.abs(np_f(bufs.entropy) - ref["H"]).max() < H_TOL
