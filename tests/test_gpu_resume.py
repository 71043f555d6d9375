"""Resuming the denoising loop from its state.  The loop's state between steps
is the canvas, the previous step's argmax and the step index (the random
numbers are counter-based Philox keyed by (seed, row, step)), so a loop
driven from the host with dg_denoise_step, stopped after step k, its state
copied to the host and back into fresh buffers, and continued, must give the
same result as an uninterrupted run -- and the same as dg_generate_block,
the loop as one CUDA graph."""
import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import DEV, np_i32, status_ok, to_dev

pytestmark = pytest.mark.gpu

N = 48


def _host_loop(x_steps, w, cfg, seed, checkpoint_at=None):
    B, L, d, V = 1, cfg.L, cfg.d, cfg.V
    bufs = dg.StepBuffers(B, L, DEV)
    bufs.canvas.copy_(torch.from_numpy(oracle.init_canvas(B * L, V, seed)))
    bufs.prev_argmax.fill_(-1)
    p0 = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=0, seed=seed)
    ws = dg.workspace(dg.denoise_step_workspace(p0), DEV)
    hist, last = [], None
    for k in range(N):
        T = oracle.temperature(k, N)
        p = dg.step_params(B, L, d, V, T, 0.1, 0.005, step=k, seed=seed)
        dg.denoise_step(x_steps[k], w, p, bufs, ws)
        torch.cuda.synchronize()
        hist.append(int(bufs.n_accepted[0]))
        last = k
        if int(bufs.stop[0]):
            break
        if checkpoint_at is not None and k == checkpoint_at:
            # the state to the host and back into new buffers and workspace
            state = {n: getattr(bufs, n).cpu().clone() for n in ("canvas", "prev_argmax")}
            del bufs, ws
            bufs = dg.StepBuffers(B, L, DEV)
            ws = dg.workspace(dg.denoise_step_workspace(p0), DEV)
            bufs.canvas.copy_(state["canvas"])
            bufs.prev_argmax.copy_(state["prev_argmax"])
    status_ok(ws)
    return dict(steps=last + 1, hist=hist, canvas=np_i32(bufs.canvas).copy(),
                argmax=np_i32(bufs.argmax).copy())


def test_resume_from_state_equals_uninterrupted_and_the_graph_loop():
    cfg = dg_synth.StepConfig("resume", L=64, d=256, V=2048, w_std=0.02, seed=18)
    wb = dg_synth.lm_weight(cfg)
    tg = dg_synth.block_targets(cfg)
    hs = np.stack([dg_synth.block_hidden(cfg, wb, tg, k) for k in range(N)])
    x_steps = [to_dev(hs[k]) for k in range(N)]
    w = to_dev(wb)
    full = _host_loop(x_steps, w, cfg, 9)
    assert 2 <= full["steps"] < N
    for ck in (0, 3, full["steps"] - 2):
        resumed = _host_loop(x_steps, w, cfg, 9, checkpoint_at=ck)
        assert resumed["steps"] == full["steps"]
        assert resumed["hist"] == full["hist"]
        assert np.array_equal(resumed["canvas"], full["canvas"])
        assert np.array_equal(resumed["argmax"], full["argmax"])
    # the same loop as one CUDA graph
    p = dg.step_params(1, cfg.L, cfg.d, cfg.V, 0.8, 0.1, 0.005, step=0, seed=9)
    bp = dg.block_params(N, 0.8, 0.4, cfg.L * cfg.d)
    bufs = dg.BlockBuffers(1, cfg.L, N, DEV)
    ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
    dg.generate_block(to_dev(hs), w, p, bp, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    assert int(bufs.steps_taken[0]) == full["steps"]
    assert np_i32(bufs.n_accepted_hist)[:full["steps"]].tolist() == full["hist"]
    assert np.array_equal(np_i32(bufs.canvas), full["canvas"])
    assert np.array_equal(np_i32(bufs.argmax), full["argmax"])
