"""The block loop's graph cache.  The seed is part of a cached graph's key, so
each new seed captures a new graph; the library keeps at most 64 and drops
the least recently used.  A seed's block must come out the same on first
use, on a replay of its cached graph and after its graph was dropped and
captured again."""
import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
from tests._helpers import DEV, np_i32, status_ok, to_dev

pytestmark = pytest.mark.gpu

N = 8


def test_block_graph_cache_drops_and_recaptures_with_the_same_results():
    cfg = dg_synth.StepConfig("cache", L=64, d=256, V=2048, w_std=0.02, seed=18)
    wb = dg_synth.lm_weight(cfg)
    tg = dg_synth.block_targets(cfg)
    h = to_dev(dg_synth.block_hidden(cfg, wb, tg, 0))
    w = to_dev(wb)
    bp = dg.block_params(N, 0.8, 0.4, 0)
    bufs = dg.BlockBuffers(1, cfg.L, N, DEV)
    p0 = dg.step_params(1, cfg.L, cfg.d, cfg.V, 0.8, 0.1, 0.005, step=0, seed=0)
    ws = dg.workspace(dg.generate_block_workspace(p0, bp), DEV)

    def run(seed):
        p = dg.step_params(1, cfg.L, cfg.d, cfg.V, 0.8, 0.1, 0.005, step=0, seed=seed)
        dg.generate_block(h, w, p, bp, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        steps = int(bufs.steps_taken[0])
        assert 1 <= steps <= N
        return (steps, np_i32(bufs.n_accepted_hist)[:steps].copy(), np_i32(bufs.canvas).copy(),
                np_i32(bufs.argmax).copy())

    # 70 keys: more than the cache holds, so the first seeds' graphs are dropped
    first = {s: run(s) for s in range(70)}
    assert len({r[2].tobytes() for r in first.values()}) > 1     # the seed matters
    for s in (0, 1, 2, 69, 68):      # dropped and captured again / still cached
        again = run(s)
        assert again[0] == first[s][0]
        for a, b in zip(again[1:], first[s][1:]):
            assert np.array_equal(a, b)
