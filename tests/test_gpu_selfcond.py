"""GPU parity of the self-conditioning read-out (dg_denoise_step_sc) against
the fp64 oracle: sc[r] = sum_v softmax(logits_r / T)_v E[v, :], folded into
the 2-SM LM head ("Parallel Denoising From an Autoregressive Checkpoint",
section "Finding": the self-conditioning block's matmul runs next to the
full-vocabulary softmax).

Tolerance of the read-out, per row: max_j |sc_j - sc*_j| <= 2e-2 max_j |sc*_j|
+ 2e-4 max |E| (the second term covers the bf16 rounding of the weights and
the fp32 summation over the vocabulary when the weighted rows cancel, e.g.
uniform weights over a zero-mean table).  Every other output of the step is checked as for
dg_denoise_step (entropies 1e-4, tokens where the margins allow).
"""
import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import (DEV, H_TOL, check_step_against_oracle, np_f, np_i32, status_ok,
                            to_dev)

pytestmark = pytest.mark.gpu

SC_REL, SC_ABS = 2e-2, 2e-4
WORKERS = 8


def _table(V, seed, R=dg.SC_DIM):
    """A bf16 table (as its fp32 values: the oracle's input)."""
    rng = np.random.default_rng(seed)
    return dg_synth.bf16_bits_to_f32(dg_synth.f32_to_bf16_bits(
        rng.standard_normal((V, R)).astype(np.float32)))


def _check_sc(got, ref, E):
    scale = np.abs(ref).max(axis=1)
    err = np.abs(got - ref).max(axis=1)
    bound = SC_REL * scale + SC_ABS * float(np.abs(E).max())
    assert (err <= bound).all(), (float((err / bound).max()), int((err / bound).argmax()))


def _run_sc(xb, wb, E, B, L, d, V, T, seed, k, canvas0=None, prev=None):
    x, w = to_dev(xb), to_dev(wb)
    Et = torch.from_numpy(E).to(DEV).to(torch.bfloat16)     # exact: E holds bf16 values
    p = dg.step_params(B, L, d, V, T, 0.1, 0.005, step=k, seed=seed)
    ws = dg.workspace(dg.denoise_step_sc_workspace(p), DEV)
    bufs = dg.StepBuffers(B, L, DEV)
    if canvas0 is not None:
        bufs.canvas.copy_(torch.from_numpy(canvas0))
    if prev is not None:
        bufs.prev_argmax.copy_(torch.from_numpy(prev))
    sc = torch.full((B * L, dg.SC_DIM), float("nan"), device=DEV)
    dg.denoise_step_sc(x, w, Et, p, bufs, sc, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    return bufs, sc.cpu().numpy()


@pytest.mark.parametrize("B,L,d,V,T", [(1, 256, 256, 4096, 0.8), (2, 100, 128, 4104, 0.5),
                                       (1, 64, 192, 16384, 0.4), (3, 256, 256, 2048, 0.8)])
def test_selfcond_step_matches_oracle(B, L, d, V, T):
    cfg = dg_synth.StepConfig("sc", B=B, L=L, d=d, V=V, w_std=0.08, seed=B * 7 + L,
                              row_scale=(0.5, 8.0))
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    E = _table(V, 3)
    rng = np.random.default_rng(1)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    bufs, sc = _run_sc(xb, wb, E, B, L, d, V, T, 11, 2, canvas0, prev)
    ref = oracle.step(xb, wb, canvas0, prev, B, L, T, 0.1, 11, 2, workers=WORKERS)
    check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)
    _check_sc(sc, oracle.self_cond(ref["logits"], T, E, workers=WORKERS), E)


def test_selfcond_other_outputs_equal_the_plain_step_on_the_same_kernel(monkeypatch):
    """With the same 2-SM kernel and tiling forced on both, every other output of
    the step is the same: the read-out adds to the fold without changing its
    decisions (tokens identical, entropies to 1e-6)."""
    cfg = dg_synth.StepConfig("sc2", B=1, L=256, d=512, V=8192, w_std=0.05, seed=5)
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    E = _table(cfg.V, 4)
    monkeypatch.setenv("DG_LM_KERNEL", "duo")
    monkeypatch.setenv("DG_LM_EPI", "8")
    bufs, _ = _run_sc(xb, wb, E, 1, cfg.L, cfg.d, cfg.V, 0.8, 3, 1)
    p = dg.step_params(1, cfg.L, cfg.d, cfg.V, 0.8, 0.1, 0.005, step=1, seed=3)
    ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
    ref = dg.StepBuffers(1, cfg.L, DEV)
    dg.denoise_step(to_dev(xb), to_dev(wb), p, ref, ws)
    torch.cuda.synchronize()
    assert dg.lm_head_plan(cfg.L, cfg.d, cfg.V)["kernel"] == "lm_head_duo_kernel"
    for name in ("argmax", "sample", "canvas", "n_accepted", "stop"):
        assert np.array_equal(np_i32(getattr(bufs, name)), np_i32(getattr(ref, name))), name
    assert np.abs(np_f(bufs.entropy) - np_f(ref.entropy)).max() <= 1e-6


def test_selfcond_special_cases():
    """Zero hidden states (every logit 0): uniform weights, the read-out is the
    mean of E's rows.  One dominant logit per row: the read-out is that
    token's row of E."""
    L, d, V = 128, 64, 4096
    E = _table(V, 5)
    bufs, sc = _run_sc(np.zeros((L, d), np.uint16), dg_synth.lm_weight(
        dg_synth.StepConfig("w", d=d, V=V, w_std=0.05, seed=6)), E, 1, L, d, V, 0.8, 1, 0)
    _check_sc(sc, np.broadcast_to(E.astype(np.float64).mean(axis=0), sc.shape), E)
    # one-hot: W has one large entry per token column group; row i hits token 3 i
    w = np.zeros((d, V), np.float32)
    w[np.arange(d), np.arange(d) * 3] = 300.0
    x = np.zeros((L, d), np.float32)
    x[np.arange(L), np.arange(L) % d] = 1.0
    bufs, sc = _run_sc(dg_synth.f32_to_bf16_bits(x), dg_synth.f32_to_bf16_bits(w), E, 1, L, d, V,
                       0.4, 1, 0)
    hot = (np.arange(L) % d) * 3
    # the row of E, up to the bf16 rounding of the chunk weights (the weight
    # is 1 within 2^-9, the softmax sum it is divided by is fp32)
    assert np.abs(sc - E[hot]).max() <= 2e-3 * float(np.abs(E).max())
    _check_sc(sc, E[hot].astype(np.float64), E)
    assert np.array_equal(np_i32(bufs.argmax), hot)


def test_selfcond_full_width_sampled_rows():
    """The full-width LM head (2816 x 262144, per-row logit scale U(0.5, 8)),
    the read-out of sampled rows against the oracle."""
    cfg = dg_synth.CONFIGS["step_full"]
    xb = dg_synth.lm_hidden(cfg)
    wb = dg_synth.lm_weight(dg_synth.StepConfig("w", d=cfg.d, V=cfg.V, w_std=cfg.w_std,
                                                seed=cfg.seed))
    E = _table(cfg.V, 7)
    bufs, sc = _run_sc(xb, wb, E, 1, cfg.L, cfg.d, cfg.V, 0.8, 0, 3)
    rows = np.arange(0, cfg.L, 9)
    lg = oracle.logits(xb, wb, rows=rows)
    _check_sc(sc[rows], oracle.self_cond(lg, 0.8, E, workers=WORKERS), E)
    s = oracle.sampler(lg, 0.8, 0, rows, 3, workers=WORKERS)
    assert np.abs(np_f(bufs.entropy)[rows] - s["H"]).max() < H_TOL
