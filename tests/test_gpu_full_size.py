"""GPU parity at the full sizes of the five synthetic workloads, in the launch
configuration the benchmark times (the default kernel plan for the device).

* full-width step: LM head 2816 x 262144 with per-row logit scale U(0.5, 8)
  against the fp64 oracle on every row (both LM-head kernels), attention with
  16/8 heads, head dim 256 and 4096 cached keys on sampled rows;
* batch sweep: the small step at 4 and 16 canvases (2048 cached keys), every
  row of the LM-head step and sampled attention rows;
* long context: attention over 32768 cached keys, sampled rows;
* block loop at 2816 x 262144: flat logits commit exactly one token per step
  for 48 steps; a three-step schedule matches the oracle's loop step by step;
  the 48-step converging loop is checked at its last steps against oracle
  steps recomputed from the same hidden states.

Oracle rows run on all host cores (rows are independent).
"""
import functools
import math
import os

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import (ATTN_TOL, DEV, H_TOL, MARGIN, acceptance_is_decided,
                            check_step_against_oracle, force_lm_kernel, np_f, np_i32, status_ok,
                            to_dev)

pytestmark = pytest.mark.gpu

WORKERS = os.cpu_count() or 1


@functools.lru_cache(maxsize=2)
def _weight_of(d, V, w_std, seed):
    return dg_synth.lm_weight(dg_synth.StepConfig("w", d=d, V=V, w_std=w_std, seed=seed))


def _weight(name):
    """The workload's W (drawn once per distinct shape / distribution / seed)."""
    c = dg_synth.CONFIGS[name]
    return _weight_of(c.d, c.V, c.w_std, c.seed)


# ------------------------------------------------------------------ single steps, every row
def _step_case(cfg, k, seed, kernel_env, monkeypatch):
    wb = _weight(cfg.name)
    xb = dg_synth.lm_hidden(cfg)
    B, L, d, V = cfg.B, cfg.L, cfg.d, cfg.V
    T = oracle.temperature(k, cfg.max_steps)
    rng = np.random.default_rng(k + 17)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    ref = oracle.step(xb, wb, canvas0, prev, B, L, T, cfg.entropy_bound, seed, k,
                      cfg.stop_threshold, workers=WORKERS)
    x, w = to_dev(xb), to_dev(wb)
    p = dg.step_params(B, L, d, V, T, cfg.entropy_bound, cfg.stop_threshold, step=k, seed=seed)
    ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
    results = []
    for env in kernel_env:
        force_lm_kernel(monkeypatch, env)
        bufs = dg.StepBuffers(B, L, DEV)
        bufs.canvas.copy_(torch.from_numpy(canvas0))
        bufs.prev_argmax.copy_(torch.from_numpy(prev))
        dg.denoise_step(x, w, p, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        decided = check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)
        assert np.array_equal(np_i32(bufs.stop), ref["stop"])
        assert np.abs(np_f(bufs.mean_entropy) - ref["mean_entropy"]).max() < H_TOL
        results.append((decided, np_f(bufs.entropy).copy()))
    force_lm_kernel(monkeypatch, None)
    return ref, results


def test_full_width_step_every_row(monkeypatch):
    """2816 x 262144 LM head: the planned kernel (2-SM UMMA pair on fused
    128-column schedule tiles, 8 epilogue warps), the same kernel on plain
    256-column tiles, with 16 epilogue warps, and the single-CTA LM-head
    kernel against the same oracle step."""
    cfg = dg_synth.CONFIGS["step_full"]
    ref, res = _step_case(cfg, k=3, seed=0, kernel_env=[None, "duo", "fused/16", "single"],
                          monkeypatch=monkeypatch)
    assert all(dec == 1 for dec, _ in res)
    # the per-row entropies span confident to uncertain rows
    assert ref["H"].min() < 0.05 and ref["H"].max() > 5.0


@pytest.mark.parametrize("name", ["batch4", "batch16"])
def test_batch_sweep_step_every_row(name, monkeypatch):
    cfg = dg_synth.CONFIGS[name]
    ref, res = _step_case(cfg, k=1, seed=0, kernel_env=[None], monkeypatch=monkeypatch)
    assert res[0][0] >= cfg.B // 2


# ------------------------------------------------------------------ attention, sampled rows
@pytest.mark.parametrize("name,stride", [("step_full", 7), ("batch4", 17), ("batch16", 61),
                                         ("long_context", 5)])
def test_attention_full_size_sampled_rows(name, stride):
    cfg = dg_synth.CONFIGS[name]
    B, L, P, Hq, Hkv, D = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D
    ai = dg_synth.attention_inputs(cfg)
    t = {k: to_dev(v) for k, v in ai.items()}
    out = torch.full_like(t["q"], float("nan"))
    scale = float(np.float32(1.0 / math.sqrt(D)))
    ws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    dg.canvas_attn(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out, scale, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    got_all = out.float().reshape(-1, D).cpu().numpy()
    assert np.isfinite(got_all).all()
    # sampled rows, plus the last row (ragged end of the sampling grid)
    rows = np.unique(np.append(np.arange(0, B * L * Hq, stride), B * L * Hq - 1))
    ref = oracle.attention_rows(ai["q"], ai["kp"], ai["vp"], ai["kc"], ai["vc"], B, L, P, Hq,
                                Hkv, D, scale, rows)
    err = np.abs(got_all[rows] - ref).max(axis=1) / np.abs(ref).max(axis=1)
    assert err.max() < ATTN_TOL, (err.max(), int(rows[err.argmax()]))


# ------------------------------------------------------------------ the block loop at full size
def _block_run(hs, wb, cfg, seed, max_steps, stride_steps=True):
    B, L, d, V = cfg.B, cfg.L, cfg.d, cfg.V
    p = dg.step_params(B, L, d, V, cfg.t_start, cfg.entropy_bound, cfg.stop_threshold, step=0,
                       seed=seed)
    bp = dg.block_params(max_steps, cfg.t_start, cfg.t_end, B * L * d if stride_steps else 0)
    bufs = dg.BlockBuffers(B, L, max_steps, DEV)
    ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
    dg.generate_block(to_dev(hs), to_dev(wb), p, bp, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    return bufs


def test_block_full_flat_logits_one_commit_per_step():
    """Zero hidden states at 2816 x 262144: every logit is 0, so every step
    accepts exactly one token, never stops, and the argmax is token 0."""
    cfg = dg_synth.CONFIGS["block_full"]
    wb = _weight("block_full")
    hid = np.zeros((cfg.L, cfg.d), np.uint16)
    bufs = _block_run(hid, wb, cfg, seed=0, max_steps=48, stride_steps=False)
    assert int(bufs.steps_taken[0]) == 48
    assert (np_i32(bufs.n_accepted_hist) == 1).all()
    assert (np_i32(bufs.argmax) == 0).all()
    assert abs(float(bufs.mean_entropy[0]) - math.log(cfg.V)) < H_TOL


def _block_hidden_all(cfg, wb, n):
    tg = dg_synth.block_targets(cfg)
    return np.stack([dg_synth.block_hidden(cfg, wb, tg, k) for k in range(n)]), tg


def test_block_full_three_step_schedule_matches_oracle():
    """The loop with a three-step schedule (T = 0.8, 0.6, 0.4) on the full-size
    converging workload against the oracle's loop: per-step commit counts where
    the acceptance is decided, and the final canvas and argmax where every
    decision of the run is clear of its margin."""
    cfg = dg_synth.CONFIGS["block_full"]
    wb = _weight("block_full")
    N = 3
    hs, _ = _block_hidden_all(cfg, wb, N)
    ref = oracle.block(lambda k: hs[k], wb, 1, cfg.L, cfg.entropy_bound, 5, max_steps=N,
                       workers=WORKERS)
    bufs = _block_run(hs, wb, cfg, seed=5, max_steps=N)
    hist = np_i32(bufs.n_accepted_hist)
    assert int(bufs.steps_taken[0]) == int(ref["steps"][0])
    all_clear = True
    for k, h in enumerate(ref["history"]):
        decided = acceptance_is_decided(h["H32"], int(h["n_accepted"][0]),
                                        float(h["boundary_gap"][0]))
        if decided:
            assert hist[k] == int(h["n_accepted"][0]), k
        acc = np.zeros(cfg.L, bool)
        acc[h["order"][0][: int(h["n_accepted"][0])]] = True
        all_clear &= (decided and bool((h["gumbel_margin"][acc] >= MARGIN).all())
                      and bool((h["argmax_margin"] >= MARGIN).all()))
    last = ref["history"][-1]
    assert abs(float(bufs.mean_entropy[0]) - float(last["mean_entropy"][0])) < H_TOL
    ok = last["argmax_margin"] >= MARGIN
    assert ok.mean() > 0.9
    assert np.array_equal(np_i32(bufs.argmax)[ok], ref["argmax"][ok])
    if all_clear:
        assert np.array_equal(np_i32(bufs.canvas), ref["canvas"])


def test_block_full_packed_weight_equals_rowmajor():
    """The full-size converging loop (48-step cap) as the benchmark runs it,
    on the packed weight: the same run as on W [d, V], bit for bit."""
    cfg = dg_synth.CONFIGS["block_full"]
    wb = _weight("block_full")
    hs, _ = _block_hidden_all(cfg, wb, cfg.max_steps)
    B, L, d, V = cfg.B, cfg.L, cfg.d, cfg.V
    w = to_dev(wb)
    hid = to_dev(hs)
    res = []
    for layout, ww in ((dg.W_ROWMAJOR, w), (dg.W_PACKED, dg.pack_lm_weight(w))):
        p = dg.step_params(B, L, d, V, cfg.t_start, cfg.entropy_bound, cfg.stop_threshold,
                           step=0, seed=5, w_layout=layout)
        bp = dg.block_params(cfg.max_steps, cfg.t_start, cfg.t_end, B * L * d)
        bufs = dg.BlockBuffers(B, L, cfg.max_steps, DEV)
        ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
        dg.generate_block(hid, ww, p, bp, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        res.append(bufs)
    a, b = res
    assert 2 <= int(a.steps_taken[0]) < cfg.max_steps
    for name in ("canvas", "argmax", "steps_taken", "mean_entropy", "n_accepted_hist"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_block_full_converging_final_steps_match_oracle():
    """The 48-step converging loop at full size.  The loop must stop before the
    cap (entropies fall with the step); at the step it stopped on, the oracle's
    step on the same hidden states and temperature gives the reported mean
    entropy and argmax, its stop test fires, and the argmax equals the
    oracle's argmax of the step before; at the step before that, the oracle's
    stop test does not fire (so the loop stopped neither early nor late)."""
    cfg = dg_synth.CONFIGS["block_full"]
    wb = _weight("block_full")
    N = cfg.max_steps
    hs, _ = _block_hidden_all(cfg, wb, N)
    bufs = _block_run(hs, wb, cfg, seed=7, max_steps=N)
    s = int(bufs.steps_taken[0])
    hist = np_i32(bufs.n_accepted_hist)
    assert 2 <= s < N
    assert (hist[:s] >= 1).all() and (hist[:s] <= cfg.L).all()
    last = s - 1

    def oracle_sampler(k):
        return oracle.sampler(oracle.logits(hs[k], wb), oracle.temperature(k, N), 7,
                              np.arange(cfg.L), k, workers=WORKERS)

    r = oracle_sampler(last)
    H32 = r["H"].astype(np.float32)
    mean_ref = float(H32.astype(np.float64).mean())
    assert abs(float(bufs.mean_entropy[0]) - mean_ref) < H_TOL
    assert mean_ref < cfg.stop_threshold + H_TOL
    ok = r["argmax_margin"] >= MARGIN
    assert ok.mean() > 0.9
    am = np_i32(bufs.argmax)
    assert np.array_equal(am[ok], r["argmax"][ok])
    r_prev = oracle_sampler(last - 1)
    ok &= r_prev["argmax_margin"] >= MARGIN
    assert np.array_equal(am[ok], r_prev["argmax"][ok])
    # the loop did not stop one step early: the oracle's stop test at step
    # last - 1 (against the argmax of step last - 2) does not fire, and the
    # decision is clear of the entropy tolerance
    if last >= 2:
        r_pp = oracle_sampler(last - 2)
        H32p = r_prev["H"].astype(np.float32)
        st = oracle.stop(r_prev["argmax"], r_pp["argmax"], H32p, last - 1, cfg.stop_threshold)
        assert st["stop"] == 0
        argmax_moved_clearly = bool(np.any((r_prev["argmax"] != r_pp["argmax"])
                                           & (r_prev["argmax_margin"] >= MARGIN)
                                           & (r_pp["argmax_margin"] >= MARGIN)))
        assert argmax_moved_clearly or st["mean_entropy"] >= cfg.stop_threshold + 2 * H_TOL


def test_canvas_step_full_width_equals_the_two_calls():
    """dg_canvas_step at the full-width step (no SMs set aside at this shape,
    the LM head on the same plan): the attention output and every step output
    equal those of dg_canvas_attn and dg_denoise_step, bit for bit."""
    cfg = dg_synth.CONFIGS["step_full"]
    B, L, P, Hq, Hkv, D, d, V = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D, cfg.d, cfg.V
    ai = dg_synth.attention_inputs(cfg)
    t = {k: to_dev(v) for k, v in ai.items()}
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(_weight("step_full"))
    scale = float(np.float32(1.0 / math.sqrt(D)))
    p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=4, seed=3)
    rng = np.random.default_rng(8)
    canvas0 = torch.from_numpy(rng.integers(0, V, B * L).astype(np.int32))
    got, ref = dg.StepBuffers(B, L, DEV), dg.StepBuffers(B, L, DEV)
    got.canvas.copy_(canvas0)
    ref.canvas.copy_(canvas0)
    out, ref_out = torch.empty_like(t["q"]), torch.empty_like(t["q"])
    ws = dg.workspace(dg.canvas_step_workspace(p, P, Hq, Hkv, D), DEV)
    dg.canvas_step(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out, scale, x, w, p, got, ws)
    aws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    sws = dg.workspace(dg.denoise_step_workspace(p), DEV)
    dg.canvas_attn(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], ref_out, scale, aws)
    dg.denoise_step(x, w, p, ref, sws)
    torch.cuda.synchronize()
    status_ok(ws)
    assert torch.equal(out, ref_out)
    for name in ("canvas", "argmax", "sample", "n_accepted", "stop", "prev_argmax"):
        assert np.array_equal(np_i32(getattr(got, name)), np_i32(getattr(ref, name))), name
    assert torch.equal(got.entropy, ref.entropy)


def _attn_case(cfg):
    ai = dg_synth.attention_inputs(cfg)
    return {k: to_dev(v) for k, v in ai.items()}


def test_canvas_step_fp8_full_width_equals_the_two_calls():
    """dg_canvas_step_fp8 at the full-width step: the attention output and every
    step output equal those of dg_canvas_attn and dg_denoise_step_fp8."""
    cfg = dg_synth.CONFIGS["step_full"]
    B, L, P, Hq, Hkv, D, d, V = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D, cfg.d, cfg.V
    t = _attn_case(cfg)
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(_weight("step_full"))
    w8 = torch.empty(V, d, dtype=torch.uint8, device=DEV)
    ws8 = torch.empty(V, dtype=torch.float32, device=DEV)
    dg.quantize_weight_e4m3(w, w8, ws8)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=2, seed=7)
    canvas0 = torch.from_numpy(np.random.default_rng(4).integers(0, V, B * L).astype(np.int32))
    got, ref = dg.StepBuffers(B, L, DEV), dg.StepBuffers(B, L, DEV)
    got.canvas.copy_(canvas0)
    ref.canvas.copy_(canvas0)
    out, ref_out = torch.empty_like(t["q"]), torch.empty_like(t["q"])
    ws = dg.workspace(dg.canvas_step_fp8_workspace(p, P, Hq, Hkv, D), DEV)
    dg.canvas_step_fp8(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out, scale, x, w8, ws8, p, got,
                       ws)
    aws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    sws = dg.workspace(dg.denoise_step_fp8_workspace(p), DEV)
    dg.canvas_attn(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], ref_out, scale, aws)
    dg.denoise_step_fp8(x, w8, ws8, p, ref, sws)
    torch.cuda.synchronize()
    status_ok(ws)
    assert torch.equal(out, ref_out)
    for name in ("canvas", "argmax", "sample", "n_accepted", "stop", "prev_argmax"):
        assert np.array_equal(np_i32(getattr(got, name)), np_i32(getattr(ref, name))), name
    assert torch.equal(got.entropy, ref.entropy)


def test_canvas_step_sc_full_width_equals_the_two_calls():
    """dg_canvas_step_sc at the full-width step on the packed weight: the
    attention output, every step output and the read-out equal those of
    dg_canvas_attn and dg_denoise_step_sc."""
    cfg = dg_synth.CONFIGS["step_full"]
    B, L, P, Hq, Hkv, D, d, V = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D, cfg.d, cfg.V
    t = _attn_case(cfg)
    x = to_dev(dg_synth.lm_hidden(cfg))
    wp = dg.pack_lm_weight(to_dev(_weight("step_full")))
    g = torch.Generator(device=DEV).manual_seed(12)
    table = (torch.randn(V, dg.SC_DIM, device=DEV, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=3, seed=8, w_layout=dg.W_PACKED)
    canvas0 = torch.from_numpy(np.random.default_rng(6).integers(0, V, B * L).astype(np.int32))
    got, ref = dg.StepBuffers(B, L, DEV), dg.StepBuffers(B, L, DEV)
    got.canvas.copy_(canvas0)
    ref.canvas.copy_(canvas0)
    out, ref_out = torch.empty_like(t["q"]), torch.empty_like(t["q"])
    sc_got = torch.empty(B * L, dg.SC_DIM, device=DEV)
    sc_ref = torch.empty(B * L, dg.SC_DIM, device=DEV)
    ws = dg.workspace(dg.canvas_step_sc_workspace(p, P, Hq, Hkv, D), DEV)
    dg.canvas_step_sc(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out, scale, x, wp, table, p, got,
                      sc_got, ws)
    aws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    sws = dg.workspace(dg.denoise_step_sc_workspace(p), DEV)
    dg.canvas_attn(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], ref_out, scale, aws)
    dg.denoise_step_sc(x, wp, table, p, ref, sc_ref, sws)
    torch.cuda.synchronize()
    status_ok(ws)
    assert torch.equal(out, ref_out)
    for name in ("canvas", "argmax", "sample", "n_accepted", "stop", "prev_argmax"):
        assert np.array_equal(np_i32(getattr(got, name)), np_i32(getattr(ref, name))), name
    assert torch.equal(got.entropy, ref.entropy)
    assert torch.equal(sc_got, sc_ref)
