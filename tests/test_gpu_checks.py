"""Device-side checks (dg_set_device_checks).  With the checks on, a normal
step, attention, encoder append and MoE layer report nothing and give the
same outputs, bit for bit, as with them off; a planted NaN among the logits,
an infinite query, or a sample outside the vocabulary is reported as
DG_ERR_DEVICE (and goes unreported with the checks off).  The planted inputs
are arithmetic only: no index the kernels use comes from them."""
import math

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import DEV, np_i32, status_ok, to_dev

pytestmark = pytest.mark.gpu

DG_ERR_DEVICE = 7


@pytest.fixture
def checks_on():
    dg.set_device_checks(True)
    try:
        yield
    finally:
        dg.set_device_checks(False)


def _canvas_step(cfg, seed):
    ai = dg_synth.attention_inputs(cfg)
    t = {k: to_dev(v) for k, v in ai.items()}
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(dg_synth.lm_weight(cfg))
    B, L, P, Hq, Hkv, D, d, V = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D, cfg.d, cfg.V
    p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=1, seed=seed)
    bufs = dg.StepBuffers(B, L, DEV)
    bufs.canvas.copy_(torch.from_numpy(oracle.init_canvas(B * L, V, seed)))
    out = torch.empty_like(t["q"])
    ws = dg.workspace(dg.canvas_step_workspace(p, P, Hq, Hkv, D), DEV)
    dg.canvas_step(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out,
                   float(np.float32(1.0 / math.sqrt(D))), x, w, p, bufs, ws)
    torch.cuda.synchronize()
    return bufs, out, ws


@pytest.mark.parametrize("name", ["step_small", "step_full"])
def test_checked_step_equals_unchecked_and_reports_nothing(name):
    cfg = dg_synth.CONFIGS[name]
    ref_bufs, ref_out, ref_ws = _canvas_step(cfg, 3)
    status_ok(ref_ws)
    dg.set_device_checks(True)
    try:
        assert dg.device_checks()
        bufs, out, ws = _canvas_step(cfg, 3)
    finally:
        dg.set_device_checks(False)
    assert not dg.device_checks()
    status_ok(ws)
    assert torch.equal(bufs.readback, ref_bufs.readback)
    assert torch.equal(bufs.entropy, ref_bufs.entropy)
    assert torch.equal(out, ref_out)


def test_checked_moe_equals_unchecked(checks_on):
    cfg = dg_synth.MoeConfig("moe_chk", M=200, d=512, f=256, E=16, top_k=4, alpha=1.0, seed=4)
    a = dg_synth.moe_inputs(cfg)
    t = {k: to_dev(v) for k, v in a.items() if k in ("x", "wr", "wg", "wu", "wd")}
    p = dg.moe_params(cfg.M, cfg.d, cfg.f, cfg.E, cfg.top_k)
    outs = []
    for on in (True, False):
        dg.set_device_checks(on)
        ws = dg.workspace(dg.moe_ffn_workspace(p), DEV)
        out = torch.empty(cfg.M, cfg.d, dtype=torch.float32, device=DEV)
        dg.moe_ffn(t["x"], t["wr"], t["wg"], t["wu"], t["wd"], out, p, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_checked_encoder_append_reports_nothing(checks_on):
    cfg = dg_synth.StepConfig("enc_chk", B=1, L=64, Hq=4, Hkv=2, D=128, P=200, seed=6)
    B, L, P, Hq, Hkv, D = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D
    ai = dg_synth.attention_inputs(cfg)
    kc = torch.zeros(B, P + L, Hkv, D, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kc[:, :P] = dg.bf16_from_bits(ai["kp"])
    vc[:, :P] = dg.bf16_from_bits(ai["vp"])
    out = torch.empty(B, L, Hq, D, dtype=torch.bfloat16, device=DEV)
    ws = dg.workspace(dg.encoder_append_workspace(B, L, P, Hq, Hkv, D), DEV)
    dg.encoder_append(to_dev(ai["q"]), kc, vc, P, to_dev(ai["kc"]), to_dev(ai["vc"]), out,
                      1.0 / math.sqrt(D), ws)
    torch.cuda.synchronize()
    status_ok(ws)


def _sampler_status(logits, B, L, V):
    p = dg.step_params(B, L, 64, V, 0.8, 0.1, 0.005, step=1, seed=9)
    bufs = dg.StepBuffers(B, L, DEV)
    ws = dg.workspace(dg.sampler_workspace(p), DEV)
    dg.sampler_from_logits(torch.from_numpy(logits).to(DEV), p, bufs, ws)
    torch.cuda.synchronize()
    return dg.read_device_status(ws), bufs


def test_nan_logits_are_reported_only_with_checks():
    B, L, V = 1, 64, 512
    logits = np.random.default_rng(1).standard_normal((B * L, V)).astype(np.float32)
    logits[7, :] = np.nan            # one row with no ordered logit at all
    assert _sampler_status(logits, B, L, V)[0] == 0
    dg.set_device_checks(True)
    try:
        st, bufs = _sampler_status(logits, B, L, V)
    finally:
        dg.set_device_checks(False)
    assert st == DG_ERR_DEVICE
    # the offending row's indices were replaced by 0 before they were stored
    assert int(np_i32(bufs.sample)[7]) == 0 and int(np_i32(bufs.argmax)[7]) == 0
    assert (np_i32(bufs.canvas) >= 0).all() and (np_i32(bufs.canvas) < V).all()


def test_infinite_query_is_reported_with_checks(checks_on):
    cfg = dg_synth.StepConfig("attn_chk", B=1, L=128, Hq=4, Hkv=1, D=128, P=256, seed=2)
    B, L, P, Hq, Hkv, D = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D
    ai = dg_synth.attention_inputs(cfg)
    t = {k: to_dev(v) for k, v in ai.items()}
    out = torch.empty_like(t["q"])
    ws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    dg.canvas_attn(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out, 1.0 / math.sqrt(D), ws)
    torch.cuda.synchronize()
    status_ok(ws)
    q = t["q"].clone()
    q[0, 5, 1, 3] = float("inf")
    dg.canvas_attn(q, t["kp"], t["vp"], t["kc"], t["vc"], out, 1.0 / math.sqrt(D), ws)
    torch.cuda.synchronize()
    assert dg.read_device_status(ws) == DG_ERR_DEVICE


def test_sample_outside_the_vocabulary_is_reported_and_replaced(checks_on):
    B, L, V = 1, 32, 1000
    H = torch.full((B * L,), 0.01, dtype=torch.float32, device=DEV)   # every position accepted
    sample = torch.arange(B * L, dtype=torch.int32, device=DEV)
    sample[4] = V + 17
    argmax = torch.zeros(B * L, dtype=torch.int32, device=DEV)
    p = dg.step_params(B, L, 64, V, 0.8, 100.0, 0.005, step=1, seed=1)
    bufs = dg.StepBuffers(B, L, DEV)
    ws = dg.workspace(256, DEV)
    dg.accept_renoise(H, sample, argmax, p, bufs, ws)
    torch.cuda.synchronize()
    assert dg.read_device_status(ws) == DG_ERR_DEVICE
    canvas = np_i32(bufs.canvas)
    assert canvas[4] == 0 and canvas[5] == 5


def test_checked_block_loop_equals_unchecked():
    """The block loop keeps one graph per setting of the checks: both give the
    same run, and the checked one reports nothing."""
    cfg = dg_synth.StepConfig("blk_chk", L=64, d=256, V=2048, w_std=0.02, seed=18)
    wb = dg_synth.lm_weight(cfg)
    tg = dg_synth.block_targets(cfg)
    N = 48
    hs = to_dev(np.stack([dg_synth.block_hidden(cfg, wb, tg, k) for k in range(N)]))
    w = to_dev(wb)
    p = dg.step_params(1, cfg.L, cfg.d, cfg.V, 0.8, 0.1, 0.005, step=0, seed=9)
    bp = dg.block_params(N, 0.8, 0.4, cfg.L * cfg.d)
    ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
    bufs = dg.BlockBuffers(1, cfg.L, N, DEV)   # the same buffers: one graph per setting
    runs = []
    for on in (False, True, False):
        dg.set_device_checks(on)
        try:
            dg.generate_block(hs, w, p, bp, bufs, ws)
            torch.cuda.synchronize()
        finally:
            dg.set_device_checks(False)
        status_ok(ws)
        runs.append({n: getattr(bufs, n).clone()
                     for n in ("steps_taken", "canvas", "argmax", "n_accepted_hist")})
    for r in runs[1:]:
        for n, v in r.items():
            assert torch.equal(v, runs[0][n]), n
