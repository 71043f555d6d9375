"""GPU parity of the FP8 (E4M3) LM head.

* Quantisation: the E4M3 codes and fp32 scales of hidden rows and of W's
  vocabulary columns are bit-exact against the oracle's.
* The FP8 step: the oracle's quantised operands give fp64 logits
  (dec(x8) sx)(dec(w8t) sw)^T; the oracle step on those logits is the
  reference the GPU step is compared with (entropies 1e-4, tokens exact away
  from near-ties), at small, ragged and full sizes.
"""
import os

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import (DEV, H_TOL, check_step_against_oracle, np_f, np_i32, status_ok,
                            to_dev)

pytestmark = pytest.mark.gpu

WORKERS = os.cpu_count() or 1


def _rows_with_edges(rows, cols, seed):
    """bf16 rows of mixed magnitude, with a zero row, a row of negative zeros and
    tiny values (codes of -0), and a row with one large outlier."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-6, 6, (rows, 1)))
    if rows >= 4:
        x[1] = 0.0
        x[2] = -1e-30 * np.abs(rng.standard_normal(cols))
        x[2, 0] = -3.0
        x[3, cols // 2] = 1e4
    return dg_synth.f32_to_bf16_bits(x.astype(np.float32))


def _u8(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(1, 1), (7, 33), (256, 1024), (300, 2816), (5, 16384),
                                       (4, 16392)])
def test_quantize_rows_bit_exact(rows, cols):
    xb = _rows_with_edges(rows, cols, rows * 131 + cols)
    q_ref, s_ref = oracle.quantize_rows_e4m3(xb)
    q = torch.full((rows, cols), 0x55, dtype=torch.uint8, device=DEV)
    s = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    dg.quantize_rows_e4m3(to_dev(xb), q, s)
    torch.cuda.synchronize()
    assert np.array_equal(_u8(q), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("d,V", [(128, 64), (100, 1000), (1024, 16384), (2816, 4104)])
def test_quantize_weight_bit_exact(d, V):
    cfg = dg_synth.StepConfig("q", d=d, V=V, w_std=0.05, seed=d + V)
    wb = dg_synth.lm_weight(cfg)
    wb[:, 3] = 0                    # an all-zero column: codes 0, scale 1
    wb[5 % d, 7] = 0x4B80           # bf16 16777216: one large outlier
    w8_ref, s_ref = oracle.quantize_weight_e4m3(wb)
    w8 = torch.full((V, d), 0x55, dtype=torch.uint8, device=DEV)
    s = torch.full((V,), float("nan"), dtype=torch.float32, device=DEV)
    dg.quantize_weight_e4m3(to_dev(wb), w8, s)
    torch.cuda.synchronize()
    assert np.array_equal(_u8(w8), w8_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert s_ref[3] == 1.0 and not w8_ref[3].any()


def _fp8_step(cfg, xb, wb, k, seed, canvas0, prev, workers=1):
    B, L, d, V = cfg.B, cfg.L, cfg.d, cfg.V
    T = oracle.temperature(k, cfg.max_steps)
    x8, sx = oracle.quantize_rows_e4m3(xb, workers=workers)
    w8t, sw = oracle.quantize_weight_e4m3(wb, workers=workers)
    lg = oracle.logits_fp8(x8, sx, w8t, sw)
    ref = oracle.step(xb, wb, canvas0, prev, B, L, T, cfg.entropy_bound, seed, k,
                      cfg.stop_threshold, workers=workers, lg=lg)
    w8d = torch.empty((V, d), dtype=torch.uint8, device=DEV)
    swd = torch.empty((V,), dtype=torch.float32, device=DEV)
    dg.quantize_weight_e4m3(to_dev(wb), w8d, swd)
    p = dg.step_params(B, L, d, V, T, cfg.entropy_bound, cfg.stop_threshold, step=k, seed=seed)
    bufs = dg.StepBuffers(B, L, DEV)
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    bufs.prev_argmax.copy_(torch.from_numpy(prev))
    ws = dg.workspace(dg.denoise_step_fp8_workspace(p), DEV)
    x = to_dev(xb)
    dg.denoise_step_fp8(x, w8d, swd, p, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    return ref, bufs, (x, w8d, swd, p, ws)


@pytest.mark.parametrize("B,L,d,V,w_std,k", [(1, 256, 1024, 16384, 0.05, 0),   # the small step
                                             (2, 256, 256, 4096, 0.08, 2),     # two row blocks
                                             (1, 100, 128, 1000, 0.2, 1),      # ragged rows / vocab
                                             (5, 200, 384, 1104, 0.1, 7),      # canvases straddle blocks
                                             (1, 1024, 128, 64, 0.1, 3)])      # largest canvas, tiny V
@pytest.mark.parametrize("kernel", ["duo", "fused"])
def test_fp8_step_matches_oracle(B, L, d, V, w_std, k, kernel, monkeypatch):
    """Plain and fused tile schedules of the 2-SM FP8 LM head."""
    monkeypatch.setenv("DG_LM_KERNEL", kernel)
    cfg = dg_synth.StepConfig("f8", B=B, L=L, d=d, V=V, w_std=w_std, seed=13)
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    rng = np.random.default_rng(B * L + V)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    ref, bufs, (x, w8d, swd, p, ws) = _fp8_step(cfg, xb, wb, k, 9, canvas0, prev)
    check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)
    assert np.array_equal(np_i32(bufs.stop), ref["stop"])
    # deterministic
    H1 = np_f(bufs.entropy).copy()
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    dg.denoise_step_fp8(x, w8d, swd, p, bufs, ws)
    torch.cuda.synchronize()
    assert np.array_equal(np_f(bufs.entropy), H1)


def test_fp8_step_full_width_every_row(monkeypatch):
    """The full-width LM head (2816 x 262144, per-row logit scale U(0.5, 8)) on
    FP8 operands, every row against the oracle: the planned tile schedule,
    then the plain 256-column one on the same inputs."""
    cfg = dg_synth.CONFIGS["step_full"]
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    rng = np.random.default_rng(3)
    canvas0 = rng.integers(0, cfg.V, cfg.M).astype(np.int32)
    prev = rng.integers(0, cfg.V, cfg.M).astype(np.int32)
    monkeypatch.delenv("DG_LM_KERNEL", raising=False)
    ref, bufs, (x, w8d, swd, p, ws) = _fp8_step(cfg, xb, wb, 4, 21, canvas0, prev,
                                                workers=WORKERS)
    decided = check_step_against_oracle(bufs, ref, cfg.B, cfg.L, exact_tokens=False)
    assert np.abs(np_f(bufs.mean_entropy) - ref["mean_entropy"]).max() < H_TOL
    assert decided == 1
    monkeypatch.setenv("DG_LM_KERNEL", "duo")
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    bufs.prev_argmax.copy_(torch.from_numpy(prev))
    dg.denoise_step_fp8(x, w8d, swd, p, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    assert check_step_against_oracle(bufs, ref, cfg.B, cfg.L, exact_tokens=False) == 1


def test_fp8_step_constant_rows():
    """A zero hidden row (scale 1, codes 0) gives uniform logits: entropy ln V,
    argmax 0; a row of one repeated value quantises to one code (448)."""
    B, L, d, V = 1, 64, 256, 2048
    cfg = dg_synth.StepConfig("c8", B=B, L=L, d=d, V=V, w_std=0.1, seed=4)
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    xb[0] = 0
    xb[1] = 0x3F80   # 1.0
    rng = np.random.default_rng(0)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    ref, bufs, _ = _fp8_step(cfg, xb, wb, 2, 1, canvas0, prev)
    check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)
    H = np_f(bufs.entropy)
    assert abs(H[0] - np.log(V)) < H_TOL and int(np_i32(bufs.argmax)[0]) == 0
