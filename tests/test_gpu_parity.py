"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bit-exact: the fp32 log, Gumbel noise, samples and argmax on identical fp32
logits, the acceptance/renoise/stop stage on identical entropies.  Within
tolerance: entropies (1e-4 absolute), attention outputs (2e-2 of the row's
largest magnitude).  Tokens from the fused GEMM path are compared where the
oracle's margins are above 1e-3.
"""
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


# ------------------------------------------------------------------ primitives
def test_logf_bit_exact():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.uniform(5.9e-8, 1.0, 6000), rng.uniform(1.0, 17.0, 6000),
        np.exp(rng.uniform(-40, 40, 6000)),
        np.array([1.0, 2.0, 0.5, 0.70710677, 0.70710683, 1.4142135, 1.4142137, 16.635532,
                  5.9604645e-08, 0.99999994, 1.0000001]),
    ]).astype(np.float32)
    x = torch.from_numpy(xs).to(DEV)
    y = torch.empty_like(x)
    dg.logf_eval(x, y)
    got = y.cpu().numpy()
    ref = np.array([oracle.logf(float(v)) for v in xs], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("seed,row,step,v0,n", [(0, 0, 0, 0, 4096),
                                                (123456789012345, 77, 5, 13, 3001),
                                                (2**64 - 1, 2**32 - 1, 47, 262144 - 1000, 1000)])
def test_gumbel_bit_exact(seed, row, step, v0, n):
    out = torch.empty(n, dtype=torch.float32, device=DEV)
    dg.gumbel_fill(seed, row, step, v0, n, out)
    ref = oracle.gumbel_fill(seed, row, step, v0, n)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ acceptance / renoise / stop
def _random_entropies(rng, L, kind):
    if kind == "exp":
        return rng.exponential(0.03, L)
    if kind == "mixed":
        h = rng.exponential(1.0, L) * rng.choice([1e-4, 1e-2, 1.0, 5.0], L)
        h[rng.integers(0, L, 5)] = 0.0
        return h
    if kind == "ties":
        return rng.choice([0.0, 0.01, 0.02, 0.5], L)
    if kind == "flat":
        return np.full(L, math.log(16384.0))
    raise ValueError(kind)


@pytest.mark.parametrize("B,L,kind", [(1, 256, "exp"), (3, 256, "mixed"), (2, 100, "ties"),
                                      (1, 1024, "exp"), (1, 1, "mixed"), (2, 256, "flat"),
                                      (4, 37, "exp")])
def test_accept_renoise_stop_bit_exact(B, L, kind):
    rng = np.random.default_rng(L * 7 + B)
    V, b, seed, step = 16384, 0.1, 99, 3
    H = np.stack([_random_entropies(rng, L, kind) for _ in range(B)]).astype(np.float32)
    if kind == "mixed":
        H[0] = np.float32(1e-4)   # canvas 0: confident, low mean entropy
    sample = rng.integers(0, V, (B, L)).astype(np.int32)
    argmax = rng.integers(0, V, (B, L)).astype(np.int32)
    prev = argmax.copy()
    if B > 1:
        prev[1, L // 2] += 1      # canvas 1: argmax changed -> no stop
    canvas = rng.integers(0, V, (B, L)).astype(np.int32)

    p = dg.step_params(B, L, 64, V, 0.8, b, 0.005, step=step, seed=seed)
    bufs = dg.StepBuffers(B, L, DEV)
    bufs.canvas.copy_(torch.from_numpy(canvas.reshape(-1)))
    bufs.prev_argmax.copy_(torch.from_numpy(prev.reshape(-1)))
    ws = dg.workspace(4096, DEV)
    dg.accept_renoise(torch.from_numpy(H.reshape(-1)).to(DEV),
                      torch.from_numpy(sample.reshape(-1)).to(DEV),
                      torch.from_numpy(argmax.reshape(-1)).to(DEV), p, bufs, ws)
    torch.cuda.synchronize()
    for bb in range(B):
        r = oracle.accept_renoise(H[bb], sample[bb], canvas[bb], V, b, seed, bb * L, step)
        s = oracle.stop(argmax[bb], prev[bb], H[bb], step)
        sl = slice(bb * L, (bb + 1) * L)
        assert np.array_equal(np_i32(bufs.canvas)[sl], r["canvas"])
        assert np.array_equal(bufs.accepted.cpu().numpy()[sl], r["accepted"])
        assert int(bufs.n_accepted[bb]) == r["n_accepted"]
        assert int(bufs.stop[bb]) == s["stop"]
        assert abs(float(bufs.mean_entropy[bb]) - s["mean_entropy"]) <= 1e-6 * max(1, s["mean_entropy"])
        assert np.array_equal(np_i32(bufs.prev_argmax)[sl], argmax[bb])
    if kind == "mixed" and L > 1:
        assert int(bufs.stop[0]) == 1 and int(bufs.n_accepted[0]) == L
    status_ok(ws)


def _edge_entropies(kind, L, b):
    """Entropies around the acceptance's in-bound set {H <= b}: its edges."""
    f = np.float32
    bf = f(b)
    h = np.full(L, f(2.0))
    if kind == "at_bound":        # H exactly b (inside) and the next float up (outside)
        h[::3] = bf
        h[1::3] = np.nextafter(bf, f(1e9))
        h[5] = f(0.0)
    elif kind == "one_out_taken":   # all but one inside, summing to 0: the outside key commits too
        h[:] = f(0.0)
        h[L // 2] = f(7.5)
    elif kind == "one_out_not":     # all but one inside, summing past b
        h[:] = f(0.01)
        h[L // 3] = f(7.5)
    elif kind == "ties_out":        # none inside; ties among the smallest outside keys
        h[:] = f(0.7)
        h[[9, 4, 30]] = f(0.3)
    elif kind == "all_inside":
        h[:] = f(b / L)
        h[::7] = f(0.0)
    elif kind == "inside_ties":     # ties inside the set and at its last committed entry
        h[:] = f(3.0)
        h[:L // 2] = np.tile(np.array([0.02, 0.0, 0.02, 0.04], np.float32), L)[:L // 2]
    elif kind == "zero_bound":      # b = 0: only exact zeros are inside
        h[::4] = f(0.0)
    else:
        raise ValueError(kind)
    return h


@pytest.mark.parametrize("kind,L,b", [("at_bound", 256, 0.1), ("one_out_taken", 256, 0.1),
                                      ("one_out_not", 256, 0.1), ("ties_out", 64, 0.1),
                                      ("all_inside", 1024, 0.1), ("inside_ties", 100, 0.1),
                                      ("zero_bound", 256, 0.0), ("at_bound", 33, 0.25)])
def test_accept_in_bound_set_edges(kind, L, b):
    """The acceptance orders only the positions within the bound (and the
    smallest key past it): its membership edge, the outside key that commits
    or not, ties inside and outside, and b = 0 -- against the oracle's full
    sort, bit for bit."""
    rng = np.random.default_rng(sum(map(ord, kind)) * 1009 + L)
    V, seed, step = 4096, 5, 2
    H = _edge_entropies(kind, L, b)[None, :]
    sample = rng.integers(0, V, (1, L)).astype(np.int32)
    argmax = rng.integers(0, V, (1, L)).astype(np.int32)
    p = dg.step_params(1, L, 64, V, 0.8, b, 0.005, step=step, seed=seed)
    bufs = dg.StepBuffers(1, L, DEV)
    bufs.prev_argmax.copy_(torch.from_numpy(argmax.reshape(-1)))
    ws = dg.workspace(4096, DEV)
    dg.accept_renoise(torch.from_numpy(H.reshape(-1)).to(DEV),
                      torch.from_numpy(sample.reshape(-1)).to(DEV),
                      torch.from_numpy(argmax.reshape(-1)).to(DEV), p, bufs, ws)
    torch.cuda.synchronize()
    r = oracle.accept_renoise(H[0], sample[0], np.zeros(L, np.int32), V, np.float32(b), seed, 0, step)
    s = oracle.stop(argmax[0], argmax[0], H[0], step)
    assert int(bufs.n_accepted[0]) == r["n_accepted"]
    assert np.array_equal(bufs.accepted.cpu().numpy(), r["accepted"])
    assert np.array_equal(np_i32(bufs.canvas), r["canvas"])
    assert int(bufs.stop[0]) == s["stop"]
    assert abs(float(bufs.mean_entropy[0]) - s["mean_entropy"]) <= 1e-6 * max(1, s["mean_entropy"])
    if kind == "one_out_taken":
        assert r["n_accepted"] == L
    if kind == "one_out_not":
        assert r["accepted"][L // 3] == 0
    if kind == "ties_out":
        assert r["n_accepted"] == 1 and r["accepted"][4] == 1
    status_ok(ws)


def test_accept_step0_never_stops():
    L, V = 64, 1024
    p = dg.step_params(1, L, 64, V, 0.8, 0.1, 0.005, step=0, seed=1)
    bufs = dg.StepBuffers(1, L, DEV)
    am = torch.arange(L, dtype=torch.int32, device=DEV)
    bufs.prev_argmax.copy_(am)
    ws = dg.workspace(4096, DEV)
    dg.accept_renoise(torch.zeros(L, device=DEV), am, am, p, bufs, ws)
    torch.cuda.synchronize()
    assert int(bufs.stop[0]) == 0 and int(bufs.n_accepted[0]) == L


# ------------------------------------------------------------------ sampler on identical fp32 logits


@pytest.mark.parametrize("B,L,V,scale", [(1, 256, 16384, 1.0), (2, 256, 4096, 4.0),
                                         (1, 64, 1000, 2.0), (3, 100, 2048, 0.5),
                                         (1, 48, 262144, 6.0), (1, 32, 262144, 0.05)])
def test_sampler_from_logits(B, L, V, scale):
    rng = np.random.default_rng(V + L)
    logits = (rng.standard_normal((B * L, V)) * scale
              * rng.uniform(0.2, 3.0, (B * L, 1))).astype(np.float32)
    logits[0, 5] = logits[0, 7] = logits[0].max() + 1.0       # tie -> lower index wins
    T, b, seed, k = 0.8, 0.1, 2024, 1
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    p = dg.step_params(B, L, 64, V, T, b, 0.005, step=k, seed=seed)
    bufs = dg.StepBuffers(B, L, DEV)
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    bufs.prev_argmax.copy_(torch.from_numpy(prev))
    ws = dg.workspace(dg.sampler_workspace(p), DEV)
    dg.sampler_from_logits(torch.from_numpy(logits).to(DEV), p, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    s = oracle.sampler(logits.astype(np.float64), T, seed, np.arange(B * L), k)
    ref = dict(s)
    ref["canvas"] = np.zeros(B * L, np.int32)
    ref["accepted"] = np.zeros(B * L, np.uint8)
    ref["n_accepted"] = np.zeros(B, np.int32)
    ref["boundary_gap"] = np.zeros(B)
    Hf = s["H"].astype(np.float32)
    for bb in range(B):
        sl = slice(bb * L, (bb + 1) * L)
        a = oracle.accept_renoise(Hf[sl], s["sample"][sl], canvas0[sl], V, b, seed, bb * L, k)
        ref["canvas"][sl], ref["accepted"][sl] = a["canvas"], a["accepted"]
        ref["n_accepted"][bb], ref["boundary_gap"][bb] = a["n_accepted"], a["boundary_gap"]
    assert int(np_i32(bufs.argmax)[0]) == 5
    check_step_against_oracle(bufs, ref, B, L, exact_tokens=True)


# ------------------------------------------------------------------ fused LM head (tcgen05 GEMM + epilogue)
@pytest.mark.parametrize("B,L,d,V,w_std,k", [(1, 256, 1024, 16384, 0.05, 0),   # the small step
                                             (2, 256, 256, 4096, 0.08, 2),     # two row blocks
                                             (1, 100, 128, 1000, 0.2, 1),      # ragged rows / vocab
                                             (3, 64, 512, 8192, 0.05, 5)])
def test_denoise_step_matches_oracle(B, L, d, V, w_std, k):
    cfg = dg_synth.StepConfig("t", B=B, L=L, d=d, V=V, w_std=w_std, seed=11)
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    T, b, seed = oracle.temperature(k, 48), 0.1, 5
    rng = np.random.default_rng(1)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    p = dg.step_params(B, L, d, V, T, b, 0.005, step=k, seed=seed)
    bufs = dg.StepBuffers(B, L, DEV)
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    bufs.prev_argmax.copy_(torch.from_numpy(prev))
    ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
    x, w = to_dev(xb), to_dev(wb)
    dg.denoise_step(x, w, p, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    ref = oracle.step(xb, wb, canvas0, prev, B, L, T, b, seed, k)
    check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)
    # repeat: same result (deterministic)
    H1 = np_f(bufs.entropy).copy()
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    dg.denoise_step(x, w, p, bufs, ws)
    torch.cuda.synchronize()
    assert np.array_equal(np_f(bufs.entropy), H1)


@pytest.mark.parametrize("kernel", [None, "single", "duo", "fused", "duo/8", "fused/16"])
@pytest.mark.parametrize("B,L,d,V", [(1, 1024, 64, 64),      # largest canvas, one k block, tiny V
                                     (2, 1, 128, 2048),      # one position per canvas
                                     (5, 200, 192, 1104)])   # canvases straddling row blocks
def test_denoise_step_edge_shapes(kernel, B, L, d, V, monkeypatch):
    """Edge shapes through every LM-head kernel (None = the planner's choice;
    "/8", "/16": the 2-SM kernel's epilogue width forced against the
    planner's, which takes 8 warps for one row block and 16 for several)."""
    force_lm_kernel(monkeypatch, kernel)
    cfg = dg_synth.StepConfig("e", B=B, L=L, d=d, V=V, w_std=0.1, seed=23)
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    T, b, seed, k = oracle.temperature(7, 48), 0.1, 17, 7
    rng = np.random.default_rng(B + L)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    p = dg.step_params(B, L, d, V, T, b, 0.005, step=k, seed=seed)
    bufs = dg.StepBuffers(B, L, DEV)
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    bufs.prev_argmax.copy_(torch.from_numpy(prev))
    ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
    dg.denoise_step(to_dev(xb), to_dev(wb), p, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    ref = oracle.step(xb, wb, canvas0, prev, B, L, T, b, seed, k)
    check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)


@pytest.mark.parametrize("kernel", ["duo", "fused", "fused/8"])
def test_shared_row_bounds_across_launches(kernel, monkeypatch):
    """The 2-SM LM head lets its units share per-row lower bounds on the best
    Gumbel score within a launch (to skip noise that cannot win).  Several
    steps on one workspace, with a status clear between them, must each match
    the oracle, and a repeated step must reproduce its outputs bit for bit
    (the shared bounds change which columns are skipped, never the result).
    Two row blocks, mixed per-row logit scales as in the full-width step."""
    force_lm_kernel(monkeypatch, kernel)
    B, L, d, V = 2, 256, 256, 65536
    cfg = dg_synth.StepConfig("rb", B=B, L=L, d=d, V=V, w_std=0.06, row_scale=(0.5, 8.0),
                              seed=31)
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    x, w = to_dev(xb), to_dev(wb)
    rng = np.random.default_rng(7)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    p0 = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=0, seed=3)
    ws = dg.workspace(dg.denoise_step_workspace(p0), DEV)
    lg = oracle.logits(xb, wb)
    first = {}
    for rep in range(2):
        for k in (0, 1, 5):
            T = oracle.temperature(k, 48)
            p = dg.step_params(B, L, d, V, T, 0.1, 0.005, step=k, seed=3)
            bufs = dg.StepBuffers(B, L, DEV)
            bufs.canvas.copy_(torch.from_numpy(canvas0))
            bufs.prev_argmax.copy_(torch.from_numpy(prev))
            dg.denoise_step(x, w, p, bufs, ws)
            torch.cuda.synchronize()
            status_ok(ws)
            out = (np_f(bufs.entropy), np_i32(bufs.sample), np_i32(bufs.argmax),
                   np_i32(bufs.canvas))
            if rep == 0:
                ref = oracle.step(xb, wb, canvas0, prev, B, L, T, 0.1, 3, k,
                                  workers=os.cpu_count() or 1, lg=lg)
                check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)
                first[k] = out
            else:
                for a_, b_ in zip(out, first[k]):
                    assert np.array_equal(a_, b_)
        dg.read_device_status(ws, clear=True)


def test_lm_head_plan_epilogue_width(monkeypatch):
    """The 2-SM kernel runs 8 epilogue warps on one 256-row block and 16 on
    several; DG_LM_EPI forces either; the other kernels report 0."""
    force_lm_kernel(monkeypatch, None)
    one = dg.lm_head_plan(256, 2816, 262144)
    assert one["kind"] in (2, 3) and one["epilogue_warps"] == 8
    assert one["kernel"] == "lm_head_duo_kernel"
    many = dg.lm_head_plan(4096, 2816, 262144)
    assert many["kind"] in (2, 3) and many["epilogue_warps"] == 16
    assert many["kernel"] == "lm_head_duo_wide_kernel"
    force_lm_kernel(monkeypatch, "fused/16")
    assert dg.lm_head_plan(256, 2816, 262144)["epilogue_warps"] == 16
    force_lm_kernel(monkeypatch, "duo/8")
    assert dg.lm_head_plan(4096, 2816, 262144)["epilogue_warps"] == 8
    force_lm_kernel(monkeypatch, "single")
    assert dg.lm_head_plan(256, 2816, 262144)["epilogue_warps"] == 0


def test_canvas_step_plan_on_the_device_equals_the_host_plan(monkeypatch):
    """sms = 0 plans for the current device: the same plan as the host-side
    query given the device's SM count."""
    force_lm_kernel(monkeypatch, None)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B, P, Hq, Hkv, D, d, V in [(1, 256, 4, 1, 128, 1024, 16384),
                                   (1, 4096, 16, 8, 256, 2816, 262144)]:
        p = dg.step_params(B, 256, d, V, 0.8)
        assert dg.canvas_step_plan(p, P, Hq, Hkv, D, 0) == \
            dg.canvas_step_plan(p, P, Hq, Hkv, D, sms)


def test_denoise_step_uniform_and_one_hot_rows():
    """Zero hidden rows give uniform logits (H = ln V, argmax 0); a row aligned
    with one vocabulary column at large scale gives H ~ 0 at that column."""
    L, d, V = 256, 128, 4096
    x = np.zeros((L, d), np.float32)
    w = np.zeros((d, V), np.float32)
    for i in range(0, L, 2):          # odd rows stay zero -> uniform
        x[i, i // 2] = 1.0
        w[i // 2, (37 * i) % V] = 200.0
    xb, wb = dg_synth.f32_to_bf16_bits(x), dg_synth.f32_to_bf16_bits(w)
    p = dg.step_params(1, L, d, V, 0.8, 0.1, 0.005, step=0, seed=3)
    bufs = dg.StepBuffers(1, L, DEV)
    ws = dg.workspace(dg.denoise_step_workspace(p), DEV)
    dg.denoise_step(to_dev(xb), to_dev(wb), p, bufs, ws)
    torch.cuda.synchronize()
    H, am = np_f(bufs.entropy), np_i32(bufs.argmax)
    assert np.abs(H[1::2] - math.log(V)).max() < H_TOL
    assert (am[1::2] == 0).all()
    assert np.abs(H[0::2]).max() < H_TOL
    assert np.array_equal(am[0::2], np.array([(37 * i) % V for i in range(0, L, 2)]))
    assert np.array_equal(np_i32(bufs.sample)[0::2], am[0::2])


# ------------------------------------------------------------------ canvas attention
def _attn_case(B, L, P, Hq, Hkv, D, seed=0, row_stride=1):
    cfg = dg_synth.StepConfig("a", B=B, L=L, P=P, Hq=Hq, Hkv=Hkv, D=D, seed=seed)
    ai = dg_synth.attention_inputs(cfg)
    t = {k: to_dev(v) for k, v in ai.items()}
    out = torch.full_like(t["q"], float("nan"))
    scale = float(np.float32(1.0 / math.sqrt(D)))
    ws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    dg.canvas_attn(t["q"], t["kp"] if P else None, t["vp"] if P else None, t["kc"], t["vc"],
                   out, scale, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    rows = np.arange(0, B * L * Hq, row_stride)
    ref = oracle.attention_rows(ai["q"], ai["kp"], ai["vp"], ai["kc"], ai["vc"], B, L, P, Hq, Hkv,
                                D, scale, rows)
    got = out.float().reshape(-1, D).cpu().numpy()[rows]
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max(axis=1) / np.abs(ref).max(axis=1)
    assert err.max() < ATTN_TOL, (err.max(), int(rows[err.argmax()]))
    return err.max()


@pytest.mark.parametrize("B,L,P,Hq,Hkv,D,stride", [
    (1, 256, 256, 4, 1, 128, 1),      # the small step's attention
    (2, 100, 37, 4, 2, 128, 1),       # ragged canvas and prefix
    (1, 64, 0, 2, 1, 128, 1),         # no cached prefix
    (1, 48, 300, 16, 8, 256, 1),      # head dim 256, G = 2, ragged
    (1, 256, 4096, 4, 1, 128, 5),     # many key tiles -> split-KV + combine
    (2, 256, 1000, 16, 8, 256, 9),    # head dim 256 with splits
    (1, 16, 5, 8, 1, 128, 1),         # G = 8, tiny
])
def test_canvas_attn_matches_oracle(B, L, P, Hq, Hkv, D, stride):
    _attn_case(B, L, P, Hq, Hkv, D, seed=B + L + P, row_stride=stride)


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("B,L,P,Hq,Hkv,D,stride", [
    (1, 256, 256, 4, 1, 128, 1),      # head dim 128
    (2, 100, 37, 4, 2, 128, 1),       # ragged canvas and prefix, odd query-tile count
    (1, 48, 300, 16, 8, 256, 1),      # head dim 256, one query tile per kv head
    (2, 256, 1000, 16, 8, 256, 9),    # head dim 256 with splits
])
def test_canvas_attn_both_kernels(kernel, B, L, P, Hq, Hkv, D, stride, monkeypatch):
    """One CTA per query tile and 2-CTA clusters with 2-SM UMMAs, whichever the
    planner picks by default for the head dim."""
    monkeypatch.setenv("DG_ATTN_KERNEL", kernel)
    _attn_case(B, L, P, Hq, Hkv, D, seed=7 + B + L, row_stride=stride)


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("B,L,P,Hq,Hkv,D", [(1, 1, 5, 16, 1, 128),    # one position, G = 16
                                          (1, 1, 0, 2, 2, 256),      # no prefix, G = 1
                                          (3, 7, 129, 8, 4, 256)])   # ragged everything
def test_canvas_attn_edge_shapes(kernel, B, L, P, Hq, Hkv, D, monkeypatch):
    monkeypatch.setenv("DG_ATTN_KERNEL", kernel)
    _attn_case(B, L, P, Hq, Hkv, D, seed=3 + P, row_stride=1)


def test_canvas_attn_pair_split_counts_on_one_workspace(monkeypatch):
    """The 2-SM kernel with 2, 3 and 4 key splits, launched in turn on one
    workspace: every launch must match the oracle, and a repeated launch with
    the same split count must reproduce its output bit for bit (nothing a
    launch leaves in the workspace changes the next one)."""
    monkeypatch.setenv("DG_ATTN_KERNEL", "pair")
    B, L, P, Hq, Hkv, D = 2, 256, 1000, 16, 8, 256
    cfg = dg_synth.StepConfig("a", B=B, L=L, P=P, Hq=Hq, Hkv=Hkv, D=D, seed=13)
    ai = dg_synth.attention_inputs(cfg)
    t = {k: to_dev(v) for k, v in ai.items()}
    scale = float(np.float32(1.0 / math.sqrt(D)))
    ws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    rows = np.arange(0, B * L * Hq, 7)
    ref = oracle.attention_rows(ai["q"], ai["kp"], ai["vp"], ai["kc"], ai["vc"], B, L, P, Hq, Hkv,
                                D, scale, rows)
    first = {}
    for splits in (4, 2, 3, 4, 2):
        monkeypatch.setenv("DG_ATTN_SPLITS", str(splits))
        out = torch.full_like(t["q"], float("nan"))
        dg.canvas_attn(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out, scale, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        got = out.float().reshape(-1, D).cpu().numpy()
        assert np.isfinite(got).all()
        err = np.abs(got[rows] - ref).max(axis=1) / np.abs(ref).max(axis=1)
        assert err.max() < ATTN_TOL, (splits, err.max())
        if splits in first:
            assert np.array_equal(got, first[splits])
        first[splits] = got


def test_canvas_attn_constant_values_and_zero_keys():
    """Constant value rows -> every output equals that row; zero keys -> mean of values."""
    B, L, P, Hq, Hkv, D = 1, 128, 200, 4, 1, 128
    cfg = dg_synth.StepConfig("a", B=B, L=L, P=P, Hq=Hq, Hkv=Hkv, D=D, seed=4)
    ai = dg_synth.attention_inputs(cfg)
    row = dg_synth.f32_to_bf16_bits(np.linspace(-2, 2, D).astype(np.float32))
    vp = np.broadcast_to(row, ai["vp"].shape).copy()
    vc = np.broadcast_to(row, ai["vc"].shape).copy()
    out = torch.empty(B, L, Hq, D, dtype=torch.bfloat16, device=DEV)
    ws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    dg.canvas_attn(to_dev(ai["q"]), to_dev(ai["kp"]), to_dev(vp), to_dev(ai["kc"]), to_dev(vc),
                   out, 0.1, ws)
    torch.cuda.synchronize()
    expect = torch.from_numpy(dg_synth.bf16_bits_to_f32(row))
    assert (out.float().cpu().reshape(-1, D) - expect).abs().max() < 2e-2
    zk = np.zeros_like(ai["kp"]), np.zeros_like(ai["kc"])
    dg.canvas_attn(to_dev(ai["q"]), to_dev(zk[0]), to_dev(ai["vp"]), to_dev(zk[1]), to_dev(ai["vc"]),
                   out, 0.1, ws)
    torch.cuda.synchronize()
    allv = np.concatenate([dg_synth.bf16_bits_to_f32(ai["vp"])[0, :, 0],
                           dg_synth.bf16_bits_to_f32(ai["vc"])[0, :, 0]]).astype(np.float64).mean(0)
    got = out.float().cpu().numpy().reshape(-1, D)
    assert np.abs(got - allv[None]).max() < 2e-2 * np.abs(allv).max() + 2e-3


# ------------------------------------------------------------------ the block loop
def _run_block(hidden_bits_steps, wb, B, L, d, V, seed, max_steps=48, stride_steps=True):
    hid = to_dev(hidden_bits_steps)
    p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=0, seed=seed)
    bp = dg.block_params(max_steps, 0.8, 0.4, B * L * d if stride_steps else 0)
    bufs = dg.BlockBuffers(B, L, max_steps, DEV)
    ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
    dg.generate_block(hid, to_dev(wb), p, bp, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    return bufs


def test_block_flat_logits_one_commit_per_step():
    """Untrained-model behaviour: exactly one commit per step, 48 steps, no stop."""
    B, L, d, V = 1, 256, 64, 4096
    wb = dg_synth.lm_weight(dg_synth.StepConfig("w", d=d, V=V))
    hid = np.zeros((L, d), np.uint16)
    bufs = _run_block(hid, wb, B, L, d, V, seed=0, stride_steps=False)
    assert int(bufs.steps_taken[0]) == 48
    assert (np_i32(bufs.n_accepted_hist) == 1).all()
    assert (np_i32(bufs.argmax) == 0).all()
    assert abs(float(bufs.mean_entropy[0]) - math.log(V)) < H_TOL


def test_block_one_hot_stops_after_two_steps_and_batches_independently():
    L, d, V = 64, 64, 1024
    w = np.zeros((d, V), np.float32)
    w[np.arange(d), np.arange(d) * 3] = 300.0
    x1 = np.zeros((L, d), np.float32)
    x1[np.arange(L), np.arange(L) % d] = 1.0
    hid = np.concatenate([dg_synth.f32_to_bf16_bits(x1), np.zeros((L, d), np.uint16)])
    bufs = _run_block(hid, dg_synth.f32_to_bf16_bits(w), 2, L, d, V, seed=1, max_steps=10,
                      stride_steps=False)
    assert np_i32(bufs.steps_taken).tolist() == [2, 10]
    assert np.array_equal(np_i32(bufs.argmax)[:L], (np.arange(L) % d) * 3)
    assert np.array_equal(np_i32(bufs.canvas)[:L], (np.arange(L) % d) * 3)
    hist = np_i32(bufs.n_accepted_hist).reshape(10, 2)
    assert hist[0, 0] == L and hist[1, 0] == L and (hist[:, 1] == 1).all()


def test_block_converging_matches_oracle():
    """A small version of the converging block workload: per-position targets and
    confidences, hidden states sharpen with the step.  The data seed is one on
    which every decision of the oracle's run is clear of its margin at every
    step (asserted below on the oracle alone), so the loop must reproduce the
    oracle's run exactly: commits per step, the stop step, the final canvas
    and the argmax output."""
    cfg = dg_synth.StepConfig("blk", L=64, d=256, V=2048, w_std=0.02, seed=18)
    wb = dg_synth.lm_weight(cfg)
    tg = dg_synth.block_targets(cfg)
    N = 48
    hs = np.stack([dg_synth.block_hidden(cfg, wb, tg, k) for k in range(N)])
    ref = oracle.block(lambda k: hs[k], wb, 1, cfg.L, 0.1, 9, max_steps=N)
    n_ref = int(ref["steps"][0])
    assert 2 <= n_ref < N
    for k, h in enumerate(ref["history"]):
        acc = np.zeros(cfg.L, bool)
        acc[h["order"][0][: int(h["n_accepted"][0])]] = True
        assert acceptance_is_decided(h["H32"], int(h["n_accepted"][0]),
                                     float(h["boundary_gap"][0])), k
        assert (h["gumbel_margin"][acc] >= MARGIN).all(), k
        assert (h["argmax_margin"] >= MARGIN).all(), k
        assert abs(float(h["mean_entropy"][0]) - 0.005) >= 2 * H_TOL, k
    bufs = _run_block(hs, wb, 1, cfg.L, cfg.d, cfg.V, seed=9, max_steps=N)
    assert int(bufs.steps_taken[0]) == n_ref
    hist = np_i32(bufs.n_accepted_hist)
    assert hist[:n_ref].tolist() == [int(h["n_accepted"][0]) for h in ref["history"]]
    assert np.array_equal(np_i32(bufs.argmax), ref["argmax"])
    assert np.array_equal(np_i32(bufs.canvas), ref["canvas"])
    last = ref["history"][-1]
    assert abs(float(bufs.mean_entropy[0]) - float(last["mean_entropy"][0])) < H_TOL


@pytest.mark.parametrize("name", ["step_small", "batch1", "batch4"])
def test_canvas_step_matches_the_two_calls_and_the_oracle(name):
    """dg_canvas_step (attention on a forked stream, the LM head planned around
    it) gives the attention output of dg_canvas_attn (bit for bit where its key
    splits are the same; capped to the SMs set aside for it, they can differ,
    and the rows then agree to bf16 rounding) and a step that matches the
    oracle."""
    cfg = dg_synth.CONFIGS[name]
    B, L, P, Hq, Hkv, D, d, V = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D, cfg.d, cfg.V
    ai = dg_synth.attention_inputs(cfg)
    t = {k: to_dev(v) for k, v in ai.items()}
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    rng = np.random.default_rng(3)
    canvas0 = rng.integers(0, V, B * L).astype(np.int32)
    prev = rng.integers(0, V, B * L).astype(np.int32)
    p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=2, seed=5)
    bufs = dg.StepBuffers(B, L, DEV)
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    bufs.prev_argmax.copy_(torch.from_numpy(prev))
    out = torch.empty_like(t["q"])
    ws = dg.workspace(dg.canvas_step_workspace(p, P, Hq, Hkv, D), DEV)
    for _ in range(2):       # the second call reuses the internal stream and events
        bufs.canvas.copy_(torch.from_numpy(canvas0))
        bufs.prev_argmax.copy_(torch.from_numpy(prev))
        dg.canvas_step(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], out, scale, to_dev(xb),
                       to_dev(wb), p, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
    ref_out = torch.empty_like(out)
    aws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), DEV)
    dg.canvas_attn(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], ref_out, scale, aws)
    torch.cuda.synchronize()
    if name == "step_small":
        assert torch.equal(out, ref_out)
    else:
        a, r = out.float(), ref_out.float()
        row_max = r.abs().amax(dim=-1, keepdim=True)
        assert ((a - r).abs() <= 2.0 ** -6 * row_max + 1e-6).all()
    ref = oracle.step(xb, wb, canvas0, prev, B, L, 0.8, 0.1, 5, 2, workers=8)
    check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)
    assert np.array_equal(np_i32(bufs.stop), ref["stop"])


def test_canvas_step_without_a_cache_and_ragged_canvases():
    """dg_canvas_step with no cached keys (P = 0), two canvases of 100
    positions (ragged against the 128-row tiles)."""
    cfg = dg_synth.StepConfig("cs_edge", B=2, L=100, Hq=4, Hkv=1, D=128, P=0, d=256, V=4096,
                              w_std=0.05, seed=12)
    B, L, Hq, Hkv, D, d, V = cfg.B, cfg.L, cfg.Hq, cfg.Hkv, cfg.D, cfg.d, cfg.V
    ai = dg_synth.attention_inputs(cfg)
    q, kc, vc = to_dev(ai["q"]), to_dev(ai["kc"]), to_dev(ai["vc"])
    xb, wb = dg_synth.lm_hidden(cfg), dg_synth.lm_weight(cfg)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    p = dg.step_params(B, L, d, V, 0.6, 0.1, 0.005, step=1, seed=2)
    bufs = dg.StepBuffers(B, L, DEV)
    canvas0 = oracle.init_canvas(B * L, V, 2)
    bufs.canvas.copy_(torch.from_numpy(canvas0))
    out = torch.full_like(q, float("nan"))
    ws = dg.workspace(dg.canvas_step_workspace(p, 0, Hq, Hkv, D), DEV)
    dg.canvas_step(q, None, None, kc, vc, out, scale, to_dev(xb), to_dev(wb), p, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    rows = np.arange(B * L * Hq)
    ref_o = oracle.attention_rows(ai["q"], ai["kp"], ai["vp"], ai["kc"], ai["vc"], B, L, 0, Hq, Hkv,
                                  D, scale, rows)
    got_o = out.float().reshape(-1, D).cpu().numpy()
    assert (np.abs(got_o - ref_o).max(axis=1) / np.abs(ref_o).max(axis=1)).max() < ATTN_TOL
    ref = oracle.step(xb, wb, canvas0, np.full(B * L, -1, np.int32), B, L, 0.6, 0.1, 2, 1)
    check_step_against_oracle(bufs, ref, B, L, exact_tokens=False)


def test_canvas_step_from_several_host_threads():
    """dg_canvas_step called from four host threads at once, each on its own
    stream, buffers and workspace (the library's forked stream and events are
    shared): every thread's repeated steps equal the same step made alone,
    bit for bit."""
    import threading
    cfg = dg_synth.CONFIGS["step_small"]
    B, L, P, Hq, Hkv, D, d, V = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D, cfg.d, cfg.V
    ai = dg_synth.attention_inputs(cfg)
    t = {k: to_dev(v) for k, v in ai.items()}
    x, w = to_dev(dg_synth.lm_hidden(cfg)), to_dev(dg_synth.lm_weight(cfg))
    scale = float(np.float32(1.0 / math.sqrt(D)))
    canvas0 = oracle.init_canvas(B * L, V, 4)

    def make(seed):
        p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=1, seed=seed)
        return dict(p=p, bufs=dg.StepBuffers(B, L, DEV), out=torch.empty_like(t["q"]),
                    ws=dg.workspace(dg.canvas_step_workspace(p, P, Hq, Hkv, D), DEV),
                    stream=torch.cuda.Stream())

    def run(c, n):
        with torch.cuda.stream(c["stream"]):
            for _ in range(n):
                c["bufs"].canvas.copy_(torch.from_numpy(canvas0))
                c["bufs"].prev_argmax.fill_(-1)
                dg.canvas_step(t["q"], t["kp"], t["vp"], t["kc"], t["vc"], c["out"], scale, x, w,
                               c["p"], c["bufs"], c["ws"], stream=c["stream"])
        c["stream"].synchronize()

    ctx = [make(10 + i) for i in range(4)]
    alone = []
    for c in ctx:
        run(c, 1)
        alone.append((c["bufs"].readback.clone(), c["out"].clone()))
    torch.cuda.synchronize()
    errs = []

    def worker(c):
        try:
            run(c, 25)
        except Exception as e:   # reported below
            errs.append(e)

    threads = [threading.Thread(target=worker, args=(c,)) for c in ctx]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errs
    for c, (rb, o) in zip(ctx, alone):
        status_ok(c["ws"])
        assert torch.equal(c["bufs"].readback, rb)
        assert torch.equal(c["out"], o)
