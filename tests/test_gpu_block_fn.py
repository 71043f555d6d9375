"""The block loop with the decoder body inside it (dg_generate_block_fn) and
block-autoregressive generation over several canvases through the library.

* dg_hidden_from_steps reproduces dg_generate_block exactly;
* dg_hidden_embed_add -- hidden states that depend on the canvas being
  denoised -- against the oracle's loop run with the same producer, on a
  data seed where every decision of the oracle's run is clear of its margin;
* a producer written in Python runs once per captured graph, not per step;
* three canvases in a row ("Parallel Denoising From an Autoregressive
  Checkpoint", section "Finding": the causal encoder appends each committed
  block to its cache; "DiffusionGemma: When the LLM Stops Writing Left to
  Right", section "What DiffusionGemma Actually Is": block-autoregressive
  multi-canvas sampling): canvas attention over the cache -> the block loop
  (its hidden states carry the attention output) -> dg_encoder_append of the
  block's argmax tokens -> the next canvas, every stage checked against the
  oracle on the inputs the previous stage produced.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import (ATTN_TOL, DEV, H_TOL, MARGIN, acceptance_is_decided, np_i32,
                            status_ok, to_dev)

pytestmark = pytest.mark.gpu

f32 = dg_synth.bf16_bits_to_f32
N = 48


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _embed_fn(base, table):
    """The oracle side of dg_hidden_embed_add: bf16(base_k + table[canvas])."""
    return lambda k, canvas: _bf16(f32(base[k]) + f32(table[canvas]))


def _run_fn(producer, user, hidden_buf, wb, B, L, d, V, seed, max_steps=N):
    p = dg.step_params(B, L, d, V, 0.8, 0.1, 0.005, step=0, seed=seed)
    bp = dg.block_params(max_steps, 0.8, 0.4, 0)
    bufs = dg.BlockBuffers(B, L, max_steps, DEV)
    ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
    dg.generate_block_fn(producer, user, hidden_buf, to_dev(wb) if isinstance(wb, np.ndarray) else wb,
                         p, bp, bufs, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    return bufs


def _converging(seed, L=64, d=256, V=2048):
    cfg = dg_synth.StepConfig("blkfn", L=L, d=d, V=V, w_std=0.02, seed=seed)
    wb = dg_synth.lm_weight(cfg)
    tg = dg_synth.block_targets(cfg)
    return cfg, wb, np.stack([dg_synth.block_hidden(cfg, wb, tg, k) for k in range(N)])


def _clear_steps(ref, L):
    out = []
    for h in ref["history"]:
        acc = np.zeros(L, bool)
        acc[h["order"][0][: int(h["n_accepted"][0])]] = True
        out.append(acceptance_is_decided(h["H32"], int(h["n_accepted"][0]),
                                         float(h["boundary_gap"][0]))
                   and bool((h["gumbel_margin"][acc] >= MARGIN).all())
                   and bool((h["argmax_margin"] >= MARGIN).all())
                   and abs(float(h["mean_entropy"][0]) - 0.005) >= 2 * H_TOL)
    return out


def test_from_steps_producer_equals_precomputed_loop():
    cfg, wb, hs = _converging(3)
    B = 2
    hs2 = np.concatenate([hs, hs[:, ::-1]], axis=1)            # two canvases: [N, 2L, d]
    hid = to_dev(np.ascontiguousarray(hs2))
    w = to_dev(wb)
    p = dg.step_params(B, cfg.L, cfg.d, cfg.V, 0.8, 0.1, 0.005, step=0, seed=4)
    bp = dg.block_params(N, 0.8, 0.4, B * cfg.L * cfg.d)
    ref = dg.BlockBuffers(B, cfg.L, N, DEV)
    ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
    dg.generate_block(hid, w, p, bp, ref, ws)
    user = dg.HiddenSteps(hid.data_ptr(), B * cfg.L * cfg.d, B * cfg.L * cfg.d)
    buf = torch.empty(B * cfg.L, cfg.d, dtype=torch.bfloat16, device=DEV)
    got = _run_fn(dg.hidden_producer("from_steps"), user, buf, w, B, cfg.L, cfg.d, cfg.V, 4)
    for name in ("canvas", "argmax", "steps_taken", "n_accepted_hist"):
        assert np.array_equal(np_i32(getattr(got, name)), np_i32(getattr(ref, name))), name
    assert torch.equal(got.mean_entropy, ref.mean_entropy)


def test_canvas_dependent_producer_matches_oracle():
    """hidden_k = bf16(base_k + E[canvas]): each step's hidden states depend on
    the canvas the previous step left; every decision of the oracle's run is
    clear of its margin on this data seed, so the whole run must match."""
    cfg, wb, hs = _converging(19)
    Eh = dg_synth._normal_bf16(dg_synth._ss(19, 300), (cfg.V, cfg.d), std=0.05)
    ref = oracle.block(_embed_fn(hs, Eh), wb, 1, cfg.L, 0.1, 9, max_steps=N)
    assert all(_clear_steps(ref, cfg.L))
    base, table = to_dev(hs), to_dev(Eh)
    user = dg.HiddenEmbed(base.data_ptr(), cfg.L * cfg.d, table.data_ptr(), cfg.L, cfg.d, cfg.V)
    buf = torch.empty(cfg.L, cfg.d, dtype=torch.bfloat16, device=DEV)
    got = _run_fn(dg.hidden_producer("embed_add"), user, buf, wb, 1, cfg.L, cfg.d, cfg.V, 9)
    n = int(ref["steps"][0])
    assert int(got.steps_taken[0]) == n
    assert np_i32(got.n_accepted_hist)[:n].tolist() == [int(h["n_accepted"][0]) for h in ref["history"]]
    assert np.array_equal(np_i32(got.argmax), ref["argmax"])
    assert np.array_equal(np_i32(got.canvas), ref["canvas"])
    # the canvas feedback matters: without it every step's entropies differ
    ref0 = oracle.block(lambda k: hs[k], wb, 1, cfg.L, 0.1, 9, max_steps=N)
    assert not np.array_equal(ref0["history"][1]["H32"], ref["history"][1]["H32"])


def test_python_producer_runs_once_per_graph():
    cfg, wb, hs = _converging(5)
    base, table = to_dev(hs), torch.zeros(cfg.V, cfg.d, dtype=torch.bfloat16, device=DEV)
    inner = dg.HiddenEmbed(base.data_ptr(), cfg.L * cfg.d, table.data_ptr(), cfg.L, cfg.d, cfg.V)
    calls = []

    def produce(step, canvas, out, stream, user):
        calls.append(1)
        return dg.lib().dg_hidden_embed_add(step, canvas, out, stream, ctypes.byref(inner))

    fn = dg.HIDDEN_FN(produce)
    user = dg.HiddenSteps(0, 0, 0)            # unused by this producer; a distinct key
    buf = torch.empty(cfg.L, cfg.d, dtype=torch.bfloat16, device=DEV)
    w = to_dev(wb)
    p = dg.step_params(1, cfg.L, cfg.d, cfg.V, 0.8, 0.1, 0.005, step=0, seed=6)
    bp = dg.block_params(N, 0.8, 0.4, 0)
    bufs = dg.BlockBuffers(1, cfg.L, N, DEV)
    ws = dg.workspace(dg.generate_block_workspace(p, bp), DEV)
    results = []
    for _ in range(3):              # the same arguments: the captured graph is replayed
        dg.generate_block_fn(fn, user, buf, w, p, bp, bufs, ws)
        torch.cuda.synchronize()
        status_ok(ws)
        results.append((np_i32(bufs.argmax).copy(), int(bufs.steps_taken[0])))
    assert len(calls) == 1
    assert all(np.array_equal(r[0], results[0][0]) and r[1] == results[0][1] for r in results)
    ref = oracle.block(lambda k: hs[k], wb, 1, cfg.L, 0.1, 6, max_steps=N)
    assert results[0][1] == int(ref["steps"][0])


def test_three_canvases_through_cache_append():
    L, Hq, Hkv, D, V = 64, 2, 1, 128, 2048
    d = Hq * D
    scale = float(np.float32(1.0 / math.sqrt(D)))
    ss = lambda t: dg_synth._ss(3, t)
    Eq = dg_synth._normal_bf16(ss(400), (V, Hq * D))
    Ek = dg_synth._normal_bf16(ss(401), (V, Hkv * D))
    Ev = dg_synth._normal_bf16(ss(402), (V, Hkv * D))
    Eh = dg_synth._normal_bf16(ss(403), (V, d), std=1e-3)
    P0, P_max = 64, 64 + 3 * L
    kcache = torch.zeros(1, P_max, Hkv, D, dtype=torch.bfloat16, device=DEV)
    vcache = torch.zeros_like(kcache)
    kcache[:, :P0] = to_dev(dg_synth._normal_bf16(ss(404), (1, P0, Hkv, D)))
    vcache[:, :P0] = to_dev(dg_synth._normal_bf16(ss(405), (1, P0, Hkv, D)))
    cfg = dg_synth.StepConfig("chain", L=L, d=d, V=V, w_std=0.02, seed=3)
    wb = dg_synth.lm_weight(cfg)
    w = to_dev(wb)
    table = to_dev(Eh)
    rows = np.arange(L * Hq)
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    P = P0
    for c in range(3):
        seed_c = 9 + c
        # 1. the canvas attends to [cache ; canvas]: its initial tokens' Q/K/V
        init = oracle.init_canvas(L, V, seed_c)
        q, kc, vc = (Eq[init].reshape(1, L, Hq, D), Ek[init].reshape(1, L, Hkv, D),
                     Ev[init].reshape(1, L, Hkv, D))
        att = torch.empty(1, L, Hq, D, dtype=torch.bfloat16, device=DEV)
        aws = dg.workspace(dg.canvas_attn_workspace(1, L, P, Hq, Hkv, D), DEV)
        dg.canvas_attn(to_dev(q), kcache[:, :P].contiguous(), vcache[:, :P].contiguous(),
                       to_dev(kc), to_dev(vc), att, scale, aws)
        torch.cuda.synchronize()
        kcb, vcb = bits(kcache[:, :P].contiguous()), bits(vcache[:, :P].contiguous())
        ref_att = oracle.attention_rows(q, kcb, vcb, kc, vc, 1, L, P, Hq, Hkv, D, scale, rows)
        got_att = att.float().reshape(-1, D).cpu().numpy()
        assert (np.abs(got_att - ref_att).max(axis=1) / np.abs(ref_att).max(axis=1)).max() < ATTN_TOL
        # 2. the block loop; its hidden states carry the attention output
        cfgc = dg_synth.StepConfig("chain", L=L, d=d, V=V, w_std=0.02, seed=30 + c)
        tg = dg_synth.block_targets(cfgc)
        hs = np.stack([dg_synth.block_hidden(cfgc, wb, tg, k) for k in range(N)])
        ab = f32(bits(att).reshape(L, d))
        base = np.stack([_bf16(f32(hs[k]) + 0.25 * ab) for k in range(N)])
        base_d = to_dev(base)
        user = dg.HiddenEmbed(base_d.data_ptr(), L * d, table.data_ptr(), L, d, V)
        buf = torch.empty(L, d, dtype=torch.bfloat16, device=DEV)
        got = _run_fn(dg.hidden_producer("embed_add"), user, buf, w, 1, L, d, V, seed_c)
        ref = oracle.block(_embed_fn(base, Eh), wb, 1, L, 0.1, seed_c, max_steps=N)
        clear = _clear_steps(ref, L)
        assert np.mean(clear) >= 0.8
        n = int(ref["steps"][0])
        assert int(got.steps_taken[0]) == n
        hist = np_i32(got.n_accepted_hist)
        for k, h in enumerate(ref["history"]):
            if clear[k]:
                assert hist[k] == int(h["n_accepted"][0]), (c, k)
        am = np_i32(got.argmax)
        ok = ref["history"][-1]["argmax_margin"] >= MARGIN
        assert ok.mean() > 0.95
        assert np.array_equal(am[ok], ref["argmax"][ok])
        # 3. the causal encoder appends the committed block (its argmax tokens)
        qe, kn, vn = (Eq[am].reshape(1, L, Hq, D), Ek[am].reshape(1, L, Hkv, D),
                      Ev[am].reshape(1, L, Hkv, D))
        eo = torch.empty(1, L, Hq, D, dtype=torch.bfloat16, device=DEV)
        ews = dg.workspace(dg.encoder_append_workspace(1, L, P, Hq, Hkv, D), DEV)
        dg.encoder_append(to_dev(qe), kcache, vcache, P, to_dev(kn), to_dev(vn), eo, scale, ews)
        torch.cuda.synchronize()
        status_ok(ews)
        assert np.array_equal(bits(kcache[:, P:P + L].contiguous()), kn)
        assert np.array_equal(bits(vcache[:, P:P + L].contiguous()), vn)
        ref_e = oracle.attention_rows(qe, kcb, vcb, kn, vn, 1, L, P, Hq, Hkv, D, scale, rows,
                                      causal=True)
        got_e = eo.float().reshape(-1, D).cpu().numpy()
        assert (np.abs(got_e - ref_e).max(axis=1) / np.abs(ref_e).max(axis=1)).max() < ATTN_TOL
        P += L
    assert P == P_max
