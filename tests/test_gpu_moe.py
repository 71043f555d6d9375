"""GPU parity of the MoE FFN (dg_moe_ffn) against the fp64 oracle.

Routing: the chosen experts must equal the oracle's on every row whose
router margin (k-th minus (k+1)-th logit) is at least 1e-3; rows below it may
pick either expert and are left out of the output comparison.  Gates: 1e-5
absolute.  Output rows: max |out - ref| <= 2e-2 max |ref| per row (bf16
operands and a bf16 intermediate activation, fp32 accumulation).
"""
import functools

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import DEV, MARGIN, status_ok

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


@functools.lru_cache(maxsize=1)
def _full_inputs():
    cfg = dg_synth.MOE_CONFIGS["moe_full"]
    return cfg, dg_synth.moe_inputs(cfg)


def _run(a, M, d, f, E, K, reps=1):
    t = {k: _dev(v) for k, v in a.items()}
    p = dg.moe_params(M, d, f, E, K)
    ws = dg.workspace(dg.moe_ffn_workspace(p), DEV)
    outs = []
    for _ in range(reps):
        out = torch.full((M, d), float("nan"), device=DEV)
        ex = torch.full((M, K), -1, dtype=torch.int32, device=DEV)
        gt = torch.zeros(M, K, device=DEV)
        dg.moe_ffn(t["x"], t["wr"], t["wg"], t["wu"], t["wd"], out, p, ws, ex, gt)
        torch.cuda.synchronize()
        status_ok(ws)
        outs.append((out.cpu().numpy(), ex.cpu().numpy(), gt.cpu().numpy()))
    return outs


def _check(got, ref, K):
    out, ex, gt = got
    clear = ref["margin"] >= MARGIN
    assert clear.mean() > 0.9
    assert np.array_equal(ex[clear], ref["experts"][clear])
    assert np.abs(gt[clear] - ref["gates"][clear]).max() < 1e-5
    err = np.abs(out - ref["out"]).max(axis=1) / np.abs(ref["out"]).max(axis=1)
    assert np.isfinite(out).all()
    assert err[clear].max() < OUT_TOL, (err[clear].max(), int(np.argmax(np.where(clear, err, 0))))


def _small(M, d, f, E, K, seed, alpha=0.8):
    cfg = dg_synth.MoeConfig("moe_small", M=M, d=d, f=f, E=E, top_k=K, alpha=alpha, seed=seed)
    return dg_synth.moe_inputs(cfg)


@pytest.mark.parametrize("M,d,f,E,K", [(64, 256, 256, 16, 4), (100, 384, 128, 20, 3),
                                       (300, 256, 384, 8, 4), (1, 256, 128, 4, 1),
                                       (17, 256, 256, 128, 8), (130, 768, 128, 40, 2),
                                       (5, 128, 128, 6, 2)])
def test_moe_matches_oracle_small(M, d, f, E, K):
    """Several tiles of f and d and k slices of the router, ragged token counts,
    an expert with more than one 128-token chunk (300 rows over 8 experts),
    a single row, 128 experts, two 128-row token chunks of the router, and the
    smallest hidden size (one k slice of the router, one d tile)."""
    a = _small(M, d, f, E, K, seed=M + E)
    ref = oracle.moe_ffn(a["x"], a["wr"], a["wg"], a["wu"], a["wd"], K)
    got, again = _run(a, M, d, f, E, K, reps=2)
    _check(got, ref, K)
    # a second call on the same workspace gives the same result, bit for bit
    assert np.array_equal(got[0], again[0]) and np.array_equal(got[1], again[1])


def test_moe_full_size_every_row():
    """The MoE workload: 256 canvas rows, d = 2816, 128 experts of f = 768,
    top-8 plus the shared expert; the router touches about 84-90 experts."""
    cfg, a = _full_inputs()
    ref = oracle.moe_ffn(a["x"], a["wr"], a["wg"], a["wu"], a["wd"], cfg.top_k)
    assert 70 <= ref["distinct"] <= 100
    (got,) = _run(a, cfg.M, cfg.d, cfg.f, cfg.E, cfg.top_k)
    _check(got, ref, cfg.top_k)


def test_moe_shared_expert_only_when_routed_down_weights_are_zero():
    M, d, f, E, K = 40, 256, 128, 12, 3
    a = _small(M, d, f, E, K, seed=9)
    a["wd"] = a["wd"].copy()
    a["wd"][:E] = 0
    ref = oracle.moe_ffn(a["x"], a["wr"], a["wg"], a["wu"], a["wd"], K)
    (got,) = _run(a, M, d, f, E, K)
    err = np.abs(got[0] - ref["out"]).max(axis=1) / np.abs(ref["out"]).max(axis=1)
    assert err.max() < OUT_TOL


@pytest.mark.parametrize("M,d,f,E,K", [(96, 256, 128, 8, 8), (2048, 256, 128, 16, 4)])
def test_moe_edges(M, d, f, E, K):
    """Every expert chosen by every row (top_k = E), and the largest M the
    routing takes (2048 rows: eight 256-token canvases)."""
    a = _small(M, d, f, E, K, seed=M + 3 * E)
    ref = oracle.moe_ffn(a["x"], a["wr"], a["wg"], a["wu"], a["wd"], K)
    (got,) = _run(a, M, d, f, E, K)
    if K == E:
        assert (np.sort(got[1], axis=1) == np.arange(E)).all()
    _check(got, ref, K)
