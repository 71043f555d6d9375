"""GPU parity of the encoder cache append (dg_encoder_append) against the
fp64 oracle's causal attention: the block's keys / values land in cache rows
P .. P+L-1 (bit-exact, other rows untouched) and canvas position i attends to
the P cached rows and the block's rows 0 .. i (2e-2 of the row's largest
magnitude), through both attention kernels."""
import math

import numpy as np
import pytest
import torch

import block_diffusion_decoding_gb300 as dg
import dg_synth
import oracle
from tests._helpers import ATTN_TOL, DEV, status_ok, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("B,L,P,Hq,Hkv,D,stride", [
    (1, 256, 256, 4, 1, 128, 1),      # the small workload's shapes
    (2, 100, 37, 4, 2, 128, 1),       # ragged block and cache
    (1, 64, 0, 2, 1, 128, 1),         # empty cache: the first block
    (2, 256, 1000, 16, 8, 256, 7),    # head dim 256 with key splits
    (1, 256, 4096, 16, 8, 256, 13),   # the full-width step's attention shapes
])
def test_encoder_append_matches_oracle(kernel, B, L, P, Hq, Hkv, D, stride, monkeypatch):
    monkeypatch.setenv("DG_ATTN_KERNEL", kernel)
    cfg = dg_synth.StepConfig("enc", B=B, L=L, P=P, Hq=Hq, Hkv=Hkv, D=D, seed=31 + P)
    ai = dg_synth.attention_inputs(cfg)
    P_max = P + L + 3
    sentinel = np.uint16(0x7FC1)   # a bf16 NaN pattern: rows past P + L must keep it
    kcache = np.full((B, P_max, Hkv, D), sentinel, np.uint16)
    vcache = np.full((B, P_max, Hkv, D), sentinel, np.uint16)
    kcache[:, :P], vcache[:, :P] = ai["kp"], ai["vp"]
    kc_d, vc_d = to_dev(kcache), to_dev(vcache)
    q, knew, vnew = to_dev(ai["q"]), to_dev(ai["kc"]), to_dev(ai["vc"])
    out = torch.full_like(q, float("nan"))
    scale = float(np.float32(1.0 / math.sqrt(D)))
    ws = dg.workspace(dg.encoder_append_workspace(B, L, P, Hq, Hkv, D), DEV)
    dg.encoder_append(q, kc_d, vc_d, P, knew, vnew, out, scale, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    # the append
    got_k = kc_d.view(torch.int16).cpu().numpy().view(np.uint16)
    got_v = vc_d.view(torch.int16).cpu().numpy().view(np.uint16)
    want_k, want_v = kcache.copy(), vcache.copy()
    want_k[:, P:P + L], want_v[:, P:P + L] = ai["kc"], ai["vc"]
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)
    # the causal attention
    rows = np.unique(np.append(np.arange(0, B * L * Hq, stride), B * L * Hq - 1))
    ref = oracle.attention_rows(ai["q"], ai["kp"], ai["vp"], ai["kc"], ai["vc"], B, L, P, Hq, Hkv,
                                D, scale, rows, causal=True)
    got = out.float().reshape(-1, D).cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got[rows] - ref).max(axis=1) / np.abs(ref).max(axis=1)
    assert err.max() < ATTN_TOL, (err.max(), int(rows[err.argmax()]))


def test_encoder_append_chains_blocks():
    """Two blocks in a row: the second block's cache holds the first block's
    tokens; its causal attention matches the oracle over the grown cache."""
    B, L, Hq, Hkv, D = 1, 128, 4, 1, 128
    cfg = dg_synth.StepConfig("chain", B=B, L=L, P=0, Hq=Hq, Hkv=Hkv, D=D, seed=5)
    blk = [dg_synth.attention_inputs(cfg, seed=s) for s in (5, 6)]
    P_max = 2 * L
    kc_d = torch.zeros(B, P_max, Hkv, D, dtype=torch.bfloat16, device=DEV)
    vc_d = torch.zeros_like(kc_d)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    out = torch.empty(B, L, Hq, D, dtype=torch.bfloat16, device=DEV)
    ws = dg.workspace(dg.encoder_append_workspace(B, L, L, Hq, Hkv, D), DEV)
    for n, ai in enumerate(blk):
        dg.encoder_append(to_dev(ai["q"]), kc_d, vc_d, n * L, to_dev(ai["kc"]), to_dev(ai["vc"]),
                          out, scale, ws)
    torch.cuda.synchronize()
    status_ok(ws)
    rows = np.arange(B * L * Hq)
    ref = oracle.attention_rows(blk[1]["q"], blk[0]["kc"], blk[0]["vc"], blk[1]["kc"],
                                blk[1]["vc"], B, L, L, Hq, Hkv, D, scale, rows, causal=True)
    got = out.float().reshape(-1, D).cpu().numpy()
    err = np.abs(got - ref).max(axis=1) / np.abs(ref).max(axis=1)
    assert err.max() < ATTN_TOL
