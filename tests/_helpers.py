"""Shared helpers of the GPU parity tests (no method arithmetic here)."""
import numpy as np

import block_diffusion_decoding_gb300 as dg

DEV = "cuda"

# Tolerances: entropies 1e-4 absolute; attention outputs within 2e-2 of the
# row's largest magnitude; tokens bit-exact unless the oracle's Gumbel /
# argmax margin or the acceptance boundary is within 1e-3 (then exempt).
H_TOL = 1e-4
ATTN_TOL = 2e-2
MARGIN = 1e-3


def to_dev(bits):
    return dg.bf16_from_bits(bits, DEV)


def np_i32(t):
    return t.detach().cpu().numpy().astype(np.int32)


def np_f(t):
    return t.detach().float().cpu().numpy()


def acceptance_is_decided(H_ref, kstar, gap, H_tol=H_TOL, margin=MARGIN):
    """True when an entropy error of up to H_tol per position cannot change the
    accepted set: the prefix sums stay clear of b and no near-tie straddles the
    boundary of the sorted order."""
    L = len(H_ref)
    if gap < margin:
        return False
    if kstar < L:
        hs = np.sort(np.asarray(H_ref, np.float64))
        if hs[kstar] - hs[kstar - 1] < 2 * H_tol:
            return False
    return True


def status_ok(ws):
    assert dg.read_device_status(ws) == 0


def check_step_against_oracle(bufs, ref, B, L, exact_tokens):
    """Compare a step's outputs (StepBuffers) with the oracle's step result; returns
    the number of canvases whose acceptance was decided clearly enough to compare."""
    H = np_f(bufs.entropy)
    assert np.abs(H - ref["H"]).max() < H_TOL, np.abs(H - ref["H"]).max()
    am, sm = np_i32(bufs.argmax), np_i32(bufs.sample)
    if exact_tokens:
        assert np.array_equal(am, ref["argmax"])
        assert np.array_equal(sm, ref["sample"])
    else:
        ok = ref["argmax_margin"] >= MARGIN
        assert ok.mean() > 0.9
        assert np.array_equal(am[ok], ref["argmax"][ok])
        ok = ref["gumbel_margin"] >= MARGIN
        assert ok.mean() > 0.9
        assert np.array_equal(sm[ok], ref["sample"][ok])
    canvas, acc = np_i32(bufs.canvas), bufs.accepted.cpu().numpy()
    checked = 0
    for bb in range(B):
        sl = slice(bb * L, (bb + 1) * L)
        if not acceptance_is_decided(ref["H"][sl], int(ref["n_accepted"][bb]),
                                     float(ref["boundary_gap"][bb])):
            continue
        checked += 1
        assert int(bufs.n_accepted[bb]) == int(ref["n_accepted"][bb])
        assert np.array_equal(acc[sl], ref["accepted"][sl])
        # accepted positions hold the sample; every other one the renoise token
        acc_ref = ref["accepted"][sl] == 1
        if exact_tokens or bool(np.all(ref["gumbel_margin"][sl][acc_ref] >= MARGIN)):
            assert np.array_equal(canvas[sl], ref["canvas"][sl])
        else:
            assert np.array_equal(canvas[sl][~acc_ref], ref["canvas"][sl][~acc_ref])
    return checked


def force_lm_kernel(monkeypatch, spec):
    """Force the LM-head choice: None = the planner's; "kind" or "kind/epi"
    (kind single | duo | fused; epi 8 | 16 epilogue warps of the
    2-SM kernel)."""
    monkeypatch.delenv("DG_LM_KERNEL", raising=False)
    monkeypatch.delenv("DG_LM_EPI", raising=False)
    if spec is None:
        return
    kind, _, epi = spec.partition("/")
    monkeypatch.setenv("DG_LM_KERNEL", kind)
    if epi:
        monkeypatch.setenv("DG_LM_EPI", epi)
