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
