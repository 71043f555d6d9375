"""The acceptance kernel orders only the positions whose entropy is within the
bound b (the set C), plus the smallest key outside C.  This checks that
reduction on the CPU, against the oracle's full sort: with an fp64 sum of
non-negative terms at least each of its terms, a sorted prefix that holds an
entropy above b sums past b, so k* counts only C's keys and at most the one
key that sorts right after them.  Random and adversarial entropy vectors:
ties, zeros, values exactly at the bound and just above it, b = 0."""
import numpy as np
import pytest

import oracle


def _kstar_reduced(H, b):
    """k* from C and the smallest key outside it, sums as the oracle takes them
    (fp64, sequential, sorted order)."""
    H = np.asarray(H, np.float32)
    L = H.shape[0]
    bd = float(np.float32(b))
    inside = np.nonzero(H.astype(np.float64) <= bd)[0]
    outside = np.nonzero(H.astype(np.float64) > bd)[0]
    keys = sorted(inside, key=lambda i: (H[i], i))
    if outside.size:
        keys.append(min(outside, key=lambda i: (H[i], i)))
    run, k = 0.0, 0
    for j, i in enumerate(keys):
        if j > 0:
            run += float(H[keys[j - 1]])
        if run <= bd:
            k = j + 1
    return max(1, k), keys


def _cases(rng):
    L = int(rng.integers(1, 300))
    kind = rng.integers(0, 6)
    if kind == 0:
        H = rng.exponential(0.02, L)
    elif kind == 1:
        H = rng.choice([0.0, 0.01, 0.02, 0.1, 0.5], L)
    elif kind == 2:
        H = rng.exponential(1.0, L) * rng.choice([1e-4, 1e-2, 1.0], L)
    elif kind == 3:
        H = np.full(L, 0.1)
        H[rng.integers(0, L, max(1, L // 3))] = np.nextafter(np.float32(0.1), np.float32(1))
    elif kind == 4:
        H = np.zeros(L)
        H[rng.integers(0, L)] = 5.0
    else:
        H = rng.uniform(0.0, 0.2, L)
    b = float(rng.choice([0.1, 0.0, 0.05, 0.3]))
    return H.astype(np.float32), b


def test_in_bound_set_reduction_matches_full_sort():
    rng = np.random.default_rng(2024)
    for _ in range(400):
        H, b = _cases(rng)
        L = H.shape[0]
        ref = oracle.accept_renoise(H, np.zeros(L, np.int32), np.zeros(L, np.int32), 4096,
                                    np.float32(b), 1, 0, 1)
        k, keys = _kstar_reduced(H, b)
        assert k == ref["n_accepted"], (L, b)
        # the accepted positions are the first k of the reduced order, which is
        # the start of the oracle's sorted order
        assert list(ref["order"][:k]) == keys[:k]
        assert np.array_equal(np.nonzero(ref["accepted"])[0], np.sort(np.array(keys[:k])))


@pytest.mark.parametrize("b", [0.0, 0.1])
def test_reduction_edges(b):
    # nothing inside: the smallest key commits alone
    H = np.array([0.7, 0.3, 0.3, 0.9], np.float32)
    assert _kstar_reduced(H, b)[0] == 1
    # everything inside with a zero sum: all commit
    H = np.zeros(17, np.float32)
    assert _kstar_reduced(H, b)[0] == 17
