"""Pins for the fp64 oracle: each checks it against something other than itself.

Closed forms, published known-answer vectors, library routines (torch /
numpy in float64), brute force on tiny inputs and the values the pages print
for a worked example.  No GPU is needed.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ Philox
def test_philox_known_answer_vectors():
    """Random123 kat_vectors for philox4x32, 10 rounds (SC'11 reference library)."""
    rows = _read_golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        vals = [int(x, 16) for x in r]
        out = oracle.philox4x32_10(vals[0:4], vals[4:6])
        assert [int(x) for x in out] == vals[6:10]


def test_philox_is_a_bijection_on_a_small_slice():
    """A keyed bijection: distinct counters give distinct outputs (sanity on 4096 counters)."""
    outs = {tuple(oracle.philox4x32_10([i, 7, 3, 1], [11, 13])) for i in range(4096)}
    assert len(outs) == 4096


# ------------------------------------------------------------------ fp32 log
def _ulp32(x: float) -> float:
    return float(np.spacing(np.float32(abs(x))))


def test_logf_accuracy_against_double_log():
    """Within 2 ulp of the correctly rounded natural log over the sampler's input range."""
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.uniform(5.9e-8, 1.0, 20000), rng.uniform(1.0, 17.0, 20000),
        np.exp(rng.uniform(-30, 30, 20000)),
        np.array([1.0, 2.0, 0.5, 0.70710677, 1.4142135, 16.635532, 5.9604645e-08, 0.99999994]),
    ]).astype(np.float32)
    worst = 0.0
    for x in xs:
        got = oracle.logf(float(x))
        ref = math.log(float(x))
        if ref == 0.0:
            assert got == 0.0
            continue
        err = abs(got - ref) / _ulp32(ref)
        worst = max(worst, err)
    assert worst <= 2.0, worst


def test_logf_exact_points():
    assert oracle.logf(1.0) == 0.0
    for k in range(-24, 25):
        assert abs(oracle.logf(2.0 ** k) - k * math.log(2.0)) <= _ulp32(k * math.log(2.0) or 1.0)


# ------------------------------------------------------------------ uniform / Gumbel
def test_uniform_open_interval_endpoints():
    assert oracle.uniform_open(0) == 2.0 ** -24
    assert oracle.uniform_open(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform_open(1 << 31) == 0.5 + 2.0 ** -24


def test_gumbel_moments():
    """Standard Gumbel: mean = Euler-Mascheroni constant, variance = pi^2/6."""
    g = np.concatenate([oracle.gumbel_fill(0, r, 0, 0, 20000) for r in range(10)]).astype(np.float64)
    n = g.size
    assert abs(g.mean() - 0.5772156649) < 5 * math.sqrt(math.pi ** 2 / 6 / n)
    assert abs(g.var() - math.pi ** 2 / 6) < 0.03
    # CDF exp(-exp(-x)) at a few points (Kolmogorov-style bound)
    for x in (-1.0, 0.0, 1.0, 3.0):
        emp = float((g <= x).mean())
        assert abs(emp - math.exp(-math.exp(-x))) < 0.005


def test_gumbel_max_sample_follows_softmax():
    """Frequency of the Gumbel-max sample over many rows matches softmax(z/T) (chi-square)."""
    V, T, n = 8, 0.8, 40000
    z = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.9, 1.7])
    logits = np.ascontiguousarray(z)
    counts = np.zeros(V)
    for r in range(n):
        s = oracle.sampler_row(logits, T, 5, r, 3)
        counts[s["sample"]] += 1
    zf = z.astype(np.float32).astype(np.float64) * float(np.float32(1.0 / T))
    p = np.exp(zf - zf.max())
    p /= p.sum()
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 24.3, chi2  # 7 dof, p = 0.001


# ------------------------------------------------------------------ entropy / argmax
def test_entropy_uniform_is_ln_V_and_pages_value():
    """Uniform logits give H = ln V; the Lab page's untrained model reads 6.91 nats at V=1000."""
    g = dict((r[0], r[1]) for r in _read_golden("lab_exp_a_untrained.txt"))
    V = int(g["vocab"])
    s = oracle.sampler_row(np.zeros(V), 0.8, 0, 0, 0)
    assert abs(s["H"] - math.log(V)) < 1e-12
    assert round(s["H"], 2) == float(g["mean_entropy_nats"])
    for V in (2, 64, 16384, 262144):
        s = oracle.sampler_row(np.full(V, 3.25), 0.4, 0, 0, 0)
        assert abs(s["H"] - math.log(V)) < 1e-9


def test_entropy_one_hot_is_zero():
    x = np.zeros(4096)
    x[1234] = 1e4
    s = oracle.sampler_row(x, 0.8, 0, 0, 0)
    assert s["H"] == 0.0
    assert s["argmax"] == 1234 and s["sample"] == 1234


def test_entropy_two_level_closed_form():
    """n entries at a, V-n at 0: H = ln Z - n a' e^{a'} / Z with a' = a/T, Z = n e^{a'} + V - n."""
    for V, n, a, T in [(1000, 3, 2.5, 0.8), (64, 10, -1.0, 0.5), (16384, 1, 7.0, 0.4)]:
        x = np.zeros(V)
        x[:n] = a
        ap = a / T
        Z = n * math.exp(ap) + V - n
        ref = math.log(Z) - n * ap * math.exp(ap) / Z
        assert abs(oracle.sampler_row(x, T, 0, 0, 0)["H"] - ref) < 1e-9 * max(1.0, abs(ref)) + 1e-11


def test_entropy_matches_torch_categorical():
    rng = np.random.default_rng(2)
    for V, T, sc in [(100, 0.8, 1.0), (5000, 0.4, 6.0), (3, 1.0, 0.1)]:
        x = rng.standard_normal(V) * sc
        ref = torch.distributions.Categorical(logits=torch.from_numpy(x / T)).entropy().item()
        assert abs(oracle.sampler_row(x, T, 0, 0, 0)["H"] - ref) < 1e-10


def test_argmax_ties_lowest_index_and_margin():
    x = np.array([1.0, 5.0, 2.0, 5.0, 4.0])
    s = oracle.sampler_row(x, 0.8, 0, 0, 0)
    assert s["argmax"] == 1 and s["argmax_margin"] == 0.0
    x[3] = 4.5
    assert oracle.sampler_row(x, 0.8, 0, 0, 0)["argmax_margin"] == 0.5


def test_gumbel_score_definition():
    """The sample is the argmax of fp32(fmaf(logit, fp32(1/T), G_v)), brute-forced here with numpy."""
    V, T, seed, row, step = 37, 0.8, 123, 9, 4
    rng = np.random.default_rng(3)
    x = rng.standard_normal(V).astype(np.float32).astype(np.float64)
    G = oracle.gumbel_fill(seed, row, step, 0, V)
    invT = np.float32(1.0 / T)
    # fmaf == round(x*invT + G) computed exactly in float64 then rounded (products of two
    # fp32 fit in fp64 exactly; the sum is then rounded once to fp32 via double rounding-safe
    # path for these magnitudes)
    score = (x.astype(np.float32).astype(np.float64) * np.float64(invT) + G.astype(np.float64)).astype(np.float32)
    s = oracle.sampler_row(x, T, seed, row, step)
    assert s["sample"] == int(np.argmax(score))


def _brute_top_two(scores):
    """Largest score, its lowest index, and the gap to the runner-up (a tie
    for the top gives 0), by sorting a copy."""
    sc = np.asarray(scores, np.float64)
    top = float(sc.max())
    first = int(np.nonzero(sc == top)[0][0])
    srt = np.sort(sc)
    return first, float(srt[-1] - srt[-2]) if sc.shape[0] > 1 else math.inf


def test_gumbel_margin_brute_force():
    """The Gumbel-max margin is the gap between the two largest fp32 scores.  At
    T = 1 (fp32(1/T) = 1) the score fmaf(logit, 1, G) is one fp32 addition, which
    numpy computes exactly the same way; the top two come from a sort."""
    rng = np.random.default_rng(11)
    for trial in range(40):
        V = int(rng.integers(2, 300))
        seed, row, step = int(rng.integers(0, 2**40)), int(rng.integers(0, 4096)), int(rng.integers(0, 48))
        x = (rng.standard_normal(V) * rng.uniform(0.1, 6.0)).astype(np.float32)
        G = oracle.gumbel_fill(seed, row, step, 0, V)
        score = x + G                               # fp32 + fp32, rounded once
        if trial % 4 == 0:
            # plant a tie for the top: a later column reaches the same score
            a = int(np.argmax(score))
            b = (a + 1 + int(rng.integers(0, V - 1))) % V
            xb = np.float32(score[a] - G[b])
            if np.float32(xb + G[b]) == score[a]:
                x[b] = xb
                score = x + G
        s = oracle.sampler_row(x.astype(np.float64), 1.0, seed, row, step)
        first, gap = _brute_top_two(score)
        assert s["sample"] == first
        assert s["gumbel_margin"] == gap
        if trial % 4 == 0 and (score == score.max()).sum() > 1:
            assert s["gumbel_margin"] == 0.0


def test_gumbel_margin_at_other_temperatures():
    """At T != 1 the brute force forms the score in float64 (the fp32 product
    is exact there) and rounds it to fp32: within one fp32 rounding of the
    oracle's fused score, so margins agree to a few ulps of the scores."""
    rng = np.random.default_rng(12)
    for T in (0.8, 0.5, 0.4123):
        V = 257
        x = (rng.standard_normal(V) * 3.0).astype(np.float32)
        G = oracle.gumbel_fill(5, 3, 2, 0, V)
        invT = np.float64(np.float32(1.0 / T))
        score = (x.astype(np.float64) * invT + G.astype(np.float64)).astype(np.float32)
        s = oracle.sampler_row(x.astype(np.float64), T, 5, 3, 2)
        _, gap = _brute_top_two(score)
        tol = 4 * float(np.spacing(np.float32(np.abs(score).max())))
        assert abs(s["gumbel_margin"] - gap) <= tol


def _brute_boundary_gap(H, b):
    """min over prefix lengths 1 .. L-1 of the (H, position)-sorted order of
    |exact sum of the prefix - b| (math.fsum: correctly rounded)."""
    order = sorted(range(len(H)), key=lambda i: (float(np.float32(H[i])), i))
    vals = [float(np.float32(H[i])) for i in order]
    return min((abs(math.fsum(vals[:j]) - b) for j in range(1, len(vals))), default=math.inf)


def test_boundary_gap_brute_force():
    rng = np.random.default_rng(13)
    for trial in range(50):
        L = int(rng.integers(2, 80))
        H = rng.exponential(rng.uniform(0.005, 0.2), L).astype(np.float32)
        b = float(rng.choice([0.0, 0.05, 0.1, 0.3]))
        r = _accept(H, b=b)
        assert abs(r["boundary_gap"] - _brute_boundary_gap(H, b)) < 1e-12
    # a prefix that sums to b exactly (dyadic entropies): the gap is 0 and the
    # prefix is accepted (the rule is <= b)
    H = np.array([0.25, 0.125, 0.5, 0.0625, 2.0], np.float32)
    r = _accept(H, b=0.4375)       # 0.0625 + 0.125 + 0.25 = 0.4375
    assert r["boundary_gap"] == 0.0
    assert r["n_accepted"] == 4    # the sum before the 4th sorted entry is exactly b


# ------------------------------------------------------------------ acceptance
def _accept(H, b=0.1, L=None, V=1 << 14, seed=0, step=0):
    H = np.asarray(H, np.float32)
    L = H.shape[0]
    smp = np.arange(L, dtype=np.int32) + 1000
    cv = np.full(L, -1, np.int32)
    return oracle.accept_renoise(H, smp, cv, V, b, seed, 0, step)


@pytest.mark.parametrize("e,expect", [(0.03, 4), (0.07, 2), (0.3, 1), (1e-5, 256), (6.91, 1)])
def test_equal_entropies(e, expect):
    """Equal entropies e: k* = 1 + floor(b/e), capped at L; e > b commits exactly one."""
    r = _accept(np.full(256, e))
    assert r["n_accepted"] == expect
    assert min(256, 1 + math.floor(0.1 / float(np.float32(e)))) == expect
    # ties go to the lower position: the first k* positions are the accepted ones
    assert r["accepted"][:expect].all() and not r["accepted"][expect:].any()


def _brute_force_kstar(H, b):
    """Largest set S that is a prefix of the (H, position) ascending order with
    sum_S H - max_S H <= b, found by enumerating every subset."""
    L = len(H)
    key = [(float(np.float32(H[i])), i) for i in range(L)]
    best = None
    for mask in range(1, 1 << L):
        S = [i for i in range(L) if mask >> i & 1]
        out = [i for i in range(L) if not mask >> i & 1]
        if out and max(key[i] for i in S) > min(key[i] for i in out):
            continue  # not a prefix of the ascending order
        vals = [key[i][0] for i in S]
        if math.fsum(vals) - max(vals) <= b + 1e-15:
            if best is None or len(S) > len(best):
                best = S
    return sorted(best)


def test_accept_brute_force_tiny():
    rng = np.random.default_rng(4)
    for trial in range(60):
        L = int(rng.integers(1, 9))
        H = rng.choice([0.0, 0.01, 0.02, 0.05, 0.07, 0.2, 1.0], size=L) * rng.uniform(0.5, 1.5, L)
        if trial % 3 == 0:
            H[rng.integers(0, L)] = H[0]  # planted ties
        b = float(rng.choice([0.0, 0.05, 0.1, 0.3]))
        r = _accept(H, b=b)
        exp_set = _brute_force_kstar(H, b)
        assert sorted(np.nonzero(r["accepted"])[0].tolist()) == exp_set
        # every permutation of the positions gives the same accepted entropies
        for perm in itertools.islice(itertools.permutations(range(L)), 6):
            rp = _accept(H[list(perm)], b=b)
            assert rp["n_accepted"] == r["n_accepted"]


def test_accept_invariants_and_monotone_in_b():
    rng = np.random.default_rng(5)
    for _ in range(20):
        H = rng.exponential(0.05, 256)
        ks = [_accept(H, b=b)["n_accepted"] for b in (0.0, 0.01, 0.1, 1.0, 10.0)]
        assert ks[0] >= 1
        assert all(a <= c for a, c in zip(ks, ks[1:]))


def test_renoise_and_commit():
    H = np.array([0.5, 0.01, 0.02, 0.9, 0.03], np.float32)
    smp = np.array([10, 11, 12, 13, 14], np.int32)
    cv = np.zeros(5, np.int32)
    r = oracle.accept_renoise(H, smp, cv, 1000, 0.1, 77, 5, 2)
    assert r["n_accepted"] == 4  # 0.01+0.02+0.03 = 0.06 <= 0.1; adding 0.5 exceeds
    assert r["order"].tolist() == [1, 2, 4, 0, 3]
    assert r["canvas"][[1, 2, 4, 0]].tolist() == [11, 12, 14, 10]
    tok = r["canvas"][3]
    assert tok == oracle.renoise_token(77, 5 + 3, 2, 1000) and 0 <= tok < 1000


def test_renoise_uniform_over_vocab():
    V = 16
    toks = np.array([oracle.renoise_token(1, r, 0, V) for r in range(32000)])
    counts = np.bincount(toks, minlength=V)
    chi2 = float(((counts - 2000) ** 2 / 2000).sum())
    assert chi2 < 37.7  # 15 dof, p = 0.001
    init = oracle.init_canvas(32000, V, 9)
    assert init.min() >= 0 and init.max() < V


# ------------------------------------------------------------------ stop / temperature
def test_stop_rule():
    a = np.arange(8, dtype=np.int32)
    lowH = np.full(8, 0.001, np.float32)
    assert oracle.stop(a, a, lowH, 0)["stop"] == 0            # step 0 has no previous step
    assert oracle.stop(a, a, lowH, 1)["stop"] == 1
    b = a.copy(); b[3] = 99
    assert oracle.stop(a, b, lowH, 5)["stop"] == 0            # argmax changed
    thr = float(np.float32(0.005))  # representable, so mean == thr exactly below
    assert oracle.stop(a, a, np.full(8, thr, np.float32), 5, thr)["stop"] == 0  # strict <
    assert oracle.stop(a, a, np.full(8, 0.0049, np.float32), 5)["stop"] == 1
    assert oracle.stop(a, a, np.full(8, 0.0051, np.float32), 5)["stop"] == 0


def test_temperature_schedule():
    g = dict((r[0], r[1]) for r in _read_golden("lab_exp_a_untrained.txt"))
    t0, t1, N = float(g["t_start"]), float(g["t_end"]), int(g["steps"])
    assert oracle.temperature(0, N, t0, t1) == t0
    assert abs(oracle.temperature(N - 1, N, t0, t1) - t1) < 1e-15
    ts = [oracle.temperature(k, N, t0, t1) for k in range(N)]
    d = np.diff(ts)
    assert np.allclose(d, (t1 - t0) / (N - 1), rtol=0, atol=1e-15)


# ------------------------------------------------------------------ attention
def _attn_inputs(B, L, P, Hq, Hkv, D, seed=0):
    rng = np.random.default_rng(seed)
    f = lambda *s: _bf16_bits(rng.standard_normal(s))
    return f(B, L, Hq, D), f(B, P, Hkv, D), f(B, P, Hkv, D), f(B, L, Hkv, D), f(B, L, Hkv, D)


def test_attention_matches_torch_sdpa_float64():
    B, L, P, Hq, Hkv, D = 2, 12, 9, 4, 2, 16
    q, kp, vp, kc, vc = _attn_inputs(B, L, P, Hq, Hkv, D)
    scale = 1.0 / math.sqrt(D)
    rows = np.arange(B * L * Hq)
    got = oracle.attention_rows(q, kp, vp, kc, vc, B, L, P, Hq, Hkv, D, scale, rows)
    f = lambda a: torch.from_numpy(oracle.bf16_bits_to_f64(a))
    Q = f(q).permute(0, 2, 1, 3)                                  # B, Hq, L, D
    K = torch.cat([f(kp), f(kc)], 1).permute(0, 2, 1, 3)          # B, Hkv, P+L, D
    Vv = torch.cat([f(vp), f(vc)], 1).permute(0, 2, 1, 3)
    K = K.repeat_interleave(Hq // Hkv, dim=1)
    Vv = Vv.repeat_interleave(Hq // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, scale=scale)
    ref = ref.permute(0, 2, 1, 3).reshape(-1, D).numpy()
    assert np.abs(got - ref).max() < 1e-12


def test_attention_special_cases():
    B, L, P, Hq, Hkv, D = 1, 5, 3, 2, 1, 8
    q, kp, vp, kc, vc = _attn_inputs(B, L, P, Hq, Hkv, D, seed=1)
    rows = np.arange(B * L * Hq)
    # every value row equal -> output equals that row
    row = _bf16_bits(np.linspace(-1, 1, D))
    vp1 = np.broadcast_to(row, vp.shape).copy()
    vc1 = np.broadcast_to(row, vc.shape).copy()
    out = oracle.attention_rows(q, kp, vp1, kc, vc1, B, L, P, Hq, Hkv, D, 0.3, rows)
    assert np.abs(out - oracle.bf16_bits_to_f64(row)[None]).max() < 1e-12
    # all keys zero -> uniform weights -> mean of the value rows
    z = np.zeros_like(kp)
    out = oracle.attention_rows(q, z, vp, np.zeros_like(kc), vc, B, L, P, Hq, Hkv, D, 0.3, rows)
    allv = np.concatenate([oracle.bf16_bits_to_f64(vp)[0, :, 0], oracle.bf16_bits_to_f64(vc)[0, :, 0]])
    assert np.abs(out - allv.mean(0)[None]).max() < 1e-12
    # a single key -> output is its value row
    out = oracle.attention_rows(q[:, :1], kp[:, :0], vp[:, :0], kc[:, :1], vc[:, :1],
                                1, 1, 0, Hq, Hkv, D, 0.3, np.arange(Hq))
    assert np.abs(out - oracle.bf16_bits_to_f64(vc)[0, 0, 0][None]).max() == 0.0


def test_causal_attention_matches_torch_sdpa_with_mask():
    """Cache-append forward: canvas position i sees all P cached keys and the
    canvas keys 0 .. i (an explicit boolean mask in torch's SDPA, float64)."""
    B, L, P, Hq, Hkv, D = 2, 11, 6, 4, 2, 16
    q, kp, vp, kc, vc = _attn_inputs(B, L, P, Hq, Hkv, D, seed=5)
    scale = 1.0 / math.sqrt(D)
    rows = np.arange(B * L * Hq)
    got = oracle.attention_rows(q, kp, vp, kc, vc, B, L, P, Hq, Hkv, D, scale, rows, causal=True)
    f = lambda a: torch.from_numpy(oracle.bf16_bits_to_f64(a))
    Q = f(q).permute(0, 2, 1, 3)
    K = torch.cat([f(kp), f(kc)], 1).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
    Vv = torch.cat([f(vp), f(vc)], 1).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
    keyj = torch.arange(P + L)[None, :]
    posi = torch.arange(L)[:, None]
    mask = (keyj < P) | (keyj - P <= posi)                       # [L, P + L]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, attn_mask=mask, scale=scale)
    ref = ref.permute(0, 2, 1, 3).reshape(-1, D).numpy()
    assert np.abs(got - ref).max() < 1e-12
    # without a cache the first canvas position sees only itself
    got0 = oracle.attention_rows(q, kp[:, :0], vp[:, :0], kc, vc, B, L, 0, Hq, Hkv, D, scale,
                                 np.arange(Hq), causal=True)
    assert np.abs(got0 - oracle.bf16_bits_to_f64(vc)[0, 0].repeat(Hq // Hkv, 0)).max() == 0.0
    # the last position sees every key: the same as the unmasked attention
    last = np.array([((b * L) + L - 1) * Hq + h for b in range(B) for h in range(Hq)])
    a = oracle.attention_rows(q, kp, vp, kc, vc, B, L, P, Hq, Hkv, D, scale, last, causal=True)
    u = oracle.attention_rows(q, kp, vp, kc, vc, B, L, P, Hq, Hkv, D, scale, last)
    assert np.array_equal(a, u)


# ------------------------------------------------------------------ LM-head GEMM
def test_logits_exact_on_small_integers():
    rng = np.random.default_rng(6)
    X = rng.integers(-8, 9, size=(7, 64)).astype(np.float32)
    W = rng.integers(-8, 9, size=(64, 100)).astype(np.float32)
    got = oracle.logits(_bf16_bits(X), _bf16_bits(W), col_chunk=33)
    ref = X.astype(np.int64) @ W.astype(np.int64)
    assert np.array_equal(got, ref.astype(np.float64))
    got_rows = oracle.logits(_bf16_bits(X), _bf16_bits(W), rows=[5, 2])
    assert np.array_equal(got_rows, ref[[5, 2]].astype(np.float64))


def test_bf16_widening_matches_torch():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(1000).astype(np.float32) * 100
    bits = _bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), ref)


# ------------------------------------------------------------------ the loop
def test_loop_flat_logits_commits_one_per_step_for_48_steps():
    """Lab EXP A: an unconfident (flat) model commits exactly one token per step,
    mean entropy stays at ln V and the loop runs to the 48-step cap."""
    g = dict((r[0], r[1]) for r in _read_golden("lab_exp_a_untrained.txt"))
    V, L, d = int(g["vocab"]), 16, 8
    w = _bf16_bits(np.random.default_rng(8).standard_normal((d, V)))
    hid = np.zeros((L, d), np.uint16)  # bf16 zeros -> every logit exactly 0
    res = oracle.block(lambda k: hid, w, 1, L, float(g["entropy_bound"]), 0,
                       max_steps=int(g["steps"]), t0=float(g["t_start"]), t1=float(g["t_end"]),
                       stop_threshold=float(g["stop_threshold"]))
    assert res["steps"][0] == int(g["steps"])
    for h in res["history"]:
        assert h["n_accepted"][0] == 1
        assert round(h["mean_entropy"][0], 2) == float(g["mean_entropy_nats"])
    assert (res["argmax"] == 0).all()


def test_loop_one_hot_stops_at_second_step():
    """One-hot logits: H = 0 at every position, argmax stable -> stops at k = 1 (2 forwards)."""
    V, L = 64, 8
    w = _bf16_bits(np.eye(V)[:L] * 1e4)          # d = L rows of W
    hid = _bf16_bits(np.eye(L))                   # position i -> logit 1e4 at vocab i
    res = oracle.block(lambda k: hid, w, 1, L, 0.1, 0, max_steps=48)
    assert res["steps"][0] == 2
    assert res["argmax"].tolist() == list(range(L))
    assert res["history"][0]["n_accepted"][0] == L  # all zero entropies fit the bound
    assert res["canvas"].tolist() == list(range(L))


def test_loop_batched_canvases_stop_independently():
    V, L = 64, 8
    w = _bf16_bits(np.eye(V)[:L] * 1e4)
    confident = _bf16_bits(np.eye(L))
    flat = np.zeros((L, L), np.uint16)
    hid = np.concatenate([confident, flat])      # canvas 0 confident, canvas 1 flat
    res = oracle.block(lambda k: hid, w, 2, L, 0.1, 3, max_steps=6)
    assert res["steps"].tolist() == [2, 6]


# ------------------------------------------------------------------ FP8 (E4M3) LM-head operands
def test_e4m3_decode_matches_torch_and_published_values():
    tab = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(tab), nan) and nan.sum() == 2       # 0x7F, 0xFF
    assert np.array_equal(tab[~nan], ref[~nan])
    # published landmarks of the format: largest finite, smallest normal and
    # subnormal, one, minus two
    assert tab[0x7E] == 448.0 and tab[0x08] == 2.0 ** -6 and tab[0x01] == 2.0 ** -9
    assert tab[0x38] == 1.0 and tab[0xC0] == -2.0 and tab[0x00] == 0.0


def test_e4m3_encode_nearest_even_and_saturating():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(3000) * 50, rng.uniform(-448, 448, 3000),
                        rng.standard_normal(1000) * 1e-3]).astype(np.float32)
    codes = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    # torch's conversion (round to nearest even) agrees on the finite range
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    # brute force: the decoded code is a nearest finite value
    tab = oracle.e4m3_table()
    fin = tab[np.isfinite(tab)]
    dist = np.abs(tab[codes] - x.astype(np.float64))
    best = np.abs(fin[None, :] - x.astype(np.float64)[:, None]).min(axis=1)
    assert np.array_equal(dist, best)
    # saturation instead of NaN beyond the largest finite value
    assert oracle.e4m3_encode(1e6) == 0x7E and oracle.e4m3_encode(-500.0) == 0xFE


def test_row_quantisation_scale_and_error_bound():
    rng = np.random.default_rng(9)
    x = _bf16_bits(rng.standard_normal((6, 300)) * rng.uniform(0.01, 100, (6, 1)))
    x[3] = 0   # an all-zero row: codes 0, scale 1
    q, sc = oracle.quantize_rows_e4m3(x)
    xf = oracle.bf16_bits_to_f64(x)
    tab = oracle.e4m3_table()
    assert (q[3] == 0).all() and sc[3] == 1.0
    for r in (0, 1, 2, 4, 5):
        amax = np.abs(xf[r]).max()
        assert sc[r] == np.float32(np.float32(amax) / np.float32(448.0))
        assert np.abs(tab[q[r]]).max() == 448.0          # the largest entry maps to 448
        # E4M3 keeps 3 mantissa bits: error <= 2^-4 of the value (normals) or
        # half the smallest subnormal step (2^-10) in code units
        err = np.abs(tab[q[r]] * sc[r] - xf[r])
        bound = np.maximum(np.abs(xf[r]) * 2.0 ** -4, 2.0 ** -10 * sc[r]) * 1.0001
        assert (err <= bound).all()


def test_fp8_logits_exact_on_small_integers():
    """Codes of small integers are exact: the FP8 logits equal the integer product."""
    rng = np.random.default_rng(10)
    X = rng.integers(-8, 9, size=(5, 64)).astype(np.float32)
    W = rng.integers(-8, 9, size=(64, 40)).astype(np.float32)
    x8 = np.array([[oracle.e4m3_encode(v) for v in row] for row in X], np.uint8)
    w8t = np.array([[oracle.e4m3_encode(v) for v in row] for row in W.T], np.uint8)
    got = oracle.logits_fp8(x8, np.ones(5, np.float32), w8t, np.ones(40, np.float32), col_chunk=7)
    assert np.array_equal(got, X.astype(np.float64) @ W.astype(np.float64))



# ------------------------------------------------------------------ self-conditioning read-out
def test_self_cond_uniform_logits_give_the_mean_row():
    """Equal logits: every token has weight 1/V, so the read-out is the mean of E's rows."""
    rng = np.random.default_rng(21)
    V, R = 1000, 30
    E = rng.standard_normal((V, R)).astype(np.float32)
    sc = oracle.self_cond(np.full((3, V), 2.5), 0.8, E)
    ref = E.astype(np.float64).mean(axis=0)
    assert np.abs(sc - ref).max() < 1e-12


def test_self_cond_one_hot_picks_the_row():
    """One logit 1e4 above the rest: every other weight underflows to 0 in fp64,
    so the read-out is that token's row of E, exactly."""
    rng = np.random.default_rng(22)
    V, R = 777, 32
    E = rng.standard_normal((V, R)).astype(np.float32)
    lg = rng.standard_normal((4, V))
    hot = [0, 5, 776, 300]
    for i, v in enumerate(hot):
        lg[i, v] = 1e4
    sc = oracle.self_cond(lg, 0.4, E)
    assert np.array_equal(sc, E[hot].astype(np.float64))


def test_self_cond_matches_torch_softmax_matmul():
    """Against torch in float64: softmax(logits / T) @ E (a library routine)."""
    rng = np.random.default_rng(23)
    V, R, T = 4096, 30, 0.8
    E = rng.standard_normal((V, R)).astype(np.float32)
    lg = rng.standard_normal((5, V)) * np.array([0.1, 1.0, 5.0, 20.0, 60.0])[:, None]
    sc = oracle.self_cond(lg, T, E)
    ref = (torch.softmax(torch.from_numpy(lg) / T, dim=1)
           @ torch.from_numpy(E.astype(np.float64))).numpy()
    assert np.abs(sc - ref).max() < 1e-12 * max(1.0, np.abs(ref).max())
    # the weights sum to one: a constant column of E reads out as that constant
    E2 = np.ones((V, 2), np.float32)
    E2[:, 1] = 3.0
    assert np.abs(oracle.self_cond(lg, T, E2) - np.array([1.0, 3.0])).max() < 1e-12


# ------------------------------------------------------------------ MoE FFN (decoder body)
def test_round_bf16_matches_torch_on_fp32_values_and_ties():
    rng = np.random.default_rng(31)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    # exact halfway cases: 8 significant bits + a half ulp, both parities
    halves = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(2.0 + 2.0 ** -7), 0.5 + 2.0 ** -9],
                      np.float32)
    x = np.concatenate([x, halves])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16_bits(x.astype(np.float64)), ref)


def test_topk_lowest_index_against_stable_sort():
    rng = np.random.default_rng(32)
    for _ in range(200):
        E = int(rng.integers(8, 130))
        k = int(rng.integers(1, min(8, E) + 1))
        row = rng.choice(np.linspace(-2, 2, 17), E)          # many ties
        ref = np.argsort(-row, kind="stable")[:k].tolist()
        assert oracle.topk_lowest_index(row, k) == ref


def test_gelu_tanh_matches_torch():
    x = np.linspace(-12, 12, 4001)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.abs(oracle.gelu_tanh(x) - ref).max() < 1e-14


def _moe_inputs(M, d, f, E, seed):
    rng = np.random.default_rng(seed)
    b = lambda a: _bf16_bits(a)
    return dict(x=b(rng.standard_normal((M, d))), wr=b(rng.standard_normal((E, d)) * 0.5),
                wg=b(rng.standard_normal((E + 1, f, d)) / np.sqrt(d)),
                wu=b(rng.standard_normal((E + 1, f, d)) / np.sqrt(d)),
                wd=b(rng.standard_normal((E + 1, d, f)) / np.sqrt(f)))


def test_moe_matches_dense_torch_evaluation():
    """Every expert on every token in torch float64, then weighted by a gate
    matrix built from torch.topk and torch.softmax: the routed sum."""
    M, d, f, E, k = 24, 64, 32, 16, 4
    a = _moe_inputs(M, d, f, E, 33)
    r = oracle.moe_ffn(a["x"], a["wr"], a["wg"], a["wu"], a["wd"], k)
    tb = lambda bits: torch.from_numpy(oracle.bf16_bits_to_f64(bits))
    X, Wr = tb(a["x"]), tb(a["wr"])
    lg = X @ Wr.T
    val, idx = torch.topk(lg, k, dim=1)
    G = torch.zeros(M, E, dtype=torch.float64)
    G.scatter_(1, idx, torch.softmax(val, dim=1))
    assert np.array_equal(np.sort(idx.numpy(), 1), np.sort(r["experts"], 1))

    def ffn(e):
        h = torch.nn.functional.gelu(X @ tb(a["wg"][e]).T, approximate="tanh") * (X @ tb(a["wu"][e]).T)
        h = torch.from_numpy(oracle.bf16_bits_to_f64(
            h.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)))
        return h @ tb(a["wd"][e]).T

    ref = ffn(E) + sum(G[:, e:e + 1] * ffn(e) for e in range(E))
    err = np.abs(r["out"] - ref.numpy()).max() / np.abs(ref.numpy()).max()
    assert err < 5e-3, err     # the two round the activation to bf16 by different paths
    assert np.abs(r["gates"].sum(axis=1) - 1).max() < 1e-12


def test_moe_top1_and_shared_only_cases():
    M, d, f, E = 8, 32, 16, 8
    a = _moe_inputs(M, d, f, E, 34)
    X = oracle.bf16_bits_to_f64(a["x"])
    tb = oracle.bf16_bits_to_f64

    def ffn(e, Xe):
        h = oracle.gelu_tanh(Xe @ tb(a["wg"][e]).T) * (Xe @ tb(a["wu"][e]).T)
        return tb(oracle.round_bf16_bits(h)) @ tb(a["wd"][e]).T

    # top-1: gate 1 on the best expert
    r = oracle.moe_ffn(a["x"], a["wr"], a["wg"], a["wu"], a["wd"], 1)
    assert np.array_equal(r["experts"][:, 0], np.argmax(X @ tb(a["wr"]).T, axis=1))
    assert (r["gates"] == 1.0).all()
    ref = ffn(E, X) + np.stack([ffn(int(e), X[t:t + 1])[0] for t, e in enumerate(r["experts"][:, 0])])
    assert np.abs(r["out"] - ref).max() < 1e-12 * np.abs(ref).max()
    # zero routed experts' down projections: only the shared expert is left
    wd = a["wd"].copy()
    wd[:E] = 0
    r = oracle.moe_ffn(a["x"], a["wr"], a["wg"], a["wu"], wd, 3)
    assert np.abs(r["out"] - ffn(E, X)).max() < 1e-12 * np.abs(r["out"]).max()
