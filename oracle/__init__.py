"""fp64 oracle for the block-diffusion denoising step -- TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library: the per-position sampler, acceptance rule, stop test, Philox and the
attention loops live in ``dg_oracle.c`` (plain single-threaded C, fp64); the
LM-head product uses numpy's float64 matmul as a library step.  bf16 tensors
are passed as raw ``uint16`` bit patterns and widened exactly to fp64.

Sources, by page title and section:
  * "DiffusionGemma Lab", section 2, items 1-7 (the sampler as coded).
  * "DiffusionGemma: Parallel Denoising From an Autoregressive Checkpoint",
    section "Finding" (entropy-bounded acceptance, temperature annealing,
    adaptive stopping; causal encoder cache + bidirectional canvas decoder).
  * Salmon et al., SC'11, for Philox4x32-10.

Parity unpinned: the number of steps a converging block loop takes (no page
gives one); everything else is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_c_i32 = ctypes.c_int32
_c_u32 = ctypes.c_uint32
_c_u64 = ctypes.c_uint64
_c_i64 = ctypes.c_int64
_c_dbl = ctypes.c_double
_c_flt = ctypes.c_float
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile dg_oracle.c into liboracle.so with gcc (no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        L.orc_philox4x32_10.argtypes = [_vp, _vp, _vp]
        L.orc_philox4x32_10.restype = None
        L.orc_gumbel_bits.argtypes = [_c_u64, _c_u32, _c_u32, _c_u32]
        L.orc_gumbel_bits.restype = _c_u32
        L.orc_renoise_token.argtypes = [_c_u64, _c_u32, _c_u32, _c_i32]
        L.orc_renoise_token.restype = _c_i32
        L.orc_init_token.argtypes = [_c_u64, _c_u32, _c_i32]
        L.orc_init_token.restype = _c_i32
        L.orc_init_canvas.argtypes = [_vp, _c_i32, _c_i32, _c_u64]
        L.orc_init_canvas.restype = None
        L.orc_logf.argtypes = [_c_flt]
        L.orc_logf.restype = _c_flt
        L.orc_uniform_open.argtypes = [_c_u32]
        L.orc_uniform_open.restype = _c_flt
        L.orc_gumbel_from_bits.argtypes = [_c_u32]
        L.orc_gumbel_from_bits.restype = _c_flt
        L.orc_sampler_row.argtypes = [_vp, _c_i32, _c_dbl, _c_u64, _c_u32, _c_u32,
                                      _vp, _vp, _vp, _vp, _vp]
        L.orc_sampler_row.restype = None
        L.orc_accept_renoise.argtypes = [_vp, _vp, _vp, _vp, _c_i32, _c_i32, _c_dbl,
                                         _c_u64, _c_u32, _c_u32, _vp, _vp]
        L.orc_accept_renoise.restype = _c_i32
        L.orc_stop.argtypes = [_vp, _vp, _vp, _c_i32, _c_i32, _c_dbl, _vp]
        L.orc_stop.restype = _c_i32
        L.orc_temperature.argtypes = [_c_i32, _c_i32, _c_dbl, _c_dbl]
        L.orc_temperature.restype = _c_dbl
        L.orc_attention_rows.argtypes = [_vp, _vp, _vp, _vp, _vp,
                                         _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                         _c_dbl, _vp, _c_i64, _vp]
        L.orc_attention_rows.restype = None
        L.orc_attention_rows_ex.argtypes = [_vp, _vp, _vp, _vp, _vp,
                                            _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                            _c_dbl, _c_i32, _vp, _c_i64, _vp]
        L.orc_attention_rows_ex.restype = None
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode.restype = _c_dbl
        L.orc_e4m3_encode.argtypes = [_c_flt]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_quantize_rows_e4m3.argtypes = [_vp, _c_i64, _c_i64, _vp, _vp]
        L.orc_quantize_rows_e4m3.restype = None
        L.orc_gumbel_fill.argtypes = [_c_u64, _c_u32, _c_u32, _c_u32, _c_i32, _vp]
        L.orc_gumbel_fill.restype = None
        L.orc_self_cond_row.argtypes = [_vp, _c_i32, _c_dbl, _vp, _c_i32, _vp]
        L.orc_self_cond_row.restype = None
        L.orc_round_bf16.argtypes = [_c_dbl]
        L.orc_round_bf16.restype = ctypes.c_uint16
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(_vp)


# ---------------------------------------------------------------- primitives
def philox4x32_10(ctr: Sequence[int], key: Sequence[int]) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def logf(x: float) -> float:
    return float(np.float32(lib().orc_logf(float(x))))


def uniform_open(bits: int) -> float:
    return float(np.float32(lib().orc_uniform_open(int(bits))))


def gumbel_from_bits(bits: int) -> float:
    return float(np.float32(lib().orc_gumbel_from_bits(int(bits))))


def gumbel_fill(seed: int, row: int, step: int, v0: int, n: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.float32)
    lib().orc_gumbel_fill(seed, row, step, v0, n, _ptr(out))
    return out


def gumbel_bits(seed: int, row: int, step: int, v: int) -> int:
    return int(lib().orc_gumbel_bits(seed, row, step, v))


def renoise_token(seed: int, row: int, step: int, V: int) -> int:
    return int(lib().orc_renoise_token(seed, row, step, V))


def init_canvas(n: int, V: int, seed: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.int32)
    lib().orc_init_canvas(_ptr(out), n, V, seed)
    return out


def temperature(k: int, N: int, t0: float = 0.8, t1: float = 0.4) -> float:
    return float(lib().orc_temperature(k, N, t0, t1))


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bit patterns (uint16) to float64."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- LM head
def logits(x_bits: np.ndarray, w_bits: np.ndarray, rows: Optional[Sequence[int]] = None,
           col_chunk: int = 32768) -> np.ndarray:
    """fp64 logits X[rows] @ W for bf16 X [M, d] and W [d, V] (raw bits).

    The product is numpy's float64 matmul (a library step); columns of W are
    widened chunk by chunk to bound host memory.
    """
    X = bf16_bits_to_f64(x_bits if rows is None else np.asarray(x_bits)[np.asarray(rows)])
    d, V = w_bits.shape
    out = np.empty((X.shape[0], V), dtype=np.float64)
    for c0 in range(0, V, col_chunk):
        c1 = min(V, c0 + col_chunk)
        out[:, c0:c1] = X @ bf16_bits_to_f64(w_bits[:, c0:c1])
    return out


# ---------------------------------------------------------------- sampler
def sampler_row(logits_row: np.ndarray, T: float, seed: int, row: int, step: int) -> dict:
    lr = np.ascontiguousarray(np.asarray(logits_row, dtype=np.float64))
    H = ctypes.c_double()
    smp = ctypes.c_int32()
    am = ctypes.c_int32()
    gm = ctypes.c_double()
    amm = ctypes.c_double()
    lib().orc_sampler_row(_ptr(lr), lr.shape[0], float(T), seed, row, step,
                          ctypes.byref(H), ctypes.byref(smp), ctypes.byref(am),
                          ctypes.byref(gm), ctypes.byref(amm))
    return dict(H=H.value, sample=smp.value, argmax=am.value,
                gumbel_margin=gm.value, argmax_margin=amm.value)


def sampler(logits_rows: np.ndarray, T: float, seed: int, rows: Sequence[int], step: int,
            workers: int = 1) -> dict:
    """Run sampler_row over a block of logits; rows[i] is the global row id of logits_rows[i].

    Rows are independent; ``workers`` > 1 runs them on that many threads (the
    C routine runs without the interpreter lock), with identical results.
    """
    n = logits_rows.shape[0]
    res = dict(H=np.zeros(n), sample=np.zeros(n, np.int32), argmax=np.zeros(n, np.int32),
               gumbel_margin=np.zeros(n), argmax_margin=np.zeros(n))

    def one(t):
        r = sampler_row(logits_rows[t], T, seed, int(rows[t]), step)
        for k in res:
            res[k][t] = r[k]

    if workers > 1 and n > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, range(n)))
    else:
        for t in range(n):
            one(t)
    return res


def accept_renoise(H: np.ndarray, sample: np.ndarray, canvas: np.ndarray, V: int, b: float,
                   seed: int, row_base: int, step: int) -> dict:
    """One canvas: returns the new canvas, accepted mask, k*, sorted order, boundary gap."""
    Hf = np.ascontiguousarray(np.asarray(H, dtype=np.float32))
    sm = np.ascontiguousarray(np.asarray(sample, dtype=np.int32))
    cv = np.ascontiguousarray(np.array(canvas, dtype=np.int32, copy=True))
    L = Hf.shape[0]
    acc = np.zeros(L, dtype=np.uint8)
    order = np.zeros(L, dtype=np.int32)
    gap = ctypes.c_double()
    k = lib().orc_accept_renoise(_ptr(Hf), _ptr(sm), _ptr(cv), _ptr(acc), L, V, float(b),
                                 seed, row_base, step, _ptr(order), ctypes.byref(gap))
    return dict(canvas=cv, accepted=acc, n_accepted=int(k), order=order, boundary_gap=gap.value)


def stop(argmax: np.ndarray, prev_argmax: np.ndarray, H: np.ndarray, step: int,
         threshold: float = 0.005) -> dict:
    a = np.ascontiguousarray(np.asarray(argmax, dtype=np.int32))
    p = np.ascontiguousarray(np.asarray(prev_argmax, dtype=np.int32))
    Hf = np.ascontiguousarray(np.asarray(H, dtype=np.float32))
    mean = ctypes.c_double()
    s = lib().orc_stop(_ptr(a), _ptr(p), _ptr(Hf), a.shape[0], step, float(threshold),
                       ctypes.byref(mean))
    return dict(stop=int(s), mean_entropy=mean.value)


def self_cond(logits_rows: np.ndarray, T: float, E: np.ndarray, workers: int = 1) -> np.ndarray:
    """Self-conditioning read-out sc[i] = sum_v softmax(logits_i / T)_v E[v, :] (fp64)
    for every row of a block of fp64 logits; E is the fp32 table [V, R].

    Rows are independent; ``workers`` > 1 runs them on that many threads
    (identical results)."""
    lg = np.ascontiguousarray(np.asarray(logits_rows, dtype=np.float64))
    Et = np.ascontiguousarray(np.asarray(E, dtype=np.float32))
    n, V = lg.shape
    R = Et.shape[1]
    assert Et.shape[0] == V
    out = np.zeros((n, R), dtype=np.float64)

    def one(t):
        lib().orc_self_cond_row(_ptr(lg[t]), V, float(T), _ptr(Et), R, _ptr(out[t]))

    if workers > 1 and n > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, range(n)))
    else:
        for t in range(n):
            one(t)
    return out


# ---------------------------------------------------------------- attention
def attention_rows(q, kp, vp, kc, vc, B, L, P, Hq, Hkv, D, scale, rows,
                   causal: bool = False) -> np.ndarray:
    """fp64 attention for the listed flat query rows (b*L+i)*Hq+h; bf16 inputs as uint16.

    causal: the encoder's cache-append forward -- the query at canvas
    position i sees the P cached keys and the canvas keys 0 .. i.
    """
    arrs = [np.ascontiguousarray(np.asarray(a, dtype=np.uint16)) for a in (q, kp, vp, kc, vc)]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((r.shape[0], D), dtype=np.float64)
    lib().orc_attention_rows_ex(*[_ptr(a) for a in arrs], B, L, P, Hq, Hkv, D, float(scale),
                                1 if causal else 0, _ptr(r), r.shape[0], _ptr(out))
    return out


# ---------------------------------------------------------------- FP8 (E4M3) LM head
def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(int(code)))


def e4m3_encode(x: float) -> int:
    return int(lib().orc_e4m3_encode(float(x)))


def e4m3_table() -> np.ndarray:
    """Values of all 256 codes (NaN for 0x7F, 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)])


def quantize_rows_e4m3(x_bits: np.ndarray, workers: int = 1):
    """Per-row E4M3 quantisation of bf16 rows [n, c] -> (codes uint8 [n, c], scale fp32 [n]).

    Rows are independent; ``workers`` > 1 runs blocks of rows on that many
    threads (the C routine runs without the interpreter lock), with identical
    results."""
    x = np.ascontiguousarray(np.asarray(x_bits, dtype=np.uint16))
    n, c = x.shape
    q = np.zeros((n, c), np.uint8)
    sc = np.zeros(n, np.float32)
    L = lib()
    L.orc_e4m3_encode(0.0)          # fills the encoder's code table before any thread runs

    def block(r0, r1):
        L.orc_quantize_rows_e4m3(_ptr(x[r0:r1]), r1 - r0, c, _ptr(q[r0:r1]), _ptr(sc[r0:r1]))

    if workers > 1 and n > 1:
        from concurrent.futures import ThreadPoolExecutor
        step = -(-n // (4 * workers))
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(lambda r0: block(r0, min(n, r0 + step)), range(0, n, step)))
    else:
        block(0, n)
    return q, sc


def quantize_weight_e4m3(w_bits: np.ndarray, workers: int = 1):
    """W [d, V] (bf16 bits) -> (W8t [V, d] codes, scale [V]): each vocabulary
    column quantised as one row."""
    return quantize_rows_e4m3(np.ascontiguousarray(np.asarray(w_bits, dtype=np.uint16).T),
                              workers=workers)


def logits_fp8(x8: np.ndarray, sx: np.ndarray, w8t: np.ndarray, sw: np.ndarray,
               col_chunk: int = 32768) -> np.ndarray:
    """fp64 logits of the quantised operands: (dec(x8) sx) (dec(w8t) sw)^T."""
    tab = e4m3_table()
    X = tab[np.asarray(x8)] * np.asarray(sx, np.float64)[:, None]
    V = w8t.shape[0]
    out = np.empty((X.shape[0], V))
    for c0 in range(0, V, col_chunk):
        c1 = min(V, c0 + col_chunk)
        Wc = tab[np.asarray(w8t[c0:c1])] * np.asarray(sw[c0:c1], np.float64)[:, None]
        out[:, c0:c1] = X @ Wc.T
    return out


# ---------------------------------------------------------------- step / block
def step(x_bits: np.ndarray, w_bits: np.ndarray, canvas: np.ndarray, prev_argmax: np.ndarray,
         B: int, L: int, T: float, b: float, seed: int, k: int,
         stop_threshold: float = 0.005, workers: int = 1, lg: Optional[np.ndarray] = None) -> dict:
    """One denoising step (LM head -> sampler -> accept/renoise -> stop) for B canvases.

    lg: precomputed fp64 logits (e.g. of the FP8 operands); x_bits/w_bits are
    then used only for the vocabulary size."""
    V = w_bits.shape[1] if lg is None else lg.shape[1]
    if lg is None:
        lg = logits(x_bits, w_bits)
    s = sampler(lg, T, seed, np.arange(B * L), k, workers=workers)
    Hf = s["H"].astype(np.float32)
    new_canvas = np.array(canvas, dtype=np.int32, copy=True).reshape(B, L)
    accepted = np.zeros((B, L), np.uint8)
    n_acc = np.zeros(B, np.int32)
    stops = np.zeros(B, np.int32)
    means = np.zeros(B)
    gaps = np.zeros(B)
    orders = np.zeros((B, L), np.int32)
    for bb in range(B):
        sl = slice(bb * L, (bb + 1) * L)
        a = accept_renoise(Hf[sl], s["sample"][sl], new_canvas[bb], V, b, seed, bb * L, k)
        new_canvas[bb] = a["canvas"]
        accepted[bb] = a["accepted"]
        n_acc[bb] = a["n_accepted"]
        gaps[bb] = a["boundary_gap"]
        orders[bb] = a["order"]
        st = stop(s["argmax"][sl], np.asarray(prev_argmax).reshape(B, L)[bb], Hf[sl], k,
                  stop_threshold)
        stops[bb] = st["stop"]
        means[bb] = st["mean_entropy"]
    return dict(logits=lg, H=s["H"], H32=Hf, sample=s["sample"], argmax=s["argmax"],
                gumbel_margin=s["gumbel_margin"], argmax_margin=s["argmax_margin"],
                canvas=new_canvas.reshape(-1), accepted=accepted.reshape(-1),
                n_accepted=n_acc, stop=stops, mean_entropy=means, boundary_gap=gaps,
                order=orders)


def block(hidden_bits_fn, w_bits: np.ndarray, B: int, L: int, b: float, seed: int,
          max_steps: int = 48, t0: float = 0.8, t1: float = 0.4,
          stop_threshold: float = 0.005, workers: int = 1) -> dict:
    """The denoising loop of a batch of B independent canvases.

    [Lab] items 1-5: uniform init, per-step sample/accept/renoise, linear
    temperature, adaptive stop; the result is the argmax canvas of the step
    at which a canvas stopped (or of the last step).  ``hidden_bits_fn(k)``
    returns the bf16 hidden states [B*L, d] of step k (the decoder body is
    outside this path); a function of two arguments is called as
    ``hidden_bits_fn(k, canvas)`` with the canvas [B*L] the step starts from
    (a decoder that reads the canvas).  Each canvas stops on its own: once its
    stop test fires, its canvas, argmax and step count are frozen.
    """
    import inspect
    two = len(inspect.signature(hidden_bits_fn).parameters) >= 2
    V = w_bits.shape[1]
    canvas = init_canvas(B * L, V, seed).reshape(B, L)
    prev = np.zeros((B, L), np.int32)
    out_argmax = np.zeros((B, L), np.int32)
    steps = np.zeros(B, np.int32)
    done = np.zeros(B, bool)
    history = []
    for k in range(max_steps):
        T = temperature(k, max_steps, t0, t1)
        hk = hidden_bits_fn(k, canvas.reshape(-1).copy()) if two else hidden_bits_fn(k)
        r = step(hk, w_bits, canvas.reshape(-1), prev.reshape(-1), B, L, T, b,
                 seed, k, stop_threshold, workers=workers)
        am = r["argmax"].reshape(B, L)
        cv = r["canvas"].reshape(B, L)
        live = ~done
        canvas[live] = cv[live]
        out_argmax[live] = am[live]
        steps[live] = k + 1
        history.append(dict(T=T, live=live.copy(), n_accepted=r["n_accepted"].copy(),
                            stop=r["stop"].copy(), mean_entropy=r["mean_entropy"].copy(),
                            argmax=r["argmax"].copy(), canvas=r["canvas"].copy(),
                            H32=r["H32"].copy(), sample=r["sample"].copy(),
                            gumbel_margin=r["gumbel_margin"].copy(),
                            argmax_margin=r["argmax_margin"].copy(),
                            boundary_gap=r["boundary_gap"].copy(), order=r["order"].copy()))
        done = done | (r["stop"] == 1)
        prev = am.copy()
        if bool(np.all(done)):
            break
    return dict(steps=steps, argmax=out_argmax.reshape(-1), canvas=canvas.reshape(-1),
                history=history)


# ---------------------------------------------------------------- MoE FFN (decoder body)
def round_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 (ties to even) of each float64, as raw bits (dg_oracle.c)."""
    a = np.asarray(x, dtype=np.float64).ravel()
    L = lib()
    out = np.fromiter((L.orc_round_bf16(float(v)) for v in a), dtype=np.uint16, count=a.shape[0])
    return out.reshape(np.shape(x))


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def topk_lowest_index(row: np.ndarray, k: int):
    """The k largest entries of a row, largest first, ties to the lower index:
    k rounds of 'take the first maximum of what is left'."""
    left = [float(v) for v in row]
    chosen = []
    for _ in range(k):
        best = None
        for e, v in enumerate(left):
            if v is None:
                continue
            if best is None or v > left[best]:
                best = e
        chosen.append(best)
        left[best] = None
    return chosen


def moe_ffn(x_bits: np.ndarray, wr_bits: np.ndarray, wg_bits: np.ndarray, wu_bits: np.ndarray,
            wd_bits: np.ndarray, top_k: int) -> dict:
    """A mixture-of-experts FFN over the canvas hidden states, fp64.

    "DiffusionGemma: When the LLM Stops Writing Left to Right", section "What
    DiffusionGemma Actually Is" (128 experts, top-8 routing plus one shared
    expert) and "Parallel Denoising From an Autoregressive Checkpoint",
    section "Finding" (the MoE layer of a canvas forward touches ~84 distinct
    experts).  Readings (the pages give no formulas): router logits
    l = X Wr^T; each token takes its top_k experts by logit (ties to the
    lower index) with gates softmax(l_selected); every expert, and the
    shared one (index E of the weight stacks, gate 1), is a gated GELU FFN
    (gelu_tanh(x Wg^T) * (x Wu^T)) Wd^T whose intermediate activation is
    stored as bf16; out = shared(x) + sum_j gate_j expert_j(x).
    Weights as raw bf16 bits: wr [E, d], wg / wu [E + 1, f, d], wd [E + 1, d, f].
    The matmuls are numpy float64 (library steps).
    """
    X = bf16_bits_to_f64(x_bits)
    Wr = bf16_bits_to_f64(wr_bits)
    M, d = X.shape
    E = Wr.shape[0]
    lg = X @ Wr.T
    experts = np.zeros((M, top_k), np.int32)
    gates = np.zeros((M, top_k))
    margin = np.full(M, np.inf)
    for t in range(M):
        sel = topk_lowest_index(lg[t], top_k)
        experts[t] = sel
        z = lg[t, sel]
        g = np.exp(z - z.max())
        gates[t] = g / g.sum()
        if top_k < E:
            rest = np.delete(lg[t], sel)
            margin[t] = lg[t, sel[-1]] - rest.max()

    def ffn(e, Xe):
        Wg = bf16_bits_to_f64(wg_bits[e])
        Wu = bf16_bits_to_f64(wu_bits[e])
        Wd = bf16_bits_to_f64(wd_bits[e])
        h = gelu_tanh(Xe @ Wg.T) * (Xe @ Wu.T)
        hb = bf16_bits_to_f64(round_bf16_bits(h))
        return hb @ Wd.T

    out = ffn(E, X)                      # the shared expert, every token
    for e in range(E):
        rows, slots = np.nonzero(experts == e)
        if rows.shape[0] == 0:
            continue
        out[rows] += gates[rows, slots][:, None] * ffn(e, X[rows])
    return dict(out=out, experts=experts, gates=gates, router_logits=lg, margin=margin,
                distinct=int(np.unique(experts).shape[0]))
