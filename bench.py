"""Benchmark of one denoising step of block diffusion on GB300.

A step = canvas attention over [KV cache ; canvas] + LM head with the fused
entropy / Gumbel-max / argmax epilogue + acceptance / renoise / stop test,
all through the C ABI of libdg.so.  The default workload is the full-width
single step (16 query / 8 kv heads, head dim 256, 4096 cached keys, LM head
2816 x 262144, per-row logit scale U(0.5, 8), T = 0.8, b = 0.1).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own independent canvas (replicas,
no data-path collective); value = total steps/s over all ranks.
The reference arm (--impl reference) times the fp64 CPU oracle on a bounded
sample of the same workload and scales it to the full step.
"""
from __future__ import annotations

import os

# The CPU oracle runs single-threaded (BLAS included) so its core count is exact.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dg_synth  # noqa: E402

DEFAULT_CONFIG = "step_full"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# nominal dense peaks of the part (HBM3e bandwidth, bf16 tensor rate), reported
# beside the measured ones
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0


# Arm cores by (implementer, part) as /proc/cpuinfo gives them
_ARM_PARTS = {("0x41", "0xd4f"): "Arm Neoverse V2", ("0x41", "0xd40"): "Arm Neoverse V1",
              ("0x41", "0xd0c"): "Arm Neoverse N1", ("0x41", "0xd49"): "Arm Neoverse N2"}


def _host_cpu():
    """The host's CPU model (best effort) and logical core count."""
    import platform
    model = platform.processor() or platform.machine()
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" not in line:
                    continue
                k, v = (x.strip() for x in line.split(":", 1))
                fields.setdefault(k.lower(), v)
    except OSError:
        pass
    if fields.get("model name"):
        model = fields["model name"]
    elif "cpu implementer" in fields and "cpu part" in fields:
        imp, part = fields["cpu implementer"].lower(), fields["cpu part"].lower()
        model = _ARM_PARTS.get((imp, part), "Arm implementer %s part %s" % (imp, part))
    return dict(cpu_model=model, machine=platform.machine(), nproc=os.cpu_count())


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _reduce_max(value, device):
    """The largest of `value` over the ranks of the initialised process group
    (the slowest replica's time), or `value` itself without one."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return value
    t = torch.tensor([value], device=device, dtype=torch.float64)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def _replica_value(world, ms):
    """Whole-job rate of `world` independent replicas whose slowest rank took
    `ms` per unit (steps/s, appends/s)."""
    return world * 1e3 / ms


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def wait_first(self, timeout=3.0):
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout:
            time.sleep(0.01)

    def mark(self, t_start, t_end):
        """The timed region; samples within 0.25 s of it are kept (nvidia-smi
        samples every 200 ms, so a short region still gets its neighbours)."""
        self.window = (t_start - 0.25, t_end + 0.25)
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 0.5 and not any(t > t_end for t, _ in self.lines):
            time.sleep(0.01)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = getattr(self, "window", (-1e30, 1e30))
        for t, ln in self.lines:
            if not lo <= t <= hi:
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle sample
def oracle_step_estimate(cfg, inputs_host, v_sample=8192, attn_rows=64, seed=0, fp8=False,
                         sc_table=None):
    """Time the CPU oracle on a bounded sample of one step and scale it to the full step.

    Sample: every canvas row of the LM head + sampler against the first v_sample
    vocabulary columns (time scaled by V / v_sample), attention for attn_rows of
    the B*L*Hq query rows (scaled by the row count), the acceptance + stop test on
    the full canvas.  fp8: the LM head on E4M3 operands (the oracle quantises
    the hidden rows and the sampled W columns, then forms the fp64 logits of the
    quantised operands).  Returns (seconds per full step, description).
    """
    import oracle
    xb, wb = inputs_host["x"], inputs_host["w"]
    vs = min(v_sample, cfg.V)
    w_s = np.ascontiguousarray(wb[:, :vs])
    t0 = time.perf_counter()
    if fp8:
        x8, sx = oracle.quantize_rows_e4m3(xb)
        w8t, sw = oracle.quantize_weight_e4m3(w_s)
        lg = oracle.logits_fp8(x8, sx, w8t, sw)
    else:
        lg = oracle.logits(xb, w_s)
    s = oracle.sampler(lg, cfg.temperature, seed, np.arange(cfg.M), 1)
    if sc_table is not None:
        oracle.self_cond(lg, cfg.temperature, np.ascontiguousarray(sc_table[:vs]))
    t_lm = time.perf_counter() - t0
    rows = np.linspace(0, cfg.B * cfg.L * cfg.Hq - 1, attn_rows).astype(np.int64)
    t0 = time.perf_counter()
    oracle.attention_rows(inputs_host["q"], inputs_host["kp"], inputs_host["vp"],
                          inputs_host["kc"], inputs_host["vc"], cfg.B, cfg.L, cfg.P, cfg.Hq,
                          cfg.Hkv, cfg.D, 1.0 / math.sqrt(cfg.D), rows)
    t_at = time.perf_counter() - t0
    t0 = time.perf_counter()
    Hf = s["H"].astype(np.float32)
    for b in range(cfg.B):
        sl = slice(b * cfg.L, (b + 1) * cfg.L)
        oracle.accept_renoise(Hf[sl], s["sample"][sl], np.zeros(cfg.L, np.int32), cfg.V,
                              cfg.entropy_bound, seed, b * cfg.L, 1)
        oracle.stop(s["argmax"][sl], s["argmax"][sl], Hf[sl], 1)
    t_acc = time.perf_counter() - t0
    full = t_lm * (cfg.V / vs) + t_at * (cfg.B * cfg.L * cfg.Hq / len(rows)) + t_acc
    desc = ("oracle (fp64 C + numpy fp64 matmul, 1 thread): all %d canvas rows x %d of %d vocab "
            "columns (%sLM head + sampler%s, scaled x%.0f), %d of %d attention rows (scaled), "
            "acceptance + stop on the full canvas" % (cfg.M, vs, cfg.V,
                                                      "E4M3 quantisation + " if fp8 else "",
                                                      " + self-conditioning read-out"
                                                      if sc_table is not None else "",
                                                      cfg.V / vs, len(rows),
                                                      cfg.B * cfg.L * cfg.Hq))
    return full, desc, dict(t_lm=t_lm, t_attn=t_at, t_accept=t_acc)


# The oracle's sample of a step, the same in the reference arm and in the GPU
# arm's cpu_baseline: every canvas row against the first ORACLE_V_SAMPLE
# vocabulary columns, ORACLE_ATTN_ROWS attention rows.
ORACLE_V_SAMPLE = 16384
ORACLE_ATTN_ROWS = 64


def host_inputs_small_sample(cfg, seed=0):
    """Host (numpy, bf16 bits) inputs of the workload for the oracle sample; W is drawn
    only for the sampled columns to keep the reference arm bounded."""
    cfg_s = dg_synth.StepConfig(cfg.name + "_cols", B=cfg.B, L=cfg.L, Hq=cfg.Hq, Hkv=cfg.Hkv,
                                D=cfg.D, P=cfg.P, d=cfg.d, V=min(cfg.V, ORACLE_V_SAMPLE),
                                w_std=cfg.w_std,
                                row_scale=cfg.row_scale, seed=seed)
    out = dict(dg_synth.attention_inputs(cfg_s))
    out["x"] = dg_synth.lm_hidden(cfg_s)
    out["w"] = dg_synth.lm_weight(cfg_s)
    return out


def run_reference(args, cfg):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    host = host_inputs_small_sample(cfg, seed=cfg.seed)
    times, walls = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        t, desc, parts = oracle_step_estimate(cfg, host, v_sample=ORACLE_V_SAMPLE,
                                              attn_rows=ORACLE_ATTN_ROWS, seed=i)
        if i >= args.warmup:
            times.append(t)
            walls.append(sum(parts.values()))
    per = sum(times) / len(times)
    value = 1.0 / per
    line = dict(impl="reference", metric="denoise steps/s (256-tok canvas, bs=1)",
                value=value, unit="steps/s", n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, ms_per_step=per * 1e3, higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                config=_config_json(cfg, l2="n/a (CPU)"),
                cpu_baseline=dict(value=value, unit="steps/s", cores=1, kind="oracle", **_host_cpu(),
                                  sample=desc),
                e2e=dict(value=value, unit="steps/s", h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0),
                # ms_per_step is the sample's time scaled to a whole step; the
                # oracle actually ran this long per timed step
                sample_wall_s_per_step=sum(walls) / len(walls))
    print(json.dumps(line), flush=True)
    return 0


def run_reference_moe(args, mcfg):
    """The oracle on the MoE workload (host cores, one thread): the whole
    layer, all canvas rows, as the GPU arm's cpu_baseline times it (a
    couple of seconds per layer)."""
    ws_, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    a = dg_synth.moe_inputs(mcfg)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.moe_ffn(a["x"], a["wr"], a["wg"], a["wu"], a["wd"], mcfg.top_k)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    walls = times
    per = sum(times) / len(times)
    value = 1.0 / per
    desc = ("oracle (numpy fp64 matmuls + plain routing, 1 thread): the whole layer, all %d "
            "rows" % mcfg.M)
    line = dict(impl="reference", metric="MoE FFN layers/s (256-token canvas)", value=value,
                unit="layers/s", n_gpus=args.gpus, steps=args.steps, warmup=args.warmup,
                ms_per_step=per * 1e3, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic",
                config={"workload": "%s: MoE FFN over the canvas, M=%d, d=%d, %d experts of f=%d, "
                                    "top-%d + 1 shared" % (mcfg.name, mcfg.M, mcfg.d, mcfg.E,
                                                           mcfg.f, mcfg.top_k),
                        "global_batch": 1, "seq_len": mcfg.M, "parallelism": "replicas",
                        "l2": "n/a (CPU)"},
                cpu_baseline=dict(value=value, unit="layers/s", cores=1, kind="oracle", **_host_cpu(),
                                  sample=desc),
                e2e=dict(value=value, unit="layers/s", h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0),
                sample_wall_s_per_step=sum(walls) / len(walls))
    print(json.dumps(line), flush=True)
    return 0


W_LAYOUTS = {0: "row-major [d, V]", 1: "packed [ceil(V/128)][d][128] (dg_pack_lm_weight, at load)"}


def _config_json(cfg, l2, lm_dtype="bf16", self_cond=False, w_layout=None):
    out = {"workload": "%s: single denoising step, B=%d L=%d, attention Hq=%d Hkv=%d D=%d "
                       "P=%d, LM head d=%d V=%d%s%s, T=%.1f b=%.1f" % (
                           cfg.name, cfg.B, cfg.L, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.d, cfg.V,
                           " (E4M3 operands, per-row / per-column scales)"
                           if lm_dtype == "fp8" else "",
                           " + self-conditioning read-out (bf16 table [V, 32])"
                           if self_cond else "",
                           cfg.temperature, cfg.entropy_bound),
           "global_batch": cfg.B, "seq_len": cfg.L, "parallelism": "replicas", "l2": l2}
    if w_layout is not None:
        out["w_layout"] = W_LAYOUTS[w_layout]
    return out


# ----------------------------------------------------------------------------- our arm
def _w_columns(w, packed, d, ncols):
    """The first ncols columns of the LM-head weight as [d, ncols] (row-major),
    from W [d, V] or from its packed form [V/128][d][128] (ncols % 128 == 0)."""
    if not packed:
        return w[:, :ncols].contiguous()
    return w.view(-1, d, 128)[:ncols // 128].permute(1, 0, 2).reshape(d, ncols)


def _traffic_record(kernel_sources, kernel, shape):
    """Per-launch DRAM bytes of the LM-head kernel from its committed ncu summary
    (profiles/<kernel>_step_full.md), valid only while the kernel sources are
    unchanged and for the same kernel and GEMM shape (rows, d, V)."""
    path = os.path.join(ROOT, "profiles", "%s_step_full.md" % kernel)
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in kernel_sources:
        with open(f, "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    rec = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("source_sha256_16") != digest or rec.get("kernel") != kernel:
        return None
    if rec.get("shape") != "x".join(str(v) for v in shape):
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def run_ours(args, cfg, emit=True):
    import torch
    import block_diffusion_decoding_gb300 as dg
    from block_diffusion_decoding_gb300 import build as dgbuild

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
    dgbuild.build()
    dg.lib()
    hbm_peak, bf16_peak, peak_kind = _peaks()

    # ---- synthetic inputs, resident in HBM (seeded per rank: independent canvases)
    g = torch.Generator(device=dev).manual_seed(1000 + rank)
    bf = torch.bfloat16
    B, L, Hq, Hkv, D, P, d, V = cfg.B, cfg.L, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.d, cfg.V
    M = B * L
    # the per-step inputs (canvas hidden states, canvas queries, canvas keys
    # and values) live in one device block, so the end-to-end run moves them
    # from one pinned host block with a single copy
    shapes = {"x": (M, d), "q": (B, L, Hq, D), "kc": (B, L, Hkv, D), "vc": (B, L, Hkv, D)}
    offs, tot = {}, 0
    for k, shp in shapes.items():
        offs[k] = tot
        tot += (math.prod(shp) * 2 + 255) // 256 * 256
    step_in = torch.empty(tot, dtype=torch.uint8, device=dev)

    def view(k):
        n = math.prod(shapes[k]) * 2
        return step_in[offs[k]:offs[k] + n].view(bf).view(shapes[k])

    q, kc, vc, x = view("q"), view("kc"), view("vc"), view("x")
    q.copy_(torch.randn(B, L, Hq, D, device=dev, generator=g))
    kp = torch.randn(B, P, Hkv, D, device=dev, generator=g).to(bf)
    vp = torch.randn(B, P, Hkv, D, device=dev, generator=g).to(bf)
    kc.copy_(torch.randn(B, L, Hkv, D, device=dev, generator=g))
    vc.copy_(torch.randn(B, L, Hkv, D, device=dev, generator=g))
    attn_out = torch.empty_like(q)
    xf = torch.randn(M, d, device=dev, generator=g)
    if cfg.row_scale is not None:
        lo, hi = cfg.row_scale
        xf *= torch.rand(M, 1, device=dev, generator=g) * (hi - lo) + lo
    x.copy_(xf)
    del xf
    w = torch.empty(d, V, device=dev, dtype=bf)
    for r0 in range(0, d, 256):
        r1 = min(d, r0 + 256)
        w[r0:r1] = (torch.randn(r1 - r0, V, device=dev, generator=g) * cfg.w_std).to(bf)
    scale = 1.0 / math.sqrt(D)
    aws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), dev)
    bufs = dg.StepBuffers(B, L, dev)
    bufs.canvas.copy_(torch.randint(0, V, (M,), device=dev, generator=g, dtype=torch.int32))
    fp8 = args.lm_dtype == "fp8"
    sc = args.self_cond
    # load-time layout of the bf16 W (not timed): where the LM head runs on
    # the 2-SM kernels, W is packed (dg_pack_lm_weight: one 16 KB stretch per
    # 128 columns x 64 hidden dimensions); FP8 reads its own E4M3 copy
    packed = not fp8 and dg.lm_head_plan(M, d, V)["kind"] >= 2
    layout = dg.W_PACKED if packed else dg.W_ROWMAJOR
    p0 = dg.step_params(B, L, d, V, cfg.temperature, cfg.entropy_bound, cfg.stop_threshold, 0,
                        seed=rank, w_layout=layout)
    if sc:
        # the self-conditioning table E [V, 32] bf16 (30 meaningful columns,
        # V x 30 = 7.86M parameters at V = 262144) and the read-out [M, 32]
        sc_table = torch.randn(V, 32, device=dev, generator=g) / math.sqrt(d)
        sc_table[:, 30:] = 0
        sc_table = sc_table.to(bf)
        sc_out = torch.empty(M, 32, device=dev)
    if fp8:
        # load-time conversion of W to E4M3 codes [V, d] + column scales (not timed);
        # the hidden states are quantised inside every step
        w8 = torch.empty(V, d, dtype=torch.uint8, device=dev)
        w_scale = torch.empty(V, dtype=torch.float32, device=dev)
        dg.quantize_weight_e4m3(w, w8, w_scale)
        sws = dg.workspace(dg.denoise_step_fp8_workspace(p0), dev)
    elif sc:
        sws = dg.workspace(dg.denoise_step_sc_workspace(p0), dev)
    else:
        sws = dg.workspace(dg.denoise_step_workspace(p0), dev)
    if packed:
        w = dg.pack_lm_weight(w)
        torch.cuda.synchronize(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > 129 MB L2
    stream = torch.cuda.current_stream(dev)

    def lm_fold():
        if fp8:
            dg.lm_head_fold_fp8(x, w8, w_scale, p0, sws)
        elif sc:
            dg.lm_head_fold_sc(x, w, sc_table, p0, sws)
        else:
            dg.lm_head_fold(x, w, p0, sws)

    # The step is one library call (dg_canvas_step and its FP8 and
    # self-conditioning forms: the canvas attention on a stream forked from the
    # step's stream; for the bf16 step the LM head is planned on the SMs a
    # short attention leaves free).
    if fp8:
        cws = dg.workspace(dg.canvas_step_fp8_workspace(p0, P, Hq, Hkv, D), dev)
    elif sc:
        cws = dg.workspace(dg.canvas_step_sc_workspace(p0, P, Hq, Hkv, D), dev)
    else:
        cws = dg.workspace(dg.canvas_step_workspace(p0, P, Hq, Hkv, D), dev)

    def step(k):
        p = dg.step_params(B, L, d, V, cfg.temperature, cfg.entropy_bound, cfg.stop_threshold,
                           k, seed=rank, w_layout=layout)
        if fp8:
            dg.canvas_step_fp8(q, kp, vp, kc, vc, attn_out, scale, x, w8, w_scale, p, bufs, cws)
        elif sc:
            dg.canvas_step_sc(q, kp, vp, kc, vc, attn_out, scale, x, w, sc_table, p, bufs, sc_out,
                              cws)
        else:
            dg.canvas_step(q, kp, vp, kc, vc, attn_out, scale, x, w, p, bufs, cws)

    def timed(fn, n, first, label="step"):
        """Per-iteration CUDA-event times (ms) with an L2 flush before each
        iteration; each iteration is an NVTX range (for a timeline profiler)."""
        evs = []
        for i in range(n):
            flush.fill_(i & 0xFF)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.nvtx.range_push(label)
            s.record(stream)
            fn(first + i)
            e.record(stream)
            torch.cuda.nvtx.range_pop()
            evs.append((s, e))
        torch.cuda.synchronize(dev)
        return [s.elapsed_time(e) for s, e in evs]

    # ---- warmup, then the timed region (barrier + sync on both sides)
    with ClockSampler(local) as clk:
        clk.wait_first()
        timed(step, args.warmup, 0)
        if world > 1:
            tdist.barrier()
        torch.cuda.synchronize(dev)
        n0 = dg.kernel_launches()
        t_start = time.perf_counter()
        ts = timed(step, args.steps, args.warmup)
        t_end = time.perf_counter()
        launches = dg.kernel_launches() - n0
        clk.mark(t_start, t_end)
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize(dev)
    step_ms = sum(ts) / len(ts)
    status = dg.read_device_status(sws) | dg.read_device_status(aws) | (
        dg.read_device_status(cws) if cws is not None else 0)
    step_ms = _reduce_max(step_ms, dev)

    # ---- per-kernel timings (same flush discipline) for the roofline
    lm_ms = statistics.mean(timed(lambda k: lm_fold(), args.steps, 0, "lm_head"))
    at_ms = statistics.mean(timed(lambda k: dg.canvas_attn(q, kp, vp, kc, vc, attn_out, scale,
                                                           aws), args.steps, 0, "canvas_attn"))
    # FP8: W codes + column scales, and the bf16 hidden states read by the row quantisation;
    # self-conditioning: + the bf16 table E [V, 32]
    lm_bytes = (d * V + 4 * V if fp8 else d * V * 2) + M * d * 2 + (V * 32 * 2 if sc else 0)
    lm_gbs = lm_bytes / (lm_ms * 1e-3) / 1e9
    lm_flops = 2.0 * M * d * V
    # E4M3 runs at twice the bf16 rate (nominal dense ratio 4.5 / 2.25 PFLOP/s)
    lm_peak = bf16_peak * (2.0 if fp8 else 1.0)
    at_flops = 4.0 * B * Hq * L * (P + L) * D
    at_bytes = 2 * (B * L * Hq * D * 2) + 2 * (B * (P + L) * Hkv * D * 2)
    lm_plan = dg.lm_head_plan(M, d, V)
    if fp8:
        lm_plan = dict(lm_plan, kernel="lm_head_duo_fp8_kernel")
    if sc:
        lm_plan = dict(lm_plan, kernel="lm_head_duo_sc_kernel")
    srcs = [os.path.join(ROOT, "block_diffusion_decoding_gb300", "csrc", f)
            for f in ("dg_lm_head.cu", "dg_lm_head_duo.cu", "dg_plan.h",
                      "dg_sampler.cuh", "dg_device.cuh", "dg_kernels.h")]
    traffic = _traffic_record(srcs, lm_plan["kernel"], (M, d, V))

    # ---- end to end through the C ABI with host buffers (pinned): per step,
    # one H2D copy of the step's inputs (hidden states, canvas Q/K/V) and one
    # D2H copy of the result (canvas, argmax, stop)
    h_in = step_in.cpu().pin_memory()
    h_out = torch.empty_like(bufs.readback, device="cpu").pin_memory()
    h2d = step_in.numel()
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step(k):
        step_in.copy_(h_in, non_blocking=True)
        step(k)
        h_out.copy_(bufs.readback, non_blocking=True)
        torch.cuda.synchronize(dev)
        return int(h_out[-1])

    for i in range(2):
        e2e_step(i)
    e2e_times = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_step(args.warmup + i)
        e2e_times.append(time.perf_counter() - t0)
    e2e_ms = 1e3 * sum(e2e_times) / len(e2e_times)
    e2e_ms = _reduce_max(e2e_ms, dev)

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = {"x": x.view(torch.int16).cpu().numpy().view(np.uint16),
                "w": _w_columns(w, packed, d, ORACLE_V_SAMPLE).view(torch.int16).cpu().numpy()
                     .view(np.uint16),
                "q": q.view(torch.int16).cpu().numpy().view(np.uint16),
                "kp": kp.view(torch.int16).cpu().numpy().view(np.uint16),
                "vp": vp.view(torch.int16).cpu().numpy().view(np.uint16),
                "kc": kc.view(torch.int16).cpu().numpy().view(np.uint16),
                "vc": vc.view(torch.int16).cpu().numpy().view(np.uint16)}
        sc_host = sc_table[:ORACLE_V_SAMPLE].float().cpu().numpy() if sc else None
        est = [oracle_step_estimate(cfg, host, v_sample=ORACLE_V_SAMPLE,
                                    attn_rows=ORACLE_ATTN_ROWS, fp8=fp8,
                                    sc_table=sc_host)[0] for _ in range(2)]
        _, desc, _ = oracle_step_estimate(cfg, host, v_sample=ORACLE_V_SAMPLE,
                                          attn_rows=ORACLE_ATTN_ROWS, fp8=fp8,
                                          sc_table=sc_host)
        cpu = dict(value=1.0 / statistics.median(est), unit="steps/s", cores=1, kind="oracle", **_host_cpu(),
                   sample=desc)
    if world > 1:
        tdist.destroy_process_group()
    if rank != 0:
        return 0
    value = _replica_value(world, step_ms)
    # each kernel's roofline: the slower of its algorithmic bytes at the
    # measured copy bandwidth and its FLOPs at the measured bf16 peak
    lm_roof_ms = max(lm_bytes / (hbm_peak * 1e9), lm_flops / (lm_peak * 1e12)) * 1e3
    at_roof_ms = max(at_bytes / (hbm_peak * 1e9), at_flops / (bf16_peak * 1e12)) * 1e3
    lm_tensor = lm_flops / (lm_peak * 1e12) > lm_bytes / (hbm_peak * 1e9)
    lm_tflops = lm_flops / (lm_ms * 1e-3) / 1e12
    if lm_tensor:
        roof = dict(bound="tensor", achieved=lm_tflops, peak=lm_peak, unit="TFLOP/s",
                    frac=lm_tflops / lm_peak, traffic=traffic, kernel=lm_plan["kernel"],
                    peak_source=peak_kind + (" (MEASURED_PEAKS.json bf16_tflops, burst, x2 for "
                                             "E4M3 by the nominal dense ratio)" if fp8 else
                                             " (MEASURED_PEAKS.json bf16_tflops, burst)"),
                    algorithmic_flops=lm_flops,
                    frac_of_nominal=lm_tflops / (NOMINAL_BF16_TFLOPS * (2.0 if fp8 else 1.0)))
    else:
        roof = dict(bound="hbm", achieved=lm_gbs, peak=hbm_peak, unit="GB/s",
                    frac=lm_gbs / hbm_peak, traffic=traffic, kernel=lm_plan["kernel"],
                    peak_source=peak_kind + " (MEASURED_PEAKS.json hbm_gbs)",
                    algorithmic_bytes=lm_bytes, frac_of_nominal=lm_gbs / NOMINAL_HBM_GBS)
    line = dict(
        metric="denoise steps/s (256-tok canvas, bs=1)", value=value, unit="steps/s",
        n_gpus=world, steps=args.steps, warmup=args.warmup, ms_per_step=step_ms,
        higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="e4m3 LM head (fp32 accumulate), bf16 attention" if fp8 else "bf16",
        data="synthetic", config=_config_json(cfg, l2="flushed (256 MiB write) before every step",
                                              lm_dtype=args.lm_dtype, self_cond=sc,
                                              w_layout=None if fp8 else layout),
        canvas_tokens_per_s=value * M,
        roofline=roof,
        kernels={lm_plan["kernel"]: {"ms": lm_ms, "GB_per_s": lm_gbs, "TFLOP_per_s": lm_tflops,
                                     "roofline_ms": lm_roof_ms, "frac_of_roofline": lm_roof_ms / lm_ms,
                                     "BN": lm_plan["BN"], "ctas": lm_plan["ctas"]},
                 "canvas_attn": {"ms": at_ms, "TFLOP_per_s": at_flops / (at_ms * 1e-3) / 1e12,
                                 "GB_per_s": at_bytes / (at_ms * 1e-3) / 1e9,
                                 "roofline_ms": at_roof_ms, "frac_of_roofline": at_roof_ms / at_ms}},
        step_roofline_ms=lm_roof_ms + at_roof_ms,
        step_frac_of_roofline=(lm_roof_ms + at_roof_ms) / step_ms,
        cpu_baseline=cpu,
        e2e=dict(value=_replica_value(world, e2e_ms), unit="steps/s", h2d_bytes_per_step=h2d,
                 d2h_bytes_per_step=d2h),
        clocks=clk.summary(), gpu_launches=launches, device_status=status)
    if not emit:
        return line
    print(json.dumps(line), flush=True)
    return 0

# ----------------------------------------------------------------------------- block loop
def run_block(args, cfg, emit=True):
    """The block loop (dg_generate_block, one CUDA graph per block) on the
    converging workload: hidden(k) = g_k(c) W[:,t]/|W[:,t]| + N(0, 1/d) for
    per-position targets t ~ U(V) and confidences c ~ U(0, 1); a block runs
    until every canvas stops (argmax unchanged and mean entropy < 0.005) or
    48 steps.  K timed blocks, L2 flushed before each; value = denoise steps
    per second inside the loop (steps taken / block time)."""
    import torch
    import block_diffusion_decoding_gb300 as dg
    from block_diffusion_decoding_gb300 import build as dgbuild

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
    dgbuild.build()
    dg.lib()
    hbm_peak, bf16_peak, peak_kind = _peaks()
    g = torch.Generator(device=dev).manual_seed(2000 + rank)
    bf = torch.bfloat16
    B, L, d, V, N = cfg.B, cfg.L, cfg.d, cfg.V, cfg.max_steps
    M = B * L
    w = torch.empty(d, V, device=dev, dtype=bf)
    for r0 in range(0, d, 256):
        r1 = min(d, r0 + 256)
        w[r0:r1] = (torch.randn(r1 - r0, V, device=dev, generator=g) * cfg.w_std).to(bf)
    t = torch.randint(0, V, (M,), device=dev, generator=g)
    c = torch.rand(M, device=dev, generator=g, dtype=torch.float64)
    cols = w[:, t].double().T
    cols /= cols.norm(dim=1, keepdim=True)
    hid = torch.empty(N, M, d, device=dev, dtype=bf)
    for k in range(N):
        gk = (2.0 + 6.0 * c) * (1.0 + k / 4.0)
        noise = torch.randn(M, d, device=dev, generator=g, dtype=torch.float64) / math.sqrt(d)
        hid[k] = (gk[:, None] * cols + noise).to(bf)
    del cols
    # W packed for the 2-SM LM-head kernels (load time, not timed); the
    # row-major copy stays for the oracle sample
    packed = dg.lm_head_plan(M, d, V)["kind"] >= 2
    layout = dg.W_PACKED if packed else dg.W_ROWMAJOR
    wl = dg.pack_lm_weight(w) if packed else w
    p = dg.step_params(B, L, d, V, cfg.t_start, cfg.entropy_bound, cfg.stop_threshold, 0,
                       seed=rank, w_layout=layout)
    bp = dg.block_params(N, cfg.t_start, cfg.t_end, M * d)
    bufs = dg.BlockBuffers(B, L, N, dev)
    bws = dg.workspace(dg.generate_block_workspace(p, bp), dev)
    sws = dg.workspace(dg.denoise_step_workspace(p), dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn, n):
        evs = []
        for i in range(n):
            flush.fill_(i & 0xFF)
            s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_.record(stream)
            fn()
            e_.record(stream)
            evs.append((s_, e_))
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b_) for a, b_ in evs]

    def block():
        dg.generate_block(hid, wl, p, bp, bufs, bws)

    with ClockSampler(local) as clk:
        clk.wait_first()
        timed(block, args.warmup)
        if world > 1:
            tdist.barrier()
        torch.cuda.synchronize(dev)
        t_start = time.perf_counter()
        ts = timed(block, args.steps)
        t_end = time.perf_counter()
        clk.mark(t_start, t_end)
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize(dev)
    status = dg.read_device_status(bws)
    steps = int(bufs.steps_taken.max().item())
    hist = bufs.n_accepted_hist.view(N, B)[:steps].float()
    block_ms = sum(ts) / len(ts)
    block_ms = _reduce_max(block_ms, dev)
    step_ms = block_ms / steps

    # flat logits (hidden = 0): exactly one commit per step, 48 steps
    flat = torch.zeros(M, d, device=dev, dtype=bf)
    fbp = dg.block_params(N, cfg.t_start, cfg.t_end, 0)
    fbufs = dg.BlockBuffers(B, L, N, dev)
    dg.generate_block(flat, wl, p, fbp, fbufs, bws)
    torch.cuda.synchronize(dev)
    flat_ok = (int(fbufs.steps_taken.min().item()) == N and
               bool((fbufs.n_accepted_hist == 1).all().item()))

    # the LM-head kernel alone on the first step's hidden states (roofline)
    lm_ms = statistics.mean(timed(lambda: dg.lm_head_fold(hid[0], wl, p, sws), args.steps))
    lm_bytes = d * V * 2 + M * d * 2
    lm_gbs = lm_bytes / (lm_ms * 1e-3) / 1e9
    lm_plan = dg.lm_head_plan(M, d, V)
    srcs = [os.path.join(ROOT, "block_diffusion_decoding_gb300", "csrc", f)
            for f in ("dg_lm_head.cu", "dg_lm_head_duo.cu", "dg_plan.h",
                      "dg_sampler.cuh", "dg_device.cuh", "dg_kernels.h")]
    traffic = _traffic_record(srcs, lm_plan["kernel"], (M, d, V))

    # end to end: the block's hidden states go up from pinned host memory,
    # the result (canvas, argmax, steps taken) comes back
    h_hid = hid.cpu().pin_memory()
    h_out = [torch.empty_like(tns, device="cpu").pin_memory()
             for tns in (bufs.canvas, bufs.argmax, bufs.steps_taken)]
    e2e_times = []
    for i in range(args.steps + 1):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        hid.copy_(h_hid, non_blocking=True)
        block()
        for h, dsrc in zip(h_out, (bufs.canvas, bufs.argmax, bufs.steps_taken)):
            h.copy_(dsrc, non_blocking=True)
        torch.cuda.synchronize(dev)
        if i > 0:
            e2e_times.append(time.perf_counter() - t0)
    e2e_ms = 1e3 * sum(e2e_times) / len(e2e_times)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = {"x": hid[0].view(torch.int16).cpu().numpy().view(np.uint16),
                "w": w[:, :16384].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)}
        est = [oracle_block_step_estimate(cfg, host)[0] for _ in range(2)]
        _, desc = oracle_block_step_estimate(cfg, host)
        cpu = dict(value=1.0 / statistics.median(est), unit="steps/s", cores=1, kind="oracle", **_host_cpu(),
                   sample=desc)
    if world > 1:
        tdist.destroy_process_group()
    if rank != 0:
        return 0
    value = _replica_value(world, step_ms)
    line = dict(
        metric="denoise steps/s (256-tok canvas, bs=1)", value=value, unit="steps/s",
        n_gpus=world, steps=args.steps, warmup=args.warmup, ms_per_step=step_ms,
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
        data="synthetic",
        config={"workload": "%s: block loop (CUDA graph, conditional while), B=%d L=%d, LM head "
                            "d=%d V=%d, T %.1f->%.1f over %d steps, b=%.1f, stop mean H < %.3f; "
                            "timed unit = one block" % (cfg.name, B, L, d, V, cfg.t_start,
                                                        cfg.t_end, N, cfg.entropy_bound,
                                                        cfg.stop_threshold),
                "global_batch": B, "seq_len": L, "parallelism": "replicas",
                "l2": "flushed (256 MiB write) before every block", "w_layout": W_LAYOUTS[layout]},
        block_ms=block_ms, steps_to_stop=steps,
        commits_per_step=float(hist.mean().item()),
        canvas_tokens_per_s=world * M / (block_ms * 1e-3),
        flat_case_one_commit_per_step_48_steps=flat_ok,
        roofline=dict(bound="hbm", achieved=lm_gbs, peak=hbm_peak, unit="GB/s",
                      frac=lm_gbs / hbm_peak, traffic=traffic, kernel=lm_plan["kernel"],
                      peak_source=peak_kind + " (MEASURED_PEAKS.json hbm_gbs)",
                      algorithmic_bytes=lm_bytes, frac_of_nominal=lm_gbs / NOMINAL_HBM_GBS),
        step_roofline_ms=lm_bytes / (hbm_peak * 1e9) * 1e3,
        step_frac_of_roofline=lm_bytes / (hbm_peak * 1e9) * 1e3 / step_ms,
        cpu_baseline=cpu,
        e2e=dict(value=world * steps * 1e3 / e2e_ms, unit="steps/s",
                 h2d_bytes_per_step=hid.numel() * 2 // steps,
                 d2h_bytes_per_step=sum(h.numel() * h.element_size() for h in h_out) // steps),
        clocks=clk.summary(),
        gpu_launches=args.steps * (1 + 2 * steps), gpu_launches_note="graph replays: loop init "
        "+ 2 kernels per step (LM head, combine/accept) per block",
        device_status=status)
    if not emit:
        return line
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- encoder append
def run_encoder(args, cfg, emit=True):
    """The encoder cache append (dg_encoder_append): the committed block's K/V
    appended to a cache holding P tokens and the block's causal attention over
    [cache ; block].  Timed per call with the L2 flushed before each; the cache
    is reset to P tokens before every call (outside the timed region)."""
    import torch
    import block_diffusion_decoding_gb300 as dg
    from block_diffusion_decoding_gb300 import build as dgbuild

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
    dgbuild.build()
    dg.lib()
    hbm_peak, bf16_peak, peak_kind = _peaks()
    g = torch.Generator(device=dev).manual_seed(3000 + rank)
    bf = torch.bfloat16
    B, L, Hq, Hkv, D, P = cfg.B, cfg.L, cfg.Hq, cfg.Hkv, cfg.D, cfg.P
    P_max = P + L
    q = torch.randn(B, L, Hq, D, device=dev, generator=g).to(bf)
    kcache = torch.randn(B, P_max, Hkv, D, device=dev, generator=g).to(bf)
    vcache = torch.randn(B, P_max, Hkv, D, device=dev, generator=g).to(bf)
    knew = torch.randn(B, L, Hkv, D, device=dev, generator=g).to(bf)
    vnew = torch.randn(B, L, Hkv, D, device=dev, generator=g).to(bf)
    out = torch.empty_like(q)
    ws = dg.workspace(dg.encoder_append_workspace(B, L, P, Hq, Hkv, D), dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale = 1.0 / math.sqrt(D)
    ts = []
    with ClockSampler(local) as clk:
        clk.wait_first()
        t_start = None
        for i in range(args.warmup + args.steps):
            if i == args.warmup:
                if world > 1:
                    tdist.barrier()
                torch.cuda.synchronize(dev)
                t_start = time.perf_counter()
            flush.fill_(i & 0xFF)
            s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_.record(stream)
            dg.encoder_append(q, kcache, vcache, P, knew, vnew, out, scale, ws)
            e_.record(stream)
            if i >= args.warmup:
                ts.append((s_, e_))
        torch.cuda.synchronize(dev)
        clk.mark(t_start, time.perf_counter())
    ms = sum(a.elapsed_time(b_) for a, b_ in ts) / len(ts)
    ms = _reduce_max(ms, dev)
    if world > 1:
        tdist.destroy_process_group()
    status = dg.read_device_status(ws)
    if rank != 0:
        return 0
    # causal: the block's position i sees P + i + 1 keys
    flops = 4.0 * B * Hq * D * (L * P + L * (L + 1) / 2)
    nbytes = 2 * (2 * B * L * Hq * D) + 2 * (2 * B * (P + L) * Hkv * D) + 2 * (2 * B * L * Hkv * D)
    roof_ms = max(flops / (bf16_peak * 1e12), nbytes / (hbm_peak * 1e9)) * 1e3
    tflops = flops / (ms * 1e-3) / 1e12
    line = dict(
        metric="encoder cache appends/s (256-token block)", value=_replica_value(world, ms),
        unit="appends/s", n_gpus=world, steps=args.steps, warmup=args.warmup, ms_per_step=ms,
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16", data="synthetic",
        config={"workload": "%s: encoder cache append, B=%d block L=%d, cache P=%d, Hq=%d Hkv=%d "
                            "D=%d, causal over [cache ; block]" % (cfg.name, B, L, P, Hq, Hkv, D),
                "global_batch": B, "seq_len": L, "parallelism": "replicas",
                "l2": "flushed (256 MiB write) before every call"},
        roofline=dict(bound="tensor", achieved=tflops, peak=bf16_peak, unit="TFLOP/s",
                      frac=tflops / bf16_peak, traffic=None, kernel="attention (causal)",
                      peak_source=peak_kind + " (MEASURED_PEAKS.json bf16_tflops, burst)",
                      algorithmic_flops=flops, frac_of_nominal=tflops / NOMINAL_BF16_TFLOPS),
        step_roofline_ms=roof_ms, step_frac_of_roofline=roof_ms / ms,
        clocks=clk.summary(), device_status=status)
    if not emit:
        return line
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- MoE FFN
def run_moe(args, mcfg, emit=True):
    """One MoE FFN layer over the canvas (dg_moe_ffn): router, top-8 of 128
    experts plus the shared one, gated GELU experts, weighted sum.  K timed
    layers, L2 flushed before each; value = layers per second.  Roofline:
    the weights of the experts the canvas touches (+ the shared expert and the
    router) at the measured HBM bandwidth, against the layer's FLOPs at the
    measured bf16 peak."""
    import torch
    import block_diffusion_decoding_gb300 as dg
    from block_diffusion_decoding_gb300 import build as dgbuild

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
    dgbuild.build()
    dg.lib()
    hbm_peak, bf16_peak, peak_kind = _peaks()
    g = torch.Generator(device=dev).manual_seed(4000 + rank)
    bf = torch.bfloat16
    M, d, f, E, K = mcfg.M, mcfg.d, mcfg.f, mcfg.E, mcfg.top_k
    c = torch.randn(d, device=dev, generator=g)
    x = ((mcfg.alpha * c[None, :] + torch.randn(M, d, device=dev, generator=g))
         / math.sqrt(1 + mcfg.alpha ** 2)).to(bf)
    wr = (torch.randn(E, d, device=dev, generator=g) / math.sqrt(d)).to(bf)
    wg = torch.empty(E + 1, f, d, device=dev, dtype=bf)
    wu = torch.empty_like(wg)
    wd = torch.empty(E + 1, d, f, device=dev, dtype=bf)
    for e in range(E + 1):
        wg[e] = (torch.randn(f, d, device=dev, generator=g) / math.sqrt(d)).to(bf)
        wu[e] = (torch.randn(f, d, device=dev, generator=g) / math.sqrt(d)).to(bf)
        wd[e] = (torch.randn(d, f, device=dev, generator=g) / math.sqrt(f)).to(bf)
    out = torch.empty(M, d, device=dev)
    experts = torch.empty(M, K, dtype=torch.int32, device=dev)
    gates = torch.empty(M, K, device=dev)
    p = dg.moe_params(M, d, f, E, K)
    ws = dg.workspace(dg.moe_ffn_workspace(p), dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def layer():
        dg.moe_ffn(x, wr, wg, wu, wd, out, p, ws, experts, gates)

    def timed(n):
        evs = []
        for i in range(n):
            flush.fill_(i & 0xFF)
            s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_.record(stream)
            layer()
            e_.record(stream)
            evs.append((s_, e_))
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b_) for a, b_ in evs]

    with ClockSampler(local) as clk:
        clk.wait_first()
        timed(args.warmup)
        if world > 1:
            tdist.barrier()
        torch.cuda.synchronize(dev)
        n0 = dg.kernel_launches()
        t_start = time.perf_counter()
        ts = timed(args.steps)
        t_end = time.perf_counter()
        launches = dg.kernel_launches() - n0
        clk.mark(t_start, t_end)
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize(dev)
    ms = _reduce_max(sum(ts) / len(ts), dev)
    status = dg.read_device_status(ws)
    distinct = int(torch.unique(experts).numel())
    # algorithmic traffic: the touched experts' and the shared expert's three
    # matrices, the router, the hidden rows in and the fp32 output rows out
    w_bytes = (distinct + 1) * 3 * f * d * 2 + E * d * 2
    nbytes = w_bytes + M * d * 2 + M * d * 4
    flops = 2.0 * M * d * E + (M * K + M) * 3 * 2.0 * d * f
    gbs = nbytes / (ms * 1e-3) / 1e9
    roof_ms = max(nbytes / (hbm_peak * 1e9), flops / (bf16_peak * 1e12)) * 1e3

    # end to end: the hidden rows up from pinned host memory, the output down
    h_x = x.cpu().pin_memory()
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    e2e = []
    for i in range(args.steps + 1):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        x.copy_(h_x, non_blocking=True)
        layer()
        h_out.copy_(out, non_blocking=True)
        torch.cuda.synchronize(dev)
        if i > 0:
            e2e.append(time.perf_counter() - t0)
    e2e_ms = _reduce_max(1e3 * sum(e2e) / len(e2e), dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        host = {k: v.view(torch.int16).cpu().numpy().view(np.uint16)
                for k, v in dict(x=x, wr=wr, wg=wg, wu=wu, wd=wd).items()}
        t0 = time.perf_counter()
        oracle.moe_ffn(host["x"], host["wr"], host["wg"], host["wu"], host["wd"], K)
        t_or = time.perf_counter() - t0
        cpu = dict(value=1.0 / t_or, unit="layers/s", cores=1, kind="oracle", **_host_cpu(),
                   sample="oracle (numpy fp64 matmuls + plain routing, 1 thread): the whole "
                          "layer, all %d rows" % M)
    if world > 1:
        tdist.destroy_process_group()
    if rank != 0:
        return 0
    line = dict(
        metric="MoE FFN layers/s (256-token canvas)", value=_replica_value(world, ms),
        unit="layers/s", n_gpus=world, steps=args.steps, warmup=args.warmup, ms_per_step=ms,
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16", data="synthetic",
        config={"workload": "%s: MoE FFN over the canvas, M=%d rows, d=%d, %d experts of f=%d, "
                            "top-%d + 1 shared, gated GELU; hidden rows share a canvas-wide "
                            "component (alpha %.1f)" % (mcfg.name, M, d, E, f, K, mcfg.alpha),
                "global_batch": 1, "seq_len": M, "parallelism": "replicas",
                "l2": "flushed (256 MiB write) before every layer"},
        distinct_experts=distinct,
        roofline=dict(bound="hbm" if nbytes / hbm_peak > flops / (bf16_peak * 1e3) else "tensor",
                      achieved=gbs, peak=hbm_peak, unit="GB/s", frac=gbs / hbm_peak,
                      traffic=None, kernel="moe_ffn_kernel (+ router, route, gather, combine)",
                      peak_source=peak_kind + " (MEASURED_PEAKS.json hbm_gbs)",
                      algorithmic_bytes=nbytes, frac_of_nominal=gbs / NOMINAL_HBM_GBS),
        step_roofline_ms=roof_ms, step_frac_of_roofline=roof_ms / ms,
        TFLOP_per_s=flops / (ms * 1e-3) / 1e12,
        cpu_baseline=cpu,
        e2e=dict(value=_replica_value(world, e2e_ms), unit="layers/s",
                 h2d_bytes_per_step=M * d * 2, d2h_bytes_per_step=M * d * 4),
        clocks=clk.summary(), gpu_launches=launches, device_status=status)
    if not emit:
        return line
    print(json.dumps(line), flush=True)
    return 0


def oracle_block_step_estimate(cfg, host, v_sample=16384):
    """One step of the block loop on the CPU oracle, column-sampled: every canvas
    row against the first v_sample vocabulary columns (LM head + sampler, time
    scaled by V / v_sample), then the acceptance and stop test."""
    import oracle
    vs = min(v_sample, cfg.V)
    t0 = time.perf_counter()
    lg = oracle.logits(host["x"], np.ascontiguousarray(host["w"][:, :vs]))
    s = oracle.sampler(lg, cfg.t_start, 0, np.arange(cfg.M), 0)
    t_lm = time.perf_counter() - t0
    t0 = time.perf_counter()
    Hf = s["H"].astype(np.float32)
    oracle.accept_renoise(Hf, s["sample"], np.zeros(cfg.M, np.int32), cfg.V, cfg.entropy_bound,
                          0, 0, 0)
    oracle.stop(s["argmax"], s["argmax"], Hf, 0)
    t_acc = time.perf_counter() - t0
    desc = ("oracle (fp64 C + numpy fp64 matmul, 1 thread): one loop step, all %d canvas rows x "
            "%d of %d vocab columns (scaled x%.0f), acceptance + stop" % (cfg.M, vs, cfg.V,
                                                                         cfg.V / vs))
    return t_lm * cfg.V / vs + t_acc, desc


def run_kernel_only(args, cfg):
    """One kernel of the step alone on the workload's shapes (for profilers:
    only that kernel's inputs are allocated).  Prints per-launch CUDA-event
    times; not the benchmark line."""
    import torch
    import block_diffusion_decoding_gb300 as dg
    from block_diffusion_decoding_gb300 import build as dgbuild
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dgbuild.build()
    g = torch.Generator(device=dev).manual_seed(1000)
    bf = torch.bfloat16
    B, L, Hq, Hkv, D, P, d, V = cfg.B, cfg.L, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.d, cfg.V
    M = B * L
    if args.kernel == "attention":
        q = torch.randn(B, L, Hq, D, device=dev, generator=g).to(bf)
        kp = torch.randn(B, P, Hkv, D, device=dev, generator=g).to(bf)
        vp = torch.randn(B, P, Hkv, D, device=dev, generator=g).to(bf)
        kc = torch.randn(B, L, Hkv, D, device=dev, generator=g).to(bf)
        vc = torch.randn(B, L, Hkv, D, device=dev, generator=g).to(bf)
        out = torch.empty_like(q)
        ws = dg.workspace(dg.canvas_attn_workspace(B, L, P, Hq, Hkv, D), dev)
        fn = lambda: dg.canvas_attn(q, kp, vp, kc, vc, out, 1.0 / math.sqrt(D), ws)
    else:
        xf = torch.randn(M, d, device=dev, generator=g)
        if cfg.row_scale is not None:
            lo, hi = cfg.row_scale
            xf *= torch.rand(M, 1, device=dev, generator=g) * (hi - lo) + lo
        x = xf.to(bf)
        del xf
        w = torch.empty(d, V, device=dev, dtype=bf)
        for r0 in range(0, d, 256):
            r1 = min(d, r0 + 256)
            w[r0:r1] = (torch.randn(r1 - r0, V, device=dev, generator=g) * cfg.w_std).to(bf)
        # W as the benchmark holds it: packed where the 2-SM kernels run
        layout = (dg.W_PACKED if args.lm_dtype != "fp8" and dg.lm_head_plan(M, d, V)["kind"] >= 2
                  else dg.W_ROWMAJOR)
        p = dg.step_params(B, L, d, V, cfg.temperature, cfg.entropy_bound, cfg.stop_threshold, 1,
                           w_layout=layout)
        if layout == dg.W_PACKED:
            w = dg.pack_lm_weight(w)
        if args.self_cond:
            sc_table = (torch.randn(V, 32, device=dev, generator=g) / math.sqrt(d)).to(bf)
            ws = dg.workspace(dg.denoise_step_sc_workspace(p), dev)
            fn = lambda: dg.lm_head_fold_sc(x, w, sc_table, p, ws)
        elif args.lm_dtype == "fp8":
            w8 = torch.empty(V, d, dtype=torch.uint8, device=dev)
            w_scale = torch.empty(V, dtype=torch.float32, device=dev)
            dg.quantize_weight_e4m3(w, w8, w_scale)
            del w
            ws = dg.workspace(dg.denoise_step_fp8_workspace(p), dev)
            fn = lambda: dg.lm_head_fold_fp8(x, w8, w_scale, p, ws)
        else:
            ws = dg.workspace(dg.denoise_step_workspace(p), dev)
            fn = lambda: dg.lm_head_fold(x, w, p, ws)
    ts = []
    for i in range(args.warmup + args.steps):
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record()
        fn()
        e_.record()
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            ts.append(s_.elapsed_time(e_))
    print(json.dumps({"kernel_only": args.kernel, "config": cfg.name,
                      "us_mean": 1e3 * sum(ts) / len(ts), "launches": args.steps,
                      "device_status": dg.read_device_status(ws)}), flush=True)
    return 0


# ----------------------------------------------------------------------------- workload sweep
SWEEP = [
    # (name in the line, config, options): every configuration of the step, the
    # block loop, the encoder append and the widened rows, each in its own
    # timed region of about half a second or more (with the L2 flush before
    # every step), so the clock sampler sees the GPU under load
    ("step_small", "step_small", {"steps": 4000}),
    ("batch1", "batch1", {"steps": 4000}),
    ("batch4", "batch4", {"steps": 3000}),
    ("batch16", "batch16", {"steps": 2000}),
    ("long_context", "long_context", {"steps": 4000}),
    ("block_full", "block_full", {"steps": 100}),
    ("step_full_fp8", "step_full", {"lm_dtype": "fp8", "steps": 2000}),
    ("step_full_self_cond", "step_full", {"self_cond": True, "steps": 1500}),
    ("encoder_full", "encoder_full", {"steps": 4000}),
    ("moe_full", "moe_full", {"steps": 2000}),
]


def _compact(line):
    """The numbers of a sub-run kept in the headline's workloads object."""
    keep = ("metric", "value", "unit", "ms_per_step", "steps", "canvas_tokens_per_s",
            "step_roofline_ms", "step_frac_of_roofline", "steps_to_stop", "commits_per_step",
            "flat_case_one_commit_per_step_48_steps", "distinct_experts", "block_ms",
            "TFLOP_per_s", "device_status", "gpu_launches")
    out = {k: line[k] for k in keep if k in line}
    out["workload"] = line["config"]["workload"]
    if line.get("roofline"):
        r = line["roofline"]
        out["roofline"] = {k: r.get(k) for k in ("bound", "achieved", "peak", "unit", "frac",
                                                  "kernel")}
    if line.get("kernels"):
        out["kernels"] = {k: {kk: v.get(kk) for kk in ("ms", "frac_of_roofline", "roofline_ms")}
                          for k, v in line["kernels"].items()}
    if line.get("e2e"):
        out["e2e"] = line["e2e"]["value"]
    if line.get("clocks"):
        out["clocks"] = line["clocks"]
    return out


def run_sweep(args):
    """Every other workload, measured in the same process after the headline."""
    import copy
    res = {}
    for name, cname, opt in SWEEP:
        a = copy.copy(args)
        a.steps = max(args.steps, opt.get("steps", 200))
        a.warmup = max(5, args.warmup)
        a.no_cpu_baseline = True
        a.lm_dtype = opt.get("lm_dtype", "bf16")
        a.self_cond = opt.get("self_cond", False)
        try:
            if cname in dg_synth.MOE_CONFIGS:
                line = run_moe(a, dg_synth.MOE_CONFIGS[cname], emit=False)
            else:
                cfg = dg_synth.CONFIGS[cname]
                if cfg.name == "block_full":
                    line = run_block(a, cfg, emit=False)
                elif cfg.name.startswith("encoder"):
                    line = run_encoder(a, cfg, emit=False)
                else:
                    line = run_ours(a, cfg, emit=False)
            res[name] = _compact(line)
        except Exception as e:      # a workload that fails is reported, not hidden
            res[name] = {"error": "%s: %s" % (type(e).__name__, e)}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG,
                    choices=sorted(dg_synth.CONFIGS) + sorted(dg_synth.MOE_CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lm-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="LM-head operands: bf16, or E4M3 codes with per-row / per-column scales")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the sweep of the other workloads after the headline step")
    ap.add_argument("--self-cond", action="store_true",
                    help="the step with the self-conditioning read-out folded into the LM head")
    ap.add_argument("--kernel", choices=["attention", "lm_head"],
                    help="run one kernel of the step alone (for profilers), not the benchmark")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.config in dg_synth.MOE_CONFIGS:
        if args.impl == "reference":
            return run_reference_moe(args, dg_synth.MOE_CONFIGS[args.config])
        return run_moe(args, dg_synth.MOE_CONFIGS[args.config])
    cfg = dg_synth.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.kernel:
        return run_kernel_only(args, cfg)
    if cfg.name == "block_full":
        return run_block(args, cfg)
    if cfg.name.startswith("encoder"):
        return run_encoder(args, cfg)
    world = _dist()[0]
    sweep = (cfg.name == DEFAULT_CONFIG and world == 1 and not args.no_workloads
             and args.lm_dtype == "bf16" and not args.self_cond)
    line = run_ours(args, cfg, emit=False)
    if line == 0:        # ranks other than 0
        return 0
    if sweep:
        line["workloads"] = run_sweep(args)
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
