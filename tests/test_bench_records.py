"""bench.py's roofline traffic field comes from the committed ncu records in
profiles/: one per LM-head kernel at the full-width step.  A record counts
only for its own kernel and GEMM shape, and only while the kernel sources
hash to the value it was taken on."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRCS = [os.path.join(ROOT, "block_diffusion_decoding_gb300", "csrc", f)
        for f in ("dg_lm_head.cu", "dg_lm_head_duo.cu", "dg_plan.h",
                  "dg_sampler.cuh", "dg_device.cuh", "dg_kernels.h")]
FULL = (256, 2816, 262144)


def _fields(kernel):
    rec = {}
    with open(os.path.join(ROOT, "profiles", "%s_step_full.md" % kernel)) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                rec[k.strip()] = v.strip()
    return rec


def test_records_are_consistent():
    # within 1% above the algorithmic bytes: W + X (bf16), codes + scales (FP8)
    algo = {"lm_head_duo_kernel": 2816 * 262144 * 2 + 256 * 2816 * 2,
            "lm_head_duo_fp8_kernel": 2816 * 262144 + 4 * 262144 + 256 * 2816 + 4 * 256,
            "lm_head_duo_sc_kernel": 2816 * 262144 * 2 + 256 * 2816 * 2 + 262144 * 32 * 2}
    for kernel, a in algo.items():
        rec = _fields(kernel)
        assert rec["kernel"] == kernel and rec["shape"] == "256x2816x262144"
        total = float(rec["dram_bytes_per_launch"])
        assert total == float(rec["dram_read_bytes"]) + float(rec["dram_write_bytes"])
        assert 1.0 <= total / a < 1.01


def test_records_match_the_current_sources():
    """Skipped (not failed) after a kernel change, until the records are
    captured again on a GPU; bench.py then reports traffic as null."""
    got = {k: bench._traffic_record(SRCS, k, FULL)
           for k in ("lm_head_duo_kernel", "lm_head_duo_fp8_kernel", "lm_head_duo_sc_kernel")}
    if any(v is None for v in got.values()):
        pytest.skip("LM-head sources changed since the ncu records were taken")
    for k, v in got.items():
        assert v == float(_fields(k)["dram_bytes_per_launch"])


def test_records_do_not_carry_over():
    assert bench._traffic_record(SRCS, "lm_head_duo_kernel", (512, 2816, 262144)) is None
    assert bench._traffic_record(SRCS, "lm_head_duo_wide_kernel", FULL) is None
    # another set of sources (here: one file short) hashes differently
    assert bench._traffic_record(SRCS[:-1], "lm_head_duo_kernel", FULL) is None


def test_oracle_sample_columns_from_either_layout():
    """bench.py's oracle sample takes the first columns of W from W [d, V] or
    from its packed form [V/128][d][128] alike."""
    import torch
    d, V = 64, 1024
    w = torch.arange(d * V, dtype=torch.float32).view(d, V)
    wp = w.view(d, V // 128, 128).permute(1, 0, 2).contiguous().view(-1)
    assert torch.equal(bench._w_columns(wp, True, d, 512), w[:, :512])
    assert torch.equal(bench._w_columns(w, False, d, 512), w[:, :512])
