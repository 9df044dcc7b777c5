"""bench.py host helpers (no GPU): the traffic lookup and the workload overrides."""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_traffic_row_is_per_kernel_and_workload():
    """A profiles/traffic.md row applies to its own kernel and workload only, and only
    while the kernel sources hash to the value it was captured on."""
    seven = bench.traffic_workload_key(synth.MLP_CONFIGS["llama7b"])
    qwen = bench.traffic_workload_key(synth.MLP_CONFIGS["qwen05b"])
    assert bench.ncu_traffic("gate_up", qwen) is None
    assert bench.ncu_traffic("rank_proj", seven) is None
    got = bench.ncu_traffic("gate_up", seven)
    if got is not None:
        # at least the algorithmic bytes: x, W_g, W_u read once, h, g, u written once
        c = synth.MLP_CONFIGS["llama7b"]
        assert got >= 2 * (c.M * c.h + 2 * c.i * c.h + 3 * c.M * c.i)


def test_rank_override_keeps_the_scale():
    args = types.SimpleNamespace(workload="gemma7b", act=None, rank=64)
    cfg = bench.mlp_config(args)
    base = synth.MLP_CONFIGS["gemma7b"]
    assert (cfg.r, cfg.h, cfg.i, cfg.M) == (64, base.h, base.i, base.M)
    assert cfg.s == pytest.approx(base.s)
    assert "r=64" in bench.workload_name(cfg)
    args = types.SimpleNamespace(workload="llama7b", act="geglu_erf", rank=0)
    cfg = bench.mlp_config(args)
    assert cfg.r == synth.MLP_CONFIGS["llama7b"].r and cfg.act == "geglu_erf"


def test_other_workloads_warm_up_by_work():
    """Each other workload warms up for at least 3 steps and about OTHER_WARMUP_TFLOP of
    work, so a small workload is timed at its own settled clocks."""
    for name in ("qwen05b", "llama7b", "gemma7b"):
        f = synth.MLP_CONFIGS[name].flops()
        n = bench.other_warmup_steps(f)
        assert n >= 3 and n * f >= bench.OTHER_WARMUP_TFLOP * 1e12 and (n - 1) * f < max(
            bench.OTHER_WARMUP_TFLOP * 1e12, 3 * f)
    assert bench.other_warmup_steps(synth.MLP_CONFIGS["qwen05b"].flops()) > 100
    assert bench.other_warmup_steps(1e15) == 3
