"""The seeded generator and the bf16 rounding (no GPU)."""

import json
import math
import os
import random

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_first_output():
    """splitmix64 (Steele, Lea and Flood 2014; Vigna's reference code) seeded with 0
    first returns 0xE220A8397B1DCDAF: the finaliser applied to the golden gamma."""
    assert synth.mix64(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_vector_draws_equal_scalar_definition():
    rnd = random.Random(3)
    for seed, sid in ((0, 0), (5, 17), (2**40 + 3, 9)):
        base = synth.stream_base(seed, sid)
        start = rnd.randrange(0, 1 << 30)
        got = synth.draws(base, start, 64).tolist()
        for j, v in enumerate(got):
            ref = synth.mix64(base + (start + j + 1) * 0x9E3779B97F4A7C15)
            assert (v & 0xFFFFFFFFFFFFFFFF) == ref


def _bf(x):
    return synth.bf16_to_f64(synth.f64_to_bf16(torch.tensor(x, dtype=torch.float64)))


def test_bf16_round_nearest_even_ties():
    one = 1.0
    assert _bf([one + 2.0 ** -8])[0] == 1.0                    # tie -> even (down)
    assert _bf([one + 3 * 2.0 ** -8])[0] == one + 2.0 ** -6    # tie -> even (up)
    assert _bf([-(one + 2.0 ** -8)])[0] == -1.0
    assert _bf([0.0])[0] == 0.0


def test_bf16_single_rounding_no_float32_detour():
    """Just above a bf16 midpoint by less than a float32 ulp: one rounding goes up,
    float64 -> float32 -> bf16 would land on the midpoint and go to even."""
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert _bf([x])[0] == 1.0 + 2.0 ** -7
    assert float(torch.tensor(x).float().to(torch.bfloat16)) == 1.0


def test_bf16_matches_torch_on_float32_values():
    x = torch.randn(200000, dtype=torch.float32, generator=torch.Generator().manual_seed(0))
    mine = synth.f64_to_bf16(x.double())
    assert torch.equal(mine.view(torch.int16), x.to(torch.bfloat16).view(torch.int16))


def test_distribution_moments():
    n = 1 << 20
    z = synth.normal_stream(0, 3, n)
    assert abs(float(z.mean())) < 5 / math.sqrt(n)
    assert abs(float(z.var()) - 1.0) < 5 * math.sqrt(2.0 / n)
    u = synth.uniform_stream(0, 4, n, 0.25)
    assert float(u.min()) >= -0.25 and float(u.max()) < 0.25
    assert abs(float(u.var()) - 0.25 ** 2 / 3) < 0.01 * 0.25 ** 2


def test_init_scales_follow_fan_in():
    cfg = synth.MLP_CONFIGS["tiny"]
    t = synth.make_mlp_inputs(cfg, seed=0)
    assert tuple(t["W_down"].shape) == (cfg.h, cfg.i)
    assert tuple(t["A_down"].shape) == (cfg.r, cfg.i)
    assert tuple(t["B_gate"].shape) == (cfg.i, cfg.r)
    w = synth.bf16_to_f64(t["W_gate"])
    assert abs(w.var() * cfg.h - 1.0) < 0.05
    a = synth.bf16_to_f64(t["A_down"])
    assert np.abs(a).max() <= (1.0 + 2.0 ** -8) / math.sqrt(cfg.i)   # bf16 rounding may round up
    b = synth.bf16_to_f64(t["B_gate"])
    assert abs(b.var() / 0.02 - 1.0) < 0.1


def test_streams_are_deterministic_and_independent():
    a = synth.normal_stream(0, 1, 1000)
    b = synth.normal_stream(0, 1, 1000)
    c = synth.normal_stream(0, 2, 1000)
    d = synth.normal_stream(1, 1, 1000)
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)
    # counter based: a later window equals the tail of a longer draw
    long = synth.normal_stream(0, 1, 1 << 25)
    assert torch.equal(long[:1000], a)


def test_golden_tiny_inputs():
    """The tiny workload's inputs, as written by tests/golden/make_golden.py."""
    with open(os.path.join(GOLDEN, "synth_tiny.json")) as f:
        gold = json.load(f)
    ins = synth.make_mlp_inputs(synth.MLP_CONFIGS[gold["config"]], seed=gold["seed"])
    for k, g in gold["tensors"].items():
        t = ins[k]
        assert list(t.shape) == g["shape"]
        got = synth.bf16_to_f64(t.reshape(-1)[:8])
        ref = synth.bf16_to_f64(np.array([int(b, 16) for b in g["first_bits"]], dtype=np.uint16))
        np.testing.assert_allclose(got, ref, rtol=2.0 ** -7, atol=0)
        assert math.isclose(float(synth.bf16_to_f64(t).sum()), g["sum"], rel_tol=1e-6, abs_tol=1e-6)


@pytest.mark.parametrize("name", ["qwen05b", "llama7b", "gemma7b"])
def test_config_flop_counts(name):
    """fwd+bwd FLOPs = 12 M h i + 18 M r (h + i) for the frozen-W LoRA MLP."""
    c = synth.MLP_CONFIGS[name]
    base = 3 * (2 * c.M * c.h * c.i) * 2      # three projections: forward product + dX product
    lora = 3 * 6 * c.M * c.r * (c.h + c.i)    # per linear: T, T B^T, U, U A, dA, dB
    assert c.flops() == pytest.approx(base + lora, rel=1e-12)


def test_positions_restart_at_each_sequence():
    assert synth.positions(7, seq=3).tolist() == [0, 1, 2, 0, 1, 2, 0]
    assert synth.positions(6, lengths=[2, 4]).tolist() == [0, 1, 0, 1, 2, 3]
    assert synth.positions(4, seq=3).dtype == torch.int32
    with pytest.raises(ValueError):
        synth.positions(5, lengths=[2, 2])
