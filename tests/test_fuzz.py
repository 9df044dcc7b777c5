"""Seeded random problem shapes against the oracle: token counts, feature sizes
(multiples of 8), ranks up to the fold limits, all three activations, and Q/K/V + O
with random head layouts, biases and RoPE.  Every draw is fixed by the seed, so a
failure names a reproducible case."""

import random

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import MLP_GRADS, f64, mlp_gpu, mlp_oracle, parity, qkvo_gpu, qkvo_oracle, to_f64_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _mlp_cases(n=30, seed=1234):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        r = rng.choice([1, 2, 3, 7, 8, 16, 33, 64, 100, 128])
        out.append(dict(M=rng.randint(1, 700), h=8 * rng.randint(1, 96), i=8 * rng.randint(1, 200), r=r,
                        alpha=float(rng.choice([r, 2 * r, 16])), act=rng.choice(oracle.ACTS)))
    return out


@pytest.mark.parametrize("case", _mlp_cases(), ids=lambda c: "M{M}-h{h}-i{i}-r{r}-{act}".format(**c))
def test_mlp_random_shapes(lib, case):
    cfg = synth.MLP_CONFIGS["tiny"].replace(**case)
    ins = synth.make_mlp_inputs(cfg, seed=case["M"])
    t = {k: x.to(DEV) for k, x in ins.items()}
    y, g = mlp_gpu(lib, t, cfg)
    f, b = mlp_oracle(to_f64_dict(ins), cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


def _qkvo_cases(n=20, seed=4321):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        d = rng.choice([64, 128, 256])
        hkv = rng.randint(1, 3)
        hq = hkv * rng.choice([1, 2, 4])
        out.append(dict(M=rng.randint(1, 600), h=8 * rng.randint(4, 96), heads_q=hq, heads_kv=hkv, head_dim=d,
                        r=rng.choice([1, 4, 8, 16, 40, 85]), rope=rng.random() < 0.7, bias=rng.random() < 0.5))
    return out


@pytest.mark.parametrize("case", _qkvo_cases(),
                         ids=lambda c: "M{M}-h{h}-q{heads_q}-kv{heads_kv}-d{head_dim}-r{r}-rope{rope}-bias{bias}".format(**c))
def test_qkvo_random_shapes(lib, case):
    c = dict(case)
    use_rope, use_bias = c.pop("rope"), c.pop("bias")
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(alpha=2.0 * c["r"], **c)
    ins = synth.make_qkvo_inputs(cfg, seed=c["M"] + 1)
    t = {k: x.to(DEV) for k, x in ins.items()}
    rg = ro = bg = bo = None
    if use_rope:
        n_pos = max(2, cfg.M // 2 + 1)
        pos = synth.positions(cfg.M, lengths=[cfg.M // 2, cfg.M - cfg.M // 2]) if cfg.M > 1 else \
            synth.positions(1, seq=1)
        cos, sin = lib.rope_table(n_pos, cfg.head_dim, device=DEV)
        rg = {"cos": cos, "sin": sin, "pos": pos.to(DEV), "head_dim": cfg.head_dim}
        oc, os_ = oracle.rope_tables(n_pos, cfg.head_dim)
        ro = {"cos": oc, "sin": os_, "pos": pos.numpy().astype(np.int64), "head_dim": cfg.head_dim}
    if use_bias:
        gen = torch.Generator().manual_seed(c["M"])
        b = synth.f64_to_bf16(torch.randn(cfg.n_q + 2 * cfg.n_kv, generator=gen, dtype=torch.float64))
        bg = b.to(DEV)
        bv = f64(b)
        bo = (bv[:cfg.n_q], bv[cfg.n_q:cfg.n_q + cfg.n_kv], bv[cfg.n_q + cfg.n_kv:])
    out, g = qkvo_gpu(lib, t, cfg, rope=rg, bias=bg)
    f, b = qkvo_oracle(to_f64_dict(ins), cfg, rope=ro, bias=bo)
    for k in ("q", "k", "v", "o"):
        parity(k, out[k], f[k])
    for k in b:
        parity(k, g[k], b[k])
