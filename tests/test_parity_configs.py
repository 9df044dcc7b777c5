"""GPU path vs the CPU float64 oracle on the five full-size workloads, every output
element compared (the oracle runs the whole problem with float64 BLAS products).

Workloads: the tiny MLP; the Qwen2.5-0.5B-shaped MLP (and its M = 4095 tail); the
7B-shaped MLP; the Gemma-7B-shaped tanh-GeGLU MLP at r = 8 and r = 64; the GQA
Q/K/V + O projections.  Inputs come from the seeded generator (made on the device,
copied to the host for the oracle, so both sides read the same bf16 values).
"""

import gc

import pytest
import torch

import synth
from helpers import MLP_GRADS, mlp_gpu, mlp_oracle, parity, qkvo_gpu, qkvo_oracle, to_f64_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

MLP_CASES = [
    ("tiny", {}),
    ("qwen05b", {}),
    ("qwen05b", {"M": 4095}),
    ("llama7b", {}),
    ("gemma7b", {}),
    ("gemma7b", {"r": 64, "alpha": 128}),
]


@pytest.mark.parametrize("name,over", MLP_CASES, ids=[f"{n}{'-' + str(o) if o else ''}" for n, o in MLP_CASES])
def test_mlp_config(lib, name, over):
    cfg = synth.MLP_CONFIGS[name].replace(**over)
    t = synth.make_mlp_inputs(cfg, seed=0, device=DEV)
    y, g = mlp_gpu(lib, t, cfg)
    got = {"y": y.cpu(), **{k: g[k].cpu() for k in MLP_GRADS}}
    v = to_f64_dict(t)
    del t, g, y
    torch.cuda.empty_cache()
    f, b = mlp_oracle(v, cfg)
    parity("y", got["y"], f["y"])
    for k in MLP_GRADS:
        parity(k, got[k], b[k])
    del f, b, v
    gc.collect()


@pytest.mark.parametrize("rope", [False, True], ids=["plain", "rope"])
def test_qkvo_config(lib, rope):
    """The GQA Q/K/V + O workload; with RoPE on q and k (positions restart every
    sequence of cfg.seq tokens, base 10000)."""
    import oracle
    cfg = synth.QKVO_CONFIGS["gqa7b"]
    t = synth.make_qkvo_inputs(cfg, seed=0, device=DEV)
    rg = ro = None
    if rope:
        pos = synth.positions(cfg.M, seq=cfg.seq)
        cos, sin = lib.rope_table(cfg.seq, cfg.head_dim, 10000.0, device=DEV)
        rg = {"cos": cos, "sin": sin, "pos": pos.to(DEV), "head_dim": cfg.head_dim}
        oc, os_ = oracle.rope_tables(cfg.seq, cfg.head_dim, 10000.0)
        ro = {"cos": oc, "sin": os_, "pos": pos.numpy().astype(int), "head_dim": cfg.head_dim}
    out, g = qkvo_gpu(lib, t, cfg, rope=rg)
    got = {**{k: out[k].cpu() for k in out}, **{k: g[k].cpu() for k in g}}
    v = to_f64_dict(t)
    del t, out, g, rg
    torch.cuda.empty_cache()
    f, b = qkvo_oracle(v, cfg, rope=ro)
    for k in ("q", "k", "v", "o"):
        parity(k, got[k], f[k])
    for k in b:
        parity(k, got[k], b[k])
