"""The autograd functions route tensors only: gradients through loss.backward() equal,
bit for bit, the library's backward called directly on the same tensors, the frozen W
gets no gradient, and leading batch dimensions pass through."""

import pytest
import torch

import synth

DEV = "cuda:0"


def test_module_imports_without_a_gpu():
    from rank_mlp_gb300 import autograd
    assert hasattr(autograd, "LoraMLPFunction") and hasattr(autograd, "LoraQKVFunction")


def _leaf(t, grad):
    return t.to(DEV).requires_grad_(grad)


def _same(a, b):
    return torch.equal(a.reshape(-1).view(torch.int16), b.reshape(-1).view(torch.int16))


@pytest.mark.gpu
def test_mlp_function_matches_the_library(lib):
    from rank_mlp_gb300 import autograd
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=256, h=256, i=520, act="geglu_tanh")
    ins = synth.make_mlp_inputs(cfg, seed=2)
    p = {k: _leaf(v, k.startswith(("A_", "B_"))) for k, v in ins.items() if k not in ("x", "dy")}
    x = ins["x"].to(DEV).reshape(4, 64, cfg.h).requires_grad_(True)
    dy = ins["dy"].to(DEV).reshape(4, 64, cfg.h)
    lin = lambda n: (p["W_" + n], p["A_" + n], p["B_" + n])  # noqa: E731
    y = autograd.lora_mlp(x, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    assert y.shape == (4, 64, cfg.h)
    y.backward(dy)
    with torch.no_grad():
        x2 = x.detach().reshape(-1, cfg.h)
        y_ref, saved = lib.mlp_forward(x2, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
        g = lib.mlp_backward(x2, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved, dy.reshape(-1, cfg.h))
    assert _same(y.detach(), y_ref)
    assert _same(x.grad, g["dx"])
    for n in ("gate", "up", "down"):
        assert p["W_" + n].grad is None
        assert _same(p["A_" + n].grad, g["dA_" + n]) and _same(p["B_" + n].grad, g["dB_" + n])


@pytest.mark.gpu
def test_qkv_and_linear_functions_match_the_library(lib):
    from rank_mlp_gb300 import autograd
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=256, h=256, heads_q=4, heads_kv=2, head_dim=64)
    ins = synth.make_qkvo_inputs(cfg, seed=4)
    p = {k: _leaf(v, k.startswith(("A_", "B_"))) for k, v in ins.items() if k[:2] in ("W_", "A_", "B_")}
    x = ins["x"].to(DEV).reshape(2, 128, cfg.h).requires_grad_(True)
    cos, sin = lib.rope_table(128, 64, device=DEV)
    rope = {"cos": cos, "sin": sin, "pos": synth.positions(256, seq=128, device=DEV), "head_dim": 64}
    g0 = torch.Generator().manual_seed(1)
    bias = synth.f64_to_bf16(torch.randn(cfg.n_q + 2 * cfg.n_kv, generator=g0, dtype=torch.float64)).to(DEV)
    lin = lambda n: (p["W_" + n], p["A_" + n], p["B_" + n])  # noqa: E731
    q, k, v = autograd.lora_qkv(x, lin("q"), lin("k"), lin("v"), cfg.s, bias=bias, rope=rope)
    dq, dk, dv = (ins["dy_" + n].to(DEV).reshape(2, 128, -1) for n in ("q", "k", "v"))
    torch.autograd.backward([q, k, v], [dq, dk, dv])
    with torch.no_grad():
        x2 = x.detach().reshape(-1, cfg.h)
        out, saved = lib.qkvo_forward(x2, lin("q"), lin("k"), lin("v"), None, None, cfg.s, bias=bias, rope=rope)
        g = lib.qkvo_backward(x2, lin("q"), lin("k"), lin("v"), None, None, cfg.s, saved,
                              dq.reshape(256, -1), dk.reshape(256, -1), dv.reshape(256, -1), None, rope=rope)
    for n, t in (("q", q), ("k", k), ("v", v)):
        assert _same(t.detach(), out[n])
        assert p["W_" + n].grad is None
        assert _same(p["A_" + n].grad, g["dA_" + n]) and _same(p["B_" + n].grad, g["dB_" + n])
    assert _same(x.grad, g["dx"])

    o_in = ins["o_in"].to(DEV).reshape(2, 128, cfg.n_q).requires_grad_(True)
    yo = autograd.lora_linear(o_in, lin("o"), cfg.s)
    dyo = ins["dy_o"].to(DEV).reshape(2, 128, cfg.h)
    yo.backward(dyo)
    with torch.no_grad():
        o2 = o_in.detach().reshape(-1, cfg.n_q)
        y_ref, sv = lib.linear_forward(o2, lin("o"), cfg.s)
        dx, dA, dB = lib.linear_backward(o2, lin("o"), cfg.s, sv, dyo.reshape(-1, cfg.h))
    assert _same(yo.detach(), y_ref) and _same(o_in.grad, dx)
    assert _same(p["A_o"].grad, dA) and _same(p["B_o"].grad, dB) and p["W_o"].grad is None
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
