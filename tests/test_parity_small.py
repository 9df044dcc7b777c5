"""GPU path vs the CPU float64 oracle on small and ragged problems (seconds each).

Sizes span several 128 x 256 tiles with ragged tails in M, N and K, ranks that
pad the folded K-segment (r = 1, 5, 8) and ranks that fill it (r = 64, 128), the
three activations (SwiGLU, tanh-GeGLU, exact GeGLU), frozen Q/K/V biases, and the
degenerate cases: one token, B = 0 (the base projections alone, adapter gradients
exactly zero) and s = 0.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import MLP_GRADS, f64, mlp_gpu, mlp_oracle, parity, qkvo_gpu, qkvo_oracle, to_f64_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _randn(shape, scale, seed):
    g = torch.Generator().manual_seed(seed)
    return synth.f64_to_bf16((torch.randn(*shape, generator=g, dtype=torch.float64) * scale))


def _linear(M, fin, fout, r, seed):
    x = _randn((M, fin), 1.0, seed)
    W = _randn((fout, fin), fin ** -0.5, seed + 1)
    A = _randn((r, fin), fin ** -0.5, seed + 2)
    B = _randn((fout, r), 0.02 ** 0.5, seed + 3)
    dy = _randn((M, fout), 1.0, seed + 4)
    return x, W, A, B, dy


@pytest.mark.parametrize("M,fin,fout,r", [
    (256, 256, 512, 8),      # whole tiles
    (300, 192, 328, 5),      # ragged M, K and N; r pads the fold
    (1, 64, 64, 1),          # one token, rank 1
    (129, 4096, 1024, 64),   # one row past a tile, full fold width
    (127, 520, 136, 16),     # K not a multiple of 64, N < one tile
    (200, 512, 384, 128),    # the widest fold of one adapter (128-column rank tiles)
    (1031, 896, 4864, 16),   # a prime token count at the Qwen-0.5B width
    (3, 8, 8, 1),            # the smallest feature sizes: every box wider than its tensor
    (70, 24, 40, 3),         # K and N below one 64-wide block, not powers of two
])
def test_linear_forward_backward(lib, M, fin, fout, r):
    s = 2.0
    x, W, A, B, dy = _linear(M, fin, fout, r, seed=M + fin)
    d = lambda t: t.to(DEV)  # noqa: E731
    y, saved = lib.linear_forward(d(x), (d(W), d(A), d(B)), s)
    dx, dA, dB = lib.linear_backward(d(x), (d(W), d(A), d(B)), s, saved, d(dy))
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
    v = [f64(t) for t in (x, W, A, B, dy)]
    parity("y", y, oracle.lora_linear(v[0], v[1], v[2], v[3], s))
    rdx, rdA, rdB = oracle.lora_linear_grad(v[0], v[1], v[2], v[3], s, v[4])
    parity("dx", dx, rdx)
    parity("dA", dA, rdA)
    parity("dB", dB, rdB)


def _mlp_inputs(cfg, seed=0, **zero):
    ins = synth.make_mlp_inputs(cfg, seed=seed)
    for k in zero:
        ins[k] = torch.zeros_like(ins[k])
    return {k: t.to(DEV) for k, t in ins.items()}, to_f64_dict(ins)


@pytest.mark.parametrize("act", ["swiglu", "geglu_tanh", "geglu_erf"])
@pytest.mark.parametrize("M", [64, 1, 127, 129])
def test_mlp_tiny(lib, act, M):
    cfg = synth.MLP_CONFIGS["tiny"].replace(act=act, M=M)
    t, v = _mlp_inputs(cfg)
    y, g = mlp_gpu(lib, t, cfg)
    f, b = mlp_oracle(v, cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


@pytest.mark.parametrize("act", ["swiglu", "geglu_tanh", "geglu_erf"])
def test_mlp_long_k_activations(lib, act):
    """h = 2304 gives the gate/up GEMM 37 k-blocks (> 32), so the forward runs the
    4-epilogue-warp pair kernel (the tiny cases take the 8-warp short-K one); each
    activation's compiled copy of the act epilogue is checked on both."""
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=260, h=2304, i=520, r=16, alpha=32, act=act)
    t, v = _mlp_inputs(cfg, seed=7)
    y, g = mlp_gpu(lib, t, cfg)
    f, b = mlp_oracle(v, cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


@pytest.mark.parametrize("M,h,i,r", [(5, 8, 16, 1), (33, 16, 8, 2)])
def test_mlp_smallest_features(lib, M, h, i, r):
    """Feature sizes of 8 and 16 (the alignment minimum): every tile and TMA box is
    mostly outside the tensors and reads zeros there."""
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=M, h=h, i=i, r=r, alpha=2.0 * r)
    t, v = _mlp_inputs(cfg, seed=M)
    y, g = mlp_gpu(lib, t, cfg)
    f, b = mlp_oracle(v, cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


@pytest.mark.parametrize("r", [1, 8, 64, 128])
def test_mlp_ranks(lib, r):
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=200, h=256, i=520, r=r, alpha=2 * r)
    t, v = _mlp_inputs(cfg, seed=r)
    y, g = mlp_gpu(lib, t, cfg)
    f, b = mlp_oracle(v, cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


@pytest.mark.parametrize("r", [5, 16])
def test_mlp_single_pass_ragged(lib, r):
    """The backward's single pass over dg, du (V and dB_g, dB_u from one read, r <= 16)
    on ragged extents: 1000 tokens (7 whole 128-token tiles and a part) and i = 1400
    (10 whole 128-feature blocks and a part), so its CTAs split both the token tiles and
    the feature blocks, and the last of each is partly outside the tensors."""
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=1000, h=384, i=1400, r=r, alpha=2 * r)
    t, v = _mlp_inputs(cfg, seed=11 + r)
    y, g = mlp_gpu(lib, t, cfg)
    f, b = mlp_oracle(v, cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


def test_mlp_zero_b_is_the_base_mlp(lib):
    """B = 0: the adapters contribute nothing and every dA is exactly zero."""
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=300)
    t, v = _mlp_inputs(cfg, B_gate=1, B_up=1, B_down=1)
    y, g = mlp_gpu(lib, t, cfg)
    f, b = mlp_oracle(v, cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])
    for k in ("dA_gate", "dA_up", "dA_down"):
        assert torch.count_nonzero(g[k]).item() == 0


def test_mlp_zero_scale_and_adapter_term(lib):
    """s = 0 gives the base MLP; the adapter's share of y, y(s) - y(0), matches the
    oracle's on its own (it is a fraction of |y|)."""
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=256)
    t, v = _mlp_inputs(cfg)
    y0, g0 = mlp_gpu(lib, t, cfg, s=0.0)
    y1, _ = mlp_gpu(lib, t, cfg)
    f0, b0 = mlp_oracle(v, cfg, s=0.0)
    f1, _ = mlp_oracle(v, cfg)
    parity("y(s=0)", y0, f0["y"])
    for k in ("dA_gate", "dA_up", "dA_down", "dB_gate", "dB_up", "dB_down"):
        assert torch.count_nonzero(g0[k]).item() == 0
    delta = f64(y1) - f64(y0)
    parity("y(s)-y(0)", torch.from_numpy(delta), f1["y"] - f0["y"], fro_tol=2e-2, max_tol=5e-2)


def test_qkvo_small(lib):
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=200, h=256, heads_q=4, heads_kv=2, head_dim=64)
    ins = synth.make_qkvo_inputs(cfg)
    t = {k: x.to(DEV) for k, x in ins.items()}
    out, g = qkvo_gpu(lib, t, cfg)
    f, b = qkvo_oracle(to_f64_dict(ins), cfg)
    for k in ("q", "k", "v", "o"):
        parity(k, out[k], f[k])
    for k in b:
        parity(k, g[k], b[k])


def test_qkvo_single_pass_rank10(lib):
    """Rank 10: the q/k/v half's single pass over dy_q, dy_k, dy_v carries three slots of
    10 columns in a 32-column projection (3 r <= 32) and reads each slot's T^T rows from
    a 16-row box that overlaps the next slot; 300 tokens (ragged)."""
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=300, h=256, heads_q=4, heads_kv=2, head_dim=64, r=10, alpha=20)
    ins = synth.make_qkvo_inputs(cfg, seed=5)
    t = {k: x.to(DEV) for k, x in ins.items()}
    out, g = qkvo_gpu(lib, t, cfg)
    f, b = qkvo_oracle(to_f64_dict(ins), cfg)
    for k in ("q", "k", "v", "o"):
        parity(k, out[k], f[k])
    for k in b:
        parity(k, g[k], b[k])


def test_qkvo_halves_independent(lib):
    """Either half can run alone (attention sits between them in a real block)."""
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=130, h=256, heads_q=4, heads_kv=2, head_dim=64, r=16)
    ins = synth.make_qkvo_inputs(cfg, seed=3)
    t = {k: x.to(DEV) for k, x in ins.items()}
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    f, b = qkvo_oracle(to_f64_dict(ins), cfg)
    out, saved = lib.qkvo_forward(t["x"], lin("q"), lin("k"), lin("v"), None, None, cfg.s)
    g = lib.qkvo_backward(t["x"], lin("q"), lin("k"), lin("v"), None, None, cfg.s, saved,
                          t["dy_q"], t["dy_k"], t["dy_v"], None)
    for k in ("q", "k", "v"):
        parity(k, out[k], f[k])
    for k in ("dx", "dA_q", "dB_q", "dA_k", "dB_k", "dA_v", "dB_v"):
        parity(k, g[k], b[k])
    out, saved = lib.qkvo_forward(None, None, None, None, t["o_in"], lin("o"), cfg.s)
    g = lib.qkvo_backward(None, None, None, None, t["o_in"], lin("o"), cfg.s, saved, dyo=t["dy_o"])
    torch.cuda.synchronize()
    parity("o", out["o"], f["o"])
    for k in ("do_in", "dA_o", "dB_o"):
        parity(k, g[k], b[k])


def test_deterministic(lib):
    """Split-K reductions run in a fixed order: repeated calls give identical bits."""
    cfg = synth.MLP_CONFIGS["qwen05b"].replace(M=1000)
    t, _ = _mlp_inputs(cfg)
    y1, g1 = mlp_gpu(lib, t, cfg)
    y2, g2 = mlp_gpu(lib, t, cfg)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    for k in MLP_GRADS:
        assert torch.equal(g1[k].view(torch.int16), g2[k].view(torch.int16)), k


def test_mlp_geglu_erf_gemma_like(lib):
    """Exact-erf GeGLU (the Gemma row of the activation table) at a Gemma-like width."""
    cfg = synth.MLP_CONFIGS["gemma7b"].replace(M=512, h=768, i=3072, act="geglu_erf")
    t, v = _mlp_inputs(cfg, seed=4)
    y, g = mlp_gpu(lib, t, cfg)
    f, b = mlp_oracle(v, cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


def test_qkvo_frozen_bias(lib):
    """Frozen base-layer q/k/v biases are added in the projection epilogue; the
    backward is unchanged."""
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=300, h=256, heads_q=4, heads_kv=2, head_dim=64)
    ins = synth.make_qkvo_inputs(cfg, seed=6)
    t = {k: x.to(DEV) for k, x in ins.items()}
    nb = cfg.n_q + 2 * cfg.n_kv
    bias = _randn((nb,), 1.0, 99).to(DEV)
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    out, saved = lib.qkvo_forward(t["x"], lin("q"), lin("k"), lin("v"), t["o_in"], lin("o"), cfg.s, bias=bias)
    g = lib.qkvo_backward(t["x"], lin("q"), lin("k"), lin("v"), t["o_in"], lin("o"), cfg.s, saved,
                          t["dy_q"], t["dy_k"], t["dy_v"], t["dy_o"])
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
    v = to_f64_dict(ins)
    bv = f64(bias)
    bsplit = (bv[:cfg.n_q], bv[cfg.n_q:cfg.n_q + cfg.n_kv], bv[cfg.n_q + cfg.n_kv:])
    L = lambda n: (v["W_" + n], v["A_" + n], v["B_" + n])  # noqa: E731
    f = oracle.qkvo_forward(v["x"], L("q"), L("k"), L("v"), v["o_in"], L("o"), cfg.s, bias=bsplit)
    b = oracle.qkvo_backward(v["x"], L("q"), L("k"), L("v"), v["o_in"], L("o"), cfg.s,
                             v["dy_q"], v["dy_k"], v["dy_v"], v["dy_o"])
    for k in ("q", "k", "v", "o"):
        parity(k, out[k], f[k])
    for k in b:
        parity(k, g[k], b[k])


@pytest.mark.parametrize("name,over,n_ex", [
    ("tiny", {}, 2),                                # seq 32: less than one 64-token block
    ("tiny", {"M": 300, "i": 520, "h": 256}, 3),    # seq 100: ragged block per example
    ("qwen05b", {"M": 2048}, 4),                    # seq 512
    ("tiny", {"M": 256, "i": 520, "h": 256, "act": "geglu_tanh"}, 4),
    ("tiny", {"M": 192, "i": 344, "h": 128, "act": "geglu_erf", "r": 64, "alpha": 128}, 3),
    ("tiny", {"M": 24}, 24),                        # seq 1: one token per example
    ("tiny", {"M": 35, "i": 520}, 5),               # seq 7: odd
])
def test_mlp_per_example_grads(lib, name, over, n_ex):
    """DP-SGD per-example adapter gradients and their squared norms."""
    cfg = synth.MLP_CONFIGS[name].replace(**over)
    t, v = _mlp_inputs(cfg, seed=8)
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    y, saved = lib.mlp_forward(t["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    g = lib.mlp_backward_per_example(t["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved,
                                     t["dy"], n_ex)
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
    args = (v["x"], v["W_gate"], v["A_gate"], v["B_gate"], v["W_up"], v["A_up"], v["B_up"],
            v["W_down"], v["A_down"], v["B_down"], cfg.s, cfg.act)
    ref = oracle.mlp_backward_per_example(*args, v["dy"], n_ex)
    parity("dx", g["dx"], ref["dx"])
    for k in ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"):
        for e in range(n_ex):
            parity(f"{k}[{e}]", g[k][e], ref[k][e])
    np.testing.assert_allclose(g["sq_norms"].double().cpu().numpy(), ref["sq_norms"], rtol=2e-2)


def test_qkvo_largest_rank(lib):
    """r = 85: three adapters fill the 256-column fold of q, k, v (the rank limit)."""
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=257, h=384, heads_q=3, heads_kv=1, head_dim=128, r=85,
                                              alpha=170)
    ins = synth.make_qkvo_inputs(cfg, seed=9)
    t = {k: x.to(DEV) for k, x in ins.items()}
    out, g = qkvo_gpu(lib, t, cfg)
    f, b = qkvo_oracle(to_f64_dict(ins), cfg)
    for k in ("q", "k", "v", "o"):
        parity(k, out[k], f[k])
    for k in b:
        parity(k, g[k], b[k])
