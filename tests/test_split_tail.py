"""The CTA-pair GEMM's split tail: when whole 256 x 256 tiles dealt round-robin would
leave pairs idle in the last wave, the tiles of that partial wave (all tiles, when
there are fewer than pairs) are each cut into 2 to 4 equal k-ranges computed by
different pairs, and the last piece of a tile to arrive adds the others' partial sums
before the epilogue.  Each case runs with every tail cut into 2, 3 and 4 pieces
(lora_set_split_tail).  On a 152-SM GPU (76 pairs) the shapes cover one tile, fewer
tiles than pairs, a full wave of whole tiles followed by a tail, ragged M and N, every
epilogue kind (plain store with bias, activation, activation derivative, RoPE) and a
launch of three groups.  Results are compared with the float64 oracle and must repeat
bit for bit."""

import pytest
import torch

import oracle
import synth
from helpers import MLP_GRADS, f64, mlp_gpu, mlp_oracle, parity, qkvo_gpu, qkvo_oracle, to_f64_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(params=[2, 3, 4])
def pieces(request, lib):
    """Every tail cut into this many pieces for the test, automatic mode after it."""
    lib.set_split_tail(request.param)
    yield request.param
    lib.set_split_tail(0)


def _linear_case(M, fin, fout, r, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *sh, sc=1.0: synth.f64_to_bf16(torch.randn(*sh, generator=g, dtype=torch.float64) * sc)  # noqa: E731
    return (mk(M, fin), mk(fout, fin, sc=fin ** -0.5), mk(r, fin, sc=fin ** -0.5), mk(fout, r, sc=0.14),
            mk(M, fout))


def _bits(t):
    return t.reshape(-1).view(torch.int16)


@pytest.mark.parametrize("M,fin,fout", [
    (256, 1024, 256),       # forward: 1 tile (the backward's 5 k-blocks stay whole)
    (1000, 1024, 1000),     # 16 ragged tiles, forward and backward
    (512, 2560, 13568),     # forward: 76 whole tiles, then a tail of 30; backward: 20 tiles
    (768, 1536, 8192),      # forward: 76 whole tiles, then a tail of 20; backward: 18 tiles
])
def test_linear_split_tail(lib, pieces, M, fin, fout):
    s, r = 1.5, 16
    x, W, A, B, dy = _linear_case(M, fin, fout, r, seed=M + fout)
    d = lambda t: t.to(DEV)  # noqa: E731
    lin = (d(W), d(A), d(B))
    outs = []
    for _ in range(2):
        y, saved = lib.linear_forward(d(x), lin, s)
        dx, dA, dB = lib.linear_backward(d(x), lin, s, saved, d(dy))
        torch.cuda.synchronize()
        outs.append((y.clone(), dx.clone(), dA.clone(), dB.clone()))
    assert lib.poll_status() == 0
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(_bits(a), _bits(b))
    v = [f64(t) for t in (x, W, A, B)]
    parity("y", outs[0][0], oracle.lora_linear(*v, s))
    ref = oracle.lora_linear_grad(*v, s, f64(dy))
    for name, got, want in zip(("dx", "dA", "dB"), outs[0][1:], ref):
        parity(name, got, want)


@pytest.mark.parametrize("act", ["swiglu", "geglu_tanh", "geglu_erf"])
def test_mlp_split_tail(lib, pieces, act):
    """512 tokens, h = 2048, i = 1024: gate/up 16 tiles (activation epilogue), act' 8
    tiles (derivative epilogue), down and dx 16 tiles each."""
    cfg = synth.MLP_CONFIGS["qwen05b"].replace(M=512, h=2048, i=1024, act=act)
    ins = synth.make_mlp_inputs(cfg, seed=31)
    t = {k: v.to(DEV) for k, v in ins.items()}
    y1, g1 = mlp_gpu(lib, t, cfg)
    y2, g2 = mlp_gpu(lib, t, cfg)
    assert torch.equal(_bits(y1), _bits(y2))
    for k in MLP_GRADS:
        assert torch.equal(_bits(g1[k]), _bits(g2[k])), k
    f, b = mlp_oracle(to_f64_dict(ins), cfg)
    parity("y", y1, f["y"])
    for k in MLP_GRADS:
        parity(k, g1[k], b[k])


def test_qkvo_split_tail_with_rope_and_bias(lib, pieces):
    """512 tokens, h = 2048, 16/4 heads of 128: the q/k/v launch has 16 + 2 x 4 tiles on
    three groups (RoPE, RoPE, bias only); O, d o_in and dx 16 tiles each."""
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=512, h=2048, heads_q=16, heads_kv=4, head_dim=128)
    ins = synth.make_qkvo_inputs(cfg, seed=32)
    t = {k: v.to(DEV) for k, v in ins.items()}
    n_pos = 256
    cos, sin = lib.rope_table(n_pos, cfg.head_dim, device=DEV)
    pos = synth.positions(cfg.M, seq=256, device=DEV)
    rope = {"cos": cos, "sin": sin, "pos": pos, "head_dim": cfg.head_dim}
    nb = cfg.n_q + 2 * cfg.n_kv
    gb = torch.Generator().manual_seed(33)
    bias = synth.f64_to_bf16(torch.randn(nb, generator=gb, dtype=torch.float64) * 0.5)
    out1, g1 = qkvo_gpu(lib, t, cfg, rope=rope, bias=bias.to(DEV))
    out2, g2 = qkvo_gpu(lib, t, cfg, rope=rope, bias=bias.to(DEV))
    for k in out1:
        assert torch.equal(_bits(out1[k]), _bits(out2[k])), k
    for k in g1:
        assert torch.equal(_bits(g1[k]), _bits(g2[k])), k
    c64, s64 = oracle.rope_tables(n_pos, cfg.head_dim)
    orope = {"cos": c64, "sin": s64, "pos": pos.cpu().numpy(), "head_dim": cfg.head_dim}
    bq = f64(bias)
    ob = (bq[:cfg.n_q], bq[cfg.n_q:cfg.n_q + cfg.n_kv], bq[cfg.n_q + cfg.n_kv:])
    f, b = qkvo_oracle(to_f64_dict(ins), cfg, rope=orope, bias=ob)
    for k in out1:
        parity(k, out1[k], f[k])
    for k in g1:
        parity(k, g1[k], b[k])
