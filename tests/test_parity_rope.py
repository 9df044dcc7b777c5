"""RoPE on q and k in the Q/K/V projection epilogue, and its transpose in the
backward, against the CPU float64 oracle ("Model Patches and Kernels", RoPE).

Head sizes 64, 128 and 256 (one, two or four heads per 256-column tile), GQA head
ratios 2, 4 and 8, q widths that end inside a tile, equal and packed sequences,
positions far into a long context, frozen biases before the rotation, and a
position outside the table (reported, not read).
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import f64, parity, qkvo_gpu, qkvo_oracle, to_f64_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("n_pos,head_dim,base", [(4096, 64, 10000.0), (2048, 128, 10000.0),
                                                 (8192, 256, 500000.0), (3, 2, 10.0)])
def test_rope_table(lib, n_pos, head_dim, base):
    cos, sin = lib.rope_table(n_pos, head_dim, base, device=DEV)
    torch.cuda.synchronize()
    oc, os_ = oracle.rope_tables(n_pos, head_dim, base)
    # computed in double, rounded once to f32
    assert np.max(np.abs(cos.cpu().double().numpy() - oc)) <= 6e-8
    assert np.max(np.abs(sin.cpu().double().numpy() - os_)) <= 6e-8


def _case(lib, M, h, hq, hkv, d, pos, n_pos, base=10000.0, bias=False, seed=0):
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=M, h=h, heads_q=hq, heads_kv=hkv, head_dim=d)
    ins = synth.make_qkvo_inputs(cfg, seed=seed)
    t = {k: x.to(DEV) for k, x in ins.items()}
    cos, sin = lib.rope_table(n_pos, d, base, device=DEV)
    rg = {"cos": cos, "sin": sin, "pos": pos.to(DEV), "head_dim": d}
    oc, os_ = oracle.rope_tables(n_pos, d, base)
    ro = {"cos": oc, "sin": os_, "pos": pos.numpy().astype(np.int64), "head_dim": d}
    bg = bo = None
    if bias:
        g = torch.Generator().manual_seed(seed + 50)
        b = synth.f64_to_bf16(torch.randn(cfg.n_q + 2 * cfg.n_kv, generator=g, dtype=torch.float64))
        bg = b.to(DEV)
        bv = f64(b)
        bo = (bv[:cfg.n_q], bv[cfg.n_q:cfg.n_q + cfg.n_kv], bv[cfg.n_q + cfg.n_kv:])
    out, grads = qkvo_gpu(lib, t, cfg, rope=rg, bias=bg)
    f, b = qkvo_oracle(to_f64_dict(ins), cfg, rope=ro, bias=bo)
    for k in ("q", "k", "v", "o"):
        parity(k, out[k], f[k])
    for k in b:
        parity(k, grads[k], b[k])


@pytest.mark.parametrize("M,h,hq,hkv,d,lengths,bias", [
    (300, 256, 4, 2, 64, [100, 100, 100], False),    # four heads per tile, ragged M
    (200, 512, 4, 1, 128, [17, 150, 33], True),      # packed sequences, GQA 4:1, bias
    (129, 512, 2, 1, 256, [64, 65], True),           # one head per tile
    (260, 384, 6, 2, 64, [260], False),              # q ends half-way into its second tile
    (192, 256, 8, 1, 64, [96, 96], True),            # GQA 8:1: k and v are 64 of a 256-wide tile
])
def test_qkvo_rope(lib, M, h, hq, hkv, d, lengths, bias):
    _case(lib, M, h, hq, hkv, d, synth.positions(M, lengths=lengths), n_pos=max(lengths), bias=bias)


def test_qkvo_rope_long_context_positions(lib):
    """Positions spread over a 32768-token context: angles up to ~3e4 rad."""
    M = 256
    g = torch.Generator().manual_seed(7)
    pos = torch.randint(0, 32768, (M,), generator=g, dtype=torch.int64).to(torch.int32)
    _case(lib, M, 256, 4, 2, 128, pos, n_pos=32768, base=500000.0, seed=3)


def test_rope_position_outside_the_table_is_reported(lib):
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=64, h=256, heads_q=2, heads_kv=1, head_dim=128)
    t = synth.make_qkvo_inputs(cfg, seed=1, device=DEV)
    cos, sin = lib.rope_table(16, 128, device=DEV)
    pos = synth.positions(64, seq=16)
    pos[5] = 16                                          # one past the table
    rg = {"cos": cos, "sin": sin, "pos": pos.to(DEV), "head_dim": 128}
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
    lib.qkvo_forward(t["x"], lin("q"), lin("k"), lin("v"), None, None, cfg.s, rope=rg)
    torch.cuda.synchronize()
    assert lib.poll_status() == 7
    pos[5] = 5
    rg["pos"] = pos.to(DEV)
    out, _ = lib.qkvo_forward(t["x"], lin("q"), lin("k"), lin("v"), None, None, cfg.s, rope=rg)
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
