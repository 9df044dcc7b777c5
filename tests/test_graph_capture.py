"""The MLP and Q/K/V + O entry points under CUDA graph capture: after one eager call
(which raises the kernels' shared-memory limits and sizes the cached workspace), a
forward + backward captured in a graph replays to the same bits as eager calls, with
the inputs updated in place between replays."""

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bits(t):
    return t.reshape(-1).view(torch.int16)


def test_mlp_step_in_a_graph(lib):
    cfg = synth.MLP_CONFIGS["qwen05b"].replace(M=1024)
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg, seed=21).items()}
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    x = ins["x"].clone()
    dy = ins["dy"].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        def step():
            y, saved = lib.mlp_forward(x, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
            g = lib.mlp_backward(x, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved, dy)
            return y, g
        step()                                        # eager: limits, workspace
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            y_g, g_g = step()
    torch.cuda.synchronize()
    for seed in (0, 1):
        x.copy_(torch.roll(ins["x"], seed * 7, dims=0))
        dy.copy_(torch.roll(ins["dy"], seed * 5, dims=0))
        graph.replay()
        torch.cuda.synchronize()
        y_e, g_e = step()
        torch.cuda.synchronize()
        assert torch.equal(_bits(y_g), _bits(y_e))
        for k in g_e:
            assert torch.equal(_bits(g_g[k]), _bits(g_e[k])), k
    assert lib.poll_status() == 0


def test_qkvo_step_with_rope_in_a_graph(lib):
    cfg = synth.QKVO_CONFIGS["gqa7b"].replace(M=512, h=512, heads_q=4, heads_kv=2, head_dim=128)
    t = {k: x.to(DEV) for k, x in synth.make_qkvo_inputs(cfg, seed=22).items()}
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    cos, sin = lib.rope_table(256, 128, device=DEV)
    rope = {"cos": cos, "sin": sin, "pos": synth.positions(512, seq=256, device=DEV), "head_dim": 128}

    def step():
        out, saved = lib.qkvo_forward(t["x"], lin("q"), lin("k"), lin("v"), t["o_in"], lin("o"), cfg.s, rope=rope)
        g = lib.qkvo_backward(t["x"], lin("q"), lin("k"), lin("v"), t["o_in"], lin("o"), cfg.s, saved,
                              t["dy_q"], t["dy_k"], t["dy_v"], t["dy_o"], rope=rope)
        return out, g

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            out_g, g_g = step()
    graph.replay()
    torch.cuda.synchronize()
    out_e, g_e = step()
    torch.cuda.synchronize()
    for k in out_e:
        assert torch.equal(_bits(out_g[k]), _bits(out_e[k])), k
    for k in g_e:
        assert torch.equal(_bits(g_g[k]), _bits(g_e[k])), k
    assert lib.poll_status() == 0
