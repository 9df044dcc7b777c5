"""torch.autograd functions over the library's entry points, for training loops that
call ``loss.backward()``.

They only route tensors: the forward and backward of each function are one call each
of ``lora_mlp_forward/backward``, ``lora_qkvo_forward/backward`` (the Q/K/V half) and
``lora_linear_forward/backward``.  The base weights W are frozen ("Model Patches and
Kernels": a frozen weight gets no gradient), so they never receive a gradient; the
adapters A, B and the input x do.  Inputs may carry leading batch dimensions
([..., features]); every tensor is bf16 on the GPU.
"""

from __future__ import annotations

import torch

from . import binding


def _flat(t: torch.Tensor) -> torch.Tensor:
    return t.reshape(-1, t.shape[-1]).contiguous()


def _bf16(t: torch.Tensor) -> torch.Tensor:
    return t if t.dtype == torch.bfloat16 else t.to(torch.bfloat16)


class LoraMLPFunction(torch.autograd.Function):
    """y = down(act(gate(x)) * up(x)), each a LoRA linear W x + s B A x."""

    @staticmethod
    def forward(ctx, x, Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, s: float, act: str = "swiglu"):
        x2 = _flat(x)
        y, saved = binding.mlp_forward(x2, (Wg, Ag, Bg), (Wu, Au, Bu), (Wd, Ad, Bd), s, act)
        ctx.save_for_backward(x2, Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, saved)
        ctx.s, ctx.act, ctx.xshape = s, act, x.shape
        return y.reshape(*x.shape[:-1], y.shape[-1])

    @staticmethod
    def backward(ctx, dy):
        x2, Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, saved = ctx.saved_tensors
        g = binding.mlp_backward(x2, (Wg, Ag, Bg), (Wu, Au, Bu), (Wd, Ad, Bd), ctx.s, ctx.act, saved,
                                 _bf16(_flat(dy)))
        return (g["dx"].reshape(ctx.xshape), None, g["dA_gate"], g["dB_gate"], None, g["dA_up"], g["dB_up"],
                None, g["dA_down"], g["dB_down"], None, None)


class LoraQKVFunction(torch.autograd.Function):
    """(q, k, v) from one input, each a LoRA linear, with optional frozen biases (one
    bf16 tensor [n_q + 2 n_kv]) and optional RoPE on q and k (dict(cos, sin, pos,
    head_dim), see ``binding.rope_table``)."""

    @staticmethod
    def forward(ctx, x, Wq, Aq, Bq, Wk, Ak, Bk, Wv, Av, Bv, s: float, bias=None, rope=None):
        x2 = _flat(x)
        out, saved = binding.qkvo_forward(x2, (Wq, Aq, Bq), (Wk, Ak, Bk), (Wv, Av, Bv), None, None, s,
                                          bias=bias, rope=rope)
        ctx.save_for_backward(x2, Wq, Aq, Bq, Wk, Ak, Bk, Wv, Av, Bv, saved)
        ctx.s, ctx.rope, ctx.xshape = s, rope, x.shape
        lead = x.shape[:-1]
        return tuple(out[n].reshape(*lead, out[n].shape[-1]) for n in ("q", "k", "v"))

    @staticmethod
    def backward(ctx, dq, dk, dv):
        x2, Wq, Aq, Bq, Wk, Ak, Bk, Wv, Av, Bv, saved = ctx.saved_tensors
        z = lambda d, W: torch.zeros(x2.shape[0], W.shape[0], dtype=torch.bfloat16, device=x2.device) \
            if d is None else _bf16(_flat(d))  # noqa: E731
        g = binding.qkvo_backward(x2, (Wq, Aq, Bq), (Wk, Ak, Bk), (Wv, Av, Bv), None, None, ctx.s, saved,
                                  z(dq, Wq), z(dk, Wk), z(dv, Wv), None, rope=ctx.rope)
        return (g["dx"].reshape(ctx.xshape), None, g["dA_q"], g["dB_q"], None, g["dA_k"], g["dB_k"],
                None, g["dA_v"], g["dB_v"], None, None, None)


class LoraLinearFunction(torch.autograd.Function):
    """y = x W^T + s (x A^T) B^T (the output projection, or any single LoRA linear)."""

    @staticmethod
    def forward(ctx, x, W, A, B, s: float):
        x2 = _flat(x)
        y, saved = binding.linear_forward(x2, (W, A, B), s)
        ctx.save_for_backward(x2, W, A, B, saved)
        ctx.s, ctx.xshape = s, x.shape
        return y.reshape(*x.shape[:-1], y.shape[-1])

    @staticmethod
    def backward(ctx, dy):
        x2, W, A, B, saved = ctx.saved_tensors
        dx, dA, dB = binding.linear_backward(x2, (W, A, B), ctx.s, saved, _bf16(_flat(dy)))
        return dx.reshape(ctx.xshape), None, dA, dB, None


def lora_mlp(x, gate, up, down, s, act="swiglu"):
    """gate, up, down: (W, A, B) triples."""
    return LoraMLPFunction.apply(x, *gate, *up, *down, s, act)


def lora_qkv(x, q, k, v, s, bias=None, rope=None):
    return LoraQKVFunction.apply(x, *q, *k, *v, s, bias, rope)


def lora_linear(x, lin, s):
    return LoraLinearFunction.apply(x, *lin, s)
