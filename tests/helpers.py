"""Shared test helpers: the parity check and runners for the GPU path and the oracle."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Tolerances for bf16 inputs/outputs with f32 accumulation, per output tensor.
FRO_TOL = 1e-2      # relative Frobenius error
MAX_TOL = 3e-2      # max-abs error / max |ref|


def f64(t) -> np.ndarray:
    return synth.bf16_to_f64(t) if isinstance(t, torch.Tensor) and t.dtype == torch.bfloat16 \
        else np.asarray(t.detach().double().cpu().numpy() if isinstance(t, torch.Tensor) else t, np.float64)


def parity(name: str, got, ref, fro_tol=FRO_TOL, max_tol=MAX_TOL):
    """Asserts got (bf16 tensor) matches the float64 reference; returns (fro, max)."""
    g = f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, f"{name}: shape {g.shape} != {ref.shape}"
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    nr = np.linalg.norm(ref)
    if nr == 0.0:
        assert np.all(g == 0.0), f"{name}: reference is exactly zero, result is not"
        return 0.0, 0.0
    fro = float(np.linalg.norm(g - ref) / nr)
    mx = float(np.abs(g - ref).max() / np.abs(ref).max())
    assert fro <= fro_tol and mx <= max_tol, f"{name}: rel-fro {fro:.3e} (<= {fro_tol}), max {mx:.3e} (<= {max_tol})"
    return fro, mx


MLP_GRADS = ("dx", "dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down")


def mlp_gpu(lib, t: dict, cfg, s=None):
    """Runs forward + backward through the library on device tensors t."""
    s = cfg.s if s is None else s
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    y, saved = lib.mlp_forward(t["x"], lin("gate"), lin("up"), lin("down"), s, cfg.act)
    g = lib.mlp_backward(t["x"], lin("gate"), lin("up"), lin("down"), s, cfg.act, saved, t["dy"])
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
    return y, g


def mlp_oracle(v: dict, cfg, s=None):
    s = cfg.s if s is None else s
    args = (v["x"], v["W_gate"], v["A_gate"], v["B_gate"], v["W_up"], v["A_up"], v["B_up"],
            v["W_down"], v["A_down"], v["B_down"], s, cfg.act)
    return oracle.mlp_forward(*args), oracle.mlp_backward(*args, v["dy"])


def qkvo_gpu(lib, t: dict, cfg, s=None, rope=None, bias=None):
    """rope: None or dict(cos, sin, pos, head_dim) of device tensors."""
    s = cfg.s if s is None else s
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    out, saved = lib.qkvo_forward(t["x"], lin("q"), lin("k"), lin("v"), t["o_in"], lin("o"), s, rope=rope,
                                  bias=bias)
    g = lib.qkvo_backward(t["x"], lin("q"), lin("k"), lin("v"), t["o_in"], lin("o"), s, saved,
                          t["dy_q"], t["dy_k"], t["dy_v"], t["dy_o"], rope=rope)
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
    return out, g


def qkvo_oracle(v: dict, cfg, s=None, rope=None, bias=None):
    """rope: None or dict(cos, sin, pos, head_dim) of numpy arrays (the oracle's own
    tables); bias: None or (b_q, b_k, b_v)."""
    s = cfg.s if s is None else s
    L = lambda n: (v["W_" + n], v["A_" + n], v["B_" + n])  # noqa: E731
    f = oracle.qkvo_forward(v["x"], L("q"), L("k"), L("v"), v["o_in"], L("o"), s, bias=bias, rope=rope)
    b = oracle.qkvo_backward(v["x"], L("q"), L("k"), L("v"), v["o_in"], L("o"), s,
                             v["dy_q"], v["dy_k"], v["dy_v"], v["dy_o"], rope=rope)
    return f, b


def to_f64_dict(t: dict) -> dict:
    return {k: f64(v) for k, v in t.items()}
