"""Pins for the CPU float64 oracle (no GPU).

Each test checks the oracle against something other than its own formula: library
routines on the special cases that reduce to them, closed forms, the LoRA merged-
weight identity, finite differences, and linearity in s.  The mutation tests at the
end plant plausible mistakes in the oracle and check that these pins catch them.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import lora as olora

RNG = np.random.default_rng(1234)


def _rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# ---------------------------------------------------------------- activations

GRID = np.linspace(-20.0, 20.0, 4001)


def test_silu_matches_torch_library():
    ref = F.silu(torch.from_numpy(GRID)).numpy()
    np.testing.assert_allclose(oracle.silu(GRID), ref, rtol=1e-14, atol=1e-14)


def test_gelu_tanh_matches_torch_library():
    ref = F.gelu(torch.from_numpy(GRID), approximate="tanh").numpy()
    np.testing.assert_allclose(oracle.gelu_tanh(GRID), ref, rtol=1e-13, atol=1e-14)


def test_gelu_erf_matches_torch_library():
    ref = F.gelu(torch.from_numpy(GRID), approximate="none").numpy()
    np.testing.assert_allclose(oracle.gelu_erf(GRID), ref, rtol=1e-13, atol=1e-14)


def test_gelu_erf_closed_values():
    # Phi(1) = (1 + erf(1/sqrt 2)) / 2; gelu(1) = Phi(1)
    assert math.isclose(oracle.gelu_erf(np.array([1.0]))[0], 0.5 * (1.0 + math.erf(1.0 / math.sqrt(2.0))),
                        rel_tol=1e-15)
    assert oracle.gelu_erf(np.array([0.0]))[0] == 0.0


def test_activation_closed_values_and_asymptotes():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert oracle.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert math.isclose(oracle.silu(np.array([1.0]))[0], 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    # silu(g) -> g for g -> +inf, -> 0 for g -> -inf; the same for gelu
    for f in (oracle.silu, oracle.gelu_tanh, oracle.gelu_erf):
        big = np.array([40.0])
        assert abs(f(big)[0] - 40.0) < 1e-12
        assert abs(f(-big)[0]) < 1e-12


@pytest.mark.parametrize("kind", oracle.ACTS)
def test_act_prime_closed_form_vs_central_difference(kind):
    eps = 1e-5
    fd = (oracle.act(GRID + eps, kind) - oracle.act(GRID - eps, kind)) / (2 * eps)
    np.testing.assert_allclose(oracle.act_prime(GRID, kind), fd, rtol=0, atol=1e-8)


def test_act_prime_limits():
    # silu'(0) = 1/2, gelu'(0) = 1/2; both tend to 1 at +inf and 0 at -inf
    for kind in oracle.ACTS:
        d = oracle.act_prime(np.array([0.0, 40.0, -40.0]), kind)
        np.testing.assert_allclose(d, [0.5, 1.0, 0.0], atol=1e-12)


# ---------------------------------------------------------------- one LoRA linear

def _linear_case(M=5, fin=7, fout=6, r=3):
    return (_rand(M, fin), _rand(fout, fin), _rand(r, fin), _rand(fout, r), 1.75)


def test_merged_weight_identity_forward():
    """LoRA's merged form: x W^T + s x A^T B^T == x (W + s B A)^T."""
    x, W, A, B, s = _linear_case()
    merged = x @ (W + s * B @ A).T
    np.testing.assert_allclose(oracle.lora_linear(x, W, A, B, s), merged, rtol=1e-12, atol=1e-12)


def test_merged_weight_identity_dx():
    x, W, A, B, s = _linear_case()
    dy = _rand(x.shape[0], W.shape[0])
    dx, _, _ = oracle.lora_linear_grad(x, W, A, B, s, dy)
    np.testing.assert_allclose(dx, dy @ (W + s * B @ A), rtol=1e-12, atol=1e-12)


def test_adapter_grads_vanish_on_zero_factor():
    x, W, A, B, s = _linear_case()
    dy = _rand(x.shape[0], W.shape[0])
    _, dA, _ = oracle.lora_linear_grad(x, W, A, np.zeros_like(B), s, dy)
    assert np.all(dA == 0.0)
    _, _, dB = oracle.lora_linear_grad(x, W, np.zeros_like(A), B, s, dy)
    assert np.all(dB == 0.0)


def test_linear_in_s():
    x, W, A, B, s = _linear_case()
    dy = _rand(x.shape[0], W.shape[0])
    y0 = oracle.lora_linear(x, W, A, B, 0.0)
    y1 = oracle.lora_linear(x, W, A, B, s)
    y2 = oracle.lora_linear(x, W, A, B, 2 * s)
    np.testing.assert_allclose(y2 - y0, 2 * (y1 - y0), rtol=1e-12, atol=1e-12)
    g1 = oracle.lora_linear_grad(x, W, A, B, s, dy)
    g2 = oracle.lora_linear_grad(x, W, A, B, 2 * s, dy)
    for a, b in zip(g1[1:], g2[1:]):
        np.testing.assert_allclose(b, 2 * a, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- finite differences

def _mlp_params(M=4, h=8, i=12, r=2, seed=7):
    rng = np.random.default_rng(seed)
    n = lambda *s: rng.standard_normal(s)  # noqa: E731
    p = {"x": n(M, h), "Wg": n(i, h) / 3, "Ag": n(r, h) / 3, "Bg": n(i, r) / 2,
         "Wu": n(i, h) / 3, "Au": n(r, h) / 3, "Bu": n(i, r) / 2,
         "Wd": n(h, i) / 3, "Ad": n(r, i) / 3, "Bd": n(h, r) / 2}
    return p, n(M, h)


def _mlp_loss(p, dy, s, kind, mod=olora):
    y = mod.mlp_forward(p["x"], p["Wg"], p["Ag"], p["Bg"], p["Wu"], p["Au"], p["Bu"],
                        p["Wd"], p["Ad"], p["Bd"], s, kind)["y"]
    return float(np.sum(dy * y))


MLP_GRAD_KEYS = {"x": "dx", "Ag": "dA_gate", "Bg": "dB_gate", "Au": "dA_up",
                 "Bu": "dB_up", "Ad": "dA_down", "Bd": "dB_down"}


def mlp_fd_error(kind, s=1.5, mod=olora, eps=1e-6):
    """Largest relative error of the oracle's MLP gradients against central
    differences of <dy, y>, over every element of x, A and B."""
    p, dy = _mlp_params()
    grads = mod.mlp_backward(p["x"], p["Wg"], p["Ag"], p["Bg"], p["Wu"], p["Au"], p["Bu"],
                             p["Wd"], p["Ad"], p["Bd"], s, kind, dy)
    worst = 0.0
    for pk, gk in MLP_GRAD_KEYS.items():
        fd = np.zeros_like(p[pk])
        for idx in np.ndindex(p[pk].shape):
            q = {k: v.copy() for k, v in p.items()}
            q[pk][idx] += eps
            lp = _mlp_loss(q, dy, s, kind, mod)
            q[pk][idx] -= 2 * eps
            lm = _mlp_loss(q, dy, s, kind, mod)
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(grads[gk] - fd)) / max(np.max(np.abs(fd)), 1e-30)
        worst = max(worst, err)
    return worst


@pytest.mark.parametrize("kind", oracle.ACTS)
def test_mlp_backward_matches_finite_differences(kind):
    assert mlp_fd_error(kind) < 1e-6


def _qkvo_params(M=4, h=8, nq=8, nkv=4, r=2, seed=11):
    rng = np.random.default_rng(seed)
    n = lambda *s: rng.standard_normal(s)  # noqa: E731
    lin = lambda fin, fout: [n(fout, fin) / 3, n(r, fin) / 3, n(fout, r) / 2]  # noqa: E731
    p = {"x": n(M, h), "o_in": n(M, nq), "q": lin(h, nq), "k": lin(h, nkv), "v": lin(h, nkv),
         "o": lin(nq, h)}
    dys = {"q": n(M, nq), "k": n(M, nkv), "v": n(M, nkv), "o": n(M, h)}
    return p, dys


def _qkvo_loss(p, dys, s, rope=None, mod=olora):
    out = mod.qkvo_forward(p["x"], p["q"], p["k"], p["v"], p["o_in"], p["o"], s, rope=rope)
    return float(sum(np.sum(dys[k] * out[k]) for k in ("q", "k", "v", "o")))


def qkvo_fd_error(rope=None, mod=olora, s=2.0, eps=1e-6, **shape):
    """Largest error of the Q/K/V + O backward against central differences of
    <dy, out>, relative to the largest difference quotient of each tensor."""
    p, dys = _qkvo_params(**shape)
    g = mod.qkvo_backward(p["x"], p["q"], p["k"], p["v"], p["o_in"], p["o"], s,
                          dys["q"], dys["k"], dys["v"], dys["o"], rope=rope)

    def fd_of(getter):
        base = getter(p)
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            orig = base[idx]
            base[idx] = orig + eps
            lp = _qkvo_loss(p, dys, s, rope, mod)
            base[idx] = orig - eps
            lm = _qkvo_loss(p, dys, s, rope, mod)
            base[idx] = orig
            fd[idx] = (lp - lm) / (2 * eps)
        return fd

    checks = [(lambda q: q["x"], g["dx"]), (lambda q: q["o_in"], g["do_in"])]
    for name in ("q", "k", "v", "o"):
        checks.append((lambda q, name=name: q[name][1], g[f"dA_{name}"]))
        checks.append((lambda q, name=name: q[name][2], g[f"dB_{name}"]))
    worst = 0.0
    for getter, got in checks:
        fd = fd_of(getter)
        worst = max(worst, float(np.max(np.abs(got - fd)) / np.max(np.abs(fd))))
    return worst


def test_qkvo_backward_matches_finite_differences():
    assert qkvo_fd_error() <= 1e-6


# ---------------------------------------------------------------- B = 0: the base MLP

def base_mlp_error(kind, mod=olora):
    """With B = 0 the block is the plain gated MLP.  Returns the largest relative
    difference of y and dx from torch float64 matmul + silu / gelu(tanh) with torch
    autograd, and whether every dA is exactly zero."""
    p, dy = _mlp_params(M=6, h=16, i=24, r=3)
    for k in ("Bg", "Bu", "Bd"):
        p[k] = np.zeros_like(p[k])
    s = 2.0
    args = (p["x"], p["Wg"], p["Ag"], p["Bg"], p["Wu"], p["Au"], p["Bu"],
            p["Wd"], p["Ad"], p["Bd"], s, kind)
    f = mod.mlp_forward(*args)
    t = {k: torch.from_numpy(v) for k, v in p.items()}
    x = t["x"].clone().requires_grad_(True)
    gate = x @ t["Wg"].T
    if kind == "swiglu":
        a = F.silu(gate)
    else:
        a = F.gelu(gate, approximate="tanh" if kind == "geglu_tanh" else "none")
    y = (a * (x @ t["Wu"].T)) @ t["Wd"].T
    (y * torch.from_numpy(dy)).sum().backward()
    b = mod.mlp_backward(*args, dy)
    rel = lambda a_, b_: np.max(np.abs(a_ - b_)) / np.max(np.abs(b_))  # noqa: E731
    err = max(rel(f["y"], y.detach().numpy()), rel(b["dx"], x.grad.numpy()))
    zero_da = all(np.all(b[k] == 0.0) for k in ("dA_gate", "dA_up", "dA_down"))
    return err, zero_da


@pytest.mark.parametrize("kind", oracle.ACTS)
def test_zero_b_reduces_to_library_base_mlp(kind):
    err, zero_da = base_mlp_error(kind)
    assert err < 1e-12
    assert zero_da


def test_merged_weight_identity_mlp():
    """The adapted MLP equals the base MLP on merged weights W + s B A."""
    p, dy = _mlp_params(M=5, h=8, i=12, r=2)
    s, kind = 1.25, "swiglu"
    f = oracle.mlp_forward(p["x"], p["Wg"], p["Ag"], p["Bg"], p["Wu"], p["Au"], p["Bu"],
                           p["Wd"], p["Ad"], p["Bd"], s, kind)
    z = lambda a: np.zeros_like(a)  # noqa: E731
    m = oracle.mlp_forward(p["x"], p["Wg"] + s * p["Bg"] @ p["Ag"], z(p["Ag"]), z(p["Bg"]),
                           p["Wu"] + s * p["Bu"] @ p["Au"], z(p["Au"]), z(p["Bu"]),
                           p["Wd"] + s * p["Bd"] @ p["Ad"], z(p["Ad"]), z(p["Bd"]), s, kind)
    np.testing.assert_allclose(f["y"], m["y"], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- mutation tests

class _Mutant:
    """A copy of the oracle module's namespace with one function replaced."""

    def __init__(self, **repl):
        self.__dict__.update({k: getattr(olora, k) for k in dir(olora) if not k.startswith("__")})
        self.__dict__.update(repl)
        # rebind the functions that call the replaced ones
        for name in ("mlp_forward", "mlp_backward", "qkvo_forward", "qkvo_backward", "apply_rope",
                     "apply_rope_transpose"):
            if name not in repl:
                self.__dict__[name] = _rebind(getattr(olora, name), self)


def _rebind(fn, ns):
    import types
    g = dict(fn.__globals__)
    g.update(ns.__dict__)
    return types.FunctionType(fn.__code__, g, fn.__name__, fn.__defaults__)


def _grad_half_db(x, W, A, B, s, dy):
    dx, dA, dB = olora.lora_linear_grad(x, W, A, B, s, dy)
    return dx, dA, 0.5 * dB


def _act_prime_sign(g, kind):
    sg = olora.sigmoid(g)
    if kind == "swiglu":
        return sg * (1.0 - g * (1.0 - sg))
    return olora.act_prime(g, kind)


def _act_prime_dropped_term(g, kind):
    if kind == "geglu_tanh":
        t = np.tanh(np.sqrt(2 / np.pi) * (g + 0.044715 * g ** 3))
        return 0.5 * (1.0 + t)
    return olora.act_prime(g, kind)


def _grad_missing_s(x, W, A, B, s, dy):
    dx, dA, dB = olora.lora_linear_grad(x, W, A, B, s, dy)
    return dx, dA / s, dB


@pytest.mark.parametrize("mutant,kind", [
    (dict(act_prime=_act_prime_sign), "swiglu"),
    (dict(act_prime=_act_prime_dropped_term), "geglu_tanh"),
    (dict(lora_linear_grad=_grad_half_db), "swiglu"),
    (dict(lora_linear_grad=_grad_missing_s), "swiglu"),
])
def test_planted_mistakes_are_caught(mutant, kind):
    m = _Mutant(**mutant)
    assert mlp_fd_error(kind, mod=m) > 1e-3


def _forward_swapped_gate_up(x, Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, s, kind):
    return olora.mlp_forward(x, Wu, Au, Bu, Wg, Ag, Bg, Wd, Ad, Bd, s, kind)


def _act_erf_for_tanh(g, kind):
    if kind == "geglu_tanh":
        from scipy.special import erf
        return 0.5 * g * (1.0 + erf(g / np.sqrt(2.0)))
    return olora.act(g, kind)


@pytest.mark.parametrize("mutant,kind", [
    (dict(mlp_forward=_forward_swapped_gate_up), "swiglu"),
    (dict(act=_act_erf_for_tanh), "geglu_tanh"),
])
def test_planted_forward_mistakes_are_caught(mutant, kind):
    m = _Mutant(**mutant)
    err, _ = base_mlp_error(kind, mod=m)
    assert err > 1e-4


def test_frozen_bias_adds_a_row_vector_and_leaves_grads():
    """A frozen Q/K/V bias shifts each output row by exactly the bias and changes no
    gradient."""
    p, dys = _qkvo_params()
    rng = np.random.default_rng(5)
    bias = (rng.standard_normal(8), rng.standard_normal(4), rng.standard_normal(4))
    a = oracle.qkvo_forward(p["x"], p["q"], p["k"], p["v"], p["o_in"], p["o"], 2.0)
    b = oracle.qkvo_forward(p["x"], p["q"], p["k"], p["v"], p["o_in"], p["o"], 2.0, bias=bias)
    for j, n in enumerate(("q", "k", "v")):
        np.testing.assert_allclose(b[n] - a[n], np.broadcast_to(bias[j], a[n].shape), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(a["o"], b["o"])


def test_per_example_grads_sum_to_the_batch_gradient():
    """Per-example adapter gradients add up to the full-batch gradient (the loss is a
    sum over examples), and each squared norm is the sum over the six adapters."""
    p, dy = _mlp_params(M=6, h=8, i=12, r=2)
    args = (p["x"], p["Wg"], p["Ag"], p["Bg"], p["Wu"], p["Au"], p["Bu"], p["Wd"], p["Ad"], p["Bd"], 1.5,
            "swiglu")
    full = oracle.mlp_backward(*args, dy)
    per = oracle.mlp_backward_per_example(*args, dy, 3)
    for k in ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"):
        assert per[k].shape == (3,) + full[k].shape
        np.testing.assert_allclose(per[k].sum(axis=0), full[k], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(per["dx"], full["dx"], rtol=1e-12, atol=1e-12)
    e1 = sum(float(np.sum(per[k][1] ** 2)) for k in ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"))
    assert math.isclose(per["sq_norms"][1], e1, rel_tol=1e-12)


@pytest.mark.parametrize("kind", ["swiglu", "geglu_tanh", "geglu_erf"])
def test_tokens_are_independent_rows(kind):
    """The block acts on each token row on its own and the adapter gradients are sums
    over tokens: permuting the tokens (x and dy together) permutes y and dx the same
    way and leaves every dA, dB unchanged.  A token index mixed into another operand
    (a transposed x, dy or saved tensor) breaks this."""
    p, dy = _mlp_params(M=7, h=8, i=12, r=3, seed=19)
    perm = np.random.default_rng(3).permutation(7)
    args = lambda x: (x, p["Wg"], p["Ag"], p["Bg"], p["Wu"], p["Au"], p["Bu"],  # noqa: E731
                      p["Wd"], p["Ad"], p["Bd"], 1.25, kind)
    y = oracle.mlp_forward(*args(p["x"]))["y"]
    yp = oracle.mlp_forward(*args(p["x"][perm]))["y"]
    np.testing.assert_allclose(yp, y[perm], rtol=1e-13, atol=1e-13)
    g = oracle.mlp_backward(*args(p["x"]), dy)
    gp = oracle.mlp_backward(*args(p["x"][perm]), dy[perm])
    np.testing.assert_allclose(gp["dx"], g["dx"][perm], rtol=1e-12, atol=1e-12)
    for k in ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"):
        np.testing.assert_allclose(gp[k], g[k], rtol=1e-12, atol=1e-12)


def test_per_example_grads_follow_their_examples():
    """Reordering whole examples (blocks of seq consecutive tokens) reorders the
    per-example gradients and squared norms the same way."""
    p, dy = _mlp_params(M=8, h=8, i=12, r=2, seed=23)
    blocks = np.array([2, 0, 3, 1])
    rows = (blocks[:, None] * 2 + np.arange(2)[None, :]).reshape(-1)
    args = lambda x: (x, p["Wg"], p["Ag"], p["Bg"], p["Wu"], p["Au"], p["Bu"],  # noqa: E731
                      p["Wd"], p["Ad"], p["Bd"], 0.75, "geglu_tanh")
    a = oracle.mlp_backward_per_example(*args(p["x"]), dy, 4)
    b = oracle.mlp_backward_per_example(*args(p["x"][rows]), dy[rows], 4)
    for k in ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"):
        np.testing.assert_allclose(b[k], a[k][blocks], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b["sq_norms"], a["sq_norms"][blocks], rtol=1e-12)


# ---------------------------------------------------------------- RoPE

def _rope(M=4, n_pos=40, head_dim=4, seed=2, base=10000.0):
    cos, sin = oracle.rope_tables(n_pos, head_dim, base)
    pos = np.random.default_rng(seed).integers(0, n_pos, M)
    return {"cos": cos, "sin": sin, "pos": pos, "head_dim": head_dim}


def test_rope_table_closed_values():
    """Frequency 0 turns 1 rad per position; with d = 4 and base 10000 the other
    frequency is 10000^(-1/2) = 0.01 rad; consecutive frequencies fall by the factor
    base^(-2/d) (RoFormer's geometric frequencies)."""
    cos, sin = oracle.rope_tables(7, 4)
    for p in range(7):
        assert math.isclose(cos[p, 0], math.cos(p), abs_tol=1e-15)
        assert math.isclose(sin[p, 0], math.sin(p), abs_tol=1e-15)
        assert math.isclose(cos[p, 1], math.cos(0.01 * p), abs_tol=1e-15)
        assert math.isclose(sin[p, 1], math.sin(0.01 * p), abs_tol=1e-15)
    cos, sin = oracle.rope_tables(2, 128, base=500000.0)
    ang = np.arctan2(sin[1], cos[1])                   # position 1: every angle below pi
    np.testing.assert_allclose(ang[1:] / ang[:-1], 500000.0 ** (-2.0 / 128), rtol=1e-12)


def rope_complex_error(mod=olora, d=8):
    """apply_rope against RoFormer's complex form: the pair (y_i, y_{i+d/2}) is the
    number y_i + 1j y_{i+d/2}, multiplied by exp(1j p theta_i), theta_i =
    10000^(-2(i-1)/d) for i = 1 .. d/2."""
    rng = np.random.default_rng(3)
    M, heads, n_pos = 6, 3, 50
    y = rng.standard_normal((M, heads * d))
    pos = rng.integers(0, n_pos, M)
    cos, sin = oracle.rope_tables(n_pos, d)
    got = mod.apply_rope(y, cos, sin, pos, d).reshape(M, heads, d)
    yh = y.reshape(M, heads, d)
    z = yh[:, :, :d // 2] + 1j * yh[:, :, d // 2:]
    theta = 10000.0 ** (-2.0 * (np.arange(1, d // 2 + 1) - 1) / d)
    w = z * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    return max(float(np.max(np.abs(got[:, :, :d // 2] - w.real))),
               float(np.max(np.abs(got[:, :, d // 2:] - w.imag))))


def test_rope_is_the_complex_rotation():
    assert rope_complex_error() < 1e-12


def test_rope_keeps_norms_and_depends_on_relative_position():
    """A rotation keeps each head's norm, position 0 is the identity, and the dot
    product of a rotated q head with a rotated k head depends only on the distance
    between their positions (RoFormer's relative-position property)."""
    d = 16
    cos, sin = oracle.rope_tables(64, d)
    rng = np.random.default_rng(9)
    q, k = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    y = rng.standard_normal((5, 3 * d))
    pos = np.array([0, 1, 7, 30, 63])
    r = oracle.apply_rope(y, cos, sin, pos, d)
    np.testing.assert_allclose(np.linalg.norm(r.reshape(5, 3, d), axis=2),
                               np.linalg.norm(y.reshape(5, 3, d), axis=2), rtol=1e-13)
    np.testing.assert_array_equal(r[0], y[0])

    def dot(pq, pk):
        return float(np.sum(oracle.apply_rope(q, cos, sin, [pq], d) * oracle.apply_rope(k, cos, sin, [pk], d)))

    assert math.isclose(dot(10, 3), dot(20, 13), rel_tol=1e-12)
    assert math.isclose(dot(40, 40), float(np.sum(q * k)), rel_tol=1e-12)
    assert not math.isclose(dot(10, 3), dot(10, 4), rel_tol=1e-3)


def test_rope_transpose_is_adjoint_and_inverse():
    rp = _rope(M=5, head_dim=8)
    rng = np.random.default_rng(4)
    y, z = rng.standard_normal((5, 16)), rng.standard_normal((5, 16))
    args = (rp["cos"], rp["sin"], rp["pos"], 8)
    ry = oracle.apply_rope(y, *args)
    assert math.isclose(float(np.sum(ry * z)), float(np.sum(y * oracle.apply_rope_transpose(z, *args))),
                        rel_tol=1e-12)
    np.testing.assert_allclose(oracle.apply_rope_transpose(ry, *args), y, atol=1e-13)


def test_qkvo_rope_backward_matches_finite_differences():
    """Q/K/V + O with RoPE on q and k (two heads of q, one of k: GQA)."""
    assert qkvo_fd_error(rope=_rope(head_dim=4)) <= 1e-6


def test_rope_leaves_v_and_o_alone():
    p, _ = _qkvo_params()
    a = oracle.qkvo_forward(p["x"], p["q"], p["k"], p["v"], p["o_in"], p["o"], 2.0)
    b = oracle.qkvo_forward(p["x"], p["q"], p["k"], p["v"], p["o_in"], p["o"], 2.0, rope=_rope())
    np.testing.assert_array_equal(a["v"], b["v"])
    np.testing.assert_array_equal(a["o"], b["o"])
    assert np.max(np.abs(a["q"] - b["q"])) > 1e-3


def _rope_no_negation(dy, cos, sin, pos, head_dim):
    return olora.apply_rope(dy, cos, sin, pos, head_dim)


def _rope_interleaved(y, cos, sin, pos, head_dim):
    M, n = y.shape
    yh = y.reshape(M, n // head_dim, head_dim // 2, 2)
    a, b = yh[..., 0], yh[..., 1]
    c, s_ = cos[pos][:, None, :], sin[pos][:, None, :]
    return np.stack([a * c - b * s_, b * c + a * s_], axis=-1).reshape(M, n)


def _rope_swapped_tables(y, cos, sin, pos, head_dim):
    return olora._rotate(y, sin, cos, pos, head_dim, 1.0)


def test_planted_rope_mistakes_are_caught():
    assert qkvo_fd_error(rope=_rope(), mod=_Mutant(apply_rope_transpose=_rope_no_negation)) > 1e-3
    assert rope_complex_error(mod=_Mutant(apply_rope=_rope_interleaved)) > 1e-3
    assert rope_complex_error(mod=_Mutant(apply_rope=_rope_swapped_tables)) > 1e-3
