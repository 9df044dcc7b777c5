"""Plain float64 definition of the LoRA block projections, forward and backward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py``; never by the CUDA library, which shares no code
with it.

Sources (web pages; each function names the passage it follows):

* "Model Patches and Kernels" (opake user guide), section "Fused LoRA operations",
  kernel table: the single LoRA linear ``x @ W.T + x @ A @ B * s`` (row
  ``opake_lora_w``), three projections sharing one input (row ``opake_lora_qkv``) and
  gate + up + activation + down in one call (row ``opake_lora_mlp``); MLP fusion
  is bias-free.
* same page, section "Triton kernels", "Activation functions" table:
  SwiGLU ``silu(gate) * up``, GeGLU Exact ``gelu(gate) * up`` (erf-based) and GeGLU
  Approx ``gelu_tanh(gate) * up``.
* same page, section "Fused linear cross-entropy", "Key design decisions": a frozen
  weight gets no gradient.  Base weights W are frozen here, so backward returns
  dX and the adapter gradients dA, dB only.
* same page, section "Rotary position embeddings (RoPE)": rotary embeddings applied
  to q and k together, with different head counts for q and k (GQA), following the
  RoFormer position encoding.
* "monkeypatch.lora_kernels" (axolotl API reference), ``apply_lora_kernel_patches``
  note: adapters have no dropout and no bias; ``original_apply_qkv`` returns
  (query, key, value) from one hidden-state input; ``original_apply_o`` is the
  output projection.

Readings where the pages leave a step open (plainest reading, stated once here):

1. ``s`` is alpha / r.
2. Layout is the PEFT one: A is [r, in], B is [out, r], so the page's
   ``x @ A @ B`` is ``x A^T B^T`` here.
3. In the gated MLP the ``gate`` projection is activated and ``up`` is linear.
4. ``gelu_tanh(g) = 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))``, the
   tanh approximation of GELU with its published constants.
5. Backward is the chain rule of the forward above, with no weight gradient, and
   dA/dB are the full gradients of the scalar <dY, Y> (no accumulation into old
   values).
6. Nothing is rounded: inputs are the bf16 values widened to float64.
7. RoPE: head j of q and k (head_dim d) is rotated pair by pair, the pair being
   features (i, i + d/2) of the head (the half-split pairing of the HF LLaMA family
   the page lists as patched; RoFormer's own pairing (2i, 2i+1) differs only by a
   fixed permutation of a head's features).  The angle of pair i at position p is
   p * base^(-2i/d), base 10000 unless stated.  It is applied after the frozen bias,
   to q and k only, and the position of each token is an input.

Every function is pinned by tests that do not restate its formula: the LoRA
merged-weight identity, the B = 0 reduction to a base MLP built from library
routines, central finite differences of <dY, Y>, closed-form activation
derivatives against finite differences, and linearity in s; RoPE by RoFormer's
complex form of the rotation, closed table values, norm preservation, the
relative-position property of rotated dot products, and finite differences.
"""

from __future__ import annotations

import numpy as np

ACTS = ("swiglu", "geglu_tanh", "geglu_erf")
_SQRT_2_OVER_PI = np.sqrt(2.0 / np.pi)
_GELU_C = 0.044715


def _mm(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """float64 matrix product (library primitive)."""
    return np.matmul(a, b)


# --------------------------------------------------------------------------------
# Activations -- "Model Patches and Kernels", "Activation functions" table.
# --------------------------------------------------------------------------------

def sigmoid(g: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g * sigmoid(g)  (SwiGLU row of the activation table)."""
    return g * sigmoid(g)


def gelu_tanh(g: np.ndarray) -> np.ndarray:
    """GELU, tanh approximation (GeGLU Approx row of the activation table)."""
    return 0.5 * g * (1.0 + np.tanh(_SQRT_2_OVER_PI * (g + _GELU_C * g ** 3)))


def gelu_erf(g: np.ndarray) -> np.ndarray:
    """Exact GELU, g * Phi(g) with Phi the standard normal CDF (GeGLU Exact row)."""
    from scipy.special import erf
    return 0.5 * g * (1.0 + erf(g / np.sqrt(2.0)))


def act(g: np.ndarray, kind: str) -> np.ndarray:
    if kind == "swiglu":
        return silu(g)
    if kind == "geglu_tanh":
        return gelu_tanh(g)
    if kind == "geglu_erf":
        return gelu_erf(g)
    raise ValueError(f"unknown activation {kind!r}")


def act_prime(g: np.ndarray, kind: str) -> np.ndarray:
    """d act / d g in closed form.

    silu'(g) = sigma(g) (1 + g (1 - sigma(g))).
    gelu_tanh'(g) = 0.5 (1 + t) + 0.5 g (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 g^2),
    t = tanh(sqrt(2/pi) (g + 0.044715 g^3)).
    gelu_erf'(g) = Phi(g) + g phi(g), phi the standard normal density.
    """
    if kind == "swiglu":
        sg = sigmoid(g)
        return sg * (1.0 + g * (1.0 - sg))
    if kind == "geglu_tanh":
        t = np.tanh(_SQRT_2_OVER_PI * (g + _GELU_C * g ** 3))
        return 0.5 * (1.0 + t) + 0.5 * g * (1.0 - t * t) * _SQRT_2_OVER_PI * (
            1.0 + 3.0 * _GELU_C * g * g)
    if kind == "geglu_erf":
        from scipy.special import erf
        return 0.5 * (1.0 + erf(g / np.sqrt(2.0))) + g * np.exp(-0.5 * g * g) / np.sqrt(2.0 * np.pi)
    raise ValueError(f"unknown activation {kind!r}")


# --------------------------------------------------------------------------------
# One LoRA linear -- "Model Patches and Kernels", "Fused LoRA operations",
# row opake_lora_w:  y = x W^T + s (x A^T) B^T.
# --------------------------------------------------------------------------------

def linear_t(x: np.ndarray, A: np.ndarray) -> np.ndarray:
    """The rank-r projection T = x A^T, [M, r]."""
    return _mm(x, A.T)


def lora_linear(x, W, A, B, s):
    """y = x W^T + s (x A^T) B^T for x [M, in], W [out, in], A [r, in], B [out, r]."""
    return _mm(x, W.T) + s * _mm(linear_t(x, A), B.T)


def lora_linear_grad(x, W, A, B, s, dy):
    """Gradients of <dy, lora_linear(x, W, A, B, s)> with W frozen.

    U = dy B [M, r];  dx = dy W + s U A;  dA = s U^T x [r, in];
    dB = s dy^T (x A^T) [out, r].
    """
    U = _mm(dy, B)
    dx = _mm(dy, W) + s * _mm(U, A)
    dA = s * _mm(U.T, x)
    dB = s * _mm(dy.T, linear_t(x, A))
    return dx, dA, dB


# --------------------------------------------------------------------------------
# Gated MLP -- row opake_lora_mlp: gate and up LoRA linears on x, activation of the
# gate times up, then the down LoRA linear.
# --------------------------------------------------------------------------------

def mlp_forward(x, Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, s, kind):
    """Returns dict(g, u, h, y) for the LoRA gated MLP."""
    g = lora_linear(x, Wg, Ag, Bg, s)
    u = lora_linear(x, Wu, Au, Bu, s)
    h = act(g, kind) * u
    y = lora_linear(h, Wd, Ad, Bd, s)
    return {"g": g, "u": u, "h": h, "y": y}


def mlp_backward(x, Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, s, kind, dy):
    """Gradients of <dy, y> for the LoRA gated MLP (frozen W): dx and dA/dB of
    gate, up and down.  The forward is recomputed in float64."""
    f = mlp_forward(x, Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, s, kind)
    g, u, h = f["g"], f["u"], f["h"]
    dh, dAd, dBd = lora_linear_grad(h, Wd, Ad, Bd, s, dy)
    dg = dh * u * act_prime(g, kind)
    du = dh * act(g, kind)
    dxg, dAg, dBg = lora_linear_grad(x, Wg, Ag, Bg, s, dg)
    dxu, dAu, dBu = lora_linear_grad(x, Wu, Au, Bu, s, du)
    return {"dx": dxg + dxu, "dA_gate": dAg, "dB_gate": dBg, "dA_up": dAu,
            "dB_up": dBu, "dA_down": dAd, "dB_down": dBd, "dg": dg, "du": du, "dh": dh}


def mlp_backward_per_example(x, Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, s, kind, dy, n_examples):
    """Per-example adapter gradients for DP-SGD ("Model Patches and Kernels": per-example
    gradients by vmap(grad) over the examples of a batch).  The block acts on each
    token independently, so example e's gradient is the backward over its own
    tokens [e seq, (e+1) seq) alone.  Returns dict(dx, dA_* [n, r, in], dB_* [n, out, r],
    sq_norms [n]); sq_norms[e] = sum of squares of example e's six adapter gradients."""
    M = x.shape[0]
    seq = M // n_examples
    keys = ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down")
    res = {k: [] for k in keys}
    dx = []
    for e in range(n_examples):
        sl = slice(e * seq, (e + 1) * seq)
        b = mlp_backward(x[sl], Wg, Ag, Bg, Wu, Au, Bu, Wd, Ad, Bd, s, kind, dy[sl])
        dx.append(b["dx"])
        for k in keys:
            res[k].append(b[k])
    out = {k: np.stack(v) for k, v in res.items()}
    out["dx"] = np.concatenate(dx, axis=0)
    out["sq_norms"] = sum(np.sum(out[k] ** 2, axis=tuple(range(1, out[k].ndim))) for k in keys)
    return out


# --------------------------------------------------------------------------------
# Attention projections -- row opake_lora_qkv (q, k, v share the input x) and the
# output projection (original_apply_qkv / original_apply_o in the axolotl API).
# The attention between them is not part of this path; o_in is its output.
# --------------------------------------------------------------------------------

# --------------------------------------------------------------------------------
# RoPE -- "Model Patches and Kernels", "Rotary position embeddings (RoPE)": rotary
# embeddings of q and k (RoFormer), GQA head counts.
# --------------------------------------------------------------------------------

def rope_tables(n_pos, head_dim, base=10000.0):
    """cos and sin of the rotation angles, [n_pos, head_dim/2]: entry (p, i) is the
    angle p * base^(-2i/head_dim) (RoFormer's frequencies)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / head_dim)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)


def _rotate(y, cos, sin, pos, head_dim, sign):
    M, n = y.shape
    half = head_dim // 2
    yh = y.reshape(M, n // head_dim, head_dim)
    a, b = yh[:, :, :half], yh[:, :, half:]
    c = cos[pos][:, None, :]
    s_ = sign * sin[pos][:, None, :]
    return np.concatenate([a * c - b * s_, b * c + a * s_], axis=2).reshape(M, n)


def apply_rope(y, cos, sin, pos, head_dim):
    """Rotates every head of y [M, heads * head_dim]: in token m's head, the pair
    (y_i, y_{i + d/2}) turns by the angle of row pos[m], column i of the tables."""
    return _rotate(y, cos, sin, pos, head_dim, 1.0)


def apply_rope_transpose(dy, cos, sin, pos, head_dim):
    """The transpose of apply_rope (each pair turned by minus the angle): the gradient
    with respect to the unrotated input, given the gradient dy of the rotated one."""
    return _rotate(dy, cos, sin, pos, head_dim, -1.0)


def qkvo_forward(x, lin_q, lin_k, lin_v, o_in, lin_o, s, bias=None, rope=None):
    """lin_p = (W, A, B).  Returns dict(q, k, v, o).

    bias: optional frozen base-layer biases (b_q, b_k, b_v) added to q, k, v
    ("Fused LoRA operations": QKV fusion supports optional frozen base-layer biases).
    A frozen bias gets no gradient and does not change the backward.
    rope: optional dict(cos, sin, pos, head_dim): q and k (bias included) are then
    rotated by apply_rope."""
    out = {}
    for j, (name, lin) in enumerate((("q", lin_q), ("k", lin_k), ("v", lin_v))):
        out[name] = lora_linear(x, *lin, s)
        if bias is not None:
            out[name] = out[name] + bias[j][None, :]
        if rope is not None and name in ("q", "k"):
            out[name] = apply_rope(out[name], rope["cos"], rope["sin"], rope["pos"], rope["head_dim"])
    out["o"] = lora_linear(o_in, *lin_o, s)
    return out


def qkvo_backward(x, lin_q, lin_k, lin_v, o_in, lin_o, s, dy_q, dy_k, dy_v, dy_o, rope=None):
    """Gradients of <dy_q, q> + <dy_k, k> + <dy_v, v> + <dy_o, o>: dx (sum over the
    three projections), d o_in, and dA/dB of q, k, v and o.  With rope, dy_q and dy_k
    are gradients of the rotated q and k and pass through apply_rope_transpose first."""
    if rope is not None:
        dy_q = apply_rope_transpose(dy_q, rope["cos"], rope["sin"], rope["pos"], rope["head_dim"])
        dy_k = apply_rope_transpose(dy_k, rope["cos"], rope["sin"], rope["pos"], rope["head_dim"])
    res = {}
    dx = None
    for name, lin, d in (("q", lin_q, dy_q), ("k", lin_k, dy_k), ("v", lin_v, dy_v)):
        dxp, dA, dB = lora_linear_grad(x, *lin, s, d)
        dx = dxp if dx is None else dx + dxp
        res[f"dA_{name}"], res[f"dB_{name}"] = dA, dB
    res["dx"] = dx
    res["do_in"], res["dA_o"], res["dB_o"] = lora_linear_grad(o_in, *lin_o, s, dy_o)
    return res
