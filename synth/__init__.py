"""Seeded synthetic inputs for the LoRA block projections.

This module is shared by the CPU oracle, the parity tests and the benchmark.  It
holds the workload shapes and the value distributions, and nothing of the method's
arithmetic: no projection, activation or gradient is computed here.

Generator (counter based, so any element can be drawn independently):

* ``splitmix64`` finaliser on a 64-bit counter.  Stream ``sid`` of seed ``seed``
  starts at ``base = mix(seed * 0x9E3779B97F4A7C15 + sid + 1)``; draw ``k`` of the
  stream is ``mix(base + (k + 1) * 0x9E3779B97F4A7C15)`` (wrapping uint64 arithmetic).
* uniform in [0, 1):   ``(bits >> 11) * 2**-53``;  uniform in (0, 1]: add one ulp.
* normal element ``n`` of a stream: Box-Muller on draws ``2n`` (u1 in (0, 1]) and
  ``2n + 1`` (u2 in [0, 1)): ``sqrt(-2 ln u1) * cos(2 pi u2)``.
* uniform element ``n`` on (-a, a): ``a * (2 u - 1)`` with u from draw ``n``.
* every value is made in float64 and rounded once, to nearest-even, to bfloat16.
  Tensors come back as torch bfloat16 (on the CPU, or on a CUDA device for
  workloads whose values need not match the oracle bit for bit);
  :func:`bf16_to_f64` widens them to float64 numpy arrays.

The arithmetic is int64 with wrapping multiplication, so the same code runs with
torch on the CPU and on the GPU.

Distributions (variance is the second argument of N): x ~ N(0, 1);
W ~ N(0, 1/fan_in); A ~ U(-1/sqrt(fan_in), 1/sqrt(fan_in)); B ~ N(0, 0.02);
upstream gradients ~ N(0, 1).  The attention output fed to the O projection is an
independent N(0, 1) tensor.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

__all__ = [
    "MlpConfig", "QkvoConfig", "MLP_CONFIGS", "QKVO_CONFIGS",
    "f64_to_bf16", "bf16_to_f64", "normal_stream", "uniform_stream", "mix64",
    "stream_base", "draws",
    "make_mlp_inputs", "make_qkvo_inputs", "MLP_TENSORS", "QKVO_TENSORS",
]

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1
_CHUNK = 1 << 24


def _s64(v: int) -> int:
    """A uint64 constant as the int64 with the same bits (torch has no wrapping uint64)."""
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def _srl(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    """splitmix64 finaliser on int64 bit patterns (multiplication wraps mod 2^64)."""
    z = z ^ _srl(z, 30)
    z = z * _s64(_M1)
    z = z ^ _srl(z, 27)
    z = z * _s64(_M2)
    return z ^ _srl(z, 31)


def mix64(v: int) -> int:
    """Scalar splitmix64 finaliser on a Python int (reference form, exact)."""
    v &= _MASK64
    v = ((v ^ (v >> 30)) * _M1) & _MASK64
    v = ((v ^ (v >> 27)) * _M2) & _MASK64
    return v ^ (v >> 31)


def stream_base(seed: int, sid: int) -> int:
    return mix64(seed * _GOLDEN + sid + 1)


def draws(base: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """Draws start .. start+count-1 (int64 bit patterns) of the stream with this base."""
    k = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    return _mix(k * _s64(_GOLDEN) + _s64(base))


def _u01_open0(bits: torch.Tensor) -> torch.Tensor:
    return (_srl(bits, 11).to(torch.float64) + 1.0) * 2.0 ** -53


def _u01(bits: torch.Tensor) -> torch.Tensor:
    return _srl(bits, 11).to(torch.float64) * 2.0 ** -53


def normal_stream(seed: int, sid: int, n: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    """n float64 normals N(0, std^2) from stream ``sid`` of ``seed``."""
    base = stream_base(seed, sid)
    out = torch.empty(n, dtype=torch.float64, device=device)
    for c0 in range(0, n, _CHUNK):
        c = min(_CHUNK, n - c0)
        d = draws(base, 2 * c0, 2 * c, device).view(c, 2)
        u1 = _u01_open0(d[:, 0])
        u2 = _u01(d[:, 1])
        out[c0:c0 + c] = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
    if std != 1.0:
        out *= std
    return out


def uniform_stream(seed: int, sid: int, n: int, a: float, device="cpu") -> torch.Tensor:
    """n float64 uniforms on (-a, a) from stream ``sid`` of ``seed``."""
    base = stream_base(seed, sid)
    out = torch.empty(n, dtype=torch.float64, device=device)
    for c0 in range(0, n, _CHUNK):
        c = min(_CHUNK, n - c0)
        out[c0:c0 + c] = a * (2.0 * _u01(draws(base, c0, c, device)) - 1.0)
    return out


def f64_to_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round float64 to bfloat16, nearest-even, in one step (no float32 detour).

    Works on the float64 bit pattern: the 52-bit fraction is rounded to 7 bits and
    the exponent re-biased from 1023 to 127.  Inputs must be zero or inside the
    normal bfloat16 range (always true for the distributions above).
    """
    b = x.contiguous().to(torch.float64).view(torch.int64)
    lsb = _srl(b, 45) & 1
    r = _srl(b + ((1 << 44) - 1) + lsb, 45)           # sign | exp11 | frac7
    sign = (r >> 18) & 1
    e64 = (r >> 7) & 0x7FF
    frac = r & 0x7F
    zero = (b & 0x7FFFFFFFFFFFFFFF) == 0
    e16 = e64 - (1023 - 127)
    bad = ~zero & ((e16 < 1) | (e16 > 254))
    if bool(bad.any()):
        raise ValueError("value outside the normal bfloat16 range")
    e16 = torch.where(zero, torch.zeros_like(e16), e16)
    frac = torch.where(zero, torch.zeros_like(frac), frac)
    bits = (sign << 15) | (e16 << 7) | frac
    return bits.to(torch.int16).view(torch.bfloat16)


def bf16_to_f64(t) -> np.ndarray:
    """Widen a bfloat16 tensor (or its uint16 bits as numpy) to a float64 numpy array."""
    if isinstance(t, np.ndarray):
        u32 = np.ascontiguousarray(t, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return u32.view(np.float32).astype(np.float64)
    return t.detach().to("cpu").to(torch.float64).numpy()


# ----------------------------------------------------------------------------------
# Workloads.  Token count M = batch * seq; every activation is token-major [M, features].
# ----------------------------------------------------------------------------------

@dataclass(frozen=True)
class MlpConfig:
    name: str
    M: int
    h: int
    i: int
    r: int
    alpha: float
    act: str            # "swiglu" or "geglu_tanh"
    batch: int = 0
    seq: int = 0

    @property
    def s(self) -> float:
        return self.alpha / self.r

    def flops(self) -> float:
        """Algorithmic fwd+bwd FLOPs with the base weights frozen (no weight gradient)."""
        M, h, i, r = self.M, self.h, self.i, self.r
        return 12.0 * M * h * i + 18.0 * M * r * (h + i)

    def replace(self, **kw) -> "MlpConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return MlpConfig(**d)


@dataclass(frozen=True)
class QkvoConfig:
    name: str
    M: int
    h: int
    heads_q: int
    heads_kv: int
    head_dim: int
    r: int
    alpha: float
    batch: int = 0
    seq: int = 0

    @property
    def s(self) -> float:
        return self.alpha / self.r

    @property
    def n_q(self) -> int:
        return self.heads_q * self.head_dim

    @property
    def n_kv(self) -> int:
        return self.heads_kv * self.head_dim

    def flops(self) -> float:
        """fwd+bwd FLOPs of the q, k, v and o LoRA linears (frozen W)."""
        tot = 0.0
        for fin, fout in ((self.h, self.n_q), (self.h, self.n_kv), (self.h, self.n_kv),
                          (self.n_q, self.h)):
            tot += 4.0 * self.M * fin * fout + 6.0 * self.M * self.r * (fin + fout)
        return tot

    def replace(self, **kw) -> "QkvoConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return QkvoConfig(**d)


MLP_CONFIGS = {
    "tiny": MlpConfig("tiny", M=64, h=128, i=344, r=8, alpha=16, act="swiglu", batch=2, seq=32),
    "qwen05b": MlpConfig("qwen05b", M=4096, h=896, i=4864, r=16, alpha=32, act="swiglu",
                         batch=4, seq=1024),
    "llama7b": MlpConfig("llama7b", M=8192, h=4096, i=14336, r=16, alpha=32, act="swiglu",
                         batch=4, seq=2048),
    "gemma7b": MlpConfig("gemma7b", M=8192, h=3072, i=24576, r=8, alpha=16, act="geglu_tanh",
                         batch=4, seq=2048),
}

QKVO_CONFIGS = {
    "gqa7b": QkvoConfig("gqa7b", M=8192, h=4096, heads_q=32, heads_kv=8, head_dim=128, r=8,
                        alpha=16, batch=4, seq=2048),
}

# Stream ids: a tensor's stream never depends on the shapes, so a tensor keeps its
# values when a test changes another tensor's size.
MLP_TENSORS = ("x", "W_gate", "A_gate", "B_gate", "W_up", "A_up", "B_up",
               "W_down", "A_down", "B_down", "dy")
QKVO_TENSORS = ("x", "W_q", "A_q", "B_q", "W_k", "A_k", "B_k", "W_v", "A_v", "B_v",
                "o_in", "W_o", "A_o", "B_o", "dy_q", "dy_k", "dy_v", "dy_o")
_B_VAR = 0.02


def _weight(seed, sid, rows, cols, fan_in, dev):
    std = 1.0 / math.sqrt(fan_in)
    return f64_to_bf16(normal_stream(seed, sid, rows * cols, std, dev)).reshape(rows, cols)


def _adapter_a(seed, sid, r, fan_in, dev):
    a = 1.0 / math.sqrt(fan_in)
    return f64_to_bf16(uniform_stream(seed, sid, r * fan_in, a, dev)).reshape(r, fan_in)


def _adapter_b(seed, sid, out, r, dev):
    std = math.sqrt(_B_VAR)
    return f64_to_bf16(normal_stream(seed, sid, out * r, std, dev)).reshape(out, r)


def _act(seed, sid, rows, cols, dev):
    return f64_to_bf16(normal_stream(seed, sid, rows * cols, 1.0, dev)).reshape(rows, cols)


def make_mlp_inputs(cfg: MlpConfig, seed: int = 0, only=None, device="cpu") -> dict:
    """bf16 tensors for one LoRA-MLP problem, keyed by MLP_TENSORS names.

    W_* are [out, in], A_* are [r, in], B_* are [out, r]; x and dy are [M, h].
    """
    M, h, i, r = cfg.M, cfg.h, cfg.i, cfg.r
    sid = {n: k for k, n in enumerate(MLP_TENSORS)}
    d = device
    makers = {
        "x": lambda: _act(seed, sid["x"], M, h, d),
        "W_gate": lambda: _weight(seed, sid["W_gate"], i, h, h, d),
        "A_gate": lambda: _adapter_a(seed, sid["A_gate"], r, h, d),
        "B_gate": lambda: _adapter_b(seed, sid["B_gate"], i, r, d),
        "W_up": lambda: _weight(seed, sid["W_up"], i, h, h, d),
        "A_up": lambda: _adapter_a(seed, sid["A_up"], r, h, d),
        "B_up": lambda: _adapter_b(seed, sid["B_up"], i, r, d),
        "W_down": lambda: _weight(seed, sid["W_down"], h, i, i, d),
        "A_down": lambda: _adapter_a(seed, sid["A_down"], r, i, d),
        "B_down": lambda: _adapter_b(seed, sid["B_down"], h, r, d),
        "dy": lambda: _act(seed, sid["dy"], M, h, d),
    }
    names = MLP_TENSORS if only is None else only
    return {n: makers[n]() for n in names}


def make_qkvo_inputs(cfg: QkvoConfig, seed: int = 0, only=None, device="cpu") -> dict:
    """bf16 tensors for one LoRA Q/K/V + O problem, keyed by QKVO_TENSORS names.

    x is [M, h]; q has n_q outputs, k and v n_kv; o_in and the O projection's
    input are [M, n_q]; W_o is [h, n_q]; dy_p matches the projection's output.
    """
    M, h, r, nq, nkv = cfg.M, cfg.h, cfg.r, cfg.n_q, cfg.n_kv
    sid = {n: k for k, n in enumerate(QKVO_TENSORS)}
    d = device
    outs = {"q": nq, "k": nkv, "v": nkv}
    makers = {"x": lambda: _act(seed, sid["x"], M, h, d),
              "o_in": lambda: _act(seed, sid["o_in"], M, nq, d),
              "W_o": lambda: _weight(seed, sid["W_o"], h, nq, nq, d),
              "A_o": lambda: _adapter_a(seed, sid["A_o"], r, nq, d),
              "B_o": lambda: _adapter_b(seed, sid["B_o"], h, r, d),
              "dy_o": lambda: _act(seed, sid["dy_o"], M, h, d)}
    for p, n_out in outs.items():
        makers[f"W_{p}"] = (lambda p=p, n_out=n_out: _weight(seed, sid[f"W_{p}"], n_out, h, h, d))
        makers[f"A_{p}"] = (lambda p=p: _adapter_a(seed, sid[f"A_{p}"], r, h, d))
        makers[f"B_{p}"] = (lambda p=p, n_out=n_out: _adapter_b(seed, sid[f"B_{p}"], n_out, r, d))
        makers[f"dy_{p}"] = (lambda p=p, n_out=n_out: _act(seed, sid[f"dy_{p}"], M, n_out, d))
    names = QKVO_TENSORS if only is None else only
    return {n: makers[n]() for n in names}


def positions(M: int, seq: int = 0, lengths=None, device="cpu") -> torch.Tensor:
    """int32 position of each of M tokens laid out as sequences end to end: the
    position restarts at 0 where a sequence starts.  Either equal sequences of `seq`
    tokens, or the explicit `lengths` (packed sequences; they must add up to M)."""
    if lengths is None:
        if seq <= 0:
            raise ValueError("give seq or lengths")
        return (torch.arange(M, dtype=torch.int64) % seq).to(torch.int32).to(device)
    if sum(lengths) != M:
        raise ValueError("lengths must add up to M")
    return torch.cat([torch.arange(n, dtype=torch.int32) for n in lengths]).to(device)
