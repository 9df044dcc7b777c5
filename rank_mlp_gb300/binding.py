"""Python binding of ``include/lora_gb300.h`` (ctypes).

Argument marshalling only: tensors are checked for dtype/contiguity/device, their
pointers and the current CUDA stream are passed to the C ABI, and status codes
become exceptions.  Every step of the computation runs in the library's kernels;
there is no fallback, and a missing library raises.

Adapters are passed as ``(W, A, B)`` tuples of bf16 CUDA tensors: W [out, in],
A [r, in], B [out, r].  Activations are token-major [M, features].
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

ACT = {"swiglu": 0, "geglu_tanh": 1, "geglu_erf": 2}
KIND_NAMES = {0: "pack", 1: "reduce", 2: "rank_proj", 3: "rank_grad", 4: "gate_up",
              5: "proj", 6: "act_bwd", 7: "dgrad", 8: "rope"}
STATUS = {0: "ok", 1: "invalid argument", 2: "alignment", 3: "unsupported",
          4: "workspace too small", 5: "CUDA error", 6: "timeout", 7: "device input out of range"}


class LoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _LIB.lora_status_string(status).decode() if _LIB is not None else STATUS.get(status, "?")
        super().__init__(f"{where}: {msg} (status {status})")


class LoraLinear(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p)]


class LoraGrads(ctypes.Structure):
    _fields_ = [("dA", ctypes.c_void_p), ("dB", ctypes.c_void_p)]


class LoraRope(ctypes.Structure):
    _fields_ = [("cos", ctypes.c_void_p), ("sin", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("n_pos", ctypes.c_int64), ("head_dim", ctypes.c_int)]


_LIB = None
_LOCK = threading.Lock()
_I64, _INT, _F32, _VP, _SZ = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

_SIGS = {
    "lora_linear_saved_bytes": (_SZ, [_I64, _I64, _I64, _INT]),
    "lora_linear_workspace_bytes": (_SZ, [_I64, _I64, _I64, _INT]),
    "lora_linear_forward": (_INT, [_I64, _I64, _I64, _INT, _F32, _VP, LoraLinear, _VP, _VP, _VP, _SZ, _VP]),
    "lora_linear_backward": (_INT, [_I64, _I64, _I64, _INT, _F32, _VP, LoraLinear, _VP, _VP, _VP, LoraGrads,
                                    _VP, _SZ, _VP]),
    "lora_linear_forward_noalloc": (_INT, [_I64, _I64, _I64, _INT, _F32, _VP, LoraLinear, _VP, _VP]),
    "lora_mlp_saved_bytes": (_SZ, [_I64, _I64, _I64, _INT]),
    "lora_mlp_workspace_bytes": (_SZ, [_I64, _I64, _I64, _INT]),
    "lora_mlp_forward": (_INT, [_I64, _I64, _I64, _INT, _F32, _INT, _VP, LoraLinear, LoraLinear, LoraLinear,
                                _VP, _VP, _VP, _SZ, _VP]),
    "lora_mlp_backward": (_INT, [_I64, _I64, _I64, _INT, _F32, _INT, _VP, LoraLinear, LoraLinear, LoraLinear,
                                 _VP, _VP, _VP, LoraGrads, LoraGrads, LoraGrads, _VP, _SZ, _VP]),
    "lora_mlp_per_example_workspace_bytes": (_SZ, [_I64, _I64, _I64, _INT, _I64]),
    "lora_mlp_backward_per_example": (_INT, [_I64, _I64, _I64, _INT, _F32, _INT, _I64, _VP, LoraLinear, LoraLinear,
                                             LoraLinear, _VP, _VP, _VP, LoraGrads, LoraGrads, LoraGrads, _VP, _VP,
                                             _SZ, _VP]),
    "lora_qkvo_saved_bytes": (_SZ, [_I64, _I64, _I64, _I64, _INT]),
    "lora_qkvo_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I64, _INT]),
    "lora_rope_table": (_INT, [_VP, _VP, _I64, _INT, ctypes.c_double, _VP]),
    "lora_qkvo_forward": (_INT, [_I64, _I64, _I64, _I64, _INT, _F32, _VP, LoraLinear, LoraLinear, LoraLinear,
                                 _VP, _VP, _VP, _VP, LoraLinear, _VP, _VP, ctypes.POINTER(LoraRope), _VP, _VP,
                                 _SZ, _VP]),
    "lora_qkvo_backward": (_INT, [_I64, _I64, _I64, _I64, _INT, _F32, _VP, LoraLinear, LoraLinear, LoraLinear,
                                  _VP, LoraLinear, _VP, ctypes.POINTER(LoraRope), _VP, _VP, _VP, _VP, _VP, _VP,
                                  LoraGrads, LoraGrads, LoraGrads, LoraGrads, _VP, _SZ, _VP]),
    "lora_poll_status": (_INT, [_VP, _VP]),
    "lora_status_string": (ctypes.c_char_p, [_INT]),
    "lora_launch_count": (ctypes.c_uint64, []),
    "lora_set_wait_timeout": (_INT, [ctypes.c_uint64]),
    "lora_wait_timeout": (ctypes.c_uint64, []),
    "lora_test_expire_waits": (_INT, [_INT]),
    "lora_set_split_tail": (_INT, [_INT]),
    "lora_split_tail": (_INT, []),
    "lora_trace_enable": (_INT, [_INT]),
    "lora_trace_kinds": (None, [ctypes.c_uint]),
    "lora_trace_read": (_INT, [ctypes.POINTER(_INT), ctypes.POINTER(_F32), _INT]),
}
EXPORTS = tuple(_SIGS)


def load(path: str | None = None):
    """Loads the library (built in-tree by ``rank_mlp_gb300.build``); raises if absent."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = path or _build.lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m rank_mlp_gb300.build` "
                               "(there is no fallback path)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        raise LoraError(status, where)


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor (got {t.dtype}, {t.device})")
    return t.data_ptr()


def _opt(t, name):
    return None if t is None else _dev(t, name)


def _lin(lin, name) -> LoraLinear:
    W, A, B = lin
    return LoraLinear(_dev(W, name + ".W"), _dev(A, name + ".A"), _dev(B, name + ".B"))


# ------------------------------------------------------------------ workspaces

_WS = {}


def workspace(nbytes: int, device) -> torch.Tensor:
    """A workspace of at least nbytes for the current stream of `device` (cached per
    device and stream, grown on demand, first 256 bytes zeroed: they hold the
    asynchronous status word).  Calls that share a workspace must not overlap on the
    GPU, so each stream gets its own; calls on one stream are ordered anyway."""
    device = torch.device(device)
    idx = device.index if device.index is not None else torch.cuda.current_device()
    key = (idx, torch.cuda.current_stream(idx).cuda_stream)
    ws = _WS.get(key)
    if ws is None or ws.numel() < nbytes:
        old = ws
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=torch.device("cuda", idx))
        if old is not None:
            ws[:4].copy_(old[:4])     # keep a status bit that has not been polled yet (same stream)
        _WS[key] = ws
    return ws


def poll_status(ws: torch.Tensor | None = None) -> int:
    lib = load()
    if ws is None:
        ws = workspace(256, torch.cuda.current_device())
    return lib.lora_poll_status(ctypes.c_void_p(ws.data_ptr()), _stream(ws.device))


def poll_noalloc_status() -> int:
    """Reads and clears the status word of lora_linear_forward_noalloc's scratch on the
    current device (lora_poll_status with ws = NULL); syncs the current stream."""
    return load().lora_poll_status(None, _stream(torch.cuda.current_device()))


def launch_count() -> int:
    return int(load().lora_launch_count())


def set_wait_timeout(ns: int):
    """Limit of the kernels' bounded waits, in ns (0 = the default of 2 s)."""
    _check(load().lora_set_wait_timeout(ns), "lora_set_wait_timeout")


def wait_timeout() -> int:
    return int(load().lora_wait_timeout())


def set_split_tail(mode: int):
    """Split-tail mode of the projection GEMMs: 0 automatic, 1 never, 2..4 every tail
    in that many pieces."""
    _check(load().lora_set_split_tail(mode), "lora_set_split_tail")


def split_tail() -> int:
    return int(load().lora_split_tail())


def test_expire_waits(launches: int):
    """Failure-path tests: the next `launches` GEMM launches let a bounded wait expire."""
    _check(load().lora_test_expire_waits(launches), "lora_test_expire_waits")


def trace_kinds(names=None):
    """Trace only these kinds (names of KIND_NAMES; None: all)."""
    if names is None:
        mask = 0xFFFFFFFF
    else:
        inv = {v: k for k, v in KIND_NAMES.items()}
        mask = 0
        for n in names:
            mask |= 1 << inv[n]
    load().lora_trace_kinds(mask)


def trace_enable(capacity: int):
    _check(load().lora_trace_enable(capacity), "lora_trace_enable")


def trace_read(max_entries: int = 4096):
    """[(kind name, ms)] of the launches recorded since the trace was (re)started."""
    kinds = (_INT * max_entries)()
    ms = (_F32 * max_entries)()
    n = load().lora_trace_read(kinds, ms, max_entries)
    if n < 0:
        raise LoraError(5, "lora_trace_read")
    return [(KIND_NAMES.get(kinds[j], str(kinds[j])), float(ms[j])) for j in range(n)]


# ------------------------------------------------------------------ single linear

def linear_forward(x, lin, s, *, y=None, saved=None, training=True, ws=None):
    lib = load()
    W, A, B = lin
    M, fin = x.shape
    fout, r = W.shape[0], A.shape[0]
    if y is None:
        y = torch.empty(M, fout, dtype=torch.bfloat16, device=x.device)
    if saved is None and training:
        saved = torch.empty(max(lib.lora_linear_saved_bytes(M, fin, fout, r), 256), dtype=torch.uint8,
                            device=x.device)
    need = lib.lora_linear_workspace_bytes(M, fin, fout, r)
    ws = workspace(need, x.device) if ws is None else ws
    _check(lib.lora_linear_forward(M, fin, fout, r, s, _dev(x, "x"), _lin(lin, "lin"), _dev(y, "y"),
                                   None if saved is None else saved.data_ptr(), ws.data_ptr(), ws.numel(),
                                   _stream(x.device)), "lora_linear_forward")
    return y, saved


def linear_forward_noalloc(x, lin, s, *, y=None):
    """Inference forward through lora_linear_forward_noalloc: the library allocates
    nothing and the caller passes no workspace (the library's fixed scratch is used)."""
    lib = load()
    W, A, B = lin
    M = x.shape[0]
    if y is None:
        y = torch.empty(M, W.shape[0], dtype=torch.bfloat16, device=x.device)
    _check(lib.lora_linear_forward_noalloc(M, x.shape[1], W.shape[0], A.shape[0], s, _dev(x, "x"),
                                           _lin(lin, "lin"), _dev(y, "y"), _stream(x.device)),
           "lora_linear_forward_noalloc")
    return y


def linear_backward(x, lin, s, saved, dy, *, dx=None, dA=None, dB=None, ws=None):
    lib = load()
    W, A, B = lin
    M, fin = x.shape
    fout, r = W.shape[0], A.shape[0]
    dev = x.device
    dx = torch.empty(M, fin, dtype=torch.bfloat16, device=dev) if dx is None else dx
    dA = torch.empty(r, fin, dtype=torch.bfloat16, device=dev) if dA is None else dA
    dB = torch.empty(fout, r, dtype=torch.bfloat16, device=dev) if dB is None else dB
    need = lib.lora_linear_workspace_bytes(M, fin, fout, r)
    ws = workspace(need, dev) if ws is None else ws
    _check(lib.lora_linear_backward(M, fin, fout, r, s, _dev(x, "x"), _lin(lin, "lin"), saved.data_ptr(),
                                    _dev(dy, "dy"), _dev(dx, "dx"), LoraGrads(_dev(dA, "dA"), _dev(dB, "dB")),
                                    ws.data_ptr(), ws.numel(), _stream(dev)), "lora_linear_backward")
    return dx, dA, dB


# ------------------------------------------------------------------ gated MLP

def mlp_sizes(M, h, i, r):
    lib = load()
    return lib.lora_mlp_saved_bytes(M, h, i, r), lib.lora_mlp_workspace_bytes(M, h, i, r)


def mlp_forward(x, gate, up, down, s, act="swiglu", *, y=None, saved=None, training=True, ws=None):
    """y = down(act(gate(x)) * up(x)); returns (y, saved)."""
    lib = load()
    M, h = x.shape
    i, r = gate[0].shape[0], gate[1].shape[0]
    if y is None:
        y = torch.empty(M, h, dtype=torch.bfloat16, device=x.device)
    if saved is None and training:
        saved = torch.empty(max(lib.lora_mlp_saved_bytes(M, h, i, r), 256), dtype=torch.uint8, device=x.device)
    need = lib.lora_mlp_workspace_bytes(M, h, i, r)
    ws = workspace(need, x.device) if ws is None else ws
    _check(lib.lora_mlp_forward(M, h, i, r, s, ACT[act], _dev(x, "x"), _lin(gate, "gate"), _lin(up, "up"),
                                _lin(down, "down"), _dev(y, "y"), None if saved is None else saved.data_ptr(),
                                ws.data_ptr(), ws.numel(), _stream(x.device)), "lora_mlp_forward")
    return y, saved


def mlp_backward(x, gate, up, down, s, act, saved, dy, *, dx=None, grads=None, ws=None):
    """Returns dict(dx, dA_gate, dB_gate, dA_up, dB_up, dA_down, dB_down)."""
    lib = load()
    M, h = x.shape
    i, r = gate[0].shape[0], gate[1].shape[0]
    dev = x.device
    e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device=dev)  # noqa: E731
    out = {"dx": e(M, h) if dx is None else dx}
    if grads is None:
        grads = {"dA_gate": e(r, h), "dB_gate": e(i, r), "dA_up": e(r, h), "dB_up": e(i, r),
                 "dA_down": e(r, i), "dB_down": e(h, r)}
    out.update(grads)
    need = lib.lora_mlp_workspace_bytes(M, h, i, r)
    ws = workspace(need, dev) if ws is None else ws
    g = lambda n: LoraGrads(_dev(out["dA_" + n], "dA_" + n), _dev(out["dB_" + n], "dB_" + n))  # noqa: E731
    _check(lib.lora_mlp_backward(M, h, i, r, s, ACT[act], _dev(x, "x"), _lin(gate, "gate"), _lin(up, "up"),
                                 _lin(down, "down"), saved.data_ptr(), _dev(dy, "dy"), _dev(out["dx"], "dx"),
                                 g("gate"), g("up"), g("down"), ws.data_ptr(), ws.numel(), _stream(dev)),
           "lora_mlp_backward")
    return out


def mlp_backward_per_example(x, gate, up, down, s, act, saved, dy, n_examples, *, norms=True, ws=None):
    """Per-example adapter gradients (DP-SGD): dict(dx, dA_gate [n, r, h], dB_gate
    [n, i, r], ..., sq_norms [n] float32 or None)."""
    lib = load()
    M, h = x.shape
    i, r = gate[0].shape[0], gate[1].shape[0]
    n = int(n_examples)
    dev = x.device
    e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device=dev)  # noqa: E731
    out = {"dx": e(M, h), "dA_gate": e(n, r, h), "dB_gate": e(n, i, r), "dA_up": e(n, r, h), "dB_up": e(n, i, r),
           "dA_down": e(n, r, i), "dB_down": e(n, h, r),
           "sq_norms": torch.empty(n, dtype=torch.float32, device=dev) if norms else None}
    need = lib.lora_mlp_per_example_workspace_bytes(M, h, i, r, n)
    ws = workspace(need, dev) if ws is None else ws
    g = lambda k: LoraGrads(_dev(out["dA_" + k], "dA_" + k), _dev(out["dB_" + k], "dB_" + k))  # noqa: E731
    _check(lib.lora_mlp_backward_per_example(
        M, h, i, r, s, ACT[act], n, _dev(x, "x"), _lin(gate, "gate"), _lin(up, "up"), _lin(down, "down"),
        saved.data_ptr(), _dev(dy, "dy"), _dev(out["dx"], "dx"), g("gate"), g("up"), g("down"),
        None if out["sq_norms"] is None else out["sq_norms"].data_ptr(), ws.data_ptr(), ws.numel(),
        _stream(dev)), "lora_mlp_backward_per_example")
    return out


# ------------------------------------------------------------------ Q/K/V + O

def rope_table(n_pos: int, head_dim: int, base: float = 10000.0, device="cuda"):
    """(cos, sin), f32 [n_pos, head_dim/2] on `device`: the angle p * base^(-2c/head_dim)."""
    dev = torch.device(device)
    cos = torch.empty(n_pos, head_dim // 2, dtype=torch.float32, device=dev)
    sin = torch.empty_like(cos)
    _check(load().lora_rope_table(cos.data_ptr(), sin.data_ptr(), n_pos, head_dim, float(base), _stream(dev)),
           "lora_rope_table")
    return cos, sin


def _rope(rope):
    """None, or dict(cos, sin, pos, head_dim): f32 tables [n_pos, head_dim/2] and int32
    positions [M] on the device."""
    if rope is None:
        return None
    cos, sin, pos = rope["cos"], rope["sin"], rope["pos"]
    for t, dt, name in ((cos, torch.float32, "cos"), (sin, torch.float32, "sin"), (pos, torch.int32, "pos")):
        if t.dtype != dt or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"rope {name}: contiguous {dt} on the GPU expected")
    if cos.shape != sin.shape or cos.shape[1] * 2 != rope["head_dim"]:
        raise ValueError("rope tables must be [n_pos, head_dim/2]")
    return ctypes.pointer(LoraRope(cos.data_ptr(), sin.data_ptr(), pos.data_ptr(), cos.shape[0], rope["head_dim"]))


def qkvo_forward(x, q, k, v, o_in, o, s, *, bias=None, rope=None, saved=None, training=True, ws=None,
                 outs=None):
    """q/k/v from x (skipped if x is None) and the O projection of o_in (skipped if
    o_in is None).  bias: None or the frozen q/k/v biases, one bf16 tensor
    [n_q + 2 n_kv].  rope: None or dict(cos, sin, pos, head_dim), applied to q and k.
    Returns (dict(q, k, v, o), saved)."""
    lib = load()
    ref = x if x is not None else o_in
    dev = ref.device
    M = ref.shape[0]
    h = q[0].shape[1] if x is not None else o[0].shape[0]
    nq = q[0].shape[0] if x is not None else o[0].shape[1]
    nkv = k[0].shape[0] if x is not None else 8
    r = (q if x is not None else o)[1].shape[0]
    e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device=dev)  # noqa: E731
    res = dict(outs or {})
    if x is not None:
        for n, w in (("q", nq), ("k", nkv), ("v", nkv)):
            res.setdefault(n, e(M, w))
    if o_in is not None:
        res.setdefault("o", e(M, h))
    if saved is None and training:
        saved = torch.empty(max(lib.lora_qkvo_saved_bytes(M, h, nq, nkv, r), 256), dtype=torch.uint8,
                            device=dev)
    need = lib.lora_qkvo_workspace_bytes(M, h, nq, nkv, r)
    ws = workspace(need, dev) if ws is None else ws
    z = LoraLinear(None, None, None)
    _check(lib.lora_qkvo_forward(
        M, h, nq, nkv, r, s, _opt(x, "x"),
        _lin(q, "q") if x is not None else z, _lin(k, "k") if x is not None else z,
        _lin(v, "v") if x is not None else z,
        _opt(res.get("q"), "yq"), _opt(res.get("k"), "yk"), _opt(res.get("v"), "yv"),
        _opt(o_in, "o_in"), _lin(o, "o") if o_in is not None else z, _opt(res.get("o"), "yo"),
        _opt(bias, "bias"), _rope(rope), None if saved is None else saved.data_ptr(), ws.data_ptr(), ws.numel(),
        _stream(dev)),
        "lora_qkvo_forward")
    return res, saved


def qkvo_backward(x, q, k, v, o_in, o, s, saved, dyq=None, dyk=None, dyv=None, dyo=None, *, rope=None,
                  ws=None):
    """Returns dict(dx, do_in, dA_q, dB_q, ..., dA_o, dB_o) for the halves present.
    With rope (the forward's), dyq and dyk are gradients of the rotated q and k."""
    lib = load()
    ref = x if x is not None else o_in
    dev = ref.device
    M = ref.shape[0]
    h = q[0].shape[1] if x is not None else o[0].shape[0]
    nq = q[0].shape[0] if x is not None else o[0].shape[1]
    nkv = k[0].shape[0] if x is not None else 8
    r = (q if x is not None else o)[1].shape[0]
    e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device=dev)  # noqa: E731
    out = {}
    z = LoraGrads(None, None)
    zl = LoraLinear(None, None, None)
    if x is not None:
        out["dx"] = e(M, h)
        for n, w in (("q", nq), ("k", nkv), ("v", nkv)):
            out["dA_" + n], out["dB_" + n] = e(r, h), e(w, r)
    if o_in is not None:
        out["do_in"] = e(M, nq)
        out["dA_o"], out["dB_o"] = e(r, nq), e(h, r)
    gr = lambda n: LoraGrads(out["dA_" + n].data_ptr(), out["dB_" + n].data_ptr()) if "dA_" + n in out else z  # noqa: E731,E501
    need = lib.lora_qkvo_workspace_bytes(M, h, nq, nkv, r)
    ws = workspace(need, dev) if ws is None else ws
    _check(lib.lora_qkvo_backward(
        M, h, nq, nkv, r, s, _opt(x, "x"),
        _lin(q, "q") if x is not None else zl, _lin(k, "k") if x is not None else zl,
        _lin(v, "v") if x is not None else zl, _opt(o_in, "o_in"),
        _lin(o, "o") if o_in is not None else zl, saved.data_ptr(), _rope(rope),
        _opt(dyq, "dyq"), _opt(dyk, "dyk"), _opt(dyv, "dyv"), _opt(out.get("dx"), "dx"),
        _opt(dyo, "dyo"), _opt(out.get("do_in"), "do_in"), gr("q"), gr("k"), gr("v"), gr("o"),
        ws.data_ptr(), ws.numel(), _stream(dev)), "lora_qkvo_backward")
    return out
