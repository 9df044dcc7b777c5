"""The C ABI on the host (no GPU): the library builds and loads, exports every
function include/lora_gb300.h declares, answers size queries, and rejects bad
arguments before anything is launched.

Only argument combinations that the library rejects during validation are used
here, so no call reaches a CUDA runtime function.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora_gb300.h")


@pytest.fixture(scope="module")
def L():
    from rank_mlp_gb300 import binding, build
    build.build()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("lora_mlp_forward", "lora_mlp_backward", "lora_qkvo_forward", "lora_qkvo_backward",
              "lora_linear_forward", "lora_linear_backward", "lora_poll_status"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    from rank_mlp_gb300 import binding
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in the header but not exported"
        assert n in binding.EXPORTS, f"{n} has no binding signature"


def test_status_strings(L):
    for code in range(8):
        s = L.lora_status_string(code)
        assert s and s != b"unknown status"
    assert L.lora_status_string(99) == b"unknown status"


def test_size_queries(L):
    a = L.lora_mlp_workspace_bytes(4096, 896, 4864, 16)
    b = L.lora_mlp_workspace_bytes(8192, 896, 4864, 16)
    assert 0 < a < b
    s = L.lora_mlp_saved_bytes(8192, 4096, 14336, 16)
    assert s >= 3 * 8192 * 14336 * 2          # g, u and h in bf16
    assert L.lora_mlp_saved_bytes(0, 128, 344, 8) >= 0
    assert L.lora_mlp_workspace_bytes(-1, 128, 344, 8) == 0
    assert L.lora_qkvo_saved_bytes(8192, 4096, 4096, 1024, 8) >= 8192 * 64 * 2
    assert L.lora_linear_workspace_bytes(64, 128, 344, 8) > 256


# ------------------------------------------------------------------ rejected calls

ALIGNED = 1 << 20          # a 256-byte aligned non-null address; never dereferenced


def _lin(L, w=ALIGNED, a=ALIGNED, b=ALIGNED):
    from rank_mlp_gb300.binding import LoraLinear
    return LoraLinear(w, a, b)


def _mlp_fwd(L, M=64, h=128, i=344, r=8, s=2.0, act=0, x=ALIGNED, y=ALIGNED, ws=ALIGNED, ws_bytes=None,
             gate=None):
    ws_bytes = L.lora_mlp_workspace_bytes(max(M, 0), h, i, r) if ws_bytes is None else ws_bytes
    return L.lora_mlp_forward(M, h, i, r, s, act, x, gate or _lin(L), _lin(L), _lin(L), y, None, ws,
                              ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), 1),                     # NULL input
    (dict(M=-1), 1),                       # negative size
    (dict(r=0), 1),                        # rank 0
    (dict(s=float("nan")), 1),             # non-finite scale
    (dict(s=float("inf")), 1),
    (dict(act=7), 1),                      # unknown activation
    (dict(act=3), 1),
    (dict(h=130), 2),                      # feature size not a multiple of 8
    (dict(x=ALIGNED + 2), 2),              # misaligned activation
    (dict(ws=ALIGNED + 16), 2),            # workspace not 256-byte aligned
    (dict(r=129), 3),                      # gate/up pair beyond the fold width
    (dict(ws_bytes=1024), 4),              # workspace too small
])
def test_mlp_forward_rejects(L, kw, code):
    before = L.lora_launch_count()
    assert _mlp_fwd(L, **kw) == code
    assert L.lora_launch_count() == before


def test_mlp_forward_zero_tokens_is_a_no_op(L):
    before = L.lora_launch_count()
    assert _mlp_fwd(L, M=0) == 0
    assert L.lora_launch_count() == before


def test_qkvo_rejects_misaligned_bias_and_large_rank(L):
    lin = _lin(L)
    ws = L.lora_qkvo_workspace_bytes(64, 256, 256, 128, 8)
    args = lambda r, bias: (64, 256, 256, 128, r, 2.0, ALIGNED, lin, lin, lin, ALIGNED, ALIGNED, ALIGNED,  # noqa
                            None, lin, None, bias, None, None, ALIGNED, ws, None)
    assert L.lora_qkvo_forward(*args(8, ALIGNED + 2)) == 2
    assert L.lora_qkvo_forward(*args(86, None)) == 3
    # both halves skipped: nothing to do is an argument error
    assert L.lora_qkvo_forward(64, 256, 256, 128, 8, 2.0, None, lin, lin, lin, None, None, None,
                               None, lin, None, None, None, None, ALIGNED, ws, None) == 1


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), 3),                # head_dim not 64, 128 or 256
    (dict(head_dim=256), 1),               # does not divide n_kv = 128
    (dict(cos=None), 1),
    (dict(pos=None), 1),
    (dict(n_pos=0), 1),
    (dict(cos=ALIGNED + 4), 2),            # tables 16-byte aligned
    (dict(pos=ALIGNED + 2), 2),            # positions 4-byte aligned
])
def test_qkvo_rejects_bad_rope(L, kw, code):
    import ctypes
    from rank_mlp_gb300.binding import LoraGrads, LoraRope
    a = dict(cos=ALIGNED, sin=ALIGNED, pos=ALIGNED, n_pos=2048, head_dim=128)
    a.update(kw)
    rope = ctypes.pointer(LoraRope(a["cos"], a["sin"], a["pos"], a["n_pos"], a["head_dim"]))
    lin = _lin(L)
    ws = L.lora_qkvo_workspace_bytes(64, 256, 256, 128, 8)
    before = L.lora_launch_count()
    assert L.lora_qkvo_forward(64, 256, 256, 128, 8, 2.0, ALIGNED, lin, lin, lin, ALIGNED, ALIGNED, ALIGNED,
                               None, lin, None, None, rope, None, ALIGNED, ws, None) == code
    g = LoraGrads(ALIGNED, ALIGNED)
    assert L.lora_qkvo_backward(64, 256, 256, 128, 8, 2.0, ALIGNED, lin, lin, lin, None, lin, ALIGNED, rope,
                                ALIGNED, ALIGNED, ALIGNED, ALIGNED, None, None, g, g, g, g, ALIGNED, ws,
                                None) == code
    assert L.lora_launch_count() == before


def test_rope_table_rejects(L):
    assert L.lora_rope_table(ALIGNED, ALIGNED, 16, 7, 10000.0, None) == 1     # odd head_dim
    assert L.lora_rope_table(ALIGNED, ALIGNED, 0, 64, 10000.0, None) == 1     # no positions
    assert L.lora_rope_table(ALIGNED, ALIGNED, 16, 64, -1.0, None) == 1       # base <= 0
    assert L.lora_rope_table(ALIGNED, ALIGNED, 16, 64, float("nan"), None) == 1
    assert L.lora_rope_table(ALIGNED + 4, ALIGNED, 16, 64, 10000.0, None) == 2


def test_backward_needs_saved(L):
    from rank_mlp_gb300.binding import LoraGrads
    g = LoraGrads(ALIGNED, ALIGNED)
    ws = L.lora_mlp_workspace_bytes(64, 128, 344, 8)
    lin = _lin(L)
    assert L.lora_mlp_backward(64, 128, 344, 8, 2.0, 0, ALIGNED, lin, lin, lin, None, ALIGNED, ALIGNED,
                               g, g, g, ALIGNED, ws, None) == 1


def test_sizes_beyond_32_bit_indices_are_unsupported(L):
    """M or a feature size above 2^31 - 1 is rejected (LORA_ERR_UNSUPPORTED) before any
    pointer is touched: the kernels index rows, columns and tiles with 32-bit ints."""
    big = 1 << 31
    assert _mlp_fwd(L, M=big, ws_bytes=1 << 62) == 3
    assert _mlp_fwd(L, h=big, ws_bytes=1 << 62) == 3
    assert _mlp_fwd(L, i=big, ws_bytes=1 << 62) == 3
    assert _mlp_fwd(L, M=big - 1, h=big - 1, r=0) == 1          # invalid arguments still win
    lin = _lin(L)
    assert L.lora_linear_forward(big, 128, 256, 8, 1.0, ALIGNED, lin, ALIGNED, None, ALIGNED, 1 << 62,
                                 None) == 3
    assert L.lora_linear_forward_noalloc(64, 128, big, 8, 1.0, ALIGNED, lin, ALIGNED, None) == 3


def test_linear_rejects(L):
    lin = _lin(L)
    ws = L.lora_linear_workspace_bytes(64, 128, 256, 8)
    assert L.lora_linear_forward(64, 128, 256, 257, 1.0, ALIGNED, lin, ALIGNED, None, ALIGNED, ws, None) == 3
    assert L.lora_linear_forward(64, 128, 256, 8, 1.0, ALIGNED, _lin(L, w=ALIGNED + 8), ALIGNED, None,
                                 ALIGNED, ws, None) == 2
    assert L.lora_linear_forward(64, 128, 256, 8, 1.0, ALIGNED, lin, ALIGNED, None, ALIGNED, 10, None) == 4
    assert L.lora_poll_status(ALIGNED + 16, None) == 1      # ws not 256-byte aligned


def test_wait_limit_range(L):
    assert L.lora_wait_timeout() == 2_000_000_000
    assert L.lora_set_wait_timeout(999_999) == 1          # below 1 ms
    assert L.lora_set_wait_timeout(60_000_000_001) == 1   # above 60 s
    assert L.lora_wait_timeout() == 2_000_000_000
    assert L.lora_set_wait_timeout(5_000_000) == 0
    assert L.lora_wait_timeout() == 5_000_000
    assert L.lora_set_wait_timeout(0) == 0                # back to the default
    assert L.lora_wait_timeout() == 2_000_000_000


def test_expiry_hook_range(L):
    assert L.lora_test_expire_waits(-1) == 1
    assert L.lora_test_expire_waits(65) == 1
    assert L.lora_test_expire_waits(0) == 0


def test_split_tail_mode_range(L):
    assert L.lora_split_tail() == 0
    assert L.lora_set_split_tail(-1) == 1
    assert L.lora_set_split_tail(5) == 1
    for m in (1, 2, 3, 4, 0):
        assert L.lora_set_split_tail(m) == 0
        assert L.lora_split_tail() == m
