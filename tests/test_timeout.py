"""Failure detection on the GPU without a fault.

A GEMM launch told to leave one pipeline stage empty (lora_test_expire_waits) has
its bounded waits expire: the kernel stops, lets its own copies finish, frees its
tensor memory and exits by itself; the status word then reads LORA_ERR_TIMEOUT.
The next call on the same CUDA context must compute the right answer.  Both GEMM
kernels are covered: the one-CTA kernel (rank-r projections) and the CTA-pair
kernel (the projections).  Nothing here faults, traps or hangs the GPU: every wait
involved is a bounded one, with a 20 ms limit.
"""

import pytest
import torch

import oracle
from helpers import MLP_GRADS, f64, mlp_gpu, mlp_oracle, parity, to_f64_dict
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LIMIT_NS = 20_000_000
TIMEOUT = 6


@pytest.fixture
def short_limit(lib):
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
    lib.set_wait_timeout(LIMIT_NS)
    assert lib.wait_timeout() == LIMIT_NS
    yield
    lib.test_expire_waits(0)
    lib.set_wait_timeout(0)


def _randn(shape, scale, seed):
    g = torch.Generator().manual_seed(seed)
    return synth.f64_to_bf16(torch.randn(*shape, generator=g, dtype=torch.float64) * scale)


def _linear(M, fin, fout, r, seed):
    x = _randn((M, fin), 1.0, seed)
    W = _randn((fout, fin), fin ** -0.5, seed + 1)
    A = _randn((r, fin), fin ** -0.5, seed + 2)
    B = _randn((fout, r), 0.02 ** 0.5, seed + 3)
    return x, W, A, B


def _check_linear(lib, x, W, A, B, s):
    d = lambda t: t.to(DEV)  # noqa: E731
    y, _ = lib.linear_forward(d(x), (d(W), d(A), d(B)), s, training=False)
    torch.cuda.synchronize()
    assert lib.poll_status() == 0
    v = [f64(t) for t in (x, W, A, B)]
    parity("y", y, oracle.lora_linear(*v, s))


@pytest.mark.parametrize("launches", [1, 2])
def test_linear_expired_wait(lib, short_limit, launches):
    """lora_linear_forward launches the rank-r projection (one-CTA kernel), then the
    projection (CTA-pair kernel): launches=1 stalls the first, 2 stalls both."""
    s = 2.0
    x, W, A, B = _linear(300, 512, 384, 8, seed=11)
    d = lambda t: t.to(DEV)  # noqa: E731
    lib.trace_enable(16)
    try:
        lib.test_expire_waits(launches)
        lib.linear_forward(d(x), (d(W), d(A), d(B)), s, training=False)
        torch.cuda.synchronize()                   # the kernels ended by themselves
        trace = lib.trace_read()
    finally:
        lib.trace_enable(0)
    assert lib.poll_status() == TIMEOUT
    assert lib.poll_status() == 0                  # polling clears the word
    gemms = [ms for kind, ms in trace if kind in ("rank_proj", "proj")]
    assert len(gemms) == 2
    # a stalled launch lasts the wait limit (wall-clock, whatever the SM clock) to
    # within 10%; the others microseconds
    for j, ms in enumerate(gemms):
        if j < launches:
            assert LIMIT_NS * 1e-6 <= ms <= 1.1 * LIMIT_NS * 1e-6, trace
        else:
            assert ms < 0.25 * LIMIT_NS * 1e-6, trace
    # the context is intact and the hook is spent: the same call is right again
    _check_linear(lib, x, W, A, B, s)


def test_mlp_expired_wait_mid_call(lib, short_limit):
    """The first three GEMM launches of a forward stall (the rank-r projection, the
    gate/up GEMM and the down projection's rank-r product); the kernels after them in
    the same call run on what was left, and the next calls are right again."""
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=200, h=256, i=520)
    ins = synth.make_mlp_inputs(cfg, seed=5)
    t = {k: v.to(DEV) for k, v in ins.items()}
    mlp_gpu(lib, t, cfg)                           # warm: workspaces, maps
    assert lib.poll_status() == 0
    lib.test_expire_waits(3)
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    lib.mlp_forward(t["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, training=False)
    lib.mlp_forward(t["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, training=False)
    torch.cuda.synchronize()
    assert lib.poll_status() == TIMEOUT
    y, g = mlp_gpu(lib, t, cfg)
    assert lib.poll_status() == 0
    f, b = mlp_oracle(to_f64_dict(ins), cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


def test_noalloc_expired_wait(lib, short_limit):
    """lora_linear_forward_noalloc keeps its status word in its fixed scratch: an
    expired wait there is read (and cleared) by lora_poll_status with no workspace,
    and the next call is right again."""
    s = 2.0
    x, W, A, B = _linear(300, 512, 384, 8, seed=13)
    d = lambda t: t.to(DEV)  # noqa: E731
    lin = (d(W), d(A), d(B))
    lib.test_expire_waits(1)
    lib.linear_forward_noalloc(d(x), lin, s)
    torch.cuda.synchronize()
    assert lib.poll_noalloc_status() == TIMEOUT
    assert lib.poll_noalloc_status() == 0
    y = lib.linear_forward_noalloc(d(x), lin, s)
    torch.cuda.synchronize()
    assert lib.poll_noalloc_status() == 0
    parity("y", y, oracle.lora_linear(*(f64(t) for t in (x, W, A, B)), s))


def test_default_limit_restored(lib):
    assert lib.wait_timeout() == 2_000_000_000
