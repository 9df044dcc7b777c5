"""lora_linear_forward_noalloc, the forward for callers that cannot allocate device
memory where they run it (for example a plugin whose host framework owns all device
memory, or a loop that must not call cudaMalloc): it takes no workspace and uses the
library's fixed 32 MiB scratch array.  Its output must match the float64 oracle on
consecutive calls (the array keeps the previous call's contents), the scratch's status
word must read clean afterwards, and the size rule must follow the forward's own
scratch need: a problem whose backward would need more than the array still runs,
one whose forward needs more is rejected before anything is launched.

The file name sorts last so that a run stopping at the first failure has already run
every other test."""

import numpy as np
import pytest
import torch

import oracle
from helpers import f64, parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCRATCH = 32 << 20


def _case(M, fin, fout, r, seed):
    import synth
    g = torch.Generator().manual_seed(seed)
    mk = lambda *sh, sc=1.0: synth.f64_to_bf16(torch.randn(*sh, generator=g, dtype=torch.float64) * sc)  # noqa: E731
    return mk(M, fin), (mk(fout, fin, sc=fin ** -0.5), mk(r, fin, sc=fin ** -0.5), mk(fout, r, sc=0.14))


def _run_twice_against_oracle(lib, M, fin, fout, r, seed, s, rows=None):
    x, lin = _case(M, fin, fout, r, seed)
    xd, lind = x.to(DEV), tuple(t.to(DEV) for t in lin)
    rows = np.arange(M) if rows is None else rows
    ref = oracle.lora_linear(f64(x)[rows], *(f64(t) for t in lin), s)
    for _ in range(2):
        y = lib.linear_forward_noalloc(xd, lind, s)
        torch.cuda.synchronize()
        parity("y", y.cpu()[torch.as_tensor(rows)], ref)
    assert lib.poll_noalloc_status() == 0


def test_noalloc_matches_oracle_on_consecutive_calls(lib):
    # several tiles and a ragged tail (300 rows, 328 columns, rank 5), then the Q/K/V
    # shape's k projection (4096 -> 1024, rank 16)
    _run_twice_against_oracle(lib, 300, 192, 328, 5, seed=1, s=2.0)
    _run_twice_against_oracle(lib, 1024, 4096, 1024, 16, seed=2, s=0.5)


def test_noalloc_size_rule_is_the_forwards_own(lib):
    """4096 tokens of a 4096 -> 4096 projection at rank 16: the forward needs about
    17 MiB of scratch, the backward (counted by lora_linear_workspace_bytes) about
    49 MiB.  The call runs; rows sampled across the tiles match the oracle."""
    M, fin, fout, r = 4096, 4096, 4096, 16
    assert lib.load().lora_linear_workspace_bytes(M, fin, fout, r) > SCRATCH
    rows = np.r_[0:64, 1000:1064, 2047:2050, 4032:4096]
    _run_twice_against_oracle(lib, M, fin, fout, r, seed=4, s=2.0, rows=rows)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    from rank_mlp_gb300.binding import LoraError
    # 8192 tokens of the same projection: the forward's split-K slab alone is 32 MiB
    x, lin = _case(8192, 4096, 4096, 16, 3)
    x, lin = x.to(DEV), tuple(t.to(DEV) for t in lin)
    before = lib.launch_count()
    with pytest.raises(LoraError) as e:
        lib.linear_forward_noalloc(x, lin, 1.0)
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert lib.launch_count() == before
