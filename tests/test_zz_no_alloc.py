"""lora_linear_forward_noalloc, the forward for callers that cannot allocate device
memory where they run it (for example a plugin whose host framework owns all device
memory, or a loop that must not call cudaMalloc): it takes no workspace and uses the
library's fixed scratch array.  Its output must match lora_linear_forward's on
consecutive calls (the array keeps the previous call's contents), and problems whose
scratch need exceeds the array are rejected before anything is launched.

The file name sorts last so that a run stopping at the first failure has already run
every other test."""

import pytest
import torch

import synth
from helpers import parity, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(M, fin, fout, r, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *sh, sc=1.0: synth.f64_to_bf16(torch.randn(*sh, generator=g, dtype=torch.float64) * sc).to(DEV)  # noqa: E731
    return mk(M, fin), (mk(fout, fin, sc=fin ** -0.5), mk(r, fin, sc=fin ** -0.5), mk(fout, r, sc=0.14))


def test_noalloc_matches_linear_forward_on_consecutive_calls(lib):
    cases = [(300, 192, 328, 5, 1, 2.0), (1024, 4096, 1024, 16, 2, 0.5)]
    for M, fin, fout, r, seed, s in cases:
        x, lin = _case(M, fin, fout, r, seed)
        ref, _ = lib.linear_forward(x, lin, s, training=False)
        for _ in range(2):
            y = lib.linear_forward_noalloc(x, lin, s)
            torch.cuda.synchronize()
            parity("y", y, f64(ref))


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    from rank_mlp_gb300.binding import LoraError
    x, lin = _case(1 << 20, 64, 64, 64, 3)       # scratch need: about 128 MiB
    before = lib.launch_count()
    with pytest.raises(LoraError) as e:
        lib.linear_forward_noalloc(x, lin, 1.0)
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert lib.launch_count() == before
