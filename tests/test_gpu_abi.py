"""The C ABI on the GPU: writes stay inside the buffers the caller passed (guard
bands around every output, the saved blob and the workspace), M = 0 backward
zero-fills the adapter gradients, errors launch nothing, the launch counter and
the event trace account for every kernel, and the status word reads OK."""

import pytest
import torch

import synth
from helpers import MLP_GRADS, f64, mlp_oracle, parity, to_f64_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 4096          # bytes of canary on each side
CANARY = 0x5A


class Guarded:
    """Contiguous bf16 views carved out of one byte buffer with canaries around each."""

    def __init__(self):
        self.parts = []

    def bf16(self, *shape):
        n = 2 * int(torch.tensor(shape).prod())
        buf = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        self.parts.append(buf)
        return buf[GUARD:GUARD + n].view(torch.bfloat16).view(*shape)

    def raw(self, nbytes):
        buf = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        self.parts.append(buf)
        return buf[GUARD:GUARD + nbytes]

    def check(self):
        torch.cuda.synchronize()
        for b in self.parts:
            assert torch.all(b[:GUARD] == CANARY) and torch.all(b[-GUARD:] == CANARY), "guard band overwritten"


@pytest.mark.parametrize("name,over", [("tiny", {}), ("qwen05b", {"M": 333, "i": 4856})])
def test_mlp_writes_stay_in_bounds(lib, name, over):
    cfg = synth.MLP_CONFIGS[name].replace(**over)
    ins = synth.make_mlp_inputs(cfg, seed=1)
    t = {k: x.to(DEV) for k, x in ins.items()}
    M, h, i, r = cfg.M, cfg.h, cfg.i, cfg.r
    saved_b, ws_b = lib.mlp_sizes(M, h, i, r)
    G = Guarded()
    y = G.bf16(M, h)
    saved = G.raw(saved_b)
    ws = G.raw(ws_b)
    ws[:256].zero_()
    grads = {"dA_gate": G.bf16(r, h), "dB_gate": G.bf16(i, r), "dA_up": G.bf16(r, h),
             "dB_up": G.bf16(i, r), "dA_down": G.bf16(r, i), "dB_down": G.bf16(h, r)}
    dx = G.bf16(M, h)
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    lib.mlp_forward(t["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, y=y, saved=saved, ws=ws)
    g = lib.mlp_backward(t["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved, t["dy"],
                         dx=dx, grads=grads, ws=ws)
    G.check()
    assert lib.poll_status(ws) == 0
    f, b = mlp_oracle(to_f64_dict(ins), cfg)
    parity("y", y, f["y"])
    for k in MLP_GRADS:
        parity(k, g[k], b[k])


def test_zero_tokens(lib):
    cfg = synth.MLP_CONFIGS["tiny"]
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg).items()}
    x0 = torch.empty(0, cfg.h, dtype=torch.bfloat16, device=DEV)
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    before = lib.launch_count()
    y, saved = lib.mlp_forward(x0, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    g = lib.mlp_backward(x0, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved, x0)
    torch.cuda.synchronize()
    assert lib.launch_count() == before
    assert y.shape == (0, cfg.h) and g["dx"].shape == (0, cfg.h)
    for k in ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"):
        assert torch.count_nonzero(g[k]).item() == 0


def test_errors_launch_nothing(lib):
    from rank_mlp_gb300.binding import LoraError
    cfg = synth.MLP_CONFIGS["tiny"]
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg).items()}
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    before = lib.launch_count()
    small = torch.zeros(512, dtype=torch.uint8, device=DEV)
    with pytest.raises(LoraError) as e:
        lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, ws=small)
    assert e.value.status == 4
    with pytest.raises(LoraError) as e:
        lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), float("nan"), cfg.act)
    with pytest.raises(ValueError):
        lib.mlp_forward(ins["x"].float(), lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    torch.cuda.synchronize()
    assert lib.launch_count() == before


def test_launch_count_and_trace(lib):
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=512)
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg).items()}
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    lib.trace_enable(256)
    before = lib.launch_count()
    y, saved = lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    lib.mlp_backward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved, ins["dy"])
    n = lib.launch_count() - before
    tr = lib.trace_read()
    lib.trace_enable(0)
    assert len(tr) == n > 0
    kinds = {k for k, _ in tr}
    assert {"gate_up", "proj", "act_bwd", "dgrad", "pack", "rank_proj", "rank_grad"} <= kinds
    assert all(ms > 0 for _, ms in tr)
    assert lib.poll_status() == 0


def test_trace_kinds_filter(lib):
    """Tracing only one kind records only its launches (the bench traces the dominant
    kernel alone inside its timed region)."""
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=512)
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg).items()}
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    lib.trace_kinds(["gate_up"])
    lib.trace_enable(64)
    try:
        for _ in range(3):
            lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, training=False)
        tr = lib.trace_read()
    finally:
        lib.trace_enable(0)
        lib.trace_kinds(None)
    assert [k for k, _ in tr] == ["gate_up"] * 3
    assert lib.poll_status() == 0


def _kinds(lib, fn):
    import collections
    lib.trace_enable(256)
    try:
        fn()
        tr = lib.trace_read()
    finally:
        lib.trace_enable(0)
    return collections.Counter(k for k, _ in tr)


def test_launches_per_call(lib):
    """The launch structure of each call.  MLP forward: pack, the two rank-r
    projections (x A^T, h A^T), the gate/up and down GEMMs, and one split-K reduction
    per rank-r projection that was split; its pack launch also packs the backward's
    adapter operands into the saved blob.  MLP backward (rank 16): the rank-r
    projection dy B_d (with its split-K sums if split), the act' GEMM, one pass over
    dg, du that gives V and dB_g, dB_u (V's partial sums added at once), the dx GEMM,
    the remaining reductions over tokens (dB_d, dA_d, dA_g, dA_u) in one launch, and one
    sum launch at the end for every dA/dB.  Q/K/V + O with RoPE (rank
    8): per half one pass over the output gradients for the projection and dB; the dA of
    all four in one launch after the dx GEMM; plus one transpose-rotation launch in the
    backward, and no pack."""
    cfg = synth.MLP_CONFIGS["qwen05b"].replace(M=1024)
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg).items()}
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    saved = {}

    def fwd():
        saved["y"], saved["s"] = lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)

    def bwd():
        lib.mlp_backward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved["s"], ins["dy"])

    f = _kinds(lib, fwd)
    assert (f["pack"], f["rank_proj"], f["gate_up"], f["proj"]) == (1, 2, 1, 1), f
    assert f["reduce"] <= 2 and set(f) <= {"pack", "rank_proj", "gate_up", "proj", "reduce"}, f
    b = _kinds(lib, bwd)
    assert (b["rank_proj"], b["rank_grad"], b["act_bwd"], b["dgrad"]) == (1, 2, 1, 1), b
    # V's sums, dy B_d's split-K sums (if split), then one for every dA/dB at the end
    assert 2 <= b["reduce"] <= 3 and set(b) <= {"rank_proj", "rank_grad", "act_bwd", "dgrad", "reduce"}, b

    qc = synth.QKVO_CONFIGS["gqa7b"].replace(M=512, h=512, heads_q=4, heads_kv=2, head_dim=128)
    t = {k: x.to(DEV) for k, x in synth.make_qkvo_inputs(qc).items()}
    ql = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    cos, sin = lib.rope_table(512, 128, device=DEV)
    rope = {"cos": cos, "sin": sin, "pos": synth.positions(512, seq=512, device=DEV), "head_dim": 128}

    def qfwd():
        saved["q"] = lib.qkvo_forward(t["x"], ql("q"), ql("k"), ql("v"), t["o_in"], ql("o"), qc.s, rope=rope)[1]

    def qbwd():
        lib.qkvo_backward(t["x"], ql("q"), ql("k"), ql("v"), t["o_in"], ql("o"), qc.s, saved["q"], t["dy_q"],
                          t["dy_k"], t["dy_v"], t["dy_o"], rope=rope)

    f = _kinds(lib, qfwd)
    assert (f["pack"], f["rank_proj"], f["proj"]) == (1, 2, 2), f
    b = _kinds(lib, qbwd)
    # rank 8: one pass over dy_o (U_o, dB_o) and one over dy_q, dy_k, dy_v (V, dB_q, dB_k,
    # dB_v), each with its partial sums, then dA_o and the q, k, v dA in one launch, and
    # the final sums
    assert (b["rope"], b["rank_proj"], b["rank_grad"], b["dgrad"]) == (1, 0, 3, 2) and "pack" not in b, b
    assert b["reduce"] == 3, b
    assert lib.poll_status() == 0


def test_qwen_shaped_step_launches(lib):
    """The Qwen-shaped forward + backward (4096 tokens, h = 896, i = 4864, r = 16) makes
    at most 13 launches: x A^T and dy B_d run unsplit (their split-K sums would cost
    more than the split saves), the forward's pack launch packs for the backward too,
    one pass over dg, du gives V and dB_g, dB_u, and the backward's other reductions
    over tokens take one launch after the dx GEMM and one for their sums."""
    cfg = synth.MLP_CONFIGS["qwen05b"]
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg, seed=4).items()}
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    y, saved = lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    lib.mlp_backward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved, ins["dy"])
    torch.cuda.synchronize()
    before = lib.launch_count()
    y, saved = lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    lib.mlp_backward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved, ins["dy"])
    torch.cuda.synchronize()
    assert lib.launch_count() - before <= 13
    assert lib.poll_status() == 0


def test_two_streams_get_their_own_workspaces(lib):
    """Calls on two streams run concurrently on separate cached workspaces and give
    the same bits as the same calls run one after the other."""
    cfg = synth.MLP_CONFIGS["qwen05b"].replace(M=1024)
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg, seed=3).items()}
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    ref, _ = lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, training=False)
    x2 = torch.flip(ins["x"], dims=[0]).contiguous()
    ref2, _ = lib.mlp_forward(x2, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, training=False)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            a, _ = lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, training=False)
        with torch.cuda.stream(s2):
            b, _ = lib.mlp_forward(x2, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, training=False)
        outs.append((a, b))
    torch.cuda.synchronize()
    for a, b in outs:
        assert torch.equal(a.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(b.view(torch.int16), ref2.view(torch.int16))
    for st in (s1, s2):
        with torch.cuda.stream(st):
            assert lib.poll_status() == 0


def test_per_example_edge_cases(lib):
    """One example is the whole batch (the per-example gradients equal the batch
    gradients, to the parity bar, and the squared norm is their sum of squares); zero
    tokens zero-fill every example's gradients and norms."""
    cfg = synth.MLP_CONFIGS["tiny"].replace(M=192, h=256, i=344)
    ins = {k: x.to(DEV) for k, x in synth.make_mlp_inputs(cfg, seed=12).items()}
    lin = lambda n: (ins["W_" + n], ins["A_" + n], ins["B_" + n])  # noqa: E731
    y, saved = lib.mlp_forward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    one = lib.mlp_backward_per_example(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved,
                                       ins["dy"], 1)
    full = lib.mlp_backward(ins["x"], lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved, ins["dy"])
    torch.cuda.synchronize()
    sq = 0.0
    for k in MLP_GRADS:
        a = one[k] if k == "dx" else one[k][0]
        parity(k, a, f64(full[k]))
        if k != "dx":
            sq += float((a.double() ** 2).sum())
    assert abs(float(one["sq_norms"][0]) - sq) <= 1e-3 * sq

    x0 = torch.empty(0, cfg.h, dtype=torch.bfloat16, device=DEV)
    _, saved0 = lib.mlp_forward(x0, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act)
    z = lib.mlp_backward_per_example(x0, lin("gate"), lin("up"), lin("down"), cfg.s, cfg.act, saved0,
                                     torch.empty(0, cfg.h, dtype=torch.bfloat16, device=DEV), 3)
    torch.cuda.synchronize()
    for k in ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"):
        assert z[k].shape[0] == 3 and bool(torch.all(z[k] == 0))
    assert bool(torch.all(z["sq_norms"] == 0))
    assert lib.poll_status() == 0
