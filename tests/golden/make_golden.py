"""Writes the stored expected values under tests/golden/.

Calls only the seeded generator (``synth``) and the CPU oracle (``oracle``):
nothing here comes from the CUDA path.  Run from the repository root:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def _bits(t):
    return [f"{int(v) & 0xFFFF:04x}" for v in t.reshape(-1)[:8].view(__import__("torch").int16).tolist()]


def synth_golden():
    cfg = synth.MLP_CONFIGS["tiny"]
    ins = synth.make_mlp_inputs(cfg, seed=0)
    out = {"config": cfg.name, "seed": 0, "tensors": {}}
    for k, t in ins.items():
        out["tensors"][k] = {"shape": list(t.shape), "first_bits": _bits(t),
                             "sum": float(synth.bf16_to_f64(t).sum())}
    return out


def oracle_golden():
    cfg = synth.MLP_CONFIGS["tiny"]
    v = {k: synth.bf16_to_f64(t) for k, t in synth.make_mlp_inputs(cfg, seed=0).items()}
    args = (v["x"], v["W_gate"], v["A_gate"], v["B_gate"], v["W_up"], v["A_up"], v["B_up"],
            v["W_down"], v["A_down"], v["B_down"], cfg.s, cfg.act)
    f = oracle.mlp_forward(*args)
    b = oracle.mlp_backward(*args, v["dy"])
    res = {"config": cfg.name, "seed": 0, "outputs": {}}
    for k, a in (("y", f["y"]),) + tuple((k, b[k]) for k in (
            "dx", "dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down")):
        res["outputs"][k] = {"fro": float(np.linalg.norm(a)), "first": a.reshape(-1)[:6].tolist()}
    return res


def main():
    with open(os.path.join(HERE, "synth_tiny.json"), "w") as f:
        json.dump(synth_golden(), f, indent=1)
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(oracle_golden(), f, indent=1)


if __name__ == "__main__":
    main()
