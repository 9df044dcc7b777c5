"""Regression pin: the oracle's outputs on the tiny workload, as stored by
tests/golden/make_golden.py (which calls only the oracle and the generator).
A change of the oracle's arithmetic shows up here first."""

import json
import os

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_oracle_tiny_matches_stored_values():
    with open(os.path.join(GOLDEN, "oracle_tiny.json")) as f:
        gold = json.load(f)
    cfg = synth.MLP_CONFIGS[gold["config"]]
    v = {k: synth.bf16_to_f64(t) for k, t in synth.make_mlp_inputs(cfg, seed=gold["seed"]).items()}
    args = (v["x"], v["W_gate"], v["A_gate"], v["B_gate"], v["W_up"], v["A_up"], v["B_up"],
            v["W_down"], v["A_down"], v["B_down"], cfg.s, cfg.act)
    got = dict(oracle.mlp_backward(*args, v["dy"]))
    got["y"] = oracle.mlp_forward(*args)["y"]
    for k, g in gold["outputs"].items():
        a = got[k]
        assert np.isclose(np.linalg.norm(a), g["fro"], rtol=1e-10)
        np.testing.assert_allclose(a.reshape(-1)[:6], g["first"], rtol=1e-9, atol=1e-12)
