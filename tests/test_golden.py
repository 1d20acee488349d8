"""Drift check: the oracle still reproduces the committed fixtures (written by
tests/golden/make_golden.py, which calls only the oracle)."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
# exp/pow of the C library may differ in the last ulp between platforms
RTOL = 1e-13


def _load(name):
    with open(os.path.join(GOLDEN, name + ".json")) as f:
        return json.load(f)


def _close(got, want):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape
    assert np.all(np.abs(got - want) <= RTOL * np.maximum(np.abs(want), 1e-300)), \
        "oracle drifted from its fixture"


def test_linear_fixture():
    fx = _load("linear_f32_small")
    y, nrm = oracle.linear(fx["inputs"]["x"], fx["inputs"]["w"], fx["inputs"]["bias"])
    _close(y, fx["y"]); _close(nrm, fx["nrm"])


def test_addmm_fixture():
    fx = _load("addmm_bf16_small")
    i = fx["inputs"]
    y, nrm = oracle.addmm(i["c"], i["a"], i["b"], i["alpha"], i["beta"])
    _close(y, fx["y"]); _close(nrm, fx["nrm"])


def test_sdpa_fixture():
    fx = _load("sdpa_causal_gqa_small")
    i = fx["inputs"]
    o, nrm = oracle.sdpa(i["q"], i["k"], i["v"], causal=i["causal"], q_offset=i["q_offset"])
    _close(o, fx["o"]); _close(nrm, fx["nrm"])


def test_fixtures_cite_the_page():
    for name in ("linear_f32_small", "addmm_bf16_small", "sdpa_causal_gqa_small"):
        assert "mlx-batch-invariant README" in _load(name)["cite"]


def test_qlinear_fixture():
    fx = _load("qlinear_4bit_small")
    i = fx["inputs"]
    wq = np.asarray(i["wq"], dtype=np.int64).astype(np.int32).view(np.uint32)
    y, nrm = oracle.qlinear(i["x"], wq, i["scales"], i["biases"], i["bits"], i["group_size"],
                            i["bias"])
    _close(y, fx["y"]); _close(nrm, fx["nrm"])
