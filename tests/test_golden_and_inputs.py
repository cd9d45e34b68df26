"""Regression fixture of the oracle and checks of the input recipe."""
import os

import numpy as np
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))



def _read_fixture():
    vals = {}
    with open(os.path.join(HERE, "golden", "tiny_gda_oracle.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            vals[" ".join(parts[:-1])] = float(parts[-1])
    return vals


def test_golden_fixture_reproduces():
    import sys
    sys.path.insert(0, os.path.join(HERE, "golden"))
    import make_golden
    stored = _read_fixture()
    fresh = {}
    for line in make_golden.compute():
        parts = line.split()
        fresh[" ".join(parts[:-1])] = float(parts[-1])
    assert stored.keys() == fresh.keys()
    for key in stored:
        assert fresh[key] == pytest.approx(stored[key], rel=1e-12, abs=1e-15), key


def test_recipe_is_deterministic_and_well_formed():
    a = inputs.tiny_gda(0)
    b = inputs.tiny_gda(0)
    for x, y in [(a.q, b.q), (a.k, b.k), (a.v, b.v), (a.g, b.g), (a.beta, b.beta)]:
        assert torch.equal(x, y)
    assert a.q.dtype == torch.float32 and a.state.abs().max() == 0
    n = a.k.double().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-6)
    assert (a.g <= 0).all() and ((a.beta > 0) & (a.beta < 1)).all()
    assert a.scale == pytest.approx(1 / 8)


def test_bf16_and_kda_shapes():
    b = inputs.make_batch(3, [70, 5], 2, 32, 16, mode="kda", n_slots=2)
    assert b.q.dtype == torch.bfloat16 and b.q.shape == (75, 2, 32)
    assert b.v.shape == (75, 2, 16) and b.g.shape == (75, 2, 32)
    assert b.state.shape == (2, 2, 32, 16) and b.state.dtype == torch.float32
    assert b.cu_seqlens.tolist() == [0, 70, 75]
    assert (b.g <= 0).all() and (b.g > -0.1 * 20).all()


def test_varlen_lengths_in_range():
    lens = inputs.varlen_lengths(4, 8)
    assert lens.shape == (8,) and lens.min() >= 512 and lens.max() <= 8192
    assert torch.equal(lens, inputs.varlen_lengths(4, 8))


def test_verify_accept_counts():
    b = inputs.verify_batch(N=32, T=8, H=1, D=64)
    na = b.meta["n_accepted"]
    assert na.shape == (32,) and na.min() >= 0 and na.max() <= 8
