"""Pins of the fp64 gated-LoRA oracle against things other than itself.

The operation ("Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
aifromscratch.in, section "Two Decoupled Weight Sets"):
    y = x.W^T + gate_row * (alpha/rank) * (x.A^T).B^T
Pins: a hand-worked golden example; gate-0 rows against numpy's matmul (a
library routine); gate-1 rows against the merged-weight form
x.(W + (alpha/rank) B.A)^T (a different association of the same product);
alpha = 0 and B = 0 reduce to x.W^T.  Non-square shapes everywhere, so a
transposed operand cannot pass.
"""
import numpy as np
import pytest

from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def test_golden_tiny(oracle_mod):
    g = read_golden("gated_lora_tiny.txt")
    M, d_in, d_out, r = (int(g[k][0]) for k in ("M", "d_in", "d_out", "rank"))
    x = np.array(g["x"]).reshape(M, d_in)
    W = np.array(g["W"]).reshape(d_out, d_in)
    A = np.array(g["A"]).reshape(r, d_in)
    B = np.array(g["B"]).reshape(d_out, r)
    gate = np.array(g["gate"], dtype=np.uint8)
    y = oracle_mod.gated_lora_linear(x, W, A, B, gate, g["alpha"][0])
    np.testing.assert_array_equal(y, np.array(g["y"]).reshape(M, d_out))


@pytest.mark.parametrize("M,d_in,d_out,r,alpha", [(7, 24, 40, 8, 16.0), (12, 64, 24, 16, 32.0)])
def test_against_numpy_forms(oracle_mod, M, d_in, d_out, r, alpha):
    rng = np.random.default_rng(7)
    x = _rand(rng, M, d_in)
    W = _rand(rng, d_out, d_in, std=0.02)
    A = _rand(rng, r, d_in, std=0.02)
    B = _rand(rng, d_out, r, std=0.01)
    gate = (np.arange(M) % 3 == 1).astype(np.uint8)
    y = oracle_mod.gated_lora_linear(x, W, A, B, gate, alpha)
    base = x @ W.T
    merged = x @ (W + (alpha / r) * (B @ A)).T
    scale = np.abs(base).max()
    for m in range(M):
        want = merged[m] if gate[m] else base[m]
        np.testing.assert_allclose(y[m], want, rtol=0, atol=1e-12 * scale)
    # the adapter really contributes on gate-1 rows (guards a dropped term)
    assert np.abs(merged - base)[gate == 1].max() > 1e-4 * scale


def test_alpha_zero_and_b_zero_reduce_to_base(oracle_mod):
    rng = np.random.default_rng(3)
    M, d_in, d_out, r = 9, 32, 20, 8
    x, W = _rand(rng, M, d_in), _rand(rng, d_out, d_in, std=0.02)
    A, B = _rand(rng, r, d_in, std=0.02), _rand(rng, d_out, r, std=0.01)
    gate = np.ones(M, np.uint8)
    base = x @ W.T
    y0 = oracle_mod.gated_lora_linear(x, W, A, B, gate, 0.0)
    yb = oracle_mod.gated_lora_linear(x, W, A, np.zeros_like(B), gate, 16.0)
    np.testing.assert_allclose(y0, base, rtol=0, atol=1e-12)
    np.testing.assert_allclose(yb, base, rtol=0, atol=1e-12)


def test_gate_zero_rows_are_exactly_base(oracle_mod):
    """gate 0 multiplies the adapter term by exactly 0: the row equals the
    rank-0 call (same summation order) bit for bit."""
    rng = np.random.default_rng(11)
    M, d_in, d_out, r = 6, 40, 16, 8
    x, W = _rand(rng, M, d_in), _rand(rng, d_out, d_in, std=0.02)
    A, B = _rand(rng, r, d_in, std=0.02), _rand(rng, d_out, r, std=0.01)
    gate = np.array([0, 1, 0, 1, 1, 0], np.uint8)
    y = oracle_mod.gated_lora_linear(x, W, A, B, gate, 256.0)
    y_rank0 = oracle_mod.gated_lora_linear(x, W, np.zeros((0, d_in)), np.zeros((d_out, 0)),
                                           gate, 256.0)
    np.testing.assert_array_equal(y[gate == 0], y_rank0[gate == 0])
    assert not np.array_equal(y[gate == 1], y_rank0[gate == 1])


def test_empty(oracle_mod):
    y = oracle_mod.gated_lora_linear(np.zeros((0, 8)), np.zeros((4, 8)), np.zeros((2, 8)),
                                     np.zeros((4, 2)), np.zeros(0, np.uint8), 1.0)
    assert y.shape == (0, 4)
