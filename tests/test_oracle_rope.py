"""Pins for the oracle's rotary position embedding.

Rotary embedding injects the absolute position into attention ("从零构建大模型
推理引擎：KV缓存、算子融合与量化优化实战", section 4.1); the decode token is
appended at its absolute RoPE position (samir-vllm README summary, section
"目前已完成的功能").  The pages fix neither the pairing nor the frequencies;
the oracle reads them as the standard rotate-half pairing (i, i + D/2) with
frequency theta^(-2i/D), theta = 500000.  The closed forms below pin that
reading: identity at position 0, norm preservation, the complex-multiplication
form, the geometric frequency ladder's end points, and the relative-position
property <R_p q, R_r k> = <R_{p-s} q, R_{r-s} k>.
"""
import math

import numpy as np
import pytest

import oracle

THETA = 500000.0
D = 64


@pytest.fixture(scope="module")
def rng():
    return np.random.default_rng(7)


def test_position_zero_is_identity(rng):
    for _ in range(20):
        x = rng.standard_normal(D)
        assert np.array_equal(oracle.rope_rotate(x, 0, THETA), x)


def test_norm_is_preserved(rng):
    for pos in [1, 15, 16, 17, 300, 2047, 100000]:
        x = rng.standard_normal(D)
        y = oracle.rope_rotate(x, pos, THETA)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) <= 1e-12 * np.linalg.norm(x)


def test_complex_multiplication_form(rng):
    # pair i as the complex number x[i] + j x[i+32], turned by exp(j * pos * f_i)
    i = np.arange(D // 2)
    freq = np.exp(-(2.0 * i / D) * math.log(THETA))
    for pos in [1, 5, 17, 999, 2047]:
        x = rng.standard_normal(D)
        z = (x[: D // 2] + 1j * x[D // 2:]) * np.exp(1j * pos * freq)
        y = oracle.rope_rotate(x, pos, THETA)
        assert np.allclose(y[: D // 2], z.real, rtol=0, atol=1e-12)
        assert np.allclose(y[D // 2:], z.imag, rtol=0, atol=1e-12)


def test_frequency_ladder_end_points():
    f = np.array([oracle.rope_inv_freq(THETA, D, i) for i in range(D // 2)])
    assert f[0] == 1.0
    assert math.isclose(f[16], 1.0 / math.sqrt(THETA), rel_tol=1e-14)
    ratios = f[:-1] / f[1:]
    assert np.allclose(ratios, ratios[0], rtol=1e-12, atol=0)
    assert math.isclose(ratios[0] ** 32, THETA, rel_tol=1e-10)


def test_rotation_direction_on_basis_vector():
    # e_0 at position p lands on (cos p, sin p) in the plane (dim 0, dim 32)
    x = np.zeros(D)
    x[0] = 1.0
    for p in [1, 2, 3]:
        y = oracle.rope_rotate(x, p, THETA)
        assert math.isclose(y[0], math.cos(p), abs_tol=1e-15)
        assert math.isclose(y[32], math.sin(p), abs_tol=1e-15)
        assert np.count_nonzero(np.delete(y, [0, 32])) == 0


def test_relative_position_property(rng):
    for _ in range(20):
        q = rng.standard_normal(D)
        k = rng.standard_normal(D)
        p, r = (int(v) for v in rng.integers(0, 2048, size=2))
        s = int(rng.integers(0, min(p, r) + 1))
        lhs = np.dot(oracle.rope_rotate(q, p, THETA), oracle.rope_rotate(k, r, THETA))
        rhs = np.dot(oracle.rope_rotate(q, p - s, THETA), oracle.rope_rotate(k, r - s, THETA))
        assert abs(lhs - rhs) <= 1e-9 * (np.linalg.norm(q) * np.linalg.norm(k))
