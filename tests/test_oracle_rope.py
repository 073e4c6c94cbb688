"""Pins for the oracle's NeoX RoPE (CPU only).

"Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA Inference Engine"
(§"The Message", §"The Float64 Decision", §"What Input Knowledge Is Required" item 1)
fixes the method: split the rope vector in half, rotate with cos/sin of an angle computed
in float64, convert to float32 at the end.  The pins use forms that do not retype the
oracle's formula: complex multiplication, a 2x2 rotation matrix, textbook trig values,
the rotation's norm preservation and its relative-position property, and torch's own
float32 -> bf16 rounding.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def ulp32(x):
    return np.spacing(np.abs(np.asarray(x, np.float32))).astype(np.float64)


def rope_complex(x, pos, base=10000.0):
    """Rotate-half RoPE as complex multiplication: z_k = x_k + i*x_{k+d/2}, z *= e^{i a}."""
    d = x.shape[-1]
    h = d // 2
    k = np.arange(h, dtype=np.float64)
    ang = np.asarray(pos, np.float64)[..., None] * (base ** (-(2.0 * k) / d))
    z = x[..., :h].astype(np.float64) + 1j * x[..., h:].astype(np.float64)
    z = z * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag], axis=-1)


def _inputs(B=3, Q=5, NH=4, D=64, seed=0, plo=0, phi=9000):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, Q, NH, D)).astype(np.float32)
    P = rng.integers(plo, phi + 1, size=B).astype(np.int32)
    depth = rng.integers(0, Q, size=(B, Q)).astype(np.int32)
    return x, P, depth


def test_position_zero_is_identity():
    x, _, _ = _inputs()
    y = oracle.rope_neox(x, np.zeros(3, np.int32), np.zeros((3, 5), np.int32))
    assert np.array_equal(x, y)


@pytest.mark.parametrize("D", [2, 16, 64, 128])
def test_matches_complex_multiplication(D):
    x, P, depth = _inputs(D=D, seed=D)
    y = oracle.rope_neox(x, P, depth)
    pos = (P[:, None] + depth)[:, :, None]
    ref = rope_complex(x, np.broadcast_to(pos, x.shape[:3]))
    # one rounding of the float64 result to float32; last-bit trig differences allowed
    assert np.all(np.abs(y - ref) <= ulp32(ref) * 1.0 + 1e-30)


def test_d2_is_plane_rotation():
    x = np.array([[[[0.75, -1.5]]]], np.float32)
    for pos in (1, 7, 123456):
        y = oracle.rope_neox(x, np.array([pos], np.int32), np.zeros((1, 1), np.int32))
        a = float(pos)
        R = np.array([[math.cos(a), -math.sin(a)], [math.sin(a), math.cos(a)]])
        ref = R @ x[0, 0, 0].astype(np.float64)
        assert np.all(np.abs(y[0, 0, 0] - ref) <= ulp32(ref))


def test_pair0_rotates_by_position_radians_and_norm_kept():
    x, P, depth = _inputs(D=64, seed=3)
    y = oracle.rope_neox(x, P, depth)
    pos = (P[:, None] + depth)[:, :, None].astype(np.float64)
    # pair k = 0 has inverse frequency exactly 1
    c, s = np.cos(pos), np.sin(pos)
    y0 = x[..., 0] * c - x[..., 32] * s
    assert np.all(np.abs(y[..., 0] - y0) <= ulp32(y0))
    # each (k, k+32) pair keeps its length up to the two float32 roundings
    nx = np.hypot(x[..., :32].astype(np.float64), x[..., 32:].astype(np.float64))
    ny = np.hypot(y[..., :32].astype(np.float64), y[..., 32:].astype(np.float64))
    assert np.all(np.abs(nx - ny) <= 4 * ulp32(nx))


def test_relative_position_property():
    """<R(m)q, R(n)k> depends only on m - n."""
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, 1, 1, 64)).astype(np.float32)
    k = rng.standard_normal((1, 1, 1, 64)).astype(np.float32)
    z = np.zeros((1, 1), np.int32)
    dots = []
    for t in (0, 17, 1000):
        rq = oracle.rope_neox(q, np.array([100 + t], np.int32), z).astype(np.float64)
        rk = oracle.rope_neox(k, np.array([60 + t], np.int32), z).astype(np.float64)
        dots.append(float((rq * rk).sum()))
    scale = float(np.abs(q).sum() * np.abs(k).sum())
    assert max(dots) - min(dots) <= 1e-6 * scale


def test_bf16_output_is_round_to_nearest_even_of_fp32():
    x, P, depth = _inputs(seed=21)
    y32 = oracle.rope_neox(x, P, depth)
    y16 = oracle.rope_neox(x, P, depth, out_bf16=True)
    ref = torch.from_numpy(y32).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(y16, ref)


def test_golden_worked_example():
    with open(os.path.join(GOLDEN, "rope_worked_example.json")) as f:
        g = json.load(f)
    x = np.array(g["x"], np.float32).reshape(1, 1, 1, -1)
    y = oracle.rope_neox(x, np.array([g["prefix_len"]], np.int32),
                         np.array([[g["depth"]]], np.int32), g["base"])
    exp = np.array(g["expected"], np.float64)
    assert np.all(np.abs(y[0, 0, 0] - exp) <= ulp32(exp))
