"""Pins for the oracle's int8-activation path: the per-32 quantizer and the
int8 x int8 matvec.

Sources: Mnemonic "In the browser", "Dot products and math" (activations
quantized to int8 per group of 32 with one scale per group; exact int32 dot
sums, then floats scaled by the activation group's scale) and ds4f-disk issue
#6, step 4 (int8 weights with per-16 E8M0 group scales).

Independent references: hand-derived codes and scales
(tests/golden/i8_quantize_pins.txt), properties every correct rounding has,
a dense numpy float64 matrix product, and the oracle's own float-activation
I8 matvec (pinned in test_oracle_pins.py) where q * d is exact in float32.
"""
import numpy as np
import pytest

import oracle
from conftest import parse_float, read_golden
from quantized_weight_matvec_gb300 import synth


def _golden_cases():
    cases = {}
    for row in read_golden("i8_quantize_pins.txt"):
        cases.setdefault(row[0], {})[row[1]] = row[2:]
    return cases


def test_quantize_golden_cases():
    for name, c in _golden_cases().items():
        x = np.zeros((1, 32), np.float32)
        for tok in c["x"]:
            col, val = tok.split(":")
            x[0, int(col)] = parse_float(val)
        want_q = np.zeros(32, np.int8)
        for tok in c["q"]:
            col, val = tok.split(":")
            want_q[int(col)] = int(val)
        want_d = np.float32(parse_float(c["d"][0]))
        q, d = oracle.i8_quantize_x(x)
        assert np.array_equal(q[0], want_q), name
        assert d.shape == (1, 1) and d[0, 0].view(np.uint32) == want_d.view(np.uint32), name


def test_quantize_groups_of_32_and_short_tail():
    """Groups are 32 consecutive columns; the last one may be shorter and has
    its own scale (C = 70: groups of 32, 32 and 6)."""
    x = np.zeros((2, 70), np.float32)
    x[0, 5], x[0, 40], x[0, 69] = 127.0, 254.0, -12.7
    x[1, 31], x[1, 32] = 1.0, -2.0
    q, d = oracle.i8_quantize_x(x)
    assert d.shape == (2, 3)
    assert np.array_equal(d[0], np.float32([1.0, 2.0, np.float32(12.7) / np.float32(127)]))
    assert q[0, 5] == 127 and q[0, 40] == 127 and q[0, 69] == -127
    assert d[1, 0] == np.float32(1.0) / np.float32(127) and d[1, 1] == np.float32(2) / np.float32(127)
    assert q[1, 31] == 127 and q[1, 32] == -127 and d[1, 2] == 0


def test_quantize_non_finite_group_gives_nan_scale():
    x = np.ones((1, 96), np.float32)
    x[0, 3] = np.inf
    x[0, 70] = np.nan
    q, d = oracle.i8_quantize_x(x)
    assert np.isnan(d[0, 0]) and np.isnan(d[0, 2]) and d[0, 1] == np.float32(1) / np.float32(127)
    assert np.all(q[0, :32] == 0) and np.all(q[0, 64:] == 0) and np.all(q[0, 32:64] == 127)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_quantize_properties(seed):
    """Properties of any correct round-to-nearest quantizer with d = m / 127:
    |q| <= 127; the largest |x| of a group maps to +/-127; each code is within
    half a step (plus the float32 quotient's rounding) of x / d; negating x
    negates q; scaling x by a power of two scales d by it and keeps q."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((4, 4096)) * rng.uniform(1e-3, 1e3, (4, 1))).astype(np.float32)
    q, d = oracle.i8_quantize_x(x)
    g = x.reshape(4, 128, 32)
    qg = q.reshape(4, 128, 32).astype(np.float64)
    assert np.all(np.abs(qg) <= 127)
    arg = np.abs(g).argmax(axis=2)
    top = np.take_along_axis(qg, arg[..., None], axis=2)[..., 0]
    assert np.all(np.abs(top) == 127)
    ratio = g.astype(np.float64) / d.astype(np.float64)[..., None]
    assert np.all(np.abs(ratio - qg) <= 0.5 + np.abs(ratio) * 2.0 ** -23)
    qn, dn = oracle.i8_quantize_x(-x)
    assert np.array_equal(qn, -q) and np.array_equal(dn, d)
    q8, d8 = oracle.i8_quantize_x(x * np.float32(8))
    assert np.array_equal(q8, q) and np.array_equal(d8, d * np.float32(8))


def _i8q_inputs(seed, R, C, batch):
    c = synth.i8_inputs(seed, R, C, 110, 124, batch)
    q, d = oracle.i8_quantize_x(c.x)
    return c.w, c.scale, q, d


@pytest.mark.parametrize("R,C,batch", [(7, 64, 1), (13, 96, 3), (5, 70, 2), (3, 16, 8)])
def test_matvec_q8_matches_dense_expansion(R, C, batch):
    w, scale, q, d = _i8q_inputs(R * C + batch, R, C, batch)
    y, mag = oracle.i8_matvec_q8(w, scale, q, d)
    sw = np.repeat(oracle.e8m0_to_f32(scale).astype(np.float64), 16, axis=1)[:, :C]
    W = w.astype(np.float64) * sw
    X = q.astype(np.float64) * np.repeat(d.astype(np.float64), 32, axis=1)[:, :C]
    assert np.allclose(y, X @ W.T, rtol=1e-12, atol=1e-300)
    assert np.allclose(mag, np.abs(X) @ np.abs(W).T, rtol=1e-12, atol=1e-300)


def test_matvec_q8_hand_case():
    """One row of 32 ones (weight scales 1 and 2 for the two 16-column
    groups), q = 1..32, d = 0.5: y = 0.5 * (1 + ... + 16 + 2 (17 + ... + 32))
    = 0.5 * (136 + 2 * 392) = 460."""
    w = np.ones((1, 32), np.int8)
    scale = np.array([[127, 128]], np.uint8)
    q = np.arange(1, 33, dtype=np.int8)[None, :]
    d = np.array([[0.5]], np.float32)
    y, mag = oracle.i8_matvec_q8(w, scale, q, d)
    assert y[0, 0] == 460.0 and mag[0, 0] == 460.0
    y2, _ = oracle.i8_matvec_q8(-w, scale, q, d)
    assert y2[0, 0] == -460.0


def test_matvec_q8_equals_float_i8_matvec_on_dequantized_x():
    """With power-of-two scales d, q * d is exact in float32, and the float
    I8 matvec over x' = q * d must give the same float64 result."""
    rng = np.random.default_rng(12)
    R, C, batch = 9, 160, 2
    c = synth.i8_inputs(4, R, C, 110, 124, batch)
    w, scale = c.w, c.scale
    q = rng.integers(-127, 128, (batch, C)).astype(np.int8)
    d = np.ldexp(1.0, rng.integers(-20, 20, (batch, (C + 31) // 32))).astype(np.float32)
    xp = (q.astype(np.float32) * np.repeat(d, 32, axis=1)[:, :C]).astype(np.float32)
    y, _ = oracle.i8_matvec_q8(w, scale, q, d)
    y_ref, _ = oracle.i8_matvec(w, scale, xp)
    assert np.allclose(y, y_ref, rtol=1e-13, atol=0)


def test_matvec_q8_nan_scale_and_nan_group():
    w, scale, q, d = _i8q_inputs(8, 4, 64, 2)
    scale = scale.copy()
    scale[1, 2] = 255
    d = d.copy()
    d[1, 1] = np.nan
    q = q.copy()
    q[1, 32:64] = 0
    y, _ = oracle.i8_matvec_q8(w, scale, q, d)
    assert np.all(np.isnan(y[:, 1])) and np.all(np.isnan(y[1, :]))
    assert np.all(np.isfinite(y[0, [0, 2, 3]]))


def test_matvec_q8_threaded_equals_single():
    w, scale, q, d = _i8q_inputs(9, 301, 128, 3)
    y1, m1 = oracle.i8_matvec_q8(w, scale, q, d)
    y4, m4 = oracle.i8_matvec_q8(w, scale, q, d, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(m1, m4)
