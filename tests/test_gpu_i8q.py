"""GPU parity of i8_quantize_x and i8_matvec_q8 (Mnemonic "In the browser",
"Dot products and math": int8 activations quantized per group of 32, exact
int32 dot sums, then the group scales; over the I8 weights of ds4f-disk
issue #6, step 4) against the oracle.

The quantizer decides integers from floats, so its codes and scales must be
bit-identical to the oracle's (both divide in IEEE float32 and round to
nearest even).  The matvec's inputs come from the oracle's quantizer, never
from the GPU's; its outputs must be within 1e-4 * sum_c |w s q d| + 1e-6 of
the oracle's float64 value.  The shapes cover the streaming kernel (many
rows), the small-matrix kernel (few rows), the general kernel (C % 16 != 0),
the tensor-core route of large matrices at batch 4-8, and ragged tails
(C % 32 == 16, a short last tile of rows)."""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_matvec_gb300 import qmv, synth

pytestmark = pytest.mark.gpu

REL, ABS = 1e-4, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qmv.load()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def within(y, ref, mag):
    with np.errstate(invalid="ignore"):
        return (np.isnan(y) & np.isnan(ref)) | (y == ref) | (np.abs(y - ref) <= REL * mag + ABS)


def check_quantize(x):
    q, d = qmv.i8_quantize_x_t(dev(x))
    torch.cuda.synchronize()
    q, d = q.cpu().numpy(), d.cpu().numpy()
    q_ref, d_ref = oracle.i8_quantize_x(x)
    assert np.array_equal(q, q_ref), (np.argwhere(q != q_ref)[:3], int((q != q_ref).sum()))
    assert np.array_equal(d.view(np.uint32), d_ref.view(np.uint32))
    return q, d


def check_matvec(f, q, d, threads=8):
    y = qmv.i8_matvec_q8_t(dev(f.w), dev(f.scale), dev(q), dev(d))
    torch.cuda.synchronize()
    y = y.cpu().numpy().astype(np.float64)
    ref, mag = oracle.i8_matvec_q8(f.w, f.scale, q, d, threads=threads)
    ok = within(y, ref, mag)
    assert ok.all(), (np.argwhere(~ok)[:3], int((~ok).sum()))
    return y


@pytest.mark.parametrize("batch", [1, 3, 8])
@pytest.mark.parametrize("C", [1, 16, 31, 32, 48, 100, 4096, 4112])
def test_quantize_bit_exact(batch, C):
    rng = np.random.default_rng(C * 10 + batch)
    x = (rng.standard_normal((batch, C)) * rng.uniform(1e-3, 1e3, (batch, 1))).astype(np.float32)
    check_quantize(x)


def test_quantize_edge_values():
    """Ties, zero groups, subnormal and underflowing scales, Inf and NaN."""
    x = np.zeros((2, 256), np.float32)
    x[0, :8] = [127, 0.5, 1.5, 2.5, -0.5, -1.5, -63.5, 3.5]            # d = 1: exact ties
    x[0, 32] = float.fromhex("0x1.7d8af0p+1")                           # tie after division
    x[0, 33] = float.fromhex("-0x1.6401a4p+1")
    x[0, 64] = 2.0 ** -140                                              # subnormal d, clamp
    x[0, 96] = -(2.0 ** -149)                                           # d underflows to 0
    x[0, 128] = np.inf
    x[0, 160], x[0, 161] = np.nan, 1.0
    x[1, :] = np.float32(3.4e38) * np.sign(np.arange(256) - 100.5)      # largest magnitudes
    x[1, 200:232] = np.float32(1e-40)                                   # subnormal inputs
    q, d = check_quantize(x)
    assert q[0, 64] == 127 and d[0, 3] == 0 and np.isnan(d[0, 4]) and np.isnan(d[0, 5])


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("R,C", [(1, 16), (1000, 4096), (4096, 4096), (150001, 32), (33, 100),
                                 (17, 7), (300, 2048), (2049, 208)])
def test_matvec_q8_shapes(batch, R, C):
    f = synth.i8_inputs(R + C + batch, R, C, 100, 130, batch=batch)
    q, d = oracle.i8_quantize_x(f.x)
    check_matvec(f, q, d)


def test_matvec_q8_extreme_scales_codes_and_nan():
    f = synth.i8_inputs(51, 700, 256, 0, 180, batch=3)  # weight scales 2^-127 .. 2^53
    rng = np.random.default_rng(5)
    q = rng.integers(-128, 128, (3, 256)).astype(np.int8)  # -128 included
    d = rng.uniform(1e-30, 1e10, (3, 8)).astype(np.float32)
    check_matvec(f, q, d)
    f.scale[9, 2] = 255
    d[1, 3] = np.nan
    y = check_matvec(f, q, d)
    assert np.isnan(y[:, 9]).all() and np.isnan(y[1]).all()
    assert not np.isnan(np.delete(y[[0, 2]], 9, axis=1)).any()


@pytest.mark.parametrize("batch,C", [(4, 256), (5, 1024), (8, 4096)])
def test_matvec_q8_tensor_core_route(batch, C):
    """Matrices large enough to stream take the tensor-core kernel from batch 4
    on (q * d split into f16 hi + lo); weight scales outside the range it folds
    exactly (2^-24 .. 2^5), the NaN scale code and a NaN activation scale take
    its exact per-element fix-up."""
    R = 50000
    f = synth.i8_inputs(60 + batch, R, C, 110, 124, batch=batch)
    q, d = oracle.i8_quantize_x(f.x)
    check_matvec(f, q, d)
    f.scale[5, 0] = 140          # 2^13: outside the folded range
    f.scale[7, 1] = 90           # 2^-37
    f.scale[9, 2] = 255          # NaN
    d = d.copy()
    d[batch - 1, 1] = np.nan
    y = check_matvec(f, q, d)
    assert np.isnan(y[:, 9]).all() and np.isnan(y[batch - 1]).all()
    assert np.isfinite(y[:batch - 1, 5]).all() and np.isfinite(y[:batch - 1, 7]).all()


def test_quantize_then_matvec_composite():
    """x -> GPU quantize -> GPU matvec against x -> oracle quantize -> oracle
    matvec (the codes agree bit for bit, so the two chains differ only by the
    matvec's float32 accumulation)."""
    f = synth.i8_inputs(52, 20000, 1024, 110, 124, batch=4)
    xq, xs = qmv.i8_quantize_x_t(dev(f.x))
    y = qmv.i8_matvec_q8_t(dev(f.w), dev(f.scale), xq, xs).cpu().numpy().astype(np.float64)
    q, d = oracle.i8_quantize_x(f.x)
    ref, mag = oracle.i8_matvec_q8(f.w, f.scale, q, d, threads=8)
    assert within(y, ref, mag).all()


def test_matvec_q8_head_full_size_every_row():
    """The 245760 x 4096 head at batch 1 and 8, every row against the
    threaded oracle."""
    f = synth.i8_inputs(7, 245760, 4096, 110, 124, batch=8)
    w, s = dev(f.w), dev(f.scale)
    q, d = oracle.i8_quantize_x(f.x)
    ref, mag = oracle.i8_matvec_q8(f.w, f.scale, q, d, threads=os.cpu_count() or 8)
    for batch in (1, 8):
        y = qmv.i8_matvec_q8_t(w, s, dev(q[:batch]), dev(d[:batch])).cpu().numpy()
        ok = within(y.astype(np.float64), ref[:batch], mag[:batch])
        assert ok.all(), (batch, np.argwhere(~ok)[:3], int((~ok).sum()))


def test_matvec_q8_deterministic():
    f = synth.i8_inputs(53, 131072, 64, 110, 124, batch=2)
    q, d = oracle.i8_quantize_x(f.x)
    args = (dev(f.w), dev(f.scale), dev(q), dev(d))
    a = qmv.i8_matvec_q8_t(*args)
    b = qmv.i8_matvec_q8_t(*args)
    assert torch.equal(a, b)
