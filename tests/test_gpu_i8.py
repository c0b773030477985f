"""GPU parity of i8_matvec (ds4f-disk issue #6, step 4: int8 weights with
per-16 E8M0 group scales) against the float64 oracle.

Matrices with many rows run on the streaming kernels: up to batch 4 the
integer-dot kernel (x in fixed-point limbs per 16-column group, exact int32
sums), above it the float32 kernel; small matrices run on the small-matrix
kernel (batch 1 at 4096..16384 columns: the split-row kernel).  The tests
below cover each route."""
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


def check(f, x=None, rows=None):
    x = f.x if x is None else x
    y = qmv.i8_matvec_t(dev(f.w), dev(f.scale), dev(x))
    torch.cuda.synchronize()
    y = y.cpu().numpy().astype(np.float64)
    ref, mag = oracle.i8_matvec(f.w, f.scale, x, threads=8)
    with np.errstate(invalid="ignore"):  # inf - inf where both sides are infinite
        ok = (np.isnan(y) & np.isnan(ref)) | (y == ref) | (np.abs(y - ref) <= REL * mag + ABS)
    assert ok.all(), (np.argwhere(~ok)[:3], int((~ok).sum()))
    return y


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("R,C", [(1, 16), (1000, 4096), (4096, 4096), (150001, 32), (33, 100),
                                 (17, 7), (300, 2048)])
def test_i8_shapes(batch, R, C):
    check(synth.i8_inputs(R + C + batch, R, C, 100, 130, batch=batch))


def test_i8_extreme_scales_and_nan():
    f = synth.i8_inputs(41, 500, 256, 0, 180, batch=2)  # 2^-127 (subnormal) up to 2^53
    check(f)
    f.scale[7, 3] = 255
    y = check(f)
    assert np.isnan(y[:, 7]).all() and not np.isnan(np.delete(y, 7, axis=1)).any()


def test_i8_extreme_weights():
    f = synth.i8_inputs(42, 64, 64, 127, 127, batch=1)
    f.w[0] = -128
    f.w[1] = 127
    check(f)


def test_i8_head_full_size_every_row():
    """All 245760 rows of the I8 head at batch 1 (integer-dot kernel) and 8
    (tensor-core kernel) against the threaded oracle."""
    f = synth.i8_inputs(7, 245760, 4096, 110, 124, batch=8)
    w, s = dev(f.w), dev(f.scale)
    ref, mag = oracle.i8_matvec(f.w, f.scale, f.x, threads=os.cpu_count() or 8)
    for batch in (1, 8):
        y = qmv.i8_matvec_t(w, s, dev(f.x[:batch])).cpu().numpy().astype(np.float64)
        ok = np.abs(y - ref[:batch]) <= REL * mag[:batch] + ABS
        assert ok.all(), (batch, np.argwhere(~ok)[:3], int((~ok).sum()))


def test_i8_deterministic():
    f = synth.i8_inputs(43, 131072, 64, 110, 124, batch=1)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    a = qmv.i8_matvec_t(w, s, x)
    b = qmv.i8_matvec_t(w, s, x)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


# Enough rows for the streaming kernels (more than four waves of tiles).
STREAM_R = 120000


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 6])
@pytest.mark.parametrize("C", [528, 1040])
def test_i8_streaming_ragged_steps(batch, C):
    """C = 528 / 1040: 33 / 65 chunks, so the last 512-column step is ragged."""
    check(synth.i8_inputs(C + batch, STREAM_R, C, 100, 130, batch=batch))


def test_i8_streaming_nonfinite_x_groups():
    f = synth.i8_inputs(50, STREAM_R, 256, 110, 124, batch=3)
    f.x[0, 37] = np.inf    # group 2 of vector 0
    f.x[1, 200] = np.nan   # group 12 of vector 1
    f.x[2, 5] = -np.inf
    f.x[2, 6] = np.inf     # -inf and +inf in one group of vector 2
    y = check(f)
    assert np.isnan(y[1]).all()
    # vector 2: NaN where the two infinite products have opposite signs,
    # +-inf where they agree
    assert not np.isfinite(y[2]).any() and np.isnan(y[2]).any() and np.isinf(y[2]).any()
    assert np.isinf(y[0]).any()


def test_i8_streaming_wide_dynamic_range_in_groups():
    """x spans six decades inside each 16-column group."""
    f = synth.i8_inputs(51, STREAM_R, 512, 110, 124, batch=2)
    rng = np.random.default_rng(51)
    f.x *= (10.0 ** rng.uniform(-3, 3, f.x.shape)).astype(np.float32)
    check(f)


@pytest.mark.parametrize("mult", [1e30, 1e-30, 0.0])
def test_i8_streaming_extreme_magnitudes(mult):
    f = synth.i8_inputs(52, STREAM_R, 256, 120, 134, batch=2)
    f.x = (f.x * np.float32(mult)).astype(np.float32)
    f.x[1, 16:48] = 0.0  # two all-zero groups
    y = qmv.i8_matvec_t(dev(f.w), dev(f.scale), dev(f.x)).cpu().numpy().astype(np.float64)
    ref, mag = oracle.i8_matvec(f.w, f.scale, f.x, threads=8)
    assert np.all(np.abs(y - ref) <= REL * mag), "relative bound without the absolute term"
    if mult == 0.0:
        assert not y.any()


def test_i8_streaming_integer_inputs_are_exact():
    """Small-integer x and unit scales: every partial sum is an integer below
    2^24, so both float32 accumulation and the integer dots are exact."""
    f = synth.i8_inputs(53, STREAM_R, 512, 127, 127, batch=2)
    rng = np.random.default_rng(53)
    f.x = rng.integers(-8, 9, f.x.shape).astype(np.float32)
    y = qmv.i8_matvec_t(dev(f.w), dev(f.scale), dev(f.x)).cpu().numpy().astype(np.float64)
    ref, _ = oracle.i8_matvec(f.w, f.scale, f.x, threads=8)
    assert np.array_equal(y, ref)


def test_i8_streaming_extreme_scales():
    f = synth.i8_inputs(54, STREAM_R, 256, 0, 180, batch=2)
    f.scale[7, 3] = 255
    y = check(f)
    assert np.isnan(y[:, 7]).all()


# ---------------------------------------------------------------------------
# Split-row kernel: batch 1, 4096..16384 columns, every T-row tile (T = 8, 4,
# 2 for up to 4096, 8192, 16384 columns) resident at once
# ---------------------------------------------------------------------------

def kernel_names(fn):
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    names = []
    for _ in range(2):  # the first profiling session of a process may record nothing
        with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
        if names:
            break
    if not names:
        pytest.skip("the profiler recorded no kernels on this box")
    return names


@pytest.mark.parametrize("R,C", [(1, 4096), (7, 4096), (9, 4096), (4100, 4096), (1001, 8192),
                                 (3, 12288), (611, 16384), (5, 4080), (4, 16400)])
def test_i8_split_shapes(R, C):
    check(synth.i8_inputs(R * 3 + C, R, C, 100, 130, batch=1))


def test_i8_split_nonfinite_x_and_nan_scale():
    f = synth.i8_inputs(44, 300, 8192, 110, 124, batch=1)
    f.scale[5, 100] = 255
    y = check(f)
    assert np.isnan(y[0, 5]) and not np.isnan(np.delete(y, 5, axis=1)).any()
    f.x[0, 3000] = np.inf
    y = check(f)
    assert not np.isfinite(y).all()


def test_i8_split_sees_activations_written_just_before():
    """Weights and scales are loaded before the dependency wait, x after it."""
    f = synth.i8_inputs(45, 4096, 4096, 110, 124, batch=4)
    w, s, src = dev(f.w), dev(f.scale), dev(f.x)
    x = torch.zeros((1, 4096), device="cuda")
    ys = []
    for v in range(4):
        x.copy_(src[v:v + 1])  # a kernel on the same stream
        ys.append(qmv.i8_matvec_t(w, s, x))
    torch.cuda.synchronize()
    ref, mag = oracle.i8_matvec(f.w, f.scale, f.x, threads=8)
    for v in range(4):
        y = ys[v].cpu().numpy()[0].astype(np.float64)
        assert (np.abs(y - ref[v]) <= REL * mag[v] + ABS).all()


@pytest.mark.parametrize("R,C,batch,expect", [
    (4096, 4096, 1, True), (611, 16384, 1, True), (1000, 2048, 1, False), (4, 16400, 1, False),
    (4096, 4096, 2, False), (65536, 4096, 1, False)])
def test_i8_split_kernel_is_the_one_launched(R, C, batch, expect):
    w = torch.zeros((R, C), dtype=torch.int8, device="cuda")
    s = torch.full((R, C // 16), 127, dtype=torch.uint8, device="cuda")
    x = torch.ones((batch, C), device="cuda")
    names = kernel_names(lambda: qmv.i8_matvec_t(w, s, x))
    assert any("i8_split_kernel" in n for n in names) == expect, names
