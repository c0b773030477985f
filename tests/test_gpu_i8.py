"""GPU parity of i8_matvec (ds4f-disk issue #6, step 4: int8 weights with
per-16 E8M0 group scales) against the float64 oracle."""
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
    ok = (np.isnan(y) & np.isnan(ref)) | (np.abs(y - ref) <= REL * mag + ABS)
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


def test_i8_head_full_size_sampled_rows():
    f = synth.i8_inputs(7, 245760, 4096, 110, 124, batch=8)
    w, s = dev(f.w), dev(f.scale)
    for batch in (1, 8):
        x = f.x[:batch]
        y = qmv.i8_matvec_t(w, s, dev(x)).cpu().numpy()
        rng = np.random.default_rng(batch)
        for r in np.unique(np.concatenate([rng.integers(0, f.R, 200), [0, f.R - 1]])):
            ref, mag = oracle.i8_matvec(f.w, f.scale, x, rows=(int(r), int(r) + 1))
            assert np.all(np.abs(y[:, r] - ref[:, r]) <= REL * mag[:, r] + ABS)


def test_i8_deterministic():
    f = synth.i8_inputs(43, 131072, 64, 110, 124, batch=1)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    a = qmv.i8_matvec_t(w, s, x)
    b = qmv.i8_matvec_t(w, s, x)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
