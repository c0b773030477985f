"""GPU parity of f8_matvec_argmax: the head matvec with fused greedy selection
(ds4f-disk issue #6, work item 3 and step 3).

The selection is an integer decided by floating point, so both sides decide
in the kernel's precision: the returned index must be the oracle's argmax of
the float32 y the same call writes, and y itself must match the float64
oracle within the matvec tolerance.
"""
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


def run(f, batch=None):
    x = f.x if batch is None else f.x[:batch]
    w, s, xd = dev(f.w), dev(f.scale), dev(x)
    y = torch.full((x.shape[0], f.R), float("nan"), device="cuda")
    idx, val = qmv.f8_matvec_argmax_t(w, s, xd, y=y)
    idx2, val2 = qmv.f8_matvec_argmax_t(w, s, xd)  # without storing y
    torch.cuda.synchronize()
    return x, y.cpu().numpy(), idx.cpu().numpy(), val.cpu().numpy(), idx2.cpu().numpy(), \
        val2.cpu().numpy()


def check(f, batch=None, full_oracle=True):
    x, y, idx, val, idx2, val2 = run(f, batch)
    assert np.array_equal(idx, oracle.argmax_rows(y))
    assert np.array_equal(idx, idx2)
    picked = y[np.arange(len(idx)), idx]
    assert np.array_equal(val.view(np.uint32), picked.view(np.uint32))
    assert np.array_equal(val2.view(np.uint32), val.view(np.uint32))
    if full_oracle:
        ref, mag = oracle.f8_matvec(f.w, f.scale, x, threads=8)
        both_nan = np.isnan(y) & np.isnan(ref)
        assert np.all(both_nan | (np.abs(y - ref) <= REL * mag + ABS))
    return idx, y


@pytest.mark.parametrize("batch", [1, 2, 3, 8])
@pytest.mark.parametrize("R,C,SR,SC", [
    (1, 16, 1, 1), (1000, 4096, 8, 32), (150001, 32, 7, 2), (64, 100, 3, 7), (257, 4096, 5, 3)])
def test_argmax_shapes(batch, R, C, SR, SC):
    check(synth.f8_inputs(R * 7 + C + batch, R, C, SR, SC, 110, 140, batch=batch))


def test_argmax_ties_pick_the_lowest_row():
    f = synth.f8_inputs(31, 3000, 256, 3, 2, 127, 127, batch=2)
    f.w[[17, 1500, 2999]] = 0x7E  # three identical rows of the largest code
    f.x[:] = np.abs(f.x)           # so those rows are the maximum
    idx, y = check(f)
    assert list(idx) == [17, 17]
    assert y[0, 17] == y[0, 1500] == y[0, 2999]


def test_argmax_nan_rows_win_first_nan():
    f = synth.f8_inputs(32, 5000, 512, 10, 4, 120, 130, batch=1)
    f.scale[4, 1] = 255  # rows of scale row 4 are NaN: rows 2000..2499
    idx, y = check(f)
    assert idx[0] == 2000 and np.isnan(y[0, 2000])


def test_argmax_all_equal_minus_inf_free_case():
    # every row identical: the lowest row wins
    f = synth.f8_inputs(33, 777, 64, 1, 1, 127, 127, batch=1)
    f.w[:] = f.w[0]
    idx, _ = check(f)
    assert idx[0] == 0


@pytest.mark.parametrize("batch", [1, 8])
def test_argmax_head_full_size(batch):
    f = synth.f8_inputs(5, 245760, 4096, 1920, 32, 118, 132, batch=8)
    x, y, idx, val, idx2, _ = run(f, batch)
    assert np.array_equal(idx, oracle.argmax_rows(y)) and np.array_equal(idx, idx2)
    for v in range(batch):
        r = int(idx[v])
        ref, mag = oracle.f8_matvec(f.w, f.scale, x, rows=(r, r + 1))
        assert np.all(np.abs(y[:, r] - ref[:, r]) <= REL * mag[:, r] + ABS)


def test_argmax_validation():
    f = synth.f8_inputs(3, 64, 64, 1, 1, 127, 127)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    small = torch.empty(qmv.f8_argmax_workspace_bytes(1) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qmv.QmvError) as e:
        qmv.f8_matvec_argmax_t(w, s, x, workspace=small)
    assert e.value.status == 2
    ws = torch.empty(qmv.f8_argmax_workspace_bytes(1) + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qmv.QmvError) as e:
        qmv.f8_matvec_argmax_t(w, s, x, workspace=ws[8:])
    assert e.value.status == 6
    idx = torch.empty(1, dtype=torch.int64, device="cuda")
    val = torch.empty(1, device="cuda")
    st = qmv.f8_matvec_argmax(w.data_ptr(), 64, 64, s.data_ptr(), 1, 1, x.data_ptr(), 1, 0,
                              idx.data_ptr(), val.data_ptr(), w.data_ptr(), 1 << 20)
    assert st == 8  # workspace overlapping the weights
