"""f8_matvec_argmax_noalloc: the fused head argmax for callers that cannot
allocate device memory (their memory pool owns the device, or their plug-in
interface offers no workspace).  It must give the same answers as
f8_matvec_argmax with a caller workspace, call after call, although every
call reuses the same scratch array inside the library.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_matvec_gb300 import qmv, synth

pytestmark = pytest.mark.gpu

REL, ABS = 1e-4, 1e-6


@pytest.mark.parametrize("batch,R,C,SR,SC", [(1, 40960, 4096, 320, 32), (4, 3001, 4096, 7, 32),
                                             (8, 513, 100, 3, 7)])
def test_noalloc_argmax_matches_workspace_variant_twice(batch, R, C, SR, SC):
    """Two calls in a row through the C ABI: the index, the value and y are
    bit for bit those of f8_matvec_argmax with a caller workspace (the same
    kernels run), and y is within the matvec tolerance of the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = synth.f8_inputs(R + batch, R, C, SR, SC, 118, 132, batch=batch)
    w, s, x = (torch.from_numpy(a).cuda() for a in (f.w, f.scale, f.x))
    sh = torch.cuda.current_stream().cuda_stream
    ref_y = torch.empty((batch, R), device="cuda")
    ref_i, ref_v = qmv.f8_matvec_argmax_t(w, s, x, y=ref_y)
    ora_y, ora_mag = oracle.f8_matvec(f.w, f.scale, f.x, threads=os.cpu_count() or 8)
    for call in range(2):
        y = torch.full((batch, R), float("nan"), device="cuda")
        idx = torch.full((batch,), -7, dtype=torch.int64, device="cuda")
        val = torch.full((batch,), float("nan"), device="cuda")
        st = qmv.f8_matvec_argmax_noalloc(w.data_ptr(), R, C, s.data_ptr(), SR, SC, x.data_ptr(),
                                          batch, y.data_ptr(), idx.data_ptr(), val.data_ptr(), sh)
        assert st == 0, qmv.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_i), call
        assert torch.equal(val.view(torch.int32), ref_v.view(torch.int32)), call
        assert torch.equal(y.view(torch.int32), ref_y.view(torch.int32)), call
        yh = y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(yh - ora_y) <= REL * ora_mag + ABS), call
        # and without storing y
        idx.fill_(-7)
        val.fill_(float("nan"))
        st = qmv.f8_matvec_argmax_noalloc(w.data_ptr(), R, C, s.data_ptr(), SR, SC, x.data_ptr(),
                                          batch, 0, idx.data_ptr(), val.data_ptr(), sh)
        assert st == 0
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_i), call
        assert torch.equal(val.view(torch.int32), ref_v.view(torch.int32)), call


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = synth.f8_inputs(3, 64, 64, 1, 1, 127, 127)
    w, s, x = (torch.from_numpy(a).cuda() for a in (f.w, f.scale, f.x))
    idx = torch.empty(9, dtype=torch.int64, device="cuda")
    val = torch.empty(9, device="cuda")
    st = qmv.f8_matvec_argmax_noalloc(w.data_ptr(), 64, 64, s.data_ptr(), 1, 1, x.data_ptr(), 9,
                                      0, idx.data_ptr(), val.data_ptr())
    assert st == 5  # QMV_ERR_BATCH
