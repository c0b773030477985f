"""GPU parity of the CQ matrix-set entry points (needle.js "part 2", section 6:
one prepared activation reused by several matrices; section 7: Q, K and V of
one input) and of prepare fused into the matvec.

Every result must be bitwise equal to running cq_prepare and cq_matvec per
matrix (same kernels, same arithmetic), and within the matvec tolerance of
the float64 oracle.
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


def make_set(outputs, inp, group, bits, batch, seed=0):
    """Matrices sharing input width, group, bits and one codebook tensor."""
    cs = [synth.cq_inputs(seed + 11 * i + 1, out, inp, group, bits, batch=batch)
          for i, out in enumerate(outputs)]
    cb = torch.from_numpy(cs[0].codebook).cuda()
    mats = [qmv.CQMatrix(c.output, c.input, c.input_padded, c.group, c.bits,
                         torch.from_numpy(c.packed).cuda(),
                         torch.from_numpy(c.norms.view(np.int16)).cuda(), cb) for c in cs]
    return cs, mats, torch.from_numpy(cs[0].x).cuda()


def separate(mats, x):
    p = qmv.cq_prepare_t(mats[0], x)
    return p, [qmv.cq_matvec_t(m, p) for m in mats]


def bits_eq(a, b):
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


SETS = [
    ((32768, 4096, 1000), 500, 128, 2, 1),   # 2-bit table kernel, vocabulary-like plus QKV-like
    ((512, 512, 512), 512, 64, 2, 1),        # three equal matrices (phiPre/phiPost/phiResidual)
    ((700, 3, 129), 500, 128, 4, 1),         # general kernel
    ((300, 2048), 512, 64, 3, 4),            # batch 4
    ((64, 65, 1, 200, 7, 33, 90, 128), 100, 32, 5, 8),  # 8 matrices, batch 8
    ((256, 0, 100), 512, 128, 2, 1),         # an empty matrix in the set
    ((40, 50), 6, 2, 2, 3),                  # group 2
]


@pytest.mark.parametrize("outputs,inp,group,bits,batch", SETS)
def test_matvec_multi_equals_per_matrix_calls(outputs, inp, group, bits, batch):
    cs, mats, x = make_set(outputs, inp, group, bits, batch)
    p, ref = separate(mats, x)
    ys = qmv.cq_matvec_multi_t(mats, p)
    torch.cuda.synchronize()
    for y, r in zip(ys, ref):
        assert bits_eq(y, r)


@pytest.mark.parametrize("outputs,inp,group,bits,batch", SETS)
def test_prepare_matvec_fused_equals_separate(outputs, inp, group, bits, batch):
    cs, mats, x = make_set(outputs, inp, group, bits, batch, seed=5)
    p, ref = separate(mats, x)
    prepared = torch.full_like(p, float("nan"))
    ys = qmv.cq_prepare_matvec_t(mats, x, prepared=prepared)
    ys2 = qmv.cq_prepare_matvec_t(mats, x)  # without storing the prepared vector
    torch.cuda.synchronize()
    assert bits_eq(prepared, p)
    for y, y2, r in zip(ys, ys2, ref):
        assert bits_eq(y, r) and bits_eq(y2, r)


def test_fused_set_against_oracle():
    cs, mats, x = make_set((32768, 1024), 500, 128, 2, 1, seed=9)
    ys = qmv.cq_prepare_matvec_t(mats, x)
    torch.cuda.synchronize()
    p = oracle.cq_prepare(cs[0].x, cs[0].input_padded, cs[0].group, mode="f32")
    for c, y in zip(cs, ys):
        om = oracle.CQMatrix(c.output, c.input, c.input_padded, c.group, c.bits, c.packed,
                             c.norms, cs[0].codebook)
        ref, mag = om.matvec(p, threads=8)
        assert np.all(np.abs(y.cpu().numpy() - ref) <= REL * mag + ABS)


def test_wide_groups_run_as_two_launches():
    cs, mats, x = make_set((100, 37), 4000, 2048, 3, 2, seed=13)
    p, ref = separate(mats, x)
    prepared = torch.empty_like(p)
    ys = qmv.cq_prepare_matvec_t(mats, x, prepared=prepared)
    torch.cuda.synchronize()
    assert bits_eq(prepared, p)
    for y, r in zip(ys, ref):
        assert bits_eq(y, r)
    with pytest.raises(qmv.QmvError) as e:  # two launches need the prepared buffer
        qmv.cq_prepare_matvec_t(mats, x)
    assert e.value.status == 1


def launches(fn):
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


def test_fused_prepare_is_one_launch_with_or_without_a_buffer():
    """Wherever the activation fits on chip, cq_prepare_matvec is one launch,
    whether or not the prepared vector is also stored; the results are the
    same bits as prepare + one call per matrix."""
    for bits, seed in ((4, 17), (2, 18)):
        cs, mats, x = make_set((2048, 2048, 2048), 512, 64, bits, 1, seed=seed)
        p, ref = separate(mats, x)
        prepared = torch.empty_like(p)
        assert len(launches(lambda: qmv.cq_prepare_matvec_t(mats, x, prepared=prepared))) == 1
        assert len(launches(lambda: qmv.cq_prepare_matvec_t(mats, x))) == 1
        ys = qmv.cq_prepare_matvec_t(mats, x, prepared=prepared)
        ys2 = qmv.cq_prepare_matvec_t(mats, x)
        torch.cuda.synchronize()
        assert bits_eq(prepared, p)
        for y, y2, r in zip(ys, ys2, ref):
            assert bits_eq(y, r) and bits_eq(y2, r)
