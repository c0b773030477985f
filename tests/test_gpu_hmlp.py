"""GPU parity of hadamard_mlp: the Hadamard MLP block of needle.js "Inference
engine, part 2: kernels and token step", section 8.

The kernel stores every value as float32 exactly as the page's Float32Array
code does, except that silu is evaluated in float32 where the page uses
float64; so the outputs are compared with the oracle (page staging, float64
silu) within 1e-5 * A, A = |d3| / sqrt(D) * sum |silu| + |residual| + |u|
(float32 silu error is a few ulps of each silu value, about 1e-6 relative
after the second transform, and the two transforms' own roundings agree).
Cases where silu is exact (zero gate, identity range) are compared bit for
bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_matvec_gb300 import qmv, synth

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-30


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qmv.load()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(f, with_res=True, with_u=True, guard=64):
    """Call through the C ABI into a NaN-filled buffer with guard elements
    past the [batch, n] result."""
    batch, n = f.x.shape
    buf = torch.full((batch * n + guard,), float("nan"), device="cuda")
    out = buf[: batch * n].view(batch, n)
    res = dev(f.residual) if with_res else None
    u = dev(f.u) if with_u else None
    qmv.hadamard_mlp_t(dev(f.x), f.D, dev(f.d1), dev(f.d2), dev(f.d3), res, u, out=out)
    torch.cuda.synchronize()
    assert torch.isnan(buf[batch * n:]).all(), "write past the result"
    return out.cpu().numpy()


def check(f, with_res=True, with_u=True):
    got = run(f, with_res, with_u)
    ref, mag = oracle.hadamard_mlp(f.x, f.D, f.d1, f.d2, f.d3,
                                   f.residual if with_res else None, f.u if with_u else None)
    both_nan = np.isnan(got) & np.isnan(ref)
    bad = ~(both_nan | (np.abs(got - ref) <= REL * mag + ABS))
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])
    return got, ref


@pytest.mark.parametrize("D", [1, 2, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384,
                               32768])
def test_hmlp_all_dimensions(D):
    for n, batch in ((D, 1), (max(1, D - 3), 3), (1, 2)):
        check(synth.hmlp_inputs(D + n + batch, n, D, batch))


@pytest.mark.parametrize("batch", [1, 2, 5, 8])
@pytest.mark.parametrize("terms", [(True, True), (True, False), (False, True), (False, False)])
def test_hmlp_batch_and_epilogue_terms(batch, terms):
    check(synth.hmlp_inputs(40 + batch, 500, 2048, batch), *terms)


@pytest.mark.parametrize("name", ["hmlp_512", "hmlp_2048"])
def test_hmlp_workloads(name):
    for batch in synth.WORKLOADS[name]["batch"]:
        check(synth.workload_inputs(name, batch=batch))


def test_hmlp_zero_gate_is_residual_minus_u_exactly():
    f = synth.hmlp_inputs(3, 500, 2048, 4)
    f.d2[:] = 0
    got = run(f)
    assert np.array_equal(got, f.residual - f.u)


@pytest.mark.parametrize("k", [0, 7, 1000])
def test_hmlp_identity_silu_collapses_exactly(k):
    """D = 1024, x = 2 e_k, d1 = 1: the first normalised transform is
    H[:, k] / 16 exactly.  With d2 = 1024 H[:, k] every silu input is +64,
    where silu is the identity in float32 and float64 alike, and the second
    transform collapses the constant 64 onto output 0: 64 sqrt(D) d3[0]
    there and zero elsewhere."""
    D = 1024
    f = synth.hmlp_inputs(11, D, D, 1)
    i = np.arange(D)
    col = np.where(np.vectorize(lambda v: bin(v).count("1") % 2)(i & k) == 0, 1.0, -1.0)
    f.x[:] = 0
    f.x[0, k] = 2.0
    f.d1[:] = 1.0
    f.d2[:] = (1024.0 * col).astype(np.float32)
    f.residual[:] = 0.5
    f.u[:] = 0.25
    got = run(f)
    want = np.full(D, np.float32(0.5) - np.float32(0.25), dtype=np.float32)
    want[0] = (np.float32(0.5) + np.float32(64.0 * math.sqrt(D)) * f.d3[0]) - np.float32(0.25)
    assert np.array_equal(got[0], want)
    ref, _ = oracle.hadamard_mlp(f.x, D, f.d1, f.d2, f.d3, f.residual, f.u)
    assert np.array_equal(ref[0], want)


def test_hmlp_nan_and_padding():
    f = synth.hmlp_inputs(4, 300, 512, 2)
    f.x[1, 17] = np.nan
    got, _ = check(f)
    assert np.all(np.isfinite(got[0])) and np.all(np.isnan(got[1]))
    g = synth.hmlp_inputs(5, 300, 512, 1)
    g.d1[400] = np.inf  # in the padding: 0 * inf
    got, _ = check(g)
    assert np.all(np.isnan(got))


def test_hmlp_deterministic():
    f = synth.hmlp_inputs(6, 512, 4096, 8)
    a, b = run(f), run(f)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_hmlp_validation_on_device_tensors():
    f = synth.hmlp_inputs(7, 64, 64, 1)
    x = dev(f.x)
    with pytest.raises(qmv.QmvError) as e:
        qmv.hadamard_mlp_t(x, 64, dev(f.d1), dev(f.d2), dev(f.d3), out=x)
    assert e.value.status == 8
    st = qmv.hadamard_mlp(x.data_ptr(), 64, 48, x.data_ptr(), x.data_ptr(), x.data_ptr(), 0, 0,
                          1, x.data_ptr())
    assert st == 2
