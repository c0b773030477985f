"""GPU parity of the fifth-generation tensor-core F8 kernel (batch 5..8).

f8_matvec at batch 5..8 goes to tcgen05.mma kind::f8f6f4 when C is a
multiple of 128 up to 4096, the matrix has at least 3 64-row units per SM,
every scale block starts on a multiple of 128 columns and 64 rows, and w and
x are 16-byte aligned: the raw E4M3 weights are the wide MMA operand
(TMA-streamed, 128-byte swizzle) and x enters as eight E4M3 pieces per
128-column block.  The bar is the matvec tolerance of ds4f-disk issue #6
step 1's definition, |y - y_oracle| <= 1e-4 * sum_c |w * s * x| + 1e-6,
against the float64 oracle.  The row counts here start at that size
threshold, R0 = 3 * 64 * (SMs of the device).

Cases: every batch 5..8; a ragged last 64-row unit; 64-row and 128-row
scale blocks; one 128-column block; blocks with unequal numbers of units
(and short last tiles); activations with a wide dynamic range inside a
block, huge, tiny, subnormal and zero; Inf / NaN in x; saturated E4M3 codes
and NaN scales; subnormal and large scales; integer inputs, where the result
is exact; the fused argmax and top-k forms (the argmax without y keeping its
logits in a large workspace); determinism; that this kernel is
the one launched, that shapes outside its conditions go elsewhere, and that
none of its waits ran out of time.
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


def r0():
    """The fewest rows the kernel takes: 3 64-row units per SM."""
    return 3 * 64 * torch.cuda.get_device_properties(0).multi_processor_count


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(f, x=None):
    x = f.x if x is None else x
    y = qmv.f8_matvec_t(dev(f.w), dev(f.scale), dev(x))
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def check(f, abs_tol=ABS):
    y = run(f)
    ref, mag = oracle.f8_matvec(f.w, f.scale, f.x, threads=8)
    with np.errstate(invalid="ignore"):  # inf - inf where both sides are infinite
        ok = (np.isnan(y) & np.isnan(ref)) | (y == ref) | (np.abs(y - ref) <= REL * mag + abs_tol)
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError("mismatch at %s: gpu %r oracle %r bound %r (%d bad)" % (
            i, y[i], ref[i], REL * mag[i] + abs_tol, int((~ok).sum())))
    return y


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


@pytest.mark.parametrize("batch", [5, 6, 7, 8])
def test_tc_every_batch_ragged_last_unit(batch):
    R = r0() + 40  # the last 64-row unit holds 40 rows
    check(synth.f8_inputs(100 + batch, R, 1024, 1, 8, 112, 140, batch=batch))


@pytest.mark.parametrize("batch,shape", [
    (5, ("r0", 2048, 128, 16)),        # 128-row x 128-column scale blocks
    (8, ("r0", 2048, 128, 16)),
    (5, ("r0+320", 1024, 64, 8)),      # 64-row scale blocks: every unit its own scale row
    (6, ("r0+1", 128, 0, 1)),          # one 128-column block, one row past a unit
    (8, ("r0+1", 128, 0, 1)),
    (8, ("2r0+273", 4096, 0, 32)),     # units split unevenly over the grid, short last tiles
    (6, ("r0", 3968, 64, 31))])        # 31 blocks of 128 columns, 64-row scale blocks
def test_tc_shapes(batch, shape):
    rspec, C, rows_per_scale, SC = shape
    R = {"r0": r0(), "r0+320": r0() + 320, "r0+1": r0() + 1, "2r0+273": 2 * r0() + 273}[rspec]
    SR = R // rows_per_scale if rows_per_scale else 1
    check(synth.f8_inputs(R % 1000 + C + batch, R, C, SR, SC, 112, 140, batch=batch))


def test_tc_wide_dynamic_range_inside_blocks():
    """x spans six decades inside every 128-column block."""
    f = synth.f8_inputs(71, r0(), 2048, r0() // 128, 16, 118, 132, batch=8)
    rng = np.random.default_rng(71)
    f.x = (f.x * (10.0 ** rng.uniform(-3, 3, f.x.shape))).astype(np.float32)
    check(f)


def test_tc_one_large_element_per_block():
    """One element per block 2^20 times the rest: the eight pieces still carry
    the others to 2^-16 of themselves (four pieces would keep only ~2^-9)."""
    f = synth.f8_inputs(72, r0(), 1024, r0() // 128, 8, 120, 134, batch=6)
    f.x[:, ::128] *= np.float32(2.0 ** 20)
    check(f)


@pytest.mark.parametrize("mult", [1e30, 1e-30, 1e-40, 0.0])
def test_tc_extreme_magnitudes(mult):
    """Huge, tiny and subnormal activations, and all-zero blocks: the relative
    bound holds without the absolute term."""
    f = synth.f8_inputs(73, r0(), 1024, r0() // 128, 8, 120, 134, batch=5)
    f.x = (f.x * np.float32(mult)).astype(np.float32)
    f.x[1, 128:384] = 0.0  # two all-zero column blocks
    y = run(f)
    ref, mag = oracle.f8_matvec(f.w, f.scale, f.x, threads=8)
    assert np.all(np.abs(y - ref) <= REL * mag), "relative bound without the absolute term"
    if mult == 0.0:
        assert not y.any()


def test_tc_subnormal_scales_and_large_exponents():
    f = synth.f8_inputs(74, r0(), 1024, r0() // 64, 8, 0, 190, batch=7)
    check(f)


def test_tc_nonfinite_x():
    f = synth.f8_inputs(75, r0(), 1024, r0() // 128, 8, 118, 132, batch=6)
    f.x[0, 37] = np.inf
    f.x[1, 700] = np.nan
    f.x[2, 5] = -np.inf
    f.x[2, 6] = np.inf
    y = check(f)
    assert np.isnan(y[1]).all()
    assert np.isinf(y[0]).any()
    assert not np.isfinite(y[2]).any()
    assert np.isfinite(y[3:]).all()


def test_tc_saturated_codes_and_nan_scale():
    R = r0()
    f = synth.f8_inputs(76, R, 4096, R // 64, 32, 120, 130, batch=8, finite_only=False)
    assert (f.w == 0x7F).any() and (f.w == 0xFF).any()
    check(f)
    f.scale[3, 5] = 255
    y = check(f)
    rows_with_nan = np.nonzero((np.arange(R) * (R // 64)) // R == 3)[0]
    assert np.isnan(y[:, rows_with_nan]).all()
    assert not np.isnan(np.delete(y, rows_with_nan, axis=1)).any()


def test_tc_integer_inputs_are_exact():
    """Integer weights (E4M3 codes of 0, +-1, +-2, 3, 4), integer x in [-8, 8]
    and unit scales: every partial sum is an integer below 2^24 and every x
    is exact in its first E4M3 piece, so the result equals the float64 oracle
    exactly."""
    rng = np.random.default_rng(77)
    codes = np.array([0x00, 0x38, 0x40, 0x44, 0x48, 0xB8, 0xC0], np.uint8)
    R, C = r0() + 512, 2048
    f = synth.F8Inputs(R, C, 1, 16, codes[rng.integers(0, len(codes), (R, C))],
                       np.full((1, 16), 127, np.uint8),
                       rng.integers(-8, 9, (8, C)).astype(np.float32))
    y = run(f)
    ref, _ = oracle.f8_matvec(f.w, f.scale, f.x, threads=8)
    assert np.array_equal(y, ref)


def test_tc_deterministic_and_writes_only_its_outputs():
    R = r0() + 1
    f = synth.f8_inputs(78, R, 1024, 1, 8, 118, 132, batch=7)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    buf = torch.full((7 * R + 64,), float("nan"), device="cuda")
    buf[7 * R:] = 3.5
    out = buf[:7 * R].view(7, R)
    qmv.f8_matvec_t(w, s, x, out=out)
    torch.cuda.synchronize()
    a = out.clone()
    qmv.f8_matvec_t(w, s, x, out=out)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), out.view(torch.int32))
    assert not torch.isnan(a).any() and bool((buf[7 * R:] == 3.5).all())


@pytest.mark.parametrize("batch", [5, 8])
def test_tc_argmax_matches_its_matvec(batch):
    """The fused greedy form: y bit for bit the plain call's, within
    tolerance of the oracle; the index is the greedy choice over that y.
    Without y the mma.sync kernel runs, whose choice must be a greedy one
    within the tolerance of the oracle's values."""
    f = synth.f8_inputs(79 + batch, r0() + 700, 2048, 1, 16, 118, 132, batch=batch)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    y_buf = torch.empty((batch, f.R), dtype=torch.float32, device="cuda")
    idx, val = qmv.f8_matvec_argmax_t(w, s, x, y=y_buf)
    y_plain = qmv.f8_matvec_t(w, s, x)
    torch.cuda.synchronize()
    assert torch.equal(y_buf.view(torch.int32), y_plain.view(torch.int32))
    y = y_buf.cpu().numpy()
    ref, mag = oracle.f8_matvec(f.w, f.scale, f.x, threads=8)
    assert np.all(np.abs(y - ref) <= REL * mag + ABS)
    idx = idx.cpu().numpy()
    assert np.array_equal(idx, oracle.argmax_rows(y))
    assert np.array_equal(val.cpu().numpy().view(np.uint32), y[np.arange(batch), idx].view(np.uint32))
    idx2, _ = qmv.f8_matvec_argmax_t(w, s, x)
    idx2 = idx2.cpu().numpy()
    for k in range(batch):
        tol = 2 * (REL * mag[k] + ABS)
        assert ref[k, idx2[k]] >= (ref[k] - tol).max() - tol[idx2[k]]


@pytest.mark.parametrize("batch", [5, 8])
def test_tc_argmax_without_y_keeps_logits_in_a_large_workspace(batch):
    """Without y, a workspace of QMV_F8_ARGMAX_WORKSPACE_TC_BYTES(batch, R)
    holds the logits behind the partials, so the call runs on this kernel:
    index and value bit for bit those of the same call with y, and the
    workspace's counter left zero.  One byte less and the mma.sync kernel
    runs."""
    R = r0() + 300
    f = synth.f8_inputs(86 + batch, R, 2048, 1, 16, 118, 132, batch=batch)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    yb = torch.empty((batch, R), dtype=torch.float32, device="cuda")
    idx, val = qmv.f8_matvec_argmax_t(w, s, x, y=yb)
    big = torch.zeros(qmv.f8_argmax_workspace_bytes(batch, R), dtype=torch.uint8, device="cuda")
    idx2, val2 = qmv.f8_matvec_argmax_t(w, s, x, workspace=big)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
    assert torch.equal(val.view(torch.int32), val2.view(torch.int32))
    assert int(big[:16].count_nonzero()) == 0
    tail = big[qmv.f8_argmax_logits_offset(batch):].view(torch.float32).view(batch, R)
    assert torch.equal(tail.view(torch.int32), yb.view(torch.int32))
    names = kernel_names(lambda: qmv.f8_matvec_argmax_t(w, s, x, workspace=big))
    assert any("f8_tc" in n for n in names), names
    short = big[:big.numel() - 1]
    names = kernel_names(lambda: qmv.f8_matvec_argmax_t(w, s, x, workspace=short))
    assert any("f8_mma" in n for n in names) and not any("f8_tc" in n for n in names), names


def test_tc_argmax_nan_and_ties():
    """A NaN result wins the greedy choice; among equal values the lower row."""
    f = synth.f8_inputs(81, r0(), 1024, 1, 8, 120, 128, batch=6)
    f.x[2, 10] = np.nan
    f.w[700] = f.w[300]
    f.x[4] = 0.0
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    yb = torch.empty((6, f.R), dtype=torch.float32, device="cuda")
    idx, _ = qmv.f8_matvec_argmax_t(w, s, x, y=yb)
    torch.cuda.synchronize()
    idx, y = idx.cpu().numpy(), yb.cpu().numpy()
    assert np.array_equal(idx, oracle.argmax_rows(y))
    assert np.isnan(y[2]).all() and idx[2] == 0  # NaN everywhere: the first row
    assert idx[4] == 0  # all zero: the first row


def test_tc_topk_sample_over_its_matvec():
    f = synth.f8_inputs(82, r0(), 2048, 1, 16, 118, 132, batch=8)
    u = np.random.default_rng(82).random(8).astype(np.float32)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    y, idx, val, _, _ = qmv.f8_matvec_topk_sample_t(w, s, x, 64, 1.0, dev(u))
    y = y.cpu().numpy()
    assert np.array_equal(y.view(np.uint32), qmv.f8_matvec_t(w, s, x).cpu().numpy().view(np.uint32))
    ref_idx, _, _ = oracle.topk_sample(y, 64, 1.0, u)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)


def test_tc_kernel_is_the_one_launched():
    f = synth.f8_inputs(83, r0(), 1024, 1, 8, 118, 132, batch=8)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    for b in (5, 8):
        names = kernel_names(lambda: qmv.f8_matvec_t(w, s, x[:b]))
        assert any("f8_tc" in n for n in names), names
    # at 2..4 vectors the mma.sync kernel runs
    names = kernel_names(lambda: qmv.f8_matvec_t(w, s, x[:4]))
    assert any("f8_mma" in n for n in names) and not any("f8_tc" in n for n in names), names
    # the argmax form: with y on this kernel; without y (and a workspace of
    # partials only), at 5..8 vectors, on mma.sync
    yb = torch.empty((8, f.R), dtype=torch.float32, device="cuda")
    names = kernel_names(lambda: qmv.f8_matvec_argmax_t(w, s, x, y=yb))
    assert any("f8_tc" in n for n in names), names
    names = kernel_names(lambda: qmv.f8_matvec_argmax_t(w, s, x))
    assert any("f8_mma" in n for n in names) and not any("f8_tc" in n for n in names), names

    # below the size threshold, and with scale rows that start off a 64-row
    # boundary, batch 8 stays on the mma.sync kernel
    g = synth.f8_inputs(84, r0() - 64, 1024, 1, 8, 118, 132, batch=8)
    gw, gs, gx = dev(g.w), dev(g.scale), dev(g.x)
    names = kernel_names(lambda: qmv.f8_matvec_t(gw, gs, gx))
    assert not any("f8_tc" in n for n in names) and any("f8_mma" in n for n in names), names
    h = synth.f8_inputs(85, 125 * 1000, 1024, 1000, 8, 118, 132, batch=8)  # scale rows of 125
    hw, hs, hx = dev(h.w), dev(h.scale), dev(h.x)
    names = kernel_names(lambda: qmv.f8_matvec_t(hw, hs, hx))
    assert not any("f8_tc" in n for n in names) and any("f8_mma" in n for n in names), names


def test_tc_reads_activations_a_preceding_kernel_wrote():
    """The kernel streams weights before its dependency wait and reads x only
    after it.  Chain: a small F8 call (mma.sync, which lets its dependents
    launch early) writes a [8, 4096] result; the large call takes it as x at
    once, on the same stream, eagerly, on a side stream and inside a CUDA
    graph.  Each time y is bit for bit the call on the settled x."""
    g = synth.f8_inputs(90, 4096, 4096, 32, 32, 118, 132, batch=8)
    f = synth.f8_inputs(91, r0() + 64, 4096, 1, 32, 118, 132, batch=8)
    gw, gs, gx = dev(g.w), dev(g.scale), dev(g.x)
    fw, fs = dev(f.w), dev(f.scale)
    mid = qmv.f8_matvec_t(gw, gs, gx)
    torch.cuda.synchronize()
    want = qmv.f8_matvec_t(fw, fs, mid.clone())
    torch.cuda.synchronize()
    want = want.cpu()

    def chain(stream=None):
        m = torch.full((8, 4096), float("nan"), device="cuda")
        y = torch.full((8, f.R), float("nan"), device="cuda")
        qmv.f8_matvec_t(gw, gs, gx, out=m, stream=stream)
        qmv.f8_matvec_t(fw, fs, m, out=y, stream=stream)
        return y

    y = chain()
    torch.cuda.synchronize()
    assert torch.equal(y.cpu().view(torch.int32), want.view(torch.int32))
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        y = chain(st)
    st.synchronize()
    assert torch.equal(y.cpu().view(torch.int32), want.view(torch.int32))
    m = torch.full((8, 4096), float("nan"), device="cuda")
    y = torch.full((8, f.R), float("nan"), device="cuda")
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        qmv.f8_matvec_t(gw, gs, gx, out=m, stream=cs)  # (warm the launch path outside capture)
        cs.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            qmv.f8_matvec_t(gw, gs, gx, out=m, stream=cs)
            qmv.f8_matvec_t(fw, fs, m, out=y, stream=cs)
    m.fill_(float("nan"))
    y.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.cpu().view(torch.int32), want.view(torch.int32))


def test_tc_back_to_back_calls_keep_their_own_inputs():
    """Three consecutive calls on one stream with different x and y: each
    result is the one its own x gives (the next call's early weight loads do
    not disturb the previous call)."""
    f = synth.f8_inputs(92, r0(), 2048, 1, 16, 118, 132, batch=6)
    w, s = dev(f.w), dev(f.scale)
    rng = np.random.default_rng(92)
    xs = [dev(rng.standard_normal(f.x.shape).astype(np.float32)) for _ in range(3)]
    singles = []
    for x in xs:
        singles.append(qmv.f8_matvec_t(w, s, x))
        torch.cuda.synchronize()
    ys = [torch.empty((6, f.R), device="cuda") for _ in range(3)]
    for x, y in zip(xs, ys):
        qmv.f8_matvec_t(w, s, x, out=y)
    torch.cuda.synchronize()
    for a, b in zip(ys, singles):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_zz_no_wait_ran_out():
    """Run last in this file: no wait of the kernel hit its time limit."""
    assert qmv.tc_wait_timeouts() == 0
