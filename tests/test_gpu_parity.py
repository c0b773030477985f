"""GPU parity: the CUDA path (through the C-ABI) against the float64 oracle.

Bars (from the method's definitions on the pages):
* cq_prepare and cq_dequantize_row: bit-exact (float32-staged FWHT of the
  needle.js "part 2" sections 2 and "Row gather").
* E4M3 / E8M0 decode inside f8_matvec: bit-exact on all 256 codes.
* cq_matvec and f8_matvec: |y - y_oracle| <= 1e-4 * A + 1e-6, A the magnitude
  sum of the terms the method adds (sum_g |norm| sum_k |level * p| for CQ,
  sum_c |w * s * x| for F8).
"""
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
    torch.cuda.init()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_close(y, ref, mag):
    y = np.asarray(y, np.float64)
    both_nan = np.isnan(y) & np.isnan(ref)
    err = np.abs(y - ref)
    bound = REL * mag + ABS
    ok = both_nan | (err <= bound)
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError("mismatch at %s: gpu %r oracle %r bound %r (%d bad)" % (
            tuple(i), y[tuple(i)], ref[tuple(i)], bound[tuple(i)], int((~ok).sum())))


def bits_equal(a, b):
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


def oracle_cq(c):
    return oracle.CQMatrix(c.output, c.input, c.input_padded, c.group, c.bits, c.packed, c.norms,
                           c.codebook)


# ---------------------------------------------------------------------------
# cq_prepare: bit-exact
# ---------------------------------------------------------------------------

PREP_CASES = [(512, 64, 1), (512, 64, 4), (500, 128, 1), (6, 2, 3), (40, 32, 2), (31, 8, 8),
              (1000, 1024, 2), (3000, 2048, 1), (4096, 4096, 2), (130, 4, 5), (17, 16, 1),
              (700, 256, 3), (1024, 512, 1), (65, 64, 7)]


@pytest.mark.parametrize("inp,group,batch", PREP_CASES)
def test_prepare_bit_exact(inp, group, batch):
    c = synth.cq_inputs(100 + inp, 4, inp, group, 2, batch=batch)
    m = qmv.CQMatrix.from_numpy(c)
    got = host(qmv.cq_prepare_t(m, dev(c.x)))
    want = oracle.cq_prepare(c.x, c.input_padded, group, mode="f32")
    assert bits_equal(got, want)


def test_prepare_scale_rounding_case():
    # group 2, x = (v, 0): both outputs RN32(RN64(v * RN64(1/sqrt 2)))
    x = np.array([[float.fromhex("0x1.4dd2f2p+0"), 0.0]], np.float32)
    c = synth.cq_inputs(1, 1, 2, 2, 2)
    m = qmv.CQMatrix.from_numpy(c)
    got = host(qmv.cq_prepare_t(m, dev(x)))[0]
    assert got[0] == got[1] == np.float32(float.fromhex("0x1.d81934p-1"))


@pytest.mark.parametrize("binade,full", [(0, True), (-60, True), (99, True), (-61, False),
                                         (100, False), (-130, False)])
def test_prepare_scale_every_mantissa(binade, full):
    """Group 2, pairs (v, 0): both outputs must be RN32(RN64(v * RN64(1/sqrt 2))).
    Every float32 mantissa of the binade [2^b, 2^(b+1)), both signs (a 2^16
    sample outside the range where the kernels use their float32 form of the
    product: there they take the float64 one; b = -130 is subnormal)."""
    if binade >= -126:
        m = np.arange(1 << 23, dtype=np.uint32)
        v = ((np.uint32(127 + binade) << 23) | m).view(np.float32)
    else:  # subnormal: exponent field 0, value m * 2^-149
        v = np.arange(1 << (binade + 149), 1 << (binade + 150), dtype=np.uint32).view(np.float32)
    if not full:
        v = np.random.default_rng(abs(binade)).choice(v, 1 << 16, replace=False)
    v = np.concatenate([v, -v])
    x = np.zeros((1, 2 * v.size), np.float32)
    x[0, 0::2] = v
    c = synth.cq_inputs(2, 1, x.shape[1], 2, 2)
    mat = qmv.CQMatrix.from_numpy(c)
    got = host(qmv.cq_prepare_t(mat, dev(x)))[0]
    s = 1.0 / np.sqrt(np.float64(2.0))
    want = (v.astype(np.float64) * s).astype(np.float32)
    assert bits_equal(got[0::2], want) and bits_equal(got[1::2], want)


def test_prepare_power_of_two_scale_edges():
    """Group 4, x = (v, 0, 0, 0): all four outputs are RN32(RN64(v / 2)), the
    power-of-two case (one float32 multiply): subnormal v (halving rounds),
    the smallest normals, huge values, +-Inf and NaN."""
    rng = np.random.default_rng(4)
    sub = rng.integers(1, 1 << 23, 4096, dtype=np.uint32).view(np.float32)
    v = np.concatenate([sub, -sub, np.array([np.finfo(np.float32).tiny, np.finfo(np.float32).max,
                                             -np.finfo(np.float32).max, np.inf, -np.inf,
                                             np.float32(1.5e-45), 0.0], np.float32)])
    x = np.zeros((1, 4 * v.size), np.float32)
    x[0, 0::4] = v
    c = synth.cq_inputs(3, 1, x.shape[1], 4, 2)
    got = host(qmv.cq_prepare_t(qmv.CQMatrix.from_numpy(c), dev(x)))[0].reshape(-1, 4)
    want = (v.astype(np.float64) * 0.5).astype(np.float32)
    for j in range(4):
        assert bits_equal(got[:, j], want)
    xn = np.zeros((1, 4), np.float32)
    xn[0, 0] = np.nan
    gn = host(qmv.cq_prepare_t(qmv.CQMatrix.from_numpy(synth.cq_inputs(3, 1, 4, 4, 2)), dev(xn)))[0]
    assert np.isnan(gn).all()


# ---------------------------------------------------------------------------
# cq_dequantize_row: bit-exact, out-of-range ids
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("inp,group", [(512, 64), (500, 128), (37, 2), (100, 32), (2000, 2048)])
def test_dequantize_row_bit_exact(bits, inp, group):
    c = synth.cq_inputs(7 + bits, 300, inp, group, bits, gather=40)
    m = qmv.CQMatrix.from_numpy(c)
    got = host(qmv.cq_dequantize_row_t(m, dev(c.rows)))
    want, bad = oracle_cq(c).dequantize_rows(c.rows)
    assert not bad
    assert bits_equal(got, want)


def test_dequantize_row_vocab_workload():
    c = synth.workload_inputs("cq2_vocab")
    m = qmv.CQMatrix.from_numpy(c)
    got = host(qmv.cq_dequantize_row_t(m, dev(c.rows)))
    want, _ = oracle_cq(c).dequantize_rows(c.rows)
    assert got.shape == (64, 500)
    assert bits_equal(got, want)


def test_dequantize_row_bad_ids_give_zero_rows_and_status():
    c = synth.cq_inputs(3, 50, 100, 32, 3)
    m = qmv.CQMatrix.from_numpy(c)
    ids = np.array([3, 50, -1, 49, 1 << 30, 0], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((6, 100), float("nan"), device="cuda")
    qmv.cq_dequantize_row_t(m, dev(ids), out=out, status=status)
    got = host(out)
    want, bad = oracle_cq(c).dequantize_rows(ids)
    assert bad and int(host(status)[0]) == 10
    assert bits_equal(got, want)
    assert np.all(got[[1, 2, 4]] == 0)
    ok = torch.zeros(1, dtype=torch.int32, device="cuda")
    qmv.cq_dequantize_row_t(m, dev(ids[[0, 3, 5]]), status=ok)
    assert int(host(ok)[0]) == 0


def test_dequantize_row_empty():
    c = synth.cq_inputs(3, 5, 64, 64, 2)
    m = qmv.CQMatrix.from_numpy(c)
    out = qmv.cq_dequantize_row_t(m, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert out.shape == (0, 64)


# ---------------------------------------------------------------------------
# cq_matvec: tolerance vs the oracle over the GPU-prepared vector
# ---------------------------------------------------------------------------

def check_cq_matvec(c):
    m = qmv.CQMatrix.from_numpy(c)
    p_gpu = qmv.cq_prepare_t(m, dev(c.x))
    y = qmv.cq_matvec_t(m, p_gpu)
    p = host(p_gpu)
    assert bits_equal(p, oracle.cq_prepare(c.x, c.input_padded, c.group, mode="f32"))
    ref, mag = oracle_cq(c).matvec(p, threads=8)
    assert_close(host(y), ref, mag)
    # also within bounds of the float64-prepared result
    ref64, mag64 = oracle_cq(c).matvec(oracle.cq_prepare(c.x, c.input_padded, c.group, mode="f64"))
    assert_close(host(y), ref64, mag64)
    return y


def test_cq_matvec_cq4_512():
    check_cq_matvec(synth.workload_inputs("cq4_512"))


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("batch", [1, 4])
def test_cq_matvec_bit_width_sweep(bits, batch):
    check_cq_matvec(synth.workload_inputs("cq_sweep", bits=bits, batch=batch))


def test_cq_matvec_vocab_workload():
    check_cq_matvec(synth.workload_inputs("cq2_vocab"))


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("out,inp,group,batch", [
    (1, 2, 2, 1), (7, 100, 32, 3), (33, 6, 2, 8), (65, 1000, 1024, 2), (300, 4000, 4096, 1),
    (129, 130, 4, 5), (40, 512, 512, 8), (3, 70, 8, 6)])
def test_cq_matvec_shapes(bits, out, inp, group, batch):
    check_cq_matvec(synth.cq_inputs(out + inp, out, inp, group, bits, batch=batch))


@pytest.mark.parametrize("P", [256, 512, 1024, 2048])
@pytest.mark.parametrize("group", [64, 128, 256])
@pytest.mark.parametrize("out", [1, 5, 1000, 5001, 9999])
def test_cq2_table_path(P, group, out):
    """2-bit, batch 1, group >= 64: the nibble-table kernel, from one row to
    several rows per warp of a full grid."""
    check_cq_matvec(synth.cq_inputs(P + group + out, out, P - 3, group, 2, batch=1,
                                    input_padded=P))


def test_cq_matvec_empty_output():
    c = synth.cq_inputs(3, 0, 64, 64, 2)
    m = qmv.CQMatrix.from_numpy(c)
    assert qmv.cq_matvec_t(m, torch.zeros(1, 64, device="cuda")).shape == (1, 0)


def test_cq_deterministic_and_writes_every_output():
    c = synth.workload_inputs("cq2_vocab")
    m = qmv.CQMatrix.from_numpy(c)
    p = qmv.cq_prepare_t(m, dev(c.x))
    buf = torch.full((c.output + 64,), float("nan"), device="cuda")
    buf[c.output:] = 12345.0
    a = qmv.cq_matvec_t(m, p, out=buf[:c.output].view(1, -1))
    first = host(a).copy()
    qmv.cq_matvec_t(m, p, out=buf[:c.output].view(1, -1))
    second = host(buf)
    assert not np.isnan(first).any()
    assert np.all(second[c.output:] == 12345.0)
    assert bits_equal(first[0], second[:c.output])


# ---------------------------------------------------------------------------
# f8_matvec
# ---------------------------------------------------------------------------

def check_f8(f, batch=None, rows=None):
    x = f.x if batch is None else f.x[:batch]
    y = host(qmv.f8_matvec_t(dev(f.w), dev(f.scale), dev(x)))
    ref, mag = oracle.f8_matvec(f.w, f.scale, x, threads=8)
    assert_close(y, ref, mag)
    return y


@pytest.mark.parametrize("C", [16, 17])
def test_e4m3_decode_bit_exact_all_codes(C):
    # row r holds code r in column 0 and zeros elsewhere; x = e_0; unit scale
    w = np.zeros((256, C), np.uint8)
    w[:, 0] = np.arange(256)
    x = np.zeros((1, C), np.float32)
    x[0, 0] = 1
    y = host(qmv.f8_matvec_t(dev(w), dev(np.full((1, 1), 127, np.uint8)), dev(x)))[0]
    want = oracle.e4m3_to_f32(np.arange(256, dtype=np.uint8))
    assert np.array_equal(y, want)  # (+0 and -0 compare equal)


@pytest.mark.parametrize("C", [16, 17])
def test_e8m0_decode_bit_exact_all_codes(C):
    w = np.zeros((256, C), np.uint8)
    w[:, 0] = 0x38  # 1.0
    x = np.zeros((1, C), np.float32)
    x[0, 0] = 1
    scale = np.arange(256, dtype=np.uint8).reshape(256, 1)
    y = host(qmv.f8_matvec_t(dev(w), dev(scale), dev(x)))[0]
    want = oracle.e8m0_to_f32(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(y), np.isnan(want))
    ok = ~np.isnan(want)
    assert bits_equal(y[ok], want[ok])


@pytest.mark.parametrize("batch", [1, 8])
def test_f8_4096(batch):
    check_f8(synth.workload_inputs("f8_4096", batch=batch))


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("R,C,SR,SC", [
    (1000, 4096, 8, 32),     # R not a multiple of the row tile
    (1030, 4096, 4, 32),     # SR does not divide R: tiles straddle scale rows
    (300, 4096, 300, 32),    # one scale row per weight row
    (257, 4096, 5, 3),       # scale blocks not aligned to 16-column chunks
    (64, 100, 3, 7),         # C not a multiple of 16 (general kernel)
    (1, 16, 1, 1), (33, 48, 2, 3), (9, 2048, 9, 128), (70, 8192, 7, 64)])
def test_f8_shapes(batch, R, C, SR, SC):
    check_f8(synth.f8_inputs(R + C + SC, R, C, SR, SC, 115, 135, batch=batch))


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("R,C,SR,SC", [
    (150001, 32, 7, 2),      # many tiles: the streaming kernel; SR does not divide R
    (131075, 48, 40000, 3),  # tiles straddle scale rows (up to 1 per 3 rows)
    (122881, 16, 1, 1)])     # one chunk per row: most lanes idle
def test_f8_streaming_kernel_shapes(batch, R, C, SR, SC):
    check_f8(synth.f8_inputs(R + C + batch, R, C, SR, SC, 110, 140, batch=batch))


def test_f8_saturated_codes_and_nan_scale():
    f = synth.f8_inputs(77, 500, 4096, 10, 32, 120, 130, batch=2, finite_only=False)
    assert (f.w == 0x7F).any() and (f.w == 0xFF).any()
    check_f8(f)
    f.scale[3, 5] = 255
    y = check_f8(f)
    rows_with_nan = np.unique(np.nonzero((np.arange(500) * 10) // 500 == 3)[0])
    assert np.isnan(y[:, rows_with_nan]).all()
    assert not np.isnan(np.delete(y, rows_with_nan, axis=1)).any()


def test_f8_subnormal_and_extreme_scales():
    # exponents down to 0 (scale 2^-127, a float32 subnormal) and up to 2^63;
    # larger scales would overflow the float32 accumulator the kernels use
    f = synth.f8_inputs(78, 256, 1024, 16, 8, 0, 190, batch=3)
    check_f8(f)


@pytest.fixture(scope="module")
def head():
    f = synth.f8_inputs(5, 245760, 4096, 1920, 32, 118, 132, batch=8)
    return f, dev(f.w), dev(f.scale)


@pytest.fixture(scope="module")
def head_ref(head):
    """The oracle over every row of the head for all 8 vectors (threaded on
    the host cores); vectors are independent, so ref[:b] serves batch b."""
    f, _, _ = head
    return oracle.f8_matvec(f.w, f.scale, f.x, threads=os.cpu_count() or 8)


@pytest.mark.parametrize("batch", [1, 2, 4, 5, 8])
def test_f8_head_full_size_every_row(head, head_ref, batch):
    """All 245760 rows of the 245760 x 4096 head (ds4f-disk issue #6, work
    item 3) against the oracle, at each batch the head runs: batch 1 on the
    streaming kernel, 2-4 on the mma.sync kernel, 5-8 on the tcgen05 one."""
    f, w_dev, s_dev = head
    y = host(qmv.f8_matvec_t(w_dev, s_dev, dev(f.x[:batch])))
    ref, mag = head_ref
    assert_close(y, ref[:batch], mag[:batch])


@pytest.mark.parametrize("batch", [1, 8])
def test_f8_head_argmax_full_size_every_row(head, head_ref, batch):
    """The fused greedy head at full size: its y is f8_matvec's bit for bit
    and within tolerance of the oracle on every row; the index is the greedy
    choice over that y and the value is y at that row."""
    f, w_dev, s_dev = head
    x = dev(f.x[:batch])
    y_buf = torch.empty((batch, f.R), dtype=torch.float32, device="cuda")
    idx, val = qmv.f8_matvec_argmax_t(w_dev, s_dev, x, y=y_buf)
    y_plain = qmv.f8_matvec_t(w_dev, s_dev, x)
    torch.cuda.synchronize()
    assert torch.equal(y_buf.view(torch.int32), y_plain.view(torch.int32))
    y = host(y_buf)
    ref, mag = head_ref
    assert_close(y, ref[:batch], mag[:batch])
    idx = idx.cpu().numpy()
    assert np.array_equal(idx, oracle.argmax_rows(y))
    assert bits_equal(val.cpu().numpy(), y[np.arange(batch), idx])


@pytest.mark.parametrize("batch", [1, 8])
def test_f8_head_topk_full_size_every_row(head, head_ref, batch):
    """The fused top-64 sampling head at full size: y within tolerance of the
    oracle on every row, and the 64 rows and their order equal to the
    oracle's selection over that y (probabilities and the draw are checked
    in the top-k tests)."""
    f, w_dev, s_dev = head
    u = np.random.default_rng(batch + 40).random(batch).astype(np.float32)
    y, idx, val, _, _ = qmv.f8_matvec_topk_sample_t(w_dev, s_dev, dev(f.x[:batch]), 64, 1.0,
                                                     dev(u))
    y = host(y)
    ref, mag = head_ref
    assert_close(y, ref[:batch], mag[:batch])
    ref_idx, _, _ = oracle.topk_sample(y, 64, 1.0, u)
    idx = idx.cpu().numpy()
    assert np.array_equal(idx, ref_idx)
    assert bits_equal(val.cpu().numpy(), np.take_along_axis(y, idx, 1))


def test_f8_deterministic_guarded_and_on_a_side_stream():
    f = synth.workload_inputs("f8_4096", batch=1)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    buf = torch.full((4096 + 64,), float("nan"), device="cuda")
    buf[4096:] = -7.0
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        qmv.f8_matvec_t(w, s, x, out=buf[:4096].view(1, -1))
    st.synchronize()
    a = host(buf).copy()
    qmv.f8_matvec_t(w, s, x, out=buf[:4096].view(1, -1))
    b = host(buf)
    assert not np.isnan(a[:4096]).any() and np.all(b[4096:] == -7.0)
    assert bits_equal(a, b)
    ref, mag = oracle.f8_matvec(f.w, f.scale, f.x)
    assert_close(a[None, :4096], ref, mag)


def test_alias_rejected_on_device():
    f = synth.f8_inputs(3, 64, 64, 1, 1, 127, 127)
    w = dev(f.w)
    with pytest.raises(qmv.QmvError) as e:
        qmv.f8_matvec_t(w, dev(f.scale), dev(f.x), out=w.view(-1).view(torch.float32)[:64].view(1, 64))
    assert e.value.status == 8
