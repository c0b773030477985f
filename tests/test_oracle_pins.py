"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources (page titles and sections):
* needle.js "Inference engine, part 2: kernels and token step" -- section 1
  (FWHT and the identity FWHT(FWHT(x)) = n x), section 2 (prepare),
  section 3 (packed-row dot, 2-bit byte table), "Row gather"
  (dequantizeRow and the matvec == dot(dequantizeRow, x) test).
* needle.js "Inference engine, part 1: loader and tokenizer" -- section 3
  (FP16 decode and its listed test cases), section 4 (CqMatrix).
* ds4f-disk issue #6 -- work item 1 / step 1 (E4M3 decode, E8M0 block
  scales indexed scale[r*SR/R][c*SC/C], "F8 matvec vs naive with per-block
  scales").

Independent references used: explicit Sylvester-Hadamard matrices and
numpy matmul, numpy float16, torch float8_e4m3fn / float8_e8m0fnu decodes,
numpy unpackbits, hand-derived golden files and closed forms.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import parse_float, read_golden
from quantized_weight_matvec_gb300 import synth


def hadamard(n: int) -> np.ndarray:
    """Sylvester-ordered Hadamard matrix H[i, j] = (-1)^popcount(i & j)."""
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


def unpack_indices(packed: np.ndarray, bits: int, ncols: int) -> np.ndarray:
    """Indices via numpy's little-endian bit unpacking (independent of the oracle)."""
    bitstream = np.unpackbits(packed, axis=1, bitorder="little")[:, : ncols * bits]
    b = bitstream.reshape(packed.shape[0], ncols, bits).astype(np.int64)
    return (b << np.arange(bits)).sum(axis=2)


def pack_indices(idx: np.ndarray, bits: int, row_bytes: int) -> np.ndarray:
    """Bit-by-bit packer: index bit i of column k goes to stream bit k*bits+i."""
    out = np.zeros((idx.shape[0], row_bytes), dtype=np.uint8)
    for r in range(idx.shape[0]):
        for k in range(idx.shape[1]):
            for i in range(bits):
                if (int(idx[r, k]) >> i) & 1:
                    t = k * bits + i
                    out[r, t // 8] |= np.uint8(1 << (t % 8))
    return out


def f16_values(u16: np.ndarray) -> np.ndarray:
    return u16.view(np.float16).astype(np.float64)


# ---------------------------------------------------------------------------
# scalar decodes
# ---------------------------------------------------------------------------

def test_f16_golden_cases():
    for code, val in read_golden("f16_pins.txt"):
        got = float(oracle.f16_to_f32(np.array([int(code, 16)]))[0])
        want = parse_float(val)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_f16_exhaustive_vs_numpy():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32(codes)
    want = codes.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_e4m3_golden_cases():
    for code, val in read_golden("e4m3_pins.txt"):
        got = float(oracle.e4m3_to_f32(np.array([int(code, 16)]))[0])
        want = parse_float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_e4m3_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    finite = np.isfinite(ref)
    # torch's e4m3fn has NaN at 0x7F / 0xFF; every other code must match bit for bit
    assert list(np.nonzero(~finite)[0]) == [0x7F, 0xFF]
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert got[0x7F] == 448.0 and got[0xFF] == -448.0
    # second formulation from the page's bit-level decode: P = 2^(e-7), M = m/8
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        mag = (m / 8) * 2.0 ** -6 if e == 0 else min((1 + m / 8) * 2.0 ** (e - 7), 448.0)
        assert float(got[b]) == (-mag if s else mag)


def test_e8m0_golden_and_exhaustive():
    for code, val in read_golden("e8m0_pins.txt"):
        got = float(oracle.e8m0_to_f32(np.array([int(code)]))[0])
        want = parse_float(val)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want, code
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e8m0_to_f32(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e8m0fnu).float().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok].view(np.uint32), ref[ok].view(np.uint32))
    # 2^-127 = 2^22 * 2^-149 is the float32 subnormal 0x00400000 (not flushed)
    assert got[:1].view(np.uint32)[0] == 0x00400000


# ---------------------------------------------------------------------------
# FWHT
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128])
def test_fwht_matches_hadamard_matrix(n):
    rng = np.random.default_rng(n)
    x = rng.standard_normal(n)
    assert np.allclose(oracle.fwht_f64(x), hadamard(n) @ x, rtol=0, atol=1e-12 * n)


@pytest.mark.parametrize("n", [2, 16, 256, 4096])
def test_fwht_involution(n):
    # needle-2 section 1: FWHT(FWHT(x)) = n x
    rng = np.random.default_rng(7)
    x = rng.standard_normal(n)
    assert np.allclose(oracle.fwht_f64(oracle.fwht_f64(x)), n * x, atol=1e-9 * n)


def test_fwht_impulse_is_all_ones():
    x = np.zeros(64)
    x[0] = 1
    assert np.array_equal(oracle.fwht_f64(x), np.ones(64))
    assert np.array_equal(oracle.fwht_f32(x), np.ones(64, np.float32))


def test_fwht_f32_stage_order_golden():
    rows = dict((r[0], r[1:]) for r in read_golden("fwht_f32_stage_order.txt"))
    x = np.array([parse_float(t) for t in rows["input"]], np.float32)
    want = np.array([parse_float(t) for t in rows["output"]], np.float32)
    got = oracle.fwht_f32(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_fwht_f32_exact_on_small_integers():
    # integer inputs whose partial sums stay below 2^24 are exact in float32
    rng = np.random.default_rng(3)
    x = rng.integers(-1000, 1000, 512).astype(np.float32)
    assert np.array_equal(oracle.fwht_f32(x), (hadamard(512) @ x.astype(np.float64)).astype(
        np.float32))


# ---------------------------------------------------------------------------
# prepare
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("inp,group", [(512, 64), (500, 128), (6, 2), (40, 32), (1, 8)])
def test_prepare_f64_matches_blockwise_hadamard(inp, group):
    P = synth.padded_width(inp, group)
    rng = np.random.default_rng(inp + group)
    x = rng.standard_normal((2, inp)).astype(np.float32)
    got = oracle.cq_prepare(x, P, group, mode="f64")
    xp = np.zeros((2, P))
    xp[:, :inp] = x
    H = hadamard(group) / math.sqrt(group)
    want = np.concatenate([xp[:, g:g + group] @ H.T for g in range(0, P, group)], axis=1)
    assert np.allclose(got, want, atol=1e-12)
    got32 = oracle.cq_prepare(x, P, group, mode="f32")
    assert np.allclose(got32, want, atol=1e-5 * np.abs(x).sum() / math.sqrt(group) + 1e-7)


def test_prepare_scale_rounding_golden():
    rows = dict((r[0], r[1:]) for r in read_golden("prepare_scale_rounding.txt"))
    group = int(rows["group"][0])
    x = np.array([[parse_float(t) for t in rows["input"]]], np.float32)
    want = np.array([parse_float(t) for t in rows["output"]], np.float32)
    got = oracle.cq_prepare(x, 2, group, mode="f32")[0]
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # group 128: the unit impulse maps to RN32(RN64(1/sqrt(128))) everywhere
    e0 = np.zeros((1, 128), np.float32)
    e0[0, 0] = 1
    s = np.float32(np.float64(1.0) / np.sqrt(np.float64(128)))
    assert np.array_equal(oracle.cq_prepare(e0, 128, 128, mode="f32")[0],
                          np.full(128, s, np.float32))


def test_prepare_pads_with_zeros():
    x = np.ones((1, 3), np.float32)
    got = oracle.cq_prepare(x, 4, 4, mode="f64")[0]
    assert np.allclose(got, hadamard(4) @ np.array([1, 1, 1, 0.0]) / 2)


# ---------------------------------------------------------------------------
# packed indices
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_index_unpack_matches_independent_packer(bits):
    rng = np.random.default_rng(bits)
    ncols = 37
    rb = synth.row_bytes_for(ncols, bits)
    idx = rng.integers(0, 1 << bits, (3, ncols))
    packed = pack_indices(idx, bits, rb)
    m = oracle.CQMatrix(3, ncols, ncols, 1, bits, packed, np.zeros((3, ncols), np.uint16),
                        np.zeros(1 << bits, np.float32))
    for r in range(3):
        for k in range(ncols):
            assert m.index(r, k) == idx[r, k]


def test_index_2bit_low_crumb_first_and_4bit_low_nibble_first():
    rng = np.random.default_rng(11)
    packed = rng.integers(0, 256, (2, 16), dtype=np.uint8)
    m2 = oracle.CQMatrix(2, 64, 64, 64, 2, packed, np.zeros((2, 1), np.uint16),
                         np.zeros(4, np.float32))
    m4 = oracle.CQMatrix(2, 32, 32, 32, 4, packed, np.zeros((2, 1), np.uint16),
                         np.zeros(16, np.float32))
    for r in range(2):
        for j in range(16):
            byte = int(packed[r, j])
            for crumb in range(4):  # needle-2 section 3: (byte >> (crumb*2)) & 3
                assert m2.index(r, 4 * j + crumb) == (byte >> (crumb * 2)) & 3
            assert m4.index(r, 2 * j) == byte & 15
            assert m4.index(r, 2 * j + 1) == byte >> 4


# ---------------------------------------------------------------------------
# cqMatvec and dequantizeRow
# ---------------------------------------------------------------------------

def _cq(bits, output=24, inp=100, group=32, seed=5, batch=2):
    c = synth.cq_inputs(seed, output, inp, group, bits, batch=batch, gather=0)
    m = oracle.CQMatrix(c.output, c.input, c.input_padded, c.group, c.bits, c.packed, c.norms,
                        c.codebook)
    return c, m


def _dense(c):
    idx = unpack_indices(c.packed, c.bits, c.input_padded)
    n = f16_values(c.norms)
    return c.codebook.astype(np.float64)[idx] * np.repeat(n, c.group, axis=1)


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_cq_matvec_matches_dense_expansion(bits):
    c, m = _cq(bits)
    p = oracle.cq_prepare(c.x, c.input_padded, c.group, mode="f32")
    y, mag = m.matvec(p)
    W = _dense(c)
    want = p.astype(np.float64) @ W.T
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(mag, np.abs(p.astype(np.float64)) @ np.abs(W).T, rtol=1e-12)


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_cq_matvec_equals_dot_with_dequantized_rows(bits):
    # needle-2 "Row gather": cqMatvec(M, x)[row] ~ dot(dequantizeRow(M, row), x)
    c, m = _cq(bits, inp=100, group=32)
    p64 = oracle.cq_prepare(c.x, c.input_padded, c.group, mode="f64")
    y, mag = m.matvec(p64)
    rows, bad = m.dequantize_rows(np.arange(c.output))
    assert not bad
    dots = c.x.astype(np.float64) @ rows.astype(np.float64).T
    assert np.allclose(y, dots, rtol=0, atol=1e-5 * mag.max())


def test_cq_matvec_single_level_closed_form():
    # every index reads the same level c: y = sum_g n_g * c * sum_{k in g} p_k
    c, _ = _cq(3, output=5, inp=64, group=16)
    cb = np.full(8, 0.75, np.float32)
    m = oracle.CQMatrix(c.output, c.input, c.input_padded, c.group, 3, c.packed, c.norms, cb)
    p = oracle.cq_prepare(c.x, c.input_padded, c.group, mode="f64")
    y, _ = m.matvec(p)
    n = f16_values(c.norms)
    psum = p.reshape(p.shape[0], -1, c.group).sum(axis=2)
    assert np.allclose(y, 0.75 * psum @ n.T, rtol=1e-13)


@pytest.mark.parametrize("bits,group", [(2, 64), (3, 8), (4, 2), (5, 128)])
def test_dequantize_row_matches_hadamard(bits, group):
    c, m = _cq(bits, output=6, inp=max(group, 70) - 3, group=group)
    got, bad = m.dequantize_rows(np.arange(6))
    assert not bad
    W = _dense(c)
    H = hadamard(group) / math.sqrt(group)
    want = np.concatenate([W[:, g:g + group] @ H.T for g in range(0, c.input_padded, group)],
                          axis=1)[:, :c.input]
    tol = 4e-7 * math.log2(group) * np.abs(W).max() * math.sqrt(group) + 1e-30
    assert np.allclose(got, want, rtol=0, atol=tol)


def test_dequantize_row_scale_rounding_golden():
    """needle-2 "Row gather" with section 2's scaling: levels times the norm
    rounded to float32, float32 butterflies, then RN32(RN64(v * s)) with
    s = 1 / sqrt(group) in float64.  The golden values are derived by hand in
    the file; a float32 scale product, or an unrounded level * norm, gives a
    different bit pattern."""
    for case, group, inp, code, l1, l2, even, odd in read_golden("dequantize_scale_rounding.txt"):
        group, inp = int(group), int(inp)
        packed = np.zeros((1, (group * 2 + 7) // 8), np.uint8)
        packed[0, 0] = 1 | (2 << 2)  # column 0 -> index 1, column 1 -> index 2
        norms = np.array([[int(code, 16)]], np.uint16)
        cb = np.array([0.0, parse_float(l1), parse_float(l2), 0.0], np.float32)
        m = oracle.CQMatrix(1, inp, group, group, 2, packed, norms, cb)
        got, bad = m.dequantize_rows(np.array([0], np.int32))
        assert not bad
        want = np.where(np.arange(inp) % 2 == 0, np.float32(parse_float(even)),
                        np.float32(parse_float(odd))).astype(np.float32)
        assert np.array_equal(got[0].view(np.uint32), want.view(np.uint32)), case


def test_dequantize_row_out_of_range_gives_zero_row():
    c, m = _cq(2, output=4, inp=32, group=32)
    got, bad = m.dequantize_rows(np.array([1, 4, -1, 0], np.int32))
    assert bad
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    assert np.array_equal(got[0], m.dequantize_rows([1])[0][0])


# ---------------------------------------------------------------------------
# F8 E4M3 + E8M0 matvec
# ---------------------------------------------------------------------------

def _decode_e4m3_torch(w):
    return torch.from_numpy(np.ascontiguousarray(w)).view(torch.float8_e4m3fn).float() \
        .numpy().astype(np.float64)


def test_f8_single_scale_is_scaled_matmul():
    f = synth.f8_inputs(9, 33, 48, 1, 1, 125, 125, batch=3)
    y, mag = oracle.f8_matvec(f.w, f.scale, f.x)
    W = _decode_e4m3_torch(f.w)
    want = (f.x.astype(np.float64) @ W.T) * 2.0 ** (125 - 127)
    assert np.allclose(y, want, rtol=1e-13, atol=1e-13)
    assert np.allclose(mag, np.abs(f.x.astype(np.float64)) @ np.abs(W).T / 4, rtol=1e-13)


def test_f8_floor_block_indexing_hand_listed():
    # R=10, SR=4: row r uses block floor(4r/10); C=12, SC=3: column c uses floor(3c/12)
    row_block = [0, 0, 0, 1, 1, 2, 2, 2, 3, 3]
    col_block = [0, 0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 2]
    f = synth.f8_inputs(10, 10, 12, 4, 3, 110, 140, batch=2)
    y, _ = oracle.f8_matvec(f.w, f.scale, f.x)
    S = np.array([[2.0 ** (int(f.scale[row_block[r], col_block[c]]) - 127) for c in range(12)]
                  for r in range(10)])
    want = f.x.astype(np.float64) @ (_decode_e4m3_torch(f.w) * S).T
    assert np.allclose(y, want, rtol=1e-13, atol=1e-30)


def test_f8_wkv_scale_shape():
    # ds4f-6 step 1: the real wkv.scale layout [4, 32]; R not a multiple of SR
    R, C, SR, SC = 1030, 4096, 4, 32
    f = synth.f8_inputs(12, R, C, SR, SC, 118, 132)
    y, _ = oracle.f8_matvec(f.w, f.scale, f.x, rows=(0, R))
    W = _decode_e4m3_torch(f.w)
    rb = (np.arange(R) * SR) // R
    cb = (np.arange(C) * SC) // C
    S = np.exp2(f.scale[rb][:, cb].astype(np.float64) - 127)
    assert np.allclose(y[0], (W * S) @ f.x[0].astype(np.float64), rtol=1e-12, atol=1e-30)


def test_f8_identity_weights():
    # one-hot rows (code 0x38 = 1.0) with unit scale reproduce x
    C = 16
    w = np.zeros((C, C), np.uint8)
    w[np.arange(C), np.arange(C)] = 0x38
    x = np.arange(1, C + 1, dtype=np.float32)[None, :]
    y, _ = oracle.f8_matvec(w, np.full((1, 1), 127, np.uint8), x)
    assert np.array_equal(y[0], x[0].astype(np.float64))


def test_f8_clamped_code_and_nan_scale():
    w = np.array([[0x7F, 0xFF]], np.uint8)
    x = np.array([[1.0, 2.0]], np.float32)
    y, _ = oracle.f8_matvec(w, np.full((1, 1), 127, np.uint8), x)
    assert y[0, 0] == 448.0 - 896.0
    y, _ = oracle.f8_matvec(w, np.full((1, 1), 255, np.uint8), x)
    assert np.isnan(y[0, 0])


def test_threaded_oracle_equals_single_threaded():
    f = synth.f8_inputs(13, 97, 64, 5, 4, 120, 130, batch=2)
    a, _ = oracle.f8_matvec(f.w, f.scale, f.x)
    b, _ = oracle.f8_matvec(f.w, f.scale, f.x, threads=4)
    assert np.array_equal(a, b)
    c, m = _cq(3, output=50)
    p = oracle.cq_prepare(c.x, c.input_padded, c.group)
    assert np.array_equal(m.matvec(p)[0], m.matvec(p, threads=3)[0])


# ---------------------------------------------------------------------------
# greedy selection over head outputs
# ---------------------------------------------------------------------------

def test_argmax_matches_numpy_including_ties_and_nans():
    rng = np.random.default_rng(21)
    for trial in range(200):
        n = int(rng.integers(1, 60))
        y = rng.integers(-3, 4, n).astype(np.float32)  # many ties
        if trial % 3 == 0:
            y[rng.integers(0, n, 2)] = np.nan
        if trial % 5 == 0:
            y[:] = -np.inf
        assert oracle.argmax_rows(y)[0] == np.argmax(y)  # numpy: first NaN, first max


def test_argmax_hand_cases():
    assert list(oracle.argmax_rows(np.array([[1, 3, 3, 2], [np.nan, 5, np.nan, 9]],
                                            np.float32))) == [1, 0]
    assert oracle.argmax_rows(np.array([[-np.inf, -np.inf]], np.float32))[0] == 0


# ---------------------------------------------------------------------------
# I8 matvec with per-16 E8M0 group scales
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("R,C", [(5, 16), (7, 37), (3, 1), (40, 100)])
def test_i8_matches_expanded_group_scales(R, C):
    f = synth.i8_inputs(R + C, R, C, 100, 140, batch=3)
    y, mag = oracle.i8_matvec(f.w, f.scale, f.x)
    S = np.exp2(np.repeat(f.scale.astype(np.float64), 16, axis=1)[:, :C] - 127)
    W = f.w.astype(np.float64) * S
    assert np.allclose(y, f.x.astype(np.float64) @ W.T, rtol=1e-13, atol=1e-300)
    assert np.allclose(mag, np.abs(f.x.astype(np.float64)) @ np.abs(W).T, rtol=1e-13)


def test_i8_hand_cases():
    # one group of 16 weights (1..16) at scale 2^1, x = 1: y = 2 * 136
    w = np.arange(1, 17, dtype=np.int8)[None, :]
    y, _ = oracle.i8_matvec(w, np.array([[128]], np.uint8), np.ones((1, 16), np.float32))
    assert y[0, 0] == 272.0
    # the 17th column starts a new group: its scale alone changes y
    w = np.zeros((1, 17), np.int8)
    w[0, 16] = -128
    y, _ = oracle.i8_matvec(w, np.array([[127, 130]], np.uint8), np.ones((1, 17), np.float32))
    assert y[0, 0] == -1024.0
    y, _ = oracle.i8_matvec(w, np.array([[127, 255]], np.uint8), np.ones((1, 17), np.float32))
    assert np.isnan(y[0, 0])


# ---------------------------------------------------------------------------
# Hadamard MLP block (needle.js "Inference engine, part 2", section 8)
# ---------------------------------------------------------------------------

def test_silu_matches_scipy_expit():
    from scipy.special import expit
    v = np.concatenate([np.linspace(-50, 50, 2001), [-745.0, -200.0, 0.0, 1e-300, 200.0, 700.0]])
    got = oracle.silu_f64(v)
    want = v * expit(v)
    assert np.allclose(got, want, rtol=4e-16, atol=0)


@pytest.mark.parametrize("D,n", [(1, 1), (2, 1), (16, 16), (64, 50), (512, 512), (1024, 700)])
def test_hadamard_mlp_f64_matches_dense_hadamard(D, n):
    """Dense-matrix restatement: two Sylvester-matrix products instead of the
    butterfly, scipy's logistic function instead of exp."""
    from scipy.special import expit
    rng = np.random.default_rng(D * 31 + n)
    x = rng.standard_normal((3, n)).astype(np.float32)
    d1, d2, d3 = (rng.uniform(-1.5, 1.5, D).astype(np.float32) for _ in range(3))
    res = rng.standard_normal((3, n)).astype(np.float32)
    u = rng.standard_normal((3, n)).astype(np.float32)
    got, mag = oracle.hadamard_mlp(x, D, d1, d2, d3, res, u, mode="f64")
    Hn = hadamard(D) / math.sqrt(D)
    z = np.zeros((3, D))
    z[:, :n] = x
    z = (z * d1) @ Hn.T
    z = d2 * z
    silu = z * expit(z)
    z = (silu @ Hn.T) * d3
    want = (res + z[:, :n]) - u
    assert np.all(np.abs(got - want) <= 1e-12 * mag + 1e-300)
    # mag is the size of exactly the terms the last transform and the
    # epilogue add: sum_j |Hn[i, j] * silu_j * d3_i| + |residual_i| + |u_i|
    want_mag = (np.abs(silu) @ np.abs(Hn).T) * np.abs(d3)
    want_mag = want_mag[:, :n] + np.abs(res) + np.abs(u)
    assert np.allclose(mag, want_mag, rtol=1e-12, atol=0)


def test_hadamard_mlp_tanh_closed_form():
    """D = 4, x = [1, 1], d1 = 1, d2 = [2, 1, -2, 1]: the first transform gives
    [1, 0, 1, 0] exactly, silu gives [s(2), 0, s(-2), 0], and since
    s(a) + s(-a) = a tanh(a/2) and s(a) - s(-a) = a the second gives
    [tanh 1, tanh 1, 1, 1]."""
    x = np.array([[1.0, 1.0]], dtype=np.float32)
    d1 = np.ones(4, dtype=np.float32)
    d2 = np.array([2, 1, -2, 1], dtype=np.float32)
    d3 = np.array([1, -3, 5, 7], dtype=np.float32)
    got64, _ = oracle.hadamard_mlp(x, 4, d1, d2, d3, mode="f64")
    assert np.allclose(got64[0], [math.tanh(1.0), -3 * math.tanh(1.0)], rtol=1e-15, atol=0)
    got32, _ = oracle.hadamard_mlp(x, 4, d1, d2, d3, mode="f32")
    assert np.allclose(got32[0], [math.tanh(1.0), -3 * math.tanh(1.0)], rtol=3e-7, atol=0)


@pytest.mark.parametrize("k", [0, 5, 13])
def test_hadamard_mlp_identity_silu_closed_form(k):
    """x = 2 e_k, D = 16, d1 = 1: the first normalised transform is
    H[:, k] / 2 exactly.  With d2 = 128 H[:, k] every silu input is +64, where
    e^-64 is below half an ulp of 1 in float64, so silu is the identity and
    the second transform collapses the constant 64 onto output 0: 256 d3[0],
    zero elsewhere, exactly."""
    D = 16
    H = hadamard(D)
    x = np.zeros((1, D), dtype=np.float32)
    x[0, k] = 2.0
    d1 = np.ones(D, dtype=np.float32)
    d2 = (128.0 * H[:, k]).astype(np.float32)
    d3 = np.linspace(-2, 3, D).astype(np.float32)
    res = np.full((1, D), 0.5, dtype=np.float32)
    u = np.full((1, D), 0.25, dtype=np.float32)
    got, _ = oracle.hadamard_mlp(x, D, d1, d2, d3, res, u, mode="f32")
    want = np.full(D, 0.25, dtype=np.float32)
    want[0] = np.float32(np.float32(0.5) + np.float32(256.0) * d3[0]) - np.float32(0.25)
    assert np.array_equal(got[0], want)


def test_hadamard_mlp_zero_gate_leaves_residual_minus_u():
    """d2 = 0: silu(0) = 0, the rest of the block is zero and the update is
    residual - u, one float32 subtraction."""
    rng = np.random.default_rng(5)
    D, n = 64, 40
    x = rng.standard_normal((2, n)).astype(np.float32)
    d1, d3 = (rng.standard_normal(D).astype(np.float32) for _ in range(2))
    res = rng.standard_normal((2, n)).astype(np.float32)
    u = rng.standard_normal((2, n)).astype(np.float32)
    got, _ = oracle.hadamard_mlp(x, D, d1, np.zeros(D, np.float32), d3, res, u)
    assert np.array_equal(got, res - u)
    bare, _ = oracle.hadamard_mlp(x, D, d1, np.zeros(D, np.float32), d3)
    assert np.array_equal(bare, np.zeros_like(bare))


def test_hadamard_mlp_pads_before_the_first_diagonal():
    """The page pads, then multiplies by d1: an infinite d1 entry in the
    padding meets a zero and makes NaN, which the transform spreads to every
    output."""
    D, n = 32, 20
    rng = np.random.default_rng(6)
    x = rng.standard_normal((1, n)).astype(np.float32)
    d1, d2, d3 = (rng.standard_normal(D).astype(np.float32) for _ in range(3))
    finite, _ = oracle.hadamard_mlp(x, D, d1, d2, d3)
    assert np.all(np.isfinite(finite))
    d1[25] = np.inf
    got, _ = oracle.hadamard_mlp(x, D, d1, d2, d3)
    assert np.all(np.isnan(got))


def test_hadamard_mlp_silu_on_the_float64_product():
    """needle-2 section 8 stores silu(d2 * z) into a Float32Array from JS
    numbers: the product d2 * z is the exact float64 one and silu is
    evaluated in float64, then rounded once.  At D = 1 both normalised
    transforms are the identity (1/sqrt(1) = 1), so with d1 = d3 = 1 the block
    returns RN32(silu(d2 * x)).  Expected values use scipy's logistic function
    (v * expit(v)); inputs whose float64 value lies within 2^-40 relative of a
    float32 rounding midpoint are skipped, so the two float64 formulations
    round the same way."""
    from scipy.special import expit
    rng = np.random.default_rng(77)
    x = rng.uniform(-6, 6, 512).astype(np.float32)
    d2 = rng.uniform(0.5, 3.0, 512).astype(np.float32)
    one = np.ones(1, np.float32)
    checked = 0
    for xi, gi in zip(x, d2):
        v = float(gi) * float(xi)  # exact: two float32 factors
        w = v * float(expit(v))
        lo = float(np.float32(w))
        nxt = float(np.nextafter(np.float32(lo), np.float32(np.inf if w > lo else -np.inf)))
        mid = (lo + nxt) / 2
        if abs(w - mid) <= 2.0 ** -40 * abs(w):
            continue
        got, _ = oracle.hadamard_mlp(np.array([[xi]], np.float32), 1, one,
                                     np.array([gi], np.float32), one, mode="f32")
        assert got[0, 0] == np.float32(w), (xi, gi)
        checked += 1
    assert checked > 500


def test_hadamard_mlp_scale_rounding_golden():
    """needle-2 section 8 with the normalized FWHT of sections 1-2 at D = 2 and
    D = 8, where 1/sqrt(D) is not a power of two: both transforms scale by the
    float64 product rounded to float32.  Values derived by hand in the file
    (silu is the identity there); a float32 scale in either transform changes
    an output bit pattern."""
    cases = {}
    for row in read_golden("hadamard_mlp_scale_rounding.txt"):
        cases.setdefault(row[0], {})[row[1]] = np.array([parse_float(t) for t in row[2:]],
                                                        np.float32)
    for name, c in cases.items():
        D = c["d1"].size
        got, _ = oracle.hadamard_mlp(c["x"][None, :], D, c["d1"], c["d2"], c["d3"],
                                     c["residual"][None, :], c["u"][None, :], mode="f32")
        assert np.array_equal(got[0].view(np.uint32), c["out"].view(np.uint32)), name


@pytest.mark.parametrize("D,n", [(256, 256), (2048, 512)])
def test_hadamard_mlp_f32_staging_within_f64_bound(D, n):
    rng = np.random.default_rng(D + n)
    x = rng.standard_normal((2, n)).astype(np.float32)
    d1, d2, d3 = (rng.uniform(-1.5, 1.5, D).astype(np.float32) for _ in range(3))
    res = rng.standard_normal((2, n)).astype(np.float32)
    u = rng.standard_normal((2, n)).astype(np.float32)
    g32, mag = oracle.hadamard_mlp(x, D, d1, d2, d3, res, u)
    g64, _ = oracle.hadamard_mlp(x, D, d1, d2, d3, res, u, mode="f64")
    assert np.all(np.abs(g32 - g64) <= 2e-6 * mag)
