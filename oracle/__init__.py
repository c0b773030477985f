"""Plain CPU oracle for the quantized-weight matvec path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.
The product library (``quantized_weight_matvec_gb300``) never imports it,
and this package never imports the product library.

The arithmetic lives in ``oracle.c`` (float64, ``-ffp-contract=off``); this
module only builds it with gcc and marshals numpy arrays through ctypes.
Every function cites the page section it follows:

* ``needle-2`` -- needle.js tutorial "Inference engine, part 2: kernels and
  token step": section 1 (FWHT), section 2 (prepare), section 3 (packed-row
  dot) and "Row gather" (dequantizeRow).
* ``needle-1`` -- needle.js tutorial "Inference engine, part 1: loader and
  tokenizer": section 3 (FP16 decode) and section 4 (CqMatrix).
* ``mnemonic`` -- Mnemonic "In the browser", "Dot products and math"
  (int8 activations quantized per group of 32, exact int32 dot sums).
* ``ds4f-6`` -- ds4f-disk issue #6 "attention + tokenizer + sampling",
  work item 1 / step 1 (F8 E4M3 + E8M0 block-scaled matvec), step 4 (I8
  matvec with per-16 E8M0 group scales), work item 3 /
  step 3 (head logits then sampling: greedy selection and top-k
  temperature sampling).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against values the pages fix, closed forms, library routines (numpy float16,
torch float8 decode, numpy matmul) or brute force.  None is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into liboracle.so next to it."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-fvisibility=hidden", "-o", tmp, _SRC,
           "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _CQ(ctypes.Structure):
    _fields_ = [("output", ctypes.c_int64), ("input", ctypes.c_int64),
                ("input_padded", ctypes.c_int64), ("group", ctypes.c_int64),
                ("bits", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("row_bytes", ctypes.c_int64),
                ("packed", ctypes.c_void_p), ("norms", ctypes.c_void_p),
                ("codebook", ctypes.c_void_p)]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    lib.orc_f16_to_f32.argtypes, lib.orc_f16_to_f32.restype = [ctypes.c_uint16], F
    lib.orc_e4m3_to_f32.argtypes, lib.orc_e4m3_to_f32.restype = [ctypes.c_uint8], F
    lib.orc_e8m0_to_f32.argtypes, lib.orc_e8m0_to_f32.restype = [ctypes.c_uint8], F
    lib.orc_fwht_f64.argtypes, lib.orc_fwht_f64.restype = [P, I64], None
    lib.orc_fwht_f32.argtypes, lib.orc_fwht_f32.restype = [P, I64], None
    lib.orc_cq_index.argtypes, lib.orc_cq_index.restype = [P, I64, I32, I64, I64], I32
    lib.orc_cq_prepare.argtypes = [P, I64, I64, I64, I64, ctypes.c_int, P, P]
    lib.orc_cq_prepare.restype = ctypes.c_int
    lib.orc_cq_matvec.argtypes = [ctypes.POINTER(_CQ), P, I64, P, P, I64, I64]
    lib.orc_cq_matvec.restype = ctypes.c_int
    lib.orc_cq_matvec_mt.argtypes = [ctypes.POINTER(_CQ), P, I64, P, P, I64, I64, ctypes.c_int]
    lib.orc_cq_matvec_mt.restype = ctypes.c_int
    lib.orc_cq_dequantize_row.argtypes = [ctypes.POINTER(_CQ), P, I64, P]
    lib.orc_cq_dequantize_row.restype = ctypes.c_int
    lib.orc_f8_matvec.argtypes = [P, I64, I64, P, I64, I64, P, I64, P, P, I64, I64]
    lib.orc_f8_matvec.restype = ctypes.c_int
    lib.orc_f8_matvec_mt.argtypes = [P, I64, I64, P, I64, I64, P, I64, P, P, I64, I64,
                                     ctypes.c_int]
    lib.orc_f8_matvec_mt.restype = ctypes.c_int
    lib.orc_i8_matvec.argtypes = [P, I64, I64, P, P, I64, P, P, I64, I64]
    lib.orc_i8_matvec.restype = ctypes.c_int
    lib.orc_i8_matvec_mt.argtypes = [P, I64, I64, P, P, I64, P, P, I64, I64, ctypes.c_int]
    lib.orc_i8_matvec_mt.restype = ctypes.c_int
    lib.orc_i8_quantize_x.argtypes = [P, I64, I64, P, P]
    lib.orc_i8_quantize_x.restype = ctypes.c_int
    lib.orc_i8_matvec_q8.argtypes = [P, I64, I64, P, P, P, I64, P, P, I64, I64]
    lib.orc_i8_matvec_q8.restype = ctypes.c_int
    lib.orc_i8_matvec_q8_mt.argtypes = [P, I64, I64, P, P, P, I64, P, P, I64, I64, ctypes.c_int]
    lib.orc_i8_matvec_q8_mt.restype = ctypes.c_int
    lib.orc_silu_f64.argtypes, lib.orc_silu_f64.restype = [ctypes.c_double], ctypes.c_double
    lib.orc_hadamard_mlp.argtypes = [P, I64, I64, P, P, P, P, P, I64, ctypes.c_int, P, P, P]
    lib.orc_hadamard_mlp.restype = ctypes.c_int
    lib.orc_argmax_f32.argtypes = [P, I64]
    lib.orc_argmax_f32.restype = I64
    lib.orc_topk_sample.argtypes = [P, I64, I64, ctypes.c_double, ctypes.c_double, P, P, P]
    lib.orc_topk_sample.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# scalar decodes
# --------------------------------------------------------------------------

def f16_to_f32(codes) -> np.ndarray:
    """IEEE binary16 bit patterns -> float32 values (needle-1 section 3)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint16).ravel()
    return np.array([lib.orc_f16_to_f32(int(h)) for h in c], dtype=np.float32).reshape(
        np.shape(codes))


def e4m3_to_f32(codes) -> np.ndarray:
    """F8 E4M3 bytes -> float32 values, e=0 subnormal, clamp at 448 (ds4f-6 item 1)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_e4m3_to_f32(int(b)) for b in c], dtype=np.float32).reshape(
        np.shape(codes))


def e8m0_to_f32(codes) -> np.ndarray:
    """E8M0 bytes -> 2^(e-127) as float32; 255 read as NaN (ds4f-6 step 1)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_e8m0_to_f32(int(b)) for b in c], dtype=np.float32).reshape(
        np.shape(codes))


# --------------------------------------------------------------------------
# FWHT and prepare
# --------------------------------------------------------------------------

def fwht_f64(x) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform in float64 (needle-2 section 1)."""
    v = _c(x, np.float64).copy()
    _load().orc_fwht_f64(_ptr(v), v.size)
    return v


def fwht_f32(x) -> np.ndarray:
    """The same transform with every butterfly result stored as float32."""
    v = _c(x, np.float32).copy()
    _load().orc_fwht_f32(_ptr(v), v.size)
    return v


def cq_prepare(x, input_padded: int, group: int, mode: str = "f32") -> np.ndarray:
    """prepare(): pad, per-group FWHT, times 1/sqrt(group) (needle-2 section 2).

    ``x`` is [batch, input] float32.  mode "f32" reproduces the page's float32
    staging exactly (bit-exact target); mode "f64" stays in float64."""
    x = _c(np.atleast_2d(x), np.float32)
    batch, inp = x.shape
    if mode == "f32":
        out = np.empty((batch, input_padded), dtype=np.float32)
        _load().orc_cq_prepare(_ptr(x), batch, inp, input_padded, group, 0, _ptr(out), None)
    elif mode == "f64":
        out = np.empty((batch, input_padded), dtype=np.float64)
        _load().orc_cq_prepare(_ptr(x), batch, inp, input_padded, group, 1, None, _ptr(out))
    else:
        raise ValueError(mode)
    return out


# --------------------------------------------------------------------------
# CQ matrix
# --------------------------------------------------------------------------

class CQMatrix:
    """The page's CqMatrix (needle-1 section 4) over numpy arrays."""

    def __init__(self, output, input, input_padded, group, bits, packed, norms, codebook):
        self.output, self.input = int(output), int(input)
        self.input_padded, self.group, self.bits = int(input_padded), int(group), int(bits)
        self.packed = _c(packed, np.uint8)
        self.norms = _c(norms, np.uint16)
        self.codebook = _c(codebook, np.float32)
        self.row_bytes = self.packed.shape[1] if self.packed.ndim == 2 else \
            (self.input_padded * self.bits + 7) // 8
        self._s = _CQ(self.output, self.input, self.input_padded, self.group, self.bits, 0,
                      self.row_bytes, _ptr(self.packed), _ptr(self.norms),
                      _ptr(self.codebook))

    def index(self, r: int, k: int) -> int:
        """Codebook index of column k in row r (little-endian bit stream)."""
        return int(_load().orc_cq_index(_ptr(self.packed), self.row_bytes, self.bits, r, k))

    def matvec(self, prepared, rows=None, threads: int = 1, with_mag: bool = True):
        """cqMatvec (needle-2 section 3) in float64.

        ``prepared`` is [batch, input_padded] (float32 or float64, read as
        float64).  Returns (y, mag), both [batch, output] float64 (only the
        rows in ``rows=(r0, r1)`` are filled when given)."""
        p = _c(np.atleast_2d(prepared), np.float64)
        batch = p.shape[0]
        r0, r1 = (0, self.output) if rows is None else rows
        y = np.zeros((batch, self.output), dtype=np.float64)
        mag = np.zeros((batch, self.output), dtype=np.float64) if with_mag else None
        lib = _load()
        if threads > 1:
            lib.orc_cq_matvec_mt(ctypes.byref(self._s), _ptr(p), batch, _ptr(y),
                                 _ptr(mag) if with_mag else None, r0, r1, threads)
        else:
            lib.orc_cq_matvec(ctypes.byref(self._s), _ptr(p), batch, _ptr(y),
                              _ptr(mag) if with_mag else None, r0, r1)
        return y, mag

    def dequantize_rows(self, rows):
        """dequantizeRow (needle-2 "Row gather") for each id: [n, input] float32.

        Returns (out, bad) where bad is True if any id was out of range (its
        row is zeros)."""
        ids = _c(np.atleast_1d(rows), np.int32)
        out = np.empty((ids.size, self.input), dtype=np.float32)
        bad = _load().orc_cq_dequantize_row(ctypes.byref(self._s), _ptr(ids), ids.size,
                                            _ptr(out))
        if bad < 0:
            raise MemoryError("oracle dequantize_row")
        return out, bool(bad)


# --------------------------------------------------------------------------
# F8 E4M3 + E8M0
# --------------------------------------------------------------------------

def f8_matvec(w, scale, x, rows=None, threads: int = 1, with_mag: bool = True):
    """Block-scaled F8 matvec (ds4f-6 step 1) in float64.

    ``w`` [R, C] uint8 E4M3, ``scale`` [SR, SC] uint8 E8M0, ``x`` [batch, C]
    float32.  Returns (y, mag) [batch, R] float64; only rows in
    ``rows=(r0, r1)`` are filled when given."""
    w = _c(w, np.uint8)
    scale = _c(scale, np.uint8)
    x = _c(np.atleast_2d(x), np.float32)
    R, C = w.shape
    SR, SC = scale.shape
    batch = x.shape[0]
    r0, r1 = (0, R) if rows is None else rows
    y = np.zeros((batch, R), dtype=np.float64)
    mag = np.zeros((batch, R), dtype=np.float64) if with_mag else None
    lib = _load()
    args = (_ptr(w), R, C, _ptr(scale), SR, SC, _ptr(x), batch, _ptr(y),
            _ptr(mag) if with_mag else None, r0, r1)
    if threads > 1:
        lib.orc_f8_matvec_mt(*args, threads)
    else:
        lib.orc_f8_matvec(*args)
    return y, mag


def argmax_rows(y) -> np.ndarray:
    """Greedy selection per row of y [batch, n] float32 (ds4f-6 work item 3 /
    step 3): NaN above every number, then the larger value, then the lower
    index.  Returns int64 [batch]."""
    y = _c(np.atleast_2d(y), np.float32)
    lib = _load()
    return np.array([lib.orc_argmax_f32(_ptr(row), row.size) for row in y], dtype=np.int64)


def topk_sample(y, k: int, temperature: float, u):
    """Top-k temperature sampling per row of y [batch, n] float32 (ds4f-6
    work item 3 / step 3), in float64: the k best entries in the greedy
    order, weights exp((l_i - l_0) / T), probabilities w / sum(w), and the
    first entry whose cumulative weight exceeds u * sum(w).  ``u`` holds one
    uniform draw per row.  Returns (index [batch, k] int64 best first,
    prob [batch, k] float64, token [batch] int64)."""
    y = _c(np.atleast_2d(y), np.float32)
    batch, n = y.shape
    u = np.broadcast_to(np.asarray(u, dtype=np.float64), (batch,))
    index = np.zeros((batch, k), dtype=np.int64)
    prob = np.zeros((batch, k), dtype=np.float64)
    token = np.zeros(batch, dtype=np.int64)
    lib = _load()
    for v in range(batch):
        rc = lib.orc_topk_sample(_ptr(y[v]), n, k, float(temperature), float(u[v]),
                                 _ptr(index[v]), _ptr(prob[v]), _ptr(token[v:]))
        if rc != 0:
            raise ValueError("topk_sample: k must be in [1, n] and temperature >= 0")
    return index, prob, token


def i8_matvec(w, scale, x, rows=None, threads: int = 1, with_mag: bool = True):
    """I8 matvec with per-16 E8M0 group scales (ds4f-6 step 4) in float64.

    ``w`` [R, C] int8, ``scale`` [R, ceil(C/16)] uint8 E8M0, ``x`` [batch, C]
    float32.  Returns (y, mag) [batch, R] float64."""
    w = _c(w, np.int8)
    scale = _c(scale, np.uint8)
    x = _c(np.atleast_2d(x), np.float32)
    R, C = w.shape
    assert scale.shape == (R, (C + 15) // 16)
    batch = x.shape[0]
    r0, r1 = (0, R) if rows is None else rows
    y = np.zeros((batch, R), dtype=np.float64)
    mag = np.zeros((batch, R), dtype=np.float64) if with_mag else None
    args = (_ptr(w), R, C, _ptr(scale), _ptr(x), batch, _ptr(y), _ptr(mag) if with_mag else None,
            r0, r1)
    lib = _load()
    if threads > 1:
        lib.orc_i8_matvec_mt(*args, threads)
    else:
        lib.orc_i8_matvec(*args)
    return y, mag


def i8_quantize_x(x):
    """Activations quantized to int8 per group of 32 columns (Mnemonic "In
    the browser", "Dot products and math"): d = max|x| / 127 and
    q = rint(x / d) clamped to [-127, 127], in float32 (see oracle.c).

    ``x`` [batch, C] float32.  Returns (q [batch, C] int8,
    d [batch, ceil(C/32)] float32)."""
    x = _c(np.atleast_2d(x), np.float32)
    batch, C = x.shape
    q = np.zeros((batch, C), dtype=np.int8)
    d = np.zeros((batch, (C + 31) // 32), dtype=np.float32)
    assert _load().orc_i8_quantize_x(_ptr(x), C, batch, _ptr(q), _ptr(d)) == 0
    return q, d


def i8_matvec_q8(w, scale, q, d, rows=None, threads: int = 1, with_mag: bool = True):
    """int8 weights (per-16 E8M0 group scales, ds4f-6 step 4) times int8
    activations with per-32 float32 scales (Mnemonic "In the browser"), in
    float64: y[v, r] = sum_c w[r, c] e8m0(scale[r, c/16]) q[v, c] d[v, c/32].

    ``w`` [R, C] int8, ``scale`` [R, ceil(C/16)] uint8, ``q`` [batch, C] int8,
    ``d`` [batch, ceil(C/32)] float32.  Returns (y, mag) [batch, R] float64."""
    w = _c(w, np.int8)
    scale = _c(scale, np.uint8)
    q = _c(np.atleast_2d(q), np.int8)
    d = _c(np.atleast_2d(d), np.float32)
    R, C = w.shape
    batch = q.shape[0]
    assert scale.shape == (R, (C + 15) // 16)
    assert q.shape == (batch, C) and d.shape == (batch, (C + 31) // 32)
    r0, r1 = (0, R) if rows is None else rows
    y = np.zeros((batch, R), dtype=np.float64)
    mag = np.zeros((batch, R), dtype=np.float64) if with_mag else None
    args = (_ptr(w), R, C, _ptr(scale), _ptr(q), _ptr(d), batch, _ptr(y),
            _ptr(mag) if with_mag else None, r0, r1)
    lib = _load()
    if threads > 1:
        lib.orc_i8_matvec_q8_mt(*args, threads)
    else:
        lib.orc_i8_matvec_q8(*args)
    return y, mag


def silu_f64(v) -> np.ndarray:
    """silu(v) = v / (1 + e^-v) in float64, elementwise (the activation of
    needle-2 section 8)."""
    v = np.asarray(v, dtype=np.float64)
    lib = _load()
    return np.array([lib.orc_silu_f64(float(t)) for t in v.ravel()]).reshape(v.shape)


def hadamard_mlp(x, D: int, d1, d2, d3, residual=None, u=None, mode: str = "f32"):
    """Hadamard MLP block of needle-2 section 8 from the normalised block input:
    pad to D, x d1, normalised FWHT, silu(d2 x .), normalised FWHT, x d3,
    first n values, then + residual and - u when given.

    ``x`` [batch, n] float32; d1..d3 [D] float32.  mode "f32" follows the
    page's Float32Array staging and returns float32; "f64" is float64
    throughout.  Returns (out, mag), both [batch, n]."""
    x = _c(np.atleast_2d(x), np.float32)
    batch, n = x.shape
    d1, d2, d3 = (_c(d, np.float32) for d in (d1, d2, d3))
    assert d1.shape == d2.shape == d3.shape == (D,) and n <= D
    res = None if residual is None else _c(np.atleast_2d(residual), np.float32)
    uu = None if u is None else _c(np.atleast_2d(u), np.float32)
    for t in (res, uu):
        assert t is None or t.shape == (batch, n)
    m = 0 if mode == "f32" else 1
    out32 = np.zeros((batch, n), dtype=np.float32)
    out64 = np.zeros((batch, n), dtype=np.float64)
    mag = np.zeros((batch, n), dtype=np.float64)
    st = _load().orc_hadamard_mlp(_ptr(x), n, D, _ptr(d1), _ptr(d2), _ptr(d3),
                                  None if res is None else _ptr(res),
                                  None if uu is None else _ptr(uu), batch, m,
                                  _ptr(out32), _ptr(out64), _ptr(mag))
    assert st == 0
    return (out32 if m == 0 else out64), mag
