"""Seeded synthetic inputs for the quantized-weight matvec path.

This module is shared by the tests, the bench and the oracle checks.  It
holds none of the method's arithmetic: it only draws random bytes, levels,
norms, activations and row ids with numpy, in a fixed sub-stream order
(packed indices, norms, x, row ids), so that the CUDA path and the oracle
see identical inputs.

Workloads (the shapes named by the pages' CQ and F8 formats):

* ``cq4_512``       CQ 4-bit, output 512, input 512, group 64, batch 1.
* ``cq_sweep``      CQ 2/3/4/5-bit, output 2048, input 512, group 64,
                    batch 1 and 4.
* ``cq2_vocab``     CQ 2-bit vocabulary-projection shape: output 32768,
                    input 500 padded to 512, group 128, x ~ 3 N(0,1), plus
                    a 64-row gather (the tied embedding lookup).
* ``f8_4096``       F8 E4M3, 4096 x 4096, E8M0 scales [32, 32] with
                    exponents in [120, 130], batch 1 and 8.
* ``f8_head``       F8 E4M3 head shape, 245760 x 4096 (~1 GB), scales
                    [1920, 32] with exponents in [118, 132], batch 1/2/4/8.
* ``i8_4096``       I8, 4096 x 4096, per-16 E8M0 group scales with
                    exponents in [110, 124], batch 1 and 8.
* ``i8_head``       I8 head shape (the run's "I8 head (246k vocab)"),
                    245760 x 4096, batch 1, 2, 4 and 8.
* ``hmlp_512``      Hadamard MLP block on the 512-value block input with no
                    widening (D = 512), batch 1 and 4.
* ``hmlp_2048``     the same block widened to D = 2048, batch 1, 4 and 8.

Hadamard MLP inputs: x ~ N(0,1) (a normalised vector has unit RMS), the
three diagonals uniform in magnitude over [0.5, 1.5] with random signs,
residual and u ~ N(0,1).

Packed CQ rows are drawn as uniform random bytes: for every bit width this
makes every index uniform over [0, 2^bits) (the 2/4-bit layouts are two
/ four codes per byte, 3/5-bit a little-endian bit stream per row).
"""
from __future__ import annotations

from dataclasses import dataclass
from statistics import NormalDist

import numpy as np


# --------------------------------------------------------------------------
# workload table
# --------------------------------------------------------------------------

WORKLOADS = {
    "cq4_512": dict(kind="cq", seed=1, output=512, input=512, group=64, bits=(4,),
                    batch=(1,), x_scale=1.0),
    "cq_sweep": dict(kind="cq", seed=2, output=2048, input=512, group=64, bits=(2, 3, 4, 5),
                     batch=(1, 4), x_scale=1.0),
    "cq2_vocab": dict(kind="cq", seed=3, output=32768, input=500, group=128, bits=(2,),
                      batch=(1,), x_scale=3.0, gather=64),
    "f8_4096": dict(kind="f8", seed=4, R=4096, C=4096, SR=32, SC=32, e_lo=120, e_hi=130,
                    batch=(1, 8)),
    "f8_head": dict(kind="f8", seed=5, R=245760, C=4096, SR=1920, SC=32, e_lo=118, e_hi=132,
                    batch=(1, 2, 4, 8)),
    "i8_4096": dict(kind="i8", seed=6, R=4096, C=4096, e_lo=110, e_hi=124, batch=(1, 8)),
    "i8_head": dict(kind="i8", seed=7, R=245760, C=4096, e_lo=110, e_hi=124, batch=(1, 2, 4, 8)),
    "hmlp_512": dict(kind="hmlp", seed=8, n=512, D=512, batch=(1, 4)),
    "hmlp_2048": dict(kind="hmlp", seed=9, n=512, D=2048, batch=(1, 4, 8)),
}


def padded_width(input_: int, group: int) -> int:
    """Smallest multiple of ``group`` that holds ``input_`` columns."""
    return -(-input_ // group) * group


def row_bytes_for(input_padded: int, bits: int) -> int:
    """Bytes per packed row: ceil(input_padded * bits / 8)."""
    return (input_padded * bits + 7) // 8


def quantile_codebook(bits: int) -> np.ndarray:
    """2^bits sorted float32 levels at the N(0,1) quantiles (i + 1/2) / 2^bits."""
    n = 1 << bits
    nd = NormalDist()
    return np.array([nd.inv_cdf((i + 0.5) / n) for i in range(n)], dtype=np.float32)


# --------------------------------------------------------------------------
# CQ inputs
# --------------------------------------------------------------------------

@dataclass
class CQInputs:
    output: int
    input: int
    input_padded: int
    group: int
    bits: int
    row_bytes: int
    packed: np.ndarray     # [output, row_bytes] uint8
    norms: np.ndarray      # [output, input_padded // group] uint16 (binary16 bits)
    codebook: np.ndarray   # [2^bits] float32
    x: np.ndarray          # [batch, input] float32
    rows: np.ndarray       # [n_gather] int32 row ids


def cq_inputs(seed: int, output: int, input: int, group: int, bits: int, batch: int = 1,
              x_scale: float = 1.0, gather: int = 0, input_padded: int | None = None,
              codebook: np.ndarray | None = None) -> CQInputs:
    """Seeded CQ matrix + activations.  Sub-streams: packed, norms, x, row ids."""
    P = padded_width(input, group) if input_padded is None else int(input_padded)
    rb = row_bytes_for(P, bits)
    ss = np.random.SeedSequence([int(seed), int(bits), int(batch), int(output), int(P)])
    g_pack, g_norm, g_x, g_rows = (np.random.default_rng(s) for s in ss.spawn(4))
    packed = g_pack.integers(0, 256, size=(output, rb), dtype=np.uint8)
    norms = (np.abs(g_norm.standard_normal((output, P // group))) + 0.1).astype(np.float16)
    x = (g_x.standard_normal((batch, input)) * x_scale).astype(np.float32)
    rows = g_rows.integers(0, max(output, 1), size=gather, dtype=np.int64).astype(np.int32)
    cb = quantile_codebook(bits) if codebook is None else np.asarray(codebook, np.float32)
    return CQInputs(output, input, P, group, bits, rb, packed, norms.view(np.uint16), cb, x,
                    rows)


# --------------------------------------------------------------------------
# F8 inputs
# --------------------------------------------------------------------------

@dataclass
class F8Inputs:
    R: int
    C: int
    SR: int
    SC: int
    w: np.ndarray       # [R, C] uint8 E4M3 codes
    scale: np.ndarray   # [SR, SC] uint8 E8M0 codes
    x: np.ndarray       # [batch, C] float32


def finite_e4m3_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniform over the 254 E4M3 byte codes other than 0x7F and 0xFF."""
    v = rng.integers(0, 254, size=shape, dtype=np.uint8)
    v += (v >= 127).astype(np.uint8)
    return v


def f8_inputs(seed: int, R: int, C: int, SR: int, SC: int, e_lo: int, e_hi: int,
              batch: int = 1, finite_only: bool = True) -> F8Inputs:
    """Seeded F8 weights, E8M0 scales (uniform integers in [e_lo, e_hi]) and x."""
    ss = np.random.SeedSequence([int(seed), int(R), int(C), int(batch)])
    g_w, g_s, g_x = (np.random.default_rng(s) for s in ss.spawn(3))
    if finite_only:
        w = finite_e4m3_codes(g_w, (R, C))
    else:
        w = g_w.integers(0, 256, size=(R, C), dtype=np.uint8)
    scale = g_s.integers(e_lo, e_hi + 1, size=(SR, SC), dtype=np.int64).astype(np.uint8)
    x = g_x.standard_normal((batch, C)).astype(np.float32)
    return F8Inputs(R, C, SR, SC, w, scale, x)


@dataclass
class I8Inputs:
    R: int
    C: int
    w: np.ndarray       # [R, C] int8
    scale: np.ndarray   # [R, ceil(C/16)] uint8 E8M0 codes
    x: np.ndarray       # [batch, C] float32


def i8_inputs(seed: int, R: int, C: int, e_lo: int, e_hi: int, batch: int = 1) -> I8Inputs:
    """Seeded int8 weights (uniform over [-128, 127]), per-16 E8M0 group scales
    (uniform integers in [e_lo, e_hi]) and x ~ N(0,1)."""
    ss = np.random.SeedSequence([int(seed), int(R), int(C), int(batch), 8])
    g_w, g_s, g_x = (np.random.default_rng(s) for s in ss.spawn(3))
    w = g_w.integers(-128, 128, size=(R, C), dtype=np.int8)
    scale = g_s.integers(e_lo, e_hi + 1, size=(R, (C + 15) // 16), dtype=np.int64).astype(np.uint8)
    x = g_x.standard_normal((batch, C)).astype(np.float32)
    return I8Inputs(R, C, w, scale, x)


@dataclass
class HMLPInputs:
    n: int
    D: int
    x: np.ndarray         # [batch, n] float32
    d1: np.ndarray        # [D] float32
    d2: np.ndarray
    d3: np.ndarray
    residual: np.ndarray  # [batch, n] float32
    u: np.ndarray         # [batch, n] float32


def hmlp_inputs(seed: int, n: int, D: int, batch: int = 1) -> HMLPInputs:
    """Seeded Hadamard MLP inputs.  Sub-streams: x, d1, d2, d3, residual, u."""
    ss = np.random.SeedSequence([int(seed), int(n), int(D), int(batch), 9])
    g = [np.random.default_rng(s) for s in ss.spawn(6)]

    def diag(r):
        mag = r.uniform(0.5, 1.5, D)
        return np.where(r.random(D) < 0.5, -mag, mag).astype(np.float32)

    x = g[0].standard_normal((batch, n)).astype(np.float32)
    d1, d2, d3 = diag(g[1]), diag(g[2]), diag(g[3])
    res = g[4].standard_normal((batch, n)).astype(np.float32)
    u = g[5].standard_normal((batch, n)).astype(np.float32)
    return HMLPInputs(n, D, x, d1, d2, d3, res, u)


def workload_inputs(name: str, bits: int | None = None, batch: int = 1):
    """Inputs for one named workload at one bit width / batch."""
    w = WORKLOADS[name]
    if w["kind"] == "cq":
        b = w["bits"][0] if bits is None else bits
        return cq_inputs(w["seed"], w["output"], w["input"], w["group"], b, batch,
                         w["x_scale"], w.get("gather", 0))
    if w["kind"] == "i8":
        return i8_inputs(w["seed"], w["R"], w["C"], w["e_lo"], w["e_hi"], batch)
    if w["kind"] == "hmlp":
        return hmlp_inputs(w["seed"], w["n"], w["D"], batch)
    return f8_inputs(w["seed"], w["R"], w["C"], w["SR"], w["SC"], w["e_lo"], w["e_hi"], batch)
