"""CPU checks of the C-ABI library: it loads, exports every declared symbol,
and rejects invalid arguments on the host before any launch.

Nothing here touches a GPU: every call below fails validation, and the
library returns its status before calling the CUDA runtime.
"""
import ctypes
import os
import re
import subprocess

import pytest

from quantized_weight_matvec_gb300 import build_lib, qmv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmv.h")

# a fake, 256-byte aligned, never dereferenced device address
FAKE = 0x7F0000000000


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"QMV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_every_entry_point():
    names = declared_functions()
    for n in ("cq_prepare", "cq_matvec", "cq_dequantize_row", "f8_matvec", "f8_matvec_argmax",
              "cq_matvec_multi", "cq_prepare_matvec", "i8_matvec", "hadamard_mlp",
              "topk_sample", "f8_matvec_topk_sample", "i8_matvec_topk_sample",
              "i8_quantize_x", "i8_matvec_q8", "qmv_status_string", "qmv_abi_version",
              "qmv_tc_wait_timeouts"):
        assert n in names


def test_library_exports_every_declared_symbol():
    path = build_lib.build()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name)


def test_only_the_abi_is_exported():
    out = subprocess.run(["nm", "-D", "--defined-only", build_lib.build()], capture_output=True,
                         text=True, check=True).stdout
    funcs = {l.split()[-1] for l in out.splitlines() if l.split() and l.split()[-2] == "T"}
    assert funcs == set(declared_functions())


def test_status_strings_and_version():
    assert qmv.abi_version() == 1
    for code, name in qmv.STATUS_NAMES.items():
        assert qmv.status_string(code).startswith(name)


def _m(**kw):
    f = dict(output=64, input=500, input_padded=512, group=128, bits=2, row_bytes=128,
             packed=FAKE, norms=FAKE, codebook=FAKE)
    f.update(kw)
    return qmv.cq_struct(**f)


@pytest.mark.parametrize("kw,code", [
    (dict(bits=1), 3), (dict(bits=6), 3),
    (dict(group=96), 4), (dict(group=1), 4), (dict(group=1024), 4), (dict(group=65536), 4),
    (dict(input=0), 2), (dict(input=513), 2),
    (dict(row_bytes=125), 2), (dict(input_padded=500, row_bytes=125), 2),
    (dict(output=-1), 2), (dict(reserved=1), 2),
])
def test_cq_shape_rejections(kw, code):
    m = _m(**kw)
    assert qmv.cq_prepare(m, FAKE, 1, FAKE + 65536) == code
    assert qmv.cq_matvec(m, FAKE, 1, FAKE + 65536) == code
    assert qmv.cq_dequantize_row(m, FAKE, 1, FAKE + 65536) == code


def test_cq_batch_null_align_alias():
    m = _m()
    assert qmv.cq_prepare(m, FAKE, 0, FAKE + 65536) == 5
    assert qmv.cq_prepare(m, FAKE, 9, FAKE + 65536) == 5
    assert qmv.cq_prepare(m, 0, 1, FAKE + 65536) == 1
    assert qmv.cq_matvec(m, FAKE, 1, 0) == 1
    assert qmv.cq_matvec(_m(packed=0), FAKE, 1, FAKE + 65536) == 1
    assert qmv.cq_matvec(m, FAKE + 2, 1, FAKE + 65536) == 6
    assert qmv.cq_matvec(_m(norms=FAKE + 1), FAKE, 1, FAKE + 65536) == 6
    # y overlapping the prepared vector, or the packed rows
    assert qmv.cq_matvec(m, FAKE, 1, FAKE + 1024) == 8
    assert qmv.cq_matvec(_m(packed=FAKE + (1 << 20)), FAKE, 1, FAKE + (1 << 20) + 64) == 8
    assert qmv.cq_prepare(m, FAKE, 1, FAKE + 512) == 8
    assert qmv.cq_dequantize_row(m, FAKE, -1, FAKE + 65536) == 2
    assert qmv.cq_dequantize_row(m, FAKE, 0, FAKE + 65536) == 0  # empty: nothing to do
    assert qmv.cq_dequantize_row(m, FAKE + 2, 3, FAKE + 65536) == 6
    # empty matrix: valid, nothing launched
    assert qmv.cq_matvec(_m(output=0), FAKE, 1, FAKE + 65536) == 0


def test_tc_wait_timeouts_rejects_null():
    # checked before any CUDA call, so it runs without a GPU
    assert qmv.load().qmv_tc_wait_timeouts(0) == 1


def test_f8_rejections():
    W, S, X, Y = FAKE, FAKE + (1 << 30), FAKE + (1 << 31), FAKE + (1 << 32)
    assert qmv.f8_matvec(W, 16, 16, S, 1, 1, X, 0, Y) == 5
    assert qmv.f8_matvec(W, 16, 0, S, 1, 1, X, 1, Y) == 2
    assert qmv.f8_matvec(W, 16, 16, S, 17, 1, X, 1, Y) == 2
    assert qmv.f8_matvec(W, 16, 16, S, 1, 17, X, 1, Y) == 2
    assert qmv.f8_matvec(W, 16, 16, S, 0, 1, X, 1, Y) == 2
    assert qmv.f8_matvec(W, -1, 16, S, 1, 1, X, 1, Y) == 2
    assert qmv.f8_matvec(W, 1 << 41, 16, S, 1, 1, X, 1, Y) == 2
    assert qmv.f8_matvec(W, 1 << 39, 1 << 39, S, 1, 1, X, 1, Y) == 7
    assert qmv.f8_matvec(0, 16, 16, S, 1, 1, X, 1, Y) == 1
    assert qmv.f8_matvec(W, 16, 16, 0, 1, 1, X, 1, Y) == 1
    assert qmv.f8_matvec(W, 16, 16, S, 1, 1, X + 2, 1, Y) == 6
    assert qmv.f8_matvec(W, 16, 16, S, 1, 1, X, 1, W + 8) == 8
    assert qmv.f8_matvec(W, 16, 16, S, 1, 1, X, 1, X + 16) == 8
    assert qmv.f8_matvec(W, 0, 16, S, 1, 1, X, 1, 0) == 0  # R = 0: nothing to do


def test_f8_argmax_rejections():
    W, S, X, Y = FAKE, FAKE + (1 << 30), FAKE + (1 << 31), FAKE + (1 << 32)
    I, V, K = FAKE + (1 << 33), FAKE + (1 << 34), FAKE + (1 << 35)
    need = qmv.f8_argmax_workspace_bytes(2)
    assert need == 16 + 2048 * 2 * 16
    assert qmv.f8_argmax_logits_offset(2) == 65792  # need rounded up to 256 bytes
    assert qmv.f8_argmax_workspace_bytes(2, 1000) == 65792 + 2 * 1000 * 4  # ..._TC_BYTES(2, 1000)
    a = qmv.f8_matvec_argmax
    assert a(W, 0, 16, S, 1, 1, X, 2, Y, I, V, K, need) == 2          # R >= 1
    assert a(W, 16, 16, S, 1, 1, X, 2, Y, I, V, K, need - 1) == 2     # workspace too small
    assert a(W, 16, 16, S, 1, 1, X, 2, Y, 0, V, K, need) == 1         # out_index NULL
    assert a(W, 16, 16, S, 1, 1, X, 2, Y, I, V, 0, need) == 1         # workspace NULL
    assert a(W, 16, 16, S, 1, 1, X, 2, Y, I + 4, V, K, need) == 6     # int64 alignment
    assert a(W, 16, 16, S, 1, 1, X, 2, Y, I, V, K + 8, need) == 6     # workspace alignment
    assert a(W, 16, 16, S, 1, 1, X, 2, Y, I, V, W, need) == 8         # workspace over weights
    assert a(W, 16, 16, S, 1, 1, X, 2, Y, I, Y + 4, K, need) == 8     # value inside y
    assert a(W, 16, 16, S, 1, 1, X, 9, Y, I, V, K, need) == 5


def test_topk_rejections():
    Y, U, I, V, P, T, K = (FAKE + (i << 30) for i in range(7))
    need = qmv.TOPK_WORKSPACE_BYTES
    assert need == 1024 * 64 * 8

    def t(y=Y, R=1000, b=2, k=8, temp=1.0, u=U, i=I, v=V, p=P, tok=T, ws=K, wsb=need):
        return qmv.topk_sample(y, R, b, k, temp, u, i, v, p, tok, ws, wsb)
    assert t(b=0) == 5 and t(b=9) == 5
    assert t(R=0) == 2                          # R >= 1
    assert t(R=1 << 31) == 7                    # rows must fit in 31 bits
    assert t(k=0) == 2 and t(k=65) == 2         # 1 <= k <= QMV_MAX_TOPK
    assert t(R=5, k=6) == 2                     # k <= R
    assert t(temp=-1.0) == 11 and t(temp=float("nan")) == 11 and t(temp=float("inf")) == 11
    assert t(y=0) == 1 and t(u=0) == 1 and t(i=0) == 1 and t(tok=0) == 1 and t(ws=0) == 1
    assert t(y=Y + 2) == 6 and t(u=U + 1) == 6 and t(i=I + 4) == 6 and t(tok=T + 4) == 6
    assert t(v=V + 2) == 6 and t(p=P + 1) == 6 and t(ws=K + 8) == 6
    assert t(wsb=need - 1) == 2                 # workspace too small
    assert t(i=Y + 64) == 8                     # index inside the logits
    assert t(p=U) == 8                          # probabilities over the draws
    assert t(ws=I) == 8                         # workspace over an output
    assert t(tok=V + 8) == 8                    # two outputs overlap
    W, S, X = FAKE + (8 << 30), FAKE + (9 << 30), FAKE + (10 << 30)

    def f(w=W, R=1000, C=64, SR=1, SC=1, y=Y, k=8, temp=0.5, i=I, ws=K):
        return qmv.f8_matvec_topk_sample(w, R, C, S, SR, SC, X, 2, y, k, temp, U, i, V, P, T,
                                         ws, need)
    assert f(R=0) == 2 and f(C=0) == 2 and f(SR=1001) == 2
    assert f(y=0) == 1 and f(w=0) == 1
    assert f(temp=-0.5) == 11
    assert f(y=W + 16) == 8                     # logits over the weights
    assert f(i=Y + 8) == 8                      # index inside the logits
    assert f(ws=X) == 8                         # workspace over x
    assert f(k=1001) == 2

    def g(w=W, R=1000, C=64, y=Y, k=8, temp=0.5, i=I, ws=K):
        return qmv.i8_matvec_topk_sample(w, R, C, S, X, 2, y, k, temp, U, i, V, P, T, ws, need)
    assert g(R=0) == 2 and g(C=0) == 2 and g(k=0) == 2
    assert g(y=0) == 1 and g(w=0) == 1
    assert g(temp=float("nan")) == 11
    assert g(y=W + 16) == 8                     # logits over the weights
    assert g(i=Y + 8) == 8                      # index inside the logits
    assert g(y=Y + 2) == 6


def test_cq_set_rejections():
    m = _m()
    other = _m(packed=FAKE + (1 << 24), norms=FAKE + (1 << 25))
    P, Y1, Y2 = FAKE + (1 << 30), FAKE + (1 << 31), FAKE + (1 << 32)
    f = qmv.cq_matvec_multi
    assert f([], P, 1, []) == 2                                    # nmats 0
    assert f([m] * 9, P, 1, [Y1 + 65536 * i for i in range(9)]) == 2   # too many
    assert f([m, _m(group=64)], P, 1, [Y1, Y2]) == 2               # group differs
    assert f([m, _m(codebook=FAKE + 64)], P, 1, [Y1, Y2]) == 2     # codebook differs
    assert f([m, other], P, 1, [Y1, 0]) == 1                        # missing output
    assert f([m, other], P, 1, [Y1, Y1 + 64]) == 8                 # outputs overlap
    assert f([m, other], P, 1, [Y1, FAKE + (1 << 24) + 16]) == 8   # output over packed rows
    assert f([m, other], 0, 1, [Y1, Y2]) == 1
    g = qmv.cq_prepare_matvec
    X = FAKE + (1 << 33)
    assert g([m, other], X, 1, X + 16, [Y1, Y2]) == 8               # prepared over x
    assert g([m, other], 0, 1, P, [Y1, Y2]) == 1
    assert g([m, other], X, 9, P, [Y1, Y2]) == 5


def test_i8_rejections():
    W, S, X, Y = FAKE, FAKE + (1 << 30), FAKE + (1 << 31), FAKE + (1 << 32)
    f = qmv.i8_matvec
    assert f(W, 16, 16, S, X, 0, Y) == 5
    assert f(W, 16, 0, S, X, 1, Y) == 2
    assert f(W, -1, 16, S, X, 1, Y) == 2
    assert f(W, 16, 16, 0, X, 1, Y) == 1
    assert f(W, 16, 16, S, 0, 1, Y) == 1
    assert f(W, 16, 16, S, X + 2, 1, Y) == 6
    assert f(W, 16, 16, S, X, 1, W + 8) == 8
    assert f(W, 16, 16, S, X, 1, S) == 8
    assert f(W, 0, 16, S, X, 1, 0) == 0


def test_i8_quantize_x_rejections():
    X, Q, D = FAKE, FAKE + (1 << 30), FAKE + (1 << 31)
    f = qmv.i8_quantize_x
    assert f(X, 64, 0, Q, D) == 5                  # batch
    assert f(X, 64, 9, Q, D) == 5
    assert f(X, 0, 1, Q, D) == 2                   # C
    assert f(0, 64, 1, Q, D) == 1                  # NULL
    assert f(X, 64, 1, 0, D) == 1
    assert f(X, 64, 1, Q, 0) == 1
    assert f(X + 2, 64, 1, Q, D) == 6              # alignment
    assert f(X, 64, 1, Q, D + 2) == 6
    assert f(X, 64, 2, X + 256, D) == 8            # codes overlap x
    assert f(X, 64, 1, Q, X + 252) == 8            # scales overlap x
    assert f(X, 64, 1, Q, Q + 60) == 8             # scales overlap codes


def test_i8_matvec_q8_rejections():
    W, S, Q, D, Y = FAKE, FAKE + (1 << 30), FAKE + (1 << 31), FAKE + (3 << 30), FAKE + (1 << 32)
    f = qmv.i8_matvec_q8
    assert f(W, 16, 64, S, Q, D, 0, Y) == 5        # batch
    assert f(W, 16, 64, S, Q, D, 9, Y) == 5
    assert f(W, 16, 0, S, Q, D, 1, Y) == 2         # shapes
    assert f(W, -1, 64, S, Q, D, 1, Y) == 2
    assert f(0, 16, 64, S, Q, D, 1, Y) == 1        # NULL
    assert f(W, 16, 64, 0, Q, D, 1, Y) == 1
    assert f(W, 16, 64, S, 0, D, 1, Y) == 1
    assert f(W, 16, 64, S, Q, 0, 1, Y) == 1
    assert f(W, 16, 64, S, Q, D, 1, 0) == 1
    assert f(W, 16, 64, S, Q, D + 2, 1, Y) == 6    # alignment
    assert f(W, 16, 64, S, Q, D, 1, Y + 2) == 6
    assert f(W, 16, 64, S, Q, D, 1, W + 64) == 8   # y overlaps w
    assert f(W, 16, 64, S, Q, D, 1, S) == 8        # y overlaps scale
    assert f(W, 16, 64, S, Q, D, 1, Q + 32) == 8   # y overlaps codes
    assert f(W, 16, 64, S, Q, D, 1, D) == 8        # y overlaps activation scales
    assert f(W, 0, 64, S, Q, D, 1, 0) == 0         # no rows: nothing to do


def test_hadamard_mlp_rejections():
    X, D1, D2, D3 = FAKE, FAKE + (1 << 30), FAKE + (1 << 31), FAKE + (3 << 30)
    R, U, O = FAKE + (1 << 32), FAKE + (5 << 30), FAKE + (6 << 30)
    f = qmv.hadamard_mlp
    assert f(X, 512, 2048, D1, D2, D3, R, U, 0, O) == 5             # batch
    assert f(X, 512, 2048, D1, D2, D3, R, U, 9, O) == 5
    assert f(X, 512, 2000, D1, D2, D3, R, U, 1, O) == 2             # D not a power of two
    assert f(X, 512, 0, D1, D2, D3, R, U, 1, O) == 2
    assert f(X, 512, 65536, D1, D2, D3, R, U, 1, O) == 2            # above the limit
    assert f(X, 0, 2048, D1, D2, D3, R, U, 1, O) == 2               # n outside [1, D]
    assert f(X, 2049, 2048, D1, D2, D3, R, U, 1, O) == 2
    assert f(0, 512, 2048, D1, D2, D3, R, U, 1, O) == 1             # NULL required pointers
    assert f(X, 512, 2048, D1, 0, D3, R, U, 1, O) == 1
    assert f(X, 512, 2048, D1, D2, D3, R, U, 1, 0) == 1
    assert f(X + 2, 512, 2048, D1, D2, D3, R, U, 1, O) == 6         # alignment
    assert f(X, 512, 2048, D1, D2, D3, R + 1, U, 1, O) == 6
    assert f(X, 512, 2048, D1, D2, D3, R, U, 1, O + 2) == 6
    assert f(X, 512, 2048, D1, D2, D3, R, U, 2, X + 1024) == 8      # out overlaps x
    assert f(X, 512, 2048, D1, D2, D3, R, U, 1, D3 + 4096) == 8     # out overlaps d3
    assert f(X, 512, 2048, D1, D2, D3, R, U, 1, R) == 8             # out overlaps residual
    assert f(X, 512, 2048, D1, D2, D3, 0, U, 1, U + 4) == 8         # out overlaps u
