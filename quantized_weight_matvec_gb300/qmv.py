"""ctypes binding of libqmv (include/qmv.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module only
checks tensor dtypes / devices / contiguity, passes ``data_ptr()`` values and
torch's current CUDA stream, and turns status codes into exceptions.  There
is no CPU fallback: if the library cannot be loaded, import fails loudly.

Raw entry points with the C names (``cq_prepare``, ``cq_matvec``,
``cq_dequantize_row``, ``f8_matvec``) take integer device pointers exactly as
the C-ABI does; the ``*_t`` helpers take torch tensors.
"""
from __future__ import annotations

import ctypes
import os

from . import build_lib

QMV_OK = 0
STATUS_NAMES = {0: "QMV_OK", 1: "QMV_ERR_NULL", 2: "QMV_ERR_SHAPE", 3: "QMV_ERR_BITS",
                4: "QMV_ERR_GROUP", 5: "QMV_ERR_BATCH", 6: "QMV_ERR_ALIGN",
                7: "QMV_ERR_OVERFLOW", 8: "QMV_ERR_ALIAS", 9: "QMV_ERR_CUDA",
                10: "QMV_ERR_ROW_ID", 11: "QMV_ERR_ARG"}
MAX_BATCH = 8
MAX_GROUP = 32768
ARGMAX_MAX_BLOCKS = 2048
MAX_TOPK = 64
TOPK_MAX_SLICES = 1024
TOPK_WORKSPACE_BYTES = TOPK_MAX_SLICES * MAX_TOPK * 8


ARGMAX_COUNTER_BYTES = 16


def f8_argmax_workspace_bytes(batch: int, R: int = 0) -> int:
    """QMV_F8_ARGMAX_WORKSPACE_BYTES(batch): the arrival counter, then the
    per-block partial results; with R, QMV_F8_ARGMAX_WORKSPACE_TC_BYTES(batch,
    R): room behind them for the batch x R logits of a call without y."""
    base = ARGMAX_COUNTER_BYTES + ARGMAX_MAX_BLOCKS * int(batch) * 16
    if not R:
        return base
    return f8_argmax_logits_offset(batch) + 4 * int(batch) * int(R)


def f8_argmax_logits_offset(batch: int) -> int:
    """QMV_F8_ARGMAX_LOGITS_OFFSET(batch): where a large workspace keeps the
    logits of a call without y."""
    return (f8_argmax_workspace_bytes(batch) + 255) // 256 * 256


class QmvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s: %s" % (where, status_string(status)))


class CQMatrixStruct(ctypes.Structure):
    """Mirror of qmv_cq_matrix."""
    _fields_ = [("output", ctypes.c_int64), ("input", ctypes.c_int64),
                ("input_padded", ctypes.c_int64), ("group", ctypes.c_int64),
                ("bits", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("row_bytes", ctypes.c_int64),
                ("packed", ctypes.c_void_p), ("norms", ctypes.c_void_p),
                ("codebook", ctypes.c_void_p)]


_lib = None


def lib_path() -> str:
    return build_lib.LIB


def load() -> ctypes.CDLL:
    """Load libqmv.so, building it first if it is missing or stale and nvcc exists."""
    global _lib
    if _lib is not None:
        return _lib
    path = build_lib.LIB
    if not build_lib.up_to_date():
        try:
            build_lib.build()
        except Exception as e:  # no toolkit: fail loudly unless a library is present
            if not os.path.exists(path):
                raise RuntimeError("libqmv.so is not built and cannot be built: %s" % e) from e
    lib = ctypes.CDLL(path)
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    CQP = ctypes.POINTER(CQMatrixStruct)
    lib.cq_prepare.argtypes = [CQP, P, I32, P, P]
    lib.cq_matvec.argtypes = [CQP, P, I32, P, P]
    lib.cq_dequantize_row.argtypes = [CQP, P, I64, P, P, P]
    lib.cq_matvec_multi.argtypes = [CQP, I32, P, I32, P, P]
    lib.cq_prepare_matvec.argtypes = [CQP, I32, P, I32, P, P, P]
    lib.f8_matvec.argtypes = [P, I64, I64, P, I64, I64, P, I32, P, P]
    lib.i8_matvec.argtypes = [P, I64, I64, P, P, I32, P, P]
    lib.i8_quantize_x.argtypes = [P, I64, I32, P, P, P]
    lib.i8_matvec_q8.argtypes = [P, I64, I64, P, P, P, I32, P, P]
    lib.f8_matvec_argmax.argtypes = [P, I64, I64, P, I64, I64, P, I32, P, P, P, P, I64, P]
    lib.f8_matvec_argmax_noalloc.argtypes = [P, I64, I64, P, I64, I64, P, I32, P, P, P, P]
    lib.hadamard_mlp.argtypes = [P, I64, I64, P, P, P, P, P, I32, P, P]
    F = ctypes.c_float
    lib.topk_sample.argtypes = [P, I64, I32, I32, F, P, P, P, P, P, P, I64, P]
    lib.f8_matvec_topk_sample.argtypes = [P, I64, I64, P, I64, I64, P, I32, P, I32, F, P, P, P,
                                          P, P, P, I64, P]
    lib.i8_matvec_topk_sample.argtypes = [P, I64, I64, P, P, I32, P, I32, F, P, P, P, P, P, P,
                                          I64, P]
    for fn in (lib.cq_prepare, lib.cq_matvec, lib.cq_dequantize_row, lib.cq_matvec_multi,
               lib.cq_prepare_matvec, lib.f8_matvec, lib.i8_matvec, lib.f8_matvec_argmax,
               lib.f8_matvec_argmax_noalloc, lib.hadamard_mlp, lib.topk_sample,
               lib.f8_matvec_topk_sample, lib.i8_matvec_topk_sample, lib.i8_quantize_x,
               lib.i8_matvec_q8):
        fn.restype = ctypes.c_int
    lib.qmv_status_string.argtypes = [ctypes.c_int]
    lib.qmv_status_string.restype = ctypes.c_char_p
    lib.qmv_abi_version.argtypes = []
    lib.qmv_abi_version.restype = I32
    lib.qmv_tc_wait_timeouts.argtypes = [P]
    lib.qmv_tc_wait_timeouts.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().qmv_status_string(int(status)).decode()


def abi_version() -> int:
    return int(load().qmv_abi_version())


def tc_wait_timeouts() -> int:
    """Waits of the fifth-generation tensor-core F8 kernel that ran out of
    their one-second limit on the current device (none, normally)."""
    out = ctypes.c_uint64(0)
    _check(load().qmv_tc_wait_timeouts(ctypes.addressof(out)), "qmv_tc_wait_timeouts")
    return int(out.value)


# --------------------------------------------------------------------------
# raw C-ABI calls (integer pointers), returning the status code
# --------------------------------------------------------------------------

def cq_struct(output, input, input_padded, group, bits, row_bytes, packed=0, norms=0,
              codebook=0, reserved=0) -> CQMatrixStruct:
    return CQMatrixStruct(int(output), int(input), int(input_padded), int(group), int(bits),
                          int(reserved), int(row_bytes), int(packed) or None, int(norms) or None,
                          int(codebook) or None)


def cq_prepare(m: CQMatrixStruct, x: int, batch: int, prepared: int, stream: int = 0) -> int:
    return load().cq_prepare(ctypes.byref(m), x or None, batch, prepared or None, stream or None)


def cq_matvec(m: CQMatrixStruct, prepared: int, batch: int, y: int, stream: int = 0) -> int:
    return load().cq_matvec(ctypes.byref(m), prepared or None, batch, y or None, stream or None)


def _set(mats, ys):
    n = len(mats)
    arr = (CQMatrixStruct * max(n, 1))(*mats)
    yarr = (ctypes.c_void_p * max(n, 1))(*[int(v) or None for v in ys])
    return arr, yarr, n


def cq_matvec_multi(mats, prepared: int, batch: int, ys, stream: int = 0) -> int:
    """mats: list of CQMatrixStruct; ys: list of device pointers."""
    arr, yarr, n = _set(mats, ys)
    return load().cq_matvec_multi(arr, n, prepared or None, batch, yarr, stream or None)


def cq_prepare_matvec(mats, x: int, batch: int, prepared: int, ys, stream: int = 0) -> int:
    arr, yarr, n = _set(mats, ys)
    return load().cq_prepare_matvec(arr, n, x or None, batch, prepared or None, yarr,
                                    stream or None)


def cq_dequantize_row(m: CQMatrixStruct, rows: int, n: int, out: int, dev_status: int = 0,
                      stream: int = 0) -> int:
    return load().cq_dequantize_row(ctypes.byref(m), rows or None, n, out or None,
                                    dev_status or None, stream or None)


def f8_matvec(w: int, R: int, C: int, scale: int, SR: int, SC: int, x: int, batch: int, y: int,
              stream: int = 0) -> int:
    return load().f8_matvec(w or None, R, C, scale or None, SR, SC, x or None, batch, y or None,
                            stream or None)


def i8_matvec(w: int, R: int, C: int, scale: int, x: int, batch: int, y: int,
              stream: int = 0) -> int:
    return load().i8_matvec(w or None, R, C, scale or None, x or None, batch, y or None,
                            stream or None)


def i8_quantize_x(x: int, C: int, batch: int, xq: int, xscale: int, stream: int = 0) -> int:
    return load().i8_quantize_x(x or None, C, batch, xq or None, xscale or None, stream or None)


def i8_matvec_q8(w: int, R: int, C: int, scale: int, xq: int, xscale: int, batch: int, y: int,
                 stream: int = 0) -> int:
    return load().i8_matvec_q8(w or None, R, C, scale or None, xq or None, xscale or None, batch,
                               y or None, stream or None)


def hadamard_mlp(x: int, n: int, D: int, d1: int, d2: int, d3: int, residual: int, u: int,
                 batch: int, out: int, stream: int = 0) -> int:
    return load().hadamard_mlp(x or None, n, D, d1 or None, d2 or None, d3 or None,
                               residual or None, u or None, batch, out or None, stream or None)


def f8_matvec_argmax(w: int, R: int, C: int, scale: int, SR: int, SC: int, x: int, batch: int,
                     y: int, out_index: int, out_value: int, workspace: int, workspace_bytes: int,
                     stream: int = 0) -> int:
    return load().f8_matvec_argmax(w or None, R, C, scale or None, SR, SC, x or None, batch,
                                   y or None, out_index or None, out_value or None,
                                   workspace or None, workspace_bytes, stream or None)


def f8_matvec_argmax_noalloc(w: int, R: int, C: int, scale: int, SR: int, SC: int, x: int,
                             batch: int, y: int, out_index: int, out_value: int,
                             stream: int = 0) -> int:
    """f8_matvec_argmax using the library's own scratch: for callers that
    cannot allocate device memory (see include/qmv.h)."""
    return load().f8_matvec_argmax_noalloc(w or None, R, C, scale or None, SR, SC, x or None,
                                           batch, y or None, out_index or None,
                                           out_value or None, stream or None)


def topk_sample(y: int, R: int, batch: int, k: int, temperature: float, u: int, top_index: int,
                top_value: int, top_prob: int, token: int, workspace: int, workspace_bytes: int,
                stream: int = 0) -> int:
    return load().topk_sample(y or None, R, batch, k, temperature, u or None, top_index or None,
                              top_value or None, top_prob or None, token or None,
                              workspace or None, workspace_bytes, stream or None)


def f8_matvec_topk_sample(w: int, R: int, C: int, scale: int, SR: int, SC: int, x: int,
                          batch: int, y: int, k: int, temperature: float, u: int, top_index: int,
                          top_value: int, top_prob: int, token: int, workspace: int,
                          workspace_bytes: int, stream: int = 0) -> int:
    return load().f8_matvec_topk_sample(w or None, R, C, scale or None, SR, SC, x or None, batch,
                                        y or None, k, temperature, u or None, top_index or None,
                                        top_value or None, top_prob or None, token or None,
                                        workspace or None, workspace_bytes, stream or None)


def i8_matvec_topk_sample(w: int, R: int, C: int, scale: int, x: int, batch: int, y: int, k: int,
                          temperature: float, u: int, top_index: int, top_value: int,
                          top_prob: int, token: int, workspace: int, workspace_bytes: int,
                          stream: int = 0) -> int:
    return load().i8_matvec_topk_sample(w or None, R, C, scale or None, x or None, batch,
                                        y or None, k, temperature, u or None, top_index or None,
                                        top_value or None, top_prob or None, token or None,
                                        workspace or None, workspace_bytes, stream or None)


# --------------------------------------------------------------------------
# torch helpers
# --------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dev(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError("%s must have dtype %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != QMV_OK:
        raise QmvError(status, where)


class CQMatrix:
    """A CQ matrix whose arrays live on the GPU (the page's CqMatrix record)."""

    def __init__(self, output, input, input_padded, group, bits, packed, norms, codebook):
        torch = _torch()
        self.output, self.input, self.input_padded = int(output), int(input), int(input_padded)
        self.group, self.bits = int(group), int(bits)
        self.row_bytes = (self.input_padded * self.bits + 7) // 8
        self.packed = _dev(packed, torch.uint8, "packed")
        self.norms = _dev(norms, (torch.int16, torch.uint16), "norms")
        self.codebook = _dev(codebook, torch.float32, "codebook")
        self.struct = cq_struct(self.output, self.input, self.input_padded, self.group, self.bits,
                                self.row_bytes, self.packed.data_ptr(), self.norms.data_ptr(),
                                self.codebook.data_ptr())

    @classmethod
    def from_numpy(cls, c, device="cuda"):
        """Upload a synth.CQInputs (or any object with the same fields)."""
        torch = _torch()
        return cls(c.output, c.input, c.input_padded, c.group, c.bits,
                   torch.from_numpy(c.packed).to(device),
                   torch.from_numpy(c.norms.view("int16")).to(device),
                   torch.from_numpy(c.codebook).to(device))


def cq_prepare_t(m: CQMatrix, x, out=None, stream=None):
    """prepared[B, P] = cq_prepare(x[B, input])."""
    torch = _torch()
    x = _dev(x, torch.float32, "x")
    batch = x.shape[0] if x.dim() == 2 else 1
    if out is None:
        out = torch.empty((batch, m.input_padded), dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    _check(cq_prepare(m.struct, x.data_ptr(), batch, out.data_ptr(), _stream(stream)), "cq_prepare")
    return out


def cq_matvec_t(m: CQMatrix, prepared, out=None, stream=None):
    """y[B, output] = cq_matvec(prepared[B, P])."""
    torch = _torch()
    prepared = _dev(prepared, torch.float32, "prepared")
    batch = prepared.shape[0] if prepared.dim() == 2 else 1
    if out is None:
        out = torch.empty((batch, m.output), dtype=torch.float32, device=prepared.device)
    _dev(out, torch.float32, "out")
    _check(cq_matvec(m.struct, prepared.data_ptr(), batch, out.data_ptr(), _stream(stream)),
           "cq_matvec")
    return out


def cq_dequantize_row_t(m: CQMatrix, rows, out=None, status=None, stream=None):
    """out[n, input] = dense rows of the given ids."""
    torch = _torch()
    rows = _dev(rows, torch.int32, "rows")
    n = rows.numel()
    if out is None:
        out = torch.empty((n, m.input), dtype=torch.float32, device=rows.device)
    _dev(out, torch.float32, "out")
    sp = 0
    if status is not None:
        sp = _dev(status, torch.int32, "status").data_ptr()
    _check(cq_dequantize_row(m.struct, rows.data_ptr(), n, out.data_ptr(), sp, _stream(stream)),
           "cq_dequantize_row")
    return out


def f8_matvec_t(w, scale, x, out=None, stream=None):
    """y[B, R] = f8_matvec(w[R, C], scale[SR, SC], x[B, C])."""
    torch = _torch()
    w = _dev(w, torch.uint8, "w")
    scale = _dev(scale, torch.uint8, "scale")
    x = _dev(x, torch.float32, "x")
    R, C = w.shape
    SR, SC = scale.shape
    batch = x.shape[0] if x.dim() == 2 else 1
    if out is None:
        out = torch.empty((batch, R), dtype=torch.float32, device=w.device)
    _dev(out, torch.float32, "out")
    _check(f8_matvec(w.data_ptr(), R, C, scale.data_ptr(), SR, SC, x.data_ptr(), batch,
                     out.data_ptr(), _stream(stream)), "f8_matvec")
    return out


def f8_matvec_argmax_t(w, scale, x, y=None, workspace=None, stream=None):
    """(index[B] int64, value[B] float32) of the row maximising y = f8_matvec(...).

    ``y`` (optional) receives the full [B, R] result; ``workspace`` (optional)
    is a uint8 CUDA tensor of at least f8_argmax_workspace_bytes(B) bytes whose
    first ARGMAX_COUNTER_BYTES bytes were zeroed before its first use (every
    call leaves them zero)."""
    torch = _torch()
    w = _dev(w, torch.uint8, "w")
    scale = _dev(scale, torch.uint8, "scale")
    x = _dev(x, torch.float32, "x")
    R, C = w.shape
    SR, SC = scale.shape
    batch = x.shape[0] if x.dim() == 2 else 1
    if workspace is None:
        workspace = torch.zeros(f8_argmax_workspace_bytes(batch), dtype=torch.uint8, device=w.device)
    _dev(workspace, torch.uint8, "workspace")
    idx = torch.empty(batch, dtype=torch.int64, device=w.device)
    val = torch.empty(batch, dtype=torch.float32, device=w.device)
    yp = 0
    if y is not None:
        yp = _dev(y, torch.float32, "y").data_ptr()
    _check(f8_matvec_argmax(w.data_ptr(), R, C, scale.data_ptr(), SR, SC, x.data_ptr(), batch, yp,
                            idx.data_ptr(), val.data_ptr(), workspace.data_ptr(), workspace.numel(),
                            _stream(stream)), "f8_matvec_argmax")
    return idx, val


def cq_matvec_multi_t(mats, prepared, stream=None):
    """[y_i] = cq_matvec(mats[i], prepared) for every CQMatrix in one launch."""
    torch = _torch()
    prepared = _dev(prepared, torch.float32, "prepared")
    batch = prepared.shape[0] if prepared.dim() == 2 else 1
    ys = [torch.empty((batch, m.output), dtype=torch.float32, device=prepared.device)
          for m in mats]
    _check(cq_matvec_multi([m.struct for m in mats], prepared.data_ptr(), batch,
                           [y.data_ptr() for y in ys], _stream(stream)), "cq_matvec_multi")
    return ys


def cq_prepare_matvec_t(mats, x, prepared=None, stream=None):
    """[y_i] for x prepared inside the launch; `prepared` (optional) receives it."""
    torch = _torch()
    x = _dev(x, torch.float32, "x")
    batch = x.shape[0] if x.dim() == 2 else 1
    ys = [torch.empty((batch, m.output), dtype=torch.float32, device=x.device) for m in mats]
    pp = 0
    if prepared is not None:
        pp = _dev(prepared, torch.float32, "prepared").data_ptr()
    _check(cq_prepare_matvec([m.struct for m in mats], x.data_ptr(), batch, pp,
                             [y.data_ptr() for y in ys], _stream(stream)), "cq_prepare_matvec")
    return ys


def i8_matvec_t(w, scale, x, out=None, stream=None):
    """y[B, R] = i8_matvec(w[R, C] int8, scale[R, ceil(C/16)] uint8, x[B, C])."""
    torch = _torch()
    w = _dev(w, torch.int8, "w")
    scale = _dev(scale, torch.uint8, "scale")
    x = _dev(x, torch.float32, "x")
    R, C = w.shape
    if tuple(scale.shape) != (R, (C + 15) // 16):
        raise ValueError("scale must be [R, ceil(C/16)]")
    batch = x.shape[0] if x.dim() == 2 else 1
    if out is None:
        out = torch.empty((batch, R), dtype=torch.float32, device=w.device)
    _dev(out, torch.float32, "out")
    _check(i8_matvec(w.data_ptr(), R, C, scale.data_ptr(), x.data_ptr(), batch, out.data_ptr(),
                     _stream(stream)), "i8_matvec")
    return out


def i8_quantize_x_t(x, xq=None, xscale=None, stream=None):
    """(xq [B, C] int8, xscale [B, ceil(C/32)] float32) = i8_quantize_x(x [B, C])."""
    torch = _torch()
    x = _dev(x, torch.float32, "x")
    batch = x.shape[0] if x.dim() == 2 else 1
    C = x.shape[-1]
    if xq is None:
        xq = torch.empty((batch, C), dtype=torch.int8, device=x.device)
    if xscale is None:
        xscale = torch.empty((batch, (C + 31) // 32), dtype=torch.float32, device=x.device)
    _dev(xq, torch.int8, "xq")
    _dev(xscale, torch.float32, "xscale")
    if xq.numel() != batch * C or xscale.numel() != batch * ((C + 31) // 32):
        raise ValueError("xq must be [B, C] and xscale [B, ceil(C/32)]")
    _check(i8_quantize_x(x.data_ptr(), C, batch, xq.data_ptr(), xscale.data_ptr(),
                         _stream(stream)), "i8_quantize_x")
    return xq, xscale


def i8_matvec_q8_t(w, scale, xq, xscale, out=None, stream=None):
    """y[B, R] = i8_matvec_q8(w[R, C] int8, scale[R, ceil(C/16)] uint8,
    xq[B, C] int8, xscale[B, ceil(C/32)] float32)."""
    torch = _torch()
    w = _dev(w, torch.int8, "w")
    scale = _dev(scale, torch.uint8, "scale")
    xq = _dev(xq, torch.int8, "xq")
    xscale = _dev(xscale, torch.float32, "xscale")
    R, C = w.shape
    batch = xq.shape[0] if xq.dim() == 2 else 1
    if tuple(scale.shape) != (R, (C + 15) // 16):
        raise ValueError("scale must be [R, ceil(C/16)]")
    if xq.numel() != batch * C or xscale.numel() != batch * ((C + 31) // 32):
        raise ValueError("xq must be [B, C] and xscale [B, ceil(C/32)]")
    if out is None:
        out = torch.empty((batch, R), dtype=torch.float32, device=w.device)
    _dev(out, torch.float32, "out")
    _check(i8_matvec_q8(w.data_ptr(), R, C, scale.data_ptr(), xq.data_ptr(), xscale.data_ptr(),
                        batch, out.data_ptr(), _stream(stream)), "i8_matvec_q8")
    return out


def hadamard_mlp_t(x, D, d1, d2, d3, residual=None, u=None, out=None, stream=None):
    """out[B, n] = hadamard_mlp(x[B, n], D, d1, d2, d3[D], residual, u)."""
    torch = _torch()
    x = _dev(x, torch.float32, "x")
    if x.dim() == 1:
        x = x.view(1, -1)
    batch, n = x.shape
    d1, d2, d3 = (_dev(d, torch.float32, name) for d, name in ((d1, "d1"), (d2, "d2"), (d3, "d3")))
    for d in (d1, d2, d3):
        if d.numel() != D:
            raise ValueError("diagonals must have D elements")
    ptrs = []
    for t, name in ((residual, "residual"), (u, "u")):
        if t is None:
            ptrs.append(0)
            continue
        t = _dev(t, torch.float32, name)
        if t.numel() != batch * n:
            raise ValueError(name + " must be [batch, n]")
        ptrs.append(t.data_ptr())
    if out is None:
        out = torch.empty((batch, n), dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    _check(hadamard_mlp(x.data_ptr(), n, D, d1.data_ptr(), d2.data_ptr(), d3.data_ptr(), ptrs[0],
                        ptrs[1], batch, out.data_ptr(), _stream(stream)), "hadamard_mlp")
    return out


def _topk_outputs(batch, k, device, workspace):
    torch = _torch()
    idx = torch.empty((batch, k), dtype=torch.int64, device=device)
    val = torch.empty((batch, k), dtype=torch.float32, device=device)
    prob = torch.empty((batch, k), dtype=torch.float32, device=device)
    tok = torch.empty(batch, dtype=torch.int64, device=device)
    if workspace is None:
        workspace = torch.empty(TOPK_WORKSPACE_BYTES, dtype=torch.uint8, device=device)
    _dev(workspace, torch.uint8, "workspace")
    return idx, val, prob, tok, workspace


def topk_sample_t(y, k, temperature, u, workspace=None, stream=None):
    """Top-k temperature sampling over logits y [B, R]: returns (top_index
    [B, k] int64 best first, top_value [B, k], top_prob [B, k], token [B]
    int64).  u [B] float32 holds one uniform draw per vector."""
    torch = _torch()
    y = _dev(y, torch.float32, "y")
    u = _dev(u, torch.float32, "u")
    batch, R = (y.shape[0], y.shape[1]) if y.dim() == 2 else (1, y.numel())
    idx, val, prob, tok, workspace = _topk_outputs(batch, int(k), y.device, workspace)
    _check(topk_sample(y.data_ptr(), R, batch, int(k), float(temperature), u.data_ptr(),
                       idx.data_ptr(), val.data_ptr(), prob.data_ptr(), tok.data_ptr(),
                       workspace.data_ptr(), workspace.numel(), _stream(stream)), "topk_sample")
    return idx, val, prob, tok


def f8_matvec_topk_sample_t(w, scale, x, k, temperature, u, y=None, workspace=None,
                            stream=None):
    """The F8 head then top-k temperature sampling: returns (y [B, R],
    top_index, top_value, top_prob, token) as topk_sample_t."""
    torch = _torch()
    w = _dev(w, torch.uint8, "w")
    scale = _dev(scale, torch.uint8, "scale")
    x = _dev(x, torch.float32, "x")
    u = _dev(u, torch.float32, "u")
    R, C = w.shape
    SR, SC = scale.shape
    batch = x.shape[0] if x.dim() == 2 else 1
    if y is None:
        y = torch.empty((batch, R), dtype=torch.float32, device=w.device)
    _dev(y, torch.float32, "y")
    idx, val, prob, tok, workspace = _topk_outputs(batch, int(k), w.device, workspace)
    _check(f8_matvec_topk_sample(w.data_ptr(), R, C, scale.data_ptr(), SR, SC, x.data_ptr(),
                                 batch, y.data_ptr(), int(k), float(temperature), u.data_ptr(),
                                 idx.data_ptr(), val.data_ptr(), prob.data_ptr(), tok.data_ptr(),
                                 workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "f8_matvec_topk_sample")
    return y, idx, val, prob, tok


def i8_matvec_topk_sample_t(w, scale, x, k, temperature, u, y=None, workspace=None,
                            stream=None):
    """The I8 head then top-k temperature sampling: returns (y [B, R],
    top_index, top_value, top_prob, token) as topk_sample_t."""
    torch = _torch()
    w = _dev(w, torch.int8, "w")
    scale = _dev(scale, torch.uint8, "scale")
    x = _dev(x, torch.float32, "x")
    u = _dev(u, torch.float32, "u")
    R, C = w.shape
    batch = x.shape[0] if x.dim() == 2 else 1
    if y is None:
        y = torch.empty((batch, R), dtype=torch.float32, device=w.device)
    _dev(y, torch.float32, "y")
    idx, val, prob, tok, workspace = _topk_outputs(batch, int(k), w.device, workspace)
    _check(i8_matvec_topk_sample(w.data_ptr(), R, C, scale.data_ptr(), x.data_ptr(), batch,
                                 y.data_ptr(), int(k), float(temperature), u.data_ptr(),
                                 idx.data_ptr(), val.data_ptr(), prob.data_ptr(), tok.data_ptr(),
                                 workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "i8_matvec_topk_sample")
    return y, idx, val, prob, tok
