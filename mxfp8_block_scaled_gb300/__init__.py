"""Python binding of the MXFP8 C-ABI library (include/mxfp8.h).

Argument marshalling only: every step of quantisation and GEMM runs in the
library's sm_103a kernels. PyTorch supplies device memory and streams. If the
shared library has not been built, importing the binding's functions raises;
there is no fallback path.

The raw entry points keep the C names (``mx_quantize``, ``mx_gemm``,
``mx_grouped_gemm``, ``mx_scale_bytes``, ``mx_grouped_padded_rows``,
``mx_status_string``, ``mx_last_error``, ``mx_abi_version``) and take integer
device pointers. ``quantize`` / ``gemm`` / ``grouped_gemm`` wrap them for
torch tensors, allocating outputs with torch.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmxfp8_gb300.so")

MX_ROWWISE, MX_COLWISE, MX_BOTH = 1, 2, 3
MX_FPROP, MX_DGRAD, MX_WGRAD = 0, 1, 2
MX_MAX_MULTI = 8
MX_MAX_GEMM_MULTI = 4
MX_MAX_GROUPS = 512
STATUS_NAMES = {0: "MX_OK", 1: "MX_ERR_INVALID_ARG", 2: "MX_ERR_UNSUPPORTED_SHAPE", 3: "MX_ERR_ALIGNMENT",
                4: "MX_ERR_CUDA", 5: "MX_ERR_DEVICE_CHECK", 6: "MX_ERR_TIMEOUT", 7: "MX_ERR_NO_DEVICE"}

# Symbols the header declares (the CPU tests check the library exports them).
EXPORTED = ("mx_scale_bytes", "mx_grouped_padded_rows", "mx_quantize", "mx_quantize_batched", "mx_quantize_f32",
            "mx_quantize_multi",
            "mx_gemm", "mx_grouped_gemm", "mx_grouped_gemm_swiglu", "mx_quantize_fp8_blockwise",
            "mx_gemm_fp8_blockwise", "mx_status_string", "mx_last_error", "mx_abi_version",
            "mx_selftest_wait_timeout", "mx_gemm_workspace_bytes", "mx_gemm_with_workspace", "mx_gemm_multi",
            "mx_gemm_static_workspace", "mx_current_amax", "mx_quantize_current", "mx_gemm_current",
            "mx_grouped_gemm_current", "mx_gemm_current_multi", "mx_grouped_gemm_swiglu_quantize")
MX_STATIC_WORKSPACE_BYTES = 40 * 1024 * 1024


class MXError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}" + (f" ({detail})" if detail else ""))


class MXOperandC(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("k", ctypes.c_int64), ("ld", ctypes.c_int64), ("orient", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class MXGemmProblemC(ctypes.Structure):
    _fields_ = [("a", MXOperandC), ("b", MXOperandC), ("c", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("mode", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class MXQuantTensorC(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ldx", ctypes.c_int64),
                ("row_data", ctypes.c_void_p), ("row_scale", ctypes.c_void_p), ("col_data", ctypes.c_void_p),
                ("col_scale", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m mxfp8_block_scaled_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.mx_scale_bytes.argtypes = [i64, i64]
    L.mx_scale_bytes.restype = ctypes.c_size_t
    L.mx_grouped_padded_rows.argtypes = [ctypes.POINTER(ctypes.c_int64), i32]
    L.mx_grouped_padded_rows.restype = i64
    L.mx_quantize.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, vp, vp, i32, i64, vp, vp]
    L.mx_quantize.restype = i32
    L.mx_quantize_batched.argtypes = [vp, i64, i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp]
    L.mx_quantize_batched.restype = i32
    L.mx_quantize_f32.argtypes = [vp, i64, i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp]
    L.mx_quantize_f32.restype = i32
    L.mx_quantize_multi.argtypes = [ctypes.POINTER(MXQuantTensorC), i32, i32, vp, vp]
    L.mx_quantize_multi.restype = i32
    L.mx_gemm.argtypes = [i32, ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC), vp, i64, vp, vp]
    L.mx_gemm.restype = i32
    L.mx_gemm_workspace_bytes.argtypes = [i32, ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC),
                                          ctypes.POINTER(ctypes.c_size_t)]
    L.mx_gemm_workspace_bytes.restype = i32
    L.mx_gemm_with_workspace.argtypes = [i32, ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC), vp, i64, vp,
                                         ctypes.c_size_t, vp, vp]
    L.mx_gemm_with_workspace.restype = i32
    L.mx_gemm_static_workspace.argtypes = [i32, ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC), vp, i64,
                                           vp, vp]
    L.mx_gemm_static_workspace.restype = i32
    L.mx_current_amax.argtypes = [vp, i64, i64, i64, i64, i64, vp, vp, vp]
    L.mx_current_amax.restype = i32
    L.mx_quantize_current.argtypes = [vp, i64, i64, i64, i64, i64, i32, vp, ctypes.c_float, vp, vp, vp, vp, i32, i64,
                                      vp, vp]
    L.mx_quantize_current.restype = i32
    L.mx_gemm_current.argtypes = [i32, ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC), vp, i64, vp, vp]
    L.mx_gemm_current.restype = i32
    L.mx_grouped_gemm_current.argtypes = [i32, ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC), vp, i32, vp,
                                          i64, vp, vp]
    L.mx_grouped_gemm_current.restype = i32
    L.mx_gemm_multi.argtypes = [ctypes.POINTER(MXGemmProblemC), i32, vp, vp]
    L.mx_gemm_multi.restype = i32
    L.mx_gemm_current_multi.argtypes = [ctypes.POINTER(MXGemmProblemC), i32, vp, vp]
    L.mx_gemm_current_multi.restype = i32
    L.mx_grouped_gemm.argtypes = [i32, ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC), vp, i32, vp, i64,
                                  vp, vp]
    L.mx_grouped_gemm.restype = i32
    L.mx_grouped_gemm_swiglu.argtypes = [ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC), vp, i32, vp, i64,
                                         vp, vp]
    L.mx_grouped_gemm_swiglu.restype = i32
    L.mx_grouped_gemm_swiglu_quantize.argtypes = [ctypes.POINTER(MXOperandC), ctypes.POINTER(MXOperandC), vp, i32, vp,
                                                  vp, vp, vp, i64, vp, vp]
    L.mx_grouped_gemm_swiglu_quantize.restype = i32
    L.mx_quantize_fp8_blockwise.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, vp]
    L.mx_quantize_fp8_blockwise.restype = i32
    L.mx_gemm_fp8_blockwise.argtypes = [vp, vp, i64, vp, vp, i64, i64, vp, i64, vp, vp]
    L.mx_gemm_fp8_blockwise.restype = i32
    L.mx_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp, vp]
    L.mx_selftest_wait_timeout.restype = i32
    L.mx_status_string.argtypes = [i32]
    L.mx_status_string.restype = ctypes.c_char_p
    L.mx_last_error.argtypes = []
    L.mx_last_error.restype = ctypes.c_char_p
    L.mx_abi_version.argtypes = []
    L.mx_abi_version.restype = i32
    _lib = L
    return L


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MXError(status, where, lib().mx_last_error().decode(errors="replace"))


# ---------------------------------------------------------------------------
# Raw entry points (same names as the C ABI; integer device pointers)
# ---------------------------------------------------------------------------

def mx_scale_bytes(rows: int, k: int) -> int:
    return int(lib().mx_scale_bytes(rows, k))


def mx_grouped_padded_rows(host_offsets) -> int:
    offs = [int(v) for v in host_offsets]
    arr = (ctypes.c_int64 * len(offs))(*offs)
    return int(lib().mx_grouped_padded_rows(arr, len(offs) - 1))


def mx_status_string(status: int) -> str:
    return lib().mx_status_string(status).decode()


def mx_last_error() -> str:
    return lib().mx_last_error().decode(errors="replace")


def mx_abi_version() -> int:
    return int(lib().mx_abi_version())


def mx_quantize(x, rows, cols, ldx, axis, row_data, row_scale, col_data, col_scale, group_offsets, n_groups,
                col_capacity, dev_status, stream) -> None:
    _check(lib().mx_quantize(x, rows, cols, ldx, axis, row_data, row_scale, col_data, col_scale, group_offsets,
                             n_groups, col_capacity, dev_status, stream), "mx_quantize")


def mx_quantize_batched(x, batch, rows, cols, ldx, x_batch_stride, axis, row_data, row_scale, col_data, col_scale,
                        dev_status, stream) -> None:
    _check(lib().mx_quantize_batched(x, batch, rows, cols, ldx, x_batch_stride, axis, row_data, row_scale, col_data,
                                     col_scale, dev_status, stream), "mx_quantize_batched")


def mx_quantize_f32(x, batch, rows, cols, ldx, x_batch_stride, axis, row_data, row_scale, col_data, col_scale,
                    dev_status, stream) -> None:
    _check(lib().mx_quantize_f32(x, batch, rows, cols, ldx, x_batch_stride, axis, row_data, row_scale, col_data,
                                 col_scale, dev_status, stream), "mx_quantize_f32")


def mx_quantize_multi(tensors, axis, dev_status, stream) -> None:
    """``tensors``: a sequence of MXQuantTensorC."""
    arr = (MXQuantTensorC * max(len(tensors), 1))(*tensors)
    _check(lib().mx_quantize_multi(arr, len(tensors), axis, dev_status, stream), "mx_quantize_multi")


def mx_quantize_fp8_blockwise(x, rows, cols, ldx, block, data, scale, dev_status, stream) -> None:
    _check(lib().mx_quantize_fp8_blockwise(x, rows, cols, ldx, block, data, scale, dev_status, stream),
           "mx_quantize_fp8_blockwise")


def mx_gemm_fp8_blockwise(a_data, a_scale, M, b_data, b_scale, N, K, c, ldc, dev_status, stream) -> None:
    _check(lib().mx_gemm_fp8_blockwise(a_data, a_scale, M, b_data, b_scale, N, K, c, ldc, dev_status, stream),
           "mx_gemm_fp8_blockwise")


def mx_selftest_wait_timeout(timeout_ns, dev_status, stream) -> None:
    _check(lib().mx_selftest_wait_timeout(timeout_ns, dev_status, stream), "mx_selftest_wait_timeout")


def _ref(op):
    return None if op is None else ctypes.byref(op)


def mx_gemm(mode, a: MXOperandC, b: MXOperandC, c, ldc, dev_status, stream) -> None:
    _check(lib().mx_gemm(mode, _ref(a), _ref(b), c, ldc, dev_status, stream), "mx_gemm")


def mx_gemm_workspace_bytes(mode, a: MXOperandC, b: MXOperandC) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().mx_gemm_workspace_bytes(mode, _ref(a), _ref(b), ctypes.byref(out)), "mx_gemm_workspace_bytes")
    return int(out.value)


def mx_gemm_with_workspace(mode, a: MXOperandC, b: MXOperandC, c, ldc, workspace, workspace_bytes, dev_status,
                           stream) -> None:
    _check(lib().mx_gemm_with_workspace(mode, _ref(a), _ref(b), c, ldc, workspace, workspace_bytes, dev_status,
                                        stream), "mx_gemm_with_workspace")


def mx_gemm_static_workspace(mode, a: MXOperandC, b: MXOperandC, c, ldc, dev_status, stream) -> None:
    _check(lib().mx_gemm_static_workspace(mode, _ref(a), _ref(b), c, ldc, dev_status, stream),
           "mx_gemm_static_workspace")


def mx_current_amax(x, batch, rows, cols, ldx, x_batch_stride, amax, dev_status, stream) -> None:
    _check(lib().mx_current_amax(x, batch, rows, cols, ldx, x_batch_stride, amax, dev_status, stream),
           "mx_current_amax")


def mx_quantize_current(x, batch, rows, cols, ldx, x_batch_stride, axis, amax, format_max, row_data, col_data, scale,
                        group_offsets, n_groups, col_capacity, dev_status, stream) -> None:
    _check(lib().mx_quantize_current(x, batch, rows, cols, ldx, x_batch_stride, axis, amax, format_max, row_data,
                                     col_data, scale, group_offsets, n_groups, col_capacity, dev_status, stream),
           "mx_quantize_current")


def mx_gemm_current(mode, a: MXOperandC, b: MXOperandC, c, ldc, dev_status, stream) -> None:
    _check(lib().mx_gemm_current(mode, _ref(a), _ref(b), c, ldc, dev_status, stream), "mx_gemm_current")


def mx_grouped_gemm_current(mode, a: MXOperandC, b: MXOperandC, group_offsets, n_groups, c, ldc, dev_status,
                            stream) -> None:
    _check(lib().mx_grouped_gemm_current(mode, _ref(a), _ref(b), group_offsets, n_groups, c, ldc, dev_status, stream),
           "mx_grouped_gemm_current")


def mx_gemm_multi(problems, dev_status, stream) -> None:
    """``problems``: a sequence of MXGemmProblemC."""
    arr = (MXGemmProblemC * max(len(problems), 1))(*problems)
    _check(lib().mx_gemm_multi(arr, len(problems), dev_status, stream), "mx_gemm_multi")


def mx_gemm_current_multi(problems, dev_status, stream) -> None:
    """``problems``: a sequence of MXGemmProblemC over current-scaled operands."""
    arr = (MXGemmProblemC * max(len(problems), 1))(*problems)
    _check(lib().mx_gemm_current_multi(arr, len(problems), dev_status, stream), "mx_gemm_current_multi")


def mx_grouped_gemm(mode, a: MXOperandC, b: MXOperandC, group_offsets, n_groups, c, ldc, dev_status,
                    stream) -> None:
    _check(lib().mx_grouped_gemm(mode, _ref(a), _ref(b), group_offsets, n_groups, c, ldc,
                                 dev_status, stream), "mx_grouped_gemm")


def mx_grouped_gemm_swiglu(a: MXOperandC, b: MXOperandC, group_offsets, n_groups, c, ldc, dev_status,
                           stream) -> None:
    _check(lib().mx_grouped_gemm_swiglu(_ref(a), _ref(b), group_offsets, n_groups, c, ldc, dev_status, stream),
           "mx_grouped_gemm_swiglu")


def mx_grouped_gemm_swiglu_quantize(a: MXOperandC, b: MXOperandC, group_offsets, n_groups, row_data, row_scale,
                                    col_data, col_scale, col_capacity, dev_status, stream) -> None:
    _check(lib().mx_grouped_gemm_swiglu_quantize(_ref(a), _ref(b), group_offsets, n_groups, row_data, row_scale,
                                                 col_data, col_scale, col_capacity, dev_status, stream),
           "mx_grouped_gemm_swiglu_quantize")


# ---------------------------------------------------------------------------
# torch-tensor wrappers
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class MXTensor:
    """One quantised copy ([rows, k] E4M3 codes + swizzled E8M0 scales)."""
    data: "object"      # torch.uint8 [rows, ld]
    scale: "object"     # torch.uint8 [mx_scale_bytes(rows, k)]
    rows: int
    k: int
    orient: int         # MX_ROWWISE or MX_COLWISE

    def c_operand(self) -> MXOperandC:
        return MXOperandC(self.data.data_ptr(), self.scale.data_ptr(), self.rows, self.k,
                          int(self.data.stride(0)), self.orient, 0)


def new_status(device=None):
    """A zeroed device int32 for the kernels' device-side status."""
    torch = _torch()
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_status(status) -> int:
    return int(status.item())


def quantize(x, axis: int = MX_BOTH, group_offsets=None, col_capacity: Optional[int] = None, status=None,
             stream=None):
    """MX-quantise a 2-D BF16 (or FP32, no groups) CUDA tensor. Returns
    (row_copy, col_copy), each an MXTensor or None. With ``group_offsets``
    (int64 CUDA tensor [E+1]) the column copy is per-group padded with width
    ``col_capacity``."""
    torch = _torch()
    assert x.dim() == 2 and x.dtype in (torch.bfloat16, torch.float32) and x.is_cuda and x.stride(1) == 1
    assert x.dtype == torch.bfloat16 or group_offsets is None
    R, C = x.shape
    dev = x.device
    row = col = None
    if axis & MX_ROWWISE:
        row = MXTensor(torch.empty((R, C), dtype=torch.uint8, device=dev),
                       torch.empty(mx_scale_bytes(R, C), dtype=torch.uint8, device=dev), R, C, MX_ROWWISE)
    n_groups = 0
    cap = 0
    if axis & MX_COLWISE:
        if group_offsets is not None:
            n_groups = group_offsets.numel() - 1
            cap = int(col_capacity) if col_capacity is not None else ((R + 127 * n_groups + 127) // 128) * 128
            col = MXTensor(torch.empty((C, cap), dtype=torch.uint8, device=dev),
                           torch.empty(mx_scale_bytes(C, cap), dtype=torch.uint8, device=dev), C, cap, MX_COLWISE)
        else:
            col = MXTensor(torch.empty((C, R), dtype=torch.uint8, device=dev),
                           torch.empty(mx_scale_bytes(C, R), dtype=torch.uint8, device=dev), C, R, MX_COLWISE)
    if x.dtype == torch.float32:
        mx_quantize_f32(x.data_ptr(), 1, R, C, x.stride(0), 0, axis,
                        _ptr(row.data) if row else None, _ptr(row.scale) if row else None,
                        _ptr(col.data) if col else None, _ptr(col.scale) if col else None,
                        _ptr(status), _stream(stream))
        return row, col
    mx_quantize(x.data_ptr(), R, C, x.stride(0), axis,
                _ptr(row.data) if row else None, _ptr(row.scale) if row else None,
                _ptr(col.data) if col else None, _ptr(col.scale) if col else None,
                _ptr(group_offsets), n_groups, cap, _ptr(status), _stream(stream))
    return row, col


def quantize_multi(xs, axis: int = MX_BOTH, status=None, stream=None):
    """MX-quantise up to MX_MAX_MULTI 2-D BF16 CUDA tensors of any shapes in
    one launch. Returns a list of (row_copy, col_copy), one per input, each
    exactly what ``quantize`` gives for that input alone."""
    torch = _torch()
    outs, descs = [], []
    for x in xs:
        assert x.dim() == 2 and x.dtype == torch.bfloat16 and x.is_cuda
        assert x.numel() == 0 or x.stride(1) == 1
        R, C = x.shape
        dev = x.device
        row = col = None
        if axis & MX_ROWWISE:
            row = MXTensor(torch.empty((R, C), dtype=torch.uint8, device=dev),
                           torch.empty(mx_scale_bytes(R, C), dtype=torch.uint8, device=dev), R, C, MX_ROWWISE)
        if axis & MX_COLWISE:
            col = MXTensor(torch.empty((C, R), dtype=torch.uint8, device=dev),
                           torch.empty(mx_scale_bytes(C, R), dtype=torch.uint8, device=dev), C, R, MX_COLWISE)
        outs.append((row, col))
        ldx = x.stride(0) if x.numel() else C  # an empty matrix's strides carry no pitch
        descs.append(MXQuantTensorC(x.data_ptr(), R, C, ldx,
                                    _ptr(row.data) if row else None, _ptr(row.scale) if row else None,
                                    _ptr(col.data) if col else None, _ptr(col.scale) if col else None))
    mx_quantize_multi(descs, axis, _ptr(status), _stream(stream))
    return outs


def gemm(mode: int, a: MXTensor, b: MXTensor, out=None, status=None, stream=None, workspace=None):
    """C[M, N] = A . B^T in BF16 (FP32 accumulation). With `workspace` (a CUDA
    uint8 tensor, see gemm_workspace) the GEMM may split its last round."""
    torch = _torch()
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.data.device)
    if workspace is None:
        mx_gemm(mode, a.c_operand(), b.c_operand(), out.data_ptr(), out.stride(0), _ptr(status), _stream(stream))
    else:
        mx_gemm_with_workspace(mode, a.c_operand(), b.c_operand(), out.data_ptr(), out.stride(0),
                               workspace.data_ptr() if workspace.numel() else None, workspace.numel(),
                               _ptr(status), _stream(stream))
    return out


def gemm_workspace(mode: int, a: MXTensor, b: MXTensor):
    """A workspace of the size mx_gemm_with_workspace uses for these operands
    (an empty tensor when the GEMM does not split)."""
    torch = _torch()
    n = mx_gemm_workspace_bytes(mode, a.c_operand(), b.c_operand())
    return torch.empty(n, dtype=torch.uint8, device=a.data.device)


def gemm_multi(problems, status=None, stream=None):
    """Several independent GEMMs (mode, a, b[, out]) in one launch; returns the
    outputs (BF16 [a.rows, b.rows], allocated where not given)."""
    torch = _torch()
    outs, descs = [], []
    for pr in problems:
        mode, a, b = pr[0], pr[1], pr[2]
        out = pr[3] if len(pr) > 3 and pr[3] is not None else \
            torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.data.device)
        outs.append(out)
        descs.append(MXGemmProblemC(a.c_operand(), b.c_operand(), out.data_ptr(), out.stride(0), mode, 0))
    mx_gemm_multi(descs, _ptr(status), _stream(stream))
    return outs


@dataclass
class MXStacked:
    """Per-expert quantised copies stacked as [E][rows][k] with per-expert
    scale blocks of mx_scale_bytes(rows, k) bytes."""
    data: "object"      # torch.uint8 [E, rows, k]
    scale: "object"     # torch.uint8 [E, mx_scale_bytes(rows, k)]
    rows: int
    k: int
    orient: int

    def c_operand(self) -> MXOperandC:
        return MXOperandC(self.data.data_ptr(), self.scale.data_ptr(), self.rows, self.k,
                          int(self.data.stride(1)), self.orient, 0)


def quantize_stacked(w, axis: int, status=None, stream=None):
    """Quantise stacked expert weights w[E, N, K] (BF16, or the FP32 master) in
    one batched launch. Returns (row_stack [E][N][K], col_stack [E][K][N]);
    entries None if not asked."""
    torch = _torch()
    E, N, K = w.shape
    dev = w.device
    row = col = None
    if axis & MX_ROWWISE:
        row = MXStacked(torch.empty((E, N, K), dtype=torch.uint8, device=dev),
                        torch.empty((E, mx_scale_bytes(N, K)), dtype=torch.uint8, device=dev), N, K, MX_ROWWISE)
    if axis & MX_COLWISE:
        col = MXStacked(torch.empty((E, K, N), dtype=torch.uint8, device=dev),
                        torch.empty((E, mx_scale_bytes(K, N)), dtype=torch.uint8, device=dev), K, N, MX_COLWISE)
    assert w.stride(2) == 1 and w.dtype in (torch.bfloat16, torch.float32)
    fn = mx_quantize_f32 if w.dtype == torch.float32 else mx_quantize_batched
    fn(w.data_ptr(), E, N, K, w.stride(1), w.stride(0), axis,
       _ptr(row.data) if row else None, _ptr(row.scale) if row else None,
       _ptr(col.data) if col else None, _ptr(col.scale) if col else None,
       _ptr(status), _stream(stream))
    return row, col


def grouped_gemm(mode: int, a, b, group_offsets, out=None, status=None, stream=None):
    """Grouped GEMM. fprop/dgrad: a MXTensor [M_total, K] (rows grouped by
    expert), b MXStacked [E][N][K] -> out [M_total, N]. wgrad: a, b grouped
    column copies (MXTensor [N, cap], [Kout, cap]) -> out [E, N, Kout]."""
    torch = _torch()
    E = group_offsets.numel() - 1
    if out is None:
        if mode == MX_WGRAD:
            out = torch.empty((E, a.rows, b.rows), dtype=torch.bfloat16, device=a.data.device)
        else:
            out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.data.device)
    ldc = out.stride(-2)
    mx_grouped_gemm(mode, a.c_operand(), b.c_operand(), group_offsets.data_ptr(), E, out.data_ptr(), ldc,
                    _ptr(status), _stream(stream))
    return out


def grouped_gemm_swiglu(a, b, group_offsets, out=None, status=None, stream=None):
    """Grouped gate_up fprop with SwiGLU in the epilogue: a MXTensor [M_total, K]
    (rows grouped by expert), b MXStacked [E][2F][K] (gate rows first) ->
    out [M_total, F] = silu(gate) * up in BF16."""
    torch = _torch()
    E = group_offsets.numel() - 1
    if out is None:
        out = torch.empty((a.rows, b.rows // 2), dtype=torch.bfloat16, device=a.data.device)
    mx_grouped_gemm_swiglu(a.c_operand(), b.c_operand(), group_offsets.data_ptr(), E, out.data_ptr(), out.stride(0),
                           _ptr(status), _stream(stream))
    return out


def grouped_gemm_swiglu_quantize(a, b, group_offsets, col_capacity: int, out=None, status=None, stream=None):
    """grouped_gemm_swiglu with the output's MX copies written instead of the
    output: returns (row_copy, col_copy) as quantize(output, MX_BOTH,
    group_offsets, col_capacity) would ([M_total, F] and the per-expert padded
    [F, col_capacity]). ``out``: an existing (row_copy, col_copy) pair to fill."""
    torch = _torch()
    E = group_offsets.numel() - 1
    R, F = a.rows, b.rows // 2
    dev = a.data.device
    if out is None:
        row = MXTensor(torch.empty((R, F), dtype=torch.uint8, device=dev),
                       torch.empty(mx_scale_bytes(R, F), dtype=torch.uint8, device=dev), R, F, MX_ROWWISE)
        col = MXTensor(torch.empty((F, col_capacity), dtype=torch.uint8, device=dev),
                       torch.empty(mx_scale_bytes(F, col_capacity), dtype=torch.uint8, device=dev), F, col_capacity,
                       MX_COLWISE)
    else:
        row, col = out
    mx_grouped_gemm_swiglu_quantize(a.c_operand(), b.c_operand(), group_offsets.data_ptr(), E, _ptr(row.data),
                                    _ptr(row.scale), _ptr(col.data), _ptr(col.scale), col_capacity, _ptr(status),
                                    _stream(stream))
    return row, col


@dataclass
class FP8Blockwise:
    """E4M3 data [rows, k] with FP32 block multipliers: block 1 -> scale
    [k/128, rows] (1 x 128 blocks), block 128 -> scale [ceil(rows/128), k/128]."""
    data: "object"
    scale: "object"
    rows: int
    k: int
    block: int


def quantize_fp8_blockwise(x, block: int, status=None, stream=None) -> FP8Blockwise:
    """DeepSeek-V3 blockwise FP8 quantisation of a 2-D BF16 CUDA tensor."""
    torch = _torch()
    assert x.dim() == 2 and x.dtype == torch.bfloat16 and x.is_cuda and x.stride(1) == 1
    R, C = x.shape
    data = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    shape = (C // 128, R) if block == 1 else ((R + 127) // 128, C // 128)
    scale = torch.empty(shape, dtype=torch.float32, device=x.device)
    mx_quantize_fp8_blockwise(x.data_ptr(), R, C, x.stride(0), block, data.data_ptr(), scale.data_ptr(),
                              _ptr(status), _stream(stream))
    return FP8Blockwise(data, scale, R, C, block)


def gemm_fp8_blockwise(a: FP8Blockwise, b: FP8Blockwise, out=None, status=None, stream=None):
    """C[M, N] = A . B^T for an activation (block 1) and a weight (block 128)."""
    torch = _torch()
    assert a.block == 1 and b.block == 128 and a.k == b.k
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.data.device)
    mx_gemm_fp8_blockwise(a.data.data_ptr(), a.scale.data_ptr(), a.rows, b.data.data_ptr(), b.scale.data_ptr(),
                          b.rows, a.k, out.data_ptr(), out.stride(0), _ptr(status), _stream(stream))
    return out


# ---------------------------------------------------------------------------
# Current-scaling variant (one FP32 scale per tensor or per expert)
# ---------------------------------------------------------------------------

CURRENT_FORMAT_MAX = 448.0


def current_amax(x, status=None, stream=None):
    """amax of a 2-D BF16 tensor ([1] FP32) or of each matrix of a 3-D stack ([E])."""
    torch = _torch()
    xs = x if x.dim() == 3 else x.unsqueeze(0)
    assert xs.dtype == torch.bfloat16 and xs.is_cuda and xs.stride(2) == 1
    E, R, C = xs.shape
    amax = torch.empty(E, dtype=torch.float32, device=x.device)
    mx_current_amax(xs.data_ptr(), E, R, C, xs.stride(1), xs.stride(0), amax.data_ptr(), _ptr(status), _stream(stream))
    return amax


def quantize_current(x, axis: int = MX_BOTH, amax=None, format_max: float = CURRENT_FORMAT_MAX, group_offsets=None,
                     col_capacity: Optional[int] = None, status=None, stream=None):
    """Current-scaling quantisation of a 2-D BF16 tensor (or a 3-D stack, one
    scale per matrix). amax: FP32 [batch] (computed here when None). Returns
    (row_copy, col_copy); each copy's `scale` is the FP32 scale tensor [batch]
    (the same tensor for both copies)."""
    torch = _torch()
    stacked = x.dim() == 3
    xs = x if stacked else x.unsqueeze(0)
    E, R, C = xs.shape
    dev = x.device
    if amax is None:
        amax = current_amax(x, status=status, stream=stream)
    scale = torch.empty(E, dtype=torch.float32, device=dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    row = col = None
    n_groups, cap = 0, 0
    if axis & MX_ROWWISE:
        d = torch.empty((E, R, C), **u8)
        row = (MXStacked(d, scale, R, C, MX_ROWWISE) if stacked else MXTensor(d[0], scale, R, C, MX_ROWWISE))
    if axis & MX_COLWISE:
        if group_offsets is not None:
            assert not stacked
            n_groups = group_offsets.numel() - 1
            cap = int(col_capacity) if col_capacity is not None else ((R + 127 * n_groups + 127) // 128) * 128
            col = MXTensor(torch.empty((C, cap), **u8), scale, C, cap, MX_COLWISE)
        else:
            d = torch.empty((E, C, R), **u8)
            col = (MXStacked(d, scale, C, R, MX_COLWISE) if stacked else MXTensor(d[0], scale, C, R, MX_COLWISE))
    mx_quantize_current(xs.data_ptr(), E, R, C, xs.stride(1), xs.stride(0), axis, amax.data_ptr(), float(format_max),
                        _ptr(row.data) if row else None, _ptr(col.data) if col else None, scale.data_ptr(),
                        _ptr(group_offsets), n_groups, cap, _ptr(status), _stream(stream))
    return row, col


def gemm_current(mode: int, a, b, out=None, status=None, stream=None):
    """C[M, N] = (A . B^T) * s_a * s_b in BF16 for current-scaled operands."""
    torch = _torch()
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.data.device)
    mx_gemm_current(mode, a.c_operand(), b.c_operand(), out.data_ptr(), out.stride(0), _ptr(status), _stream(stream))
    return out


def gemm_current_multi(problems, status=None, stream=None):
    """Several independent current-scaled GEMMs (mode, a, b[, out]) in one
    launch; returns the outputs (BF16 [a.rows, b.rows], allocated where not
    given)."""
    torch = _torch()
    outs, descs = [], []
    for pr in problems:
        mode, a, b = pr[0], pr[1], pr[2]
        out = pr[3] if len(pr) > 3 and pr[3] is not None else \
            torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.data.device)
        outs.append(out)
        descs.append(MXGemmProblemC(a.c_operand(), b.c_operand(), out.data_ptr(), out.stride(0), mode, 0))
    mx_gemm_current_multi(descs, _ptr(status), _stream(stream))
    return outs


def grouped_gemm_current(mode: int, a, b, group_offsets, out=None, status=None, stream=None):
    """Grouped GEMM on current-scaled operands (layouts as grouped_gemm; the
    stacked weights carry one scale per expert)."""
    torch = _torch()
    E = group_offsets.numel() - 1
    if out is None:
        shape = (E, a.rows, b.rows) if mode == MX_WGRAD else (a.rows, b.rows)
        out = torch.empty(shape, dtype=torch.bfloat16, device=a.data.device)
    mx_grouped_gemm_current(mode, a.c_operand(), b.c_operand(), group_offsets.data_ptr(), E, out.data_ptr(),
                            out.stride(-2), _ptr(status), _stream(stream))
    return out
