"""Thin Python binding of libvnm's C ABI (include/vnm.h), same names.

Argument marshalling only: PyTorch provides device memory and streams, and
every step of the computation runs in libvnm's CUDA kernels. There is no CPU
or PyTorch fallback: if libvnm.so is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Tuple

import torch

from . import build as _build

VNM_OK = 0
VNM_ERR_INVALID_ARG = 1
VNM_ERR_UNSUPPORTED = 2
VNM_ERR_CUDA = 3
VNM_ERR_NONFINITE = 4
VNM_ERR_TIMEOUT = 5
VNM_ERR_INTERNAL = 6

VNM_F16 = 0
VNM_F32 = 1

VNM_PATH_NONE = 0
VNM_PATH_TC = 1
VNM_PATH_SIMT = 2

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class VnmError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class vnm_spmm_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("splits", ctypes.c_int32), ("lift", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]

    def as_dict(self):
        return {k: getattr(self, k) for k in ("path", "tile_m", "tile_n", "stages", "splits", "lift")}


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    L.vnm_status_string.argtypes = [ctypes.c_int]
    L.vnm_status_string.restype = ctypes.c_char_p
    L.vnm_version.argtypes = []
    L.vnm_version.restype = i32
    L.vnm_sizes.argtypes = [i64, i64, i32, i32, p, p, p]
    L.vnm_matrix_create.argtypes = [i64, i64, i32, i32, p, p, p, p]
    L.vnm_matrix_destroy.argtypes = [p]
    L.vnm_compress.argtypes = [p, p, i64, p]
    L.vnm_decompress.argtypes = [p, p, i64, p]
    L.vnm_gemm_compress.argtypes = [p, p, i64, p, i64, i64, p, i64, p]
    L.vnm_energy.argtypes = [p, p, i64, ctypes.c_int, p, sz, p, p, p, p]
    L.vnm_linear.argtypes = [p, p, i64, i64, p, ctypes.c_int, p, i64, ctypes.c_int, p, sz, p]
    L.vnm_linear_workspace_size.argtypes = [p, i64, p]
    L.vnm_bitmap_sizes.argtypes = [i64, i64, p, p, p, p]
    L.vnm_bitmap_encode.argtypes = [p, i64, i64, i64, p, p, p, p, i64, p, p]
    L.vnm_bitmap_spmm.argtypes = [i64, i64, p, p, p, p, p, i64, i64, p, i64, ctypes.c_int, p, sz, p]
    L.vnm_bitmap_spmm_workspace_size.argtypes = [i64, i64, i64, p]
    L.vnm_energy_workspace_size.argtypes = [p, p]
    L.vnm_spmm.argtypes = [p, p, i64, i64, p, i64, ctypes.c_int, p, sz, p]
    L.vnm_spmm_workspace_size.argtypes = [p, i64, p]
    L.vnm_spmm_plan_query.argtypes = [p, p, i64, i64, ctypes.c_int, sz, ctypes.POINTER(vnm_spmm_plan)]
    L.vnm_spmm_with_plan.argtypes = [p, ctypes.POINTER(vnm_spmm_plan), p, i64, i64, p, i64, ctypes.c_int, p, sz, p]
    L.vnm_get_status.argtypes = [p, p]
    L.vnm_spmm_noalloc.argtypes = [i64, i64, i32, i32, p, p, p, p, i64, i64, p, i64, ctypes.c_int, p, p]
    L.vnm_testing_spmm_skip_stage.argtypes = [p, p, i64, i64, p, i64, ctypes.c_int, p, sz, i32, p]
    for name in ("vnm_sizes", "vnm_matrix_create", "vnm_matrix_destroy", "vnm_compress", "vnm_decompress",
                 "vnm_spmm", "vnm_spmm_workspace_size", "vnm_spmm_plan_query", "vnm_spmm_with_plan",
                 "vnm_get_status", "vnm_spmm_noalloc", "vnm_testing_spmm_skip_stage"):
        getattr(L, name).restype = ctypes.c_int
    return L


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """libvnm, loaded once. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB_PATH):
                raise RuntimeError(
                    f"libvnm is not built ({_build.LIB_PATH} missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            _lib = _declare(ctypes.CDLL(_build.LIB_PATH))
        return _lib


def status_string(code: int) -> str:
    return lib().vnm_status_string(code).decode()


def _check(code: int, what: str) -> None:
    if code != VNM_OK:
        raise VnmError(code, what)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _rowmajor(t: torch.Tensor, name: str) -> int:
    """Leading dimension (elements) of a row-major 2-D tensor."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major tensor (stride(1) == 1)")
    return max(int(t.stride(0)), int(t.shape[1]), 1)


def vnm_version() -> int:
    return int(lib().vnm_version())


def vnm_sizes(R: int, K: int, V: int, M: int) -> Tuple[int, int, int]:
    """Byte sizes (values, meta, colidx) of the compressed arrays."""
    v, m, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().vnm_sizes(R, K, V, M, ctypes.byref(v), ctypes.byref(m), ctypes.byref(c)), "vnm_sizes")
    return v.value, m.value, c.value


@dataclass
class VnmMatrix:
    """A handle plus the caller-owned compressed arrays it describes."""

    handle: int
    R: int
    K: int
    V: int
    M: int
    values: torch.Tensor  # fp16 [R, 2K/M]
    meta: torch.Tensor    # uint8 [R, ceil(2K/M/4)]
    colidx: torch.Tensor  # uint8 [R/V, K/M, 4]

    def __del__(self):
        try:
            if self.handle:
                vnm_matrix_destroy(self)
        except Exception:
            pass


def vnm_matrix_create(R: int, K: int, V: int, M: int, values: torch.Tensor, meta: torch.Tensor,
                      colidx: torch.Tensor) -> VnmMatrix:
    h = ctypes.c_void_p()
    _check(lib().vnm_matrix_create(R, K, V, M, values.data_ptr() or None, meta.data_ptr() or None,
                                   colidx.data_ptr() or None, ctypes.byref(h)), "vnm_matrix_create")
    return VnmMatrix(int(h.value), R, K, V, M, values, meta, colidx)


def vnm_matrix_alloc(R: int, K: int, V: int, M: int, device=None) -> VnmMatrix:
    """Allocate the three arrays with torch on ``device`` and create a handle."""
    vb, mb, cb = vnm_sizes(R, K, V, M)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    values = torch.empty((R, 2 * (K // M)), dtype=torch.float16, device=dev)
    meta = torch.empty((R, (2 * (K // M) + 3) // 4), dtype=torch.uint8, device=dev)
    colidx = torch.empty((R // V, K // M, 4), dtype=torch.uint8, device=dev)
    assert values.numel() * 2 == vb and meta.numel() == mb and colidx.numel() == cb
    with torch.cuda.device(dev):
        return vnm_matrix_create(R, K, V, M, values, meta, colidx)


def vnm_matrix_destroy(A: VnmMatrix) -> None:
    h, A.handle = A.handle, 0
    if h:
        _check(lib().vnm_matrix_destroy(h), "vnm_matrix_destroy")


def vnm_compress(A: VnmMatrix, W: torch.Tensor, stream=None) -> None:
    if W.dtype != torch.float16 or not W.is_cuda or tuple(W.shape) != (A.R, A.K):
        raise ValueError("W must be a CUDA fp16 tensor of shape (R, K)")
    _check(lib().vnm_compress(A.handle, W.data_ptr() or None, _rowmajor(W, "W"), _stream_ptr(stream)),
           "vnm_compress")


def vnm_decompress(A: VnmMatrix, W_out: torch.Tensor, stream=None) -> None:
    if W_out.dtype != torch.float16 or not W_out.is_cuda or tuple(W_out.shape) != (A.R, A.K):
        raise ValueError("W_out must be a CUDA fp16 tensor of shape (R, K)")
    _check(lib().vnm_decompress(A.handle, W_out.data_ptr() or None, _rowmajor(W_out, "W_out"), _stream_ptr(stream)),
           "vnm_decompress")


def vnm_gemm_compress(A: VnmMatrix, X: torch.Tensor, Y: torch.Tensor, W_out: Optional[torch.Tensor] = None,
                      stream=None) -> None:
    """W = X . Y^T (X: R x D, Y: K x D, fp16), compressed into A in the GEMM's
    epilogue; W_out (R x K fp16), if given, also receives W."""
    if X.dtype != torch.float16 or not X.is_cuda or X.dim() != 2 or X.shape[0] != A.R:
        raise ValueError("X must be a CUDA fp16 tensor of shape (R, D)")
    if Y.dtype != torch.float16 or not Y.is_cuda or Y.dim() != 2 or Y.shape[0] != A.K or Y.shape[1] != X.shape[1]:
        raise ValueError("Y must be a CUDA fp16 tensor of shape (K, D)")
    D = int(X.shape[1])
    w_ptr, ld_w = None, max(A.K, 1)
    if W_out is not None:
        if W_out.dtype != torch.float16 or not W_out.is_cuda or tuple(W_out.shape) != (A.R, A.K):
            raise ValueError("W_out must be a CUDA fp16 tensor of shape (R, K)")
        w_ptr, ld_w = W_out.data_ptr() or None, _rowmajor(W_out, "W_out")
    ld_x = _rowmajor(X, "X") if D > 0 else 1
    ld_y = _rowmajor(Y, "Y") if D > 0 else 1
    _check(lib().vnm_gemm_compress(A.handle, X.data_ptr() or None, ld_x, Y.data_ptr() or None, ld_y, D, w_ptr, ld_w,
                                   _stream_ptr(stream)), "vnm_gemm_compress")


class BitmapMatrix:
    """A matrix in the bitmap format (bitmaps, offsets, bases, values as torch
    tensors on one device), made by bitmap_encode."""

    def __init__(self, R: int, K: int, bitmaps, offsets, bases, values, values_storage=None):
        self.R, self.K = R, K
        self.bitmaps, self.offsets, self.bases, self.values = bitmaps, offsets, bases, values
        # an allocation holding `values` (an empty slice has no address of its own)
        self._values_storage = values if values_storage is None else values_storage

    def values_ptr(self) -> int:
        return self.values.data_ptr() if self.values.numel() else self._values_storage.data_ptr()


def bitmap_encode(W: torch.Tensor, stream=None) -> BitmapMatrix:
    """Encode fp16 W (R x K, R % 64 == 0) into the bitmap format (two passes:
    the arrays of positions, then the values once their length is known)."""
    if W.dtype != torch.float16 or not W.is_cuda or W.dim() != 2:
        raise ValueError("W must be a CUDA fp16 matrix")
    R, K = int(W.shape[0]), int(W.shape[1])
    nb = ctypes.c_size_t(0); no = ctypes.c_size_t(0); nbase = ctypes.c_size_t(0); nv = ctypes.c_size_t(0)
    _check(lib().vnm_bitmap_sizes(R, K, ctypes.byref(nb), ctypes.byref(no), ctypes.byref(nbase), ctypes.byref(nv)),
           "vnm_bitmap_sizes")
    dev = W.device
    bitmaps = torch.empty(max(1, nb.value // 8), dtype=torch.int64, device=dev)
    offsets = torch.empty(max(1, no.value // 4), dtype=torch.int32, device=dev)
    bases = torch.empty(nbase.value // 8, dtype=torch.int64, device=dev)
    ld = _rowmajor(W, "W") if K > 0 else 1
    need = ctypes.c_int64(0)
    code = lib().vnm_bitmap_encode(W.data_ptr() or None, ld, R, K, bitmaps.data_ptr(), offsets.data_ptr(),
                                   bases.data_ptr(), None, 0, ctypes.byref(need), _stream_ptr(stream))
    values = torch.empty(max(8, int(need.value)), dtype=torch.float16, device=dev)
    if code == VNM_ERR_INVALID_ARG and need.value > 0:
        code = lib().vnm_bitmap_encode(W.data_ptr() or None, ld, R, K, bitmaps.data_ptr(), offsets.data_ptr(),
                                       bases.data_ptr(), values.data_ptr(), values.numel(), ctypes.byref(need),
                                       _stream_ptr(stream))
    _check(code, "vnm_bitmap_encode")
    return BitmapMatrix(R, K, bitmaps, offsets, bases, values[:int(need.value)], values)


def bitmap_spmm_workspace_size(R: int, K: int, N: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().vnm_bitmap_spmm_workspace_size(R, K, N, ctypes.byref(n)), "vnm_bitmap_spmm_workspace_size")
    return int(n.value)


def bitmap_spmm(A: BitmapMatrix, B: torch.Tensor, C: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                stream=None) -> None:
    """C = A . B for A in the bitmap format (B fp16 K x N, C fp16 or fp32 R x N)."""
    if B.dtype != torch.float16 or not B.is_cuda or B.dim() != 2 or B.shape[0] != A.K:
        raise ValueError("B must be a CUDA fp16 tensor of shape (K, N)")
    N = int(B.shape[1])
    if not C.is_cuda or tuple(C.shape) != (A.R, N):
        raise ValueError("C must be a CUDA tensor of shape (R, N)")
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().vnm_bitmap_spmm(A.R, A.K, A.bitmaps.data_ptr(), A.offsets.data_ptr(), A.bases.data_ptr(),
                                 A.values_ptr() or None, B.data_ptr() or None, _rowmajor(B, "B") if N else 1, N,
                                 C.data_ptr() or None, _rowmajor(C, "C") if N else 1, _c_type(C), ws_ptr, ws_bytes,
                                 _stream_ptr(stream)), "vnm_bitmap_spmm")


VNM_ACT_NONE, VNM_ACT_RELU, VNM_ACT_GELU = 0, 1, 2


def vnm_linear_workspace_size(A: VnmMatrix, T: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().vnm_linear_workspace_size(A.handle, int(T), ctypes.byref(n)), "vnm_linear_workspace_size")
    return int(n.value)


def vnm_linear(A: VnmMatrix, X: torch.Tensor, Y: torch.Tensor, bias: Optional[torch.Tensor] = None,
               act: int = VNM_ACT_NONE, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Y = act(X . A^T + bias): X (T x K fp16), Y (T x R, fp16 or fp32), bias (R fp16) or None."""
    if X.dtype != torch.float16 or not X.is_cuda or X.dim() != 2 or X.shape[1] != A.K:
        raise ValueError("X must be a CUDA fp16 tensor of shape (T, K)")
    T = int(X.shape[0])
    if not Y.is_cuda or Y.dim() != 2 or tuple(Y.shape) != (T, A.R):
        raise ValueError("Y must be a CUDA tensor of shape (T, R)")
    if bias is not None and (bias.dtype != torch.float16 or not bias.is_cuda or tuple(bias.shape) != (A.R,)
                             or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous CUDA fp16 tensor of shape (R,)")
    if workspace is None:
        n = vnm_linear_workspace_size(A, T)
        workspace = torch.empty(n, dtype=torch.uint8, device=X.device) if n else None
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    ld_x = _rowmajor(X, "X") if A.K > 0 else 1
    _check(lib().vnm_linear(A.handle, X.data_ptr() or None, ld_x, T,
                            bias.data_ptr() if bias is not None else None, int(act), Y.data_ptr() or None,
                            _rowmajor(Y, "Y"), _c_type(Y), ws_ptr, ws_bytes, _stream_ptr(stream)), "vnm_linear")


VNM_PATTERN_VNM, VNM_PATTERN_UNSTRUCTURED, VNM_PATTERN_VECTORWISE = 0, 1, 2


def vnm_energy_workspace_size(A: VnmMatrix) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().vnm_energy_workspace_size(A.handle, ctypes.byref(n)), "vnm_energy_workspace_size")
    return int(n.value)


def vnm_energy(A: VnmMatrix, W: torch.Tensor, pattern: int, workspace: Optional[torch.Tensor] = None,
               stream=None) -> Tuple[float, int, int]:
    """Energy of pruning W (R x K fp16) with `pattern` at density 2/M:
    (energy, kept units, total units), the sums exact in units of 2^-24.
    VNM_PATTERN_VNM reads A, which must hold vnm_compress(A, W)."""
    if W.dtype != torch.float16 or not W.is_cuda or tuple(W.shape) != (A.R, A.K):
        raise ValueError("W must be a CUDA fp16 tensor of shape (R, K)")
    if workspace is None:
        workspace = torch.empty(vnm_energy_workspace_size(A), dtype=torch.uint8, device=W.device)
    kept = (ctypes.c_uint64 * 2)()
    total = (ctypes.c_uint64 * 2)()
    e = ctypes.c_double(0.0)
    _check(lib().vnm_energy(A.handle, W.data_ptr() or None, _rowmajor(W, "W"), int(pattern), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), kept, total, ctypes.byref(e),
                            _stream_ptr(stream)), "vnm_energy")
    return float(e.value), int(kept[0]) | (int(kept[1]) << 64), int(total[0]) | (int(total[1]) << 64)


def _c_type(C: torch.Tensor) -> int:
    if C.dtype == torch.float16:
        return VNM_F16
    if C.dtype == torch.float32:
        return VNM_F32
    raise ValueError("C must be fp16 or fp32")


def _spmm_operands(A: VnmMatrix, B: torch.Tensor, C: torch.Tensor):
    if B.dtype != torch.float16 or not B.is_cuda or B.dim() != 2 or B.shape[0] != A.K:
        raise ValueError("B must be a CUDA fp16 tensor of shape (K, N)")
    N = int(B.shape[1])
    if not C.is_cuda or tuple(C.shape) != (A.R, N):
        raise ValueError("C must be a CUDA tensor of shape (R, N)")
    return N, _rowmajor(B, "B"), _rowmajor(C, "C"), _c_type(C)


def vnm_spmm_workspace_size(A: VnmMatrix, N: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().vnm_spmm_workspace_size(A.handle, N, ctypes.byref(b)), "vnm_spmm_workspace_size")
    return b.value


def vnm_spmm_plan_query(A: VnmMatrix, B: torch.Tensor, c_dtype=torch.float16, workspace_bytes: int = 0
                        ) -> vnm_spmm_plan:
    plan = vnm_spmm_plan()
    N = int(B.shape[1])
    ct = VNM_F16 if c_dtype == torch.float16 else VNM_F32
    _check(lib().vnm_spmm_plan_query(A.handle, B.data_ptr() or None, _rowmajor(B, "B"), N, ct, workspace_bytes,
                                     ctypes.byref(plan)), "vnm_spmm_plan_query")
    return plan


def vnm_spmm(A: VnmMatrix, B: torch.Tensor, C: torch.Tensor, workspace: Optional[torch.Tensor] = None,
             stream=None) -> None:
    """C = A . B on ``stream`` (default: torch's current stream)."""
    N, ld_b, ld_c, ct = _spmm_operands(A, B, C)
    wp = workspace.data_ptr() if workspace is not None and workspace.numel() else None
    wb = workspace.numel() * workspace.element_size() if wp else 0
    _check(lib().vnm_spmm(A.handle, B.data_ptr() or None, ld_b, N, C.data_ptr() or None, ld_c, ct, wp, wb,
                          _stream_ptr(stream)), "vnm_spmm")


def vnm_spmm_with_plan(A: VnmMatrix, plan: vnm_spmm_plan, B: torch.Tensor, C: torch.Tensor,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    N, ld_b, ld_c, ct = _spmm_operands(A, B, C)
    wp = workspace.data_ptr() if workspace is not None and workspace.numel() else None
    wb = workspace.numel() * workspace.element_size() if wp else 0
    _check(lib().vnm_spmm_with_plan(A.handle, ctypes.byref(plan), B.data_ptr() or None, ld_b, N,
                                    C.data_ptr() or None, ld_c, ct, wp, wb, _stream_ptr(stream)),
           "vnm_spmm_with_plan")


def vnm_testing_spmm_skip_stage(A: VnmMatrix, B: torch.Tensor, C: torch.Tensor, skip_stage: int,
                                workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Test support: vnm_spmm with the first CTA's loads of one pipeline stage
    never issued, so that its bounded waits run out (include/vnm_testing.h)."""
    N, ld_b, ld_c, ct = _spmm_operands(A, B, C)
    wp = workspace.data_ptr() if workspace is not None and workspace.numel() else None
    wb = workspace.numel() * workspace.element_size() if wp else 0
    _check(lib().vnm_testing_spmm_skip_stage(A.handle, B.data_ptr() or None, ld_b, N, C.data_ptr() or None, ld_c,
                                             ct, wp, wb, int(skip_stage), _stream_ptr(stream)),
           "vnm_testing_spmm_skip_stage")


def vnm_get_status(A: VnmMatrix, stream=None) -> int:
    """Synchronise the stream and return (and clear) the kernels' first error code."""
    return int(lib().vnm_get_status(A.handle, _stream_ptr(stream)))


def workspace_for(A: VnmMatrix, N: int, device=None) -> Optional[torch.Tensor]:
    """A torch-allocated workspace of the size vnm_spmm's plan wants (None if 0)."""
    nbytes = vnm_spmm_workspace_size(A, N)
    if nbytes == 0:
        return None
    dev = device if device is not None else A.values.device
    return torch.empty(nbytes // 4 + 64, dtype=torch.float32, device=dev)


def vnm_spmm_noalloc(R: int, K: int, V: int, M: int, values: torch.Tensor, meta: torch.Tensor,
                     colidx: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                     status: Optional[torch.Tensor] = None, stream=None) -> None:
    """C = A . B from the compressed arrays, without any device allocation.

    For callers that cannot call cudaMalloc (memory held in full by another
    allocator, or a path that must not synchronise the device): the split-K
    scratch is a static 8 MiB device array inside libvnm. ``status`` is an
    optional int32 CUDA tensor of 3 zeroed words that receives kernel errors.
    """
    if B.dtype != torch.float16 or not B.is_cuda or B.dim() != 2 or B.shape[0] != K:
        raise ValueError("B must be a CUDA fp16 tensor of shape (K, N)")
    N = int(B.shape[1])
    if not C.is_cuda or tuple(C.shape) != (R, N):
        raise ValueError("C must be a CUDA tensor of shape (R, N)")
    sp = None
    if status is not None:
        if status.dtype != torch.int32 or not status.is_cuda or status.numel() < 3:
            raise ValueError("status must be a CUDA int32 tensor of at least 3 words")
        sp = status.data_ptr()
    _check(lib().vnm_spmm_noalloc(R, K, V, M, values.data_ptr() or None, meta.data_ptr() or None,
                                  colidx.data_ptr() or None, B.data_ptr() or None, _rowmajor(B, "B"), N,
                                  C.data_ptr() or None, _rowmajor(C, "C"), _c_type(C), sp, _stream_ptr(stream)),
           "vnm_spmm_noalloc")
