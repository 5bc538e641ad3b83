"""CPU oracle for the V:N:M format and SpMM (ctypes wrapper of vnm_oracle.c).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``structured_sparse_matmul_gb300``) never imports
it, and the two share no code.

The C source restates "VENOM: A Vectorized N:M Format for Unleashing the
Power of Sparse Tensor Cores", section 3 (Figures 2 and 3) and section 4
(Figure 4), with the 2:4 packing of the lecture notes "2:4 sparsity on sparse
tensor cores" ("The compressed format", "Worked: compress a 2 x 8 matrix").
:func:`gemm_compress` composes numpy's fp64 matmul with the C compress
(DFSS sections 4.2-4.3). Every function is pinned by tests/test_oracle.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vnm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_vnm.so")
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

OK, INVALID, NONFINITE, NOMEM = 0, 1, 4, 6


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} returned {code}")
        self.code = code


def build(src: str = _SRC, out: str = _LIB_PATH, defines: Sequence[str] = ()) -> str:
    """Compile the oracle with gcc (plain C11, no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           *[f"-D{d}" for d in defines], src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.oracle_sizes.argtypes = [i64, i64, i32, i32, p, p, p]
    lib.oracle_compress.argtypes = [p, i64, i64, i64, i32, i32, p, p, p]
    lib.oracle_decompress.argtypes = [p, p, p, i64, i64, i32, i32, p, i64]
    spmm_args = [p, p, p, i64, i64, i32, i32, p, i64, i64, p, i64, p]
    lib.oracle_spmm_f32.argtypes = spmm_args
    lib.oracle_spmm_f64.argtypes = spmm_args
    for f in (lib.oracle_sizes, lib.oracle_compress, lib.oracle_decompress, lib.oracle_spmm_f32,
              lib.oracle_spmm_f64):
        f.restype = ctypes.c_int
    return lib


def load_from(path: str) -> ctypes.CDLL:
    """Load an oracle shared library built from ``path`` (tests load variants)."""
    return _declare(ctypes.CDLL(path))


def lib() -> ctypes.CDLL:
    """The oracle library, built on first use if missing or older than its source."""
    global _lib
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = load_from(_LIB_PATH)
        return _lib


def _ptr(a: Optional[np.ndarray]) -> Optional[int]:
    return None if a is None else a.ctypes.data


def sizes(R: int, K: int, V: int, M: int, L: Optional[ctypes.CDLL] = None) -> Tuple[int, int, int]:
    """(number of fp16 values, bytes of m-indices, bytes of column-loc)."""
    L = L or lib()
    v, m, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    rc = L.oracle_sizes(R, K, V, M, ctypes.byref(v), ctypes.byref(m), ctypes.byref(c))
    if rc != OK:
        raise OracleError(rc, "sizes")
    return v.value, m.value, c.value


def meta_pitch(K: int, M: int) -> int:
    """Bytes per row of m-indices (2 bits per stored value, rounded up)."""
    return (2 * (K // M) + 3) // 4


def compress(W: np.ndarray, V: int, M: int, L: Optional[ctypes.CDLL] = None):
    """Magnitude V:N:M compress of an fp16 R x K matrix.

    Returns ``(values, meta, colidx)``: values uint16 [R, 2K/M] (fp16 bit
    patterns), meta uint8 [R, ceil(2K/M/4)], colidx uint8 [R/V, K/M, 4].
    """
    L = L or lib()
    W = np.ascontiguousarray(W, dtype=np.float16)
    R, K = W.shape
    nv, nm, nc = sizes(R, K, V, M, L)
    values = np.zeros((R, 2 * (K // M)), dtype=np.uint16)
    meta = np.zeros((R, meta_pitch(K, M)), dtype=np.uint8)
    colidx = np.zeros((R // V, K // M, 4), dtype=np.uint8)
    assert values.size == nv and meta.size == nm and colidx.size == nc
    rc = L.oracle_compress(_ptr(W), K, R, K, V, M, _ptr(values), _ptr(meta), _ptr(colidx))
    if rc != OK:
        raise OracleError(rc, "compress")
    return values, meta, colidx


def gemm_compress(X: np.ndarray, Y: np.ndarray, V: int, M: int, L: Optional[ctypes.CDLL] = None):
    """The fused GEMM + prune-and-encode: W = X . Y^T, then ``compress(W)``.

    Restates "Dynamic N:M fine-grained structured sparse attention" (DFSS),
    sections 4.2-4.3: the dense product that yields the sparse operand (there
    Q K^T) is pruned and encoded as it is produced; the pruning rule here is
    that of :func:`compress` (VENOM section 3). X is fp16 R x D, Y fp16 K x D.
    The product step is numpy's matmul in fp64 (every product of two fp16
    values is exact in fp64); W is rounded once from fp64 to fp16, to nearest
    even. Returns ``(W, (values, meta, colidx))`` with W fp16 R x K.
    """
    X = np.asarray(X, dtype=np.float16)
    Y = np.asarray(Y, dtype=np.float16)
    assert X.ndim == 2 and Y.ndim == 2 and X.shape[1] == Y.shape[1]
    with np.errstate(over="ignore"):  # beyond the fp16 range: Inf, reported by compress()
        W = (X.astype(np.float64) @ Y.astype(np.float64).T).astype(np.float16)
    return W, compress(W, V, M, L)


def bitmap_encode(W: np.ndarray):
    """The bitmap format of "Coruscant" section 3.1 (Figure 7) for fp16 W
    (R x K, R % 64 == 0): column tiles of 64 rows; tile (i, k) is rows
    64i .. 64i+63 of column k. Returns ``(bitmaps, offsets, bases, values)``:
    bitmaps uint64 [R/64, K] with bit r set when W[64i + r, k] is not +-0;
    values fp16 bit patterns, per tile (row-block major, then column) its
    non-zero values in row order followed by +0.0 up to a multiple of 8;
    offsets uint32 [R/64, K] the start of each tile's values relative to its
    row block's first value; bases int64 [R/64 + 1] those firsts (the last
    is the total length)."""
    W = np.ascontiguousarray(W, dtype=np.float16)
    R, K = W.shape
    assert R % 64 == 0
    nb = R // 64
    bits = W.view(np.uint16)
    bitmaps = np.zeros((nb, K), dtype=np.uint64)
    offsets = np.zeros((nb, K), dtype=np.uint32)
    bases = np.zeros(nb + 1, dtype=np.int64)
    chunks = []
    total = 0
    for i in range(nb):
        start = total
        for k in range(K):
            col = bits[64 * i:64 * (i + 1), k]
            rows = [r for r in range(64) if int(col[r]) & 0x7FFF]
            bitmaps[i, k] = np.uint64(sum(1 << r for r in rows))
            offsets[i, k] = total - start
            padded = (len(rows) + 7) // 8 * 8
            chunk = np.zeros(padded, dtype=np.uint16)
            chunk[:len(rows)] = col[rows]
            chunks.append(chunk)
            total += padded
        bases[i + 1] = total
    values = np.concatenate(chunks) if chunks else np.zeros(0, dtype=np.uint16)
    return bitmaps, offsets, bases, values


def bitmap_decode(bitmaps: np.ndarray, offsets: np.ndarray, bases: np.ndarray, values: np.ndarray, R: int,
                  K: int) -> np.ndarray:
    """Dense fp16 R x K from the bitmap format (positions without a bit: +0.0)."""
    W = np.zeros((R, K), dtype=np.uint16)
    for i in range(R // 64):
        for k in range(K):
            bm = int(bitmaps[i, k])
            at = int(bases[i]) + int(offsets[i, k])
            n = 0
            for r in range(64):
                if (bm >> r) & 1:
                    W[64 * i + r, k] = values[at + n]
                    n += 1
    return W.view(np.float16)


def bitmap_spmm(bitmaps, offsets, bases, values, R: int, K: int, B: np.ndarray) -> np.ndarray:
    """C = A . B in fp64 for A in the bitmap format (numpy's matmul of the
    decoded A; fp16 products are exact in fp64)."""
    A = bitmap_decode(bitmaps, offsets, bases, values, R, K).astype(np.float64)
    return A @ np.asarray(B, dtype=np.float16).astype(np.float64)


ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2


def linear(values: np.ndarray, meta: np.ndarray, colidx: np.ndarray, R: int, K: int, V: int, M: int,
           X: np.ndarray, bias: Optional[np.ndarray] = None, act: int = ACT_NONE) -> np.ndarray:
    """Y = act(X . A^T + bias) in fp64 (the Linear-layer form of the SpMM, as
    "VENOM" section 7's transformer layers apply a pruned weight): the fp64
    :func:`spmm` of A by X^T, transposed, plus the fp16 bias, then ReLU
    max(y, 0) or GELU y * (1 + erf(y / sqrt 2)) / 2. X is fp16 T x K."""
    import math
    X = np.asarray(X, dtype=np.float16)
    C = spmm(values, meta, colidx, R, K, V, M, np.ascontiguousarray(X.T), acc="f64")  # R x T
    Y = C.T.copy()
    if bias is not None:
        Y += np.asarray(bias, dtype=np.float16).astype(np.float64)[None, :]
    if act == ACT_RELU:
        Y = np.maximum(Y, 0.0)
    elif act == ACT_GELU:
        Y = Y * (1.0 + np.vectorize(math.erf)(Y / math.sqrt(2.0))) / 2.0
    return Y


PATTERN_VNM, PATTERN_UNSTRUCTURED, PATTERN_VECTORWISE = 0, 1, 2


def _units(h16: np.ndarray) -> np.ndarray:
    """|w| of fp16 values in units of 2^-24, as exact integers (uint64): the
    fp16 -> fp64 conversion is exact and every |fp16| is a multiple of 2^-24
    below 2^41."""
    return (np.abs(np.asarray(h16, dtype=np.float16).astype(np.float64)) * 2.0 ** 24).astype(np.uint64)


def energy(W: np.ndarray, V: int, M: int, pattern: int, L: Optional[ctypes.CDLL] = None):
    """Energy (magnitude preservation) of pruning fp16 W at density 2/M.

    Restates "VENOM", section 5 (Figure 11): the sum of the kept |w| over the
    sum of all |w|. ``pattern``: PATTERN_VNM keeps the values of
    :func:`compress` (V:N:M); PATTERN_UNSTRUCTURED the R*2K/M largest |w|;
    PATTERN_VECTORWISE, per panel of V rows, the 2K/M columns of largest L1
    norm over the panel (vectors of V x 1). Returns ``(energy, kept, total)``
    with kept and total exact Python integers in units of 2^-24 (energy 1.0
    for an all-zero W).
    """
    W = np.ascontiguousarray(W, dtype=np.float16)
    R, K = W.shape
    u = _units(W)
    total = int(u.sum(dtype=np.uint64)) if u.size else 0
    k = 2 * (K // M)
    if pattern == PATTERN_VNM:
        values = compress(W, V, M, L)[0]
        kept = int(_units(values.view(np.float16)).sum(dtype=np.uint64)) if values.size else 0
    elif pattern == PATTERN_UNSTRUCTURED:
        flat = np.sort(u.ravel())[::-1]
        kept = sum(int(x) for x in flat[:R * k])
    elif pattern == PATTERN_VECTORWISE:
        kept = 0
        for i in range(R // V):
            col = u[i * V:(i + 1) * V].sum(axis=0, dtype=np.uint64)  # exact: below 2^53
            kept += sum(int(x) for x in np.sort(col)[::-1][:k])
    else:
        raise ValueError(f"no pattern {pattern}")
    return (1.0 if total == 0 else kept / total), kept, total


def decompress(values: np.ndarray, meta: np.ndarray, colidx: np.ndarray, R: int, K: int, V: int,
               M: int, L: Optional[ctypes.CDLL] = None) -> np.ndarray:
    """Dense fp16 R x K from the compressed arrays (pruned positions +0.0)."""
    L = L or lib()
    values = np.ascontiguousarray(values, dtype=np.uint16)
    meta = np.ascontiguousarray(meta, dtype=np.uint8)
    colidx = np.ascontiguousarray(colidx, dtype=np.uint8)
    W = np.empty((R, K), dtype=np.uint16)
    rc = L.oracle_decompress(_ptr(values), _ptr(meta), _ptr(colidx), R, K, V, M, _ptr(W), K)
    if rc != OK:
        raise OracleError(rc, "decompress")
    return W.view(np.float16)


def spmm(values: np.ndarray, meta: np.ndarray, colidx: np.ndarray, R: int, K: int, V: int, M: int,
         B: np.ndarray, rows: Optional[Sequence[int]] = None, acc: str = "f32",
         L: Optional[ctypes.CDLL] = None) -> np.ndarray:
    """C[rows, :] = A_vnm[rows, :] . B, accumulated in ``acc`` ("f32" or "f64").

    B is fp16 K x N. Returns float32 (acc="f32") or float64 (acc="f64") of
    shape [len(rows), N] (all R rows when ``rows`` is None).
    """
    L = L or lib()
    values = np.ascontiguousarray(values, dtype=np.uint16)
    meta = np.ascontiguousarray(meta, dtype=np.uint8)
    colidx = np.ascontiguousarray(colidx, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.float16)
    assert B.shape[0] == K
    N = B.shape[1]
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_rows = R if rows_arr is None else rows_arr.size
    dt = np.float32 if acc == "f32" else np.float64
    C = np.zeros((n_rows, N), dtype=dt)
    fn = L.oracle_spmm_f32 if acc == "f32" else L.oracle_spmm_f64
    rc = fn(_ptr(values), _ptr(meta), _ptr(colidx), R, K, V, M, _ptr(B), N, N, _ptr(rows_arr),
            n_rows, _ptr(C))
    if rc != OK:
        raise OracleError(rc, "spmm")
    return C
