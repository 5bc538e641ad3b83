"""The C ABI without a GPU: libvnm loads, exports every function include/*.h
declares, and its host-only calls (sizes, status strings, argument checks
that fail before any CUDA call) behave as documented."""
import ctypes
import os
import re
import shutil

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


def _declared_functions():
    names = set()
    for header in HEADERS:
        text = open(header).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"^[A-Za-z_][\w \*]*?\b(vnm_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def libvnm():
    from structured_sparse_matmul_gb300 import build, vnm
    if not build.up_to_date():
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available and libvnm not built")
        build.build()
    return vnm.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("vnm_sizes", "vnm_matrix_create", "vnm_matrix_destroy", "vnm_compress", "vnm_decompress",
                 "vnm_spmm", "vnm_spmm_workspace_size", "vnm_spmm_plan_query", "vnm_spmm_with_plan",
                 "vnm_get_status", "vnm_status_string", "vnm_version", "vnm_gemm_compress", "vnm_energy", "vnm_energy_workspace_size", "vnm_linear",
                 "vnm_linear_workspace_size", "vnm_bitmap_sizes", "vnm_bitmap_encode", "vnm_bitmap_spmm",
                 "vnm_bitmap_spmm_workspace_size"):
        assert want in names, want


def test_every_declared_symbol_is_exported(libvnm):
    for name in _declared_functions():
        assert hasattr(libvnm, name), f"libvnm does not export {name}"
        assert ctypes.cast(getattr(libvnm, name), ctypes.c_void_p).value


def test_version_and_status_strings(libvnm):
    from structured_sparse_matmul_gb300 import vnm
    assert vnm.vnm_version() == 100
    for code, name in ((0, "VNM_OK"), (1, "VNM_ERR_INVALID_ARG"), (2, "VNM_ERR_UNSUPPORTED"), (3, "VNM_ERR_CUDA"),
                       (4, "VNM_ERR_NONFINITE"), (5, "VNM_ERR_TIMEOUT"), (6, "VNM_ERR_INTERNAL")):
        assert vnm.status_string(code) == name


@pytest.mark.parametrize("R,K,V,M", [(2, 8, 1, 4), (512, 1024, 1, 4), (256, 256, 16, 4), (4096, 4096, 64, 8),
                                     (1024, 4096, 128, 16), (49152, 12288, 128, 32), (12, 60, 4, 5),
                                     (8, 512, 8, 256), (0, 64, 16, 8), (16, 0, 16, 8)])
def test_sizes_match_oracle(libvnm, R, K, V, M):
    from structured_sparse_matmul_gb300 import vnm
    vb, mb, cb = vnm.vnm_sizes(R, K, V, M)
    nv, nm, nc = oracle.sizes(R, K, V, M)
    assert (vb, mb, cb) == (2 * nv, nm, nc)


@pytest.mark.parametrize("R,K,V,M", [(10, 16, 4, 8), (8, 18, 4, 8), (8, 16, 4, 3), (8, 512, 4, 257),
                                     (8192, 16, 8192, 8), (8, 16, 0, 8), (-4, 16, 4, 8)])
def test_invalid_shapes_rejected(libvnm, R, K, V, M):
    from structured_sparse_matmul_gb300 import vnm
    with pytest.raises(vnm.VnmError) as e:
        vnm.vnm_sizes(R, K, V, M)
    assert e.value.code == vnm.VNM_ERR_INVALID_ARG
    # the same check runs first in vnm_matrix_create (no CUDA call is made)
    h = ctypes.c_void_p()
    assert libvnm.vnm_matrix_create(R, K, V, M, None, None, None, ctypes.byref(h)) == vnm.VNM_ERR_INVALID_ARG
    assert not h.value


def test_handle_checks_without_gpu(libvnm):
    from structured_sparse_matmul_gb300 import vnm
    # NULL handles and out-pointers are argument errors, found before any CUDA call
    assert libvnm.vnm_matrix_create(16, 64, 16, 8, None, None, None, None) == vnm.VNM_ERR_INVALID_ARG
    assert libvnm.vnm_compress(None, None, 64, None) == vnm.VNM_ERR_INVALID_ARG
    assert libvnm.vnm_decompress(None, None, 64, None) == vnm.VNM_ERR_INVALID_ARG
    assert libvnm.vnm_spmm(None, None, 8, 8, None, 8, 0, None, 0, None) == vnm.VNM_ERR_INVALID_ARG
    assert libvnm.vnm_get_status(None, None) == vnm.VNM_ERR_INVALID_ARG
    assert libvnm.vnm_matrix_destroy(None) == vnm.VNM_OK
    b = ctypes.c_size_t()
    assert libvnm.vnm_spmm_workspace_size(None, 8, ctypes.byref(b)) == vnm.VNM_ERR_INVALID_ARG
    # arrays must be 16-byte aligned device allocations
    assert libvnm.vnm_matrix_create(16, 64, 16, 8, 8, 16, 32, ctypes.byref(ctypes.c_void_p())) == \
        vnm.VNM_ERR_INVALID_ARG


@pytest.mark.parametrize("R,K", [(64, 1), (128, 40), (4096, 11008), (0, 7), (64, 0)])
def test_bitmap_sizes_match_oracle(libvnm, R, K):
    """vnm_bitmap_sizes (host only) against the oracle's arrays: one 8-byte
    bitmap and one 4-byte offset per 64-row column tile, R/64 + 1 bases, and
    at most R*K fp16 values (every tile full)."""
    rng = np.random.default_rng(R + K)
    W = (rng.standard_normal((R, K)) * (rng.random((R, K)) > 0.5)).astype(np.float16)
    bm, off, bases, _ = oracle.bitmap_encode(W)
    out = [ctypes.c_size_t() for _ in range(4)]
    assert libvnm.vnm_bitmap_sizes(R, K, *[ctypes.byref(o) for o in out]) == 0
    assert [o.value for o in out] == [bm.nbytes, off.nbytes, bases.nbytes, 2 * R * K]


@pytest.mark.parametrize("R,K", [(100, 8), (-64, 8), (64, -1), (64, 1 << 27)])
def test_bitmap_sizes_rejected(libvnm, R, K):
    from structured_sparse_matmul_gb300 import vnm
    assert libvnm.vnm_bitmap_sizes(R, K, None, None, None, None) == vnm.VNM_ERR_INVALID_ARG


def test_product_path_does_not_import_the_oracle():
    """The package never imports, loads or names the oracle."""
    pkg = os.path.join(ROOT, "structured_sparse_matmul_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "liboracle" not in text and "from oracle" not in text, f
