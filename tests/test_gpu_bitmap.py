"""The bitmap format for unstructured sparsity on the GPU ("Coruscant",
section 3.1, Figure 7) and its small-N SpMM (section 3.2) against the CPU
oracle: the encoded arrays bit for bit, the product within
1e-2 * (1 + |C_oracle|) and the fp32 summation bound."""
import numpy as np
import pytest
import torch

import oracle
from structured_sparse_matmul_gb300 import inputs, vnm

pytestmark = pytest.mark.gpu

from gpu_util import TOL, check_close, device, to_dev  # noqa: E402


def _sparse(R, K, sparsity, seed):
    """N(0, 0.02) weights with the smallest |w| fraction `sparsity` zeroed (magnitude pruning)."""
    W = inputs.normal_f16((R, K), seed, 0, 0.02)
    mags = np.abs(W.astype(np.float64)).ravel()
    cut = np.sort(mags)[int(sparsity * mags.size)] if sparsity > 0 else -1.0
    W[np.abs(W.astype(np.float64)) < cut] = 0
    return W


def _enc(W, ld=None):
    A = vnm.bitmap_encode(to_dev(W, ld))
    got = (A.bitmaps.cpu().numpy().view(np.uint64).reshape(A.R // 64, A.K),
           A.offsets.cpu().numpy().view(np.uint32).reshape(A.R // 64, A.K), A.bases.cpu().numpy(),
           A.values.cpu().numpy().view(np.uint16))
    return A, got


@pytest.mark.parametrize("R,K,sparsity", [(64, 40, 0.5), (256, 1000, 0.3), (512, 777, 0.7), (128, 256, 0.0),
                                          (192, 96, 0.95)])
def test_encode_bit_exact(R, K, sparsity):
    W = _sparse(R, K, sparsity, seed=R + K)
    W[1, 2] = -0.0
    A, got = _enc(W, ld=K + 8)
    want = oracle.bitmap_encode(W)
    for name, a, b in zip(("bitmaps", "offsets", "bases", "values"), got, want):
        assert np.array_equal(a, b), f"{name} differ at {np.argwhere(a != b)[:4].tolist()}"


@pytest.mark.parametrize("R,K,N,sparsity", [(4096, 4096, 1, 0.5), (1024, 2048, 8, 0.3), (512, 1000, 16, 0.7),
                                            (256, 640, 32, 0.5), (128, 300, 40, 0.6), (64, 64, 3, 0.5),
                                            (256, 1100, 2, 0.0), (128, 700, 5, 0.999)])
def test_spmm(R, K, N, sparsity):
    W = _sparse(R, K, sparsity, seed=R + N)
    B = inputs.normal_f16((K, N), R + N, 1, 1.0)
    A, enc = _enc(W)
    ref = oracle.bitmap_spmm(*enc, R, K, B)
    mag = np.abs(W.astype(np.float64)) @ np.abs(B.astype(np.float64))
    Bd = to_dev(B)
    for c_dtype in (torch.float16, torch.float32):
        for ws in (None, True):
            C = torch.empty((R, N), dtype=c_dtype, device=device())
            w = None
            if ws:
                n = vnm.bitmap_spmm_workspace_size(R, K, N)
                w = torch.empty(max(1, n // 4), dtype=torch.float32, device=device())
            vnm.bitmap_spmm(A, Bd, C, workspace=w)
            got = C.float().cpu().numpy()
            check_close(got, ref, f"bitmap {R}x{K}x{N}")
            if c_dtype == torch.float32:
                err = np.abs(got.astype(np.float64) - ref)
                assert (err <= K * 2.0 ** -22 * mag + 1e-30).all(), "beyond the fp32 summation bound"


def test_capacity_and_shape_checks():
    W = _sparse(128, 64, 0.5, seed=3)
    Wd = to_dev(W)
    lib = vnm.lib()
    import ctypes
    bm = torch.empty(2 * 64, dtype=torch.int64, device=device())
    off = torch.empty(2 * 64, dtype=torch.int32, device=device())
    bases = torch.empty(3, dtype=torch.int64, device=device())
    vals = torch.empty(8, dtype=torch.float16, device=device())
    need = ctypes.c_int64(0)
    code = lib.vnm_bitmap_encode(Wd.data_ptr(), 64, 128, 64, bm.data_ptr(), off.data_ptr(), bases.data_ptr(),
                                 vals.data_ptr(), 8, ctypes.byref(need), None)
    assert code == vnm.VNM_ERR_INVALID_ARG and need.value == oracle.bitmap_encode(W)[2][-1]
    assert lib.vnm_bitmap_sizes(100, 64, None, None, None, None) == vnm.VNM_ERR_INVALID_ARG  # R % 64 != 0


def test_spmm_all_zero():
    """No value at all (every bitmap zero, every run empty): C = 0."""
    R, K, N = 128, 520, 4
    A, _ = _enc(np.zeros((R, K), np.float16))
    assert A.values.numel() == 0 or not A.values.any()
    B = to_dev(inputs.normal_f16((K, N), 9, 1, 1.0))
    for ws in (None, True):
        C = torch.full((R, N), 7.0, dtype=torch.float32, device=device())
        w = torch.empty(max(1, vnm.bitmap_spmm_workspace_size(R, K, N) // 4), dtype=torch.float32,
                        device=device()) if ws else None
        vnm.bitmap_spmm(A, B, C, workspace=w)
        assert (C == 0).all()
