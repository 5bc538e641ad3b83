"""vnm_gemm_compress on the GPU against the CPU oracle: the fused dense GEMM
W = X . Y^T whose epilogue prunes and encodes W (DFSS "Dynamic N:M
fine-grained structured sparse attention", sections 4.2-4.3, with the V:N:M
rule of VENOM section 3).

The pruning decisions depend on W's fp16 bits, which the GPU (fp32
accumulation) and the oracle (fp64) may round differently when W is not
exact. So: with inputs whose products and sums are exact in fp32 (small
multiples of 1/4) both sides hold the same W and every array must match bit
for bit; with N(0, 1) inputs the W the GPU also writes must lie within the
fp32 summation bound of the oracle's fp64 product, and the arrays must equal
the oracle's compress of that W."""
import numpy as np
import pytest
import torch

import oracle
from structured_sparse_matmul_gb300 import inputs, vnm

pytestmark = pytest.mark.gpu

from gpu_util import device  # noqa: E402


def _exact_operands(R, K, D, seed):
    rng = np.random.default_rng(seed)
    X = (rng.integers(-3, 4, (R, D)) * 0.25).astype(np.float16)
    Y = (rng.integers(-3, 4, (K, D)) * 0.25).astype(np.float16)
    return X, Y


def _run(X, Y, V, M, want_w=True):
    R, K = X.shape[0], Y.shape[0]
    A = vnm.vnm_matrix_alloc(R, K, V, M, device())
    Wd = torch.full((R, K), float("nan"), dtype=torch.float16, device=device()) if want_w else None
    vnm.vnm_gemm_compress(A, torch.from_numpy(X).to(device()), torch.from_numpy(Y).to(device()), Wd)
    st = vnm.vnm_get_status(A)
    arrays = (A.values.cpu().numpy().view(np.uint16), A.meta.cpu().numpy(), A.colidx.cpu().numpy())
    return st, arrays, (Wd.cpu().numpy() if want_w else None)


def _assert_arrays(got, want, what):
    for name, a, b in zip(("values", "meta", "column-loc"), got, want):
        assert np.array_equal(a, b), f"{what}: {name} differ at {np.argwhere(a != b)[:4].tolist()}"


SHAPES = [
    # R, K, D, V, M
    (128, 128, 64, 16, 8),      # one tile, one stage
    (256, 384, 192, 64, 8),     # several tiles and stages
    (384, 512, 136, 128, 16),   # D % 64 != 0 (zero-filled tail)
    (160, 200, 72, 16, 8),      # ragged rows and columns (R % 128, K % 128 != 0)
    (96, 136, 40, 32, 8),       # an odd number of blocks in the last column tile
    (128, 256, 64, 1, 4),       # plain 2:4 per row (V = 1)
    (256, 256, 128, 8, 32),
    (128, 320, 96, 4, 64),
    (512, 1024, 64, 16, 4),     # the attention-score shape class: a short D
]


@pytest.mark.parametrize("R,K,D,V,M", SHAPES)
def test_exact_inputs_bit_exact(R, K, D, V, M):
    X, Y = _exact_operands(R, K, D, seed=R + K + D)
    st, got, W = _run(X, Y, V, M)
    assert st == vnm.VNM_OK, vnm.status_string(st)
    Wo, want = oracle.gemm_compress(X, Y, V, M)
    assert W.tobytes() == Wo.tobytes(), "W differs"
    _assert_arrays(got, want, f"{R}x{K}x{D} {V}:2:{M}")
    # the same arrays as vnm_compress of W
    A2 = vnm.vnm_matrix_alloc(R, K, V, M, device())
    vnm.vnm_compress(A2, torch.from_numpy(Wo).to(device()))
    assert vnm.vnm_get_status(A2) == vnm.VNM_OK
    _assert_arrays(got, (A2.values.cpu().numpy().view(np.uint16), A2.meta.cpu().numpy(), A2.colidx.cpu().numpy()),
                   "against vnm_compress")


@pytest.mark.parametrize("R,K,D,V,M", [(256, 384, 256, 64, 8), (160, 208, 72, 16, 16), (384, 256, 1000, 128, 8)])
def test_normal_inputs(R, K, D, V, M):
    X = inputs.normal_f16((R, D), 71, 0, 1.0)
    Y = inputs.normal_f16((K, D), 71, 1, 1.0)
    st, got, W = _run(X, Y, V, M)
    assert st == vnm.VNM_OK, vnm.status_string(st)
    ref = X.astype(np.float64) @ Y.astype(np.float64).T
    mag = np.abs(X.astype(np.float64)) @ np.abs(Y.astype(np.float64)).T
    # fp32 accumulation (D - 1 roundings of the running sum, bound 2^-22 per term)
    # then one rounding to fp16 (half an ulp: 2^-11 relative)
    bound = D * 2.0 ** -22 * mag + 2.0 ** -11 * np.abs(ref) + 2.0 ** -24
    err = np.abs(W.astype(np.float64) - ref)
    assert (err <= bound).all(), f"W beyond the bound at {np.argwhere(err > bound)[:4].tolist()}"
    _assert_arrays(got, oracle.compress(W, V, M), f"normal {R}x{K}x{D}")


def test_w_out_optional():
    R, K, D, V, M = 256, 256, 128, 16, 8
    X, Y = _exact_operands(R, K, D, seed=5)
    st, got, _ = _run(X, Y, V, M, want_w=False)
    assert st == vnm.VNM_OK
    _assert_arrays(got, oracle.gemm_compress(X, Y, V, M)[1], "without W_out")


def test_zero_depth():
    """D = 0: W = 0, compressed like an all-zero matrix."""
    R, K, V, M = 128, 128, 16, 8
    st, got, W = _run(np.zeros((R, 0), np.float16), np.zeros((K, 0), np.float16), V, M)
    assert st == vnm.VNM_OK
    assert not W.astype(np.float64).any()
    _assert_arrays(got, oracle.compress(np.zeros((R, K), np.float16), V, M), "D = 0")


def test_overflow_reports_nonfinite():
    R, K, D, V, M = 128, 128, 64, 16, 8
    X = np.full((R, D), 8.0, np.float16)
    Y = np.full((K, D), 256.0, np.float16)  # 64 * 8 * 256 = 131072 > 65504
    st, _, _ = _run(X, Y, V, M)
    assert st == vnm.VNM_ERR_NONFINITE


@pytest.mark.parametrize("V,M", [(256, 8), (16, 128), (48, 8)])
def test_unserved_shapes(V, M):
    A = vnm.vnm_matrix_alloc(2 * V if V > 16 else 256, 256, V, M, device())
    X = torch.zeros((A.R, 64), dtype=torch.float16, device=device())
    Y = torch.zeros((A.K, 64), dtype=torch.float16, device=device())
    with pytest.raises(vnm.VnmError) as e:
        vnm.vnm_gemm_compress(A, X, Y)
    assert e.value.code == vnm.VNM_ERR_UNSUPPORTED


def test_strided_operands():
    R, K, D, V, M = 256, 256, 96, 64, 8
    X, Y = _exact_operands(R, K, D, seed=9)
    Xb = torch.zeros((R, 104), dtype=torch.float16, device=device())
    Yb = torch.zeros((K, 128), dtype=torch.float16, device=device())
    Xb[:, :D] = torch.from_numpy(X).to(device())
    Yb[:, :D] = torch.from_numpy(Y).to(device())
    Wb = torch.full((R, K + 8), float("nan"), dtype=torch.float16, device=device())
    A = vnm.vnm_matrix_alloc(R, K, V, M, device())
    vnm.vnm_gemm_compress(A, Xb[:, :D], Yb[:, :D], Wb[:, :K])
    assert vnm.vnm_get_status(A) == vnm.VNM_OK
    Wo, want = oracle.gemm_compress(X, Y, V, M)
    assert Wb[:, :K].cpu().numpy().tobytes() == Wo.tobytes()
    assert torch.isnan(Wb[:, K:]).all()
    _assert_arrays((A.values.cpu().numpy().view(np.uint16), A.meta.cpu().numpy(), A.colidx.cpu().numpy()), want,
                   "strided")
