"""vnm_compress / vnm_decompress on the GPU against the CPU oracle: bit-exact
values, m-indices and column-loc (VENOM section 3, Figures 2-3)."""
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import read_fixture
from structured_sparse_matmul_gb300 import inputs, vnm, workloads

pytestmark = pytest.mark.gpu

from gpu_util import assert_compress_bitexact, device, gpu_compress  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_worked_example():
    fx = read_fixture(os.path.join(GOLDEN, "worked_2x8.txt"))
    W = np.array([[float(x) for x in fx["dense_row0"].split()], [float(x) for x in fx["dense_row1"].split()]],
                 dtype=np.float16)
    for V in (1, 2):
        A, st = gpu_compress(W, V, 4)
        assert st == vnm.VNM_OK
        assert_compress_bitexact(A, W, V, 4)
        got = A.values.cpu().numpy()
        for r in range(2):
            want = np.array([float(x) for x in fx[f"values_row{r}"].split()], dtype=np.float16)
            assert got[r].tobytes() == want.tobytes()
        assert A.meta.cpu().numpy()[:, 0].tolist() == [0xD8, 0xC9]


SHAPES = [
    (256, 256, 16, 4),      # plain 2:4 with V = 16
    (384, 1024, 128, 8),
    (128, 4096, 128, 16),
    (64, 8192, 64, 32),
    (32, 600, 8, 5),        # odd M, K not a multiple of the tile
    (24, 56, 8, 7),
    (16, 1000, 16, 10),
    (128, 512, 128, 256),   # V x 2M above the tile budget: block-pair kernel
    (4, 4096, 1, 4),
    (8, 64, 8, 64),
    (256, 4096, 256, 8),
    (64, 296, 16, 8),       # M in {8, 16, 32} with an odd number of blocks per row
    (32, 80, 4, 16),
    (36, 96, 12, 32),
    (384, 640, 192, 16),    # V above 128: the two-pass (re-read) variant
]


@pytest.mark.parametrize("R,K,V,M", SHAPES)
def test_random_shapes(R, K, V, M):
    W = inputs.normal_f16((R, K), 11, R + K + M, 0.02)
    A, st = gpu_compress(W, V, M)
    assert st == vnm.VNM_OK
    assert_compress_bitexact(A, W, V, M)


@pytest.mark.parametrize("R,K,V,M,ld", [(64, 256, 16, 8, 264), (32, 600, 8, 5, 640), (128, 512, 128, 256, 520)])
def test_padded_rows(R, K, V, M, ld):
    W = inputs.normal_f16((R, K), 12, K, 0.02)
    A, st = gpu_compress(W, V, M, ld=ld)
    assert st == vnm.VNM_OK
    assert_compress_bitexact(A, W, V, M)


@pytest.mark.parametrize("R,K,V,M", [(32, 96, 4, 6), (64, 512, 16, 8), (16, 256, 8, 16), (16, 768, 16, 12),
                                     (64, 1056, 32, 32), (128, 72, 128, 8), (256, 96, 256, 16)])
def test_tie_heavy(R, K, V, M):
    W = inputs.choice_f16((R, K), 13, M, [0, 0.5, -0.5, 1, -1, 0.0])
    A, st = gpu_compress(W, V, M)
    assert st == vnm.VNM_OK
    assert_compress_bitexact(A, W, V, M)


def test_subnormals_and_signed_zeros():
    tiny = [1023 * 2.0 ** -24, -1023 * 2.0 ** -24, 1.5 * 2.0 ** -14, 2.0 ** -13, -(2.0 ** -13), 3 * 2.0 ** -24,
            0.0, -0.0]
    W = inputs.choice_f16((64, 512), 14, 0, tiny)
    for V, M in ((16, 8), (64, 4), (8, 32)):
        A, st = gpu_compress(W, V, M)
        assert st == vnm.VNM_OK
        assert_compress_bitexact(A, W, V, M)


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_nonfinite_reported(bad):
    for (R, K, V, M) in ((64, 256, 16, 8), (128, 512, 128, 256), (256, 512, 128, 32), (256, 128, 256, 8)):
        W = inputs.normal_f16((R, K), 15, 0, 0.02)
        W[R // 2, K - 3] = bad
        A, st = gpu_compress(W, V, M)
        assert st == vnm.VNM_ERR_NONFINITE
        # the status word is cleared once read
        assert vnm.vnm_get_status(A) == vnm.VNM_OK


@pytest.mark.parametrize("R,K,V,M", [(256, 256, 16, 4), (128, 1000, 16, 10), (64, 8192, 64, 32), (24, 56, 8, 7)])
def test_decompress_matches_oracle(R, K, V, M):
    W = inputs.normal_f16((R, K), 16, K, 0.02)
    A, st = gpu_compress(W, V, M)
    values, meta, colidx = assert_compress_bitexact(A, W, V, M)
    D = torch.empty((R, K), dtype=torch.float16, device=device())
    vnm.vnm_decompress(A, D)
    assert vnm.vnm_get_status(A) == vnm.VNM_OK
    want = oracle.decompress(values, meta, colidx, R, K, V, M)
    assert np.array_equal(D.cpu().numpy().view(np.uint16), want.view(np.uint16))


def test_empty():
    for (R, K) in ((0, 64), (16, 0)):
        A = vnm.vnm_matrix_alloc(R, K, 16, 8, device())
        vnm.vnm_compress(A, torch.zeros((R, K), dtype=torch.float16, device=device()))
        assert vnm.vnm_get_status(A) == vnm.VNM_OK


@pytest.mark.parametrize("case", [c for w in (1, 2, 3, 4) for c in workloads.workload_cases(w)
                                  if c.N in (1, 2048, 8192, 64)], ids=lambda c: c.name)
def test_workload_shapes(case):
    W = inputs.normal_f16((case.R, case.K), case.seed, case.a_stream, workloads.A_SIGMA)
    A, st = gpu_compress(W, case.V, case.M)
    assert st == vnm.VNM_OK
    assert_compress_bitexact(A, W, case.V, case.M)
