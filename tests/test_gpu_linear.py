"""vnm_linear on the GPU against the CPU oracle: the Linear-layer form
Y = act(X . A^T + bias) ("VENOM" section 7's transformer layers apply a
pruned weight to token activations), i.e. the SpMM C = A . X^T written
transposed, with the bias and activation applied as C is written. Every
path: the tensor cores reading X in place (2:4, and M = 8 re-encoded), the
gather through a transposed copy of X, split K, the streaming small-T
kernel and the CUDA-core kernel reading X with strides. Tolerance as for the
SpMM: |Y - Y_oracle| <= 1e-2 * (1 + |Y_oracle|)."""
import numpy as np
import pytest
import torch

import oracle
from structured_sparse_matmul_gb300 import inputs, vnm

pytestmark = pytest.mark.gpu

from gpu_util import assert_compress_bitexact, check_close, device, gpu_compress  # noqa: E402

ACTS = [(vnm.VNM_ACT_NONE, oracle.ACT_NONE), (vnm.VNM_ACT_RELU, oracle.ACT_RELU), (vnm.VNM_ACT_GELU, oracle.ACT_GELU)]


def _layer(R, K, V, M, seed):
    W = inputs.normal_f16((R, K), seed, 0, 0.02)
    A, st = gpu_compress(W, V, M)
    assert st == vnm.VNM_OK
    comp = assert_compress_bitexact(A, W, V, M)
    bias = inputs.normal_f16((1, R), seed, 2, 0.5)[0]
    return A, comp, bias


def _run(A, X, bias, act, y_dtype=torch.float16, ld_y=None, x_offset=0, ld_x=None):
    T, K = X.shape
    if ld_x is None and x_offset == 0:
        Xd = torch.from_numpy(X).to(device())
    else:
        ld = ld_x or K
        buf = torch.zeros(x_offset + T * ld, dtype=torch.float16, device=device())
        Xd = buf[x_offset:].view(T, ld)[:, :K]
        Xd.copy_(torch.from_numpy(X).to(device()))
    ldy = ld_y or A.R
    Ybuf = torch.full((T, ldy), float("nan"), dtype=y_dtype, device=device())
    Y = Ybuf[:, :A.R]
    bd = torch.from_numpy(bias).to(device()) if bias is not None else None
    vnm.vnm_linear(A, Xd, Y, bd, act)
    st = vnm.vnm_get_status(A)
    assert st == vnm.VNM_OK, vnm.status_string(st)
    if ldy > A.R:
        assert torch.isnan(Ybuf[:, A.R:]).all(), "a write landed outside Y"
    return Y.float().cpu().numpy()


@pytest.mark.parametrize("R,K,V,M,T", [(384, 1024, 64, 4, 300),    # 2:4: X read in place (K-major TMA)
                                       (256, 1024, 64, 8, 520),    # M = 8 re-encoded: X in place
                                       (256, 2048, 128, 16, 200),  # gather: X transposed first
                                       (512, 1024, 16, 8, 40)])    # lift with V = 16, narrow tile
@pytest.mark.parametrize("act", ACTS, ids=["none", "relu", "gelu"])
def test_tensor_core_paths(R, K, V, M, T, act):
    A, comp, bias = _layer(R, K, V, M, seed=R + T)
    X = inputs.normal_f16((T, K), R + T, 1, 1.0)
    for y_dtype in (torch.float16, torch.float32):
        got = _run(A, X, bias, act[0], y_dtype)
        check_close(got, oracle.linear(*comp, R, K, V, M, X, bias, act[1]), f"linear {R}x{K} T={T} {V}:2:{M}")


@pytest.mark.parametrize("R,K,V,M,T", [(128, 2048, 64, 4, 64),     # one tile: split K, reduction applies the epilogue
                                       (1024, 2048, 64, 8, 5),     # T <= 8: streaming kernel, X with strides
                                       (96, 600, 8, 5, 24),        # CUDA-core kernel, X with strides
                                       (256, 1024, 128, 4, 33)])   # ragged T against the 16-column tile
def test_other_paths(R, K, V, M, T):
    A, comp, bias = _layer(R, K, V, M, seed=R + T + 7)
    X = inputs.normal_f16((T, K), R + T, 1, 1.0)
    for act in ACTS:
        got = _run(A, X, bias, act[0], torch.float32, ld_y=R + 8)
        check_close(got, oracle.linear(*comp, R, K, V, M, X, bias, act[1]), f"linear {R}x{K} T={T} {V}:2:{M}")


def test_unaligned_x_and_no_bias():
    R, K, V, M, T = 256, 1024, 64, 4, 96
    A, comp, _ = _layer(R, K, V, M, seed=91)
    X = inputs.normal_f16((T, K), 91, 1, 1.0)
    got = _run(A, X, None, vnm.VNM_ACT_NONE, x_offset=1, ld_x=K + 3)  # rows not 16-byte aligned: transposed copy
    check_close(got, oracle.linear(*comp, R, K, V, M, X, None), "unaligned X")


def test_zero_depth_gives_activation_of_bias():
    R, K, V, M, T = 128, 0, 16, 8, 12
    A = vnm.vnm_matrix_alloc(R, K, V, M, device())
    bias = inputs.normal_f16((1, R), 92, 2, 1.0)[0]
    for act in ACTS:
        got = _run(A, np.zeros((T, 0), np.float16), bias, act[0], torch.float32)
        want = oracle.linear(np.zeros((R, 0), np.uint16), np.zeros((R, 0), np.uint8), np.zeros((R // V, 0, 4), np.uint8),
                             R, K, V, M, np.zeros((T, 0), np.float16), bias, act[1])
        check_close(got, want, "K = 0")
