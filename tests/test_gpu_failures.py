"""Failure handling on the GPU without a fault: a pipeline stage whose loads
are never issued makes the tensor-core kernel's bounded waits run out; the
kernel must record VNM_ERR_TIMEOUT, free what it holds and leave the device
usable. Out-of-bounds writes are checked with canary-padded outputs."""
import numpy as np
import pytest
import torch

from structured_sparse_matmul_gb300 import inputs, vnm

pytestmark = pytest.mark.gpu

from gpu_util import check_close, device, gpu_compress, sample_rows  # noqa: E402
import oracle  # noqa: E402


def _product(R, K, N, V, M, seed):
    W = inputs.normal_f16((R, K), seed, 0, 0.02)
    B = inputs.normal_f16((K, N), seed, 1, 1.0)
    A, st = gpu_compress(W, V, M)
    assert st == vnm.VNM_OK
    values, meta, colidx = oracle.compress(W, V, M)
    return A, B, (values, meta, colidx)


# shapes with enough tiles that K is not split, so the first CTA runs every
# stage of its tiles (persistent schedule: CTA 0 takes tiles 0, 152, ...)
@pytest.mark.parametrize("R,K,N,V,M,skip", [(2048, 2048, 1024, 128, 4, 3),    # B by TMA
                                            (2048, 2048, 1024, 64, 16, 2),    # B gathered
                                            (4096, 2048, 2048, 64, 16, 9),    # third tile of four (4 stages each)
                                            (16384, 2048, 256, 32, 8, 2),     # A re-encoded as 2:4 on chip (lift)
                                            (20480, 2048, 256, 32, 8, 20),    # second tile of two (16 stages each)
                                            (4096, 2048, 2048, 64, 8, 3)])    # A written out as 2:4 first
def test_bounded_wait_reports_timeout_and_device_stays_usable(R, K, N, V, M, skip):
    A, B, comp = _product(R, K, N, V, M, seed=80 + M)
    Bd = torch.from_numpy(B).to(device())
    C = torch.empty((R, N), dtype=torch.float16, device=device())
    plan = vnm.vnm_spmm_plan_query(A, Bd)
    assert plan.path == vnm.VNM_PATH_TC and plan.splits == 1, plan.as_dict()
    vnm.vnm_testing_spmm_skip_stage(A, Bd, C, skip, workspace=vnm.workspace_for(A, N))
    assert vnm.vnm_get_status(A) == vnm.VNM_ERR_TIMEOUT
    # the next products on the same device and matrix are correct
    for _ in range(2):
        vnm.vnm_spmm(A, Bd, C, workspace=vnm.workspace_for(A, N))
        assert vnm.vnm_get_status(A) == vnm.VNM_OK
    rows = sample_rows(R, V, 24)
    ref = oracle.spmm(*comp, R, K, V, M, B, rows=rows)
    check_close(C.float().cpu().numpy()[rows], ref, "after the timeout")


def test_skip_stage_needs_the_tensor_core_path():
    A, B, _ = _product(64, 512, 4, 16, 4, seed=90)
    Bd = torch.from_numpy(B).to(device())
    C = torch.empty((64, 4), dtype=torch.float16, device=device())
    with pytest.raises(vnm.VnmError) as e:
        vnm.vnm_testing_spmm_skip_stage(A, Bd, C, 0)
    assert e.value.code == vnm.VNM_ERR_UNSUPPORTED


@pytest.mark.parametrize("R,K,N,V,M", [(272, 256, 72, 16, 4),     # tensor cores, ragged rows and columns
                                       (256, 1024, 296, 64, 16),  # gather, ragged against the tile
                                       (144, 1024, 296, 16, 8),   # lift, ragged rows and columns
                                       (192, 768, 5, 64, 8),      # streaming small N
                                       (96, 600, 33, 8, 5)])      # CUDA-core rows
def test_outputs_stay_inside_c(R, K, N, V, M):
    """C sits inside a larger NaN-filled buffer (padding rows and columns on
    every side); after the product the padding must still be NaN."""
    A, B, comp = _product(R, K, N, V, M, seed=95)
    Bd = torch.from_numpy(B).to(device())
    pad = 8
    for c_dtype in (torch.float16, torch.float32):
        big = torch.full((R + 2 * pad, N + 2 * pad + 3), float("nan"), dtype=c_dtype, device=device())
        C = big[pad:pad + R, pad:pad + N]
        vnm.vnm_spmm(A, Bd, C, workspace=vnm.workspace_for(A, N))
        assert vnm.vnm_get_status(A) == vnm.VNM_OK
        host = big.float().cpu().numpy()
        inside = np.zeros(host.shape, dtype=bool)
        inside[pad:pad + R, pad:pad + N] = True
        assert np.isnan(host[~inside]).all(), "a write landed outside C"
        check_close(host[inside].reshape(R, N), oracle.spmm(*comp, R, K, V, M, B), f"{R}x{K}x{N}")
