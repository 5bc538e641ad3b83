"""vnm_spmm_noalloc: the SpMM entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc where they need the product
(their device memory is held in full by another caching allocator, or the
path must not take the device synchronisation of cudaMalloc/cudaFree): the
split-K scratch is a static device array inside libvnm. These tests call it
through the C ABI (ctypes on libvnm) and compare it with the CPU oracle and
with vnm_spmm (given a torch-allocated workspace), within the parity
tolerance, on two calls in a row (the second call finds the first call's
scratch contents).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from structured_sparse_matmul_gb300 import inputs, vnm

pytestmark = pytest.mark.gpu

TOL = 1e-2  # the parity tolerance of the other GPU tests: |x - y| <= TOL * (1 + |y|)


def _close(got, ref):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    return bool((np.abs(got - ref) <= TOL * (1.0 + np.abs(ref))).all())


def _compressed(R, K, V, M, seed):
    """The GPU's compressed matrix and the oracle's arrays of the same W."""
    dev = torch.device("cuda", 0)
    W_h = inputs.normal_f16((R, K), seed, 0, 0.02)
    A = vnm.vnm_matrix_alloc(R, K, V, M, dev)
    vnm.vnm_compress(A, torch.from_numpy(W_h).to(dev))
    assert vnm.vnm_get_status(A) == vnm.VNM_OK
    return A, oracle.compress(W_h, V, M)


def _noalloc_call(A, B, C, status=None):
    """One call of vnm_spmm_noalloc through the C ABI."""
    L = vnm.lib()
    N = int(B.shape[1])
    rc = L.vnm_spmm_noalloc(A.R, A.K, A.V, A.M, A.values.data_ptr(), A.meta.data_ptr(), A.colidx.data_ptr(),
                            B.data_ptr(), B.stride(0), N, C.data_ptr(), C.stride(0),
                            vnm.VNM_F32 if C.dtype == torch.float32 else vnm.VNM_F16,
                            None if status is None else status.data_ptr(),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("R,K,N,V,M", [(4096, 4096, 32, 64, 4), (4096, 4096, 16, 64, 8), (1024, 2048, 40, 128, 16),
                                       (128, 4096, 256, 128, 4)])
def test_matches_vnm_spmm_on_two_calls(R, K, N, V, M):
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    A, comp = _compressed(R, K, V, M, seed=31 + M)
    # these shapes split K on the tensor-core path, so the scratch is used
    plan = vnm.vnm_spmm_plan_query(A, torch.empty((K, N), dtype=torch.float16, device=dev), torch.float16,
                                   1 << 40)
    assert plan.path == vnm.VNM_PATH_TC and plan.splits > 1, plan.as_dict()
    for call in range(2):
        B_h = inputs.normal_f16((K, N), 41 + call, M, 1.0)
        B = torch.from_numpy(B_h).to(dev)
        ref = torch.empty((R, N), dtype=torch.float16, device=dev)
        vnm.vnm_spmm(A, B, ref, workspace=vnm.workspace_for(A, N))
        assert vnm.vnm_get_status(A) == vnm.VNM_OK
        got = torch.full((R, N), float("nan"), dtype=torch.float16, device=dev)
        status = torch.zeros(3, dtype=torch.int32, device=dev)
        assert _noalloc_call(A, B, got, status) == vnm.VNM_OK
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0, 0]
        got_h = got.float().cpu().numpy()
        assert _close(got_h, oracle.spmm(*comp, R, K, V, M, B_h)), f"call {call} against the oracle"
        assert _close(got_h, ref.float().cpu().numpy()), f"call {call} against vnm_spmm"


def test_without_status_pointer_and_fp32_output():
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    R, K, N, V, M = 2048, 4096, 24, 64, 4
    A, comp = _compressed(R, K, V, M, seed=51)
    for call in range(2):
        B_h = inputs.normal_f16((K, N), 61 + call, 0, 1.0)
        B = torch.from_numpy(B_h).to(dev)
        ref = torch.empty((R, N), dtype=torch.float32, device=dev)
        vnm.vnm_spmm(A, B, ref, workspace=vnm.workspace_for(A, N))
        got = torch.empty((R, N), dtype=torch.float32, device=dev)
        assert _noalloc_call(A, B, got) == vnm.VNM_OK
        torch.cuda.synchronize()
        assert _close(got.cpu().numpy(), oracle.spmm(*comp, R, K, V, M, B_h)), f"call {call} against the oracle"
        assert _close(got.cpu().numpy(), ref.cpu().numpy()), f"call {call} against vnm_spmm"


def test_rejects_scratch_beyond_the_static_maximum():
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    # 9 x 6 tiles of 128 x 192 split K in two: 2 x 1152 x 1024 fp32 partials > 8 MiB
    R, K, N, V, M = 1152, 4096, 1024, 128, 4
    A, _ = _compressed(R, K, V, M, seed=71)
    B = torch.zeros((K, N), dtype=torch.float16, device=dev)
    C = torch.zeros((R, N), dtype=torch.float16, device=dev)
    plan = vnm.vnm_spmm_plan_query(A, B, torch.float16, 1 << 40)
    assert plan.path == vnm.VNM_PATH_TC and plan.splits * R * N * 4 > (8 << 20), plan.as_dict()
    assert _noalloc_call(A, B, C) == vnm.VNM_ERR_INVALID_ARG
