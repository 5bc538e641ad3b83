"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the CPU oracle on the same seeded host buffers."""
import numpy as np
import torch

import oracle
from structured_sparse_matmul_gb300 import vnm

TOL = 1e-2  # |C_gpu - C_oracle| <= TOL * (1 + |C_oracle|), fp16 inputs, fp32 accumulation


def device():
    return torch.device("cuda", 0)


def to_dev(a: np.ndarray, ld: int = None) -> torch.Tensor:
    """Host fp16 array -> device tensor; ``ld`` > columns pads each row."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    if ld is None or ld == a.shape[1]:
        return t.to(device())
    buf = torch.full((a.shape[0], ld), float("nan"), dtype=t.dtype, device=device())
    buf[:, : a.shape[1]] = t.to(device())
    return buf[:, : a.shape[1]]


def gpu_compress(W: np.ndarray, V: int, M: int, ld: int = None):
    R, K = W.shape
    A = vnm.vnm_matrix_alloc(R, K, V, M, device())
    Wd = to_dev(W, ld)
    vnm.vnm_compress(A, Wd)
    st = vnm.vnm_get_status(A)
    return A, st


def assert_compress_bitexact(A, W: np.ndarray, V: int, M: int):
    values, meta, colidx = oracle.compress(W, V, M)
    gv = A.values.cpu().numpy().view(np.uint16)
    gm = A.meta.cpu().numpy()
    gc = A.colidx.cpu().numpy()
    assert np.array_equal(gc, colidx), f"colidx differs at {np.argwhere(gc != colidx)[:5].tolist()}"
    assert np.array_equal(gm, meta), f"meta differs at {np.argwhere(gm != meta)[:5].tolist()}"
    assert np.array_equal(gv, values), f"values differ at {np.argwhere(gv != values)[:5].tolist()}"
    return values, meta, colidx


def check_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    excess = np.abs(got - ref) - TOL * (1.0 + np.abs(ref))
    bad = np.argwhere(~(excess <= 0))
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of tolerance, first {bad[:4].tolist()}: "
                           f"got {[got[tuple(b)] for b in bad[:4]]} want {[ref[tuple(b)] for b in bad[:4]]}")


def run_spmm(A, B: np.ndarray, c_dtype=torch.float16, plan=None, ld_b=None, ld_c=None, workspace=True):
    N = B.shape[1]
    Bd = to_dev(B, ld_b)
    if ld_c is None:
        C = torch.empty((A.R, N), dtype=c_dtype, device=device())
    else:
        C = torch.empty((A.R, ld_c), dtype=c_dtype, device=device())[:, :N]
    if plan is None:
        ws = vnm.workspace_for(A, N) if workspace else None
        vnm.vnm_spmm(A, Bd, C, workspace=ws)
    else:
        s = max(1, plan.splits)
        ws = torch.empty(s * A.R * N + 64, dtype=torch.float32, device=device()) if s > 1 and workspace else None
        vnm.vnm_spmm_with_plan(A, plan, Bd, C, workspace=ws)
    st = vnm.vnm_get_status(A)
    assert st == vnm.VNM_OK, vnm.status_string(st)
    return C.float().cpu().numpy(), Bd


def sample_rows(R: int, V: int, count: int, seed: int = 0):
    """Rows spread over all V-blocks, always including the first and last row."""
    rng = np.random.default_rng(seed)
    rows = set([0, R - 1, V - 1, R - V])
    blocks = np.linspace(0, R // V - 1, num=min(count, R // V)).astype(np.int64)
    for b in blocks:
        rows.add(int(b * V + rng.integers(0, V)))
    return sorted(r for r in rows if 0 <= r < R)


def check_tight_f32(got: np.ndarray, comp, R: int, K: int, V: int, M: int, B: np.ndarray, rows=None,
                    what: str = ""):
    """fp32 C against the oracle's fp64 product within the fp32 summation
    bound: every product of two fp16 values is exact in fp32, so only the
    accumulation of the 2K/M kept products of a row rounds. With n terms
    the rounding error of any summation order is at most (n - 1) ulps of
    the running sum, i.e. below n * 2^-23 * sum |a||b| even when each
    addition truncates instead of rounding; the bound below allows twice
    that. A single dropped or mis-selected product (|a||b| ~ 0.02 here) is
    far above it, unlike the 1e-2 * (1 + |C|) tolerance."""
    values, meta, colidx = comp
    n_terms = 2 * (K // M)
    ref64 = oracle.spmm(values, meta, colidx, R, K, V, M, B, rows=rows, acc="f64")
    mag = oracle.spmm(values & np.uint16(0x7FFF), meta, colidx, R, K, V, M, np.abs(B), rows=rows, acc="f64")
    bound = n_terms * 2.0 ** -22 * mag + 1e-30
    err = np.abs(got.astype(np.float64) - ref64)
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, (f"{what}: {len(bad)} elements beyond the fp32 summation bound, first {bad[:4].tolist()}: "
                           f"err {[err[tuple(b)] for b in bad[:4]]} bound {[bound[tuple(b)] for b in bad[:4]]}")
