"""vnm_spmm on the GPU against the CPU oracle: C within 1e-2 * (1 + |C_oracle|)
(fp16 inputs, fp32 accumulation; VENOM section 4, Figure 4), on the
tensor-core path and on the CUDA-core path, with multi-tile and ragged
shapes, split-K, both C types, and the workload shapes."""
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import read_fixture
from structured_sparse_matmul_gb300 import inputs, vnm, workloads

pytestmark = pytest.mark.gpu

from gpu_util import (assert_compress_bitexact, check_close, check_tight_f32, device, gpu_compress,  # noqa: E402
                      run_spmm, sample_rows, to_dev)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _setup(R, K, N, V, M, seed=21, a_sigma=0.02):
    W = inputs.normal_f16((R, K), seed, 0, a_sigma)
    B = inputs.normal_f16((K, N), seed, 1, 1.0)
    A, st = gpu_compress(W, V, M)
    assert st == vnm.VNM_OK
    values, meta, colidx = assert_compress_bitexact(A, W, V, M)
    return A, B, (values, meta, colidx)


def _ref(comp, R, K, V, M, B, rows=None):
    values, meta, colidx = comp
    return oracle.spmm(values, meta, colidx, R, K, V, M, B, rows=rows)


def test_worked_example_product():
    """Row 0 of the 2 x 8 worked example times B = 0.9*b0 - 0.4*b2 + 0.7*b5 - 1.2*b7."""
    fx = read_fixture(os.path.join(GOLDEN, "worked_2x8.txt"))
    W = np.array([[float(x) for x in fx["dense_row0"].split()], [float(x) for x in fx["dense_row1"].split()]],
                 dtype=np.float16)
    B = np.zeros((8, 3), dtype=np.float16)
    B[:, 0] = np.arange(1, 9)
    B[:, 1] = [0.5, -2, 3, 0.25, 7, -1, 1.5, 4]
    B[:, 2] = 1
    A, st = gpu_compress(W, 1, 4)
    got, _ = run_spmm(A, B, torch.float32)
    f = lambda x: float(np.float16(x))  # noqa: E731
    want0 = [f(0.9) * float(B[0, n]) + f(-0.4) * float(B[2, n]) + f(0.7) * float(B[5, n]) + f(-1.2) * float(B[7, n])
             for n in range(3)]
    assert np.allclose(got[0], want0, rtol=1e-6, atol=1e-6)


TC_SHAPES = [
    # R, K, N, V, M
    (384, 512, 64, 128, 4),
    (384, 512, 128, 128, 4),
    (256, 1024, 200, 128, 8),
    (384, 1536, 256, 128, 8),
    (256, 2048, 48, 128, 16),
    (128, 4096, 16, 128, 32),
    (272, 256, 72, 16, 4),     # ragged rows (R % 128 != 0), plain 2:4
    (256, 1024, 24, 256, 8),   # V = 256: two tiles per block row
    (128, 512, 8, 128, 4),     # N = 8: one MMA of N = 16 with zero-filled columns
    (256, 1024, 128, 64, 16),  # V = 64: 64-row tiles (M = 64 MMA), gathered B
    (256, 1024, 128, 64, 8),
    (272, 1024, 88, 16, 8),    # V = 16, M = 8: A re-encoded as 2:4 (lift), ragged rows
    (192, 2048, 40, 64, 16),
    (64, 4096, 256, 64, 32),
    (320, 512, 72, 64, 4),     # V = 64 with M = 4: 128-row tiles, ragged rows
]


@pytest.mark.parametrize("R,K,N,V,M", TC_SHAPES)
@pytest.mark.parametrize("c_dtype", [torch.float16, torch.float32], ids=["f16", "f32"])
def test_tensor_core_path(R, K, N, V, M, c_dtype):
    A, B, comp = _setup(R, K, N, V, M)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B), c_dtype)
    assert plan.path == vnm.VNM_PATH_TC, plan.as_dict()
    got, _ = run_spmm(A, B, c_dtype)
    check_close(got, _ref(comp, R, K, V, M, B), f"tc {R}x{K}x{N} {V}:2:{M}")
    if c_dtype == torch.float32:
        check_tight_f32(got, comp, R, K, V, M, B, what=f"tc {R}x{K}x{N} {V}:2:{M}")


@pytest.mark.parametrize("tile_n", [16, 32, 64, 128, 192, 256])
@pytest.mark.parametrize("V,tile_m", [(128, 128), (64, 64), (128, 64)])
def test_tensor_core_tiles(tile_n, V, tile_m):
    """Gathered B (lift = 0) at every tile width and both MMA heights."""
    R, K, N, M = 256, 1024, 296, 8  # N % 8 == 0 (TMA rows), ragged against every tile_n
    A, B, comp = _setup(R, K, N, V, M, seed=22)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    assert plan.path == vnm.VNM_PATH_TC and plan.lift == 0
    plan.tile_m = tile_m
    plan.tile_n = tile_n
    plan.stages = 0  # the default depth for this tile
    plan.splits = 1
    got, _ = run_spmm(A, B, plan=plan)
    check_close(got, _ref(comp, R, K, V, M, B), f"tile_n {tile_n}")


@pytest.mark.parametrize("tile_n", [16, 32, 64, 192, 256])
def test_tensor_core_tiles_plain_2to4(tile_n):
    """M = 4 (B rows by TMA, no gather) at several tile widths, ragged N."""
    R, K, N, V, M = 256, 1024, 296, 16, 4
    A, B, comp = _setup(R, K, N, V, M, seed=30)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    assert plan.path == vnm.VNM_PATH_TC
    plan.tile_n = tile_n
    plan.stages = 0
    plan.splits = 1
    got, _ = run_spmm(A, B, plan=plan)
    check_close(got, _ref(comp, R, K, V, M, B), f"plain 2:4 tile_n {tile_n}")


# ---------------------------------------------------------------- M = 8 re-encoded as 2:4 (lift)

def _lift_plan(A, B, c_dtype=torch.float16):
    """The plan vnm_spmm would use, asked for the re-encoded path (the
    default only where the gather cannot run)."""
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B), c_dtype)
    assert plan.path == vnm.VNM_PATH_TC, plan.as_dict()
    plan.lift = 1
    plan.tile_m = 128
    plan.stages = 0
    return plan


def _all_pairs_weights(R, K, V, seed):
    """W (R x K, M = 8) in which every V-block row keeps, in block j, the
    pair of columns PAIRS[(j + 3 * vb) % 28]: all rows of the V-block are
    non-zero there (with random signs and magnitudes) and zero elsewhere, so
    the column selection takes those two columns first and every row keeps
    both. Every one of the 28 pairs d0 < d1 of an 8-column block appears,
    in every position of a 16-block stage."""
    pairs = [(a, b) for a in range(8) for b in range(a + 1, 8)]
    rng = np.random.default_rng(seed)
    W = np.zeros((R, K), dtype=np.float16)
    for vb in range(R // V):
        for j in range(K // 8):
            d0, d1 = pairs[(j + 3 * vb) % 28]
            rows = slice(vb * V, (vb + 1) * V)
            W[rows, 8 * j + d0] = (rng.uniform(0.5, 2.0, V) * rng.choice([-1, 1], V)).astype(np.float16)
            W[rows, 8 * j + d1] = (rng.uniform(0.5, 2.0, V) * rng.choice([-1, 1], V)).astype(np.float16)
    return W


@pytest.mark.parametrize("V", [16, 64, 128])
def test_lift_every_column_pair(V):
    """Every (d0, d1) placement of a row's two kept values in an 8-column
    block: the 2:4 re-encoding (both in the first group, both in the second,
    one in each, with column 0 or 4 among them or not) against the oracle,
    with the fp32 summation bound."""
    R, K, N = 256, 2048, 136
    W = _all_pairs_weights(R, K, V, seed=61)
    B = inputs.normal_f16((K, N), 61, 1, 1.0)
    A, st = gpu_compress(W, V, 8)
    assert st == vnm.VNM_OK
    comp = assert_compress_bitexact(A, W, V, 8)
    plan = _lift_plan(A, B, torch.float32)
    got, _ = run_spmm(A, B, torch.float32, plan=plan)
    check_close(got, _ref(comp, R, K, V, 8, B), f"all pairs V={V}")
    check_tight_f32(got, comp, R, K, V, 8, B, what=f"all pairs V={V}")


@pytest.mark.parametrize("R,K,N,V", [(128, 128, 16, 16),     # one tile, one stage
                                     (144, 384, 40, 16),     # ragged rows (R % 128 = 16) and columns
                                     (320, 1024, 296, 32),   # V = 32
                                     (384, 1152, 520, 64),   # three row tiles, N over two 256-column tiles
                                     (512, 1024, 64, 256)])  # V = 256: two row tiles share column-loc
@pytest.mark.parametrize("c_dtype", [torch.float16, torch.float32], ids=["f16", "f32"])
def test_lift_shapes(R, K, N, V, c_dtype):
    A, B, comp = _setup(R, K, N, V, 8, seed=62)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B), c_dtype)
    assert plan.path == vnm.VNM_PATH_TC and plan.lift == (1 if V % 64 or (K // 8) % 32 else 0), plan.as_dict()
    got, _ = run_spmm(A, B, c_dtype, plan=_lift_plan(A, B, c_dtype))
    check_close(got, _ref(comp, R, K, V, 8, B), f"lift {R}x{K}x{N} V={V}")
    if c_dtype == torch.float32:
        check_tight_f32(got, comp, R, K, V, 8, B, what=f"lift {R}x{K}x{N} V={V}")


@pytest.mark.parametrize("tile_n", [16, 32, 64, 128, 192, 256])
def test_lift_tiles(tile_n):
    R, K, N, V = 256, 1024, 296, 64
    A, B, comp = _setup(R, K, N, V, 8, seed=63)
    plan = _lift_plan(A, B)
    plan.tile_n = tile_n
    plan.stages = 0
    plan.splits = 1
    got, _ = run_spmm(A, B, torch.float32, plan=plan)
    check_close(got, _ref(comp, R, K, V, 8, B), f"lift tile_n {tile_n}")
    check_tight_f32(got, comp, R, K, V, 8, B, what=f"lift tile_n {tile_n}")


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_lift_split_k(splits):
    R, K, N, V = 256, 2560, 40, 128
    A, B, comp = _setup(R, K, N, V, 8, seed=64)
    plan = _lift_plan(A, B)
    plan.splits = splits
    for c_dtype in (torch.float16, torch.float32):
        got, _ = run_spmm(A, B, c_dtype, plan=plan)
        check_close(got, _ref(comp, R, K, V, 8, B), f"lift splits {splits}")
    check_tight_f32(got, comp, R, K, V, 8, B, what=f"lift splits {splits}")


def test_lift_agrees_with_gather():
    """Both tensor-core formulations of one M = 8 product (the MMAs over the
    condensed K with gathered rows of B, and over the whole K with A
    re-encoded) are within the fp32 bound of the oracle."""
    R, K, N, V = 512, 2048, 264, 128
    A, B, comp = _setup(R, K, N, V, 8, seed=65)
    lifted, _ = run_spmm(A, B, torch.float32, plan=_lift_plan(A, B))
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    assert plan.lift == 0
    gathered, _ = run_spmm(A, B, torch.float32, plan=plan)
    for got, what in ((lifted, "lift"), (gathered, "gather")):
        check_tight_f32(got, comp, R, K, V, 8, B, what=what)


@pytest.mark.parametrize("R,K,N,V", [(4096, 2048, 2048, 64),   # the planner's choice (wide B, 64-row gather)
                                     (320, 1024, 600, 64),     # ragged rows and columns
                                     (256, 1152, 136, 32)])    # a plan asking for it on a narrow product
def test_lift_written_out(R, K, N, V):
    """lift = 2: A written out as a plain 2:4 matrix over the whole K in the
    workspace by a first kernel, then the 2:4 path (split K after it)."""
    A, B, comp = _setup(R, K, N, V, 8, seed=68)
    rows = None if R <= 512 else sample_rows(R, V, 64)
    if N >= 512:
        plan = vnm.vnm_spmm_plan_query(A, to_dev(B), torch.float32, vnm.vnm_spmm_workspace_size(A, N))
        assert plan.lift == 2 and plan.tile_m == 128, plan.as_dict()
        got, _ = run_spmm(A, B, torch.float32)  # through vnm_spmm with vnm_spmm_workspace_size bytes
    else:
        plan = _lift_plan(A, B, torch.float32)
        plan.lift = 2
        plan.splits = 3
        ws = torch.empty((R * K + R * K // 8 + 1024) // 4 + 3 * R * N + 64, dtype=torch.float32, device=device())
        C = torch.empty((R, N), dtype=torch.float32, device=device())
        vnm.vnm_spmm_with_plan(A, plan, to_dev(B), C, workspace=ws)
        assert vnm.vnm_get_status(A) == vnm.VNM_OK
        got = C.cpu().numpy()
    g = got if rows is None else got[rows]
    check_close(g, _ref(comp, R, K, V, 8, B, rows=rows), f"lift 2 {R}x{K}x{N}")
    check_tight_f32(g, comp, R, K, V, 8, B, rows=rows, what=f"lift 2 {R}x{K}x{N}")
    # a workspace without room for the written-out form is refused for this plan
    if N < 512:
        with pytest.raises(vnm.VnmError) as e:
            vnm.vnm_spmm_with_plan(A, plan, to_dev(B), C, workspace=torch.empty(1024, dtype=torch.float32,
                                                                                  device=device()))
        assert e.value.code == vnm.VNM_ERR_INVALID_ARG


def test_lift_plan_checks():
    R, K, N, V = 256, 1024, 64, 128
    A, B, _ = _setup(R, K, N, V, 8, seed=66)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    assert plan.lift == 0 and plan.tile_m == 128
    plan.lift = 3
    with pytest.raises(vnm.VnmError) as e:
        run_spmm(A, B, plan=plan)
    assert e.value.code == vnm.VNM_ERR_INVALID_ARG
    plan.lift = 1
    plan.tile_m = 64
    with pytest.raises(vnm.VnmError) as e:
        run_spmm(A, B, plan=plan)
    assert e.value.code == vnm.VNM_ERR_UNSUPPORTED
    # K % 128 != 0 (but K/M % 32 == 0 is not met either): the CUDA-core path
    A2, B2, comp2 = _setup(64, 1088, 40, 16, 8, seed=67)
    plan2 = vnm.vnm_spmm_plan_query(A2, to_dev(B2))
    assert plan2.path == vnm.VNM_PATH_SIMT and plan2.lift == 0
    got, _ = run_spmm(A2, B2)
    check_close(got, _ref(comp2, 64, 1088, 16, 8, B2), "K % 128 != 0")


def test_reserved_plan_fields_rejected():
    """A plan whose reserved words are not zero is refused before any launch."""
    R, K, N, V, M = 256, 512, 128, 128, 4
    A, B, _ = _setup(R, K, N, V, M, seed=34)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    plan.reserved[0] = 2
    with pytest.raises(vnm.VnmError) as e:
        run_spmm(A, B, plan=plan)
    assert e.value.code == vnm.VNM_ERR_INVALID_ARG


@pytest.mark.parametrize("splits", [2, 3, 5])
def test_tensor_core_split_k(splits):
    R, K, N, V, M = 256, 2560, 40, 128, 4
    A, B, comp = _setup(R, K, N, V, M, seed=23)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    assert plan.path == vnm.VNM_PATH_TC
    plan.splits = splits
    for c_dtype in (torch.float16, torch.float32):
        got, _ = run_spmm(A, B, c_dtype, plan=plan)
        check_close(got, _ref(comp, R, K, V, M, B), f"splits {splits}")
    check_tight_f32(got, comp, R, K, V, M, B, what=f"splits {splits}")


@pytest.mark.parametrize("R,K,N,V,M", [(256, 1024, 200, 128, 8), (272, 256, 72, 16, 4), (96, 600, 33, 8, 5),
                                       (128, 512, 40, 64, 8), (64, 4096, 17, 64, 4)])
def test_cuda_core_path(R, K, N, V, M):
    A, B, comp = _setup(R, K, N, V, M, seed=24)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    plan.path = vnm.VNM_PATH_SIMT
    for c_dtype in (torch.float16, torch.float32):
        got, _ = run_spmm(A, B, c_dtype, plan=plan)
        check_close(got, _ref(comp, R, K, V, M, B), f"simt {R}x{K}x{N}")
    check_tight_f32(got, comp, R, K, V, M, B, what=f"simt {R}x{K}x{N}")


@pytest.mark.parametrize("N", [1, 2, 3, 5, 7])
def test_small_n(N):
    R, K, V, M = 256, 2048, 64, 8
    A, B, comp = _setup(R, K, N, V, M, seed=25)
    got, _ = run_spmm(A, B)
    check_close(got, _ref(comp, R, K, V, M, B), f"N={N}")


def test_unaligned_and_strided_operands():
    R, K, N, V, M = 256, 1024, 37, 128, 8
    A, B, comp = _setup(R, K, N, V, M, seed=26)
    ref = _ref(comp, R, K, V, M, B)
    got, _ = run_spmm(A, B, ld_b=N)            # ld_b % 8 != 0: CUDA-core path
    check_close(got, ref, "ld_b = N")
    got, _ = run_spmm(A, B, ld_b=48, ld_c=41)  # aligned B, padded C rows
    check_close(got, ref, "ld_b = 48, ld_c = 41")


def test_unservable_plan_rejected():
    R, K, N, V, M = 128, 512, 64, 64, 16
    A, B, comp = _setup(R, K, N, V, M, seed=27)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    assert plan.path == vnm.VNM_PATH_TC and plan.tile_m == 64 and plan.lift == 0
    plan.tile_m = 128  # a 128-row tile would span two column-loc blocks
    with pytest.raises(vnm.VnmError) as e:
        run_spmm(A, B, plan=plan)
    assert e.value.code == vnm.VNM_ERR_UNSUPPORTED
    plan.tile_m = 64
    plan.lift = 1  # M = 16 cannot be re-encoded as 2:4 over 8-column blocks
    with pytest.raises(vnm.VnmError) as e:
        run_spmm(A, B, plan=plan)
    assert e.value.code == vnm.VNM_ERR_UNSUPPORTED


def test_empty_products():
    R, K, V, M = 128, 512, 128, 4
    A, B, comp = _setup(R, K, 8, V, M)
    C = torch.full((R, 0), 1.0, dtype=torch.float16, device=device())
    vnm.vnm_spmm(A, torch.zeros((K, 0), dtype=torch.float16, device=device()), C)
    Z = vnm.vnm_matrix_alloc(64, 0, 16, 8, device())
    C = torch.full((64, 5), 7.0, dtype=torch.float32, device=device())
    vnm.vnm_spmm(Z, torch.zeros((0, 5), dtype=torch.float16, device=device()), C)
    assert vnm.vnm_get_status(Z) == vnm.VNM_OK
    assert not C.any().item()


def _workload_case(case: workloads.Case, max_rows: int):
    W = inputs.normal_f16((case.R, case.K), case.seed, case.a_stream, workloads.A_SIGMA)
    B = inputs.normal_f16((case.K, case.N), case.seed, case.b_stream, workloads.B_SIGMA)
    A, st = gpu_compress(W, case.V, case.M)
    assert st == vnm.VNM_OK
    comp = assert_compress_bitexact(A, W, case.V, case.M)
    c_dtype = torch.float32 if case.c_f32 else torch.float16
    got, Bd = run_spmm(A, B, c_dtype)
    rows = None if case.R <= max_rows else sample_rows(case.R, case.V, max_rows // 2)
    ref = _ref(comp, case.R, case.K, case.V, case.M, B, rows=rows)
    check_close(got if rows is None else got[rows], ref, case.name)
    if case.c_f32:
        check_tight_f32(got if rows is None else got[rows], comp, case.R, case.K, case.V, case.M, B, rows=rows,
                        what=case.name)
    return A, Bd


@pytest.mark.parametrize("case", [c for w in (1, 2, 3, 4) for c in workloads.workload_cases(w)],
                         ids=lambda c: c.name)
def test_workloads(case):
    _workload_case(case, max_rows=256 if case.N >= 2048 else 1024)


def _oracle_compress_parallel(W, V, M):
    """The oracle's compress of all of W, one host thread per group of whole
    V-block rows (each call is the same plain oracle on its rows; the C code
    runs outside the GIL). The result equals one call on all of W: the
    format is computed per V-block row."""
    from concurrent.futures import ThreadPoolExecutor
    R = W.shape[0]
    nb = R // V
    threads = max(1, min(nb, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 8))
    bounds = [nb * q // threads * V for q in range(threads + 1)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda q: oracle.compress(W[bounds[q]:bounds[q + 1]], V, M), range(threads)))
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(3))


@pytest.mark.parametrize("case", workloads.workload_cases(5), ids=lambda c: c.name)
def test_workload5_full_size_sampled(case):
    """The large FFN shape at full size, through the same calls and plan the
    bench times: the whole W is compressed on the GPU and its values,
    m-indices and column-loc must match the oracle's compress of the whole W
    bit for bit; C (computed by the GPU for all rows) is checked against the
    oracle on a sample of rows from the first, middle and last V-block rows
    and 40 more spread over R."""
    R, K, N, V, M = case.R, case.K, case.N, case.V, case.M
    W = inputs.normal_f16((R, K), case.seed, case.a_stream, workloads.A_SIGMA)
    B = inputs.normal_f16((K, N), case.seed, case.b_stream, workloads.B_SIGMA)
    A, st = gpu_compress(W, V, M)
    assert st == vnm.VNM_OK
    got, _ = run_spmm(A, B, torch.float16)
    values, meta, colidx = _oracle_compress_parallel(W, V, M)
    del W
    gv = A.values.cpu().numpy().view(np.uint16)
    assert np.array_equal(gv, values), f"values differ at {np.argwhere(gv != values)[:4].tolist()}"
    del gv
    gm = A.meta.cpu().numpy()
    assert np.array_equal(gm, meta), f"meta differs at {np.argwhere(gm != meta)[:4].tolist()}"
    gc = A.colidx.cpu().numpy()
    assert np.array_equal(gc, colidx), f"column-loc differs at {np.argwhere(gc != colidx)[:4].tolist()}"
    nb = R // V
    rng = np.random.default_rng(5)
    rows = set(sample_rows(R, V, 40))
    for i in (0, nb // 2, nb - 1):
        rows.update(i * V + r for r in [0, 1, V // 2, V - 1] + rng.integers(0, V, 4).tolist())
    rows = sorted(rows)
    ref = oracle.spmm(values, meta, colidx, R, K, V, M, B, rows=rows)
    check_close(got[rows], ref, f"{case.name} sampled rows")


STREAM_SHAPES = [
    (64, 512, 8, 4, 3),       # V < 16: rows of a block row spread over fewer warps
    (96, 600, 8, 5, 2),       # odd M, K not a multiple of the stage
    (256, 1024, 128, 8, 1),
    (272, 256, 16, 4, 7),
    (512, 8192, 32, 16, 4),   # several staged chunks per split
    (4096, 4096, 64, 4, 1),   # decode shape
]


@pytest.mark.parametrize("R,K,V,M,N", STREAM_SHAPES)
@pytest.mark.parametrize("c_dtype", [torch.float16, torch.float32], ids=["f16", "f32"])
def test_streaming_small_n(R, K, V, M, N, c_dtype):
    """N <= 8 takes the streaming CUDA-core path: with the workspace it asks
    for (split K, partials reduced in order) and without one (one split)."""
    A, B, comp = _setup(R, K, N, V, M, seed=28)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B), c_dtype, 1 << 40)
    assert plan.path == vnm.VNM_PATH_SIMT, plan.as_dict()
    rows = None if R <= 512 else sample_rows(R, V, 64)
    ref = _ref(comp, R, K, V, M, B, rows=rows)
    for ws in (True, False):
        got, _ = run_spmm(A, B, c_dtype, workspace=ws)
        check_close(got if rows is None else got[rows], ref, f"stream {R}x{K}x{N} {V}:2:{M} ws={ws}")
        if c_dtype == torch.float32:
            check_tight_f32(got if rows is None else got[rows], comp, R, K, V, M, B, rows=rows,
                            what=f"stream {R}x{K}x{N} {V}:2:{M} ws={ws}")


@pytest.mark.parametrize("splits", [1, 2, 4, 8])
@pytest.mark.parametrize("R,K,N,V,M", [(192, 4096, 5, 64, 8),
                                       (256, 256, 3, 128, 4)])  # two row passes; 64 blocks: most splits empty
def test_streaming_split_clusters(splits, R, K, N, V, M):
    """The streaming kernel's K splits (1, 2, 4 or 8 CTAs of a V-block row in
    one cluster, reduced in split order through distributed shared memory),
    ragged N, both C types; the same C bit for bit on a second run."""
    A, B, comp = _setup(R, K, N, V, M, seed=36)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    assert plan.path == vnm.VNM_PATH_SIMT, plan.as_dict()
    plan.splits = splits
    ref = _ref(comp, R, K, V, M, B)
    for c_dtype in (torch.float16, torch.float32):
        got, _ = run_spmm(A, B, c_dtype, plan=plan, workspace=False)
        check_close(got, ref, f"stream splits {splits}")
        again, _ = run_spmm(A, B, c_dtype, plan=plan, workspace=False)
        assert np.array_equal(got, again)


def test_streaming_at_n8_by_plan():
    """N = 8 runs on the tensor cores by default; a plan may ask for the
    streaming path instead, with a chosen split."""
    R, K, N, V, M = 1024, 4096, 8, 64, 8
    A, B, comp = _setup(R, K, N, V, M, seed=29)
    plan = vnm.vnm_spmm_plan_query(A, to_dev(B))
    plan.path = vnm.VNM_PATH_SIMT
    plan.splits = 3
    got, _ = run_spmm(A, B, plan=plan)
    check_close(got, _ref(comp, R, K, V, M, B), "stream N=8")


@pytest.mark.parametrize("R,K,N,V,M", [(1024, 4096, 512, 32, 8),   # tensor cores, re-encoded A (lift)
                                       (1024, 4096, 512, 64, 16),  # tensor cores, gathered B
                                       (256, 2560, 40, 128, 4),    # tensor cores, split K
                                       (512, 4096, 3, 64, 8)])     # streaming small N, split K
def test_repeatable_bit_for_bit(R, K, N, V, M):
    """The same inputs give the same C bit for bit (fixed accumulation and
    split-K reduction orders)."""
    A, B, _ = _setup(R, K, N, V, M, seed=31)
    first, _ = run_spmm(A, B)
    for _ in range(2):
        again, _ = run_spmm(A, B)
        assert np.array_equal(first.view(np.uint32), again.view(np.uint32))
