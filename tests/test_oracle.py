"""Pins for the CPU oracle (no GPU).

Each ``check_*`` function pins one part of the oracle against something other
than the oracle itself: the worked example printed in the lecture notes "2:4
sparsity on sparse tensor cores", the storage arithmetic printed there and in
"VENOM" section 3, brute-force enumeration of every candidate subset, format
invariants, round trips, and numpy's own fp64 matmul. ``test_mutants_are_caught``
plants plausible mistakes in copies of the oracle source and checks that at
least one pin fails for each.
"""
import itertools
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from conftest import read_fixture
from structured_sparse_matmul_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _floats(s):
    return [float(x) for x in s.split()]


def _slots_of(meta_row, n):
    """Decode n 2-bit slots of one m-index row under the LSB-first reading."""
    return [(int(meta_row[t // 4]) >> (2 * (t % 4))) & 3 for t in range(n)]


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def check_worked_example(L):
    """The 2 x 8 matrix of "Worked: compress a 2 x 8 matrix and count bits"."""
    fx = read_fixture(os.path.join(GOLDEN, "worked_2x8.txt"))
    W = np.array([_floats(fx["dense_row0"]), _floats(fx["dense_row1"])], dtype=np.float16)
    for V in (1, 2):
        values, meta, colidx = oracle.compress(W, V, 4, L)
        for r in range(2):
            want_vals = np.array(_floats(fx[f"values_row{r}"]), dtype=np.float16)
            assert values[r].tobytes() == want_vals.tobytes(), (V, r, values[r])
            want_idx = [int(b, 2) for b in fx[f"indices_row{r}"].split()]
            assert _slots_of(meta[r], 4) == want_idx, (V, r, meta[r])
            # indices are the kept slots of each group, ascending
            kept = [tuple(int(x) for x in g.split(",")) for g in fx[f"kept_row{r}"].split()]
            assert [tuple(want_idx[0:2]), tuple(want_idx[2:4])] == kept
            # the packed byte of the 4 printed 2-bit tags, LSB first
            assert int(meta[r][0]) == sum(want_idx[t] << (2 * t) for t in range(4))
        # M = 4: column-loc is the identity in every block
        assert (colidx == np.array([0, 1, 2, 3], dtype=np.uint8)).all()
    # the printed bytes of this packing: row 0 -> 0xD8, row 1 -> 0xC9
    values, meta, colidx = oracle.compress(W, 1, 4, L)
    assert meta[:, 0].tolist() == [0xD8, 0xC9]


def check_worked_local_index(L):
    """Indices are local to their group: slot 1 of group 1 decompresses to column 5."""
    fx = read_fixture(os.path.join(GOLDEN, "worked_2x8.txt"))
    W = np.array([_floats(fx["dense_row0"]), _floats(fx["dense_row1"])], dtype=np.float16)
    values, meta, colidx = oracle.compress(W, 1, 4, L)
    D = oracle.decompress(values, meta, colidx, 2, 8, 1, 4, L)
    g = dict(kv.split("=") for kv in fx["local_index"].split())
    col = int(g["column"])
    assert col == 4 * int(g["group"]) + int(g["slot"])
    assert D[0, col] == np.float16(0.7)
    # kept positions hold the dense values, pruned ones are +0.0
    kept0 = {0, 2, 5, 7}
    for k in range(8):
        if k in kept0:
            assert D[0, k] == W[0, k]
        else:
            assert D[0, k].view(np.uint16) == 0


def check_worked_product(L):
    """Row 0 times B: 0.9*b0 - 0.4*b2 + 0.7*b5 - 1.2*b7 (with fp16 weights)."""
    fx = read_fixture(os.path.join(GOLDEN, "worked_2x8.txt"))
    W = np.array([_floats(fx["dense_row0"]), _floats(fx["dense_row1"])], dtype=np.float16)
    values, meta, colidx = oracle.compress(W, 1, 4, L)
    terms = []
    for term in fx["product_row0"].split():
        coef, b = term.split("*")
        terms.append((float(np.float16(float(coef))), int(b[1:])))
    B = np.zeros((8, 3), dtype=np.float16)
    B[:, 0] = np.arange(1, 9)
    B[:, 1] = np.array([0.5, -2, 3, 0.25, 7, -1, 1.5, 4])
    B[:, 2] = 1
    want = np.array([sum(c * float(B[k, n]) for c, k in terms) for n in range(3)])
    got64 = oracle.spmm(values, meta, colidx, 2, 8, 1, 4, B, rows=[0], acc="f64", L=L)[0]
    assert np.allclose(got64, want, rtol=1e-15, atol=0)
    got32 = oracle.spmm(values, meta, colidx, 2, 8, 1, 4, B, rows=[0], acc="f32", L=L)[0]
    assert np.allclose(got32, want, rtol=1e-6, atol=1e-7)


def check_storage_arithmetic(L):
    """Storage counts printed in the lecture notes and in VENOM section 3."""
    fx = read_fixture(os.path.join(GOLDEN, "worked_2x8.txt"))
    bits = dict(kv.split("=") for kv in fx["fp16_bits"].split())
    nv, nm, nc = oracle.sizes(2, 8, 1, 4, L)
    assert nv * 16 == int(bits["values"])
    assert nm * 8 == int(bits["indices"])
    assert nv * 16 + nm * 8 == int(bits["total"])
    assert (nv * 16 + nm * 8) / (2 * 8 * 16) == float(bits["ratio"])
    nv, nm, nc = oracle.sizes(512, 1024, 1, 4, L)
    assert nm * 8 == int(fx["meta_bits_512x1024"])
    assert nm == 64 * 1024
    # VENOM Figure 3: values and m-indices R x K/M*2, column-loc R/V x K/M x 4
    f3 = read_fixture(os.path.join(GOLDEN, "venom_fig3.txt"))
    R, K, V, M = (int(f3[k]) for k in ("R", "K", "V", "M"))
    nv, nm, nc = oracle.sizes(R, K, V, M, L)
    assert nv == len(f3["m_indices"].split()) == R * K // M * 2
    assert nc == len(f3["column_loc"].split()) == R // V * K // M * 4
    # VENOM section 3: about 13.28 % overhead at V = 128 (2-bit m-index per value + an
    # 8-bit column-loc entry per 4 columns every V rows) over 16-bit values
    nv, nm, nc = oracle.sizes(1024, 4096, 128, 8, L)
    overhead = (nm * 8 + nc * 8) / (nv * 16)
    assert round(100 * overhead, 2) == float(f3["overhead_v128_percent"])


def _brute_force_compress(W, V, M):
    """All-subset enumeration: the 4-column subset of largest total L1 per
    block, then the 2-of-4 pair of largest |a|+|b| per row; on ties the
    lexicographically smallest subset (itertools.combinations order)."""
    R, K = W.shape
    Wd = W.astype(np.float64)
    sel = np.zeros((R // V, K // M, 4), dtype=np.int64)
    pairs = np.zeros((R, K // M, 2), dtype=np.int64)
    for i in range(R // V):
        for j in range(K // M):
            blk = np.abs(Wd[i * V:(i + 1) * V, j * M:(j + 1) * M])
            l1 = [sum(blk[:, c].tolist()) for c in range(M)]  # exact for these dyadic values
            best, best_s = None, None
            for sub in itertools.combinations(range(M), 4):
                s = sum(l1[c] for c in sub)
                if best_s is None or s > best_s:
                    best, best_s = sub, s
            sel[i, j] = best
            for r in range(V):
                a = [abs(float(Wd[i * V + r, j * M + c])) for c in best]
                bp, bs = None, None
                for pr in itertools.combinations(range(4), 2):
                    s = a[pr[0]] + a[pr[1]]
                    if bs is None or s > bs:
                        bp, bs = pr, s
                pairs[i * V + r, j] = bp
    return sel, pairs


def _check_against_brute_force(L, W, V, M):
    R, K = W.shape
    values, meta, colidx = oracle.compress(W, V, M, L)
    sel, pairs = _brute_force_compress(W, V, M)
    assert (colidx.astype(np.int64) == sel).all(), "column-loc differs from brute force"
    Wb = W.view(np.uint16)
    for r in range(R):
        slots = _slots_of(meta[r], 2 * (K // M))
        for j in range(K // M):
            assert (slots[2 * j], slots[2 * j + 1]) == tuple(pairs[r, j]), (r, j)
            for t in range(2):
                c = j * M + int(sel[r // V, j, pairs[r, j][t]])
                assert values[r, 2 * j + t] == Wb[r, c], (r, j, t)


def check_brute_force_ties(L):
    """Tie-heavy inputs: values from {0, +-0.5, +-1}, many equal sums."""
    k = 0
    for M in (4, 5, 6, 8, 12):
        for V in (1, 2, 4):
            W = inputs.choice_f16((2 * V, 3 * M), 77, k, [0, 0.5, -0.5, 1, -1, 0.0])
            k += 1
            _check_against_brute_force(L, W, V, M)


def check_brute_force_subnormals(L):
    """Mixed subnormal / normal magnitudes, where the exact values decide."""
    tiny = [1023 * 2.0 ** -24, -1023 * 2.0 ** -24, 1.5 * 2.0 ** -14, 2.0 ** -13, -(2.0 ** -13),
            3 * 2.0 ** -24, 0.0, -0.0]
    for k, (V, M) in enumerate(((1, 6), (2, 8), (3, 5))):
        W = inputs.choice_f16((2 * V, 4 * M), 91, k, tiny)
        _check_against_brute_force(L, W, V, M)


def check_brute_force_normal(L):
    """N(0, 0.02) inputs (the workloads' distribution), M up to 16."""
    for k, (V, M) in enumerate(((4, 4), (2, 7), (4, 8), (1, 16))):
        W = inputs.normal_f16((2 * V, 2 * M), 55, k, 0.02)
        _check_against_brute_force(L, W, V, M)


def check_invariants_and_round_trip(L):
    """Format invariants and decompress(compress(W)) on random shapes."""
    k = 0
    for (R, K, V, M) in ((32, 64, 16, 4), (64, 128, 64, 8), (128, 96, 32, 12), (16, 512, 8, 32),
                         (8, 256, 8, 256)):
        W = inputs.normal_f16((R, K), 42, k, 0.02)
        k += 1
        values, meta, colidx = oracle.compress(W, V, M, L)
        # column-loc: 4 distinct, strictly ascending indices < M per block
        assert (np.diff(colidx.astype(np.int64), axis=2) > 0).all()
        assert int(colidx.max()) < M
        D = oracle.decompress(values, meta, colidx, R, K, V, M, L)
        Wb, Db = W.view(np.uint16), D.view(np.uint16)
        kept = np.zeros((R, K), dtype=bool)
        for r in range(R):
            slots = _slots_of(meta[r], 2 * (K // M))
            for j in range(K // M):
                s0, s1 = slots[2 * j], slots[2 * j + 1]
                assert s0 < s1  # two distinct slots, ascending
                for s in (s0, s1):
                    kept[r, j * M + int(colidx[r // V, j, s])] = True
        # exactly 2 kept per (row, block): density 2/M
        assert kept.sum() == R * (K // M) * 2
        assert (kept.reshape(R, K // M, M).sum(axis=2) == 2).all()
        # kept positions are bit copies of W, pruned ones +0.0
        assert (Db[kept] == Wb[kept]).all()
        assert (Db[~kept] == 0).all()
        # kept columns lie inside the block's column-loc
        cols = kept.reshape(R // V, V, K // M, M).any(axis=1)
        for i in range(R // V):
            for j in range(K // M):
                assert set(np.nonzero(cols[i, j])[0]) <= set(colidx[i, j].tolist())
        # the 2 kept of each row are the 2 largest |w| of its 4 selected
        for r in range(min(R, 8)):
            for j in range(K // M):
                sel = colidx[r // V, j].astype(np.int64) + j * M
                mags = np.abs(W[r, sel].astype(np.float64))
                kept_mags = np.abs(D[r, sel].astype(np.float64))[kept[r, sel]]
                assert sorted(kept_mags) == sorted(mags)[2:]
        # compress is idempotent on its own output (value-equal: +-0 may move)
        v2, m2, c2 = oracle.compress(D, V, M, L)
        D2 = oracle.decompress(v2, m2, c2, R, K, V, M, L)
        assert (D2.astype(np.float64) == D.astype(np.float64)).all()


def check_spmm_against_numpy(L):
    """fp64 oracle SpMM equals numpy's fp64 matmul of the decompressed A."""
    k = 0
    for (R, K, N, V, M) in ((16, 32, 5, 8, 4), (32, 64, 17, 16, 8), (12, 60, 3, 4, 5),
                            (8, 64, 9, 8, 16)):
        A = inputs.normal_f16((R, K), 7, k, 0.02)
        B = inputs.normal_f16((K, N), 7, k + 100, 1.0)
        k += 1
        values, meta, colidx = oracle.compress(A, V, M, L)
        D = oracle.decompress(values, meta, colidx, R, K, V, M, L).astype(np.float64)
        ref = D @ B.astype(np.float64)
        got = oracle.spmm(values, meta, colidx, R, K, V, M, B, acc="f64", L=L)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)
        # fp32 accumulation: within the standard bound K * 2^-24 * sum |a||b|
        got32 = oracle.spmm(values, meta, colidx, R, K, V, M, B, acc="f32", L=L).astype(np.float64)
        bound = K * 2.0 ** -24 * (np.abs(D) @ np.abs(B.astype(np.float64))) + 1e-30
        assert (np.abs(got32 - ref) <= bound).all()
        # a row subset gives the same rows
        rows = [R - 1, 0, R // 2]
        sub = oracle.spmm(values, meta, colidx, R, K, V, M, B, rows=rows, acc="f64", L=L)
        assert np.array_equal(sub, got[rows])
    # subnormal and signed-zero operands: numpy converts fp16 exactly
    tiny = [1023 * 2.0 ** -24, -3 * 2.0 ** -24, 2.0 ** -14, -0.0, 0.0, 1.0, -2.0]
    A = inputs.choice_f16((8, 32), 3, 0, tiny)
    B = inputs.choice_f16((32, 6), 3, 1, tiny)
    values, meta, colidx = oracle.compress(A, 4, 8, L)
    D = oracle.decompress(values, meta, colidx, 8, 32, 4, 8, L).astype(np.float64)
    got = oracle.spmm(values, meta, colidx, 8, 32, 4, 8, B, acc="f64", L=L)
    assert np.array_equal(got, D @ B.astype(np.float64))


def check_fig3_fixture(L):
    """VENOM Figure 3: ascending m-index pairs and column-loc decompress to
    exactly 2 non-zeros per (row, block), inside the block's column-loc."""
    f3 = read_fixture(os.path.join(GOLDEN, "venom_fig3.txt"))
    R, K, V, M = (int(f3[k]) for k in ("R", "K", "V", "M"))
    midx = [int(x) for x in f3["m_indices"].split()]
    cl = np.array([int(x) for x in f3["column_loc"].split()], dtype=np.uint8).reshape(R // V, K // M, 4)
    vpr = 2 * (K // M)
    meta = np.zeros((R, (vpr + 3) // 4), dtype=np.uint8)
    for r in range(R):
        for t in range(vpr):
            meta[r, t // 4] |= midx[r * vpr + t] << (2 * (t % 4))
    labels = np.arange(1, R * vpr + 1, dtype=np.float16).reshape(R, vpr)  # label + 1: non-zero
    D = oracle.decompress(labels.view(np.uint16), meta, cl, R, K, V, M, L).astype(np.float64)
    for r in range(R):
        for j in range(K // M):
            blk = D[r, j * M:(j + 1) * M]
            nz = np.nonzero(blk)[0]
            assert len(nz) == 2
            assert set(nz.tolist()) <= set(cl[r // V, j].tolist())
            # row-major order: the two labels of a block increase left to right
            assert blk[nz[0]] < blk[nz[1]]
    for pair in zip(midx[0::2], midx[1::2]):
        assert pair[0] < pair[1]
    assert (np.diff(cl.astype(np.int64), axis=2) > 0).all()


def check_gemm_compress_identity(L):
    """X = I: the fused op's W is Y^T exactly (orientation W = X . Y^T), and
    its arrays are compress(Y^T)."""
    rng = np.random.default_rng(7)
    R, K = 64, 96
    Y = (rng.standard_normal((K, R)) * 0.5).astype(np.float16)
    X = np.eye(R, dtype=np.float16)
    for V, M in ((16, 8), (1, 4), (64, 32)):
        W, got = oracle.gemm_compress(X, Y, V, M, L)
        assert W.tobytes() == np.ascontiguousarray(Y.T).tobytes()
        want = oracle.compress(np.ascontiguousarray(Y.T), V, M, L)
        for a, b in zip(got, want):
            assert np.array_equal(a, b)


def check_gemm_compress_rank1(L):
    """D = 1 with powers of two: W[r][k] = x[r] * y[k] exactly, a column's L1
    over any rows is |y[k]| times a common factor, so every block keeps the 4
    columns of largest |y| (lower column on ties), and every row the 2 of
    those with the largest |y|: the expected arrays in closed form."""
    rng = np.random.default_rng(8)
    R, K, V, M = 32, 64, 8, 16
    x = (2.0 ** rng.integers(-6, 4, R) * rng.choice([-1, 1], R)).astype(np.float16)
    y = (2.0 ** rng.integers(-6, 4, K) * rng.choice([-1, 1], K)).astype(np.float16)
    W, (values, meta, colidx) = oracle.gemm_compress(x[:, None], y[:, None], V, M, L)
    assert np.array_equal(W.astype(np.float64), np.outer(x.astype(np.float64), y.astype(np.float64)))
    for j in range(K // M):
        mags = np.abs(y[j * M:(j + 1) * M].astype(np.float64))
        order = sorted(range(M), key=lambda c: (-mags[c], c))
        cols = sorted(order[:4])
        keep = sorted(sorted(range(4), key=lambda s: (-mags[cols[s]], s))[:2])
        for i in range(R // V):
            assert colidx[i, j].tolist() == cols
        for r in range(R):
            want = [np.float16(x[r] * y[j * M + cols[s]]) for s in keep]
            assert values[r, 2 * j:2 * j + 2].tobytes() == np.array(want, dtype=np.float16).tobytes()
            assert _slots_of(meta[r], 2 * (K // M))[2 * j:2 * j + 2] == keep


def check_gemm_compress_rounding(L):
    """W is rounded once, to nearest even: exact sums halfway between two
    fp16 values (1 + 2^-11, 1 + 3 * 2^-11, 1 - 2^-12, 2049) go to the even
    neighbour (1, 1 + 2^-9, 1, 2048); an fp16 overflow is non-finite."""
    X = np.array([[1, 2.0 ** -11], [1, 3 * 2.0 ** -11], [1, -(2.0 ** -12)], [2048, 1]], dtype=np.float16)
    Y = np.zeros((4, 2), dtype=np.float16)
    Y[0] = [1, 1]
    W, (values, meta, colidx) = oracle.gemm_compress(X, Y, 1, 4, L)
    want = np.array([1.0, 1 + 2.0 ** -9, 1.0, 2048.0], dtype=np.float16)
    assert W[:, 0].tobytes() == want.tobytes()
    assert not W[:, 1:].any()
    # each row keeps column 0 and the lowest of the zero columns
    assert values[:, 0].tobytes() == want.tobytes() and not values[:, 1].any()
    with pytest.raises(oracle.OracleError) as e:
        oracle.gemm_compress(np.full((4, 1), 256, np.float16), np.full((4, 1), 256, np.float16), 1, 4, L)
    assert e.value.code == oracle.NONFINITE


def check_energy_worked_example(L):
    """The 2 x 8 matrix of the 2:4 notes' worked example at density 1/2: V:N:M
    (V = 2, 2:4) keeps the printed values 0.9 -0.4 0.7 -1.2 / 0.3 0.5 -0.8 0.6;
    unstructured keeps the 8 largest magnitudes 1.2 0.9 0.8 0.7 0.6 0.5 0.4 0.4;
    vector-wise (one panel of both rows) keeps the 4 columns of largest L1
    norm, columns 7, 0, 5, 2 (norms 1.8, 1.1, 1.1, 0.9)."""
    fx = read_fixture(os.path.join(GOLDEN, "worked_2x8.txt"))
    W = np.array([_floats(fx["dense_row0"]), _floats(fx["dense_row1"])], dtype=np.float16)
    h = lambda xs: sum(abs(float(np.float16(x))) for x in xs)  # noqa: E731
    total = h(_floats(fx["dense_row0"]) + _floats(fx["dense_row1"]))
    want = {oracle.PATTERN_VNM: h([0.9, -0.4, 0.7, -1.2, 0.3, 0.5, -0.8, 0.6]),
            oracle.PATTERN_UNSTRUCTURED: h([1.2, 0.9, 0.8, 0.7, 0.6, 0.5, 0.4, 0.4]),
            oracle.PATTERN_VECTORWISE: h([1.2, 0.6, 0.9, 0.2, 0.7, 0.4, -0.4, 0.5])}
    for pattern, kept in want.items():
        e, k_units, t_units = oracle.energy(W, 2, 4, pattern, L)
        assert k_units == round(kept * 2 ** 24) and t_units == round(total * 2 ** 24), (pattern, k_units, t_units)
        assert abs(e - kept / total) < 1e-15


def check_energy_invariants(L):
    """Equal magnitudes keep exactly the density 2/M; on any matrix the
    unstructured selection (the ideal) keeps at least as much as V:N:M and
    vector-wise; V:N:M with V = 1 and M = 4 equals the sum of the two largest
    |w| of every group of 4 (brute force)."""
    rng = np.random.default_rng(11)
    R, K = 64, 128
    ones = (rng.choice([-1.0, 1.0], (R, K))).astype(np.float16)
    for M in (4, 8, 16):
        for pattern in (oracle.PATTERN_VNM, oracle.PATTERN_UNSTRUCTURED, oracle.PATTERN_VECTORWISE):
            e, kept, total = oracle.energy(ones, 16, M, pattern, L)
            assert kept * M == total * 2, (M, pattern)
    W = (rng.standard_normal((R, K)) * 0.02).astype(np.float16)
    for V, M in ((16, 8), (64, 16), (1, 4)):
        ideal = oracle.energy(W, V, M, oracle.PATTERN_UNSTRUCTURED, L)[1]
        assert ideal >= oracle.energy(W, V, M, oracle.PATTERN_VNM, L)[1]
        assert ideal >= oracle.energy(W, V, M, oracle.PATTERN_VECTORWISE, L)[1]
    groups = np.abs(W.astype(np.float64)).reshape(R, K // 4, 4)
    brute = np.sort(groups, axis=2)[:, :, 2:].sum()
    assert oracle.energy(W, 1, 4, oracle.PATTERN_VNM, L)[1] == round(brute * 2 ** 24)


def check_linear_worked_row(L):
    """The worked row 0 of the 2:4 notes as a one-output Linear layer: y =
    0.9 x0 - 0.4 x2 + 0.7 x5 - 1.2 x7 + bias, then ReLU or GELU; GELU(y) -
    GELU(-y) = y and GELU(0) = 0 (x * Phi(x) with Phi(-x) = 1 - Phi(x))."""
    fx = read_fixture(os.path.join(GOLDEN, "worked_2x8.txt"))
    W = np.array([_floats(fx["dense_row0"])], dtype=np.float16)
    values, meta, colidx = oracle.compress(W, 1, 4, L)
    X = np.array([[1, 2, 3, 4, 5, 6, 7, 8], [-1, 0.5, 2, 0, 0, -3, 1, 0.25]], dtype=np.float16)
    f = lambda x: float(np.float16(x))  # noqa: E731
    want = np.array([f(0.9) * x[0] - f(0.4) * x[2] + f(0.7) * x[5] - f(1.2) * x[7] for x in X.astype(np.float64)])
    bias = np.array([0.5], dtype=np.float16)
    y = oracle.linear(values, meta, colidx, 1, 8, 1, 4, X, bias)
    assert np.allclose(y[:, 0], want + 0.5, rtol=0, atol=1e-12)
    assert np.allclose(oracle.linear(values, meta, colidx, 1, 8, 1, 4, X, bias, oracle.ACT_RELU)[:, 0],
                       np.maximum(want + 0.5, 0), rtol=0, atol=1e-12)
    g = oracle.linear(values, meta, colidx, 1, 8, 1, 4, X, bias, oracle.ACT_GELU)[:, 0]
    gneg = oracle.linear(values, meta, colidx, 1, 8, 1, 4, -X, -bias, oracle.ACT_GELU)[:, 0]
    assert np.allclose(g - gneg, want + 0.5, rtol=0, atol=1e-12)
    zero = oracle.linear(values, meta, colidx, 1, 8, 1, 4, np.zeros((1, 8), np.float16), None, oracle.ACT_GELU)
    assert zero[0, 0] == 0.0
    # GELU(1) = Phi(1), the standard normal distribution function at 1 (erf form, not the tanh approximation)
    one = oracle.linear(values, meta, colidx, 1, 8, 1, 4, np.zeros((1, 8), np.float16), np.ones(1, np.float16),
                        oracle.ACT_GELU)
    assert abs(one[0, 0] - 0.8413447460685429) < 1e-12


def check_bitmap_format(L):
    """The bitmap format on a hand-made 64 x 3 matrix: column 0 holds 1 at
    row 0, -2 at row 5 and 3 at row 63 (bitmap bits 0, 5, 63; three values
    padded to 8); column 1 only -0.0 (no bit, no values); column 2 is full
    (all 64 bits, 64 values). Offsets 0, 8, 8; the length 72. An all-zero
    matrix has no values; a matrix without zeros has full tiles and no
    padding. Then random matrices of 30-70% zeros decode back to themselves
    (-0.0 as +0.0), and the product equals numpy's of the dense matrix."""
    W = np.zeros((64, 3), dtype=np.float16)
    W[0, 0], W[5, 0], W[63, 0] = 1, -2, 3
    W[7, 1] = -0.0
    W[:, 2] = np.arange(1, 65)
    bm, off, bases, vals = oracle.bitmap_encode(W)
    assert int(bm[0, 0]) == (1 | 1 << 5 | 1 << 63) and int(bm[0, 1]) == 0 and int(bm[0, 2]) == (1 << 64) - 1
    assert off[0].tolist() == [0, 8, 8] and bases.tolist() == [0, 72]
    assert vals.view(np.float16)[:8].tolist() == [1, -2, 3, 0, 0, 0, 0, 0]
    assert vals.view(np.float16)[8:].tolist() == list(range(1, 65))
    # no non-zero at all: empty values, every offset and base 0; no zero at all: full tiles, no padding
    bm, off, bases, vals = oracle.bitmap_encode(np.zeros((128, 5), np.float16))
    assert not bm.any() and not off.any() and bases.tolist() == [0, 0, 0] and vals.size == 0
    full = np.arange(1, 64 * 3 + 1, dtype=np.float16).reshape(64, 3)
    bm, off, bases, vals = oracle.bitmap_encode(full)
    assert all(int(b) == (1 << 64) - 1 for b in bm[0]) and off[0].tolist() == [0, 64, 128]
    assert bases.tolist() == [0, 192] and vals.view(np.float16)[64:128].tolist() == full[:, 1].tolist()
    rng = np.random.default_rng(13)
    for sparsity in (0.3, 0.5, 0.7):
        D = (rng.standard_normal((128, 40)) * (rng.random((128, 40)) >= sparsity)).astype(np.float16)
        D[3, 4] = -0.0
        enc = oracle.bitmap_encode(D)
        back = oracle.bitmap_decode(*enc, 128, 40)
        assert np.array_equal(back.astype(np.float64), D.astype(np.float64))
        assert int(enc[2][-1]) == sum((int(c) + 7) // 8 * 8 for c in (D.reshape(2, 64, 40) != 0).sum(axis=1).ravel())
        B = rng.standard_normal((40, 5)).astype(np.float16)
        assert np.allclose(oracle.bitmap_spmm(*enc, 128, 40, B), D.astype(np.float64) @ B.astype(np.float64),
                           rtol=0, atol=1e-12)


PINS = [check_worked_example, check_worked_local_index, check_worked_product,
        check_storage_arithmetic, check_brute_force_ties, check_brute_force_subnormals,
        check_brute_force_normal, check_invariants_and_round_trip, check_spmm_against_numpy,
        check_fig3_fixture, check_gemm_compress_identity, check_gemm_compress_rank1,
        check_gemm_compress_rounding, check_energy_worked_example, check_energy_invariants,
        check_linear_worked_row, check_bitmap_format]


# ----------------------------------------------------------------------------
# tests
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.lib())


def test_nonfinite_rejected():
    L = oracle.lib()
    for bad in (np.inf, -np.inf, np.nan):
        W = inputs.normal_f16((8, 16), 1, 0, 0.02)
        W[3, 5] = bad
        with pytest.raises(oracle.OracleError) as e:
            oracle.compress(W, 4, 8, L)
        assert e.value.code == oracle.NONFINITE


@pytest.mark.parametrize("R,K,V,M", [(10, 16, 4, 8), (8, 18, 4, 8), (8, 16, 4, 3), (8, 512, 4, 257),
                                     (8192, 16, 8192, 8), (8, 16, 0, 8)])
def test_invalid_shapes(R, K, V, M):
    with pytest.raises(oracle.OracleError) as e:
        oracle.sizes(R, K, V, M)
    assert e.value.code == oracle.INVALID


def test_empty_inputs():
    L = oracle.lib()
    assert oracle.sizes(0, 64, 16, 8, L) == (0, 0, 0)
    v, m, c = oracle.compress(np.zeros((0, 64), dtype=np.float16), 16, 8, L)
    assert v.shape == (0, 16) and m.shape == (0, 4) and c.shape == (0, 8, 4)
    v, m, c = oracle.compress(np.zeros((16, 0), dtype=np.float16), 16, 8, L)
    assert v.shape == (16, 0) and c.shape == (1, 0, 4)
    C = oracle.spmm(v, m, c, 16, 0, 16, 8, np.zeros((0, 5), dtype=np.float16), L=L)
    assert C.shape == (16, 5) and not C.any()


def test_generator_matches_its_definition():
    """The shared input generator against a scalar restatement of SplitMix64."""
    mask = (1 << 64) - 1

    def mix(z):
        z ^= z >> 30
        z = (z * 0xBF58476D1CE4E5B9) & mask
        z ^= z >> 27
        z = (z * 0x94D049BB133111EB) & mask
        return z ^ (z >> 31)

    seed, stream = 1002, 3
    key = mix((seed * 0x9E3779B97F4A7C15) & mask) ^ mix(((stream + 1) * 0xD1B54A32D192ED03) & mask)
    want = [mix((key + (i + 1) * 0x9E3779B97F4A7C15) & mask) for i in range(8)]
    assert inputs.raw_u64(seed, stream, 0, 8).tolist() == want
    assert inputs.raw_u64(seed, stream, 5, 3).tolist() == want[5:]
    x = inputs.normal_f16((1 << 16,), 1, 0, 0.02).astype(np.float64)
    assert abs(x.mean()) < 3e-4 and abs(x.std() - 0.02) < 3e-4
    # any chunk boundary gives the same stream
    big = inputs.normal_range(0, 1000, 9, 2)
    assert np.array_equal(inputs.normal_range(400, 1000, 9, 2), big[400:])


# planted mistakes: (description, regex on the oracle source, replacement)
MUTANTS = [
    ("ties go to the higher index", r"score\[c\] > score\[best\]", "score[c] >= score[best]"),
    ("keep the smallest instead of the largest", r"score\[c\] > score\[best\]", "score[c] < score[best]"),
    ("m-index fields packed MSB first", r"\(uint8_t\)\(slot << \(2 \* \(t % 4\)\)\)",
     "(uint8_t)(slot << (2 * (3 - t % 4)))"),
    ("column-loc not sorted", r"out\[b - 1\] > out\[b\]", "0"),
    ("signed instead of absolute column sums", r"s \+= fabs\(half_to_double", "s += (half_to_double"),
    ("column-loc slot reversed on decompress", r"colidx\[\(i \* nblk \+ j\) \* 4 \+ slot\]",
     "colidx[(i * nblk + j) * 4 + (3 - slot)]"),
    ("SpMM drops the last k", r"for \(int64_t k = 0; k < K; \+\+k\) \{\n                const double ak",
     "for (int64_t k = 0; k < K - 1; ++k) {\n                const double ak"),
    ("subnormal scale off by one", r"ldexp\(\(double\)f, -24\)", "ldexp((double)f, -25)"),
    ("values taken from the unselected column", r"W\[row \* ld_w \+ j \* M \+ sel\[keep\[t\]\]\]",
     "W[row * ld_w + j * M + keep[t]]"),
]


def test_mutants_are_caught(tmp_path):
    """Every planted mistake in a copy of the oracle fails at least one pin."""
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "vnm_oracle.c")).read()
    for k, (what, pat, rep) in enumerate(MUTANTS):
        new, n = re.subn(pat, rep, src, count=1)
        assert n == 1, f"mutant pattern not found: {what}"
        path = tmp_path / f"mutant{k}.c"
        path.write_text(new)
        so = str(tmp_path / f"libmutant{k}.so")
        oracle.build(str(path), so)
        L = oracle.load_from(so)
        failed = []
        for pin in PINS:
            try:
                pin(L)
            except (AssertionError, oracle.OracleError, IndexError, ValueError):
                failed.append(pin.__name__)
        assert failed, f"no pin caught the planted mistake: {what}"


# Planted mistakes in the oracle's Python functions (the Linear form, the
# energy and the bitmap format): (what, pattern in oracle/__init__.py,
# replacement, the function it lands in).
PY_MUTANTS = [
    ("bitmap bits MSB-first", r"np\.uint64\(sum\(1 << r for r in rows\)\)",
     "np.uint64(sum(1 << (63 - r) for r in rows))", "bitmap_encode"),
    ("bitmap values not padded", r"padded = \(len\(rows\) \+ 7\) // 8 \* 8", "padded = len(rows)", "bitmap_encode"),
    ("bitmap counts -0.0 as a non-zero", r"if int\(col\[r\]\) & 0x7FFF\]", "if int(col[r])]", "bitmap_encode"),
    ("bitmap decode ignores the row block's base", r"at = int\(bases\[i\]\) \+ int\(offsets\[i, k\]\)",
     "at = int(offsets[i, k])", "bitmap_decode"),
    ("unstructured keeps the smallest", r"flat = np\.sort\(u\.ravel\(\)\)\[::-1\]", "flat = np.sort(u.ravel())",
     "energy"),
    ("vector-wise ranks columns by their largest |w|",
     r"col = u\[i \* V:\(i \+ 1\) \* V\]\.sum\(axis=0, dtype=np\.uint64\)",
     "col = u[i * V:(i + 1) * V].max(axis=0)", "energy"),
    ("GELU by the tanh approximation",
     r"Y = Y \* \(1\.0 \+ np\.vectorize\(math\.erf\)\(Y / math\.sqrt\(2\.0\)\)\) / 2\.0",
     "Y = 0.5 * Y * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (Y + 0.044715 * Y ** 3)))", "linear"),
    ("bias dropped", r"Y \+= np\.asarray\(bias, dtype=np\.float16\)", "Y += 0 * np.asarray(bias, dtype=np.float16)",
     "linear"),
]


def test_python_mutants_are_caught(monkeypatch):
    """Every planted mistake in the oracle's Python functions fails at least
    one pin (the mutated function replaces the oracle's for the run)."""
    path = os.path.join(os.path.dirname(oracle.__file__), "__init__.py")
    src = open(path).read()
    L = oracle.lib()
    for what, pat, rep, fn in PY_MUTANTS:
        new, n = re.subn(pat, rep, src, count=1)
        assert n == 1, f"mutant pattern not found: {what}"
        ns = {"__name__": "oracle_mutant", "__file__": path}
        exec(compile(new, path, "exec"), ns)
        failed = []
        with monkeypatch.context() as m:
            m.setattr(oracle, fn, ns[fn])
            for pin in PINS:
                try:
                    pin(L)
                except (AssertionError, oracle.OracleError, IndexError, ValueError):
                    failed.append(pin.__name__)
        assert failed, f"no pin caught the planted mistake: {what}"
