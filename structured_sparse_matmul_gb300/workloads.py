"""The five synthetic V:N:M workloads: shapes, sparsity patterns, dtypes, seeds.

Pure data (no arithmetic of the method). Shapes follow the experiments of
"VENOM: A Vectorized N:M Format for Unleashing the Power of Sparse Tensor
Cores" (BERT-large linear layers 1024 x 4096 and 4096 x 1024 with 16 x 512
tokens, section 7.1 / Figure 14; GPT-3-scale FFN layers, section 7.2) and the
decode-like small-N products of "Coruscant" (section 2, Llama-style 4096 and
11008 projections). A is R x K (sparse weights), B is K x N (dense
activations), C is R x N.

Values: A ~ N(0, 0.02), B ~ N(0, 1), both fp16 (round-to-nearest-even),
drawn by :mod:`structured_sparse_matmul_gb300.inputs` with seed
``1000 + index`` (index 1..5); A is stream ``2 * case`` and B stream
``2 * case + 1`` where ``case`` numbers the shapes inside one workload.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Tuple

A_SIGMA = 0.02
B_SIGMA = 1.0


@dataclass(frozen=True)
class Case:
    """One SpMM problem C[R x N] = A_vnm[R x K] . B[K x N]."""

    workload: int      # 1..5
    case: int          # index inside the workload
    R: int
    K: int
    N: int
    V: int
    M: int
    c_f32: bool        # C written as fp32 (else fp16)

    @property
    def seed(self) -> int:
        return 1000 + self.workload

    @property
    def a_stream(self) -> int:
        return 2 * self.case

    @property
    def b_stream(self) -> int:
        return 2 * self.case + 1

    @property
    def name(self) -> str:
        return (f"w{self.workload}.{self.case}:{self.R}x{self.K}x{self.N}"
                f"-{self.V}:2:{self.M}-{'f32' if self.c_f32 else 'f16'}")

    def dense_flops(self) -> float:
        """Dense-equivalent flops 2*R*N*K."""
        return 2.0 * self.R * self.N * self.K

    def effective_flops(self) -> float:
        """Flops on kept non-zeros only: 2*R*N*K*2/M."""
        return 2.0 * self.R * self.N * self.K * 2.0 / self.M


def workload_cases(w: int) -> List[Case]:
    """All cases of workload ``w`` (1..5)."""
    out: List[Case] = []
    if w == 1:
        # tiny plain 2:4 (V=16), fp32 C
        out.append(Case(1, 0, 256, 256, 64, 16, 4, True))
    elif w == 2:
        # square compute-bound: V=64, 2:8, fp16 C
        out.append(Case(2, 0, 4096, 4096, 2048, 64, 8, False))
    elif w == 3:
        # transformer-encoder linear sweep, V=128, M in {4, 8, 16}, 8192 tokens
        c = 0
        for (R, K) in ((1024, 4096), (4096, 1024)):
            for M in (4, 8, 16):
                out.append(Case(3, c, R, K, 8192, 128, M, False))
                c += 1
    elif w == 4:
        # decode-like memory-bound SpMM, V=64, M in {4, 8}, N in {1, 8, 16, 32}
        c = 0
        for (R, K) in ((4096, 4096), (11008, 4096), (4096, 11008)):
            for M in (4, 8):
                for N in (1, 8, 16, 32):
                    out.append(Case(4, c, R, K, N, 64, M, False))
                    c += 1
    elif w == 5:
        # large FFN-scale: V=128, M in {16, 32}
        for c, M in enumerate((16, 32)):
            out.append(Case(5, c, 49152, 12288, 4096, 128, M, False))
    else:
        raise ValueError(f"no workload {w}")
    return out


def all_cases() -> List[Case]:
    return [c for w in range(1, 6) for c in workload_cases(w)]


def shape_a(c: Case) -> Tuple[int, int]:
    return (c.R, c.K)


def shape_b(c: Case) -> Tuple[int, int]:
    return (c.K, c.N)
