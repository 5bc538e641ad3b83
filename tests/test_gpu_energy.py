"""vnm_energy on the GPU against the CPU oracle: the energy (magnitude
preservation) of V:N:M, unstructured and vector-wise pruning at density 2/M
("VENOM", section 5, Figure 11). The kept and total sums are exact integers
(units of 2^-24) and must equal the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from structured_sparse_matmul_gb300 import inputs, vnm

pytestmark = pytest.mark.gpu

from gpu_util import device, gpu_compress, to_dev  # noqa: E402

PATTERNS = [(vnm.VNM_PATTERN_VNM, oracle.PATTERN_VNM), (vnm.VNM_PATTERN_UNSTRUCTURED, oracle.PATTERN_UNSTRUCTURED),
            (vnm.VNM_PATTERN_VECTORWISE, oracle.PATTERN_VECTORWISE)]


def _check(W, V, M, ld=None):
    A, st = gpu_compress(W, V, M, ld)
    assert st == vnm.VNM_OK
    Wd = to_dev(W, ld)
    for gp, op in PATTERNS:
        e, kept, total = vnm.vnm_energy(A, Wd, gp)
        oe, okept, ototal = oracle.energy(W, V, M, op)
        assert (kept, total) == (okept, ototal), (gp, kept - okept, total - ototal)
        assert e == pytest.approx(oe, rel=1e-15, abs=0)


@pytest.mark.parametrize("R,K,V,M", [(768, 768, 16, 4), (768, 768, 64, 8), (768, 768, 128, 16), (768, 768, 1, 32),
                                     (768, 960, 32, 40), (768, 960, 128, 20), (272, 520, 16, 8), (4096, 4096, 64, 8)])
def test_normal_weights(R, K, V, M):
    _check(inputs.normal_f16((R, K), 51, 0, 0.02), V, M)


def test_tie_heavy_and_padded_rows():
    rng = np.random.default_rng(52)
    W = rng.choice(np.array([0, 0.5, -0.5, 1, -1], dtype=np.float16), (256, 384))
    _check(W, 32, 8, ld=392)


def test_zero_and_nonfinite():
    R, K, V, M = 128, 256, 16, 8
    Z = np.zeros((R, K), np.float16)
    A, _ = gpu_compress(Z, V, M)
    for gp, _op in PATTERNS:
        assert vnm.vnm_energy(A, to_dev(Z), gp) == (1.0, 0, 0)
    W = inputs.normal_f16((R, K), 53, 0, 0.02)
    W[5, 7] = np.inf
    with pytest.raises(vnm.VnmError) as e:
        vnm.vnm_energy(A, to_dev(W), vnm.VNM_PATTERN_UNSTRUCTURED)
    assert e.value.code == vnm.VNM_ERR_NONFINITE


def test_workspace_checked():
    R, K, V, M = 128, 256, 16, 8
    W = inputs.normal_f16((R, K), 54, 0, 0.02)
    A, _ = gpu_compress(W, V, M)
    small = torch.empty(vnm.vnm_energy_workspace_size(A) - 16, dtype=torch.uint8, device=device())
    with pytest.raises(vnm.VnmError) as e:
        vnm.vnm_energy(A, to_dev(W), vnm.VNM_PATTERN_VECTORWISE, workspace=small)
    assert e.value.code == vnm.VNM_ERR_INVALID_ARG
