"""Seeded synthetic inputs, shared by the oracle tests, the GPU tests and bench.py.

This module draws numbers and nothing else: it holds none of the V:N:M
method's arithmetic (no pruning, packing or products), so that the CPU oracle
and the CUDA path can both read the same host buffers without sharing code.

Generator (counter-based, so any element can be drawn independently):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): ``x_i = mix64(key + (i + 1) * GAMMA)`` with
  ``GAMMA = 0x9E3779B97F4A7C15`` and the published finaliser
  ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
  z *= 0x94D049BB133111EB; z ^= z >> 31``.
* The key of stream ``s`` under seed ``seed`` is
  ``mix64(seed * GAMMA) ^ mix64((s + 1) * 0xD1B54A32D192ED03)``.
* Uniforms in (0, 1): ``((x >> 11) + 0.5) * 2**-53``.
* Normals: Box and Muller (1958), in float64, from the uniform pair
  ``(u_{2p}, u_{2p+1})``: element ``2p`` takes the cosine branch and element
  ``2p + 1`` the sine branch.
* fp16 values: ``sigma * normal`` in float64, rounded once to binary16 with
  round-to-nearest-even (numpy's float64 -> float16 conversion).

The draws are bit-stable on one platform. Across CPU architectures the
float64 ``log``/``cos``/``sin`` of numpy may differ in the last ulp, which can
move an fp16 rounding in rare elements; every test and the benchmark generate
their inputs in the same process that checks them, so nothing depends on that.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    _mix64_inplace(z, np.empty_like(z))
    return z


def _mix64_inplace(z: np.ndarray, tmp: np.ndarray) -> None:
    with np.errstate(over="ignore"):
        np.right_shift(z, np.uint64(30), out=tmp)
        np.bitwise_xor(z, tmp, out=z)
        np.multiply(z, _M1, out=z)
        np.right_shift(z, np.uint64(27), out=tmp)
        np.bitwise_xor(z, tmp, out=z)
        np.multiply(z, _M2, out=z)
        np.right_shift(z, np.uint64(31), out=tmp)
        np.bitwise_xor(z, tmp, out=z)


def stream_key(seed: int, stream: int) -> np.uint64:
    """Key of one named stream of draws under one seed."""
    with np.errstate(over="ignore"):
        a = mix64(np.array([seed], dtype=np.uint64) * GAMMA)[0]
        b = mix64(np.array([stream + 1], dtype=np.uint64) * _STREAM_MUL)[0]
    return np.uint64(a ^ b)


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of one stream, as uint64."""
    key = stream_key(seed, stream)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(key + idx * GAMMA)


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform float64 draws in the open interval (0, 1)."""
    x = raw_u64(seed, stream, start, count)
    return ((x >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal_range(c0: int, c1: int, seed: int, stream: int) -> np.ndarray:
    """Standard normal float64 draws ``c0 .. c1-1`` of one stream (``c0`` even)."""
    if c0 % 2:
        raise ValueError("normal_range starts on a pair boundary")
    n = c1 - c0
    npairs = (n + 1) // 2
    out = np.empty(2 * npairs, dtype=np.float64)
    key = stream_key(seed, stream)
    blk = 1 << 15  # pairs per block: keeps the temporaries in cache
    z = np.empty(2 * blk, dtype=np.uint64)
    tmp = np.empty(2 * blk, dtype=np.uint64)
    u = np.empty(2 * blk, dtype=np.float64)
    rad = np.empty(blk, dtype=np.float64)
    ang = np.empty(blk, dtype=np.float64)
    with np.errstate(over="ignore"):
        for p0 in range(0, npairs, blk):
            m = min(blk, npairs - p0)
            zz, tt, uu = z[: 2 * m], tmp[: 2 * m], u[: 2 * m]
            # counters c0 + 2*p0 + 1 ... (1-based draw index)
            zz[:] = np.arange(c0 + 2 * p0 + 1, c0 + 2 * (p0 + m) + 1, dtype=np.uint64)
            np.multiply(zz, GAMMA, out=zz)
            np.add(zz, key, out=zz)
            _mix64_inplace(zz, tt)
            np.right_shift(zz, np.uint64(11), out=zz)
            uu[:] = zz
            uu += 0.5
            uu *= 2.0 ** -53
            r, g = rad[:m], ang[:m]
            np.log(uu[0::2], out=r)
            r *= -2.0
            np.sqrt(r, out=r)
            np.multiply(uu[1::2], 2.0 * np.pi, out=g)
            dst = out[2 * p0: 2 * (p0 + m)]
            np.cos(g, out=dst[0::2])
            dst[0::2] *= r
            np.sin(g, out=dst[1::2])
            dst[1::2] *= r
    return out[:n]


def normal_f16(shape, seed: int, stream: int, sigma: float) -> np.ndarray:
    """fp16 array of ``shape`` drawn from N(0, sigma), row-major, RNE-rounded."""
    shape = tuple(int(s) for s in shape)
    count = int(np.prod(shape)) if shape else 1
    out = np.empty(count, dtype=np.float16)
    step = 1 << 24  # even, so every chunk starts on a pair boundary
    for c0 in range(0, count, step):
        c1 = min(count, c0 + step)
        out[c0:c1] = (sigma * normal_range(c0, c1, seed, stream)).astype(np.float16)
    return out.reshape(shape)


def choice_f16(shape, seed: int, stream: int, choices) -> np.ndarray:
    """fp16 array whose elements are drawn uniformly from ``choices``.

    Used for tie-heavy inputs (for example ``{0, +-0.5, +-1}``), where many
    column sums and magnitudes are equal and the tie rules decide.
    """
    shape = tuple(int(s) for s in shape)
    count = int(np.prod(shape)) if shape else 1
    table = np.asarray(choices, dtype=np.float16)
    x = raw_u64(seed, stream, 0, count)
    pick = (x % np.uint64(len(table))).astype(np.int64)
    return table[pick].reshape(shape)
