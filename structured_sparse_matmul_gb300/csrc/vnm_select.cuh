// Device-side selection rules of the V:N:M magnitude pruning, shared by the
// compress kernels and the fused GEMM + prune-and-encode kernel.
//
// VENOM: A Vectorized N:M Format for Unleashing the Power of Sparse Tensor
// Cores, section 3, Figure 2: per V x M block keep the 4 most significant
// columns (here: largest exact L1 norm over the block's rows, lower column
// on ties), then per row 2 of those 4 (largest |w|, lower slot on ties).
#pragma once

#include <stdint.h>

namespace vnm {

// |h| in units of 2^-24 (binary16: 5 exponent bits, bias 15, 10 fraction bits).
__device__ __forceinline__ uint64_t mag_units(uint16_t h) {
    const uint32_t e = (h >> 10) & 0x1Fu, f = h & 0x3FFu;
    return e == 0 ? static_cast<uint64_t>(f) : static_cast<uint64_t>(1024u + f) << (e - 1u);
}

__device__ __forceinline__ bool half_nonfinite(uint16_t h) { return (h & 0x7C00u) == 0x7C00u; }

// The 4 largest of a stream of (score, index) pairs offered in increasing
// index order: largest first, the lower index first on ties (a later equal
// score never displaces an earlier one). Registers only: the four best keys
// (score + 1; 0 = empty) shift down as a larger key arrives.
struct Top4 {
    uint64_t k0 = 0, k1 = 0, k2 = 0, k3 = 0;
    uint32_t i0 = 0, i1 = 0, i2 = 0, i3 = 0;

    __device__ __forceinline__ void offer(uint64_t score, uint32_t c) {
        const uint64_t k = score + 1;
        if (k <= k3) return;
        if (k > k2) {
            k3 = k2;
            i3 = i2;
            if (k > k1) {
                k2 = k1;
                i2 = i1;
                if (k > k0) {
                    k1 = k0;
                    i1 = i0;
                    k0 = k;
                    i0 = c;
                } else {
                    k1 = k;
                    i1 = c;
                }
            } else {
                k2 = k;
                i2 = c;
            }
        } else {
            k3 = k;
            i3 = c;
        }
    }

    // the four indices ascending (a sorting network of 5 compare-exchanges),
    // packed in bytes 0..3
    __device__ __forceinline__ uint32_t word() const {
        uint32_t a = i0, b = i1, c = i2, d = i3;
        auto cx = [](uint32_t& x, uint32_t& y) {
            const uint32_t lo = min(x, y), hi = max(x, y);
            x = lo;
            y = hi;
        };
        cx(a, b);
        cx(c, d);
        cx(a, c);
        cx(b, d);
        cx(b, c);
        return a | (b << 8) | (c << 16) | (d << 24);
    }
};

// Top 4 of n >= 4 scores as 4 ascending column indices packed in bytes 0..3.
__device__ __forceinline__ uint32_t top4_ascending(const uint64_t* score, int n) {
    Top4 t;
    for (int c = 0; c < n; ++c) t.offer(score[c], static_cast<uint32_t>(c));
    return t.word();
}

// 2 of the 4 values a[0..3] with the largest |a| (lower slot on ties), in
// ascending slot order. Returns the 4-bit code s0 | s1 << 2 and the two
// fp16 bit patterns. Branch-free: slot i is kept when fewer than two slots
// beat it, slot j < i beating i when |a_j| >= |a_i| and slot j > i when
// |a_j| > |a_i| (finite fp16 magnitudes order like their integer bits).
__device__ __forceinline__ uint32_t keep2of4(const uint16_t a[4], uint16_t& v0, uint16_t& v1) {
    const uint32_t m0 = a[0] & 0x7FFFu, m1 = a[1] & 0x7FFFu, m2 = a[2] & 0x7FFFu, m3 = a[3] & 0x7FFFu;
    const uint32_t g01 = m0 >= m1, g02 = m0 >= m2, g03 = m0 >= m3;
    const uint32_t g12 = m1 >= m2, g13 = m1 >= m3, g23 = m2 >= m3;
    const uint32_t r0 = (1u - g01) + (1u - g02) + (1u - g03);
    const uint32_t r1 = g01 + (1u - g12) + (1u - g13);
    const uint32_t r2 = g02 + g12 + (1u - g23);
    const uint32_t r3 = g03 + g13 + g23;
    const uint32_t keep = (r0 < 2u) | ((r1 < 2u) << 1) | ((r2 < 2u) << 2) | ((r3 < 2u) << 3);
    const uint32_t s0 = __ffs(keep) - 1u;  // exactly two bits are set
    const uint32_t s1 = 31u - __clz(keep);
    v0 = s0 == 0u ? a[0] : (s0 == 1u ? a[1] : a[2]);
    v1 = s1 == 3u ? a[3] : (s1 == 2u ? a[2] : a[1]);
    return s0 | (s1 << 2);
}

}  // namespace vnm
