// sampling_math.cuh -- numeric helpers shared by the sampler and the
// speculative-decoding verifier: order-preserving float keys, 2^-40 fixed-point
// masses of temperature weights (exact integer sums, so every cut and every
// draw is deterministic), exact ceil(p * S), and the Philox4x64-10 generator.
#pragma once

#include <stdint.h>

namespace pkv {

// ------------------------------------------------------------------ numeric helpers
// Order-preserving key of a float (larger float -> larger key); -0.0 is folded
// onto +0.0 so that equal logits have equal keys.
__device__ __forceinline__ uint32_t okey(float z) {
    uint32_t u = __float_as_uint(z);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}
// floor(w * 2^40) for w in [0, 1], from the bits of w with integer ALU
// operations (a float -> 64-bit integer conversion is a slow multi-cycle
// operation, and the sampler takes one per logit): a normal w is m * 2^(e-150)
// with m its 24-bit significand (implicit 1 included), so w * 2^40 =
// m * 2^(e-110); a left shift (e >= 110) is exact, a right shift drops exactly
// the fraction, and zero or subnormal w (e = 0) gives 0.  The same value as
// truncating w * 2^40, which is exact in float.
__device__ __forceinline__ uint64_t fx40(float w) {
    const uint32_t u = __float_as_uint(w);
    const uint64_t m = (u & 0x7fffffu) | 0x800000u;
    const int sh = static_cast<int>(u >> 23) - 110;
    return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0ull);
}
// floor(w * 2^24) = fx40(w) >> 16, in 32 bits by the same construction.
__device__ __forceinline__ uint32_t fx24(float w) {
    const uint32_t u = __float_as_uint(w);
    const uint32_t m = (u & 0x7fffffu) | 0x800000u;
    const int sh = static_cast<int>(u >> 23) - 126;
    return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0u);
}
// 2^x by the hardware's approximate base-2 exponential (subnormal results flush
// to zero; they are below 2^-40 and weigh nothing anyway).
__device__ __forceinline__ float hw_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Weight of a logit relative to the row maximum, w = 2^((z - zmax) * c2) with
// c2 = log2(e) / T clamped to a finite value, so that the maximum weighs 2^0 = 1
// and a banned (-inf) logit weighs 2^-inf = 0.
__device__ __forceinline__ float weight(float z, float zmax, float c2) { return hw_exp2((z - zmax) * c2); }
// Its 64-bit fixed-point mass floor(w * 2^40).
__device__ __forceinline__ uint64_t mass(float z, float zmax, float c2) { return fx40(weight(z, zmax, c2)); }
// Sort key with (z desc, id asc) as descending u64 order.
__device__ __forceinline__ uint64_t sort_key(float z, int id) {
    return (static_cast<uint64_t>(okey(z)) << 32) | static_cast<uint32_t>(0xffffffffu - static_cast<uint32_t>(id));
}
__device__ __forceinline__ int sort_key_id(uint64_t k) {
    return static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
}
// ceil(p * S) for p a float in (0, 1) and S < 2^63, exactly.
__device__ __forceinline__ uint64_t ceil_mul_p(float p, uint64_t S) {
    const uint32_t u = __float_as_uint(p);
    const int e = static_cast<int>((u >> 23) & 0xffu);
    const uint64_t m = e ? static_cast<uint64_t>((u & 0x7fffffu) | 0x800000u) : static_cast<uint64_t>(u & 0x7fffffu);
    const int sh = e ? 150 - e : 149;  // p = m * 2^-sh
    const unsigned __int128 N = static_cast<unsigned __int128>(m) * S;
    if (N == 0) return 0ull;
    if (sh >= 127) return 1ull;
    const unsigned __int128 one = 1;
    return static_cast<uint64_t>((N + ((one << sh) - 1)) >> sh);
}

// Philox4x64-10 (Salmon et al., SC'11) under key (seed, 0) at counter
// (offset, j, 0, 0), word 0 only.
__device__ __forceinline__ uint64_t philox_word0(uint64_t seed, uint64_t offset, uint64_t j = 0) {
    uint64_t x0 = offset, x1 = j, x2 = 0, x3 = 0;
    uint64_t k0 = seed, k1 = 0;
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint64_t lo0 = 0xD2E7470EE14C6C93ull * x0, hi0 = __umul64hi(0xD2E7470EE14C6C93ull, x0);
        const uint64_t lo1 = 0xCA5A826395121157ull * x2, hi1 = __umul64hi(0xCA5A826395121157ull, x2);
        const uint64_t y0 = hi1 ^ x1 ^ k0, y2 = hi0 ^ x3 ^ k1;
        x0 = y0;
        x1 = lo1;
        x2 = y2;
        x3 = lo0;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
    return x0;
}

}  // namespace pkv
