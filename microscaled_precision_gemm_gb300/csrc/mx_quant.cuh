// MXFP6 encoding of fp32 values, shared by the fused epilogues of the GEMM and
// the fused normalisation quantizer. The rule is the quantizer's (OCP MX v1.0
// conversion): amax over 32 values; E8M0 code = max(floor(log2 amax) - 2, -127)
// + 127; each value times 2^-s rounded to the nearest E2M3 value, ties to even,
// saturating at +-7.5; a block holding Inf/NaN gets code 0xFF and zero codes.
#pragma once

#include <cstdint>

#include "mx_layout.cuh"
#include "ptx.cuh"

namespace mxk {

// Three- and two-input maxima, NaN if any input is NaN (PTX max.NaN).
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Block amax of 32 fp32 values as magnitude bits: +0 .. 0x7F7FFFFF finite, 0x7F800000
// Inf, above that NaN (max.NaN returns the canonical NaN 0x7FFFFFFF). A tree of
// three-input maxima of |v| (the absolute value folds into the max): 32 -> 11 -> 4 -> 1.
__device__ __forceinline__ uint32_t amax_bits32(const float (&g)[32]) {
  float m[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) m[i] = max3_nan(fabsf(g[3 * i]), fabsf(g[3 * i + 1]), fabsf(g[3 * i + 2]));
  m[10] = max_nan(fabsf(g[30]), fabsf(g[31]));
  const float n0 = max3_nan(m[0], m[1], m[2]);
  const float n1 = max3_nan(m[3], m[4], m[5]);
  const float n2 = max3_nan(m[6], m[7], m[8]);
  const float n3 = max_nan(m[9], m[10]);
  return __float_as_uint(max_nan(max3_nan(n0, n1, n2), n3));
}

// Four values (already scaled by 2^-s) -> their E2M3 codes, one per byte (value i
// in byte i): two paired converts joined into one 32-bit register.
__device__ __forceinline__ uint32_t cvt_e2m3x4(float a0, float a1, float a2, float a3) {
  uint32_t q;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e2m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(q)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return q;
}

// Four codes one per byte (c0 | c1 << 8 | c2 << 16 | c3 << 24) -> the 24-bit group
// c0 | c1 << 6 | c2 << 12 | c3 << 18: per 16-bit half c + 256 c' - 192 c' = c + 64 c',
// then lo + 65536 hi - 61440 hi = lo + 4096 hi.
__device__ __forceinline__ uint32_t pack_codes4(uint32_t q) {
  const uint32_t odd = __byte_perm(q, 0u, 0x4341u);   // c1 | c3 << 16
  const uint32_t t = q - 192u * odd;
  return t - 61440u * (t >> 16);
}

// Eight 24-bit groups (32 codes) -> the six little-endian words of their 24 bytes
// (group j at bits [24 j, 24 j + 24) of the block's bit string).
__device__ __forceinline__ void pack_groups(const uint32_t (&grp)[8], uint32_t (&w)[6]) {
  w[0] = grp[0] + (grp[1] << 24);
  w[1] = (grp[1] >> 8) + (grp[2] << 16);
  w[2] = (grp[2] >> 16) + (grp[3] << 8);
  w[3] = grp[4] + (grp[5] << 24);
  w[4] = (grp[5] >> 8) + (grp[6] << 16);
  w[5] = (grp[6] >> 16) + (grp[7] << 8);
}

// MXFP6 encoding of one 32-value block: returns the E8M0 code and the block's 24
// code bytes as six little-endian words (the quantizer's rule, on fp32 values).
__device__ __forceinline__ uint32_t quant_block32(const float (&g)[32], uint32_t (&w)[6]) {
  const uint32_t amax = amax_bits32(g);
  if (amax >= 0x7F800000u) {  // Inf or NaN: E8M0 NaN, zero codes
#pragma unroll
    for (int i = 0; i < 6; ++i) w[i] = 0;
    return 0xFFu;
  }
  const int e = static_cast<int>(amax >> 23);
  const uint32_t sc = static_cast<uint32_t>(e > 2 ? e - 2 : 0);
  const float fac = __uint_as_float((254u - sc) << 23);  // 2^-s, exact
  const uint64_t fac2 = f2_pack(fac, fac);
  uint32_t grp[8];   // 24-bit groups of four codes
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float t0, t1, t2, t3;   // the values times 2^-s (exact), two per packed multiply
    f2_unpack(f2_mul(f2_pack(g[4 * j], g[4 * j + 1]), fac2), t0, t1);
    f2_unpack(f2_mul(f2_pack(g[4 * j + 2], g[4 * j + 3]), fac2), t2, t3);
    grp[j] = pack_codes4(cvt_e2m3x4(t0, t1, t2, t3));
  }
  pack_groups(grp, w);
  return sc;
}

}  // namespace mxk
