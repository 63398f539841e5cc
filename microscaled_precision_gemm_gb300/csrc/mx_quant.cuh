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

// MXFP6 encoding of one 32-value block: returns the E8M0 code and the block's 24
// code bytes as six little-endian words (the quantizer's rule, on fp32 values).
__device__ __forceinline__ uint32_t quant_block32(const float (&g)[32], uint32_t (&w)[6]) {
  // |g| order = unsigned order of the magnitude bits (NaN/Inf sort last); a tree keeps it shallow
  uint32_t m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    m[i] = max(__float_as_uint(g[2 * i]) & 0x7FFFFFFFu, __float_as_uint(g[2 * i + 1]) & 0x7FFFFFFFu);
#pragma unroll
  for (int w2 = 8; w2 >= 1; w2 >>= 1)
#pragma unroll
    for (int i = 0; i < w2; ++i) m[i] = max(m[i], m[i + w2]);
  const uint32_t amax = m[0];
  if (amax >= 0x7F800000u) {  // Inf or NaN: E8M0 NaN, zero codes
#pragma unroll
    for (int i = 0; i < 6; ++i) w[i] = 0;
    return 0xFFu;
  }
  const int e = static_cast<int>(amax >> 23);
  const uint32_t sc = static_cast<uint32_t>(e > 2 ? e - 2 : 0);
  const float fac = __uint_as_float((254u - sc) << 23);  // 2^-s, exact
  uint32_t grp[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t lo = cvt_e2m3x2(g[4 * j + 1] * fac, g[4 * j] * fac);
    const uint32_t hi = cvt_e2m3x2(g[4 * j + 3] * fac, g[4 * j + 2] * fac);
    grp[j] = pack4(lo | (hi << 16));
  }
  pack32(grp, w);
  return sc;
}

}  // namespace mxk
