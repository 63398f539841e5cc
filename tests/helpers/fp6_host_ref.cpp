// Test helper: CUDA's own host-side FP6 (E2M3) conversions from cuda_fp6.h,
// called as library routines to pin the oracle's table and rounding.
//   fp6_host_ref decode          -> prints the fp16 bit pattern of codes 0..63
//   fp6_host_ref encode < f32s   -> writes one code byte per input float
#include <cuda_fp6.h>
#include <cstdio>
#include <cstring>
#include <vector>

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  if (std::strcmp(argv[1], "decode") == 0) {
    for (int c = 0; c < 64; ++c) {
      __half_raw h = __nv_cvt_fp6_to_halfraw(static_cast<__nv_fp6_storage_t>(c), __NV_E2M3);
      std::printf("%u\n", static_cast<unsigned>(h.x));
    }
    return 0;
  }
  if (std::strcmp(argv[1], "encode") == 0) {
    std::vector<float> buf(1 << 16);
    size_t n;
    while ((n = std::fread(buf.data(), sizeof(float), buf.size(), stdin)) > 0) {
      std::vector<unsigned char> out(n);
      for (size_t i = 0; i < n; ++i)
        out[i] = static_cast<unsigned char>(__nv_cvt_float_to_fp6(buf[i], __NV_E2M3, cudaRoundNearest));
      std::fwrite(out.data(), 1, n, stdout);
    }
    return 0;
  }
  return 2;
}
