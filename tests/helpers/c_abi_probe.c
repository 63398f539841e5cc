/* Plain C11 caller of the library: include/mx.h must compile as C and every call
 * below must link and run without a GPU (size queries, status strings, host-side
 * argument checks and layout helpers). Prints one "name value" line per check. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "mx.h"

int main(void) {
  printf("version %d\n", mx_version());
  printf("codes_bytes %zu\n", mx_codes_bytes(128, 256));
  printf("scales_bytes %zu\n", mx_scales_bytes(300, 256));
  printf("workspace_bytes %zu\n", mx_mlp_workspace_bytes(256, 512, 1024));
  /* K % 128 != 0 is rejected before any device call */
  printf("bad_shape %d\n", (int)mx_quantize((const void*)0x10000, 128, 100, 100, (void*)0x20000, (void*)0x30000, 0));
  /* a null pointer is rejected before any device call */
  printf("null_ptr %d\n", (int)mx_gemm(0, 0, 0, 0, 0, 128, 256, 128, MX_EPI_BIAS_BF16, 0, 0, 0, 0, 0, 0));
  printf("gemm_workspace_bytes %zu\n", mx_gemm_workspace_bytes(20480, 3072, 12288));
  printf("status_ok %s\n", mx_status_string(MX_OK));
  /* host layout round trip: plain -> tiled -> plain */
  uint8_t plain[130 * 4], tiled[256 * 4], back[130 * 4];
  for (int i = 0; i < 130 * 4; ++i) plain[i] = (uint8_t)(i * 7 + 3);
  int st1 = (int)mx_scales_from_plain(plain, tiled, 130, 128);
  int st2 = (int)mx_scales_to_plain(tiled, back, 130, 128);
  printf("layout_round_trip %d\n", st1 == 0 && st2 == 0 && memcmp(plain, back, sizeof(plain)) == 0);
  return 0;
}
