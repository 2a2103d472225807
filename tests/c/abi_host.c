/* The C boundary from plain C (no Python, no torch): sizes, error codes and
 * host-side argument checks of libmoe.so, none of which needs a GPU.
 * Exits 0 when every check holds, else prints the failing line. */
#include <stdio.h>
#include <string.h>

#include "moe.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
      return 1;                                               \
    }                                                         \
  } while (0)

int main(void) {
  moe_desc d = {8192, 7168, 2048, 256, 8, MOE_BF16, 0};
  size_t ws = moe_workspace_size(&d);
  CHECK(ws > 0);
  moe_desc fp8 = d;
  fp8.flags = MOE_FP8_BLOCK;
  CHECK(moe_workspace_size(&fp8) > 0);
  fp8.flags = MOE_FP8_GATE_UP;
  CHECK(moe_workspace_size(&fp8) > 0);
  moe_desc bad = d;
  bad.k = 33;
  CHECK(moe_workspace_size(&bad) == 0);
  bad = d;
  bad.dtype = 7;
  CHECK(moe_workspace_size(&bad) == 0);
  CHECK(moe_workspace_size(NULL) == 0);

  moe_region regs[16];
  int n = moe_workspace_regions(&d, regs, 16);
  CHECK(n == 12);
  CHECK(strcmp(regs[0].name, "router_part") == 0);
  for (int i = 1; i < n; ++i) CHECK(regs[i].offset % 256 == 0);

  CHECK(strcmp(moe_error_string(MOE_OK), "unknown error") != 0);
  CHECK(strcmp(moe_error_string(12345), "unknown error") == 0);

  /* argument errors are found on the host, before any launch */
  moe_expert_w w = {(const void*)0x10000, (const void*)0x10000, (const void*)0x10000};
  CHECK(moe_forward(&d, NULL, (const float*)0x10000, (const float*)0x10000, &w, &w,
                    (void*)0x10000, (int32_t*)0x10000, (float*)0x10000, (int32_t*)0x10000,
                    (void*)0x10000, ws, NULL) == MOE_ERR_NULL);
  CHECK(moe_forward(&d, (const void*)0x10008, (const float*)0x10000, (const float*)0x10000, &w,
                    &w, (void*)0x10000, (int32_t*)0x10000, (float*)0x10000, (int32_t*)0x10000,
                    (void*)0x10000, ws, NULL) == MOE_ERR_ALIGN);
  CHECK(moe_forward(&d, (const void*)0x10000, (const float*)0x10000, (const float*)0x10000, &w,
                    &w, (void*)0x10000, (int32_t*)0x10000, (float*)0x10000, (int32_t*)0x10000,
                    (void*)0x10000, ws - 1, NULL) == MOE_ERR_WORKSPACE);
  CHECK(moe_bias_update(NULL, (float*)0x10000, 1e-3f, 256, 65536, NULL) == MOE_ERR_NULL);
  CHECK(moe_e4m3_packed_bytes(10, 24) == 256 + 40);
  /* 128 x 640 codes, then 1 block row x 2 words of exponents */
  CHECK(moe_e4m3_block_packed_bytes(128, 640) == 128 * 640 + 8);
  CHECK(moe_e4m3_block_packed_bytes(100, 640) == 0);
  CHECK(moe_quantize_blocks_e4m3((const void*)0x10000, 128, 100, (void*)0x10000, NULL) ==
        MOE_ERR_SHAPE);
  moe_desc both = d;
  both.flags = MOE_FP8_BLOCK | MOE_FP8_GATE_UP;
  CHECK(moe_workspace_size(&both) == 0);
  CHECK(moe_quantize_rows_e4m3((const void*)0x10000, 4, 100, (void*)0x10000, NULL) ==
        MOE_ERR_SHAPE);
  CHECK(moe_selftest_timeout(0, NULL) == MOE_ERR_SHAPE);
  CHECK(moe_sm_clock_record(NULL, 0) == MOE_ERR_NULL);
  CHECK(moe_selftest_silu(NULL, NULL, -1, NULL) == MOE_ERR_SHAPE);
  CHECK(moe_selftest_silu(NULL, (float*)0x10000, 4, NULL) == MOE_ERR_NULL);
  CHECK(MOE_CLOCK_SLOTS == 4);
  /* routing with the static array: a problem whose scratch exceeds it is
   * refused before any device is touched */
  moe_desc big = {65536, 128, 128, 256, 1, MOE_BF16, MOE_ROUTE_ONLY};
  CHECK(moe_workspace_size(&big) > MOE_STATIC_SCRATCH_BYTES);
  CHECK(moe_route_noalloc(&big, (const void*)0x10000, (const float*)0x10000,
                          (const float*)0x10000, (int32_t*)0x10000, (float*)0x10000,
                          (int32_t*)0x10000, NULL) == MOE_ERR_WORKSPACE);
  puts("C ABI host checks passed");
  return 0;
}
