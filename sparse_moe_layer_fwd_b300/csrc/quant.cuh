// quant.cuh -- per-row e4m3 quantization for the fp8 gate/up products.
//
// The official V3 model ("DeepSeek V3 viết lại bằng 190 dòng JAX thuần",
// section "Những gì có trong 190 dòng code") computes its expert products in
// FP8; the re-creation leaves that out.  Here the scaling unit is one row:
// each row of W_gate / W_up (one hidden unit) and each token row of x gets
//   scale = amax(|row|) / 448   (1 for an all-zero row)
//   code  = e4m3(row / scale)   (nearest, ties to even, saturating)
// so that a gate/up product is (code_w . code_x) * scale_w * scale_x with the
// code dot product on the tensor cores (kind::f8f6f4).  448 is the largest
// finite e4m3 value.  Scale and quotient are IEEE fp32 operations.
//
// Packed layout of a quantized [rows, cols] matrix (one buffer):
//   bytes [0, rows*cols)              codes, row-major, one byte each
//   bytes [S, S + 4*rows)             fp32 scales, S = rows*cols rounded up to 256
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

__host__ __device__ inline size_t e4m3_scale_offset(long long rows, long long cols) {
  return ((size_t)rows * (size_t)cols + 255) / 256 * 256;
}

// Two fp32 values to e4m3 codes, nearest-even with saturation to +-448:
// lo in the low byte.
MOE_DEV uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One warp per row; cols a multiple of 8 (each lane reads 8 bf16 per step).
// A row holding a NaN gets scale 1 (the NaN propagates into its code).
template <typename TX>
__global__ void __launch_bounds__(256) k_quant_rows(const TX* __restrict__ a, long long rows,
                                                    int cols, uint8_t* __restrict__ codes,
                                                    float* __restrict__ scales) {
  static_assert(sizeof(TX) == 2, "bf16 rows");
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(a + row * cols);
  const int n8 = cols / 8;
  float amax = 0.f;
  bool nan = false;
  for (int i = lane; i < n8; i += 32) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
      nan |= (lo != lo) | (hi != hi);
      amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  nan = __any_sync(0xffffffffu, nan);
  const float scale = (!nan && amax > 0.f) ? __fdiv_rn(amax, 448.f) : 1.f;
  if (lane == 0) scales[row] = scale;
  uint2* dst = reinterpret_cast<uint2*>(codes + row * cols);
  for (int i = lane; i < n8; i += 32) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t q[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t a0 = w[2 * j], a1 = w[2 * j + 1];
      const uint16_t c0 = cvt_e4m3x2(__fdiv_rn(__uint_as_float(a0 << 16), scale),
                                     __fdiv_rn(__uint_as_float(a0 & 0xffff0000u), scale));
      const uint16_t c1 = cvt_e4m3x2(__fdiv_rn(__uint_as_float(a1 << 16), scale),
                                     __fdiv_rn(__uint_as_float(a1 & 0xffff0000u), scale));
      q[j] = (uint32_t)c0 | ((uint32_t)c1 << 16);
    }
    dst[i] = make_uint2(q[0], q[1]);
  }
}
