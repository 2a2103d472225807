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

// ---------------------------------------------------------------- block scales
// Block-scaled e4m3 (the official model's tile granularity): weights in
// 128 x 128 blocks, activation rows in 1 x 128 blocks.  A block with largest
// magnitude amax gets the scale 2^e, e the smallest integer with amax <=
// 448 * 2^e (0 for a block of zeros or one whose maximum is not finite,
// clamped to [-127, 127]), stored as the byte e + 127; its codes are
// e4m3(v * 2^-e), nearest-even, saturating (NaN stays NaN).  The exponent
// bytes of four consecutive blocks along a row share one 32-bit word (byte j
// = block 4 w + j), the unit the block-scaled MMA's scale copies move.
//
// Packed weight matrix [rows, cols] (rows, cols multiples of 128): codes
// [rows, cols] at byte 0, exponent words [rows / 128][ceil(cols / 512)] at
// byte e4m3_scale_offset(rows, cols).  Activation rows: codes [rows, cols],
// exponent words [ceil(cols / 512)][rows] (column-group major, so that a
// tile's tokens are consecutive words).
__host__ __device__ inline int e4m3_block_words(long long cols) {
  return (int)((cols / 128 + 3) / 4);
}
__host__ __device__ inline size_t e4m3_block_packed_bytes(long long rows, long long cols) {
  return e4m3_scale_offset(rows, cols) + (size_t)(rows / 128) * e4m3_block_words(cols) * 4;
}

// Eight bf16 values (one 16-byte vector) times 2^-e to e4m3 codes, in order.
MOE_DEV uint2 e4m3x8_scaled(const uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t q[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t a0 = w[2 * j], a1 = w[2 * j + 1];
    const uint16_t c0 = cvt_e4m3x2(__uint_as_float(a0 << 16) * inv,
                                   __uint_as_float(a0 & 0xffff0000u) * inv);
    const uint16_t c1 = cvt_e4m3x2(__uint_as_float(a1 << 16) * inv,
                                   __uint_as_float(a1 & 0xffff0000u) * inv);
    q[j] = (uint32_t)c0 | ((uint32_t)c1 << 16);
  }
  return make_uint2(q[0], q[1]);
}

// Largest |value| of eight bf16 values as fp32 bits (NaN above inf above any
// finite value).
MOE_DEV uint32_t absmax_bits8(const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    m = max(m, (w[j] << 16) & 0x7fffffffu);
    m = max(m, w[j] & 0x7fff0000u);
  }
  return m;
}

// Weights: one CTA of 128 threads per 128 x 128 block (grid: column blocks
// x row blocks); thread r quantizes row r of the block.
__global__ void __launch_bounds__(128) k_quant_wblocks(const __nv_bfloat16* __restrict__ a,
                                                        int cols, uint8_t* __restrict__ codes,
                                                        uint32_t* __restrict__ words) {
  __shared__ uint32_t part[4];
  const int r = threadIdx.x, cb = blockIdx.x;
  const long long row = (long long)blockIdx.y * 128 + r;
  const uint4* src = reinterpret_cast<const uint4*>(a + row * cols + (size_t)cb * 128);
  uint4 v[16];
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = src[i];
    m = max(m, absmax_bits8(v[i]));
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((r & 31) == 0) part[r >> 5] = m;
  __syncthreads();
  m = max(max(part[0], part[1]), max(part[2], part[3]));
  const int e = block_exp_from_bits(m);
  const float inv = exp2_neg(e);
  uint4* dst = reinterpret_cast<uint4*>(codes + row * cols + (size_t)cb * 128);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint2 lo = e4m3x8_scaled(v[2 * i], inv), hi = e4m3x8_scaled(v[2 * i + 1], inv);
    dst[i] = make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  if (r == 0)
    reinterpret_cast<uint8_t*>(words)[((size_t)blockIdx.y * e4m3_block_words(cols) + (cb >> 2)) * 4 +
                                      (cb & 3)] = (uint8_t)(e + 127);
}

// Activation rows: one warp per row, a half-warp per 128-column block (16
// lanes x 8 values).
__global__ void __launch_bounds__(256) k_quant_ablocks(const __nv_bfloat16* __restrict__ a,
                                                        int rows, int cols,
                                                        uint8_t* __restrict__ codes,
                                                        uint32_t* __restrict__ words) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int nb = cols / 128, sub = lane & 15;
  for (int b0 = 0; b0 < nb; b0 += 2) {
    const int b = b0 + (lane >> 4);
    const bool active = b < nb;
    const size_t off = (size_t)row * cols + (size_t)b * 128 + sub * 8;
    const uint4 v = active ? *reinterpret_cast<const uint4*>(a + off) : make_uint4(0, 0, 0, 0);
    uint32_t m = absmax_bits8(v);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = block_exp_from_bits(m);
    if (active) {
      *reinterpret_cast<uint2*>(codes + off) = e4m3x8_scaled(v, exp2_neg(e));
      if (sub == 0)
        reinterpret_cast<uint8_t*>(words)[((size_t)(b >> 2) * rows + row) * 4 + (b & 3)] =
            (uint8_t)(e + 127);
    }
  }
}
