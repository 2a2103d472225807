// combine.cuh -- gated combine and the bias update.
//
// k_combine: y[t] = Y_sh[t] + sum_{j=0..k-1} g[t,j] * Y_perm[inv[t*k+j]],
//   one fp32 fused multiply-add per slot in that fixed slot order, rounded
//   once to the output type.  (The gate multiplies the expert's output row
//   here rather than in the down-projection epilogue: the same product, and
//   the tensor-core epilogue, which stalls the MMAs while it drains the
//   accumulators, loses its per-token broadcasts.)  One CTA per token, 8
//   elements (16 bytes of bf16) per thread per step, so every load and store
//   is a coalesced 16-byte vector.  Deterministic: no atomics.
// k_bias_update: b[e] = fp32(b[e] - fp32(gamma) * sgn(E*load[e] - TK))
//   ("190行JAX复刻DeepSeek V3", section "最有价值的实验:无辅助损失均衡真的有效":
//   an expert above the mean load T*k/E is lowered, one below it raised).
#pragma once

#include "ptx.cuh"

MOE_DEV void load8(const float* p, float* v) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

MOE_DEV void load8(const __nv_bfloat16* p, float* v) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

MOE_DEV void store8(float* p, const float* v) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

MOE_DEV void store8(__nv_bfloat16* p, const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename TA>
__global__ void __launch_bounds__(128)
k_combine(const float* __restrict__ y_sh, const TA* __restrict__ y_perm,
          const int32_t* __restrict__ inv, const float* __restrict__ gates, int T, int d, int k,
          TA* __restrict__ y) {
  __shared__ int rows[32];
  __shared__ float gs[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    rows[threadIdx.x] = inv[(size_t)t * k + threadIdx.x];
    gs[threadIdx.x] = gates[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float acc[8];
    load8(y_sh + (size_t)t * d + c, acc);
    for (int j = 0; j < k; ++j) {
      float v[8];
      load8(y_perm + (size_t)rows[j] * d + c, v);
      const float g = gs[j];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(g, v[q], acc[q]);
    }
    store8(y + (size_t)t * d + c, acc);
  }
}

__global__ void k_bias_update(const int32_t* __restrict__ load, float* __restrict__ bias,
                              float gamma, int E, int TK) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const long long diff = (long long)E * load[e] - (long long)TK;
  const float sgn = diff > 0 ? 1.0f : (diff < 0 ? -1.0f : 0.0f);
  bias[e] = __fsub_rn(bias[e], gamma * sgn);
}
