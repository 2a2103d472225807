// combine.cuh -- gated combine and the bias update.
//
// k_combine: y[t] = Y_perm[TK + t] + sum_{j=0..k-1} g[t,j] * Y_perm[inv[t*k+j]]
//   (row TK + t: the shared expert's output for token t), one fp32 fused
//   multiply-add per slot in that fixed slot order, rounded once to the
//   output type.  (The gate multiplies the expert's output row
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
k_combine(const TA* __restrict__ y_perm, const int32_t* __restrict__ inv,
          const float* __restrict__ gates, int T, int d, int k, TA* __restrict__ y) {
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
    load8(y_perm + ((size_t)T * k + t) * d + c, acc);
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

// k_seq_balance_loss: the sequence-wise balance loss that the pages keep
// beside the bias (alpha = 1e-4; "DeepSeek V3 viết lại bằng 190 dòng JAX
// thuần", section "Những gì có trong 190 dòng code"), per sequence of S
// consecutive tokens as the original report defines it:
//   f_e = E/(k S) * #{t : e selected},  s'[t,e] = s[t,e] / sum_j s[t,j],
//   P_e = (1/S) sum_t s'[t,e],          L = alpha * sum_e f_e P_e.
// One CTA (8 warps) per sequence, reading the router's partial logits from
// the workspace.  Warp w takes tokens w, w+8, ... of the sequence: u = sum
// of the partials in slice order, s = 1/(1+exp(-u)), the token's sum of s
// by a fixed butterfly, and s' accumulated per expert in registers.
// Selections are counted in shared memory (integers).  P_e sums the warps
// in warp order; warp 0 sums count_e * P_e over the experts in a fixed order.
// Every floating-point sum has a fixed order: the result is deterministic.
template <int EPL>
__global__ void __launch_bounds__(256)
k_seq_balance_loss(const float* __restrict__ part, int n_split, const int32_t* __restrict__ topk_idx,
                   int T, int E, int k, int S, float alpha, float* __restrict__ loss) {
  extern __shared__ float sm_bal[];
  float* ppart = sm_bal;                                // [8][E]
  int* cnt = reinterpret_cast<int*>(sm_bal + 8 * E);  // [E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * S, t1 = min(T, t0 + S);
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
  for (int t = t0 + warp; t < t1; t += 8) {
    float sv[EPL];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      sv[i] = 0.f;
      if (e < E) {
        float u = 0.f;
        for (int s = 0; s < n_split; ++s) u += part[((size_t)s * T + t) * E + e];
        sv[i] = 1.0f / (1.0f + expf(-u));
        sum += sv[i];
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] += sv[i] / sum;
    if (lane < k) atomicAdd(&cnt[topk_idx[(size_t)t * k + lane]], 1);
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) ppart[warp * E + e] = acc[i];
  }
  __syncthreads();
  if (warp == 0) {
    float total = 0.f;
    for (int e = lane; e < E; e += 32) {
      float P = 0.f;
      for (int w = 0; w < 8; ++w) P += ppart[w * E + e];
      total += (float)cnt[e] * P;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
    const float Sq = (float)(t1 - t0);
    if (lane == 0) loss[blockIdx.x] = alpha * ((float)E / ((float)k * Sq)) * (total / Sq);
  }
}
