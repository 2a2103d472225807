// router.cuh -- router affinity and biased top-k ("190行JAX复刻DeepSeek V3",
// sections "190行代码到底装进了什么" and "最有价值的实验:无辅助损失均衡真的有效").
//
// k_router_logits: partial logits part[s][t][e] = sum over the s-th slice of
//   the model dimension of x[t][i] * W_r[e][i], fp32 FFMA on CUDA cores.
//   Each output accumulates its slice in one fixed sequential order that does
//   not depend on e, so two experts with identical router rows get
//   bit-identical logits (exact ties stay exact).  The multiply-adds are
//   issued as packed fp32 pairs (fma.rn.f32x2: two IEEE fp32 FMAs per
//   instruction), halving the instruction count of the inner product.
// k_router_topk: one warp per token.  u = sum_s part[s] in slice order,
//   s = 1/(1+exp(-u)), z = s + b.  The k largest z are picked one at a time
//   by a warp arg-max (larger z wins, equal z -> lower index, NaN ranks
//   below every number), slots in pick order; gates are the picked unbiased
//   s divided by their sum (summed in slot order).
#pragma once

#include "ptx.cuh"

template <typename TX>
MOE_DEV void load4_as_float(const TX* p, float* out);

template <>
MOE_DEV void load4_as_float<float>(const float* p, float* out) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}

template <>
MOE_DEV void load4_as_float<__nv_bfloat16>(const __nv_bfloat16* p, float* out) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  out[0] = fa.x; out[1] = fa.y; out[2] = fb.x; out[3] = fb.y;
}

// Packed fp32 pairs: fma.rn.f32x2 performs two IEEE fp32 fused multiply-adds
// (exactly what two fmaf calls would) in one instruction.
MOE_DEV unsigned long long f32x2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
MOE_DEV void f32x2_fma(unsigned long long& d, unsigned long long a, unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
MOE_DEV float2 f32x2_unpack(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

// Block tile BM tokens x BN experts, K step BK; 256 threads, each owning a
// TM x TN block of outputs made of 4 x 4 sub-blocks spaced BM/(TM/4) rows and
// BN/(TN/4) columns apart, so that every shared-memory read is a 16-byte
// vector.  The next K step's tiles are loaded into registers while the
// current one is multiplied (double buffering).  grid = (ceil(E/BN),
// ceil(T/BM), n_split); split z covers columns [z*kchunk, (z+1)*kchunk).
template <typename TX, int BM, int BN, int BK, int TM, int TN>
__global__ void __launch_bounds__(256)
k_router_logits(const TX* __restrict__ x, const float* __restrict__ w, float* __restrict__ part,
                int T, int E, int d, int kchunk) {
  constexpr int NT = 256;
  constexpr int TXN = BN / TN;  // threads along experts
  static_assert((BM / TM) * (BN / TN) == NT, "thread count");
  static_assert(TM % 4 == 0 && TN % 4 == 0, "4x4 sub-blocks");
  constexpr int MI = TM / 4, NJ = TN / 4;        // sub-blocks per thread
  constexpr int XV = BM * BK / 4 / NT;           // 4-element x loads per thread
  constexpr int WV = BN * BK / 4 / NT;           // 4-element w loads per thread
  static_assert(XV >= 1 && WV >= 1 && (BM * BK / 4) % NT == 0 && (BN * BK / 4) % NT == 0,
                "load split");
  __shared__ __align__(16) float As[2][BK][BM];
  __shared__ __align__(16) float Bs[2][BK][BN];

  const int tid = threadIdx.x;
  const int tx = tid % TXN, ty = tid / TXN;
  const int e0 = blockIdx.x * BN, t0 = blockIdx.y * BM;
  const int kbeg = blockIdx.z * kchunk;
  const int kend = min(d, kbeg + kchunk);

  // acc[i][2 jj], acc[i][2 jj + 1] packed in one 64-bit register
  unsigned long long acc[TM][TN / 2];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN / 2; ++j) acc[i][j] = 0ull;

  // Load slot i covers row i / (BK/4), columns 4 * (i % (BK/4)) .. +3, so
  // each row's BK columns are read by neighbouring lanes (coalesced).
  float xr[XV][4], wr[WV][4];
  auto gload = [&](int k0) {
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int i = tid + v * NT;
      const int row = i / (BK / 4), c4 = (i % (BK / 4)) * 4;
      xr[v][0] = xr[v][1] = xr[v][2] = xr[v][3] = 0.f;
      if (t0 + row < T) load4_as_float<TX>(x + (size_t)(t0 + row) * d + k0 + c4, xr[v]);
    }
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + v * NT;
      const int row = i / (BK / 4), c4 = (i % (BK / 4)) * 4;
      wr[v][0] = wr[v][1] = wr[v][2] = wr[v][3] = 0.f;
      if (e0 + row < E) load4_as_float<float>(w + (size_t)(e0 + row) * d + k0 + c4, wr[v]);
    }
  };
  auto sstore = [&](int buf) {
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int i = tid + v * NT;
      const int row = i / (BK / 4), c4 = (i % (BK / 4)) * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) As[buf][c4 + q][row] = xr[v][q];
    }
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + v * NT;
      const int row = i / (BK / 4), c4 = (i % (BK / 4)) * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) Bs[buf][c4 + q][row] = wr[v][q];
    }
  };

  int buf = 0;
  if (kbeg < kend) {
    gload(kbeg);
    sstore(0);
  }
  __syncthreads();
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    const bool more = k0 + BK < kend;
    if (more) gload(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[TM];
      unsigned long long b[TN / 2];
#pragma unroll
      for (int mi = 0; mi < MI; ++mi) {
        const float4 v = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4 + mi * (BM / MI)]);
        a[mi * 4 + 0] = v.x; a[mi * 4 + 1] = v.y; a[mi * 4 + 2] = v.z; a[mi * 4 + 3] = v.w;
      }
#pragma unroll
      for (int nj = 0; nj < NJ; ++nj) {
        const float4 v = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4 + nj * (BN / NJ)]);
        b[nj * 2 + 0] = f32x2_pack(v.x, v.y);
        b[nj * 2 + 1] = f32x2_pack(v.z, v.w);
      }
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const unsigned long long ai = f32x2_pack(a[i], a[i]);
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) f32x2_fma(acc[i][j], ai, b[j]);
      }
    }
    if (more) sstore(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
  float* out = part + (size_t)blockIdx.z * T * E;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int t = t0 + ty * 4 + (i / 4) * (BM / MI) + (i % 4);
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int e = e0 + tx * 4 + (j / 4) * (BN / NJ) + (j % 4);
      const float2 v = f32x2_unpack(acc[i][j / 2]);
      if (e < E) out[(size_t)t * E + e] = (j & 1) ? v.y : v.x;
    }
  }
}

// One warp per token; EPL = experts held per lane (E <= 32 * EPL).
template <int EPL>
__global__ void __launch_bounds__(256)
k_router_topk(const float* __restrict__ part, int n_split, const float* __restrict__ bias,
              int T, int E, int k, int32_t* __restrict__ topk_idx, float* __restrict__ gates) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;

  float key[EPL], sval[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = -INFINITY;
    sval[i] = 0.f;
    if (e < E) {
      float u = 0.f;
      for (int s = 0; s < n_split; ++s) u += part[((size_t)s * T + t) * E + e];
      const float sg = 1.0f / (1.0f + expf(-u));
      const float z = sg + bias[e];
      sval[i] = sg;
      key[i] = isnan(z) ? -INFINITY : z;
    }
  }
  uint32_t taken = 0;
  int my_idx = 0;
  float my_s = 0.f;
  float ssum = 0.f;
  for (int j = 0; j < k; ++j) {
    // best candidate of this lane
    float bk = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken >> i & 1u)) {
        if (key[i] > bk || (key[i] == bk && e < bi)) { bk = key[i]; bi = e; }
      }
    }
    // warp arg-max: larger key, then lower index -- two warp reductions: the
    // largest key as order-preserving bits, then the lowest index among the
    // lanes holding it (keys are never -0: z = s + b with s > 0)
    {
      const uint32_t kb = __float_as_uint(bk);
      const uint32_t ob = (kb & 0x80000000u) ? ~kb : (kb | 0x80000000u);
      const uint32_t mx = __reduce_max_sync(0xffffffffu, ob);
      bi = (int)__reduce_min_sync(0xffffffffu, ob == mx ? (uint32_t)bi : 0xffffffffu);
    }
    const int owner = bi & 31, slot = bi >> 5;
    float s_win = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i == slot) s_win = sval[i];
    s_win = __shfl_sync(0xffffffffu, s_win, owner);
    if (lane == owner) taken |= 1u << slot;
    if (lane == j) { my_idx = bi; my_s = s_win; }
    ssum += s_win;
  }
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = my_idx;
    gates[(size_t)t * k + lane] = my_s / ssum;
  }
}
