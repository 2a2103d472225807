// experts_simt.cuh -- grouped SwiGLU expert GEMMs on CUDA cores (fp32 FFMA).
//
// This is the expert path of the fp32 workloads (tensor-core TF32 would not
// meet an fp32 tolerance) and, for bf16, a cross-check of the tensor-core
// kernels with the same rounding points (H and Y_perm stored in the
// activation type, accumulation in fp32).
//
// Groups g < E are routed experts over their permuted rows; group E is the
// shared expert over all T tokens.  Tile = SIMT_TM tokens x SIMT_TN outputs;
// the group table (dispatch.cuh) lists each group's token tiles.
//   first GEMM  (DOWN = false): H[row] = silu(X W_gate^T) * (X W_up^T)
//   second GEMM (DOWN = true) : Y_perm[row] = H[row] W_down^T for the routed
//                               rows (the gate is applied in the combine) and
//                               for the shared expert's rows TK + t
#pragma once

#include "dispatch.cuh"

#define SIMT_TM 32
#define SIMT_TN 64
#define SIMT_TK 32

MOE_DEV float to_f(float v) { return v; }
MOE_DEV float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> MOE_DEV T from_f(float v);
template <> MOE_DEV float from_f<float>(float v) { return v; }
template <> MOE_DEV __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

MOE_DEV float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Locate tile b among the groups: the g with toff[g] <= b < toff[g+1].
MOE_DEV int find_group(const int32_t* toff, int E, int b) {
  int lo = 0, hi = E;  // answer in [0, E]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (toff[mid] <= b) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename T, bool DOWN>
__global__ void __launch_bounds__(256)
k_expert_simt(const T* __restrict__ wa0, const T* __restrict__ wa1, const T* __restrict__ sa0,
              const T* __restrict__ sa1, const T* __restrict__ b_routed,
              const T* __restrict__ b_shared, const int32_t* __restrict__ groups, int E, int K,
              int n_out, T* __restrict__ out) {
  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  const int32_t* toff = DOWN ? G.toff_b : G.toff_a;
  const int b = blockIdx.x;
  if (b >= toff[E + 1]) return;
  const int g = find_group(toff, E, b);
  const int nt = G.ntt[g];
  const int local = b - toff[g];
  const int ft = local / nt, tt = local % nt;
  const int n_g = G.off[g + 1] - G.off[g];
  const int tok0 = tt * G.tsz[g];
  const int ntok = min(G.tsz[g], n_g - tok0);
  const int f0 = ft * SIMT_TN;
  const bool shared = g == E;

  const T* A0 = shared ? sa0 : wa0 + (size_t)g * n_out * K;
  const T* A1 = DOWN ? nullptr : (shared ? sa1 : wa1 + (size_t)g * n_out * K);
  // B rows: first GEMM reads X_perm (routed) or x (shared); second reads H.
  const T* B = (!DOWN && shared) ? b_shared + (size_t)tok0 * K
                                 : b_routed + (size_t)(G.off[g] + tok0) * K;

  __shared__ float Xs[SIMT_TM][SIMT_TK + 1];
  __shared__ float As0[SIMT_TN][SIMT_TK + 1];
  __shared__ float As1[DOWN ? 1 : SIMT_TN][SIMT_TK + 1];

  const int tid = threadIdx.x;
  const int tf = tid % 16, tr = tid / 16;  // outputs tf*4..+3, tokens tr*2..+1
  float acc0[2][4], acc1[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc0[i][q] = acc1[i][q] = 0.f;

  for (int k0 = 0; k0 < K; k0 += SIMT_TK) {
    for (int i = tid; i < SIMT_TM * SIMT_TK; i += 256) {
      const int r = i / SIMT_TK, c = i % SIMT_TK;
      Xs[r][c] = r < ntok ? to_f(B[(size_t)r * K + k0 + c]) : 0.f;
    }
    for (int i = tid; i < SIMT_TN * SIMT_TK; i += 256) {
      const int r = i / SIMT_TK, c = i % SIMT_TK;
      As0[r][c] = to_f(A0[(size_t)(f0 + r) * K + k0 + c]);
      if (!DOWN) As1[r][c] = to_f(A1[(size_t)(f0 + r) * K + k0 + c]);
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SIMT_TK; ++kk) {
      const float x0 = Xs[tr * 2][kk], x1 = Xs[tr * 2 + 1][kk];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = As0[tf * 4 + q][kk];
        acc0[0][q] = fmaf(x0, a, acc0[0][q]);
        acc0[1][q] = fmaf(x1, a, acc0[1][q]);
        if (!DOWN) {
          const float c = As1[tf * 4 + q][kk];
          acc1[0][q] = fmaf(x0, c, acc1[0][q]);
          acc1[1][q] = fmaf(x1, c, acc1[1][q]);
        }
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = tr * 2 + i;
    if (r >= ntok) continue;
    const int row = G.off[g] + tok0 + r;  // H row (first GEMM) / Y_perm row (routed)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int f = f0 + tf * 4 + q;
      if (!DOWN) {
        out[(size_t)row * n_out + f] = from_f<T>(silu_f(acc0[i][q]) * acc1[i][q]);
      } else {
        out[(size_t)row * n_out + f] = from_f<T>(acc0[i][q]);
      }
    }
  }
}
