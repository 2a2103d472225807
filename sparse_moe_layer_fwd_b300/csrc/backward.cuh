// backward.cuh -- gradients of the MoE layer (the pages train with it: "DeepSeek
// V3 viết lại bằng 190 dòng JAX thuần", section "Những gì có trong 190 dòng
// code", and "190行JAX复刻DeepSeek V3", section "如何在Mac上复现").
//
// For an output gradient dy [T, d], with the forward's selection idx, gates
// g = s_sel / sum s_sel (s = sigmoid router affinities), H = silu(A) * B,
// A = X W_gate^T, B = X W_up^T per expert:
//   dY_pair = g dy                       dG_pair = <dy, Y_pair>  (Y ungated)
//   dH = dY W_down                       dA = dH B silu'(A),  dB = dH silu(A)
//   dX_pair = dA W_gate + dB W_up        dW_down = dY^T H,  dW_gate = dA^T X,
//                                        dW_up = dB^T X      (per expert)
//   ds_j = (dG_j - sum_i dG_i g_i) / sum s_sel,  du = ds s (1 - s)
//   dW_r = du^T x,   dx = dX_shared + sum_j dX_pair + du W_r
// The selection is piecewise constant and carries no gradient; the bias has
// none (it moves by the sign rule).  The shared expert is the same with g = 1.
//
// Row layouts: dY and dA|dB use "padded" rows -- every group (expert, then the
// shared expert) starts on a multiple of 16 rows and the gap rows are zero --
// so that the weight-gradient products can run their K loop (over a group's
// rows) in whole MMA steps of 16; their other operand (H, x_perm, x) keeps the
// forward's rows, whose next rows are finite.
#pragma once

#include "dispatch.cuh"
#include "experts_tc2.cuh"

// ---------------------------------------------------------------- tables
// One CTA: padded group offsets, the tile prefix of the dH product (ft_c
// output tiles per token tile), zeroed tile counters of the backward GEMMs.
__global__ void __launch_bounds__(1024)
k_bwd_tables(int32_t* __restrict__ groups, int E, int ft_c) {
  __shared__ int buf[MOE_MAX_E + 2];
  __shared__ int warp_tot[32];
  GroupTable G = group_table(groups, E);
  const int tid = threadIdx.x;
  for (int g = tid; g <= E; g += blockDim.x) buf[g] = (G.off[g + 1] - G.off[g] + 15) / 16 * 16;
  __syncthreads();
  int tot = cta_exclusive_scan(buf, E + 1, warp_tot);
  for (int g = tid; g <= E; g += blockDim.x) G.poff[g] = buf[g];
  if (tid == 0) G.poff[E + 1] = tot;
  __syncthreads();
  for (int g = tid; g <= E; g += blockDim.x) buf[g] = G.ntt[g] * ft_c;
  __syncthreads();
  tot = cta_exclusive_scan(buf, E + 1, warp_tot);
  for (int g = tid; g <= E; g += blockDim.x) G.toff_c[g] = buf[g];
  if (tid == 0) {
    G.toff_c[E + 1] = tot;
    for (int i = 2; i < 8; ++i) G.next[i] = 0;
  }
}

// ---------------------------------------------------------------- prep
// One warp per routed pair position: dY row (gate times dy, bf16, padded row)
// and dG = <dy, Y_perm> (fp32, lanes in a fixed order).  Row bytes multiple
// of 16 (d a multiple of 64).
__global__ void __launch_bounds__(256)
k_bwd_prep(const int32_t* __restrict__ groups, int E, const int32_t* __restrict__ perm,
           const int32_t* __restrict__ topk_idx, const float* __restrict__ gates, int TK, int k,
           int d, const __nv_bfloat16* __restrict__ dy, const __nv_bfloat16* __restrict__ y_perm,
           __nv_bfloat16* __restrict__ dyp, float* __restrict__ dg) {
  const int lane = threadIdx.x & 31;
  const int pos = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (pos >= TK) return;
  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  const int p = perm[pos];
  const int t = p / k;
  const int e = topk_idx[p];
  const float gv = gates[p];
  const int prow = G.poff[e] + (pos - G.off[e]);
  const uint4* src = reinterpret_cast<const uint4*>(dy + (size_t)t * d);
  const uint4* yp = reinterpret_cast<const uint4*>(y_perm + (size_t)pos * d);
  uint4* dst = reinterpret_cast<uint4*>(dyp + (size_t)prow * d);
  float acc = 0.f;
  for (int i = lane; i < d / 8; i += 32) {
    const uint4 a = src[i], b = yp[i];
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
    uint32_t wo[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[m]));
      const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[m]));
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
      const __nv_bfloat162 o = __floats2bfloat162_rn(gv * fa.x, gv * fa.y);
      wo[m] = *reinterpret_cast<const uint32_t*>(&o);
    }
    dst[i] = make_uint4(wo[0], wo[1], wo[2], wo[3]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) dg[pos] = acc;
}

// Zero the gap rows of the padded layouts: dY (routed groups, `dcols`
// columns) and dA|dB (every group, 2h columns).  One CTA per group.
__global__ void __launch_bounds__(256)
k_bwd_zero_gaps(const int32_t* __restrict__ groups, int E, __nv_bfloat16* __restrict__ dyp,
                int dcols, __nv_bfloat16* __restrict__ dab, int abcols) {
  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  const int g = blockIdx.x;
  const int n = G.off[g + 1] - G.off[g];
  const int r0 = G.poff[g] + n, r1 = G.poff[g + 1];
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int r = r0; r < r1; ++r) {
    if (g < E) {
      uint4* a = reinterpret_cast<uint4*>(dyp + (size_t)r * dcols);
      for (int i = threadIdx.x; i < dcols / 8; i += blockDim.x) a[i] = z;
    }
    uint4* b = reinterpret_cast<uint4*>(dab + (size_t)r * abcols);
    for (int i = threadIdx.x; i < abcols / 8; i += blockDim.x) b[i] = z;
  }
}

// ---------------------------------------------------------------- SwiGLU gradient
// dA = dH B silu'(A), dB = dH silu(A) from the pre-activations the training
// forward stored (A|B rows [rows, 2h], bf16, the forward's row order) and dH
// ([rows, h]); written to the padded dA|dB rows ([., 2h]).  One warp per
// row, 8 columns per lane per step; silu'(a) = s (1 + a (1 - s)), s =
// sigmoid(a).
__global__ void __launch_bounds__(256)
k_bwd_swiglu(const int32_t* __restrict__ groups, int E, int rows, int h,
             const __nv_bfloat16* __restrict__ ab, const __nv_bfloat16* __restrict__ dh,
             __nv_bfloat16* __restrict__ dab) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  int lo = 0, hi = E;  // the group g with off[g] <= r < off[g + 1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (G.off[mid] <= r) lo = mid; else hi = mid - 1;
  }
  const int prow = G.poff[lo] + (r - G.off[lo]);
  const uint4* pa = reinterpret_cast<const uint4*>(ab + (size_t)r * 2 * h);
  const uint4* pb = reinterpret_cast<const uint4*>(ab + (size_t)r * 2 * h + h);
  const uint4* pg = reinterpret_cast<const uint4*>(dh + (size_t)r * h);
  uint4* qa = reinterpret_cast<uint4*>(dab + (size_t)prow * 2 * h);
  uint4* qb = reinterpret_cast<uint4*>(dab + (size_t)prow * 2 * h + h);
  for (int i = lane; i < h / 8; i += 32) {
    const uint4 va = pa[i], vb = pb[i], vg = pg[i];
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w},
                   wg[4] = {vg.x, vg.y, vg.z, vg.w};
    uint32_t oa[4], ob[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[m]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[m]));
      const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wg[m]));
      const float s0 = 1.0f / (1.0f + __expf(-a.x)), s1 = 1.0f / (1.0f + __expf(-a.y));
      oa[m] = pack_bf16x2(g.x * b.x * (s0 * (1.0f + a.x * (1.0f - s0))),
                          g.y * b.y * (s1 * (1.0f + a.y * (1.0f - s1))));
      ob[m] = pack_bf16x2(g.x * (a.x * s0), g.y * (a.y * s1));
    }
    qa[i] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    qb[i] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// ---------------------------------------------------------------- router
// One warp per token: lane j < k takes slot j.  s_j = sigmoid(u_j) from the
// router's partial logits (summed in slice order, as the top-k did), g_j =
// s_j / S with S = sum_j s_j, ds_j = (dG_j - sum_i dG_i g_i) / S,
// du_j = ds_j s_j (1 - s_j).  Sums over slots in slot order.
__global__ void __launch_bounds__(256)
k_bwd_router(const float* __restrict__ part, int n_split, const int32_t* __restrict__ topk_idx,
             const int32_t* __restrict__ inv, const float* __restrict__ dg, int T, int E, int k,
             float* __restrict__ du) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float sv = 0.f, dgv = 0.f;
  if (lane < k) {
    const int e = topk_idx[(size_t)t * k + lane];
    float u = 0.f;
    for (int s = 0; s < n_split; ++s) u += part[((size_t)s * T + t) * E + e];
    sv = 1.0f / (1.0f + expf(-u));
    dgv = dg[inv[(size_t)t * k + lane]];
  }
  float S = 0.f, dot = 0.f;
  for (int j = 0; j < k; ++j) S += __shfl_sync(0xffffffffu, sv, j);
  const float g = sv / S;
  for (int j = 0; j < k; ++j) dot += __shfl_sync(0xffffffffu, dgv * g, j);
  if (lane < k) {
    const float ds = (dgv - dot) / S;
    du[(size_t)t * k + lane] = ds * sv * (1.0f - sv);
  }
}

// dW_r[e][c] = sum over the pairs of expert e, in row order, of du * x[token]
// (fp32).  grid (E, ceil(d / 1024)), 128 threads: thread = eight columns (one
// 16-byte load per row), four rows' loads in flight before their FMAs, which
// still run in row order.
template <typename TX>
__global__ void __launch_bounds__(128)
k_bwd_router_wgrad(const int32_t* __restrict__ groups, int E, const int32_t* __restrict__ perm,
                   const float* __restrict__ du, const TX* __restrict__ x, int d, int k,
                   float* __restrict__ dwr) {
  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  const int e = blockIdx.x, c = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (c >= d) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int r1 = G.off[e + 1];
  int pos = G.off[e];
  for (; pos + 4 <= r1; pos += 4) {
    float u[4], v[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int p = perm[pos + i];
      u[i] = du[p];
      load8(x + (size_t)(p / k) * d + c, v[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(u[i], v[i][q], acc[q]);
  }
  for (; pos < r1; ++pos) {
    const int p = perm[pos];
    float v[8];
    load8(x + (size_t)(p / k) * d + c, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = fmaf(du[p], v[q], acc[q]);
  }
  float4* o = reinterpret_cast<float4*>(dwr + (size_t)e * d + c);
  o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// ---------------------------------------------------------------- combine
// dx[t] = dX_shared[t] + sum_j dX_pair[inv[t,j]] + sum_j du[t,j] W_r[idx[t,j]],
// in that order, fp32, rounded once.  One CTA per token, 8 columns per thread.
template <typename TA>
__global__ void __launch_bounds__(128)
k_bwd_combine(const float* __restrict__ dxs, const __nv_bfloat16* __restrict__ dxp,
              const int32_t* __restrict__ inv, const int32_t* __restrict__ topk_idx,
              const float* __restrict__ du, const float* __restrict__ w_router, int T, int d,
              int k, TA* __restrict__ dx) {
  __shared__ int rows[32], ex[32];
  __shared__ float dus[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    rows[threadIdx.x] = inv[(size_t)t * k + threadIdx.x];
    ex[threadIdx.x] = topk_idx[(size_t)t * k + threadIdx.x];
    dus[threadIdx.x] = du[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float acc[8];
    load8(dxs + (size_t)t * d + c, acc);
    for (int j = 0; j < k; ++j) {
      float v[8];
      load8(dxp + (size_t)rows[j] * d + c, v);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += v[q];
    }
    for (int j = 0; j < k; ++j) {
      float w[8];
      load8(w_router + (size_t)ex[j] * d + c, w);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(dus[j], w[q], acc[q]);
    }
    store8(dx + (size_t)t * d + c, acc);
  }
}

// ---------------------------------------------------------------- weight gradients
// dW[g] = P_g^T Q_g for every group g (E routed experts, then the shared
// expert): P = dY (dW_down), dA or dB (dW_gate, dW_up), padded rows; Q = H,
// x_perm (x for the shared expert), the forward's rows.  K = the group's
// rows, rounded up to 16 (P's extra rows are zero).  Output dW[g] [M, N]
// fp32, row-major (M, N multiples of 128; partial 256 blocks are masked).  CTA pairs: a tile is 256 rows (M) x 256 columns (N), CTA
// r holding rows 128 r .. +127 of P's block and columns 128 r .. +127 of Q's;
// both operands MN-major (stored K rows of contiguous M / N elements), loaded
// as 64-element x 64-row boxes.  Two TMEM buffers: the epilogue of one tile
// overlaps the MMAs of the next.  Tiles: (E + 1) groups x M/256 x N/256,
// groups without rows write zeros.  The fp32 output leaves through shared
// memory: each epilogue warp stages 32 rows x 32 columns (a 128-byte-swizzled
// 4 KB box, so that the row-per-lane writes spread over all banks) and stores
// it with one TMA store.
struct WgMapsDev {
  CUtensorMap p, ps;  // P rows: routed (padded layout), shared
  CUtensorMap q, qs;  // Q rows: routed, shared
  CUtensorMap o, os;  // fp32 output rows: routed [(E) M, N], shared [M, N]; 32 x 32 boxes
};

#ifndef WG_STAGES
#define WG_STAGES 5
#endif
#ifndef WG_BOXES
#define WG_BOXES 2  // staged output boxes per epilogue warp, used round robin
#endif
#define WG_HALF_BYTES 16384  // 128 elements x 64 K rows (two 64-element blocks)
#define WG_STAGE_BYTES (2 * WG_HALF_BYTES)
#define WG_BOX_BYTES 4096                      // 32 x 32 fp32
#define WG_STG_OFF (WG_STAGES * WG_STAGE_BYTES)   // two boxes per epilogue warp
#define WG_BAR_OFF (WG_STG_OFF + TC_EPI_WARPS * WG_BOXES * WG_BOX_BYTES)
#define WG_N_BARS (2 * WG_STAGES + 4 + 2 * TC_TILE_RING + 1)
#define WG_SMEM_BYTES (WG_BAR_OFF + 8 * WG_N_BARS + 4 * TC_TILE_RING + 32 + 1024)
#define WG_THREADS (32 * (2 + TC_EPI_WARPS))  // producer, MMA, epilogue warps
#define WG_CONSUMERS (TC_EPI_WARPS + 2)       // per CTA: epilogue warps, MMA warp, producer

struct WgTile {
  int g, m0, n0, rows, nkb;
  int prow, qrow;  // first P / Q row of the group
  bool shared;
};

MOE_DEV WgTile wg_tile(const GroupTable& G, int E, int b, int MB, int NB, int pcol0, int qcol0) {
  WgTile t;
  t.g = b / (MB * NB);
  const int r = b % (MB * NB);
  t.m0 = (r / NB) * 256;
  t.n0 = (r % NB) * 256;
  t.shared = t.g == E;
  t.rows = G.off[t.g + 1] - G.off[t.g];
  t.nkb = (t.rows + 63) / 64;
  t.prow = G.poff[t.g];
  t.qrow = t.shared ? 0 : G.off[t.g];
  (void)pcol0;
  (void)qcol0;
  return t;
}

// pcol0 / qcol0: first column of P / Q read (dB lives in the columns h .. 2h
// of dA|dB); M, N: output rows / columns per group; `shared_p_from_ps`: the
// shared group's P rows come from the map ps at row 0 (dy) rather than the
// routed map at the shared group's padded row; same for Q.
// BF16OUT: the fp32 sums are rounded once to bf16 and stored as 32 x 32 bf16
// boxes (64-byte rows, 64-byte swizzle), half the bytes of the fp32 output.
template <bool BF16OUT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(WG_THREADS, 1)
k_wgrad_tc2(const __grid_constant__ WgMapsDev maps, const int32_t* __restrict__ groups, int E,
            int M, int N, int pcol0, int qcol0, int counter_slot, int shared_p_from_ps,
            int shared_q_from_qs) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  const int MB = (M + 255) / 256, NB = (N + 255) / 256;
  const int total = (E + 1) * MB * NB;
  int* counter = G.next + counter_slot;
  if ((int)(blockIdx.x >> 1) >= total) return;
  const SmClockStart clk_start = sm_clock_start();

  uint8_t* bar_base = smem + WG_BAR_OFF;
  auto bar = [&](int i) { return smem_u32(bar_base + 8 * i); };
  auto full = [&](int s) { return bar(s); };
  auto empty = [&](int s) { return bar(WG_STAGES + s); };
  auto acc_full = [&](int u) { return bar(2 * WG_STAGES + u); };
  auto acc_empty = [&](int u) { return bar(2 * WG_STAGES + 2 + u); };
  auto tile_full = [&](int s) { return bar(2 * WG_STAGES + 4 + s); };
  auto tile_empty = [&](int s) { return bar(2 * WG_STAGES + 4 + TC_TILE_RING + s); };
  const uint32_t drain_bar = bar(2 * WG_STAGES + 4 + 2 * TC_TILE_RING);
  uint8_t* misc = bar_base + 8 * WG_N_BARS;
  volatile int* tile_id = reinterpret_cast<volatile int*>(misc);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(misc + 4 * TC_TILE_RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4 * TC_TILE_RING + 4);
  volatile int* progress = reinterpret_cast<volatile int*>(misc + 4 * TC_TILE_RING + 8);

  if (threadIdx.x == 0) {
    for (int s = 0; s < WG_STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(acc_full(u), 1);
      mbar_init(acc_empty(u), 2 * TC_EPI_WARPS);
    }
    for (int s = 0; s < TC_TILE_RING; ++s) {
      mbar_init(tile_full(s), 1);
      mbar_init(tile_empty(s), 2 * WG_CONSUMERS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    progress[0] = progress[1] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool mma_issued = false;

  auto release_tile = [&](int s) {
    if (leader) mbar_arrive(tile_empty(s)); else mbar_arrive_cluster(cluster_map(tile_empty(s), 0));
  };
  auto next_tile = [&](int i) -> int {
    const int s = i % TC_TILE_RING;
    if (!mbar_wait_cluster(tile_full(s), (i / TC_TILE_RING) & 1)) {
      *abort_flag = 1;
      return -1;
    }
    return tile_id[s];
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------- producer of both operands; in the leader also the scheduler ----------
      const uint64_t pol = l2_policy_evict_last();
      int it = 0;
      for (int i = 0;; ++i) {
        int b;
        if (leader) {
          const int s = i % TC_TILE_RING;
          if (i >= TC_TILE_RING &&
              !mbar_wait_cluster(tile_empty(s), ((i / TC_TILE_RING) & 1) ^ 1)) {
            *abort_flag = 1;
            break;
          }
          b = *abort_flag ? total : atomicAdd(counter, 1);
          if (b >= total) b = -1;
          tile_id[s] = b;
          st_cluster_u32(cluster_map(smem_u32(const_cast<int*>(&tile_id[s])), 1), (uint32_t)b);
          mbar_arrive(tile_full(s));
          mbar_arrive_cluster(cluster_map(tile_full(s), 1));
        } else {
          b = next_tile(i);
        }
        if (b >= 0) release_tile(i % TC_TILE_RING);
        if (b < 0) break;
        const WgTile t = wg_tile(G, E, b, MB, NB, pcol0, qcol0);
        const CUtensorMap* mp = t.shared && shared_p_from_ps ? &maps.ps : &maps.p;
        const CUtensorMap* mq = t.shared && shared_q_from_qs ? &maps.qs : &maps.q;
        const int prow = t.shared && shared_p_from_ps ? 0 : t.prow;
        const int qrow = t.shared && shared_q_from_qs ? 0 : (t.shared ? G.off[E] : t.qrow);
        const int pc = pcol0 + t.m0 + 128 * (int)rank, qc = qcol0 + t.n0 + 128 * (int)rank;
        for (int kb = 0; kb < t.nkb; ++kb, ++it) {
          const int st = it % WG_STAGES, r = it / WG_STAGES;
          if (*abort_flag || (it >= WG_STAGES && !mbar_wait(empty(st), (r & 1) ^ 1))) {
            *abort_flag = 1;
            break;
          }
          uint8_t* a = smem + st * WG_STAGE_BYTES;
          const uint32_t fb = leader ? full(st) : cluster_map(full(st), 0);
          if (leader) mbar_arrive_expect_tx(full(st), 2u * WG_STAGE_BYTES);
          const int y = kb * 64;
          tma_load_2d_pair(smem_u32(a), mp, fb, pc, prow + y, pol);
          tma_load_2d_pair(smem_u32(a + 8192), mp, fb, pc + 64, prow + y, pol);
          tma_load_2d_pair(smem_u32(a + WG_HALF_BYTES), mq, fb, qc, qrow + y, pol);
          tma_load_2d_pair(smem_u32(a + WG_HALF_BYTES + 8192), mq, fb, qc + 64, qrow + y, pol);
          progress[0] = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the loop (both CTAs keep the tile ring in step);
    // in the leader one elected lane issues the tcgen05 instructions, with
    // one descriptor per operand and stage (the 16-row K slices are constant
    // offsets of 2048 bytes = 128 units in the start-address field).  Every
    // wait's outcome is made warp-uniform.
    const uint32_t F = 0xffffffffu;
    int it = 0, tl = 0;
    for (int i = 0;; ++i) {
      const int b = __shfl_sync(F, next_tile(i), 0);
      __syncwarp();
      if (lane == 0 && b >= 0) release_tile(i % TC_TILE_RING);
      if (b < 0) break;
      if (!leader) continue;  // the peer only keeps the tile ring in step
      if (__any_sync(F, *abort_flag != 0)) continue;
      // ---------- MMA issuer (leader) ----------
      const WgTile t = wg_tile(G, E, b, MB, NB, pcol0, qcol0);
      const int u = tl & 1;
      if (tl >= 2 && !__all_sync(F, mbar_wait_cluster(acc_empty(u), ((tl >> 1) - 1) & 1))) {
        if (lane == 0) *abort_flag = 1;
        continue;
      }
      tc_fence_after();
      const uint32_t idesc = umma_idesc_bf16(256, 256) | (1u << 15) | (1u << 16);
      const int ksteps = (t.rows + 15) / 16;  // rows rounded up to 16
      bool ok = true;
      for (int kb = 0; kb < t.nkb; ++kb, ++it) {
        const int st = it % WG_STAGES;
        if (!__all_sync(F, mbar_wait(full(st), (it / WG_STAGES) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + st * WG_STAGE_BYTES), bq = a + WG_HALF_BYTES;
        const uint64_t ad = umma_desc_sw128_mn(a, 8192), bd = umma_desc_sw128_mn(bq, 8192);
        const int kk_n = min(4, ksteps - 4 * kb);
        if (elect_one()) {
          for (int kk = 0; kk < kk_n; ++kk)
            umma_bf16_pair(tmem + (uint32_t)(u * 256), ad + (uint64_t)(128 * kk),
                           bd + (uint64_t)(128 * kk), idesc, (kb | kk) != 0);
          umma_commit_pair(empty(st));
          progress[1] = it + 1;
        }
        __syncwarp();
        mma_issued = true;
      }
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        continue;
      }
      if (elect_one()) umma_commit_pair(acc_full(u));
      __syncwarp();
      ++tl;
    }
    __syncwarp();
  } else {
    // ---------- epilogue: TMEM lane = output row, column = output column ----------
    const int q = warp & 3, hv = (warp - 2) >> 2;  // lanes 32 q .., columns 128 hv ..
    const uint32_t stg = smem_u32(smem + WG_STG_OFF) + (uint32_t)((warp - 2) * WG_BOXES * WG_BOX_BYTES);
    int tl = 0, nbox = 0;
    for (int i = 0;; ++i) {
      const int b = next_tile(i);
      __syncwarp();
      if (lane == 0 && b >= 0) release_tile(i % TC_TILE_RING);
      if (b < 0) break;
      const WgTile t = wg_tile(G, E, b, MB, NB, pcol0, qcol0);
      const int u = tl & 1;
      if (*abort_flag || !mbar_wait(acc_full(u), (tl >> 1) & 1)) {
        *abort_flag = 1;
        continue;  // keep reading the tile ring until the scheduler says "none"
      }
      tc_fence_after();
      const int row0 = t.m0 + 128 * (int)rank + 32 * q;  // this warp's first output row
      const bool row_ok = t.m0 + 128 * (int)rank < M;    // M a multiple of 128
      const CUtensorMap* om = t.shared ? &maps.os : &maps.o;
      const int orow = (t.shared ? 0 : t.g * M) + row0;
      for (int c = 128 * hv; c < 128 * hv + 128; c += 32) {
        float v[32];
        tmem_load_32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(u * 256) + c, v);
        if (t.rows == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        if (!row_ok || t.n0 + c >= N) continue;  // N a multiple of 32; warp-uniform
        const uint32_t box = stg + (uint32_t)((nbox % WG_BOXES) * WG_BOX_BYTES);
        if (lane == 0) bulk_wait_read<WG_BOXES - 1>();  // the box's previous store has read it
        __syncwarp();
        if (BF16OUT) {
          // row `lane` of the box: 32 bf16 in four 16-byte chunks, chunk j at
          // j ^ ((lane >> 1) & 3)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t a = box + (uint32_t)(lane * 64 + 16 * (j ^ ((lane >> 1) & 3)));
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                         "r"(pack_bf16x2(v[8 * j], v[8 * j + 1])),
                         "r"(pack_bf16x2(v[8 * j + 2], v[8 * j + 3])),
                         "r"(pack_bf16x2(v[8 * j + 4], v[8 * j + 5])),
                         "r"(pack_bf16x2(v[8 * j + 6], v[8 * j + 7]))
                         : "memory");
          }
        } else {
          // row `lane` of the box, 16-byte chunk j at chunk j ^ (lane & 7)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t a = box + (uint32_t)(lane * 128 + 16 * (j ^ (lane & 7)));
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v[4 * j]),
                         "f"(v[4 * j + 1]), "f"(v[4 * j + 2]), "f"(v[4 * j + 3])
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(om, box, t.n0 + c, orow);
          bulk_commit();
        }
        ++nbox;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(acc_empty(u)); else mbar_arrive_cluster(cluster_map(acc_empty(u), 0));
      }
      ++tl;
    }
    if (lane == 0) bulk_wait_all();  // this warp's stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && leader) {
    if (warp == 0 && lane == 0) {
      for (int it = progress[1]; it < progress[0]; ++it)
        mbar_wait(full(it % WG_STAGES), (it / WG_STAGES) & 1);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      umma_commit_pair_local(drain_bar);
      mbar_wait(drain_bar, 0);
    }
    __syncthreads();
  }
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
  if (threadIdx.x == 0) sm_clock_add(2, clk_start);
}
