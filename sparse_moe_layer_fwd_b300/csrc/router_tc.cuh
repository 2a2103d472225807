// router_tc.cuh -- router logits on the tensor cores ("190行JAX复刻DeepSeek V3",
// section "190行代码到底装进了什么": every token scores every routed expert).
//
// u[t][e] = sum_i x[t][i] W_r[e][i], x bf16, W_r fp32.  W_r is split into
// three bf16 terms, W1 = bf16(W_r), W2 = bf16(W_r - W1), W3 = bf16(W_r - W1 -
// W2), which together carry the 24 significant bits of the fp32 value, so
// every product x W_j is exact in fp32 and u = x W1^T + x W2^T + x W3^T.
// The MMA's fp32 accumulator loses a little to each addition of a partial
// dot product, always toward zero, so a chain of the 3 x d/16 MMAs of one
// slice would shrink u by ~1e-5 relative at d = 7168 (measured; the error
// grows in proportion to the chain's length).  So each 64-deep K step goes
// into fresh TMEM accumulators and the epilogue warps add them into fp32
// registers with round-to-nearest adds while the MMAs of the next steps run:
// a hardware chain is 12 MMAs long, the W3 and W2 terms first, so that only
// the four W1 MMAs add to a sum of u's magnitude.  The token tile is issued as
// two MMAs of N = 128 (token rows 0..63 and 64..127 of each CTA's half) into
// four 128-column accumulators used in turn, so a drain has one and a half K
// steps of MMAs to hide behind.
//
// k_router_split: Wsplit[j][e][i], j = 0..2, e < E_pad (rows e >= E zero).
// k_router_tc: CTA pairs (cta_group::2) in the swap-AB orientation: M = 256
//   experts (CTA r holds experts 128 r .. +127 of its block: three 16 KB
//   split tiles per 64-deep K step), N = up to 256 tokens (half per CTA),
//   K = one slice of d (split-K; k_router_topk sums the partials in slice
//   order).  Epilogue: TMEM lane = expert, column = token; eight warps, each
//   holding 32 experts x one MMA half's 128 tokens in registers; at the end,
//   for every token a warp writes its 32 experts' logits as one 128-byte
//   piece of part[s][t][e].
#pragma once

#include "ptx.cuh"

#define RT_THREADS 320  // warp 0: TMA producer, warp 1: TMEM + MMA, warps 2-9: epilogue
#define RT_STAGES 3
#define RT_A_BYTES 16384                      // 128 expert rows x 64 K of one split term
#define RT_A_STAGE (3 * RT_A_BYTES)
#define RT_STAGE (RT_A_STAGE + 16384)         // + up to 128 token rows x 64 K
#define RT_BAR_OFF (RT_STAGES * RT_STAGE)
#define RT_N_ACC 4                     // 128-column accumulators
#define RT_N_BARS (2 * RT_STAGES + 2 * RT_N_ACC + 1)  // full, empty; acc_full, acc_empty; drain
#define RT_SMEM_BYTES (RT_BAR_OFF + 8 * RT_N_BARS + 16 + 1024)
#define RT_TMEM_COLS 512  // four 128-column accumulators
#define RT_EPI_WARPS 8

struct RouterMapsDev {
  CUtensorMap w;               // Wsplit viewed as [3 E_pad, d], 64 x 128 boxes
  CUtensorMap x128, x64, x16;  // token rows of x, 64 x {128, 64, 16} boxes
};

// Four consecutive elements of one row per thread (d is a multiple of 64).
__global__ void k_router_split(const float* __restrict__ w, __nv_bfloat16* __restrict__ ws, int E,
                               int E_pad, int d) {
  const size_t n4 = (size_t)E_pad * d / 4, plane = (size_t)E_pad * d;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t o = 4 * i;
    const int e = (int)(o / d);
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (e < E) {
      const float4 f = *reinterpret_cast<const float4*>(w + o);
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
    __nv_bfloat16 b[3][4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const __nv_bfloat16 b1 = __float2bfloat16_rn(v[c]);
      const float r1 = v[c] - __bfloat162float(b1);  // exact: b1 is v rounded
      const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(b2);
      const bool fin = isfinite(v[c]);
      b[0][c] = b1;
      b[1][c] = fin ? b2 : __float2bfloat16_rn(0.f);
      b[2][c] = fin ? __float2bfloat16_rn(r2) : __float2bfloat16_rn(0.f);
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      uint2 pk;
      pk.x = (uint32_t)__bfloat16_as_ushort(b[j][0]) | ((uint32_t)__bfloat16_as_ushort(b[j][1]) << 16);
      pk.y = (uint32_t)__bfloat16_as_ushort(b[j][2]) | ((uint32_t)__bfloat16_as_ushort(b[j][3]) << 16);
      *reinterpret_cast<uint2*>(ws + j * plane + o) = pk;
    }
  }
}

// One pair per (expert block, token tile, K slice) unit; grid = 2 x units.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(RT_THREADS, 1)
k_router_tc(const __grid_constant__ RouterMapsDev maps, int T, int E, int E_pad, int d,
            int kchunk, int n_tt, int n_eb, float* __restrict__ part) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const SmClockStart clk_start = sm_clock_start();

  const int pid = blockIdx.x >> 1;  // the same unit in both CTAs of the pair
  const int eb = pid % n_eb, tt = (pid / n_eb) % n_tt, s = pid / (n_eb * n_tt);
  const int t0 = tt * 256;
  const int ntok = min(256, T - t0);
  const int npad = (ntok + 31) & ~31, half = npad / 2;
  const int k0 = s * kchunk;
  const int nkb = (min(d, k0 + kchunk) - k0) / 64;

  uint8_t* bar_base = smem + RT_BAR_OFF;
  auto full = [&](int i) { return smem_u32(bar_base + 8 * i); };
  auto empty = [&](int i) { return smem_u32(bar_base + 8 * (RT_STAGES + i)); };
  auto acc_full = [&](int u) { return smem_u32(bar_base + 8 * (2 * RT_STAGES + u)); };
  auto acc_empty = [&](int u) { return smem_u32(bar_base + 8 * (2 * RT_STAGES + RT_N_ACC + u)); };
  const uint32_t drain_bar = smem_u32(bar_base + 8 * (2 * RT_STAGES + 2 * RT_N_ACC));
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_base + 8 * RT_N_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_base + 8 * RT_N_BARS + 4);
  volatile int* progress = reinterpret_cast<volatile int*>(bar_base + 8 * RT_N_BARS + 8);

  if (threadIdx.x == 0) {
    for (int i = 0; i < RT_STAGES; ++i) {
      mbar_init(full(i), 1);   // the leader's arrive + both CTAs' bytes
      mbar_init(empty(i), 1);  // the leader's multicast commit
    }
    for (int u = 0; u < RT_N_ACC; ++u) {
      mbar_init(acc_full(u), 1);                   // the leader's multicast commit
      mbar_init(acc_empty(u), RT_EPI_WARPS);       // the 4 warps of its half, both CTAs
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    progress[0] = progress[1] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), RT_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool mma_issued = false;

  if (warp == 0) {
    if (lane == 0) {
      // ---------- producer: three split tiles of 128 experts + half the tokens ----------
      const uint64_t pol_w = l2_policy_evict_last();   // read by every pair
      const uint64_t pol_x = l2_policy_evict_first();  // read by one pair per K slice
      const uint32_t abytes = 2u * RT_A_STAGE + (uint32_t)npad * 128u;  // both CTAs
      for (int kb = 0; kb < nkb; ++kb) {
        const int st = kb % RT_STAGES, r = kb / RT_STAGES;
        if (*abort_flag || (kb >= RT_STAGES && !mbar_wait(empty(st), (r & 1) ^ 1))) {
          *abort_flag = 1;
          break;
        }
        const uint32_t fb = leader ? full(st) : cluster_map(full(st), 0);
        if (leader) mbar_arrive_expect_tx(full(st), abytes);
        uint8_t* a = smem + st * RT_STAGE;
        const int x = k0 + kb * 64;
#pragma unroll
        for (int j = 0; j < 3; ++j)
          tma_load_2d_pair(smem_u32(a + j * RT_A_BYTES), &maps.w, fb, x,
                           j * E_pad + eb * 256 + (int)rank * 128, pol_w);
        uint8_t* bsm = a + RT_A_STAGE;
        const int row = t0 + (int)rank * half;
        int i = 0;
        for (; i + 128 <= half; i += 128)
          tma_load_2d_pair(smem_u32(bsm + i * 128), &maps.x128, fb, x, row + i, pol_x);
        for (; i + 64 <= half; i += 64)
          tma_load_2d_pair(smem_u32(bsm + i * 128), &maps.x64, fb, x, row + i, pol_x);
        for (; i < half; i += 16)
          tma_load_2d_pair(smem_u32(bsm + i * 128), &maps.x16, fb, x, row + i, pol_x);
        progress[0] = kb + 1;
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ---------- MMA issuer: per stage and token half, 3 split terms x 4 ----------
      // ---------- K=16 steps into a fresh accumulator (2 kb + h) mod 4   ----------
      // The whole warp runs the loop and one elected lane issues (the issue
      // costs a lone thread more than an N = 128 MMA takes); descriptors are
      // built once per stage, the terms, slices and token halves are
      // constant offsets (16-byte units) in their start-address fields.
      const uint32_t F = 0xffffffffu;
      const uint32_t idesc = umma_idesc_bf16(256, 128);
      bool ok = true;
      for (int kb = 0; ok && kb < nkb; ++kb) {
        const int st = kb % RT_STAGES;
        const bool got = !*abort_flag && mbar_wait(full(st), (kb / RT_STAGES) & 1);
        if (!__all_sync(F, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + st * RT_STAGE), b = a + RT_A_STAGE;
        const uint64_t ad = umma_desc_sw128(a), bd = umma_desc_sw128(b);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = 2 * kb + h, u = n % RT_N_ACC;  // n-th use of the accumulators
          if (n >= RT_N_ACC &&
              !__all_sync(F, mbar_wait(acc_empty(u), ((n / RT_N_ACC) - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // smallest term first: while W3 and W2 products accumulate, the sum
          // is 2^8 to 2^16 times smaller than u, so only the four W1 MMAs add
          // at full magnitude.  B: token rows 64 h .. +63 of each CTA's half.
          if (elect_one()) {
#pragma unroll
            for (int jj = 0; jj < 3; ++jj)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16_pair(tmem + (uint32_t)(u * 128),
                               ad + (uint64_t)(((2 - jj) * RT_A_BYTES) / 16 + 2 * kk),
                               bd + (uint64_t)((h * 64 * 128) / 16 + 2 * kk), idesc,
                               (jj | kk) != 0);
            umma_commit_pair(acc_full(u));
          }
          __syncwarp();
          mma_issued = true;
        }
        if (!ok) break;
        if (elect_one()) {
          umma_commit_pair(empty(st));
          progress[1] = kb + 1;
        }
        __syncwarp();
      }
      if (!ok && lane == 0) *abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ---------- epilogue: TMEM lanes 32 q .. +31 = experts, columns = tokens; ----------
    // ---------- token half hv: its accumulators summed in registers           ----------
    // Column c of a half-h accumulator: token row 64 h + c % 64 of CTA c / 64's
    // half of the tile (the MMA's N concatenates the two CTAs' B rows).
    const int q = warp & 3, hv = (warp - 2) >> 2;
    const uint32_t lanes = tmem + ((uint32_t)(q * 32) << 16);
    float acc[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) acc[j] = 0.f;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int n = 2 * kb + hv, u = n % RT_N_ACC;
      if (*abort_flag || !mbar_wait(acc_full(u), (n / RT_N_ACC) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        float v[32];
        tmem_load_32(lanes + (uint32_t)(u * 128 + c), v);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[c + j] = __fadd_rn(acc[c + j], v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(acc_empty(u));
        else mbar_arrive_cluster(cluster_map(acc_empty(u), 0));
      }
    }
    if (ok) {
      const int e = eb * 256 + (int)rank * 128 + q * 32 + lane;
      float* out = part + (size_t)s * T * E;
#pragma unroll
      for (int j = 0; j < 128; ++j) {
        const int r = 64 * hv + (j & 63);               // row within its CTA's half
        const int t = t0 + (j < 64 ? 0 : half) + r;
        if (r < half && t < T && e < E) out[(size_t)t * E + e] = acc[j];
      }
    } else {
      *abort_flag = 1;
    }
  }

  __syncthreads();
  if (*abort_flag && leader) {
    // unwind: wait (bounded) for the copies issued, then for the MMAs
    if (warp == 0 && lane == 0) {
      for (int kb = progress[1]; kb < progress[0]; ++kb)
        mbar_wait(full(kb % RT_STAGES), (kb / RT_STAGES) & 1);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      umma_commit_pair_local(drain_bar);
      mbar_wait(drain_bar, 0);
    }
    __syncthreads();
  }
  cluster_sync_all();  // neither CTA leaves while the other may still use its memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, RT_TMEM_COLS);
  if (threadIdx.x == 0) sm_clock_add(3, clk_start);
}
