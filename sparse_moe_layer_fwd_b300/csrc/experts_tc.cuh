// experts_tc.cuh -- grouped SwiGLU expert GEMMs on the sm_103a tensor cores.
//
// The expert FFNs are where the layer is a dense contraction (the pages place
// the layer's cost in the expert matmuls: "190行JAX复刻DeepSeek V3", section
// "190行代码到底装进了什么"), so this is the one place the tensor cores are used.
//
// Formulation ("swap-AB"): the weights are the MMA's M side and the tokens
// its N side,
//     D^T[out, tok] = W[out, :] . X[tok, :]^T
// so a tile is 128 weight rows x N tokens with N = the group's token count
// rounded up to 16 (<= BN).  A routed expert in the V3 prefill workload gets
// about 256 +- 16 tokens, so 16-token granularity wastes ~3% of the MMA work
// where 128-token M tiles would waste ~25%; in decode (about 4 tokens per
// expert) the same kernel streams each weight tile once with N = 16.
//
// Each CTA owns one tile and two fp32 TMEM accumulators of BN columns each:
//   first GEMM (DOWN = false): acc0 = W_gate rows f0..f0+127, acc1 = W_up rows
//       f0..f0+127 (same B tile) -> H[row, f] = bf16(silu(acc0) * acc1)
//   second GEMM (DOWN = true): acc0 / acc1 = W_down rows f0..+127 / f0+128..+255
//       -> routed: Y_perm[row, f] = bf16(g(row) * acc); shared: Y_sh[t, f] = acc
// Both GEMMs therefore read 2 A sub-tiles (2 x 16 KB) per B tile (N x 128 B)
// per 64-deep K step.
//
// Warp roles (192 threads): warp 0 = TMA producer (one lane), warp 1 = TMEM
// allocator + MMA issuer (one lane), warps 2-5 = epilogue (TMEM -> registers
// -> global; warp w reads TMEM lanes 32*(w%4)..+31).  A STAGES-deep ring of
// shared-memory stages, each with a "full" mbarrier (TMA transaction bytes)
// and an "empty" mbarrier (tcgen05.commit from the MMA lane).  Operands are
// K-major with the 128-byte swizzle.  Weights are loaded with an L2
// evict-first hint (each weight tile is read by one CTA, or by the CTAs of
// one expert's token tiles that run side by side), token rows with
// evict-last (re-read by every output tile of the group).
//
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains its copies in
// flight with bounded waits, frees its TMEM and returns, leaving the device
// error word set.  Later CTAs see the word and return at once.
#pragma once

#include "experts_simt.cuh"

#define TC_BM 128
#define TC_BK 64
#define TC_THREADS 192

template <int BN, int STAGES>
struct TcCfg {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
  static constexpr int B_BYTES = BN * TC_BK * 2;     // BN * 128 B
  static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 1) + 16;
  static constexpr int GATE_OFF = BAR_OFF + ((BAR_BYTES + 127) / 128) * 128;
  static constexpr int SMEM_BYTES = GATE_OFF + BN * 4 + 1024;  // + 1024 for base alignment
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(SMEM_BYTES > 232448 / 2, "one CTA per SM: the TMEM allocation assumes it");
};

template <int BN, int STAGES, bool DOWN>
__global__ void __launch_bounds__(TC_THREADS, 1)
k_expert_tc(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
            const __grid_constant__ CUtensorMap tm_sa0, const __grid_constant__ CUtensorMap tm_sa1,
            const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_bs,
            const int32_t* __restrict__ groups, int E, int K, int n_out,
            __nv_bfloat16* __restrict__ out, float* __restrict__ y_sh,
            const int32_t* __restrict__ perm, const float* __restrict__ gates) {
  using C = TcCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile of this CTA (uniform across the CTA) ----
  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  const int32_t* toff = DOWN ? G.toff_b : G.toff_a;
  const int b = blockIdx.x;
  if (b >= toff[E + 1]) return;
  {
    // a CTA-uniform decision: one thread reads the error word
    __shared__ int s_skip;
    if (threadIdx.x == 0) s_skip = *reinterpret_cast<volatile unsigned*>(&g_moe_dev_error) != 0u;
    __syncthreads();
    if (s_skip) return;
  }
  const int g = find_group(toff, E, b);
  const bool shared = g == E;
  const int nt = G.ntt[g];
  const int local = b - toff[g];
  const int ft = local / nt, tt = local % nt;
  const int n_g = G.off[g + 1] - G.off[g];
  const int tsz = G.tsz[g];
  const int tok0 = tt * tsz;
  const int ntok = min(tsz, n_g - tok0);
  const int npad = (ntok + 15) & ~15;
  const int f0 = ft * (DOWN ? 2 * TC_BM : TC_BM);
  const bool has_a1 = DOWN ? (f0 + TC_BM < n_out) : true;
  const int row_a0 = (shared ? 0 : g * n_out) + f0;
  const int row_a1 = DOWN ? row_a0 + TC_BM : row_a0;
  const int row_b = (!DOWN && shared) ? tok0 : G.off[g] + tok0;
  const CUtensorMap* mA0 = shared ? &tm_sa0 : &tm_a0;
  const CUtensorMap* mA1 = DOWN ? mA0 : (shared ? &tm_sa1 : &tm_a1);
  const CUtensorMap* mB = (!DOWN && shared) ? &tm_bs : &tm_b;

  uint8_t* bar_base = smem + C::BAR_OFF;
  auto full_bar = [&](int s) { return smem_u32(bar_base + 8 * s); };
  auto empty_bar = [&](int s) { return smem_u32(bar_base + 8 * (STAGES + s)); };
  const uint32_t acc_bar = smem_u32(bar_base + 8 * (2 * STAGES));
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_base + 8 * (2 * STAGES + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_base + 8 * (2 * STAGES + 1) + 4);
  volatile int* progress = reinterpret_cast<volatile int*>(bar_base + 8 * (2 * STAGES + 1) + 8);
  float* gate_s = reinterpret_cast<float*>(smem + C::GATE_OFF);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_bar, 1);
    *abort_flag = 0;
    progress[0] = 0;  // k-blocks issued by the producer
    progress[1] = 0;  // k-blocks consumed by the MMA lane
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(mA0);
    prefetch_tensormap(mA1);
    prefetch_tensormap(mB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nkb = K / TC_BK;
  bool mma_committed = false;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      const uint32_t bytes = (has_a1 ? 2u : 1u) * C::A_BYTES + (uint32_t)npad * (TC_BK * 2);
      int kb = 0;
      for (; kb < nkb; ++kb) {
        const int s = kb % STAGES, r = kb / STAGES;
        if (kb >= STAGES && !mbar_wait(empty_bar(s), (r & 1) ^ 1)) { *abort_flag = 1; break; }
        uint8_t* st = smem + s * C::STAGE_BYTES;
        const uint32_t fb = full_bar(s);
        mbar_arrive_expect_tx(fb, bytes);
        tma_load_2d(smem_u32(st), mA0, fb, kb * TC_BK, row_a0, pol_w);
        if (has_a1) tma_load_2d(smem_u32(st + C::A_BYTES), mA1, fb, kb * TC_BK, row_a1, pol_w);
        uint8_t* sb = st + 2 * C::A_BYTES;
        for (int i = 0; i < npad; i += 16)
          tma_load_2d(smem_u32(sb + i * (TC_BK * 2)), mB, fb, kb * TC_BK, row_b + i, pol_x);
        progress[0] = kb + 1;
        if (*abort_flag) { ++kb; break; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(TC_BM, npad);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES, r = kb / STAGES;
        if (!mbar_wait(full_bar(s), r & 1)) { *abort_flag = 1; break; }
        tc_fence_after();
        uint8_t* st = smem + s * C::STAGE_BYTES;
        const uint32_t a0 = smem_u32(st), a1 = smem_u32(st + C::A_BYTES);
        const uint32_t bb = smem_u32(st + 2 * C::A_BYTES);
#pragma unroll
        for (int kk = 0; kk < TC_BK / 16; ++kk) {
          const uint64_t bdesc = umma_desc_sw128(bb + kk * 32);
          const uint32_t acc = (kb | kk) != 0;
          umma_bf16(tmem, umma_desc_sw128(a0 + kk * 32), bdesc, idesc, acc);
          if (has_a1) umma_bf16(tmem + BN, umma_desc_sw128(a1 + kk * 32), bdesc, idesc, acc);
        }
        umma_commit(empty_bar(s));
        progress[1] = kb + 1;
        if (*abort_flag) break;
      }
      umma_commit(acc_bar);
      mma_committed = true;
    }
    __syncwarp();
  } else {
    // ---- epilogue warps 2..5 ----
    const int et = threadIdx.x - 64;  // 0..127
    if (DOWN && !shared) {
      for (int i = et; i < ntok; i += 128) gate_s[i] = gates[perm[G.off[g] + tok0 + i]];
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const bool ok = mbar_wait(acc_bar, 0);
    if (!ok) *abort_flag = 1;
    tc_fence_after();
    const int q = warp & 3;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const int f = f0 + q * 32 + lane;
    const bool write = ok && (*abort_flag == 0);
    for (int c = 0; c < npad; c += 32) {
      float va[32], vb[32];
      tmem_load_2x32(tl + c, tl + BN + c, va, vb);
      if (!write) continue;
      if (!DOWN) {
        __nv_bfloat16* o = out + (size_t)(G.off[g] + tok0 + c) * n_out + f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c + j < ntok) o[(size_t)j * n_out] = __float2bfloat16_rn(silu_f(va[j]) * vb[j]);
      } else if (shared) {
        float* o = y_sh + (size_t)(tok0 + c) * n_out + f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c + j < ntok) {
            o[(size_t)j * n_out] = va[j];
            if (has_a1) o[(size_t)j * n_out + TC_BM] = vb[j];
          }
      } else {
        __nv_bfloat16* o = out + (size_t)(G.off[g] + tok0 + c) * n_out + f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c + j < ntok) {
            const float gv = gate_s[c + j];
            o[(size_t)j * n_out] = __float2bfloat16_rn(gv * va[j]);
            if (has_a1) o[(size_t)j * n_out + TC_BM] = __float2bfloat16_rn(gv * vb[j]);
          }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Unwind: let every copy this CTA issued land and every MMA it issued
    // finish (each wait bounded) before the shared memory and TMEM go away.
    if (warp == 0 && lane == 0) {
      for (int kb = progress[1]; kb < progress[0]; ++kb)
        mbar_wait(full_bar(kb % STAGES), (kb / STAGES) & 1);
    }
    if (warp == 1 && lane == 0 && mma_committed) mbar_wait(acc_bar, 0);
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}
