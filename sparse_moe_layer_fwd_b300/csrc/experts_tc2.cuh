// experts_tc2.cuh -- the grouped expert GEMMs on CTA pairs (2-SM tensor-core
// MMA, cta_group::2), for token tiles of up to 256 tokens.
//
// Same computation and tile table as experts_tc.cuh (swap-AB: weights are the
// MMA's M side, tokens its N side), with one tile spread over a cluster of
// two CTAs on two SMs:
//   first GEMM : a pair tile covers 256 rows of W_gate and the same 256 rows
//                of W_up; CTA r holds rows f0 + 128 r .. +127 of both, so its
//                two TMEM accumulators hold gate and up for its own 128
//                hidden units and the SwiGLU epilogue stays local.
//   second GEMM: a pair tile covers 512 rows of W_down, two blocks of 256;
//                CTA r holds rows f0 + 128 r .. +127 and f0 + 256 + 128 r ..
//                +127 in its two accumulators.  (One block per tile with two
//                TMEM buffers, so that the epilogue overlaps the next tile's
//                MMAs, streams the token tile twice as often and measured
//                slower.)
//   Token rows: CTA r holds rows r * N/2 .. of the N-token tile (N a
//   multiple of 16), so each CTA streams half of the token tile.
// Per 64-deep K step a CTA loads 32 KB of weights + N/2 x 128 B of tokens
// (48 KB at N = 256) instead of 64 KB, so the same shared memory holds a
// deeper weight ring (5 stages) and each SM moves a quarter fewer bytes.
//
// Roles per CTA as in the 1-SM kernel (warp 0: weights [+ tile scheduler in
// the leader], warp 1: MMA in the leader, warps 2-9: epilogue, warp 10:
// token rows).  The weight, MMA and token-row warps run their loops as whole
// warps and issue the TMA copies and tcgen05 instructions from one elected
// lane (the issue then keeps up with an MMA of N >= 128; from a loop that
// one lane runs alone it did not).  Only the leader (cluster rank 0) issues
// MMAs; both CTAs'
// TMA loads complete on the leader's "full" barriers (.cta_group::2 TMA), the
// leader's commits arrive on both CTAs' "empty" and "acc_full" barriers
// (multicast), and the peer's roles arrive remotely on the leader's
// tile_empty and acc_empty barriers.  The leader's scheduler takes pair
// tiles in table order from the global counter and writes each tile id into
// both CTAs' tile rings.
//
// Every wait is bounded; every decision to leave is the same in both CTAs of
// a pair, so both reach the final cluster barrier.
#pragma once

#include "experts_tc.cuh"

// Operations of the CTA-pair grouped GEMM.  Rows of a weight matrix are the
// MMA's M side and token rows its N side in all of them.
enum : int {
  TC2_FWD_UP = 0,    // H = silu(X W_gate^T) * (X W_up^T)                      K = d
  TC2_FWD_DOWN = 1,  // Y = H W_down^T                                          K = h
  TC2_BWD_DH = 2,    // dH = dY W_down (W_down read transposed)                 K = d
  // (3: unused -- the SwiGLU gradient is an elementwise kernel on the
  //  pre-activations the training forward stores, TC2_FWD_UP_T)
  TC2_BWD_DX = 4,    // dX = dA W_gate + dB W_up (weights read transposed)      K = 2h
  TC2_FWD_UP_FP8 = 5,  // H as TC2_FWD_UP from e4m3 codes of weights and tokens
                       // with per-row scales (kind::f8f6f4)          K = d (bytes)
  TC2_FWD_UP_B8 = 7,     // H as TC2_FWD_UP from block-scaled e4m3 codes (kind::mxf8f6f4), H
                         // written as e4m3 codes with one scale per 1 x 128 block   K = d (bytes)
  TC2_FWD_DOWN_B8 = 8,   // Y as TC2_FWD_DOWN from block-scaled e4m3 codes of W_down and H
  TC2_FWD_UP_T = 9,      // H as TC2_FWD_UP, and (for the backward) the pre-activations
                         // A = X W_gate^T, B = X W_up^T as bf16 rows [rows, 2h]
};
// two blocks of 256 rows of one matrix per tile (else gate and up rows)
__host__ __device__ constexpr bool tc2_down(int op) {
  return op == TC2_FWD_DOWN || op == TC2_BWD_DH || op == TC2_BWD_DX || op == TC2_FWD_DOWN_B8;
}
// block-scaled e4m3 products: scales in TMEM, one more warp stages them
__host__ __device__ constexpr bool tc2_blk(int op) {
  return op == TC2_FWD_UP_B8 || op == TC2_FWD_DOWN_B8;
}
__host__ __device__ constexpr int tc2_threads(int op) {
  return 32 * (3 + TC_EPI_WARPS + (tc2_blk(op) ? 1 : 0));
}
#define TC2_SF_WARP (TC_TOKEN_WARP + 1)
// Token tiles of the block-scaled products hold at most 240 tokens: TMEM
// keeps two accumulators of N columns (0.. and 256..) and two scale sets of
// 16 columns (240.. and 496..).
#define TC2_BLK_BN 240

// Exponent words of the block-scaled products: one byte per 128-wide block,
// the scale 2^(byte - 127), four consecutive blocks of a row per word (byte
// j = block 4 w + j).  Weights: [row blocks][wg] words (wa0 / wa1 routed:
// gate / up, or down for both; swa0 / swa1 shared).  Activations: act
// [ceil(K / 512)][act_rows] words -- the tokens x for gate/up (a routed
// row's token is perm[row] / k), the hidden rows for down.  hq / hq_exp:
// the first GEMM's outputs, H as codes [hq_rows, h] and its exponent words
// [ceil(h / 512)][hq_rows].
struct Fp8Blk {
  const uint32_t *wa0, *wa1, *swa0, *swa1;
  int wg;
  const uint32_t* act;
  int act_rows;
  const int32_t* perm;
  int k;
  uint8_t* hq;
  uint32_t* hq_exp;
  int hq_rows;
};

// 4 x 4 byte transpose inside each group of 4 consecutive lanes: lane i
// holds row i (byte j = column j) and ends up with column i.
MOE_DEV uint32_t transpose4x4_b8(uint32_t w, int lane) {
  uint32_t r = __shfl_xor_sync(0xffffffffu, w, 2);
  w = (lane & 2) ? __byte_perm(w, r, 0x3276) : __byte_perm(w, r, 0x5410);
  r = __shfl_xor_sync(0xffffffffu, w, 1);
  return (lane & 1) ? __byte_perm(w, r, 0x3715) : __byte_perm(w, r, 0x6240);
}
// the weight operand is MN-major (the weights' transpose is multiplied)
__host__ __device__ constexpr bool tc2_mn_a(int op) { return op == TC2_BWD_DH || op == TC2_BWD_DX; }

#define TC2_THREADS TC_THREADS
#define TC2_CONSUMERS (TC_EPI_WARPS + 2)  // per CTA: epilogue warps, token producer, MMA or weight producer

// NACC accumulators of 256 columns per tile (2: gate and up, or two blocks
// of down-projection rows; 1: one block) and NBUF TMEM buffers of them
// (NACC * NBUF <= 2): with two buffers the epilogue of one tile overlaps the
// MMAs of the next.
// OUTB: output boxes staged per epilogue warp (0: the epilogue stores from
// registers; 1 or 2: bf16 outputs go out by TMA store from shared memory).
template <int SA, int SB, int NACC, int NBUF, int OUTB, bool BLK = false>
struct Tc2Cfg {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;  // 16 KB per weight sub-tile
  static constexpr int A_STAGE = NACC * A_BYTES;
  static constexpr int B_STAGE = 128 * TC_BK * 2;    // half of a 256-token tile
  static constexpr int B_OFF = SA * A_STAGE;
  static constexpr int STG_OFF = B_OFF + SB * B_STAGE;
  // block-scaled products: two stages of scale words (four 32 x 16-byte
  // copy sources each), then the H-amax exchange [2 halves][2][4 warps][32]
  static constexpr int SF_STAGE = 2048;
  static constexpr int SF_OFF = STG_OFF + TC_EPI_WARPS * OUTB * TC_BOX_BYTES;
  static constexpr int XCH_OFF = SF_OFF + (BLK ? 2 * SF_STAGE : 0);
  static constexpr int BAR_OFF = XCH_OFF + (BLK ? 2 * 2 * 4 * 32 * 4 : 0);
  // a_full, a_empty [SA]; b_full, b_empty [SB]; acc_full, acc_empty [2];
  // drain; tile_full, tile_empty [RING]
  // (+ block-scaled: sf_full, sf_empty [2]; the exchange's [2 halves][2])
  static constexpr int N_BARS = 2 * SA + 2 * SB + 5 + 2 * TC_TILE_RING + (BLK ? 8 : 0);
  static constexpr int MISC_BYTES = 4 * TC_TILE_RING + 4 * 5;
  static constexpr int SMEM_BYTES = BAR_OFF + 8 * N_BARS + MISC_BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(NACC * NBUF <= 2 && NACC >= 1 && NBUF >= 1, "TMEM holds two 256-column blocks");
  static_assert(SMEM_BYTES + 64 <= 232448, "shared memory");
  static_assert(SMEM_BYTES > 232448 / 2, "one CTA per SM: the TMEM allocation assumes it");
};

// Geometry of one pair tile as seen by CTA `rank`.
struct Tc2Tile {
  bool shared, v0, v1;  // this CTA's weight sub-tiles exist (rows < n_out)
  bool mma1;            // the second accumulator is computed
  bool reread;          // another token tile of this group reads the same weight rows
  int g, ntok, npad, half, tok0, row_a0, row_a1, row_b, out_row0, pout_row0, out_f0, out_f1;
  uint32_t bytes_a;     // weight bytes of one K step, both CTAs together
};

template <int OP, int NACC>
MOE_DEV Tc2Tile tc2_tile(const GroupTable& G, const int32_t* toff, int E, int b, int n_out,
                         uint32_t rank) {
  constexpr bool DOWN = tc2_down(OP);
  Tc2Tile t;
  const int g = find_group(toff, E, b);
  t.g = g;
  t.shared = g == E;
  const int nt = G.ntt[g];
  t.reread = nt > 1;
  const int local = b - toff[g];
  const int ft = local / nt, tt = local % nt;
  const int n_g = G.off[g + 1] - G.off[g];
  const int tsz = G.tsz[g];
  t.tok0 = tt * tsz;
  t.ntok = min(tsz, n_g - t.tok0);
  t.npad = (t.ntok + 15) & ~15;  // N of the pair MMA: a multiple of 16, half per CTA
  t.half = t.npad / 2;
  // rows of the tile: first GEMM 256 (gate and up alike); second GEMM 256 per
  // accumulator
  const int f0 = ft * (DOWN ? 2 * TC_BM * NACC : 2 * TC_BM);
  const int base = t.shared ? 0 : g * n_out;
  int nsub = 0;  // valid weight sub-tiles of both CTAs
  for (int r = 0; r < 2; ++r) {
    const int a = f0 + TC_BM * r, c = DOWN ? f0 + 2 * TC_BM + TC_BM * r : a;
    nsub += (a < n_out) + (NACC == 2 && c < n_out);
  }
  t.out_f0 = f0 + TC_BM * (int)rank;
  t.out_f1 = DOWN ? f0 + 2 * TC_BM + TC_BM * (int)rank : t.out_f0;
  t.v0 = t.out_f0 < n_out;
  t.v1 = NACC == 2 && t.out_f1 < n_out;
  t.mma1 = NACC == 2 && (DOWN ? f0 + 2 * TC_BM < n_out : true);
  t.row_a0 = base + t.out_f0;
  t.row_a1 = base + t.out_f1;
  t.bytes_a = (uint32_t)nsub * (TC_BM * TC_BK * 2);
  // token rows: x_perm / x (shared) for the gate/up products, H for the
  // down projection, the padded dY rows / dy (shared) for dH, the padded
  // dA|dB rows for dX
  int rb;
  if (OP == TC2_FWD_UP || OP == TC2_FWD_UP_FP8 || OP == TC2_FWD_UP_B8 || OP == TC2_FWD_UP_T)
    rb = t.shared ? t.tok0 : G.off[g] + t.tok0;
  else if (OP == TC2_FWD_DOWN || OP == TC2_FWD_DOWN_B8)
    rb = G.off[g] + t.tok0;
  else if (OP == TC2_BWD_DH) rb = t.shared ? t.tok0 : G.poff[g] + t.tok0;
  else rb = G.poff[g] + t.tok0;
  t.row_b = rb + (int)rank * t.half;
  t.out_row0 = G.off[g] + t.tok0;
  t.pout_row0 = G.poff[g] + t.tok0;
  return t;
}

template <int SA, int SB, int NACC, int NBUF, int OUTB, int OP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(tc2_threads(OP), 1)
k_expert_tc2(const __grid_constant__ TcMapsDev maps, const int32_t* __restrict__ groups, int E,
             int K, int n_out, __nv_bfloat16* __restrict__ out, float* __restrict__ y_sh,
             const __nv_bfloat16* __restrict__ aux, const Fp8Scales fs, const Fp8Blk fb,
             __nv_bfloat16* __restrict__ out2) {
  constexpr bool DOWN = tc2_down(OP);
  constexpr bool MNA = tc2_mn_a(OP);
  constexpr bool FP8U = OP == TC2_FWD_UP_FP8;
  constexpr bool FP8 = FP8U;  // per-row scales, applied in the epilogue
  constexpr bool BLK = tc2_blk(OP);   // block scales, applied by the MMA
  constexpr bool UPB = OP == TC2_FWD_UP_B8;
  constexpr bool UPT = OP == TC2_FWD_UP_T;  // also A|B (out2; TMA stores through maps.aux)
  constexpr int KB_ELEMS = (FP8 || BLK) ? 128 : TC_BK;  // elements per 128-byte K step
  using C = Tc2Cfg<SA, SB, NACC, NBUF, OUTB, BLK>;
  static_assert(OUTB >= 0 && OUTB <= 3, "staged boxes per epilogue warp");
  static_assert(OP != TC2_FWD_UP_T || OUTB == 0 || OUTB == 3, "H, A and B out");
  // second GEMM with both 256-row blocks in one TMEM buffer: staggered blocks
  constexpr bool STAG = DOWN && NACC == 2 && NBUF == 1;
  static_assert(!DOWN || STAG || NACC == 1, "second GEMM: two staggered blocks or one block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  const int32_t* toff = (OP == TC2_FWD_UP || FP8U || UPB || UPT) ? G.toff_a
                        : (OP == TC2_BWD_DH ? G.toff_c : G.toff_b);
  int* counter = G.next + ((FP8U || UPB || UPT) ? TC2_FWD_UP : BLK ? TC2_FWD_DOWN : OP);
  const int total = toff[E + 1];
  // the same decision in both CTAs of the pair (same cluster index)
  if ((int)(blockIdx.x >> 1) >= total) return;
  const SmClockStart clk_start = sm_clock_start();

  uint8_t* bar_base = smem + C::BAR_OFF;
  auto bar = [&](int i) { return smem_u32(bar_base + 8 * i); };
  auto a_full = [&](int s) { return bar(s); };
  auto a_empty = [&](int s) { return bar(SA + s); };
  auto b_full = [&](int s) { return bar(2 * SA + s); };
  auto b_empty = [&](int s) { return bar(2 * SA + SB + s); };
  auto acc_full = [&](int u) { return bar(2 * SA + 2 * SB + u); };
  auto acc_empty = [&](int u) { return bar(2 * SA + 2 * SB + 2 + u); };
  const uint32_t drain_bar = bar(2 * SA + 2 * SB + 4);
  auto tile_full = [&](int s) { return bar(2 * SA + 2 * SB + 5 + s); };
  auto tile_empty = [&](int s) { return bar(2 * SA + 2 * SB + 5 + TC_TILE_RING + s); };
  constexpr int SFB0 = 2 * SA + 2 * SB + 5 + 2 * TC_TILE_RING;
  auto sf_full = [&](int s) { return bar(SFB0 + s); };
  auto sf_empty = [&](int s) { return bar(SFB0 + 2 + s); };
  auto xch_bar = [&](int hf, int par) { return bar(SFB0 + 4 + 2 * hf + par); };
  uint8_t* misc = bar_base + 8 * C::N_BARS;
  volatile int* tile_id = reinterpret_cast<volatile int*>(misc);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(misc + 4 * TC_TILE_RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4 * TC_TILE_RING + 4);
  volatile int* progress = reinterpret_cast<volatile int*>(misc + 4 * TC_TILE_RING + 8);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(a_full(s), 1);   // the leader's arrive + both CTAs' bytes
      mbar_init(a_empty(s), 1);  // the leader's multicast commit
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_empty(s), 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(acc_full(u), 1);
      mbar_init(acc_empty(u), 2 * TC_EPI_WARPS);  // epilogue warps of both CTAs
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < TC_TILE_RING; ++s) {
      mbar_init(tile_full(s), 1);
      mbar_init(tile_empty(s), 2 * (TC2_CONSUMERS + (BLK ? 1 : 0)));  // consumers of both CTAs
    }
    if (BLK) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(sf_full(s), 2);   // the scale warps of both CTAs (leader's barrier)
        mbar_init(sf_empty(s), 1);  // the leader's multicast commit
      }
      for (int i = 0; i < 4; ++i) mbar_init(xch_bar(i >> 1, i & 1), 4);  // the four lane quarters
    }
    *abort_flag = 0;
    progress[0] = progress[1] = progress[2] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nkb = K / TC_BK;
  bool mma_issued = false;

  // leader's barriers as seen from this CTA
  auto lead = [&](uint32_t a) { return leader ? a : cluster_map(a, 0); };
  auto release_tile = [&](int s) {
    if (leader) mbar_arrive(tile_empty(s)); else mbar_arrive_cluster(cluster_map(tile_empty(s), 0));
  };
  auto next_tile = [&](int i, bool arrive) -> int {
    const int s = i % TC_TILE_RING;
    if (!mbar_wait_cluster(tile_full(s), (i / TC_TILE_RING) & 1)) {
      *abort_flag = 1;
      return -1;
    }
    const int b = tile_id[s];
    if (arrive) release_tile(s);
    return b;
  };

  if (warp == 0) {
    // ---------- weight (A) producer; in the leader also the scheduler.  The
    // whole warp runs the loop (waits and tile geometry warp-uniform); lane 0
    // takes tiles and publishes them, one elected lane issues the copies ----------
    const uint32_t F = 0xffffffffu;
    // weight rows read by one token tile: evict first; rows that the group's
    // other token tiles (taken at about the same time by other pairs) read
    // again: normal priority, so that they meet in L2
    const uint64_t pol_once = l2_policy_evict_first(), pol_again = l2_policy_evict_normal();
    int it = 0;
    for (int i = 0;; ++i) {
      int b;
      if (leader) {
        const int s = i % TC_TILE_RING;
        if (i >= TC_TILE_RING &&
            !__all_sync(F, mbar_wait_cluster(tile_empty(s), ((i / TC_TILE_RING) & 1) ^ 1))) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        int bl = 0;
        if (lane == 0) {
          bl = *abort_flag ? total : atomicAdd(counter, 1);
          if (bl >= total) bl = -1;
          tile_id[s] = bl;
          st_cluster_u32(cluster_map(smem_u32(const_cast<int*>(&tile_id[s])), 1), (uint32_t)bl);
          mbar_arrive(tile_full(s));
          mbar_arrive_cluster(cluster_map(tile_full(s), 1));
        }
        b = __shfl_sync(F, bl, 0);
      } else {
        b = __shfl_sync(F, next_tile(i, false), 0);
        __syncwarp();
        if (lane == 0) release_tile(i % TC_TILE_RING);
      }
      if (b < 0) break;
      const Tc2Tile t = tc2_tile<OP, NACC>(G, toff, E, b, n_out, rank);
      const CUtensorMap* mA0 = t.shared ? &maps.sa0 : &maps.a0;
      const CUtensorMap* mA1 = DOWN ? mA0 : (t.shared ? &maps.sa1 : &maps.a1);
      const uint64_t pol_w = t.reread ? pol_again : pol_once;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int sa = it % SA, r = it / SA;
        const bool ok1 = !*abort_flag && (it < SA || mbar_wait(a_empty(sa), (r & 1) ^ 1));
        if (!__all_sync(F, ok1)) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + sa * C::A_STAGE;
        const uint32_t fb = lead(a_full(sa));
        if (elect_one()) {
          if (leader) mbar_arrive_expect_tx(a_full(sa), t.bytes_a);
          if (MNA) {
            // rows kb*64 .. +63 of the K dimension of the transposed weights,
            // M columns out_f .. +127 as two 64-column blocks 8 KB apart
            const int kr = OP == TC2_BWD_DX ? K / 2 : K;  // K rows per matrix
            const int kk0 = kb * TC_BK;
            const bool second = OP == TC2_BWD_DX && kk0 >= kr;
            const CUtensorMap* mA = t.shared ? (second ? &maps.sa1 : &maps.sa0)
                                             : (second ? &maps.a1 : &maps.a0);
            const int y = (t.shared ? 0 : t.g * kr) + (second ? kk0 - kr : kk0);
            if (t.v0) {
              tma_load_2d_pair(smem_u32(st), mA, fb, t.out_f0, y, pol_w);
              tma_load_2d_pair(smem_u32(st + C::A_BYTES / 2), mA, fb, t.out_f0 + 64, y, pol_w);
            }
            if (t.v1) {
              tma_load_2d_pair(smem_u32(st + C::A_BYTES), mA, fb, t.out_f1, y, pol_w);
              tma_load_2d_pair(smem_u32(st + C::A_BYTES + C::A_BYTES / 2), mA, fb, t.out_f1 + 64,
                               y, pol_w);
            }
          } else {
            if (t.v0) tma_load_2d_pair(smem_u32(st), mA0, fb, kb * KB_ELEMS, t.row_a0, pol_w);
            if (t.v1)
              tma_load_2d_pair(smem_u32(st + C::A_BYTES), mA1, fb, kb * KB_ELEMS, t.row_a1, pol_w);
          }
          progress[0] = it + 1;
        }
        __syncwarp();
      }
    }
    __syncwarp();
  } else if (warp == TC_TOKEN_WARP) {
    // ---------- token-row (B) producer: this CTA's half of the tile (the
    // whole warp runs the loop, one elected lane issues the copies) ----------
    const uint32_t F = 0xffffffffu;
    const uint64_t pol_x = l2_policy_evict_last();
    int it = 0;
    for (int i = 0;; ++i) {
      const int b = __shfl_sync(F, next_tile(i, false), 0);
      __syncwarp();
      if (lane == 0) release_tile(i % TC_TILE_RING);
      if (b < 0) break;
      const Tc2Tile t = tc2_tile<OP, NACC>(G, toff, E, b, n_out, rank);
      const bool bs =
          (OP == TC2_FWD_UP || OP == TC2_BWD_DH || FP8U || UPB || UPT) &&
          t.shared;
      const CUtensorMap* m128 = bs ? &maps.bs128 : &maps.b128;
      const CUtensorMap* m64 = bs ? &maps.bs64 : &maps.b64;
      const CUtensorMap* m16 = bs ? &maps.bs16 : &maps.b16;
      const CUtensorMap* m8 = bs ? &maps.bs8 : &maps.b8;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int sb = it % SB, r = it / SB;
        const bool ok1 = !*abort_flag && (it < SB || mbar_wait(b_empty(sb), (r & 1) ^ 1));
        if (!__all_sync(F, ok1)) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + C::B_OFF + sb * C::B_STAGE;
        const uint32_t fb = lead(b_full(sb));
        const int kx = kb * KB_ELEMS;
        if (elect_one()) {
          if (leader) mbar_arrive_expect_tx(b_full(sb), (uint32_t)t.npad * (TC_BK * 2));
          int j = 0;
          for (; j + 128 <= t.half; j += 128)
            tma_load_2d_pair(smem_u32(st + j * (TC_BK * 2)), m128, fb, kx, t.row_b + j, pol_x);
          for (; j + 64 <= t.half; j += 64)
            tma_load_2d_pair(smem_u32(st + j * (TC_BK * 2)), m64, fb, kx, t.row_b + j, pol_x);
          for (; j + 16 <= t.half; j += 16)
            tma_load_2d_pair(smem_u32(st + j * (TC_BK * 2)), m16, fb, kx, t.row_b + j, pol_x);
          for (; j < t.half; j += 8)
            tma_load_2d_pair(smem_u32(st + j * (TC_BK * 2)), m8, fb, kx, t.row_b + j, pol_x);
          progress[1] = it + 1;
        }
        __syncwarp();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (leader) {
      // ---------- MMA issuer (leader only): the whole warp runs the loop
      // (waits, tile geometry, descriptors), one elected lane issues the
      // tcgen05 instructions; every wait's outcome is made warp-uniform ----------
      const uint32_t F = 0xffffffffu;
      int it = 0, tl = 0;
      int qsf = 0;  // block-scaled: scale groups (4 K steps each) of the tiles before this one
      for (int i = 0;; ++i) {
        const int b = __shfl_sync(F, next_tile(i, false), 0);
        __syncwarp();
        if (lane == 0) release_tile(i % TC_TILE_RING);
        if (b < 0) break;
        if (__any_sync(F, *abort_flag != 0)) continue;  // keep reading the tile ring until "none"
        const Tc2Tile t = tc2_tile<OP, NACC>(G, toff, E, b, n_out, 0);
        const uint32_t idesc = FP8 ? umma_idesc_e4m3(2 * TC_BM, t.npad)
                                   : umma_idesc_bf16(2 * TC_BM, t.npad) | (MNA ? (1u << 15) : 0u);
        // Block-scaled: the scale words of K steps 4 j .. 4 j + 3 (group
        // j) are copied from the scale warps' stage into TMEM set (qsf + j)
        // & 1 before the group's first MMA (the copy and the MMAs issued
        // after it run in order), and the set and stage are released by a
        // commit after the group's last MMA.  The copy into a set comes
        // after the scale warp refilled its stage, which it does only after
        // that commit: the MMAs of the group two back have completed.
        int g_loaded = -1;
        auto sf_col = [&](int kb) {
          return tmem + (((qsf + (kb >> 2)) & 1) ? 496u : 240u);
        };
        auto ensure_sf = [&](int kb) -> bool {
          if constexpr (BLK) {
            while (g_loaded < (kb >> 2)) {
              ++g_loaded;
              const int q = qsf + g_loaded;
              if (!__all_sync(F, mbar_wait_cluster(sf_full(q & 1), (q >> 1) & 1))) return false;
              tc_fence_after();
              const uint32_t col = tmem + ((q & 1) ? 496u : 240u);
              const uint32_t src = smem_u32(smem + C::SF_OFF + (q & 1) * C::SF_STAGE);
              if (elect_one()) {
                tmem_cp_pair_32x128b(col, smem_desc_rows16(src));             // A rows, accumulator 0
                tmem_cp_pair_32x128b(col + 4, smem_desc_rows16(src + 512));   // A rows, accumulator 1
                tmem_cp_pair_32x128b(col + 8, smem_desc_rows16(src + 1024));  // tokens 0 .. 127
                if (t.npad > 128) tmem_cp_pair_32x128b(col + 12, smem_desc_rows16(src + 1536));
              }
              __syncwarp();
            }
          }
          return true;
        };
        auto release_sf = [&](int kb, int w) {
          if (BLK && w == (t.mma1 ? 1 : 0) && ((kb & 3) == 3 || kb == nkb - 1)) {
            if (elect_one()) umma_commit_pair(sf_empty((qsf + (kb >> 2)) & 1));
            __syncwarp();
          }
        };
        const int u = tl % NBUF;  // TMEM buffer of this tile
        // k step kb of this tile uses ring stage it + kb
        auto stage_ready = [&](int kb) -> bool {
          const int st = it + kb;
          const bool ok1 =
              mbar_wait(a_full(st % SA), (st / SA) & 1) && mbar_wait(b_full(st % SB), (st / SB) & 1);
          if (!__all_sync(F, ok1)) return false;
          tc_fence_after();
          return true;
        };
        auto acc_ready = [&](int ab, int parity) -> bool {
          const bool ok1 = mbar_wait_cluster(acc_empty(ab), parity);
          return __all_sync(F, ok1);
        };
        // the four K=16 MMAs of k step kb into accumulator w (0: columns
        // 256 u, 1: columns 256).  Operand descriptors: one per operand and
        // call, the four K slices as constant offsets in the start-address
        // field (32 bytes = 2 units for K-major rows, 2048 bytes = 128 units
        // for 16-row MN-major slices; the field stays below 2^14 for every
        // shared-memory address).
        auto issue = [&](int kb, int w) {
          const int st = it + kb;
          const uint32_t a = smem_u32(smem + (st % SA) * C::A_STAGE) + (uint32_t)(w * C::A_BYTES);
          const uint32_t bb = smem_u32(smem + C::B_OFF + (st % SB) * C::B_STAGE);
          const uint32_t d = tmem + (w ? 256u : (uint32_t)(u * 256));
          const uint64_t ad = MNA ? umma_desc_sw128_mn(a, C::A_BYTES / 2) : umma_desc_sw128(a);
          const uint64_t bd = umma_desc_sw128(bb);
          constexpr uint64_t A_STEP = MNA ? (2048 >> 4) : (32 >> 4);
          if (BLK) {
            const uint32_t id = umma_idesc_mx_e4m3(2 * TC_BM, t.npad, (uint32_t)(kb & 3));
            const uint32_t sfa = sf_col(kb) + (w ? 4u : 0u), sfb = sf_col(kb) + 8u;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // four 32-byte K slices
                umma_mx_pair(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), id, sfa, sfb,
                             (kb | kk) != 0);
            }
          } else if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (FP8)
                umma_f8_pair(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc,
                             (kb | kk) != 0);
              else
                umma_bf16_pair(d, ad + A_STEP * kk, bd + (uint64_t)(2 * kk), idesc,
                               (kb | kk) != 0);
            }
          }
          __syncwarp();
          mma_issued = true;
        };
        auto release = [&](int kb) {  // the stage is free once its MMAs complete
          const int st = it + kb;
          if (elect_one()) {
            umma_commit_pair(a_empty(st % SA));
            umma_commit_pair(b_empty(st % SB));
            progress[2] = st + 1;
          }
          __syncwarp();
        };
        auto commit_acc = [&](int ab) {
          if (elect_one()) umma_commit_pair(acc_full(ab));
          __syncwarp();
        };
        bool ok;
        if (STAG) {
          // Second GEMM: block 0 runs S k steps ahead of block 1 at the
          // start of the tile and finishes S k steps before it, so the
          // drain of each block overlaps MMAs of the other.
          // (block-scaled: S <= 4, so block 0 is never more than one scale
          // group ahead of block 1 and two TMEM scale sets suffice)
          const int S = min(min(min(SA, SB), nkb / 2), BLK ? 4 : 64);
          ok = tl == 0 || acc_ready(0, (tl - 1) & 1);
          tc_fence_after();
          for (int kb = 0; ok && kb < S; ++kb)
            if ((ok = stage_ready(kb) && ensure_sf(kb))) {
              issue(kb, 0);
              release_sf(kb, 0);
            }
          ok = ok && (tl == 0 || acc_ready(1, (tl - 1) & 1));
          tc_fence_after();
          for (int kb = 0; ok && kb < S; ++kb) {
            if (t.mma1) issue(kb, 1);
            release_sf(kb, 1);
            release(kb);
          }
          for (int kb = S; ok && kb < nkb - S; ++kb) {
            if ((ok = stage_ready(kb) && ensure_sf(kb))) {
              issue(kb, 0);
              release_sf(kb, 0);
              if (t.mma1) issue(kb, 1);
              release_sf(kb, 1);
              release(kb);
            }
          }
          for (int kb = nkb - S; ok && kb < nkb; ++kb)
            if ((ok = stage_ready(kb) && ensure_sf(kb))) {
              issue(kb, 0);
              release_sf(kb, 0);
            }
          if (ok) commit_acc(0);
          for (int kb = nkb - S; ok && kb < nkb; ++kb) {
            if (t.mma1) issue(kb, 1);
            release_sf(kb, 1);
            release(kb);
          }
          if (ok) commit_acc(1);
        } else {
          ok = tl < NBUF || acc_ready(u, ((tl / NBUF) - 1) & 1);
          tc_fence_after();
          for (int kb = 0; ok && kb < nkb; ++kb) {
            if ((ok = stage_ready(kb) && ensure_sf(kb))) {
              issue(kb, 0);
              release_sf(kb, 0);
              if (t.mma1) issue(kb, 1);
              release_sf(kb, 1);
              release(kb);
            }
          }
          if (ok) commit_acc(u);
        }
        if (!ok) {
          if (lane == 0) *abort_flag = 1;
          __syncwarp();
          continue;
        }
        it += nkb;
        qsf += (nkb + 3) >> 2;
        ++tl;
      }
    }  // the peer has no MMA role
    __syncwarp();
  } else if (BLK && warp == TC2_SF_WARP) {
    // ---------- block scales (both CTAs): the exponent words of each group
    // of 4 K steps, in the layout tcgen05.cp .32x128b.warpx4 copies into
    // TMEM -- 32 rows of 16 bytes, row r holding the words of rows (or
    // tokens) r, r + 32, r + 64, r + 96.  This CTA's 128 weight rows of each
    // accumulator share one block row, so their 32 x 4 words are all that
    // block's word; every token column needs its own word, and both CTAs
    // hold all the tile's tokens (each CTA's rows meet every token). ----------
    const uint32_t F = 0xffffffffu;
    const int ng = (nkb + 3) >> 2;
    int q = 0;
    for (int i = 0;; ++i) {  // after an abort, keep reading the tile ring until "none"
      int b = 0;
      if (lane == 0) b = next_tile(i, true);
      b = __shfl_sync(F, b, 0);
      if (b < 0) break;
      const Tc2Tile t = tc2_tile<OP, NACC>(G, toff, E, b, n_out, rank);
      const uint32_t* wa0 = t.shared ? fb.swa0 : fb.wa0;
      const uint32_t* wa1 = t.shared ? fb.swa1 : fb.wa1;
      const int rb0 = t.row_a0 / TC_BM, rb1 = t.row_a1 / TC_BM;
      int arow[8];  // activation row of token column lane + 32 j (-1: none)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int n = lane + 32 * j;
        arow[j] = n >= t.ntok ? -1
                  : !UPB      ? t.out_row0 + n
                  : t.shared  ? t.tok0 + n
                              : fb.perm[t.out_row0 + n] / fb.k;
      }
      for (int gi = 0; gi < ng; ++gi, ++q) {
        const int s = q & 1;
        int ok = 1;
        if (lane == 0)
          ok = !*abort_flag && (q < 2 || mbar_wait(sf_empty(s), ((q >> 1) - 1) & 1));
        if (!__shfl_sync(F, ok, 0)) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + C::SF_OFF + s * C::SF_STAGE;
        const uint32_t w0 = t.v0 ? wa0[(size_t)rb0 * fb.wg + gi] : 0x7f7f7f7fu;
        const uint32_t w1 = (NACC == 2 && (UPB || t.v1)) ? wa1[(size_t)rb1 * fb.wg + gi] : 0x7f7f7f7fu;
        uint32_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v[j] = arow[j] >= 0 ? fb.act[(size_t)gi * fb.act_rows + arow[j]] : 0x7f7f7f7fu;
        reinterpret_cast<uint4*>(st)[lane] = make_uint4(w0, w0, w0, w0);
        reinterpret_cast<uint4*>(st + 512)[lane] = make_uint4(w1, w1, w1, w1);
        reinterpret_cast<uint4*>(st + 1024)[lane] = make_uint4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<uint4*>(st + 1536)[lane] = make_uint4(v[4], v[5], v[6], v[7]);
        fence_proxy_async_smem();  // visible to the tensor core's copy
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(sf_full(s)); else mbar_arrive_cluster(cluster_map(sf_full(s), 0));
        }
      }
    }
  } else {
    // ---------- epilogue warps 2 .. 2+TC_EPI_WARPS-1 (both CTAs) ----------
    // Warp (q, half) drains TMEM lanes 32 q .. +31 (its 32 output rows),
    // token columns 32 half + 64 j.  Gate/up tiles drain both accumulators
    // at once (SwiGLU, or its gradient); two-block tiles drain block 0, free
    // it, then block 1.  bf16 outputs of 32 whole tokens go out through
    // shared memory by TMA store; the rest (a ragged last chunk, the shared
    // expert's fp32 dX rows of the backward) from registers.
    constexpr bool F32SH = OP == TC2_BWD_DX;  // the shared expert's dX rows in fp32
    const int q = warp & 3, half = (warp - 2) >> 2;
    const uint32_t stg = smem_u32(smem + C::STG_OFF) + (uint32_t)((warp - 2) * OUTB * TC_BOX_BYTES);
    const uint32_t lanes = tmem + ((uint32_t)(q * 32) << 16);
    int tl = 0, nbox = 0, nch = 0;
    for (int i = 0;; ++i) {
      const int b = next_tile(i, false);
      __syncwarp();
      if (lane == 0) release_tile(i % TC_TILE_RING);
      if (b < 0) break;
      const Tc2Tile t = tc2_tile<OP, NACC>(G, toff, E, b, n_out, rank);
      const int u = tl % NBUF;
      for (int ph = 0; ph < (STAG ? 2 : 1); ++ph) {
        const int bi = STAG ? ph : u;  // barrier pair of this phase
        if (*abort_flag || !mbar_wait(acc_full(bi), STAG ? (tl & 1) : ((tl / NBUF) & 1))) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t ta = lanes + (uint32_t)((STAG ? ph : u) * 256);  // this phase's accumulator
        const uint32_t tb = lanes + 256;                                // GEMM 1: up projection
        const bool valid = ph ? t.v1 : t.v0;
        const int of = (ph ? t.out_f1 : t.out_f0) + 32 * q;  // first output column of the warp
        // fp8: scales of this warp's weight rows (row of + lane for the
        // register path; of + lane/4 + 8 r for the fragment layout)
        float rsg[4] = {1.f, 1.f, 1.f, 1.f}, rsu[4] = {1.f, 1.f, 1.f, 1.f}, rlg = 1.f, rlu = 1.f;
        if (FP8 && valid) {
          const float* sgp = t.shared ? fs.sg : fs.g + (size_t)t.g * n_out;
          const float* sup = t.shared ? fs.su : fs.u + (size_t)t.g * n_out;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            rsg[r] = sgp[of + (lane >> 2) + 8 * r];
            rsu[r] = sup[of + (lane >> 2) + 8 * r];
          }
          rlg = sgp[of + lane];
          rlu = sup[of + lane];
        }
        for (int c = 32 * half; c < t.npad; c += 64) {
          if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
          if (UPB) {
            // H of 32 tokens x this warp's 32 hidden units, quantized: the
            // CTA's 128 hidden units of a token are one 1 x 128 block, spread
            // over the four lane quarters, so the four warps of this half
            // exchange their per-token maxima (|h| as bits: NaN above inf
            // above every finite value) through shared memory.  (valid is
            // the same for the four warps: it depends only on the CTA.)
            if (!valid) continue;
            const uint32_t F = 0xffffffffu;
            float va[32], vb[32];
            tmem_load_2x32(ta + c, tb + c, va, vb);
            uint32_t mine = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              va[j] = silu_fast(va[j]) * vb[j];
              const uint32_t m = __reduce_max_sync(F, __float_as_uint(va[j]) & 0x7fffffffu);
              if (lane == j) mine = m;
            }
            const int par = nch & 1;
            volatile uint32_t* xch = reinterpret_cast<volatile uint32_t*>(smem + C::XCH_OFF) +
                                     (size_t)((half * 2 + par) * 4) * 32;
            xch[q * 32 + lane] = mine;
            __syncwarp();
            if (lane == 0) mbar_arrive(xch_bar(half, par));
            const bool got = mbar_wait(xch_bar(half, par), (nch >> 1) & 1);
            ++nch;
            if (!__all_sync(F, got)) {
              if (lane == 0) *abort_flag = 1;
              break;
            }
            const uint32_t amax = max(max(xch[lane], xch[32 + lane]), max(xch[64 + lane], xch[96 + lane]));
            const int e = block_exp_from_bits(amax);
            const float inv = exp2_neg(e);
            const int kbh = t.out_f0 / TC_BM;  // the block's index along h
            if (q == 0 && c + lane < t.ntok)
              reinterpret_cast<uint8_t*>(fb.hq_exp)[((size_t)(kbh >> 2) * fb.hq_rows + t.out_row0 + c +
                                                     lane) * 4 + (kbh & 3)] = (uint8_t)(e + 127);
            // codes: word p of this lane = tokens 4p .. 4p+3 of its hidden
            // unit, then a 4 x 4 byte transpose per group of 4 lanes gives
            // lane 4m + i token 4p + i's hidden units 4m .. 4m + 3
            uint8_t* hq = fb.hq + (size_t)(t.out_row0 + c) * n_out + of + 4 * (lane >> 2);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const float i0 = __shfl_sync(F, inv, 4 * p), i1 = __shfl_sync(F, inv, 4 * p + 1);
              const float i2 = __shfl_sync(F, inv, 4 * p + 2), i3 = __shfl_sync(F, inv, 4 * p + 3);
              uint32_t w = (uint32_t)cvt_e4m3x2(va[4 * p] * i0, va[4 * p + 1] * i1) |
                           ((uint32_t)cvt_e4m3x2(va[4 * p + 2] * i2, va[4 * p + 3] * i3) << 16);
              w = transpose4x4_b8(w, lane);
              const int tok = 4 * p + (lane & 3);
              if (c + tok < t.ntok) *reinterpret_cast<uint32_t*>(hq + (size_t)tok * n_out) = w;
            }
            continue;
          }
          if (UPT && OUTB == 3 && c + 32 <= t.ntok) {
            // 32 whole tokens: H, and the pre-activations A (gate) and B
            // (up) for the backward, staged as three boxes and stored by TMA
            // (H rows of `out`; A|B rows [rows, 2h] through maps.aux)
            if (lane == 0) bulk_wait_read<0>();  // the last chunk's stores have read the boxes
            __syncwarp();
            stage_box_bf16<true>(ta + c, tb + c, stg, lane);
            stage_box_bf16<false>(ta + c, tb + c, stg + TC_BOX_BYTES, lane);
            stage_box_bf16<false>(tb + c, tb + c, stg + 2 * TC_BOX_BYTES, lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (elect_one()) {  // lane 0 of the converged warp, as for the waits
              if (valid) {
                tma_store_2d(&maps.out, stg, of, t.out_row0 + c);
                tma_store_2d(&maps.aux, stg + TC_BOX_BYTES, of, t.out_row0 + c);
                tma_store_2d(&maps.aux, stg + 2 * TC_BOX_BYTES, n_out + of, t.out_row0 + c);
              }
              bulk_commit();
            }
            __syncwarp();
            continue;
          }
          // fp8: scale of token column c + lane (the token's row of x)
          float tsl = 0.f;
          if (FP8 && c + lane < t.ntok)
            tsl = fs.tok[t.shared ? t.tok0 + c + lane : fs.perm[t.out_row0 + c + lane] / fs.k];
          if (OUTB > 0 && c + 32 <= t.ntok && !(F32SH && t.shared)) {
            // 32 whole tokens of bf16 output: stage the box in shared
            // memory and store it with TMA (boxes used round robin)
            const uint32_t box = stg + (uint32_t)((nbox % (OUTB > 0 ? OUTB : 1)) * TC_BOX_BYTES);
            if (lane == 0) bulk_wait_read<(OUTB > 0 ? OUTB - 1 : 0)>();  // the box's last store read it
            __syncwarp();
            if (FP8) {
              float tsc[8];
#pragma unroll
              for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                  tsc[2 * i + e] = __shfl_sync(0xffffffffu, tsl, 8 * i + 2 * (lane & 3) + e);
              stage_box_scaled<FP8U>(ta + c, tb + c, box, lane, rsg, rsu, tsc);
            } else {
              stage_box_bf16<OP == TC2_FWD_UP>(ta + c, tb + c, box, lane);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (elect_one()) {  // lane 0 of the converged warp, as for the waits
              if (valid) tma_store_2d(&maps.out, box, of, t.out_row0 + c);
              bulk_commit();
            }
            __syncwarp();
            ++nbox;
            continue;
          }
          // from registers: a ragged last chunk, or the shared expert's fp32 dX rows
          float va[32], vb[32];
          if (!DOWN)
            tmem_load_2x32(ta + c, tb + c, va, vb);
          else
            tmem_load_32(ta + c, va);
          if (!valid) continue;
          if (FP8U) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float ts = __shfl_sync(0xffffffffu, tsl, j);
              va[j] = silu_fast(va[j] * (rlg * ts)) * (vb[j] * (rlu * ts));
            }
            store_rows_bf16(out + (size_t)(t.out_row0 + c) * n_out + of, n_out, va, c, t.ntok, lane);
          } else if (OP == TC2_FWD_UP || UPT) {
            if (UPT) {  // the pre-activations first, then H in place
              __nv_bfloat16* ab = out2 + (size_t)(t.out_row0 + c) * (2 * n_out) + of;
              store_rows_bf16(ab, 2 * n_out, va, c, t.ntok, lane);
              store_rows_bf16(ab + n_out, 2 * n_out, vb, c, t.ntok, lane);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) va[j] = silu_fast(va[j]) * vb[j];
            store_rows_bf16(out + (size_t)(t.out_row0 + c) * n_out + of, n_out, va, c, t.ntok, lane);
          } else if (F32SH && t.shared) {
            store_rows_f32(y_sh + (size_t)(t.tok0 + c) * n_out + of, n_out, va, c, t.ntok, lane);
          } else {
            store_rows_bf16(out + (size_t)(t.out_row0 + c) * n_out + of, n_out, va, c, t.ntok, lane);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(acc_empty(bi)); else mbar_arrive_cluster(cluster_map(acc_empty(bi), 0));
        }
      }
      ++tl;
    }
    if (OUTB > 0 && lane == 0) bulk_wait_all();  // this warp's stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && leader) {
    // Unwind (leader): the full barriers count both CTAs' copies; wait for
    // what was issued, then for the MMAs (each wait bounded).
    if (warp == 0 && lane == 0) {
      for (int it = progress[2]; it < progress[0]; ++it)
        mbar_wait(a_full(it % SA), (it / SA) & 1);
    }
    if (warp == TC_TOKEN_WARP && lane == 0) {
      for (int it = progress[2]; it < progress[1]; ++it)
        mbar_wait(b_full(it % SB), (it / SB) & 1);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      umma_commit_pair_local(drain_bar);
      mbar_wait(drain_bar, 0);
    }
    __syncthreads();
  }
  cluster_sync_all();  // neither CTA leaves while the other may still use its memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, C::TMEM_COLS);
  if (threadIdx.x == 0)
    sm_clock_add(MNA ? 2 : DOWN ? 1 : 0, clk_start);  // backward / down / gate-up
}
