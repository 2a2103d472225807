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
// Each tile has two fp32 TMEM accumulators of BN columns:
//   first GEMM (DOWN = false): acc0 = W_gate rows f0..f0+127, acc1 = W_up rows
//       f0..f0+127 (same B tile) -> H[row, f] = bf16(silu(acc0) * acc1)
//   second GEMM (DOWN = true): acc0 / acc1 = W_down rows f0..+127 / f0+128..+255
//       -> Y_perm[row, f] = bf16(acc), for the routed rows and the shared
//       expert's rows TK + t (the gates are applied in the combine)
//
// Pipeline: K steps of 64 elements (128-byte rows, 128-byte swizzle).  The
// weights (A: 2 x 16 KB per step, streamed from DRAM, long latency) and the
// token rows (B: N x 128 B per step, re-read by every output tile of the
// group, mostly L2 hits) have separate shared-memory rings fed by separate
// producer warps, so the weight ring can run deeper than the token ring in
// the same shared memory.  Each ring slot has a "full" mbarrier (TMA
// transaction bytes) and an "empty" mbarrier (tcgen05.commit of the MMAs
// that read it).
//
// Persistent, in order: one CTA per SM; warp 0's lane takes tiles from a
// global counter (zeroed by the scan kernel) in table order, so the tiles in
// flight across the GPU are always a contiguous window of the table -- the
// token tiles of one expert run side by side and share each weight tile
// through L2.  The tile index goes to the other roles through a small ring
// of (tile id, full, empty) slots in shared memory.
//
// Warp roles (352 threads): warp 0 = tile scheduler + weight producer,
// warp 1 = TMEM allocator + MMA issuer, warps 2-9 = epilogue (TMEM ->
// registers -> global; warp w reads TMEM lanes 32*(w%4)..+31, half of the
// token columns each), warp 10 = token-row producer.  The epilogue writes
// whole 16-byte row segments: an 8 x 8 shuffle transpose per group of 8
// lanes turns the accumulator's one-output-row-per-lane layout into 8
// consecutive outputs of one token per lane.  The MMA lane starts a tile once the epilogue has
// drained the previous tile's accumulators ("acc_empty", one arrive per
// epilogue warp) and hands the tile over with "acc_full"; the producers keep
// filling their rings meanwhile.
//
// Every wait is bounded (ptx.cuh).  On a timeout the role stops, the CTA
// drains its copies and MMAs in flight with bounded waits, frees its TMEM
// and returns, leaving the device error word set.
#pragma once

#include "experts_simt.cuh"

#define TC_BM 128
#define TC_BK 64
#define TC_EPI_WARPS 8                         // two per TMEM lane quarter
#define TC_THREADS (32 * (3 + TC_EPI_WARPS))  // scheduler/weights, MMA, epilogue, tokens
#define TC_TOKEN_WARP (2 + TC_EPI_WARPS)
#define TC_TILE_RING 8

// silu(z) = z * sigmoid(z) with the fast exponential and division: their
// relative error (~1e-6) is far below the bf16 rounding of the stored H.
// Where 1 + e^-z exceeds 2^126 (z below about -87.3) the fast division
// gives z * 0: -0, or NaN for z = -inf.  (moe_selftest_silu exposes it to
// the accuracy tests.)
MOE_DEV float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// 8 x 8 transpose of 16-bit values inside each group of 8 consecutive lanes:
// lane i of a group holds row i (positions p = 0..7, w[m] = p 2m | p 2m+1 <<
// 16) and ends up holding column i, packed the same way.  Three butterfly
// stages exchange, with lane i ^ k, the values whose position bit k differs
// from lane bit k (k = 4, 2, 1); six shuffles in all.
MOE_DEV void transpose8x8_b16(uint32_t (&w)[4], int lane) {
  const uint32_t F = 0xffffffffu;
  {
    const bool hi = lane & 4;
    const uint32_t r0 = __shfl_xor_sync(F, hi ? w[0] : w[2], 4);
    const uint32_t r1 = __shfl_xor_sync(F, hi ? w[1] : w[3], 4);
    if (hi) { w[0] = r0; w[1] = r1; } else { w[2] = r0; w[3] = r1; }
  }
  {
    const bool hi = lane & 2;
    const uint32_t r0 = __shfl_xor_sync(F, hi ? w[0] : w[1], 2);
    const uint32_t r1 = __shfl_xor_sync(F, hi ? w[2] : w[3], 2);
    if (hi) { w[0] = r0; w[2] = r1; } else { w[1] = r0; w[3] = r1; }
  }
  {
    const bool hi = lane & 1;
    const uint32_t s0 = hi ? __byte_perm(w[0], w[1], 0x5410) : __byte_perm(w[0], w[1], 0x7632);
    const uint32_t s1 = hi ? __byte_perm(w[2], w[3], 0x5410) : __byte_perm(w[2], w[3], 0x7632);
    const uint32_t r0 = __shfl_xor_sync(F, s0, 1), r1 = __shfl_xor_sync(F, s1, 1);
    if (hi) {
      w[0] = __byte_perm(r0, w[0], 0x7610);
      w[1] = __byte_perm(r0, w[1], 0x7632);
      w[2] = __byte_perm(r1, w[2], 0x7610);
      w[3] = __byte_perm(r1, w[3], 0x7632);
    } else {
      w[0] = __byte_perm(w[0], r0, 0x5410);
      w[1] = __byte_perm(w[1], r0, 0x7610);
      w[2] = __byte_perm(w[2], r1, 0x5410);
      w[3] = __byte_perm(w[3], r1, 0x7610);
    }
  }
}

// 4 x 4 transpose of 32-bit values inside each group of 4 consecutive lanes
// (lane i: row i in f[0..3] -> column i), two butterfly stages.
MOE_DEV void transpose4x4_f32(float (&f)[4], int lane) {
  const uint32_t F = 0xffffffffu;
  {
    const bool hi = lane & 2;
    const float r0 = __shfl_xor_sync(F, hi ? f[0] : f[2], 2);
    const float r1 = __shfl_xor_sync(F, hi ? f[1] : f[3], 2);
    if (hi) { f[0] = r0; f[1] = r1; } else { f[2] = r0; f[3] = r1; }
  }
  {
    const bool hi = lane & 1;
    const float r0 = __shfl_xor_sync(F, hi ? f[0] : f[1], 1);
    const float r1 = __shfl_xor_sync(F, hi ? f[2] : f[3], 1);
    if (hi) { f[0] = r0; f[2] = r1; } else { f[1] = r0; f[3] = r1; }
  }
}

MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Store 32 values of this lane's output row (one per token c0 + j) for the
// warp's 32 consecutive output rows as 16-byte vectors: 8 outputs of one
// token per lane after an 8 x 8 transpose per group of 8 lanes.
// dst = &out[token c0][first output of the warp]; tokens >= ntok are skipped.
MOE_DEV void store_rows_bf16(__nv_bfloat16* dst, size_t ld, const float (&v)[32], int c0,
                             int ntok, int lane) {
  const int grp = lane >> 3, u = lane & 7;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    uint32_t w[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) w[m] = pack_bf16x2(v[8 * r + 2 * m], v[8 * r + 2 * m + 1]);
    transpose8x8_b16(w, lane);
    const int tok = 8 * r + u;
    if (c0 + tok < ntok)
      *reinterpret_cast<uint4*>(dst + (size_t)tok * ld + 8 * grp) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The same for fp32 outputs: 4 outputs of one token per lane (4 x 4 transpose).
MOE_DEV void store_rows_f32(float* dst, size_t ld, const float (&v)[32], int c0, int ntok,
                            int lane) {
  const int grp = lane >> 2, u = lane & 3;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float f[4] = {v[4 * r], v[4 * r + 1], v[4 * r + 2], v[4 * r + 3]};
    transpose4x4_f32(f, lane);
    const int tok = 4 * r + u;
    if (c0 + tok < ntok)
      *reinterpret_cast<float4*>(dst + (size_t)tok * ld + 4 * grp) = make_float4(f[0], f[1], f[2], f[3]);
  }
}

// Staged output box: 32 tokens x 32 outputs of bf16 in shared memory, one
// 64-byte row per token, its four 16-byte chunks swizzled as the TMA 64-byte
// swizzle expects (chunk ^ ((row >> 1) & 3)), so that the eight rows written
// by each stmatrix fall into eight different bank groups.
#define TC_BOX_BYTES 2048

// One warp stages TMEM columns c .. c+31 of its 32 lanes (ta, tb: the
// addresses of column c in the warp's lane quarter) into `box`: box row j =
// column c + j (a token), 32 outputs (the lanes) per row.  Values are
// silu(acc a) * acc b when SWIGLU, else acc a, rounded to bf16.  The 16x256b
// loads give each thread pairs of adjacent columns of one lane -- the
// fragment layout of an 8 x 8 matrix -- and stmatrix .trans writes the
// transpose, 8 outputs of one token per 16-byte row piece.
template <bool SWIGLU>
MOE_DEV void stage_box_bf16(uint32_t ta, uint32_t tb, uint32_t box, int lane) {
  const int mm = lane >> 3, ii = lane & 7;
#pragma unroll
  for (int L = 0; L < 32; L += 16) {
    uint32_t ra[16], rb[16];
    if (SWIGLU)
      tmem_load_16x256b_2(ta + ((uint32_t)L << 16), tb + ((uint32_t)L << 16), ra, rb);
    else
      tmem_load_16x256b(ta + ((uint32_t)L << 16), ra);
    // matrix m = 2 i + hf: lanes L + 8 hf .. +7, columns 8 i .. 8 i + 7
    uint32_t w[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      float lo = __uint_as_float(ra[2 * m]), hi = __uint_as_float(ra[2 * m + 1]);
      if (SWIGLU) {
        lo = silu_fast(lo) * __uint_as_float(rb[2 * m]);
        hi = silu_fast(hi) * __uint_as_float(rb[2 * m + 1]);
      }
      w[m] = pack_bf16x2(lo, hi);
    }
    // stmatrix ip covers matrices 4 ip .. 4 ip + 3; thread 8 mm + ii gives
    // the row of token 8 i + ii, outputs L + 8 hf .. +7, of matrix 4 ip + mm
#pragma unroll
    for (int ip = 0; ip < 2; ++ip) {
      const int tok = 8 * (2 * ip + (mm >> 1)) + ii, chunk = (L >> 3) + (mm & 1);
      stmatrix_x4_trans(box + (uint32_t)(tok * 64 + 16 * (chunk ^ ((tok >> 1) & 3))), w[4 * ip],
                        w[4 * ip + 1], w[4 * ip + 2], w[4 * ip + 3]);
    }
  }
}

// stage_box_bf16 for the per-row fp8 products: the accumulators hold sums
// of code products, so each value is first multiplied by its weight row's
// scale and its token's scale (SWIGLU: gate and up, each with its own row
// scales).
// rsg / rsu: scales of the rows (lane >> 2) + 8 r, r = 0..3 of the warp's 32;
// tsc[2 i + e]: scale of token column 8 i + 2 (lane & 3) + e.
template <bool SWIGLU>
MOE_DEV void stage_box_scaled(uint32_t ta, uint32_t tb, uint32_t box, int lane,
                              const float (&rsg)[4], const float (&rsu)[4],
                              const float (&tsc)[8]) {
  const int mm = lane >> 3, ii = lane & 7;
#pragma unroll
  for (int L = 0; L < 32; L += 16) {
    uint32_t ra[16], rb[16];
    if (SWIGLU)
      tmem_load_16x256b_2(ta + ((uint32_t)L << 16), tb + ((uint32_t)L << 16), ra, rb);
    else
      tmem_load_16x256b(ta + ((uint32_t)L << 16), ra);
    uint32_t w[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {  // m = 2 i + hf: rows L + 8 hf + lane/4, columns 8 i ..
      const int r = (L >> 3) + (m & 1), i = m >> 1;
      float o[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float g = __uint_as_float(ra[2 * m + e]) * (rsg[r] * tsc[2 * i + e]);
        if (SWIGLU) {
          const float u = __uint_as_float(rb[2 * m + e]) * (rsu[r] * tsc[2 * i + e]);
          o[e] = silu_fast(g) * u;
        } else {
          o[e] = g;
        }
      }
      w[m] = pack_bf16x2(o[0], o[1]);
    }
#pragma unroll
    for (int ip = 0; ip < 2; ++ip) {
      const int tok = 8 * (2 * ip + (mm >> 1)) + ii, chunk = (L >> 3) + (mm & 1);
      stmatrix_x4_trans(box + (uint32_t)(tok * 64 + 16 * (chunk ^ ((tok >> 1) & 3))), w[4 * ip],
                        w[4 * ip + 1], w[4 * ip + 2], w[4 * ip + 3]);
    }
  }
}

template <int BN, int SA, int SB>
struct TcCfg {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;  // 16 KB per weight sub-tile
  static constexpr int A_STAGE = 2 * A_BYTES;        // both sub-tiles
  static constexpr int B_STAGE = BN * TC_BK * 2;     // BN rows of 128 B
  static constexpr int B_OFF = SA * A_STAGE;
  static constexpr int BAR_OFF = B_OFF + SB * B_STAGE;
  // a_full[SA], a_empty[SA], b_full[SB], b_empty[SB], acc_full, acc_empty,
  // drain, tile_full[RING], tile_empty[RING]
  static constexpr int N_BARS = 2 * SA + 2 * SB + 3 + 2 * TC_TILE_RING;
  // then: tile ids [RING], tmem slot, abort flag, 3 progress counters
  static constexpr int MISC_BYTES = 4 * TC_TILE_RING + 4 * 5;
  static constexpr int SMEM_BYTES = BAR_OFF + 8 * N_BARS + MISC_BYTES + 1024;  // + base alignment
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(SMEM_BYTES + 64 <= 232448, "shared memory");
  static_assert(SMEM_BYTES > 232448 / 2, "one CTA per SM: the TMEM allocation assumes it");
};

// Geometry of one tile, computed identically by every role.
struct TcTile {
  bool shared, has_a1;
  bool reread;  // another token tile of this group reads the same weight rows
  int ntok, npad, tok0, f0, row_a0, row_a1, row_b, out_row0;
};

template <bool DOWN>
MOE_DEV TcTile tc_tile(const GroupTable& G, const int32_t* toff, int E, int b, int n_out) {
  TcTile t;
  const int g = find_group(toff, E, b);
  t.shared = g == E;
  const int nt = G.ntt[g];
  t.reread = nt > 1;
  const int local = b - toff[g];
  const int ft = local / nt, tt = local % nt;
  const int n_g = G.off[g + 1] - G.off[g];
  const int tsz = G.tsz[g];
  t.tok0 = tt * tsz;
  t.ntok = min(tsz, n_g - t.tok0);
  t.npad = (t.ntok + 15) & ~15;
  t.f0 = ft * (DOWN ? 2 * TC_BM : TC_BM);
  t.has_a1 = DOWN ? (t.f0 + TC_BM < n_out) : true;
  t.row_a0 = (t.shared ? 0 : g * n_out) + t.f0;
  t.row_a1 = DOWN ? t.row_a0 + TC_BM : t.row_a0;
  t.row_b = (!DOWN && t.shared) ? t.tok0 : G.off[g] + t.tok0;
  t.out_row0 = G.off[g] + t.tok0;  // H row (first GEMM) / Y_perm row (routed, second)
  return t;
}

// Scales of the per-row fp8 gate/up products: per weight row (g, u routed
// [E*h]; sg, su shared [h]) and per token (tok [T]; a routed row's token is
// perm[row] / k).
struct Fp8Scales {
  const float *g, *u, *sg, *su, *tok;
  const int32_t* perm;
  int k;
};

struct TcMapsDev {
  CUtensorMap a0, a1, sa0, sa1;   // weights, 128-row boxes (routed, shared)
  CUtensorMap b128, b64, b16, b8;     // token rows of the routed groups
  CUtensorMap bs128, bs64, bs16, bs8;  // token rows of the shared group
  CUtensorMap out;                // bf16 output rows (H or Y_perm), 32 x 32 boxes, 64-byte swizzle
  CUtensorMap aux;                // bf16 rows read by the epilogue (dH), boxes as `out`
};

template <int BN, int SA, int SB, bool DOWN>
__global__ void __launch_bounds__(TC_THREADS, 1)
k_expert_tc(const __grid_constant__ TcMapsDev maps, const int32_t* __restrict__ groups, int E,
            int K, int n_out, __nv_bfloat16* __restrict__ out) {
  using C = TcCfg<BN, SA, SB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  GroupTable G = group_table(const_cast<int32_t*>(groups), E);
  const int32_t* toff = DOWN ? G.toff_b : G.toff_a;
  int* counter = G.next + (DOWN ? 1 : 0);
  const int total = toff[E + 1];
  if ((int)blockIdx.x >= total) return;
  const SmClockStart clk_start = sm_clock_start();
  {
    // a CTA-uniform decision: one thread reads the error word
    __shared__ int s_skip;
    if (threadIdx.x == 0) s_skip = *reinterpret_cast<volatile unsigned*>(&g_moe_dev_error) != 0u;
    __syncthreads();
    if (s_skip) return;
  }

  uint8_t* bar_base = smem + C::BAR_OFF;
  auto bar = [&](int i) { return smem_u32(bar_base + 8 * i); };
  auto a_full = [&](int s) { return bar(s); };
  auto a_empty = [&](int s) { return bar(SA + s); };
  auto b_full = [&](int s) { return bar(2 * SA + s); };
  auto b_empty = [&](int s) { return bar(2 * SA + SB + s); };
  const uint32_t acc_full = bar(2 * SA + 2 * SB), acc_empty = bar(2 * SA + 2 * SB + 1);
  const uint32_t drain_bar = bar(2 * SA + 2 * SB + 2);
  auto tile_full = [&](int s) { return bar(2 * SA + 2 * SB + 3 + s); };
  auto tile_empty = [&](int s) { return bar(2 * SA + 2 * SB + 3 + TC_TILE_RING + s); };
  uint8_t* misc = bar_base + 8 * C::N_BARS;
  volatile int* tile_id = reinterpret_cast<volatile int*>(misc);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(misc + 4 * TC_TILE_RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4 * TC_TILE_RING + 4);
  // k-steps issued by the weight producer, by the token producer, consumed by the MMA
  volatile int* progress = reinterpret_cast<volatile int*>(misc + 4 * TC_TILE_RING + 8);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(a_full(s), 1);
      mbar_init(a_empty(s), 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_empty(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, TC_EPI_WARPS);  // one arrive per epilogue warp
    mbar_init(drain_bar, 1);
    for (int s = 0; s < TC_TILE_RING; ++s) {
      mbar_init(tile_full(s), 1);
      mbar_init(tile_empty(s), TC_EPI_WARPS + 2);  // MMA lane, epilogue warps, token producer
    }
    *abort_flag = 0;
    progress[0] = progress[1] = progress[2] = 0;
    fence_barrier_init();
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
  bool mma_issued = false;

  // Tile i of this CTA for a consumer role (-1: no more tiles).  Waits for
  // the scheduler to publish slot i and reads it; `arrive` releases the slot.
  auto next_tile = [&](int i, bool arrive) -> int {
    const int s = i % TC_TILE_RING;
    if (!mbar_wait(tile_full(s), (i / TC_TILE_RING) & 1)) {
      *abort_flag = 1;
      return -1;
    }
    const int b = tile_id[s];
    if (arrive) mbar_arrive(tile_empty(s));
    return b;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------- tile scheduler + weight (A) producer -------------
      // weight rows read by one token tile: evict first; rows that the
      // group's other token tiles (running at about the same time on other
      // SMs) read again: normal priority, so that they meet in L2
      const uint64_t pol_once = l2_policy_evict_first(), pol_again = l2_policy_evict_normal();
      int it = 0;
      for (int i = 0;; ++i) {
        const int s = i % TC_TILE_RING;
        if (i >= TC_TILE_RING && !mbar_wait(tile_empty(s), ((i / TC_TILE_RING) & 1) ^ 1)) {
          *abort_flag = 1;
          break;
        }
        int b = *abort_flag ? total : atomicAdd(counter, 1);
        if (b >= total) b = -1;
        tile_id[s] = b;
        mbar_arrive(tile_full(s));
        if (b < 0) break;
        const TcTile t = tc_tile<DOWN>(G, toff, E, b, n_out);
        const CUtensorMap* mA0 = t.shared ? &maps.sa0 : &maps.a0;
        const CUtensorMap* mA1 = DOWN ? mA0 : (t.shared ? &maps.sa1 : &maps.a1);
        const uint32_t bytes = (t.has_a1 ? 2u : 1u) * C::A_BYTES;
        const uint64_t pol_w = t.reread ? pol_again : pol_once;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int sa = it % SA, r = it / SA;
          if (it >= SA && !mbar_wait(a_empty(sa), (r & 1) ^ 1)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* st = smem + sa * C::A_STAGE;
          const uint32_t fb = a_full(sa);
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_2d(smem_u32(st), mA0, fb, kb * TC_BK, t.row_a0, pol_w);
          if (t.has_a1) tma_load_2d(smem_u32(st + C::A_BYTES), mA1, fb, kb * TC_BK, t.row_a1, pol_w);
          progress[0] = it + 1;
        }
        // after an abort the next published tile is "none" (b = -1 above)
      }
    }
  } else if (warp == TC_TOKEN_WARP) {
    if (lane == 0) {
      // ------------- token-row (B) producer -------------
      const uint64_t pol_x = l2_policy_evict_last();
      int it = 0;
      for (int i = 0;; ++i) {
        const int b = next_tile(i, true);
        if (b < 0) break;
        const TcTile t = tc_tile<DOWN>(G, toff, E, b, n_out);
        const bool bs = !DOWN && t.shared;
        const CUtensorMap* m128 = bs ? &maps.bs128 : &maps.b128;
        const CUtensorMap* m64 = bs ? &maps.bs64 : &maps.b64;
        const CUtensorMap* m16 = bs ? &maps.bs16 : &maps.b16;
        const uint32_t bytes = (uint32_t)t.npad * (TC_BK * 2);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int sb = it % SB, r = it / SB;
          if (*abort_flag || (it >= SB && !mbar_wait(b_empty(sb), (r & 1) ^ 1))) {
            *abort_flag = 1;
            break;
          }
          uint8_t* st = smem + C::B_OFF + sb * C::B_STAGE;
          const uint32_t fb = b_full(sb);
          const int kx = kb * TC_BK;
          mbar_arrive_expect_tx(fb, bytes);
          int j = 0;
          for (; j + 128 <= t.npad; j += 128)
            tma_load_2d(smem_u32(st + j * (TC_BK * 2)), m128, fb, kx, t.row_b + j, pol_x);
          for (; j + 64 <= t.npad; j += 64)
            tma_load_2d(smem_u32(st + j * (TC_BK * 2)), m64, fb, kx, t.row_b + j, pol_x);
          for (; j < t.npad; j += 16)
            tma_load_2d(smem_u32(st + j * (TC_BK * 2)), m16, fb, kx, t.row_b + j, pol_x);
          progress[1] = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------- MMA issuer -------------
      int it = 0, tl = 0;
      for (int i = 0;; ++i) {
        const int b = next_tile(i, true);
        if (b < 0) break;
        const TcTile t = tc_tile<DOWN>(G, toff, E, b, n_out);
        const uint32_t idesc = umma_idesc_bf16(TC_BM, t.npad);
        if (*abort_flag || (tl > 0 && !mbar_wait(acc_empty, (tl - 1) & 1))) {
          *abort_flag = 1;
          continue;  // keep reading the tile ring until the scheduler says "none"
        }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int sa = it % SA, sb = it % SB;
          if (!mbar_wait(a_full(sa), (it / SA) & 1) || !mbar_wait(b_full(sb), (it / SB) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + sa * C::A_STAGE), a1 = a0 + C::A_BYTES;
          const uint32_t bb = smem_u32(smem + C::B_OFF + sb * C::B_STAGE);
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            const uint64_t bdesc = umma_desc_sw128(bb + kk * 32);
            const uint32_t acc = (kb | kk) != 0;
            umma_bf16(tmem, umma_desc_sw128(a0 + kk * 32), bdesc, idesc, acc);
            if (t.has_a1) umma_bf16(tmem + BN, umma_desc_sw128(a1 + kk * 32), bdesc, idesc, acc);
          }
          mma_issued = true;
          umma_commit(a_empty(sa));
          umma_commit(b_empty(sb));
          progress[2] = it + 1;
        }
        if (!ok) {
          *abort_flag = 1;
          continue;
        }
        umma_commit(acc_full);
        ++tl;
      }
    }
    __syncwarp();
  } else {
    // ------------- epilogue warps 2 .. 2+TC_EPI_WARPS-1 -------------
    // Warp w reads TMEM lane quarter w % 4 (its 32 output rows) for every
    // other 32-token chunk (w - 2) / 4 = 0 or 1.  No epilogue warp waits on
    // another: each decides on its own when to stop, so a timeout cannot
    // leave one waiting at a barrier for ever.
    const int q = warp & 3, half = (warp - 2) >> 2;
    const uint32_t tl_addr = tmem + ((uint32_t)(q * 32) << 16);
    int tl = 0;
    for (int i = 0;; ++i) {
      const int b = next_tile(i, false);
      __syncwarp();
      if (lane == 0) mbar_arrive(tile_empty(i % TC_TILE_RING));
      if (b < 0) break;
      const TcTile t = tc_tile<DOWN>(G, toff, E, b, n_out);
      if (*abort_flag || !mbar_wait(acc_full, tl & 1)) {
        *abort_flag = 1;
        continue;  // keep reading the tile ring until the scheduler says "none"
      }
      tc_fence_after();
      const int fw = t.f0 + q * 32;  // first output row of this warp
      for (int c = 32 * half; c < t.npad; c += 64) {
        float va[32], vb[32];
        tmem_load_2x32(tl_addr + c, tl_addr + BN + c, va, vb);
        if (__any_sync(0xffffffffu, *abort_flag != 0)) continue;  // warp-uniform (shuffles below)
        if (!DOWN) {
#pragma unroll
          for (int j = 0; j < 32; ++j) va[j] = silu_fast(va[j]) * vb[j];
          store_rows_bf16(out + (size_t)(t.out_row0 + c) * n_out + fw, n_out, va, c, t.ntok, lane);
        } else {
          __nv_bfloat16* o = out + (size_t)(t.out_row0 + c) * n_out + fw;
          store_rows_bf16(o, n_out, va, c, t.ntok, lane);
          if (t.has_a1) store_rows_bf16(o + TC_BM, n_out, vb, c, t.ntok, lane);
        }
      }
      // the accumulators may be overwritten once every epilogue warp has read them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      ++tl;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Unwind: let every copy this CTA issued land and every MMA it issued
    // finish (each wait bounded) before the shared memory and TMEM go away.
    if (warp == 0 && lane == 0) {
      for (int it = progress[2]; it < progress[0]; ++it)
        mbar_wait(a_full(it % SA), (it / SA) & 1);
    }
    if (warp == TC_TOKEN_WARP && lane == 0) {
      for (int it = progress[2]; it < progress[1]; ++it)
        mbar_wait(b_full(it % SB), (it / SB) & 1);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
  if (threadIdx.x == 0) sm_clock_add(DOWN ? 1 : 0, clk_start);
}
