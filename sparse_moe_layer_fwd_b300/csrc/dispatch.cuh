// dispatch.cuh -- per-expert load counts and a stable token permutation.
//
// The pages' code has no sparse dispatch ("DeepSeek V3 viết lại bằng 190 dòng
// JAX thuần", section "Những gì đã được đơn giản hóa": every expert runs on
// every token).  Here each (token, slot) pair p = t*k + j with expert
// e = topk_idx[p] gets a row pos(p) in an expert-major permuted order:
//   pos(p) = off[e] + #{p' < p : topk_idx[p'] = e},   off = exclusive scan of load
// i.e. a stable counting sort of the pairs by expert.  load[e] is the count
// that drives the bias update ("190行JAX复刻DeepSeek V3", section
// "最有价值的实验:无辅助损失均衡真的有效").
//
// k_block_rank   : one warp per block of PAIRS_PER_BLOCK pairs, in pair order,
//                  __match_any_sync groups equal experts in a 32-pair chunk;
//                  gives each pair its rank among same-expert pairs of the
//                  block and the block's per-expert histogram.
// k_scan_groups  : one CTA.  Per-expert totals (= load counts) and per-block
//                  bases, the exclusive scan off[], and the GEMM tile table
//                  (token tiles per group, tile prefix sums).  Group E is the
//                  shared expert, whose rows are all T tokens.
// k_permute_gather: one warp per pair: pos = base[block][e] + rank,
//                  perm[pos] = p, inv[p] = pos, X_perm[pos] = x[t].
#pragma once

#include "ptx.cuh"

#define MOE_PAIRS_PER_BLOCK 1024
#define MOE_MAX_E 1024

__global__ void __launch_bounds__(32)
k_block_rank(const int32_t* __restrict__ topk_idx, int TK, int E, int32_t* __restrict__ pair_rank,
             int32_t* __restrict__ blk_hist) {
  __shared__ int run[MOE_MAX_E];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) run[e] = 0;
  __syncwarp();
  const int beg = blockIdx.x * MOE_PAIRS_PER_BLOCK;
  const int end = min(TK, beg + MOE_PAIRS_PER_BLOCK);
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = beg; base < end; base += 32) {
    const int p = base + lane;
    const bool valid = p < end;
    const int e = valid ? topk_idx[p] : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int r = __popc(peers & lt);
    int cur = 0;
    if (valid) cur = run[e];
    __syncwarp();
    if (valid) {
      pair_rank[p] = cur + r;
      if (r == 0) run[e] = cur + __popc(peers);
    }
    __syncwarp();
  }
  for (int e = lane; e < E; e += 32) blk_hist[(size_t)blockIdx.x * E + e] = run[e];
}

// Exclusive scan of n ints in shared memory by the whole CTA (blockDim.x a
// multiple of 32, <= 1024).  Returns the total to every thread.
__device__ int cta_exclusive_scan(int* data, int n, int* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  int carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + tid;
    const int v = i < n ? data[i] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) warp_tot[wid] = inc;
    __syncthreads();
    if (wid == 0) {
      int w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nw) warp_tot[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    const int wpre = wid > 0 ? warp_tot[wid - 1] : 0;
    const int chunk_total = warp_tot[nw - 1];
    if (i < n) data[i] = carry + wpre + inc - v;
    __syncthreads();
    carry += chunk_total;
  }
  return carry;
}

// Group table layout (int32, inside the workspace):
//   off[E+2]     first row of group g in the permuted row space; off[E] = TK
//                is the shared expert's first row (in H), off[E+1] = TK + T
//   ntt[E+1]     token tiles of group g (0 if the group is empty)
//   tsz[E+1]     rows per token tile (multiple of tile_round, <= bn)
//   toff_a[E+2]  prefix sum of ntt[g] * ft_a (tiles of the first GEMM)
//   toff_b[E+2]  prefix sum of ntt[g] * ft_b (tiles of the second GEMM)
//   toff_c[E+2]  prefix sum of ntt[g] * ft_c (backward: tiles of dH = dY W_d)
//   poff[E+2]    backward: first row of group g with every group padded to a
//                multiple of 16 rows (poff[E] = the shared group's first row,
//                poff[E+1] = all rows)
//   next[16]     tile counters of the GEMMs' schedulers: 0, 1 the forward's
//                (zeroed here), 2..7 the backward's (zeroed by its tables);
//                8..15 spare
#define MOE_GROUP_NEXT 16
#define MOE_GROUP_INTS(E) (7 * (E) + 12 + MOE_GROUP_NEXT)
struct GroupTable {
  int32_t *off, *ntt, *tsz, *toff_a, *toff_b, *toff_c, *poff, *next;
};

MOE_DEV GroupTable group_table(int32_t* base, int E) {
  GroupTable g;
  g.off = base;
  g.ntt = g.off + (E + 2);
  g.tsz = g.ntt + (E + 1);
  g.toff_a = g.tsz + (E + 1);
  g.toff_b = g.toff_a + (E + 2);
  g.toff_c = g.toff_b + (E + 2);
  g.poff = g.toff_c + (E + 2);
  g.next = g.poff + (E + 2);
  return g;
}

__global__ void __launch_bounds__(1024)
k_scan_groups(int32_t* __restrict__ blk_hist, int n_blocks, int E, int T, int TK,
              int32_t* __restrict__ load_counts, int32_t* __restrict__ groups, int bn, int ft_a,
              int ft_b, int tile_round) {
  __shared__ int buf[MOE_MAX_E + 2];
  __shared__ int load_s[MOE_MAX_E + 1];
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x;
  GroupTable G = group_table(groups, E);

  // per-expert totals; blk_hist becomes each block's exclusive prefix
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int b = 0; b < n_blocks; ++b) {
      const int c = blk_hist[(size_t)b * E + e];
      blk_hist[(size_t)b * E + e] = run;
      run += c;
    }
    load_s[e] = run;
    load_counts[e] = run;
    buf[e] = run;
  }
  __syncthreads();
  cta_exclusive_scan(buf, E, warp_tot);
  for (int e = tid; e < E; e += blockDim.x) G.off[e] = buf[e];
  if (tid == 0) {
    G.off[E] = TK;
    G.off[E + 1] = TK + T;
  }
  // absolute base row of every (block, expert)
  for (int e = tid; e < E; e += blockDim.x) {
    const int o = buf[e];
    for (int b = 0; b < n_blocks; ++b) blk_hist[(size_t)b * E + e] += o;
  }
  __syncthreads();
  if (bn <= 0) return;  // route-only: no GEMM tile table
  // token tiles per group (group E = shared expert with all T tokens)
  for (int g = tid; g <= E; g += blockDim.x) {
    const int n = g < E ? load_s[g] : T;
    const int nt = n > 0 ? (n + bn - 1) / bn : 0;
    const int per = nt > 0 ? (n + nt - 1) / nt : 0;
    G.ntt[g] = nt;
    G.tsz[g] = (per + tile_round - 1) / tile_round * tile_round;
    buf[g] = nt * ft_a;
  }
  __syncthreads();
  int tot = cta_exclusive_scan(buf, E + 1, warp_tot);
  for (int g = tid; g <= E; g += blockDim.x) G.toff_a[g] = buf[g];
  if (tid == 0) G.toff_a[E + 1] = tot;
  __syncthreads();
  for (int g = tid; g <= E; g += blockDim.x) buf[g] = G.ntt[g] * ft_b;
  __syncthreads();
  tot = cta_exclusive_scan(buf, E + 1, warp_tot);
  for (int g = tid; g <= E; g += blockDim.x) G.toff_b[g] = buf[g];
  if (tid == 0) {
    G.toff_b[E + 1] = tot;
    G.next[0] = 0;
    G.next[1] = 0;
  }
}

// One warp per pair; row_bytes a multiple of 16.
__global__ void __launch_bounds__(256)
k_permute_gather(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ pair_rank,
                 const int32_t* __restrict__ blk_base, int TK, int E, int k,
                 const uint8_t* __restrict__ x, uint8_t* __restrict__ x_perm, size_t row_bytes,
                 int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  const int lane = threadIdx.x & 31;
  const int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (p >= TK) return;
  const int e = topk_idx[p];
  const int b = p / MOE_PAIRS_PER_BLOCK;
  const int pos = blk_base[(size_t)b * E + e] + pair_rank[p];
  if (lane == 0) {
    perm[pos] = p;
    inv[p] = pos;
  }
  const int t = p / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * row_bytes);
  uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)pos * row_bytes);
  const int nv = (int)(row_bytes / 16);
  for (int i = lane; i < nv; i += 32) dst[i] = src[i];
}
