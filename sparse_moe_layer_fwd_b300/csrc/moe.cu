// moe.cu -- libmoe.so: the C ABI declared in include/moe.h.
//
// Host side of the DeepSeekMoE layer forward on one sm_103a GPU: argument
// validation, the workspace layout, TMA tensor maps, and the launch sequence
//   router logits -> router top-k -> block ranks -> scan + tile table ->
//   permute/gather -> expert GEMM 1 (gate/up + SwiGLU) -> expert GEMM 2
//   (down projection) -> combine (gates applied)
// all enqueued on the caller's stream with no host synchronisation (tile
// counts live in device memory; GEMM grids are sized by an upper bound and
// surplus CTAs return at once).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <math.h>

#include <mutex>

#include "../../include/moe.h"
#include "combine.cuh"
#include "dispatch.cuh"
#include "experts_simt.cuh"
#include "experts_tc.cuh"
#include "experts_tc2.cuh"
#include "ptx.cuh"
#include "router.cuh"
#include "router_tc.cuh"
#include "backward.cuh"
#include "quant.cuh"
#include "selftest.cuh"

namespace {

constexpr double kRouterCtaSlots = 296;  // router GEMM CTAs resident at once: 2 per SM
constexpr double kRouterPairs = 74;      // tensor-core router: one CTA pair per two SMs
                                         // on 148 SMs (fixed, so the split and hence
                                         // the results do not depend on the device)
constexpr int kRouterBK = 16;

// Tensor-core GEMM variants: BN tokens per tile, weight-ring and token-ring
// depths (each fills ~224 KB of shared memory).
constexpr int kSmallBN = 64, kSmallSA = 6, kSmallSB = 4;  // 1-SM kernel, small token tiles
constexpr int kBigBN = 256, kBigSA = 4, kBigSB = 3;        // 1-SM kernel, up to 256 tokens
// CTA-pair kernels, up to 256 tokens, two 256-column accumulators per tile
// (gate and up rows; two blocks of down-projection rows).  (One accumulator
// with two TMEM buffers, which overlaps the epilogue with the next tile's MMAs,
// measured slower for the second GEMM: it re-reads the token rows for every
// 256 output rows instead of every 512.)
// Ring depths and staged output boxes per epilogue warp (used round robin)
// of each pair GEMM: the bf16 outputs go out through shared memory by TMA
// store, and the staging boxes take the place of ring stages.
constexpr int kPairBN = 256;
#ifndef MOE_PAIR1_SA
#define MOE_PAIR1_SA 4
#endif
#ifndef MOE_PAIR1_SB
#define MOE_PAIR1_SB 4
#endif
#ifndef MOE_PAIR1_OUTB
#define MOE_PAIR1_OUTB 2
#endif
#ifndef MOE_PAIR2_SA
#define MOE_PAIR2_SA 4
#endif
#ifndef MOE_PAIR2_SB
#define MOE_PAIR2_SB 4
#endif
#ifndef MOE_PAIR2_OUTB
#define MOE_PAIR2_OUTB 2
#endif
// Kernel of each GEMM for the large token tiles: 1 = CTA pairs, 0 = one SM.
#ifndef MOE_PAIR_GEMM1
#define MOE_PAIR_GEMM1 1
#endif
#ifndef MOE_PAIR_GEMM2
#define MOE_PAIR_GEMM2 1
#endif

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Plan {
  int T, d, h, E, k, TK;
  bool f32, route_only, simt, big_router, big_tiles, tc_router;
  bool training;  // the backward's buffers follow the forward's
  bool fp8;       // gate/up products on per-row e4m3 codes (packed weights, tokens quantized here)
  bool fp8_blk;   // both products on block-scaled e4m3 codes (packed block weights)
  int el;  // bytes per activation / weight element
  // router: CUDA-core tiles (r_bm x r_bn) or tensor-core pairs over E_pad
  // experts (rt_eb blocks of 256) x rt_tt token tiles x n_split K slices
  int r_bm, r_bn, n_split, kchunk, E_pad, rt_eb, rt_tt;
  // dispatch
  int n_pair_blocks;
  // expert tiling
  int bn, ft_a, ft_b, ft_c, tile_round, max_tiles_a, max_tiles_b, max_tiles_c;
  // workspace regions (byte offsets)
  size_t o_part, o_w3, o_hist, o_rank, o_groups, o_perm, o_inv, o_xperm, o_h, o_yperm,
      o_xq, o_hq, total;
  // backward: padded dY rows, dG, du, dH, padded dA|dB rows, dX rows, shared dX;
  // the training forward's pre-activations A|B
  size_t o_dyp, o_dg, o_du, o_dh, o_dab, o_dxp, o_dxs, o_ab;
  long long rows_dyp, rows_dab;  // allocated padded rows
  size_t b_part, b_w3, b_hist, b_rank, b_groups, b_perm, b_inv, b_xperm, b_h, b_yperm,
      b_xq, b_hq;
};

int validate_desc(const moe_desc* d) {
  if (!d) return MOE_ERR_NULL;
  if (d->dtype != MOE_F32 && d->dtype != MOE_BF16) return MOE_ERR_DTYPE;
  if (d->flags & ~(MOE_ROUTE_ONLY | MOE_SIMT_EXPERTS | MOE_TRAINING | MOE_FP8_GATE_UP |
                   MOE_FP8_BLOCK | MOE_GRAD_BF16))
    return MOE_ERR_DTYPE;
  if ((d->flags & MOE_GRAD_BF16) && !(d->flags & MOE_TRAINING)) return MOE_ERR_DTYPE;
  if ((d->flags & (MOE_FP8_GATE_UP | MOE_FP8_BLOCK)) &&
      (d->dtype != MOE_BF16 || (d->flags & (MOE_SIMT_EXPERTS | MOE_ROUTE_ONLY | MOE_TRAINING))))
    return MOE_ERR_DTYPE;
  if ((d->flags & MOE_FP8_BLOCK) && (d->flags & MOE_FP8_GATE_UP)) return MOE_ERR_DTYPE;
  if ((d->flags & MOE_TRAINING) &&
      (d->dtype != MOE_BF16 || (d->flags & (MOE_SIMT_EXPERTS | MOE_ROUTE_ONLY))))
    return MOE_ERR_DTYPE;
  if ((d->flags & MOE_SIMT_EXPERTS) && d->dtype != MOE_BF16) return MOE_ERR_DTYPE;
  if (d->T < 0 || d->d <= 0 || d->h <= 0 || d->E < 1 || d->E > MOE_MAX_E || d->k < 1 ||
      d->k > d->E || d->k > 32)
    return MOE_ERR_SHAPE;
  if (d->d % 64 || d->h % 64) return MOE_ERR_SHAPE;
  const bool tc = d->dtype == MOE_BF16 && !(d->flags & MOE_SIMT_EXPERTS);
  if (tc && (d->d % 128 || d->h % 128)) return MOE_ERR_SHAPE;
  const long long TK = (long long)d->T * d->k;
  const long long wmax = d->d > d->h ? d->d : d->h;
  if ((TK + d->T) * wmax >= (1LL << 31)) return MOE_ERR_SHAPE;
  if ((long long)d->E * wmax >= (1LL << 31)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

Plan make_plan(const moe_desc* d) {
  Plan p;
  memset(&p, 0, sizeof(p));
  p.T = d->T; p.d = d->d; p.h = d->h; p.E = d->E; p.k = d->k; p.TK = d->T * d->k;
  p.f32 = d->dtype == MOE_F32;
  p.route_only = d->flags & MOE_ROUTE_ONLY;
  p.simt = p.f32 || (d->flags & MOE_SIMT_EXPERTS);
  p.el = p.f32 ? 4 : 2;
  p.fp8 = d->flags & MOE_FP8_GATE_UP;
  p.fp8_blk = d->flags & MOE_FP8_BLOCK;

  // router GEMM tiling and split of the model dimension
  p.big_router = p.E >= 96;
  p.r_bm = p.big_router ? 128 : 64;
  p.r_bn = p.big_router ? 128 : 64;
  // Split of the model dimension: the count whose CTAs fill whole waves best
  // (2 CTAs per SM on 148 SMs), with the partial logits kept under 24 MiB.
  const long long tiles = (long long)((p.T + p.r_bm - 1) / p.r_bm) * ((p.E + p.r_bn - 1) / p.r_bn);
  const int kblocks = p.d / kRouterBK;
  const long long te_bytes = (long long)p.T * p.E * 4;
  long long ns_max = te_bytes > 0 ? (24LL << 20) / te_bytes : 64;
  ns_max = ns_max < 1 ? 1 : (ns_max > 64 ? 64 : ns_max);
  ns_max = ns_max > kblocks ? kblocks : ns_max;
  int ns = 1;
  double best = -1.0;
  for (int c = 1; c <= ns_max && tiles > 0; ++c) {
    const double ctas = (double)tiles * c;
    const double waves = ceil(ctas / kRouterCtaSlots);
    const double eff = ctas / (waves * kRouterCtaSlots);
    if (eff > best + 1e-9) {
      best = eff;
      ns = c;
    }
  }
  p.kchunk = ((kblocks + ns - 1) / ns) * kRouterBK;
  p.n_split = (p.d + p.kchunk - 1) / p.kchunk;

  // bf16 tokens and a hundred experts or more: tensor-core router on CTA
  // pairs, split-K count chosen to fill whole waves of 74 pairs (partials
  // under 24 MiB, at least 4 K steps per slice)
  p.tc_router = !p.f32 && p.E >= 96 && p.T > 0;
  if (p.tc_router) {
    p.E_pad = (p.E + 255) / 256 * 256;
    p.rt_eb = p.E_pad / 256;
    p.rt_tt = (p.T + 255) / 256;
    const long long units1 = (long long)p.rt_eb * p.rt_tt;
    const int kb64 = p.d / 64;
    long long smax = te_bytes > 0 ? (24LL << 20) / te_bytes : 1;
    smax = smax < 1 ? 1 : smax;
    smax = smax > kb64 / 4 ? kb64 / 4 : smax;
    smax = smax < 1 ? 1 : smax;
    int sbest = 1;
    double eff_best = -1.0;
    for (int c = 1; c <= smax; ++c) {
      const double u = (double)units1 * c;
      const double eff = u / (ceil(u / kRouterPairs) * kRouterPairs);
      if (eff > eff_best + 1e-9) {
        eff_best = eff;
        sbest = c;
      }
    }
    p.kchunk = (kb64 + sbest - 1) / sbest * 64;
    p.n_split = (p.d + p.kchunk - 1) / p.kchunk;
  }

  p.n_pair_blocks = (p.TK + MOE_PAIRS_PER_BLOCK - 1) / MOE_PAIRS_PER_BLOCK;

  // expert tiling
  if (!p.route_only) {
    p.tile_round = 16;
    if (p.simt) {
      p.bn = SIMT_TM;
      p.ft_a = p.h / SIMT_TN;
      p.ft_b = p.d / SIMT_TN;
    } else {
      // about a hundred tokens per expert or more: CTA-pair tiles of up to
      // 256 tokens (N a multiple of 16) over 256 (first GEMM) or 512 (second)
      // weight rows; fewer: 1-SM tiles of up to 64 tokens over 128 / 256 rows
      const double per_expert = p.E > 0 ? (double)p.TK / p.E : 0.0;
      // (training: always the CTA-pair tiles, whose tile table the
      // backward's products share)
      // (fp8: the CTA-pair kernel alone has the e4m3 product)
      p.big_tiles =
          per_expert >= 96.0 || (d->flags & (MOE_TRAINING | MOE_FP8_GATE_UP | MOE_FP8_BLOCK));
      if (p.big_tiles) {
        // (block-scaled: TMEM also holds the scale sets, 240 tokens at most)
        p.bn = p.fp8_blk ? TC2_BLK_BN : kPairBN;
        p.ft_a = MOE_PAIR_GEMM1 ? (p.h + 2 * TC_BM - 1) / (2 * TC_BM) : p.h / TC_BM;
        p.ft_b = MOE_PAIR_GEMM2 ? (p.d + 4 * TC_BM - 1) / (4 * TC_BM) : (p.d / TC_BM + 1) / 2;
      } else {
        p.bn = kSmallBN;
        p.ft_a = p.h / TC_BM;
        p.ft_b = (p.d / TC_BM + 1) / 2;
      }
    }
    const long long tok_tiles = (long long)p.TK / p.bn + (p.TK < p.E ? p.TK : p.E) +
                                (p.T + p.bn - 1) / p.bn + 1;
    p.max_tiles_a = (int)(tok_tiles * p.ft_a);
    p.max_tiles_b = (int)(tok_tiles * p.ft_b);
    p.ft_c = (p.h + 4 * TC_BM - 1) / (4 * TC_BM);  // backward dH: 512 hidden rows per tile
    p.max_tiles_c = (int)(tok_tiles * p.ft_c);
  }

  // workspace
  size_t off = 0;
  auto region = [&](size_t bytes, size_t& o, size_t& b) {
    o = off;
    b = bytes;
    off = align_up(off + bytes, 256);
  };
  region((size_t)p.n_split * p.T * p.E * 4, p.o_part, p.b_part);
  region(p.tc_router ? (size_t)3 * p.E_pad * p.d * 2 : 0, p.o_w3, p.b_w3);
  region((size_t)p.n_pair_blocks * p.E * 4, p.o_hist, p.b_hist);
  region((size_t)p.TK * 4, p.o_rank, p.b_rank);
  region((size_t)MOE_GROUP_INTS(p.E) * 4, p.o_groups, p.b_groups);
  if (!p.route_only) {
    region((size_t)p.TK * 4, p.o_perm, p.b_perm);
    region((size_t)p.TK * 4, p.o_inv, p.b_inv);
    region((size_t)p.TK * p.d * ((p.fp8 || p.fp8_blk) ? 1 : p.el), p.o_xperm, p.b_xperm);
    region(p.fp8_blk ? 0 : (size_t)(p.TK + p.T) * p.h * p.el, p.o_h, p.b_h);
    // Y_perm: the routed rows in expert order, then the shared expert's rows
    // in token order (row TK + t)
    region((size_t)(p.TK + p.T) * p.d * p.el, p.o_yperm, p.b_yperm);
    // x_q: codes [T, d], then fp32 row scales [T] (per row) or exponent
    // words [ceil(d / 512)][T] (blocks); h_q: the block-quantized rows of H
    region(p.fp8 ? e4m3_scale_offset(p.T, p.d) + (size_t)p.T * 4
           : p.fp8_blk ? e4m3_scale_offset(p.T, p.d) + (size_t)e4m3_block_words(p.d) * p.T * 4
                       : 0,
           p.o_xq, p.b_xq);
    const long long rows_h = (long long)p.TK + p.T;
    region(p.fp8_blk ? e4m3_scale_offset(rows_h, p.h) + (size_t)e4m3_block_words(p.h) * rows_h * 4
                     : 0,
           p.o_hq, p.b_hq);
  }
  p.training = d->flags & MOE_TRAINING;
  if (p.training) {
    size_t b;
    // every group padded to 16 rows: at most 15 extra rows per group
    p.rows_dyp = (long long)p.TK + 15LL * p.E;
    p.rows_dab = (long long)p.TK + p.T + 15LL * (p.E + 1);
    region((size_t)p.rows_dyp * p.d * 2, p.o_dyp, b);
    region((size_t)p.TK * 4, p.o_dg, b);
    region((size_t)p.TK * 4, p.o_du, b);
    region((size_t)(p.TK + p.T) * p.h * 2, p.o_dh, b);
    region((size_t)p.rows_dab * 2 * p.h * 2, p.o_dab, b);
    region((size_t)p.TK * p.d * 2, p.o_dxp, b);
    region((size_t)p.T * p.d * 4, p.o_dxs, b);
    region((size_t)(p.TK + p.T) * 2 * p.h * 2, p.o_ab, b);
  }
  p.total = off > 0 ? off : 256;
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- TMA tensor maps ------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// bf16 matrix [rows, cols] (row-major) read in boxes of 64 columns (128
// bytes) x box_rows rows with the 128-byte swizzle; rows past the end read
// as zero.
// bf16 output rows [rows, cols] for TMA stores of 32 x 32 boxes with the
// 64-byte swizzle (the epilogue's staging layout).
bool make_out_map(CUtensorMap* m, const void* base, long long rows, long long cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output rows [rows, cols] for TMA stores of 32 x 32 boxes, 128-byte
// swizzle (the weight-gradient epilogue's staging layout).
bool make_out_map_f32(CUtensorMap* m, const void* base, long long rows, long long cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 codes [rows, cols] (one byte each) read in boxes of 128 columns (128
// bytes) x box_rows rows with the 128-byte swizzle; rows past the end read
// as zero.
bool make_map_u8(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

int device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_DEVICE;
  if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
  return MOE_OK;
}

template <typename TX>
void launch_router(const Plan& p, const TX* x, const float* w_router, float* part,
                   cudaStream_t s) {
  if (p.big_router) {
    dim3 grid((p.E + 127) / 128, (p.T + 127) / 128, p.n_split);
    k_router_logits<TX, 128, 128, kRouterBK, 8, 8>
        <<<grid, 256, 0, s>>>(x, w_router, part, p.T, p.E, p.d, p.kchunk);
  } else {
    dim3 grid((p.E + 63) / 64, (p.T + 63) / 64, p.n_split);
    k_router_logits<TX, 64, 64, kRouterBK, 4, 4>
        <<<grid, 256, 0, s>>>(x, w_router, part, p.T, p.E, p.d, p.kchunk);
  }
}

void launch_topk(const Plan& p, const float* part, const float* bias, int32_t* idx, float* gates,
                 cudaStream_t s) {
  const int grid = (p.T + 7) / 8;
  const int epl = (p.E + 31) / 32;
#define MOE_TOPK(N) \
  k_router_topk<N><<<grid, 256, 0, s>>>(part, p.n_split, bias, p.T, p.E, p.k, idx, gates)
  if (epl <= 1) MOE_TOPK(1);
  else if (epl <= 2) MOE_TOPK(2);
  else if (epl <= 4) MOE_TOPK(4);
  else if (epl <= 8) MOE_TOPK(8);
  else if (epl <= 16) MOE_TOPK(16);
  else MOE_TOPK(32);
#undef MOE_TOPK
}

struct TcMaps {
  TcMapsDev up;    // first GEMM: W_gate, W_up; token rows of X_perm and x
  TcMapsDev down;  // second GEMM: W_down; rows of H
};

// Token-row maps with 128-, 64-, 16- and (if m8) 8-row boxes: a tile of n
// rows is loaded as the fewest boxes that cover it exactly.
bool make_rows_maps(CUtensorMap* m128, CUtensorMap* m64, CUtensorMap* m16, CUtensorMap* m8,
                    const void* base, long long rows, long long cols) {
  return make_map(m128, base, rows, cols, 128) && make_map(m64, base, rows, cols, 64) &&
         make_map(m16, base, rows, cols, 16) && (!m8 || make_map(m8, base, rows, cols, 8));
}

// All tensor maps of the two tensor-core GEMMs, built before anything is
// launched so that a failure here leaves the stream untouched.
bool make_tc_maps(const Plan& p, const void* x, const moe_expert_w* ex, const moe_expert_w* sh,
                  uint8_t* ws, TcMaps* m) {
  bool ok = true;
  if (p.fp8 || p.fp8_blk) {
    // e4m3 codes: packed weights (codes first), X_perm codes, x codes
    const uint8_t* xq = ws + p.o_xq;
    ok &= make_map_u8(&m->up.a0, ex->w_gate, (long long)p.E * p.h, p.d, TC_BM);
    ok &= make_map_u8(&m->up.a1, ex->w_up, (long long)p.E * p.h, p.d, TC_BM);
    ok &= make_map_u8(&m->up.sa0, sh->w_gate, p.h, p.d, TC_BM);
    ok &= make_map_u8(&m->up.sa1, sh->w_up, p.h, p.d, TC_BM);
    for (int i = 0; i < 4; ++i) {
      static const int rows[4] = {128, 64, 16, 8};
      CUtensorMap* b[4] = {&m->up.b128, &m->up.b64, &m->up.b16, &m->up.b8};
      CUtensorMap* bs[4] = {&m->up.bs128, &m->up.bs64, &m->up.bs16, &m->up.bs8};
      ok &= make_map_u8(b[i], ws + p.o_xperm, p.TK, p.d, rows[i]);
      ok &= make_map_u8(bs[i], xq, p.T, p.d, rows[i]);
    }
  } else {
    ok &= make_map(&m->up.a0, ex->w_gate, (long long)p.E * p.h, p.d, TC_BM);
    ok &= make_map(&m->up.a1, ex->w_up, (long long)p.E * p.h, p.d, TC_BM);
    ok &= make_map(&m->up.sa0, sh->w_gate, p.h, p.d, TC_BM);
    ok &= make_map(&m->up.sa1, sh->w_up, p.h, p.d, TC_BM);
    ok &= make_rows_maps(&m->up.b128, &m->up.b64, &m->up.b16, &m->up.b8, ws + p.o_xperm, p.TK,
                         p.d);
    ok &= make_rows_maps(&m->up.bs128, &m->up.bs64, &m->up.bs16, &m->up.bs8, x, p.T, p.d);
  }
  if (p.fp8_blk) {
    // e4m3 codes: packed W_down (codes first), rows of H quantized
    ok &= make_map_u8(&m->down.a0, ex->w_down, (long long)p.E * p.d, p.h, TC_BM);
    ok &= make_map_u8(&m->down.sa0, sh->w_down, p.d, p.h, TC_BM);
    ok &= make_map_u8(&m->down.b128, ws + p.o_hq, (long long)p.TK + p.T, p.h, 128);
    ok &= make_map_u8(&m->down.b64, ws + p.o_hq, (long long)p.TK + p.T, p.h, 64);
    ok &= make_map_u8(&m->down.b16, ws + p.o_hq, (long long)p.TK + p.T, p.h, 16);
    ok &= make_map_u8(&m->down.b8, ws + p.o_hq, (long long)p.TK + p.T, p.h, 8);
  } else {
    ok &= make_map(&m->down.a0, ex->w_down, (long long)p.E * p.d, p.h, TC_BM);
    ok &= make_map(&m->down.sa0, sh->w_down, p.d, p.h, TC_BM);
    ok &= make_rows_maps(&m->down.b128, &m->down.b64, &m->down.b16, &m->down.b8, ws + p.o_h,
                         (long long)p.TK + p.T, p.h);
  }
  m->down.a1 = m->down.a0;
  m->down.sa1 = m->down.sa0;
  m->down.bs128 = m->down.b128;
  m->down.bs64 = m->down.b64;
  m->down.bs16 = m->down.b16;
  m->down.bs8 = m->down.b8;
  ok &= make_out_map(&m->up.out, ws + p.o_h, (long long)p.TK + p.T, p.h);
  if (p.training)  // the pre-activations A|B rows, stored by the training forward
    ok &= make_out_map(&m->up.aux, ws + p.o_ab, (long long)p.TK + p.T, 2LL * p.h);
  ok &= make_out_map(&m->down.out, ws + p.o_yperm, (long long)p.TK + p.T, p.d);
  return ok;
}

// The CTA-pair kernel of each operation: ring depths and staged boxes.  The
// backward's two-block products (dH, dX) take the second GEMM's
// configuration; the training forward's gate/up product stages three boxes
// per epilogue warp (H, A, B).
// (block-scaled: the first GEMM writes H codes from registers, no staged
// boxes; the second keeps one staged box per warp to leave room for the
// scale stages)
template <int OP> struct PairCfg {
  static constexpr bool UP = OP == TC2_FWD_UP || OP == TC2_FWD_UP_FP8 || OP == TC2_FWD_UP_B8;
  static constexpr bool B3 = OP == TC2_FWD_UP_T;  // three staged boxes per chunk (H, A, B)
  static constexpr int SA = B3 ? 4 : (UP ? MOE_PAIR1_SA : MOE_PAIR2_SA);
  static constexpr int SB = B3 ? 3 : (UP ? MOE_PAIR1_SB : MOE_PAIR2_SB);
  static constexpr int OUTB = B3                      ? 3
                              : OP == TC2_FWD_UP_B8   ? 0
                              : OP == TC2_FWD_DOWN_B8 ? 1
                              : (UP ? MOE_PAIR1_OUTB : MOE_PAIR2_OUTB);
  static constexpr int NACC = 2, NBUF = 1;
  using Cfg = Tc2Cfg<SA, SB, NACC, NBUF, OUTB, tc2_blk(OP)>;
};

template <int OP>
bool set_tc2_smem() {
  using P = PairCfg<OP>;
  return cudaFuncSetAttribute(k_expert_tc2<P::SA, P::SB, P::NACC, P::NBUF, P::OUTB, OP>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              P::Cfg::SMEM_BYTES) == cudaSuccess;
}

// One grouped product on CTA pairs, persistent: one pair per two SMs, at
// most one pair per tile.
template <int OP>
void launch_pair(const Plan& p, const TcMapsDev& m, int max_tiles, int32_t* groups, int K,
                 int n_out, __nv_bfloat16* out, float* ysh, const __nv_bfloat16* aux,
                 cudaStream_t s, const Fp8Scales& fs = Fp8Scales{}, const Fp8Blk& fb = Fp8Blk{},
                 __nv_bfloat16* out2 = nullptr) {
  const int pairs = sm_count() / 2;
  const int grid = 2 * (max_tiles < pairs ? max_tiles : pairs);
  using P = PairCfg<OP>;
  k_expert_tc2<P::SA, P::SB, P::NACC, P::NBUF, P::OUTB, OP>
      <<<grid, tc2_threads(OP), P::Cfg::SMEM_BYTES, s>>>(m, groups, p.E, K, n_out, out, ysh, aux,
                                                         fs, fb, out2);
}

template <int BN, int SA, int SB, bool DOWN>
bool set_tc1_smem() {
  return cudaFuncSetAttribute(k_expert_tc<BN, SA, SB, DOWN>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TcCfg<BN, SA, SB>::SMEM_BYTES) == cudaSuccess;
}

// One expert GEMM on CTA pairs (one pair per two SMs) or on single SMs (one
// CTA per SM), at most one CTA (pair) per tile.
template <bool DOWN>
void launch_gemm(const Plan& p, const TcMapsDev& m, bool pair, int BN, int max_tiles,
                 int32_t* groups, __nv_bfloat16* out, cudaStream_t s) {
  const int sms = sm_count();
  const int K = DOWN ? p.h : p.d, n_out = DOWN ? p.d : p.h;
  if (pair) {
    launch_pair<DOWN ? TC2_FWD_DOWN : TC2_FWD_UP>(p, m, max_tiles, groups, K, n_out, out,
                                                  nullptr, nullptr, s);
  } else if (BN == kBigBN) {
    const int grid = max_tiles < sms ? max_tiles : sms;
    k_expert_tc<kBigBN, kBigSA, kBigSB, DOWN><<<grid, TC_THREADS,
                                                  TcCfg<kBigBN, kBigSA, kBigSB>::SMEM_BYTES, s>>>(
        m, groups, p.E, K, n_out, out);
  } else {
    const int grid = max_tiles < sms ? max_tiles : sms;
    k_expert_tc<kSmallBN, kSmallSA, kSmallSB, DOWN>
        <<<grid, TC_THREADS, TcCfg<kSmallBN, kSmallSA, kSmallSB>::SMEM_BYTES, s>>>(
            m, groups, p.E, K, n_out, out);
  }
}

template <typename T>
void launch_simt(const Plan& p, const void* x, const moe_expert_w* ex, const moe_expert_w* sh,
                 uint8_t* ws, int32_t* groups, cudaStream_t s, cudaEvent_t between) {
  const T* xp = reinterpret_cast<const T*>(ws + p.o_xperm);
  T* hbuf = reinterpret_cast<T*>(ws + p.o_h);
  T* yperm = reinterpret_cast<T*>(ws + p.o_yperm);
  k_expert_simt<T, false><<<p.max_tiles_a, 256, 0, s>>>(
      (const T*)ex->w_gate, (const T*)ex->w_up, (const T*)sh->w_gate, (const T*)sh->w_up, xp,
      (const T*)x, groups, p.E, p.d, p.h, hbuf);
  if (between) cudaEventRecord(between, s);
  k_expert_simt<T, true><<<p.max_tiles_b, 256, 0, s>>>(
      (const T*)ex->w_down, nullptr, (const T*)sh->w_down, nullptr, hbuf, hbuf, groups, p.E, p.h,
      p.d, yperm);
}

int forward_impl(const moe_desc* desc, const void* x, const float* w_router, const float* bias,
                 const moe_expert_w* experts, const moe_expert_w* shared, void* y,
                 int32_t* topk_idx, float* gates, int32_t* load_counts, void* workspace,
                 size_t ws_bytes, cudaStream_t s, void* const* events = nullptr) {
  auto mark = [&](int i) {
    if (events) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
  };
  int rc = validate_desc(desc);
  if (rc != MOE_OK) return rc;
  const Plan p = make_plan(desc);
  const bool need_out = !p.route_only && p.T > 0;
  if (!w_router || !bias || !load_counts || !workspace) return MOE_ERR_NULL;
  if (p.T > 0 && (!x || !topk_idx || !gates)) return MOE_ERR_NULL;
  if (need_out) {
    if (!y || !experts || !shared) return MOE_ERR_NULL;
    if (!experts->w_gate || !experts->w_up || !experts->w_down || !shared->w_gate ||
        !shared->w_up || !shared->w_down)
      return MOE_ERR_NULL;
    if (!aligned16(y) || !aligned16(experts->w_gate) || !aligned16(experts->w_up) ||
        !aligned16(experts->w_down) || !aligned16(shared->w_gate) || !aligned16(shared->w_up) ||
        !aligned16(shared->w_down))
      return MOE_ERR_ALIGN;
  }
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace)) return MOE_ERR_ALIGN;
  if (ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  rc = device_ok();
  if (rc != MOE_OK) return rc;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  RouterMapsDev rmaps;
  if (p.tc_router) {
    if (!make_map(&rmaps.w, ws + p.o_w3, 3LL * p.E_pad, p.d, 128) ||
        !make_rows_maps(&rmaps.x128, &rmaps.x64, &rmaps.x16, nullptr, x, p.T, p.d))
      return MOE_ERR_DEVICE;
    if (cudaFuncSetAttribute(k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             RT_SMEM_BYTES) != cudaSuccess)
      return MOE_ERR_LAUNCH;
  }
  const bool use_tc = need_out && !p.simt;
  TcMaps maps;
  if (use_tc) {
    if (!make_tc_maps(p, x, experts, shared, ws, &maps)) return MOE_ERR_DEVICE;
    const bool ok =
        p.fp8_blk ? (set_tc2_smem<TC2_FWD_UP_B8>() && set_tc2_smem<TC2_FWD_DOWN_B8>()) :
        p.big_tiles
            ? ((p.fp8        ? set_tc2_smem<TC2_FWD_UP_FP8>()
                : p.training ? set_tc2_smem<TC2_FWD_UP_T>()
                      : MOE_PAIR_GEMM1 ? set_tc2_smem<TC2_FWD_UP>()
                               : set_tc1_smem<kBigBN, kBigSA, kBigSB, false>()) &&
               (MOE_PAIR_GEMM2 ? set_tc2_smem<TC2_FWD_DOWN>()
                               : set_tc1_smem<kBigBN, kBigSA, kBigSB, true>()))
            : (set_tc1_smem<kSmallBN, kSmallSA, kSmallSB, false>() &&
               set_tc1_smem<kSmallBN, kSmallSA, kSmallSB, true>());
    if (!ok) return MOE_ERR_LAUNCH;
  }
  float* part = reinterpret_cast<float*>(ws + p.o_part);
  int32_t* hist = reinterpret_cast<int32_t*>(ws + p.o_hist);
  int32_t* rank = reinterpret_cast<int32_t*>(ws + p.o_rank);
  int32_t* groups = reinterpret_cast<int32_t*>(ws + p.o_groups);

  cudaGetLastError();  // clear a stale error so the check below is ours
  mark(0);
  if (p.T > 0) {
    if (p.f32)
      launch_router<float>(p, static_cast<const float*>(x), w_router, part, s);
    else
      if (p.tc_router) {
        k_router_split<<<2 * sm_count(), 256, 0, s>>>(
            w_router, reinterpret_cast<__nv_bfloat16*>(ws + p.o_w3), p.E, p.E_pad, p.d);
        k_router_tc<<<2 * p.rt_eb * p.rt_tt * p.n_split, RT_THREADS, RT_SMEM_BYTES, s>>>(
            rmaps, p.T, p.E, p.E_pad, p.d, p.kchunk, p.rt_tt, p.rt_eb, part);
      } else {
        launch_router<__nv_bfloat16>(p, static_cast<const __nv_bfloat16*>(x), w_router, part, s);
      }
    launch_topk(p, part, bias, topk_idx, gates, s);
  }
  mark(1);
  if (p.T > 0) {
    k_block_rank<<<p.n_pair_blocks, 32, 0, s>>>(topk_idx, p.TK, p.E, rank, hist);
  }
  k_scan_groups<<<1, 1024, 0, s>>>(hist, p.n_pair_blocks, p.E, p.T, p.TK, load_counts, groups,
                                   need_out ? p.bn : 0, p.ft_a, p.ft_b, p.tile_round);
  if (need_out) {
    int32_t* perm = reinterpret_cast<int32_t*>(ws + p.o_perm);
    int32_t* inv = reinterpret_cast<int32_t*>(ws + p.o_inv);
    uint8_t* xq = ws + p.o_xq;
    float* xs = reinterpret_cast<float*>(xq + e4m3_scale_offset(p.T, p.d));
    uint32_t* xw = reinterpret_cast<uint32_t*>(xs);  // block-scaled: exponent words
    if (p.fp8)  // the tokens' codes and scales; the gather moves codes
      k_quant_rows<__nv_bfloat16><<<(p.T + 7) / 8, 256, 0, s>>>(
          static_cast<const __nv_bfloat16*>(x), p.T, p.d, xq, xs);
    if (p.fp8_blk)
      k_quant_ablocks<<<(p.T + 7) / 8, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), p.T,
                                                     p.d, xq, xw);
    const bool codes = p.fp8 || p.fp8_blk;
    k_permute_gather<<<(p.TK + 7) / 8, 256, 0, s>>>(
        topk_idx, rank, hist, p.TK, p.E, p.k, codes ? xq : static_cast<const uint8_t*>(x),
        ws + p.o_xperm, (size_t)p.d * (codes ? 1 : p.el), perm, inv);
    mark(2);
    cudaEvent_t between = events ? static_cast<cudaEvent_t>(events[3]) : nullptr;
    if (p.f32) {
      launch_simt<float>(p, x, experts, shared, ws, groups, s, between);
    } else if (p.simt) {
      launch_simt<__nv_bfloat16>(p, x, experts, shared, ws, groups, s, between);
    } else {
      __nv_bfloat16* hbuf = reinterpret_cast<__nv_bfloat16*>(ws + p.o_h);
      __nv_bfloat16* yperm = reinterpret_cast<__nv_bfloat16*>(ws + p.o_yperm);
      if (p.fp8_blk) {
        // both products on block-scaled codes: GEMM 1 writes H as codes and
        // exponent words, GEMM 2 reads them (K counted in 64-element bf16
        // steps of 128 bytes: d codes = d / 2)
        const long long rows_h = (long long)p.TK + p.T;
        uint8_t* hq = ws + p.o_hq;
        uint32_t* hw = reinterpret_cast<uint32_t*>(hq + e4m3_scale_offset(rows_h, p.h));
        auto words = [](const void* w, long long rows, long long cols) {
          return reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(w) +
                                                   e4m3_scale_offset(rows, cols));
        };
        const Fp8Blk f1{words(experts->w_gate, (long long)p.E * p.h, p.d),
                        words(experts->w_up, (long long)p.E * p.h, p.d),
                        words(shared->w_gate, p.h, p.d), words(shared->w_up, p.h, p.d),
                        e4m3_block_words(p.d), xw, p.T, perm, p.k, hq, hw, (int)rows_h};
        launch_pair<TC2_FWD_UP_B8>(p, maps.up, p.max_tiles_a, groups, p.d / 2, p.h, nullptr,
                                   nullptr, nullptr, s, Fp8Scales{}, f1);
        if (between) cudaEventRecord(between, s);
        const uint32_t* wd = words(experts->w_down, (long long)p.E * p.d, p.h);
        const uint32_t* swd = words(shared->w_down, p.d, p.h);
        const Fp8Blk f2{wd, wd, swd, swd, e4m3_block_words(p.h), hw, (int)rows_h, nullptr, p.k,
                        nullptr, nullptr, 0};
        launch_pair<TC2_FWD_DOWN_B8>(p, maps.down, p.max_tiles_b, groups, p.h / 2, p.d, yperm,
                                     nullptr, nullptr, s, Fp8Scales{}, f2);
      } else {
      if (p.fp8) {
        const size_t so = e4m3_scale_offset((long long)p.E * p.h, p.d),
                     ss = e4m3_scale_offset(p.h, p.d);
        auto scl = [](const void* w, size_t o) {
          return reinterpret_cast<const float*>(static_cast<const uint8_t*>(w) + o);
        };
        const Fp8Scales fs{scl(experts->w_gate, so), scl(experts->w_up, so),
                           scl(shared->w_gate, ss), scl(shared->w_up, ss), xs, perm, p.k};
        // K in bf16 units of 128 bytes per step: d codes = d / 2 "elements"
        launch_pair<TC2_FWD_UP_FP8>(p, maps.up, p.max_tiles_a, groups, p.d / 2, p.h, hbuf,
                                    nullptr, nullptr, s, fs);
      } else if (p.training) {
        // the pre-activations A|B as well, for the backward's SwiGLU gradient
        launch_pair<TC2_FWD_UP_T>(p, maps.up, p.max_tiles_a, groups, p.d, p.h, hbuf, nullptr,
                                  nullptr, s, Fp8Scales{}, Fp8Blk{},
                                  reinterpret_cast<__nv_bfloat16*>(ws + p.o_ab));
      } else {
        launch_gemm<false>(p, maps.up, p.big_tiles && MOE_PAIR_GEMM1, p.bn, p.max_tiles_a,
                           groups, hbuf, s);
      }
      if (between) cudaEventRecord(between, s);
      launch_gemm<true>(p, maps.down, p.big_tiles && MOE_PAIR_GEMM2, p.bn, p.max_tiles_b, groups,
                        yperm, s);
      }
    }
    mark(4);
    if (p.f32)
      k_combine<float><<<p.T, 128, 0, s>>>(reinterpret_cast<const float*>(ws + p.o_yperm), inv,
                                           gates, p.T, p.d, p.k, static_cast<float*>(y));
    else
      k_combine<__nv_bfloat16><<<p.T, 128, 0, s>>>(
          reinterpret_cast<const __nv_bfloat16*>(ws + p.o_yperm), inv, gates, p.T, p.d, p.k,
          static_cast<__nv_bfloat16*>(y));
  } else {
    mark(2);
    mark(3);
    mark(4);
  }
  mark(5);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // namespace

extern "C" {

size_t moe_workspace_size(const moe_desc* desc) {
  if (validate_desc(desc) != MOE_OK) return 0;
  return make_plan(desc).total;
}

int moe_forward(const moe_desc* desc, const void* x, const float* w_router, const float* bias,
                const moe_expert_w* experts, const moe_expert_w* shared, void* y,
                int32_t* topk_idx, float* gates, int32_t* load_counts, void* workspace,
                size_t ws_bytes, void* stream) {
  return forward_impl(desc, x, w_router, bias, experts, shared, y, topk_idx, gates, load_counts,
                      workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

int moe_forward_profiled(const moe_desc* desc, const void* x, const float* w_router,
                         const float* bias, const moe_expert_w* experts,
                         const moe_expert_w* shared, void* y, int32_t* topk_idx, float* gates,
                         int32_t* load_counts, void* workspace, size_t ws_bytes, void* stream,
                         void* const* events) {
  if (!events) return MOE_ERR_NULL;
  for (int i = 0; i < MOE_N_PHASE_EVENTS; ++i)
    if (!events[i]) return MOE_ERR_NULL;
  return forward_impl(desc, x, w_router, bias, experts, shared, y, topk_idx, gates, load_counts,
                      workspace, ws_bytes, static_cast<cudaStream_t>(stream), events);
}

size_t moe_host_io_extra_bytes(const moe_desc* desc) {
  if (validate_desc(desc) != MOE_OK) return 0;
  const size_t el = desc->dtype == MOE_F32 ? 4 : 2;
  return 2 * align_up((size_t)desc->T * desc->d * el, 256);
}

int moe_forward_host_io(const moe_desc* desc, const void* x_host, const float* w_router,
                        const float* bias, const moe_expert_w* experts,
                        const moe_expert_w* shared, void* y_host, int32_t* topk_idx,
                        float* gates, int32_t* load_counts, void* workspace, size_t ws_bytes,
                        void* stream) {
  int rc = validate_desc(desc);
  if (rc != MOE_OK) return rc;
  if (!workspace) return MOE_ERR_NULL;
  const size_t base = make_plan(desc).total;
  const size_t el = desc->dtype == MOE_F32 ? 4 : 2;
  const size_t xbytes = (size_t)desc->T * desc->d * el;
  if (ws_bytes < base + moe_host_io_extra_bytes(desc)) return MOE_ERR_WORKSPACE;
  if (desc->T > 0 && !x_host) return MOE_ERR_NULL;
  const bool need_y = !(desc->flags & MOE_ROUTE_ONLY) && desc->T > 0;
  if (need_y && !y_host) return MOE_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* xdev = static_cast<uint8_t*>(workspace) + base;
  uint8_t* ydev = xdev + align_up(xbytes, 256);
  if (xbytes && cudaMemcpyAsync(xdev, x_host, xbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_DEVICE;
  rc = forward_impl(desc, xdev, w_router, bias, experts, shared, need_y ? ydev : nullptr,
                    topk_idx, gates, load_counts, workspace, base, s);
  if (rc != MOE_OK) return rc;
  if (need_y && cudaMemcpyAsync(y_host, ydev, xbytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_DEVICE;
  return MOE_OK;
}

int moe_selftest_timeout(unsigned limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 10000) return MOE_ERR_SHAPE;
  int rc = device_ok();
  if (rc != MOE_OK) return rc;
  cudaGetLastError();
  k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_ms * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int moe_selftest_silu(const float* z, float* out, int n, void* stream) {
  if (n < 0) return MOE_ERR_SHAPE;
  if (n == 0) return MOE_OK;
  if (!z || !out) return MOE_ERR_NULL;
  int rc = device_ok();
  if (rc != MOE_OK) return rc;
  cudaGetLastError();
  k_selftest_silu<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(z, out, n);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

size_t moe_e4m3_packed_bytes(long long rows, int cols) {
  if (rows < 0 || cols <= 0) return 0;
  return e4m3_scale_offset(rows, cols) + (size_t)rows * 4;
}

int moe_quantize_rows_e4m3(const void* a, long long rows, int cols, void* packed, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 8 || rows > (1LL << 40) / cols) return MOE_ERR_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!a || !packed) return MOE_ERR_NULL;
  if (!aligned16(a) || !aligned16(packed)) return MOE_ERR_ALIGN;
  int rc = device_ok();
  if (rc != MOE_OK) return rc;
  cudaGetLastError();
  uint8_t* q = static_cast<uint8_t*>(packed);
  k_quant_rows<__nv_bfloat16><<<(unsigned)((rows + 7) / 8), 256, 0,
                                static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(a), rows, cols, q,
      reinterpret_cast<float*>(q + e4m3_scale_offset(rows, cols)));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

size_t moe_e4m3_block_packed_bytes(long long rows, int cols) {
  if (rows < 0 || cols <= 0 || rows % 128 || cols % 128) return 0;
  return e4m3_block_packed_bytes(rows, cols);
}

int moe_quantize_blocks_e4m3(const void* a, long long rows, int cols, void* packed,
                             void* stream) {
  if (rows < 0 || cols <= 0 || rows % 128 || cols % 128 || rows > (1LL << 40) / cols ||
      rows / 128 > 65535)
    return MOE_ERR_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!a || !packed) return MOE_ERR_NULL;
  if (!aligned16(a) || !aligned16(packed)) return MOE_ERR_ALIGN;
  int rc = device_ok();
  if (rc != MOE_OK) return rc;
  cudaGetLastError();
  uint8_t* q = static_cast<uint8_t*>(packed);
  const dim3 grid((unsigned)(cols / 128), (unsigned)(rows / 128));
  k_quant_wblocks<<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(a), cols, q,
      reinterpret_cast<uint32_t*>(q + e4m3_scale_offset(rows, cols)));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int moe_bias_update(const int32_t* load_counts, float* bias, float gamma, int E, int TK,
                    void* stream) {
  if (!load_counts || !bias) return MOE_ERR_NULL;
  if (E < 1 || E > MOE_MAX_E || TK < 0) return MOE_ERR_SHAPE;
  int rc = device_ok();
  if (rc != MOE_OK) return rc;
  cudaGetLastError();
  k_bias_update<<<(E + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(load_counts, bias,
                                                                                 gamma, E, TK);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

// ---- backward ---------------------------------------------------------------
// Tensor maps of the backward's products, built before anything is launched.
struct BwdMaps {
  TcMaps fwd;        // the forward's (gate/up recomputation reuses fwd.up)
  TcMapsDev dh, dx;  // dH = dY W_down, dX = dA W_gate + dB W_up (weights transposed)
  WgMapsDev wd, wg, wu; // weight gradients: dW_down, dW_gate, dW_up
};

bool make_bwd_maps(const Plan& p, const void* x, const moe_expert_w* ex, const moe_expert_w* sh,
                   const void* dy, uint8_t* ws, const moe_expert_grad* dex,
                   const moe_expert_grad* dsh, bool grad_bf16, BwdMaps* m) {
  // weight-gradient outputs: fp32, or bf16 with MOE_GRAD_BF16
  auto out_map = [&](CUtensorMap* mm, const void* base, long long rows, long long cols) {
    return grad_bf16 ? make_out_map(mm, base, rows, cols) : make_out_map_f32(mm, base, rows, cols);
  };
  bool ok = make_tc_maps(p, x, ex, sh, ws, &m->fwd);
  const long long rows_h = (long long)p.TK + p.T;
  // dH: W_down [E*d rows, h cols] read as d-row x h-column boxes (MN-major)
  ok &= make_map(&m->dh.a0, ex->w_down, (long long)p.E * p.d, p.h, 64);
  ok &= make_map(&m->dh.sa0, sh->w_down, p.d, p.h, 64);
  m->dh.a1 = m->dh.a0;
  m->dh.sa1 = m->dh.sa0;
  ok &= make_rows_maps(&m->dh.b128, &m->dh.b64, &m->dh.b16, &m->dh.b8, ws + p.o_dyp, p.rows_dyp,
                       p.d);
  ok &= make_rows_maps(&m->dh.bs128, &m->dh.bs64, &m->dh.bs16, &m->dh.bs8, dy, p.T, p.d);
  ok &= make_out_map(&m->dh.out, ws + p.o_dh, rows_h, p.h);
  // dX: W_gate, W_up [E*h rows, d cols] (MN-major), dA|dB rows [rows, 2h]
  ok &= make_map(&m->dx.a0, ex->w_gate, (long long)p.E * p.h, p.d, 64);
  ok &= make_map(&m->dx.a1, ex->w_up, (long long)p.E * p.h, p.d, 64);
  ok &= make_map(&m->dx.sa0, sh->w_gate, p.h, p.d, 64);
  ok &= make_map(&m->dx.sa1, sh->w_up, p.h, p.d, 64);
  ok &= make_rows_maps(&m->dx.b128, &m->dx.b64, &m->dx.b16, &m->dx.b8, ws + p.o_dab, p.rows_dab,
                       2LL * p.h);
  m->dx.bs128 = m->dx.b128;
  m->dx.bs64 = m->dx.b64;
  m->dx.bs16 = m->dx.b16;
  m->dx.bs8 = m->dx.b8;
  ok &= make_out_map(&m->dx.out, ws + p.o_dxp, p.TK, p.d);
  // weight gradients: both operands MN-major, 64-column x 64-row boxes
  ok &= make_map(&m->wd.p, ws + p.o_dyp, p.rows_dyp, p.d, 64);
  ok &= make_map(&m->wd.ps, dy, p.T, p.d, 64);
  ok &= make_map(&m->wd.q, ws + p.o_h, rows_h, p.h, 64);
  m->wd.qs = m->wd.q;
  ok &= out_map(&m->wd.o, dex->d_down, (long long)p.E * p.d, p.h);
  ok &= out_map(&m->wd.os, dsh->d_down, p.d, p.h);
  ok &= make_map(&m->wg.p, ws + p.o_dab, p.rows_dab, 2LL * p.h, 64);
  m->wg.ps = m->wg.p;
  ok &= make_map(&m->wg.q, ws + p.o_xperm, p.TK, p.d, 64);
  ok &= make_map(&m->wg.qs, x, p.T, p.d, 64);
  m->wu = m->wg;
  ok &= out_map(&m->wg.o, dex->d_gate, (long long)p.E * p.h, p.d);
  ok &= out_map(&m->wg.os, dsh->d_gate, p.h, p.d);
  ok &= out_map(&m->wu.o, dex->d_up, (long long)p.E * p.h, p.d);
  ok &= out_map(&m->wu.os, dsh->d_up, p.h, p.d);
  return ok;
}

int moe_backward(const moe_desc* desc, const void* x, const float* w_router,
                 const moe_expert_w* experts, const moe_expert_w* shared,
                 const int32_t* topk_idx, const float* gates, const void* dy, void* dx,
                 const moe_expert_grad* d_experts, const moe_expert_grad* d_shared,
                 float* d_router, void* workspace, size_t ws_bytes, void* stream) {
  int rc = validate_desc(desc);
  if (rc != MOE_OK) return rc;
  if (!(desc->flags & MOE_TRAINING)) return MOE_ERR_DTYPE;
  const Plan p = make_plan(desc);
  if (!w_router || !experts || !shared || !d_experts || !d_shared || !d_router || !workspace)
    return MOE_ERR_NULL;
  if (!experts->w_gate || !experts->w_up || !experts->w_down || !shared->w_gate ||
      !shared->w_up || !shared->w_down || !d_experts->d_gate || !d_experts->d_up ||
      !d_experts->d_down || !d_shared->d_gate || !d_shared->d_up || !d_shared->d_down)
    return MOE_ERR_NULL;
  if (p.T > 0 && (!x || !topk_idx || !gates || !dy || !dx)) return MOE_ERR_NULL;
  const void* ptrs[] = {x, w_router, experts->w_gate, experts->w_up, experts->w_down,
                        shared->w_gate, shared->w_up, shared->w_down, dy, dx,
                        d_experts->d_gate, d_experts->d_up, d_experts->d_down, d_shared->d_gate,
                        d_shared->d_up, d_shared->d_down, d_router, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_ALIGN;
  if (ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  rc = device_ok();
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool gb = desc->flags & MOE_GRAD_BF16;
  const size_t gel = gb ? 2 : 4;  // bytes per weight-gradient element
  const size_t e_hd = (size_t)p.E * p.h * p.d * gel, hd = (size_t)p.h * p.d * gel;
  cudaGetLastError();
  if (p.T == 0) {  // no tokens: every gradient is zero
    const bool ok = cudaMemsetAsync(d_experts->d_gate, 0, e_hd, s) == cudaSuccess &&
                    cudaMemsetAsync(d_experts->d_up, 0, e_hd, s) == cudaSuccess &&
                    cudaMemsetAsync(d_experts->d_down, 0, e_hd, s) == cudaSuccess &&
                    cudaMemsetAsync(d_shared->d_gate, 0, hd, s) == cudaSuccess &&
                    cudaMemsetAsync(d_shared->d_up, 0, hd, s) == cudaSuccess &&
                    cudaMemsetAsync(d_shared->d_down, 0, hd, s) == cudaSuccess &&
                    cudaMemsetAsync(d_router, 0, (size_t)p.E * p.d * 4, s) == cudaSuccess;
    return ok ? MOE_OK : MOE_ERR_LAUNCH;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BwdMaps maps;
  if (!make_bwd_maps(p, x, experts, shared, dy, ws, d_experts, d_shared, gb, &maps))
    return MOE_ERR_DEVICE;
  if (!set_tc2_smem<TC2_BWD_DH>() || !set_tc2_smem<TC2_BWD_DX>() ||
      cudaFuncSetAttribute(k_wgrad_tc2<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           WG_SMEM_BYTES) != cudaSuccess ||
      cudaFuncSetAttribute(k_wgrad_tc2<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           WG_SMEM_BYTES) != cudaSuccess)
    return MOE_ERR_LAUNCH;

  int32_t* groups = reinterpret_cast<int32_t*>(ws + p.o_groups);
  const int32_t* perm = reinterpret_cast<const int32_t*>(ws + p.o_perm);
  const int32_t* inv = reinterpret_cast<const int32_t*>(ws + p.o_inv);
  const float* part = reinterpret_cast<const float*>(ws + p.o_part);
  __nv_bfloat16* dyp = reinterpret_cast<__nv_bfloat16*>(ws + p.o_dyp);
  float* dg = reinterpret_cast<float*>(ws + p.o_dg);
  float* du = reinterpret_cast<float*>(ws + p.o_du);
  __nv_bfloat16* dh = reinterpret_cast<__nv_bfloat16*>(ws + p.o_dh);
  __nv_bfloat16* dab = reinterpret_cast<__nv_bfloat16*>(ws + p.o_dab);
  __nv_bfloat16* dxp = reinterpret_cast<__nv_bfloat16*>(ws + p.o_dxp);
  float* dxs = reinterpret_cast<float*>(ws + p.o_dxs);
  const __nv_bfloat16* dyb = static_cast<const __nv_bfloat16*>(dy);

  k_bwd_tables<<<1, 1024, 0, s>>>(groups, p.E, p.ft_c);
  k_bwd_prep<<<(p.TK + 7) / 8, 256, 0, s>>>(
      groups, p.E, perm, topk_idx, gates, p.TK, p.k, p.d, dyb,
      reinterpret_cast<const __nv_bfloat16*>(ws + p.o_yperm), dyp, dg);
  k_bwd_zero_gaps<<<p.E + 1, 256, 0, s>>>(groups, p.E, dyp, p.d, dab, 2 * p.h);
  k_bwd_router<<<(p.T + 7) / 8, 256, 0, s>>>(part, p.n_split, topk_idx, inv, dg, p.T, p.E, p.k,
                                               du);
  launch_pair<TC2_BWD_DH>(p, maps.dh, p.max_tiles_c, groups, p.d, p.h, dh, nullptr, nullptr, s);
  // SwiGLU gradient from the pre-activations the forward stored
  k_bwd_swiglu<<<(unsigned)((p.TK + p.T + 7) / 8), 256, 0, s>>>(
      groups, p.E, p.TK + p.T, p.h, reinterpret_cast<const __nv_bfloat16*>(ws + p.o_ab), dh, dab);
  launch_pair<TC2_BWD_DX>(p, maps.dx, p.max_tiles_b, groups, 2 * p.h, p.d, dxp, dxs, nullptr, s);
  const int pairs = sm_count() / 2;
  auto wgrad = [&](const WgMapsDev& m, int M, int N, int pcol0, int slot, int p_from_ps,
                   int q_from_qs) {
    const long long tiles = (long long)(p.E + 1) * ((M + 255) / 256) * ((N + 255) / 256);
    const int grid = 2 * (int)(tiles < pairs ? tiles : pairs);
    if (gb)
      k_wgrad_tc2<true><<<grid, WG_THREADS, WG_SMEM_BYTES, s>>>(m, groups, p.E, M, N, pcol0, 0,
                                                                slot, p_from_ps, q_from_qs);
    else
      k_wgrad_tc2<false><<<grid, WG_THREADS, WG_SMEM_BYTES, s>>>(m, groups, p.E, M, N, pcol0, 0,
                                                                 slot, p_from_ps, q_from_qs);
  };
  wgrad(maps.wd, p.d, p.h, 0, 5, 1, 0);
  wgrad(maps.wg, p.h, p.d, 0, 6, 0, 1);
  wgrad(maps.wu, p.h, p.d, p.h, 7, 0, 1);
  k_bwd_router_wgrad<__nv_bfloat16><<<dim3(p.E, (p.d + 1023) / 1024), 128, 0, s>>>(
      groups, p.E, perm, du, static_cast<const __nv_bfloat16*>(x), p.d, p.k, d_router);
  k_bwd_combine<__nv_bfloat16><<<p.T, 128, 0, s>>>(dxs, dxp, inv, topk_idx, du, w_router, p.T,
                                                    p.d, p.k, static_cast<__nv_bfloat16*>(dx));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int moe_seq_balance_loss(const moe_desc* desc, int seq_len, float alpha, const int32_t* topk_idx,
                         const void* workspace, size_t ws_bytes, float* loss, void* stream) {
  int rc = validate_desc(desc);
  if (rc != MOE_OK) return rc;
  if (seq_len < 1) return MOE_ERR_SHAPE;
  const Plan p = make_plan(desc);
  if (p.T == 0) return MOE_OK;
  if (!topk_idx || !workspace || !loss) return MOE_ERR_NULL;
  if (ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MOE_ERR_ALIGN;
  rc = device_ok();
  if (rc != MOE_OK) return rc;
  const float* part =
      reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + p.o_part);
  const int nseq = (p.T + seq_len - 1) / seq_len;
  const size_t smem = (size_t)9 * p.E * 4;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  const int epl = (p.E + 31) / 32;
#define MOE_BAL(N)                                                                          \
  k_seq_balance_loss<N><<<nseq, 256, smem, s>>>(part, p.n_split, topk_idx, p.T, p.E, p.k, \
                                                seq_len, alpha, loss)
  if (epl <= 1) MOE_BAL(1);
  else if (epl <= 2) MOE_BAL(2);
  else if (epl <= 4) MOE_BAL(4);
  else if (epl <= 8) MOE_BAL(8);
  else if (epl <= 16) MOE_BAL(16);
  else MOE_BAL(32);
#undef MOE_BAL
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

static_assert(MOE_CLOCK_SLOTS == MOE_CLOCK_NSLOT, "clock slots");

int moe_sm_clock_record(unsigned long long* out, int reset) {
  if (!out) return MOE_ERR_NULL;
  unsigned long long v[MOE_CLOCK_NSLOT][2];
  if (cudaMemcpyFromSymbol(v, g_moe_clock, sizeof(v)) != cudaSuccess) return MOE_ERR_DEVICE;
  for (int s = 0; s < MOE_CLOCK_NSLOT; ++s) {
    out[2 * s] = v[s][0];
    out[2 * s + 1] = v[s][1];
  }
  if (reset) {
    const unsigned long long zero[MOE_CLOCK_NSLOT][2] = {};
    if (cudaMemcpyToSymbol(g_moe_clock, zero, sizeof(zero)) != cudaSuccess) return MOE_ERR_DEVICE;
  }
  return MOE_OK;
}

int moe_last_error(void) {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_moe_dev_error, sizeof(v)) != cudaSuccess) return MOE_ERR_DEVICE;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_moe_dev_error, &zero, sizeof(zero)) != cudaSuccess)
    return MOE_ERR_DEVICE;
  return v ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

const char* moe_error_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_SHAPE: return "sizes out of range";
    case MOE_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_DTYPE: return "unsupported dtype or flags";
    case MOE_ERR_LAUNCH: return "kernel launch failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out of time";
    case MOE_ERR_DEVICE: return "no usable sm_103 device or CUDA call failed";
    default: return "unknown error";
  }
}

int moe_workspace_regions(const moe_desc* desc, moe_region* regions, int cap) {
  const int rc = validate_desc(desc);
  if (rc != MOE_OK) return rc;
  const Plan p = make_plan(desc);
  const struct { const char* n; size_t o, b; } all[] = {
      {"router_part", p.o_part, p.b_part}, {"router_w3", p.o_w3, p.b_w3},
      {"blk_hist", p.o_hist, p.b_hist},
      {"pair_rank", p.o_rank, p.b_rank},   {"groups", p.o_groups, p.b_groups},
      {"perm", p.o_perm, p.b_perm},        {"inv", p.o_inv, p.b_inv},
      {"x_perm", p.o_xperm, p.b_xperm},    {"h", p.o_h, p.b_h},
      {"y_perm", p.o_yperm, p.b_yperm},
      {"x_q", p.o_xq, p.b_xq},             {"h_q", p.o_hq, p.b_hq},
  };
  const int n = p.route_only ? 5 : (int)(sizeof(all) / sizeof(all[0]));
  for (int i = 0; i < n && i < cap && regions; ++i) {
    memset(regions[i].name, 0, sizeof(regions[i].name));
    strncpy(regions[i].name, all[i].n, sizeof(regions[i].name) - 1);
    regions[i].offset = all[i].o;
    regions[i].bytes = all[i].b;
  }
  return n;
}

// ---- routing with static scratch (no allocation, no caller workspace) ----
// File-scope device array: the scratch of moe_route_noalloc.  Host code must
// not pass its name to a kernel (on the host it is only a stand-in for the
// symbol); its device address is looked up on every call, with the caller's
// device current.
static __device__ __align__(256) unsigned char g_route_scratch[MOE_STATIC_SCRATCH_BYTES];

namespace {

// Device address of g_route_scratch in the current context.  Not cached: a
// context that is destroyed and created again (cudaDeviceReset) loads the
// module anew, possibly at another address, and the lookup costs about a
// microsecond.
void* route_scratch_address() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_route_scratch) != cudaSuccess) return nullptr;
  return ptr;
}

}  // namespace

int moe_route_noalloc(const moe_desc* desc, const void* x, const float* w_router,
                      const float* bias, int32_t* topk_idx, float* gates, int32_t* load_counts,
                      void* stream) {
  if (!desc) return MOE_ERR_NULL;
  moe_desc d = *desc;
  d.flags = MOE_ROUTE_ONLY;
  const int rc = validate_desc(&d);
  if (rc != MOE_OK) return rc;
  const size_t need = make_plan(&d).total;
  if (need > MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  const int dev_rc = device_ok();
  if (dev_rc != MOE_OK) return dev_rc;
  void* scratch = route_scratch_address();
  if (!scratch) return MOE_ERR_DEVICE;
  return forward_impl(&d, x, w_router, bias, nullptr, nullptr, nullptr, topk_idx, gates,
                      load_counts, scratch, MOE_STATIC_SCRATCH_BYTES,
                      static_cast<cudaStream_t>(stream));
}

}  // extern "C"
