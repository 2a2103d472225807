// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, TMA tensor
// loads, and the 5th-generation tensor core (tcgen05: TMEM allocation, MMA,
// commit, TMEM loads).  Every wait on an mbarrier is bounded in time; a wait
// that runs out records MOE_DEV_ERR_TIMEOUT in the device error word and
// returns false so the caller can unwind instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

// Device error word: OR of MOE_DEV_ERR_* bits, read by moe_last_error().
static __device__ unsigned int g_moe_dev_error;
#define MOE_DEV_ERR_TIMEOUT 1u

// Upper bound on any single mbarrier wait (ns of %globaltimer).  A tile of
// the largest workload takes well under a millisecond; 4 s only trips when
// something is genuinely stuck.
#define MOE_WAIT_LIMIT_NS 4000000000ull

// In-band SM clock record: per kernel class (slot), the sums over CTAs of
// the SM clock cycles and of the %globaltimer ns from a CTA's start to its
// end (read by moe_sm_clock_record).
#define MOE_CLOCK_NSLOT 4
static __device__ unsigned long long g_moe_clock[MOE_CLOCK_NSLOT][2];

MOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEV uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct SmClockStart {
  uint64_t clk, ns;
};
MOE_DEV SmClockStart sm_clock_start() { return {(uint64_t)clock64(), global_timer_ns()}; }
MOE_DEV void sm_clock_add(int slot, SmClockStart s0) {
  const uint64_t clk = (uint64_t)clock64() - s0.clk, ns = global_timer_ns() - s0.ns;
  atomicAdd(&g_moe_clock[slot][0], (unsigned long long)clk);
  atomicAdd(&g_moe_clock[slot][1], (unsigned long long)ns);
}

// true in one lane of the converged warp (elect.sync).  Single-thread
// tcgen05 instructions are issued from such a lane inside loops that the
// whole warp runs: their control flow and operands then stay warp-uniform.
// (Issued from a loop that one lane runs alone, the same MMA sequence cost
// its thread about 105 cycles per MMA instead of at most 66 -- less than the
// MMA itself takes only for N above 200.)
MOE_DEV bool elect_one() {
  uint32_t p;
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}\n"
      : "=r"(p));
  return p != 0;
}

// ------------------------------------------------------------------ mbarrier
MOE_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

MOE_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

MOE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Bounded by
// MOE_WAIT_LIMIT_NS of wall time and by an iteration cap; returns false (and
// flags the device error word) if either runs out.
MOE_DEV bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && global_timer_ns() - t0 > MOE_WAIT_LIMIT_NS) break;
  }
  atomicOr(&g_moe_dev_error, MOE_DEV_ERR_TIMEOUT);
  return false;
}

// ------------------------------------------------------------------ TMA
// 2-D tiled tensor load global -> shared, completion counted in bytes on
// `bar`.  x is the innermost (contiguous) coordinate in elements; callers
// only pass multiples of 64 bf16 elements (128 bytes), so every copy starts
// on a 16-byte boundary.
MOE_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

MOE_DEV uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MOE_DEV uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MOE_DEV uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MOE_DEV void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
MOE_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

MOE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major bf16 operand tile stored as
// rows of 128 bytes (64 elements) with the 128-byte swizzle that TMA's
// CU_TENSOR_MAP_SWIZZLE_128B writes: 8-row atoms of 1024 bytes stacked
// densely (stride byte offset 1024).  Fields: start address >> 4 (bits
// 0-13), leading byte offset >> 4 (16-29; unused for swizzled K-major, set to
// 1), stride byte offset >> 4 (32-45), descriptor version 1 (46-47), base
// offset 0 (49-51; tiles are 1024-byte aligned), layout 2 = SWIZZLE_128B
// (61-63).  The k-th 16-element K slice of a row starts 32*k bytes further on.
MOE_DEV uint64_t umma_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// The same for an MN-major operand (the matrix stored transposed: K rows of
// contiguous M (or N) elements), as TMA writes a box of 64 elements x 64 K
// rows with the 128-byte swizzle: 8-row K groups of 1024 bytes (stride byte
// offset 1024), blocks of 64 M elements `lbo` bytes apart (leading byte
// offset).  The k-th 16-row K slice starts 2048*k bytes further on.  The
// instruction descriptor must mark the operand transposed (bit 15 for A).
MOE_DEV uint64_t umma_desc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

MOE_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B, fp32
// accumulator, both operands K-major, no negation, dense: D format (bits
// 4-5) = 1 (F32), A format (7-9) = 1 (BF16), B format (10-12) = 1 (BF16),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
MOE_DEV uint32_t umma_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
MOE_DEV void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
MOE_DEV void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

#define MOE_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                  "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])

// One 32-column load of this warp's 32 TMEM lanes (one fp32 value per lane
// per column) and its wait, in one asm statement so that no register is read
// before the wait.
MOE_DEV void tmem_load_32(uint32_t ta, float* a) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : MOE_R8(0), MOE_R8(8), MOE_R8(16), MOE_R8(24)
      : "r"(ta)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) a[i] = __uint_as_float(r[i]);
}

// Two such loads, from column addresses ta and tb, and one wait.
MOE_DEV void tmem_load_2x32(uint32_t ta, uint32_t tb, float* a, float* b) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : MOE_R8(0), MOE_R8(8), MOE_R8(16), MOE_R8(24), MOE_R8(32), MOE_R8(40), MOE_R8(48),
        MOE_R8(56)
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[32 + i]);
  }
}
#undef MOE_R8

// TMEM -> registers in the 16x256b shape, four repetitions along columns:
// for a TMEM address with lane field b (a multiple of 16 inside the warp's
// 32-lane quarter) and column c, thread t receives in r[4 i + j] lane
// b + t/4 + 8 (j/2), column c + 8 i + 2 (t%4) + (j%2), i = 0..3 -- the
// accumulator-fragment layout that stmatrix consumes.  Two loads, one wait.
#define MOE_R16(r) "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), \
    "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),    \
    "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
MOE_DEV void tmem_load_16x256b_2(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : MOE_R16(a), MOE_R16(b)
      : "r"(ta), "r"(tb)
      : "memory");
}
MOE_DEV void tmem_load_16x256b(uint32_t ta, uint32_t (&a)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : MOE_R16(a)
      : "r"(ta)
      : "memory");
}
#undef MOE_R16

// Four 8 x 8 b16 matrices from fragment registers (thread t: row t/4,
// columns 2 (t%4) and +1 of each) to shared memory, transposed: the row whose
// address thread 8 m + i gives receives column i of matrix m.
MOE_DEV void stmatrix_x4_trans(uint32_t addr, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};"
               :: "r"(addr), "r"(w0), "r"(w1), "r"(w2), "r"(w3) : "memory");
}

// The inverse: four 8 x 8 b16 matrices from shared memory into fragment
// registers, transposed (the row whose address thread 8 m + i gives is read
// as column i of matrix m).
MOE_DEV void ldmatrix_x4_trans(uint32_t addr, uint32_t& w0, uint32_t& w1, uint32_t& w2,
                               uint32_t& w3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
               : "r"(addr)
               : "memory");
}

// Generic-proxy writes to shared memory become visible to the async proxy
// (TMA) once the writing threads execute this fence.
MOE_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// TMA store of one box from shared memory; completion tracked by bulk groups.
MOE_DEV void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               :: "l"(map), "r"(x), "r"(y), "r"(src) : "memory");
}
MOE_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed store has finished reading its shared-memory source
MOE_DEV void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all but the N most recently committed stores have read their sources
template <int N>
MOE_DEV void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory"); }
// every committed store has completed
MOE_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------------ CTA pairs
// Primitives for the 2-SM (cta_group::2) tensor-core MMA: a cluster of two
// CTAs on two SMs computes one M = 256 tile; each CTA holds half of A (128
// rows) and half of B (N/2 rows) at the same shared-memory offsets, and its
// own TMEM receives its 128 rows of D.

MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full barrier across the CTAs of the cluster (every CTA must reach it).
MOE_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
MOE_DEV uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

MOE_DEV void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

MOE_DEV void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (here: the leader's).
MOE_DEV void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t mbar_cluster, int x,
                              int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar_cluster), "l"(policy)
      : "memory");
}

MOE_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

MOE_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D (+)= A * B^T with M = 256 over the CTA pair, issued by one thread of the
// leader CTA.
MOE_DEV void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with e4m3 A and B (kind::f8f6f4, K = 32 per instruction, so one
// 32-byte K slice of a 128-byte row as for bf16).
MOE_DEV void umma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f8f6f4 with e4m3 A and B (format 0), fp32
// accumulator, both K-major: the bf16 descriptor's fields without the bf16
// format codes.
MOE_DEV uint32_t umma_idesc_e4m3(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Arrive once on the mbarrier at the same offset in both CTAs of the pair
// when every pair MMA issued so far has completed.
MOE_DEV void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], "
      "%1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

// Bounded wait with cluster-scope acquire, for barriers that the other CTA of
// the pair arrives on (its preceding writes become visible here).
MOE_DEV bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

MOE_DEV bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 63u && global_timer_ns() - t0 > MOE_WAIT_LIMIT_NS) break;
  }
  atomicOr(&g_moe_dev_error, MOE_DEV_ERR_TIMEOUT);
  return false;
}

// Arrive on this CTA's own mbarrier when the pair MMAs issued so far complete.
MOE_DEV void umma_commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Two fp32 values to e4m3 codes, nearest-even with saturation to +-448 (NaN
// stays NaN): lo in the low byte.
MOE_DEV uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------------ block-scaled MMA
// tcgen05.mma kind::mxf8f6f4 with block scaling (scale_vec::1X: one UE8M0
// scale byte, 2^(byte - 127), per row of A and per column of B for each
// K = 32 slice), e4m3 A and B, fp32 accumulator.  The scales live in TMEM:
// the scale of A row m (of this CTA's 128) is read from lane m, column
// sfa + m / 32; the scale of B column n from lane n % 32 of the quarter that
// computes the row, column sfb + n / 32, so every lane quarter holds a copy
// (tcgen05.cp .32x128b.warpx4 writes exactly that).  Each 32-bit TMEM cell
// holds four scale bytes; the instruction descriptor's scale-factor IDs pick
// the byte (bits 29-30 for A, 4-5 for B).  Descriptor: B scale ID (4-5), A
// and B format e4m3 = 0 (7-9, 10-12), K-major, N >> 3 (17-22), scale type
// UE8M0 = 1 (23), M >> 4 (24-28), A scale ID (29-30).
MOE_DEV uint32_t umma_idesc_mx_e4m3(int m, int n, uint32_t sf_id) {
  return (sf_id << 4) | ((uint32_t)(n >> 3) << 17) | (1u << 23) | ((uint32_t)(m >> 4) << 24) |
         (sf_id << 29);
}

// D (+)= A * B^T with block scales, M = 256 over the CTA pair (leader only).
MOE_DEV void umma_mx_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte matrix (no swizzle, rows of
// 16 bytes stored densely: 8-row core groups 128 bytes apart), the source of
// a .32x128b copy.
MOE_DEV uint64_t smem_desc_rows16(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// Copy 32 rows of 16 bytes from shared memory into TMEM columns taddr ..
// taddr + 3 (row r -> lane r of every lane quarter, word w -> column w), in
// both CTAs of the pair, each from its own shared memory; issued by the
// leader's MMA thread, ordered before the MMAs it issues afterwards.
MOE_DEV void tmem_cp_pair_32x128b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Exponent e of the power-of-two scale of a block whose largest magnitude
// has the fp32 bit pattern `amax_bits` (sign cleared): the smallest integer
// with amax <= 448 * 2^e, 0 for a block of zeros or one whose maximum is not
// finite, clamped to [-127, 127].  With amax = m * 2^E, m in [1, 2): e = E - 8
// when m <= 1.75 (448 = 1.75 * 2^8), else E - 7; subnormal maxima give
// exponents below -127.
MOE_DEV int block_exp_from_bits(uint32_t amax_bits) {
  if (amax_bits == 0u || amax_bits >= 0x7f800000u) return 0;
  const int ef = (int)(amax_bits >> 23);
  if (ef == 0) return -127;
  const int E = ef - 127;
  const int e = (amax_bits & 0x7fffffu) <= 0x600000u ? E - 8 : E - 7;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as fp32 for the exponents block_exp_from_bits gives finite maxima
// (-127 <= e <= 120).
MOE_DEV float exp2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }
