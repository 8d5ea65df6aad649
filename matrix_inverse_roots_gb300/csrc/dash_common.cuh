// Shared device helpers for the dashroot kernels: operand formats, bounded
// mbarrier waits, TMA and tcgen05 (5th-generation tensor core) wrappers.
// Everything here is written for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dash {

// Storage format of a stacked matrix inside the library.
enum Fmt : int {
  FMT_F32 = 0,    // plain fp32
  FMT_TF32 = 1,   // fp32 container holding a value rounded to TF32 (RNA)
  FMT_SPLIT = 2,  // two fp32 arrays: hi = rna_tf32(x), lo = rna_tf32(x - hi)
  FMT_F16 = 3,
  FMT_BF16 = 4,
  // Unevaluated sum of two 16-bit numbers in two arrays: hi = rn16(x), lo =
  // rn16(x - hi) (x - hi is exact in fp32).  About 22 significant bits (fp16) or
  // 16 (bf16) in the range of the 16-bit type; a tensor-core operand of this
  // format takes two products, one per part.
  FMT_F16X2 = 5,
  FMT_BF16X2 = 6,
};

// Tensor-core operand kinds.  The _SPLITB kinds take B in FMT_F16X2 / FMT_BF16X2:
// C = A B_hi + A B_lo, both products of one 16-bit type.
enum Kind : int {
  KIND_F16 = 0,
  KIND_BF16 = 1,
  KIND_TF32 = 2,
  KIND_TF32X3 = 3,
  KIND_F16_SPLITB = 4,
  KIND_BF16_SPLITB = 5
};

// Device error codes recorded in g_dash_error (mirrors dash_status values).
constexpr int DEV_ERR_TIMEOUT = 5;
constexpr int DEV_ERR_CONFLICT = 6;

// Time limit of any single device-side wait, in nanoseconds of %globaltimer.
constexpr unsigned long long WAIT_LIMIT_NS = 4000000000ull;

// One flag per translation unit; each unit exports a host reader for it.
static __device__ int g_dash_error = 0;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Upper bound, in ns, on how long one try_wait may keep its thread suspended before
// returning false; the thread resumes as soon as the phase completes.  Waiting warps
// then issue less while they wait: in the benchmark step, timed launch by launch on
// two boxes, the step ran 0.7% and 1.4% faster than with the default limit.
constexpr uint32_t SUSPEND_HINT_NS = 20000u;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(SUSPEND_HINT_NS)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity of barrier `bar` has completed.
// Gives up when *abort becomes non-zero (another role gave up) or after
// WAIT_LIMIT_NS; on a time-out it raises *abort and the device error flag.
// Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort = 1;
        atomicExch(&g_dash_error, DEV_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// mbar_wait with acquire at cluster scope, for a barrier that other CTAs of the
// cluster arrive on (their release orders their earlier accesses before ours).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort) {
  const unsigned long long t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((++n & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort = 1;
        atomicExch(&g_dash_error, DEV_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      atomicExch(&g_dash_error, DEV_ERR_TIMEOUT);
      return;
    }
  }
}

// Sum over the 32 lanes of x[c] for every c; lane l returns the total of column l.
__device__ __forceinline__ float butterfly_colsum(float (&x)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      // Keep the half of the columns this lane is responsible for, send the other.
      const float send = upper ? x[i] : x[i + half];
      const float keep = upper ? x[i + half] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  return x[0];
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled bulk tensor load global -> shared, completion on mbarrier `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full barrier across the thread block cluster (every thread of every CTA).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// 3-D tiled store shared -> global, tracked as a bulk async-group of this thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to TMA.
__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-wide TMEM allocation; the base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Shared-memory matrix layouts understood by tcgen05 descriptors.
constexpr uint32_t LAYOUT_SW128 = 2;         // 128-byte swizzle of 16-byte chunks
constexpr uint32_t LAYOUT_SW128_BASE32 = 1;  // 128-byte swizzle of 32-byte chunks (MN-major TF32)

// Shared-memory matrix descriptor, descriptor version 1.  lbo / sbo in bytes
// (multiples of 16); layout one of LAYOUT_*.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // version
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return smem_desc(saddr, lbo, sbo, LAYOUT_SW128);
}

// Instruction descriptor for kind::f16 / kind::tf32 with fp32 accumulation.
// fmt: 0 = F16, 1 = BF16, 2 = TF32.  major: 0 = K-major, 1 = MN-major.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t fmt, uint32_t a_mn, uint32_t b_mn,
                                                  uint32_t M, uint32_t N) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) |
         ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (TMEM) += A (TMEM) * B (shared-memory descriptor), TF32.  A holds one 32-bit
// element per TMEM column, row m in lane m; a_tmem addresses its first column.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ---- pair-of-CTAs (cta_group::2) forms: one MMA spans the TMEM and shared
// memory of two peer CTAs (cluster ranks 2k, 2k+1); the even CTA issues it.

// Address of the same shared-memory object in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly a peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// The same arrive with the default (release, CTA scope) semantics: no cluster-wide
// memory fence.  For handing a tensor-memory buffer back to the peer that issues
// the MMAs, where the only accesses to order are this thread's tcgen05.ld, already
// completed (tcgen05.wait::ld) and ordered by tcgen05.fence::before_thread_sync.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 3-D tiled load into this CTA's shared memory whose completion is counted on
// `bar`, which may be the peer CTA's barrier (shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile"
      ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` in every CTA of cta_mask once the pair MMAs issued so far are done.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Each thread writes 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Ties the registers of r to a preceding tcgen05.wait::ld (see tmem_wait_ld).
__device__ __forceinline__ void tmem_fence_regs(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])::"memory");
}

// Waits for outstanding tcgen05.ld and ties the registers of r to the wait, so
// that no use of r can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])::"memory");
}

// ---------------------------------------------------------------- packed fp32 pairs
// Two fp32 values in one 64-bit register (lo = first), added lane by lane with
// round-to-nearest: bit for bit two __fadd_rn, in one instruction.

__device__ __forceinline__ uint64_t f32x2_pack(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

__device__ __forceinline__ void f32x2_unpack(uint64_t v, uint32_t& lo, uint32_t& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}

__device__ __forceinline__ void f32x2_add_rn(uint64_t& acc, uint64_t v) {
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(v));
}

// ---------------------------------------------------------------- formats

// Round an fp32 value to the nearest TF32 value (ties away from zero).
__device__ __forceinline__ float rna_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Bytes per element of a storage format (both halves for the split formats).
__host__ __device__ constexpr int fmt_bytes(int fmt) {
  return fmt == FMT_SPLIT ? 8 : ((fmt == FMT_F16 || fmt == FMT_BF16) ? 2 : 4);
}

__host__ __device__ constexpr bool fmt_is_pair16(int fmt) {
  return fmt == FMT_F16X2 || fmt == FMT_BF16X2;
}

// The two 16-bit parts of x: hi = rn16(x), lo = rn16(x - hi), packed two values
// per 32-bit word (a in the low half).
__device__ __forceinline__ void pair16_pack(bool bf, float a, float b, uint32_t& hi, uint32_t& lo) {
  if (bf) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
  } else {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
  }
}

// Value of one packed word pair (two elements) of a pair format.
__device__ __forceinline__ float2 pair16_unpack(bool bf, uint32_t hi, uint32_t lo) {
  if (bf) {
    const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi));
    const float2 l = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&lo));
    return make_float2(h.x + l.x, h.y + l.y);
  }
  const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  const float2 l = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  return make_float2(h.x + l.x, h.y + l.y);
}

// Element offset helpers use 64-bit arithmetic throughout.
__device__ __forceinline__ float load_elem(int fmt, const void* hi, const void* lo, int64_t i) {
  switch (fmt) {
    case FMT_F16:
      return __half2float(static_cast<const __half*>(hi)[i]);
    case FMT_BF16:
      return __bfloat162float(static_cast<const __nv_bfloat16*>(hi)[i]);
    case FMT_SPLIT:
      return static_cast<const float*>(hi)[i] + static_cast<const float*>(lo)[i];
    case FMT_F16X2:
      return __half2float(static_cast<const __half*>(hi)[i]) +
             __half2float(static_cast<const __half*>(lo)[i]);
    case FMT_BF16X2:
      return __bfloat162float(static_cast<const __nv_bfloat16*>(hi)[i]) +
             __bfloat162float(static_cast<const __nv_bfloat16*>(lo)[i]);
    default:
      return static_cast<const float*>(hi)[i];
  }
}

// Loads 4 consecutive elements starting at i (i a multiple of 4).
__device__ __forceinline__ void load4(int fmt, const void* hi, const void* lo, int64_t i,
                                      float (&v)[4]) {
  if (fmt == FMT_F16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __half*>(hi) + i);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  } else if (fmt == FMT_BF16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(hi) + i);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  } else if (fmt_is_pair16(fmt)) {
    const bool bf = (fmt == FMT_BF16X2);
    const uint2 h = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(hi) + i);
    const uint2 l = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(lo) + i);
    const float2 a = pair16_unpack(bf, h.x, l.x);
    const float2 b = pair16_unpack(bf, h.y, l.y);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  } else {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(hi) + i);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    if (fmt == FMT_SPLIT) {
      const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(lo) + i);
      v[0] += b.x; v[1] += b.y; v[2] += b.z; v[3] += b.w;
    }
  }
}

// Stores 4 consecutive elements starting at i (i a multiple of 4).
__device__ __forceinline__ void store4(int fmt, void* hi, void* lo, int64_t i, const float (&v)[4]) {
  if (fmt == FMT_F16) {
    __half2 a = __floats2half2_rn(v[0], v[1]);
    __half2 b = __floats2half2_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__half*>(hi) + i) = u;
  } else if (fmt == FMT_BF16) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(hi) + i) = u;
  } else if (fmt_is_pair16(fmt)) {
    const bool bf = (fmt == FMT_BF16X2);
    uint2 h, l;
    pair16_pack(bf, v[0], v[1], h.x, l.x);
    pair16_pack(bf, v[2], v[3], h.y, l.y);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(hi) + i) = h;
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(lo) + i) = l;
  } else if (fmt == FMT_TF32) {
    float4 a = make_float4(rna_tf32(v[0]), rna_tf32(v[1]), rna_tf32(v[2]), rna_tf32(v[3]));
    *reinterpret_cast<float4*>(static_cast<float*>(hi) + i) = a;
  } else if (fmt == FMT_SPLIT) {
    float h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[j] = rna_tf32(v[j]);
      l[j] = rna_tf32(v[j] - h[j]);
    }
    *reinterpret_cast<float4*>(static_cast<float*>(hi) + i) = make_float4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<float4*>(static_cast<float*>(lo) + i) = make_float4(l[0], l[1], l[2], l[3]);
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(hi) + i) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// ---------------------------------------------------------------- 256-bit access
// 32 consecutive bytes per thread: a whole L2 sector per access.

__device__ __forceinline__ void st_v8(void* p, const uint32_t (&r)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void ld_v8(const void* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Stores 16 consecutive elements starting at i (i a multiple of 16) with 256-bit
// stores; the base pointers must be 32-byte aligned.
__device__ __forceinline__ void store16_v8(int fmt, void* hi, void* lo, int64_t i,
                                           const float (&v)[16]) {
  if (fmt == FMT_F16 || fmt == FMT_BF16) {
    uint32_t r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      r[j] = (fmt == FMT_F16) ? pack_half2(v[2 * j], v[2 * j + 1])
                              : pack_bf162(v[2 * j], v[2 * j + 1]);
    st_v8(static_cast<uint16_t*>(hi) + i, r);
    return;
  }
  if (fmt_is_pair16(fmt)) {
    uint32_t rh[8], rl[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) pair16_pack(fmt == FMT_BF16X2, v[2 * j], v[2 * j + 1], rh[j], rl[j]);
    st_v8(static_cast<uint16_t*>(hi) + i, rh);
    st_v8(static_cast<uint16_t*>(lo) + i, rl);
    return;
  }
  uint32_t h[16], l[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float x = v[j];
    if (fmt == FMT_TF32 || fmt == FMT_SPLIT) x = rna_tf32(v[j]);
    h[j] = __float_as_uint(x);
    if (fmt == FMT_SPLIT) l[j] = __float_as_uint(rna_tf32(v[j] - x));
  }
  float* ph = static_cast<float*>(hi) + i;
  st_v8(ph, *reinterpret_cast<const uint32_t(*)[8]>(&h[0]));
  st_v8(ph + 8, *reinterpret_cast<const uint32_t(*)[8]>(&h[8]));
  if (fmt == FMT_SPLIT) {
    float* pl = static_cast<float*>(lo) + i;
    st_v8(pl, *reinterpret_cast<const uint32_t(*)[8]>(&l[0]));
    st_v8(pl + 8, *reinterpret_cast<const uint32_t(*)[8]>(&l[8]));
  }
}

// Loads 16 consecutive elements starting at i (i a multiple of 16) with 256-bit
// loads; the base pointers must be 32-byte aligned.
__device__ __forceinline__ void load16_v8(int fmt, const void* hi, const void* lo, int64_t i,
                                          float (&v)[16]) {
  if (fmt == FMT_F16 || fmt == FMT_BF16) {
    uint32_t r[8];
    ld_v8(static_cast<const uint16_t*>(hi) + i, r);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (fmt == FMT_F16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r[j]));
        v[2 * j] = f.x;
        v[2 * j + 1] = f.y;
      } else {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r[j]));
        v[2 * j] = f.x;
        v[2 * j + 1] = f.y;
      }
    }
    return;
  }
  if (fmt_is_pair16(fmt)) {
    uint32_t rh[8], rl[8];
    ld_v8(static_cast<const uint16_t*>(hi) + i, rh);
    ld_v8(static_cast<const uint16_t*>(lo) + i, rl);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = pair16_unpack(fmt == FMT_BF16X2, rh[j], rl[j]);
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
    return;
  }
  uint32_t a[8], b[8];
  const float* ph = static_cast<const float*>(hi) + i;
  ld_v8(ph, a);
  ld_v8(ph + 8, b);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = __uint_as_float(a[j]);
    v[8 + j] = __uint_as_float(b[j]);
  }
  if (fmt == FMT_SPLIT) {
    const float* pl = static_cast<const float*>(lo) + i;
    ld_v8(pl, a);
    ld_v8(pl + 8, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] += __uint_as_float(a[j]);
      v[8 + j] += __uint_as_float(b[j]);
    }
  }
}

__device__ __forceinline__ bool aligned32(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 31u) == 0;
}

}  // namespace dash
