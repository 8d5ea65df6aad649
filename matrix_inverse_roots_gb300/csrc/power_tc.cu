// One power-iteration product W = (A + ridge I) V D for every block, on the
// 5th-generation tensor cores in 3xTF32 (fp32-level accuracy).
//
// A is the caller's fp32 stack; V is B x 32 per block (row stride 32, the 32
// start-vector columns); D = diag(1 / ||previous column||) is applied to the
// accumulator, since (A V) D = A (V D).  The product is a skinny GEMM
// (M = B rows, N = 32, K = B) whose cost is reading A once, so the kernel is
// built to stream A from HBM at full rate, with as many bytes in flight as the
// shared memory holds:
//   warp 0      TMA producer: per k-block a 128 x 32 fp32 tile of A (K-major,
//               128B swizzle) and the 32 x 32 tile of V (MN-major: the 32
//               vectors are one 128-byte atom, 32-byte swizzle atoms) into a
//               ring of nine 24 KB stages.
//   warps 2..5  converters: each thread reads one row of the A tile, splits it
//               into TF32 hi and lo and writes both into a TMEM operand buffer
//               (tcgen05.st), so the split costs no shared-memory writes and the
//               ring holds only raw data; the small V tile is split in place
//               (hi over the fp32 data, lo beside it).
//   warp 1      one thread issues, per K = 8 slice, A_hi [V_hi | V_lo] (N = 64:
//               V_lo sits one operand atom after V_hi) and A_lo V_hi (N = 32) into
//               a 64-column TMEM accumulator, A read from TMEM and V from shared
//               memory; two accumulators alternate.  The epilogue adds the halves.
//   warps 6..9  epilogue: one accumulator row per thread; scale, ridge term,
//               W stored as contiguous 128-byte rows; column sums (W^2, or v.w and
//               v.v on the last product) reduced with a butterfly shuffle and one
//               atomic per warp and column.
// The CTA grid is persistent over 128-row slabs, ordered block-major.
// Every wait is bounded; a time-out sets the device flag and the CTA drains
// its copies and MMAs, frees TMEM and returns.
#include "dash_common.cuh"
#include "dash_internal.h"

namespace dash {

int power_tc_read_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_dash_error, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_dash_error, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

namespace {

constexpr int PT_BM = 128;
constexpr int PT_BK = 32;                 // fp32 elements per 128-byte row
constexpr int PT_NV = 32;
constexpr int PT_A_BYTES = PT_BM * 128;   // 16 KB
constexpr int PT_V_BYTES = PT_BK * 128;   // 4 KB
// Stage: A (raw fp32) | V (hi after conversion) | V lo.
constexpr int PT_STAGE_BYTES = PT_A_BYTES + 2 * PT_V_BYTES;  // 24 KB
constexpr int PT_STAGES = 9;
// TMEM: two 64-column accumulators at column 0 (A_hi V_hi + A_lo V_hi | A_hi V_lo);
// PT_ABUFS A-operand buffers of 64 columns (hi in the first 32, lo in the next 32)
// from column PT_ACOL.
constexpr int PT_ACC_COLS = 2 * PT_NV;
constexpr int PT_ABUFS = 4;
constexpr int PT_ACOL = 256;
constexpr int PT_TMEM_COLS = 512;
constexpr int PT_THREADS = 320;
// mbarriers: full, conv, empty per stage; 2 + 2 accumulator; fin; one per A buffer.
constexpr int PT_NBAR = 3 * PT_STAGES + 5 + PT_ABUFS;
constexpr int PT_BAR_AREA = 512;
static_assert(PT_NBAR * 8 + 16 <= PT_BAR_AREA, "barrier area");
constexpr int PT_SMEM_BYTES = PT_STAGES * PT_STAGE_BYTES + 1024 + PT_BAR_AREA;
static_assert(PT_SMEM_BYTES <= 232448, "shared memory budget");

struct PowerParams {
  int dim;
  long long nblocks;
  long long slabs;  // nblocks * dim / 128
  int nkb;          // dim / 32
  uint32_t idesc;     // M = 128, N = 64
  uint32_t idesc32;   // M = 128, N = 32
  float ridge;
  const float* Vin;       // (nblocks, dim, 32)
  const float* in_nrm2;   // (nblocks, 32) or null
  float* Wout;            // (nblocks, dim, 32); unused on the last product
  float* acc0;            // W.W per column, or v.w on the last product
  float* acc1;            // v.v per column on the last product
  int nv;
  int last;
};

__global__ void __launch_bounds__(PT_THREADS, 1)
    power_tc_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tV,
                    const __grid_constant__ PowerParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;
  uint8_t* bar_area = smem + PT_STAGES * PT_STAGE_BYTES;
  const uint32_t bar0 = sbase + PT_STAGES * PT_STAGE_BYTES;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto conv_bar = [&](int s) { return bar0 + 8u * (PT_STAGES + s); };
  auto empty_bar = [&](int s) { return bar0 + 8u * (2 * PT_STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (3 * PT_STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (3 * PT_STAGES + 2 + a); };
  const uint32_t fin_bar = bar0 + 8u * (3 * PT_STAGES + 4);
  auto aempty_bar = [&](int b) { return bar0 + 8u * (3 * PT_STAGES + 5 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * PT_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * PT_NBAR + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int slabs_per_blk = p.dim / PT_BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PT_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(conv_bar(s), 4);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(fin_bar, 1);
    for (int b = 0; b < PT_ABUFS; ++b) mbar_init(aempty_bar(b), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tA);
    tma_prefetch_desc(&tV);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), PT_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (long long sl = blockIdx.x; sl < p.slabs && ok; sl += gridDim.x) {
        const int blk = static_cast<int>(sl / slabs_per_blk);
        const int m0 = static_cast<int>(sl % slabs_per_blk) * PT_BM;
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, PT_A_BYTES + PT_V_BYTES);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          const uint32_t s0 = sbase + stage * PT_STAGE_BYTES;
          tma_load_3d(s0, &tA, fb, kb * PT_BK, m0, blk);
          tma_load_3d(s0 + PT_A_BYTES, &tV, fb, 0, kb * PT_BK, blk);
          if (++stage == PT_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < PT_STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (long long sl = blockIdx.x; sl < p.slabs && ok; sl += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PT_ACC_COLS);
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!mbar_wait(conv_bar(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sV = sbase + stage * PT_STAGE_BYTES + PT_A_BYTES;
          const uint32_t ta = tmem_base + static_cast<uint32_t>(PT_ACOL + abuf * 64);
#pragma unroll
          for (int kk = 0; kk < PT_BK / 8; ++kk) {
            // V is MN-major TF32: 32-byte swizzle atoms, 4-row K slabs (SBO 512);
            // the next N atom (LBO) is V_lo, so N = 64 reads [V_hi | V_lo].
            const uint64_t dv = smem_desc(sV + kk * 8 * 128, PT_V_BYTES, 512, LAYOUT_SW128_BASE32);
            const uint32_t a_hi = ta + kk * 8, a_lo = ta + 32 + kk * 8;
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            mma_tf32_ts(d_tmem, a_hi, dv, p.idesc, accum);
            mma_tf32_ts(d_tmem, a_lo, dv, p.idesc32, 1u);
          }
          mma_commit(empty_bar(stage));
          mma_commit(aempty_bar(abuf));
          if (++stage == PT_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (++abuf == PT_ABUFS) abuf = 0;
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      mma_commit(fin_bar);
      mbar_wait_drain(fin_bar, 0);
    }
  } else if (warp < 6) {
    // -------------------------------------------------------------- converters
    const int ct = threadIdx.x - 64;  // 0..127
    const int q = warp & 3;           // TMEM lane quarter this warp may write
    const int r = q * 32 + lane;      // A-tile row this thread splits
    int stage = 0;
    uint32_t phase = 0;
    int abuf = 0;
    uint32_t aphase = 0;
    bool ok = true;
    for (long long sl = blockIdx.x; sl < p.slabs && ok; sl += gridDim.x) {
      for (int kb = 0; kb < p.nkb; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag) ||
            !mbar_wait(aempty_bar(abuf), aphase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* st = smem + stage * PT_STAGE_BYTES;
        // Row r of the 128B-swizzled tile: logical 16-byte chunk j sits at j ^ (r & 7).
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 x = *reinterpret_cast<const float4*>(st + r * 128 + ((j ^ (r & 7)) << 4));
          const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float h = rna_tf32(xs[e]);
            hi[4 * j + e] = __float_as_uint(h);
            lo[4 * j + e] = __float_as_uint(rna_tf32(xs[e] - h));
          }
        }
        const uint32_t ta = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(PT_ACOL + abuf * 64);
        tmem_st16(ta, reinterpret_cast<const uint32_t(&)[16]>(hi[0]));
        tmem_st16(ta + 16, reinterpret_cast<const uint32_t(&)[16]>(hi[16]));
        tmem_st16(ta + 32, reinterpret_cast<const uint32_t(&)[16]>(lo[0]));
        tmem_st16(ta + 48, reinterpret_cast<const uint32_t(&)[16]>(lo[16]));
        // V: 256 16-byte chunks, element-wise, so the swizzle is kept.
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = ct + 128 * i;
          float4* hp = reinterpret_cast<float4*>(st + PT_A_BYTES + 16 * c);
          float4* lp = reinterpret_cast<float4*>(st + PT_A_BYTES + PT_V_BYTES + 16 * c);
          const float4 x = *hp;
          float4 h, l;
          h.x = rna_tf32(x.x); l.x = rna_tf32(x.x - h.x);
          h.y = rna_tf32(x.y); l.y = rna_tf32(x.y - h.y);
          h.z = rna_tf32(x.z); l.z = rna_tf32(x.z - h.z);
          h.w = rna_tf32(x.w); l.w = rna_tf32(x.w - h.w);
          *hp = h;
          *lp = l;
        }
        tmem_wait_st();
        fence_async_shared();  // generic-proxy writes -> tensor-core reads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(conv_bar(stage));
        if (++stage == PT_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++abuf == PT_ABUFS) {
          abuf = 0;
          aphase ^= 1u;
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row_in = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (long long sl = blockIdx.x; sl < p.slabs; sl += gridDim.x) {
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) break;
      tc_fence_after();
      const long long blk = sl / slabs_per_blk;
      const int row = static_cast<int>(sl % slabs_per_blk) * PT_BM + row_in;
      uint32_t r0[16], r1[16], r2[16], r3[16];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * PT_ACC_COLS);
      tmem_ld16(taddr, r0);
      tmem_ld16(taddr + 16, r1);
      tmem_ld16(taddr + 32, r2);
      tmem_ld16(taddr + 48, r3);
      tmem_wait_ld(r0);
      tmem_fence_regs(r1);
      tmem_fence_regs(r2);
      tmem_fence_regs(r3);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));  // accumulator copied to registers
      float sc[PT_NV];
#pragma unroll
      for (int c = 0; c < PT_NV; ++c) {
        float s = 0.0f;
        if (c < p.nv)
          s = (p.in_nrm2 != nullptr) ? 1.0f / sqrtf(p.in_nrm2[blk * PT_NV + c]) : 1.0f;
        sc[c] = s;
      }
      const float* vr = p.Vin + (blk * p.dim + row) * static_cast<long long>(PT_NV);
      float w[PT_NV], v[PT_NV];
#pragma unroll
      for (int c = 0; c < PT_NV; c += 4) {
        const float4 t = *reinterpret_cast<const float4*>(vr + c);
        v[c] = t.x * sc[c];
        v[c + 1] = t.y * sc[c + 1];
        v[c + 2] = t.z * sc[c + 2];
        v[c + 3] = t.w * sc[c + 3];
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float a0 = __uint_as_float(r0[c]) + __uint_as_float(r2[c]);
        const float a1 = __uint_as_float(r1[c]) + __uint_as_float(r3[c]);
        w[c] = fmaf(p.ridge, v[c], a0 * sc[c]);
        w[16 + c] = fmaf(p.ridge, v[16 + c], a1 * sc[16 + c]);
      }
      float s0[PT_NV], s1[PT_NV];
      if (p.last) {
#pragma unroll
        for (int c = 0; c < PT_NV; ++c) {
          s0[c] = v[c] * w[c];
          s1[c] = v[c] * v[c];
        }
      } else {
        float* wr = p.Wout + (blk * p.dim + row) * static_cast<long long>(PT_NV);
#pragma unroll
        for (int c = 0; c < PT_NV; c += 4)
          *reinterpret_cast<float4*>(wr + c) = make_float4(w[c], w[c + 1], w[c + 2], w[c + 3]);
#pragma unroll
        for (int c = 0; c < PT_NV; ++c) s0[c] = w[c] * w[c];
      }
      const float t0 = butterfly_colsum(s0, lane);
      if (lane < p.nv) atomicAdd(p.acc0 + blk * PT_NV + lane, t0);
      if (p.last) {
        const float t1 = butterfly_colsum(s1, lane);
        if (lane < p.nv) atomicAdd(p.acc1 + blk * PT_NV + lane, t1);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, PT_TMEM_COLS);
  }
}

// ---------------------------------------------------------------- half precision
// The power product in half precision ([pt] Principais Contribuicoes item 4: an
// efficient half-precision power iteration).  A is a 16-bit copy of the block
// (fp16 or bf16) and the 32 vectors are kept transposed, (32, B) per block, so
// both operands are K-major 128-byte rows: TMA brings them straight into the
// layout kind::f16 reads (no split, no converters), half the bytes of fp32.
//   warp 0      TMA producer: per k-block (64 elements) a 128 x 64 tile of A and
//               the 32 x 64 tile of V^T, ten 20 KB stages.
//   warp 1      one thread issues four M = 128, N = 32, K = 16 MMAs per k-block
//               into one of two 32-column TMEM accumulators (fp32).
//   warps 2..5  epilogue: one accumulator row per thread; scale by the previous
//               column norms, ridge term, W^T stored in the 16-bit format
//               (coalesced across the warp), fp32 column sums of the stored values.
constexpr int PH_BK = 64;                             // 16-bit elements per 128-byte row
constexpr int PH_A_BYTES = PT_BM * 128;               // 16 KB
constexpr int PH_V_BYTES = PT_NV * 128;               // 4 KB
constexpr int PH_STAGE_BYTES = PH_A_BYTES + PH_V_BYTES;
constexpr int PH_STAGES = 10;
constexpr int PH_NBAR = 2 * PH_STAGES + 5;            // full, empty; tfull x2, tempty x2; fin
constexpr int PH_THREADS = 192;
constexpr int PH_TMEM_COLS = 64;
constexpr int PH_SMEM_BYTES = PH_STAGES * PH_STAGE_BYTES + 1024 + PT_BAR_AREA;
static_assert(PH_NBAR * 8 + 16 <= PT_BAR_AREA, "barrier area");
static_assert(PH_SMEM_BYTES <= 232448, "shared memory budget");

struct PowerHalfParams {
  int dim;
  long long slabs;
  int nkb;
  uint32_t idesc;
  float ridge;
  const float* blk_scale;  // (nblocks) power-of-two scale of each 16-bit block, or null
  const uint16_t* Vt_in;  // (nblocks, 32, dim): previous vectors, transposed
  const float* in_nrm2;   // (nblocks, 32) or null
  uint16_t* Vt_out;       // (nblocks, 32, dim); unused on the last product
  float* acc0;            // W.W per column, or v.w on the last product
  float* acc1;            // v.v per column on the last product
  int nv;
  int last;
};

template <bool BF>
__device__ __forceinline__ float h16_to_f(uint16_t x) {
  if (BF) return __uint_as_float(static_cast<uint32_t>(x) << 16);
  return __half2float(__ushort_as_half(x));
}

template <bool BF>
__device__ __forceinline__ uint16_t f_to_h16(float x) {
  if (BF) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  return __half_as_ushort(__float2half_rn(x));
}

template <bool BF>
__global__ void __launch_bounds__(PH_THREADS, 1)
    power_half_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tV,
                      const __grid_constant__ PowerHalfParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;
  uint8_t* bar_area = smem + PH_STAGES * PH_STAGE_BYTES;
  const uint32_t bar0 = sbase + PH_STAGES * PH_STAGE_BYTES;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (PH_STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * PH_STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * PH_STAGES + 2 + a); };
  const uint32_t fin_bar = bar0 + 8u * (2 * PH_STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * PH_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * PH_NBAR + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int slabs_per_blk = p.dim / PT_BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PH_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(fin_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tA);
    tma_prefetch_desc(&tV);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), PH_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (long long sl = blockIdx.x; sl < p.slabs && ok; sl += gridDim.x) {
        const int blk = static_cast<int>(sl / slabs_per_blk);
        const int m0 = static_cast<int>(sl % slabs_per_blk) * PT_BM;
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, PH_STAGE_BYTES);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          const uint32_t s0 = sbase + stage * PH_STAGE_BYTES;
          tma_load_3d(s0, &tA, fb, kb * PH_BK, m0, blk);
          tma_load_3d(s0 + PH_A_BYTES, &tV, fb, kb * PH_BK, 0, blk);
          if (++stage == PH_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < PH_STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (long long sl = blockIdx.x; sl < p.slabs && ok; sl += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PT_NV);
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sbase + stage * PH_STAGE_BYTES;
          const uint32_t sV = sA + PH_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < PH_BK / 16; ++kk) {
            const uint64_t da = smem_desc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t dv = smem_desc_sw128(sV + kk * 32, 16, 1024);
            mma_f16(d_tmem, da, dv, p.idesc, (kb | kk) ? 1u : 0u);
          }
          mma_commit(empty_bar(stage));
          if (++stage == PH_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      mma_commit(fin_bar);
      mbar_wait_drain(fin_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row_in = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (long long sl = blockIdx.x; sl < p.slabs; sl += gridDim.x) {
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) break;
      tc_fence_after();
      const long long blk = sl / slabs_per_blk;
      const int row = static_cast<int>(sl % slabs_per_blk) * PT_BM + row_in;
      uint32_t r0[16], r1[16];
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * PT_NV);
      tmem_ld16(taddr, r0);
      tmem_ld16(taddr + 16, r1);
      tmem_wait_ld(r0);
      tmem_fence_regs(r1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));  // accumulator copied to registers
      float sc[PT_NV];
#pragma unroll
      for (int c = 0; c < PT_NV; ++c) {
        float s = 0.0f;
        if (c < p.nv)
          s = (p.in_nrm2 != nullptr) ? 1.0f / sqrtf(p.in_nrm2[blk * PT_NV + c]) : 1.0f;
        sc[c] = s;
      }
      // Element (c, row) of this block's V^T; consecutive lanes read consecutive rows.
      const uint16_t* vin = p.Vt_in + blk * PT_NV * static_cast<long long>(p.dim) + row;
      float w[PT_NV], v[PT_NV];
#pragma unroll
      for (int c = 0; c < PT_NV; ++c) v[c] = h16_to_f<BF>(vin[static_cast<long long>(c) * p.dim]) * sc[c];
      // The 16-bit copy holds sigma A, so the ridge term is sigma ridge.
      const float rb = (p.blk_scale != nullptr) ? p.ridge * p.blk_scale[blk] : p.ridge;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        w[c] = fmaf(rb, v[c], __uint_as_float(r0[c]) * sc[c]);
        w[16 + c] = fmaf(rb, v[16 + c], __uint_as_float(r1[c]) * sc[16 + c]);
      }
      float s0[PT_NV], s1[PT_NV];
      if (p.last) {
#pragma unroll
        for (int c = 0; c < PT_NV; ++c) {
          s0[c] = v[c] * w[c];
          s1[c] = v[c] * v[c];
        }
      } else {
        uint16_t* wout = p.Vt_out + blk * PT_NV * static_cast<long long>(p.dim) + row;
#pragma unroll
        for (int c = 0; c < PT_NV; ++c) {
          const uint16_t hw = f_to_h16<BF>(w[c]);
          wout[static_cast<long long>(c) * p.dim] = hw;
          const float wr = h16_to_f<BF>(hw);  // the next product sees the stored value
          s0[c] = wr * wr;
        }
      }
      const float t0 = butterfly_colsum(s0, lane);
      if (lane < p.nv) atomicAdd(p.acc0 + blk * PT_NV + lane, t0);
      if (p.last) {
        const float t1 = butterfly_colsum(s1, lane);
        if (lane < p.nv) atomicAdd(p.acc1 + blk * PT_NV + lane, t1);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, PH_TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

bool map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t nblk,
            uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t gdim[3] = {inner, outer, nblk};
  cuuint64_t gstride[2] = {inner * 4, inner * outer * 4};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), gdim, gstride, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_3d_h16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t nblk,
                uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t gdim[3] = {inner, outer, nblk};
  cuuint64_t gstride[2] = {inner * 2, inner * outer * 2};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), gdim, gstride, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool map_3d_u16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t nblk,
                uint32_t box_inner, uint32_t box_outer) {
  return map_3d_h16(m, base, inner, outer, nblk, box_inner, box_outer);
}

dash_status launch_power_step_half(const void* Ah, int bf16, float ridge, const float* blk_scale,
                                   int dim, long long nblocks, const uint16_t* Vt_in, int nv,
                                   const float* in_nrm2, uint16_t* Vt_out, float* acc0,
                                   float* acc1, int last, cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  CUtensorMap tA, tV;
  if (!map_3d_h16(&tA, Ah, dim, dim, nblocks, PH_BK, PT_BM)) return DASH_ERR_CUDA;
  if (!map_3d_h16(&tV, Vt_in, dim, PT_NV, nblocks, PH_BK, PT_NV)) return DASH_ERR_CUDA;
  PowerHalfParams p;
  p.dim = dim;
  p.slabs = nblocks * (dim / PT_BM);
  p.nkb = dim / PH_BK;
  p.idesc = make_idesc(bf16 ? 1u : 0u, 0, 0, PT_BM, PT_NV);
  p.ridge = ridge;
  p.blk_scale = blk_scale;
  p.Vt_in = Vt_in;
  p.in_nrm2 = in_nrm2;
  p.Vt_out = Vt_out;
  p.acc0 = acc0;
  p.acc1 = acc1;
  p.nv = nv;
  p.last = last;
  auto kern = bf16 ? power_half_kernel<true> : power_half_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PH_SMEM_BYTES) !=
      cudaSuccess)
    return DASH_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return DASH_ERR_CUDA;
  const long long grid = p.slabs < sms ? p.slabs : sms;
  const int rec = trace_begin(st);
  kern<<<static_cast<unsigned>(grid), PH_THREADS, PH_SMEM_BYTES, st>>>(tA, tV, p);
  const cudaError_t err = cudaGetLastError();
  const double bb = static_cast<double>(dim) * dim * nblocks;
  const double vb = static_cast<double>(dim) * nblocks * 2.0 * PT_NV;
  trace_end(rec, st, DASH_TRACE_POWER, 2.0 * bb * nv, 2.0 * bb + vb * (last ? 1 : 2));
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

dash_status launch_power_step_tc(const float* A, float ridge, int dim, long long nblocks,
                                 const float* Vin, int nv, const float* in_nrm2, float* Wout,
                                 float* acc0, float* acc1, int last, cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  CUtensorMap tA, tV;
  if (!map_3d(&tA, A, dim, dim, nblocks, PT_BK, PT_BM, CU_TENSOR_MAP_SWIZZLE_128B))
    return DASH_ERR_CUDA;
  if (!map_3d(&tV, Vin, PT_NV, dim, nblocks, PT_NV, PT_BK, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B))
    return DASH_ERR_CUDA;
  PowerParams p;
  p.dim = dim;
  p.nblocks = nblocks;
  p.slabs = nblocks * (dim / PT_BM);
  p.nkb = dim / PT_BK;
  p.idesc = make_idesc(2, 0, 1, PT_BM, PT_ACC_COLS);
  p.idesc32 = make_idesc(2, 0, 1, PT_BM, PT_NV);
  p.ridge = ridge;
  p.Vin = Vin;
  p.in_nrm2 = in_nrm2;
  p.Wout = Wout;
  p.acc0 = acc0;
  p.acc1 = acc1;
  p.nv = nv;
  p.last = last;
  if (cudaFuncSetAttribute(power_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PT_SMEM_BYTES) != cudaSuccess)
    return DASH_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return DASH_ERR_CUDA;
  const long long grid = p.slabs < sms ? p.slabs : sms;
  const int rec = trace_begin(st);
  power_tc_kernel<<<static_cast<unsigned>(grid), PT_THREADS, PT_SMEM_BYTES, st>>>(tA, tV, p);
  const cudaError_t err = cudaGetLastError();
  const double bb = static_cast<double>(dim) * dim * nblocks;
  const double vb = static_cast<double>(dim) * nblocks * 4.0;
  trace_end(rec, st, DASH_TRACE_POWER, 2.0 * bb * nv, 4.0 * bb + vb * (32 + (last ? 0 : 32)));
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

}  // namespace dash
