// Batched square GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA)
// with a fused epilogue.  Every dense B x B x B product of the preconditioner
// step (factor accumulation, the Coupled Newton / Newton-Denman-Beavers /
// Clenshaw iterations, the preconditioned update) runs through this kernel.
//
// Design (one CTA per SM, persistent; for B a multiple of 256 the CTAs run in
// pairs, cta_group::2, that share one 256 x 256 tile: each stages its own 128
// rows of A and half of B, the even CTA issues the MMAs, each CTA holds 128
// accumulator rows):
//   warp 0      TMA producer: streams 128-byte-wide, 128B-swizzled operand tiles
//               into a ring of shared-memory stages (mbarrier full/empty pairs).
//   warp 10     in the fixed-order pair instances, a second producer thread that
//               loads the B operand while warp 0 loads A: one thread's loop of
//               barrier waits and tiled TMA issues caps the copies it can start
//               (about one 16 KB box per 600 cycles), and two threads double it.
//               Each arms the stage's barrier for its own bytes (two arrivals).
//   warp 1      allocates TMEM and issues tcgen05.mma from one thread into one of
//               two TMEM accumulators (128 x BN fp32 each), so the epilogue of
//               tile i overlaps the MMAs of tile i+1.
//   warps 2..9  epilogue, two warps per TMEM lane quarter, each taking half of
//               the tile's columns: tcgen05.ld the accumulator (one TMEM lane =
//               one row per thread), apply D = mult*(alpha C + gamma I + eps E),
//               optional residual sum (C - I)^2 and identity padding, and store
//               in the requested format (fp32, TF32-rounded, hi/lo split, fp16,
//               bf16).  Chunks away from the diagonal take a branch-free path.
// Tiles are ordered block-major so that concurrently running CTAs share the
// operands of a few blocks in L2.  The mirrored-store pair instances (fp32 results
// of symmetric products) hand the tiles out in that order at run time (a global
// counter per launch, drawn by the even CTA's producer and passed to every role of
// the pair through a small ring in shared memory): with a fixed round-robin split,
// pairs that run slightly faster drift ahead over a long stack, the tiles in flight
// spread over more blocks than L2 holds, and operands are read from DRAM more than
// once.
// Precisions: kind::f16 (fp16 / bf16 operands), kind::tf32, and 3xTF32, which
// issues hi*lo, lo*hi and hi*hi products into the same accumulator.
// Every wait is bounded (see mbar_wait); a time-out sets the device error flag
// and the CTA drains its in-flight copies and MMAs, frees TMEM and returns.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "dash_common.cuh"
#include "dash_internal.h"

#ifndef DASH_STAGED_EPILOGUE
#define DASH_STAGED_EPILOGUE 1  // build-time: 0 stores every output directly
#endif
#ifndef DASH_KPS
#define DASH_KPS 2  // k-blocks per pipeline stage of the 16-bit and TF32 pair kernels
#endif
#ifndef DASH_ACC_KPS
#define DASH_ACC_KPS 1  // k-blocks per pipeline stage of the accurate 3xTF32 pair kernel
#endif
#ifndef DASH_DYN_SCHED
#define DASH_DYN_SCHED 1  // build-time: 0 gives the pair kernels the fixed round-robin order
#endif

namespace dash {

int gemm_read_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_dash_error, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_dash_error, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

// KT: 0 = 16-bit operands (kind::f16), 1 = TF32, 2 = 3xTF32, 3 = 16-bit A and a
//     16-bit pair B (FMT_F16X2 / FMT_BF16X2): A B_lo, then A B_hi, per K slice
//     into the same accumulator.
// MODE: 0 = one CTA per 128 x BN tile;
//       2 = CTA pairs running one 256 x BN MMA (cta_group::2): each CTA stages
//           its own 128 rows of A and half of B, the even CTA issues the MMA and
//           both CTAs hold 128 rows of the accumulator.
// Every CTA loads its own operand tiles; no load is shared between CTAs.
template <int BN, int KT, int MODE>
struct Cfg {
  static_assert(MODE == 0 || MODE == 2, "MODE is 0 (single CTA) or 2 (CTA pair)");
  static constexpr int CL = MODE ? 2 : 1;       // CTAs per cluster
  static constexpr int BM = 128;                // accumulator rows per CTA
  static constexpr bool H16 = (KT == 0 || KT == 3);  // 16-bit operands (kind::f16)
  static constexpr int EB = H16 ? 2 : 4;        // operand element bytes
  static constexpr int BK = 128 / EB;           // elements per 128-byte row
  static constexpr int UK = H16 ? 16 : 8;       // K of one MMA
  static constexpr int NSUB = BK / UK;          // MMAs per k-block
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_ROWS = (MODE == 2) ? BN / 2 : BN;  // B rows staged per CTA
  static constexpr int B_BYTES = B_ROWS * 128;
  // Operand parts staged per k-block: hi and lo of both operands for 3xTF32, of
  // B alone for KT 3.  Stage layout: A | B | A_lo | B_lo (3xTF32), A | B | B_lo (KT 3).
  static constexpr int NPART_A = (KT == 2) ? 2 : 1;
  static constexpr int NPART_B = (KT == 2 || KT == 3) ? 2 : 1;
  static constexpr int NPART = NPART_B;
  static constexpr int LO_A = A_BYTES + B_BYTES;                     // A_lo after sA
  static constexpr int LO_B = (KT == 2) ? A_BYTES + B_BYTES : B_BYTES;  // B_lo after sB
  // K-blocks per stage.  The 16-bit and TF32 pair kernels take two per barrier round
  // trip (three 64 KB stages instead of six of 32 KB): the MMA warp then waits,
  // issues and commits once per eight MMAs instead of four.  Measured on CN FP16
  // (1024^2 blocks): 13% fewer cycles per tile, 3% less wall time under the power cap.
  static constexpr int KPS =
      (MODE == 2 && (KT == 0 || KT == 1)) ? DASH_KPS : ((MODE == 2 && KT == 2) ? DASH_ACC_KPS : 1);
  static constexpr int SUB_BYTES = A_BYTES * NPART_A + B_BYTES * NPART_B;  // one k-block
  static constexpr int STAGE_BYTES = KPS * SUB_BYTES;
  // Bytes the barrier owner waits for per stage (both CTAs' loads for a pair).
  static constexpr int EXPECT_BYTES = (MODE == 2 ? 2 : 1) * STAGE_BYTES;
  // fp16/bf16-operand kernels stage 16-bit output tiles through shared memory
  // (4 KB per epilogue warp) so that global stores cover whole rows.
  static constexpr int EPI_WARP_BYTES = 4096;
  static constexpr int EPI_BYTES = (H16 && DASH_STAGED_EPILOGUE) ? 8 * EPI_WARP_BYTES : 0;
  static constexpr int STAGES_RAW = (224 * 1024 - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int MMA_M = (MODE == 2) ? 256 : 128;
  static constexpr int MN_ATOM = 128 / EB;      // elements in one 128-byte MN row
  static constexpr int A_BOXES_MN = BM / MN_ATOM;
  static constexpr int B_BOXES_MN = B_ROWS / MN_ATOM;  // MN-major boxes of B per CTA tile
  static constexpr int MN_BOX_BYTES = BK * 128;  // one MN-major box: BK rows of 128 B
  // MN-major 32-bit operands are read with 32-byte swizzle atoms; that layout
  // groups K in slabs of 4 rows (512 B), the 16-byte-atom layout in slabs of 8.
  static constexpr uint32_t MN_LAYOUT = H16 ? LAYOUT_SW128 : LAYOUT_SW128_BASE32;
  static constexpr uint32_t MN_SBO = H16 ? 1024 : 512;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES + EPI_BYTES;
  static_assert(STAGES >= 2, "need at least two pipeline stages");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct KParams {
  CUtensorMap tO[2];  // 16-bit outputs of the staged epilogue (TMA store maps)
  // Symmetric operands (sym_in): the other-major views of A and B, used for the
  // k-blocks that lie in the unstored lower triangle (A(m,k) = A(k,m)).
  CUtensorMap tAm, tBm;
  CUtensorMap tAlm, tBlm;  // the same for the lo parts of 3xTF32 operands
  int dim;
  int tiles_m, tiles_n;
  long long total_tiles;
  long long total_units;  // tiles / cluster size: one unit per cluster step
  int nkb;
  uint32_t idesc;
  int a_mn, b_mn;
  int staged;  // all outputs 16-bit (at most two): tiles leave through TMA stores
  // Symmetric-half iterates (CTA pairs only).  sym_in / sym_in_b: A / B is
  // symmetric and only its 256 x 256 tiles on or above the diagonal are read.
  // sym_out: only those tiles of C are computed and written (C symmetric by
  // construction).  sym_any = sym_in | sym_in_b.
  int sym_in, sym_in_b, sym_out, sym_any;
  int t256;         // dim / 256
  uint32_t idesc0;  // instruction descriptor without the operand-major bits
  // Run-time tile order (CTA-pair kernels): this launch's counter, whose high word
  // is the launch's tag sched_id and low word the units drawn so far; nullptr for
  // the fixed order cid, cid + ncl, ...
  unsigned long long* sched;
  uint32_t sched_id;
  EpiParams epi;
};

// The next unit of a launch from its tile counter *w: (sched_id << 32) + units
// handed out; t is the value an atomicAdd(w, 1) returned (issued earlier, so that
// its latency overlaps other work).  A counter tagged by an earlier launch, or
// untagged (0), is re-tagged, the caller taking unit 0.  A counter tagged by a later
// launch means two launches overlap on it: `conflict` is set and -1 returned.
// Returns -1 too once every unit is handed out.  Each of the launch's `parts`
// drawers (CTA pairs) stops at its first index past the end, so the one that draws
// total + parts - 1 is the last to touch the counter: it clears the tag, and a
// replay of the same launch (a captured graph, same tag) starts afresh.
__device__ __forceinline__ long long resolve_unit(unsigned long long* w, uint32_t id,
                                                  long long total, long long parts,
                                                  unsigned long long t, bool& conflict) {
  for (int n = 0; n < 1024; ++n) {
    if (n > 0) t = atomicAdd(w, 1ull);
    uint32_t hi = static_cast<uint32_t>(t >> 32);
    if (hi == id) {
      const long long u = static_cast<long long>(t & 0xffffffffull);
      if (u < total) return u;
      if (u == total + parts - 1) {
        const unsigned long long fin =
            (static_cast<unsigned long long>(id) << 32) | static_cast<unsigned long long>(total + parts);
        atomicCAS(w, fin, 0ull);
      }
      return -1;
    }
    unsigned long long cur = t + 1ull;
    for (int m = 0; m < 1024; ++m) {
      hi = static_cast<uint32_t>(cur >> 32);
      if (hi == id) break;  // re-tagged by another pair: draw again
      if (hi != 0u && static_cast<int32_t>(hi - id) > 0) {
        conflict = true;
        return -1;
      }
      const unsigned long long tagged = (static_cast<unsigned long long>(id) << 32) | 1ull;
      const unsigned long long prev = atomicCAS(w, cur, tagged);
      if (prev == cur) {
        if (total > 0) return 0;
        if (parts == 1) atomicCAS(w, tagged, 0ull);  // that was the launch's only draw
        return -1;
      }
      cur = prev;
    }
    if (static_cast<uint32_t>(cur >> 32) != id) break;
  }
  conflict = true;
  return -1;
}

// 64-bit store into shared memory of a CTA of the cluster (shared::cluster address)
// that completes 8 bytes of transaction count on that CTA's mbarrier `bar`.
__device__ __forceinline__ void st_async_b64(uint32_t addr, long long v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(
                   addr),
               "l"(v), "r"(bar)
               : "memory");
}

// A unit is the group of CL tiles one cluster computes together: the CTAs of a
// cluster take adjacent 128-row M tiles that share one BN-wide N tile.
template <int CL>
__device__ __forceinline__ void decode_unit(long long u, const KParams& p, uint32_t crank,
                                            long long& blk, int& m0, int& n0, int bn) {
  if (p.sym_out) {
    // 256 x 256 tiles (mt, nt) with nt >= mt, row by row: T(T+1)/2 per block, each
    // split into 256 / bn column tiles of width bn.
    const int T = p.t256;
    const int nh = 256 / bn;
    const long long per = static_cast<long long>(T) * (T + 1) / 2 * nh;
    blk = u / per;
    int t = static_cast<int>(u - blk * per);
    const int h = t % nh;
    t /= nh;
    int mt = 0;
    while (t >= T - mt) {
      t -= T - mt;
      ++mt;
    }
    m0 = mt * 256 + static_cast<int>(crank) * 128;
    n0 = (mt + t) * 256 + h * bn;
    return;
  }
  const long long per = static_cast<long long>(p.tiles_m / CL) * p.tiles_n;
  blk = u / per;
  const int r = static_cast<int>(u - blk * per);
  m0 = ((r / p.tiles_n) * CL + static_cast<int>(crank)) * 128;
  n0 = (r % p.tiles_n) * bn;
}

// Per-tile constants of the epilogue, read once per tile: the per-block output
// multipliers and the valid size of a padded block.  (Read inside the chunk loop
// they would be reloaded after every store, which may alias them.)
struct TileEpi {
  float m[3];
  int pv;
  uint32_t plain;  // bit o: output o is the accumulator itself (D = C)
};

__device__ __forceinline__ TileEpi tile_epi(const EpiParams& e, long long blk) {
  TileEpi t;
  t.plain = 0u;
#pragma unroll
  for (int o = 0; o < 3; ++o) {
    t.m[o] = (o < e.nout && e.out[o].mult != nullptr) ? e.out[o].mult[blk] : 1.0f;
    if (o < e.nout) {
      const EpiOut& O = e.out[o];
      if (O.alpha == 1.0f && O.gamma == 0.0f && (O.eps == 0.0f || e.E_hi == nullptr) &&
          t.m[o] == 1.0f && e.pad_valid == nullptr)
        t.plain |= 1u << o;
    }
  }
  t.pv = (e.pad_valid != nullptr) ? e.pad_valid[blk] : 0x7fffffff;
  return t;
}

// Residual term and E operand for 16 consecutive columns of one row.  E reads are
// 256-bit when the base pointers allow it, 128-bit otherwise.
__device__ __forceinline__ void epi_pre16(const EpiParams& e, int rg, int cg0, long long idx,
                                          const float (&c)[16], float& rsum, bool diag,
                                          float (&ev)[16]) {
  // diag: this warp's rows and these 16 columns share a diagonal element (a
  // warp-uniform flag: off-diagonal chunks skip every identity term).
  if (e.E_hi != nullptr) {
    if (aligned32(e.E_hi) && (e.E_fmt != FMT_SPLIT || aligned32(e.E_lo))) {
      load16_v8(e.E_fmt, e.E_hi, e.E_lo, idx, ev);
    } else {
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float t[4];
        load4(e.E_fmt, e.E_hi, e.E_lo, idx + 4 * g, t);
#pragma unroll
        for (int j = 0; j < 4; ++j) ev[4 * g + j] = t[j];
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) ev[j] = 0.0f;
  }
  if (e.resid_acc != nullptr) {
    // Residual of the iterate: C itself, or C + E when the iterate is stored as its
    // deviation from a matrix the epilogue adds (E).
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = e.resid_plus_e ? c[j] + ev[j] : c[j];
    if (diag) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float d = x[j] - ((rg == cg0 + j) ? 1.0f : 0.0f);
        rsum = fmaf(d, d, rsum);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) rsum = fmaf(x[j], x[j], rsum);
    }
  }
}

// Output o's values D = mult (alpha C + gamma I + eps E), identity outside the
// valid part of a padded block.
__device__ __forceinline__ void epi_out16(const EpiParams& e, const TileEpi& te, int o, int rg,
                                          int cg0, const float (&c)[16], const float (&ev)[16],
                                          bool diag, float (&d)[16]) {
  const EpiOut& O = e.out[o];
  const float m = te.m[o];
  if ((te.plain >> o) & 1u) {
    // alpha 1, no gamma, E or multiplier: the products' sum as it stands.
#pragma unroll
    for (int j = 0; j < 16; ++j) d[j] = c[j];
    return;
  }
  if (!diag && e.pad_valid == nullptr) {
#pragma unroll
    for (int j = 0; j < 16; ++j) d[j] = m * fmaf(O.alpha, c[j], O.eps * ev[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int col = cg0 + j;
      float v = fmaf(O.alpha, c[j], O.eps * ev[j]);
      if (rg == col) v += O.gamma;
      v *= m;
      if (rg >= te.pv || col >= te.pv) v = (rg == col) ? 1.0f : 0.0f;
      d[j] = v;
    }
  }
}

// Epilogue for 16 consecutive columns of one row, stored straight to global
// memory (256-bit stores when the base pointers allow it, 128-bit otherwise).
// mir: the tile lies above the diagonal of a symmetric output, and element
// (rg, cg0 + j) is also written to (cg0 + j, rg) for outputs flagged mirror.  The
// lanes of a warp hold consecutive rows, so each of these stores covers 128
// contiguous bytes of a row of the mirrored tile.
__device__ __forceinline__ void epilogue16f(const EpiParams& e, const TileEpi& te, int rg,
                                            int cg0, long long idx, const float (&c)[16],
                                            float& rsum, bool diag, bool mir, int dim) {
  float ev[16];
  epi_pre16(e, rg, cg0, idx, c, rsum, diag, ev);
#pragma unroll
  for (int o = 0; o < 3; ++o) {
    if (o < e.nout) {
      const EpiOut& O = e.out[o];
      float d[16];
      epi_out16(e, te, o, rg, cg0, c, ev, diag, d);
      if (aligned32(O.hi) && (O.fmt != FMT_SPLIT || aligned32(O.lo))) {
        store16_v8(O.fmt, O.hi, O.lo, idx, d);
      } else {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float q[4] = {d[4 * g], d[4 * g + 1], d[4 * g + 2], d[4 * g + 3]};
          store4(O.fmt, O.hi, O.lo, idx + 4 * g, q);
        }
      }
      if (mir && O.mirror && (O.fmt == FMT_F32 || O.fmt == FMT_TF32)) {
        // idx = blk dim^2 + rg dim + cg0  ->  blk dim^2 + cg0 dim + rg
        float* mp = static_cast<float*>(O.hi) + (idx - cg0 + rg) +
                    static_cast<long long>(cg0 - rg) * dim;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          *mp = (O.fmt == FMT_TF32) ? rna_tf32(d[j]) : d[j];
          mp += dim;
        }
      }
    }
  }
}

// Position of 16-byte unit u of staging row r: the TMA store's swizzle (128-byte
// rows: SWIZZLE_128B, unit ^ (r & 7); 64-byte rows: SWIZZLE_64B, unit ^ ((r >> 1)
// & 3)).  Both spread a warp's row-wise writes over all banks.
__device__ __forceinline__ int stage_unit(int u, int r, int U) {
  return (U == 8) ? (u ^ (r & 7)) : (u ^ ((r >> 1) & 3));
}

// Staged variant for 16-bit outputs: chunk jr of the current round is packed and
// written to this thread's row of the warp's staging buffer (per output a box of
// 32 rows x U 16-byte units in the TMA store's swizzled layout).
__device__ __forceinline__ void epilogue16s(const EpiParams& e, const TileEpi& te, int rg,
                                            int cg0, long long idx, const float (&c)[16],
                                            float& rsum, bool diag, uint8_t* wst, int lane,
                                            int jr, int U) {
  float ev[16];
  epi_pre16(e, rg, cg0, idx, c, rsum, diag, ev);
#pragma unroll
  for (int o = 0; o < 2; ++o) {
    if (o < e.nout) {
      float d[16];
      epi_out16(e, te, o, rg, cg0, c, ev, diag, d);
      uint32_t r[8];
      const bool half = (e.out[o].fmt == FMT_F16);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        r[j] = half ? pack_half2(d[2 * j], d[2 * j + 1]) : pack_bf162(d[2 * j], d[2 * j + 1]);
      uint8_t* rowp = wst + o * 32 * U * 16 + lane * U * 16;
      *reinterpret_cast<uint4*>(rowp + (stage_unit(2 * jr, lane, U) << 4)) =
          make_uint4(r[0], r[1], r[2], r[3]);
      *reinterpret_cast<uint4*>(rowp + (stage_unit(2 * jr + 1, lane, U) << 4)) =
          make_uint4(r[4], r[5], r[6], r[7]);
    }
  }
}

// Hands one staged round to the TMA engine: a 32-row box per output at (col0,
// row0) of block blk.  The buffer may be rewritten once the stores have read it.
__device__ __forceinline__ void flush_round_tma(const KParams& p, uint32_t wst_s, int lane, int U,
                                                int row0, long long blk, int col0) {
  fence_async_shared();  // this thread's staging writes -> the TMA engine
  __syncwarp();
  if (lane == 0) {
    for (int o = 0; o < p.epi.nout; ++o)
      tma_store_3d(&p.tO[o], wst_s + o * 32 * U * 16, col0, row0, static_cast<int>(blk));
    bulk_commit_group();
  }
}

__device__ __forceinline__ void epilogue16(const EpiParams& e, const TileEpi& te, int rg,
                                           int cg0, long long idx, const uint32_t (&r)[16],
                                           float& rsum, bool diag, bool mir, int dim) {
  float c[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) c[j] = __uint_as_float(r[j]);
  epilogue16f(e, te, rg, cg0, idx, c, rsum, diag, mir, dim);
}

// Whether rows [r0, r0 + 32) and columns [c0, c0 + 16) contain a diagonal element.
__device__ __forceinline__ bool chunk_on_diag(int r0, int c0) {
  return c0 < r0 + 32 && r0 < c0 + 16;
}

// Instances with the second (B) producer thread, warp 10: the pair kernels whose
// tile order is fixed (the run-time order's ring is read by one producer only).
template <int MODE, bool MIR>
constexpr bool gemm_split() {
  return MODE == 2 && !(MIR && DASH_DYN_SCHED != 0);
}
template <int MODE, bool MIR>
constexpr int gemm_threads() {
  return gemm_split<MODE, MIR>() ? 352 : 320;
}

template <int BN, int KT, int MODE, bool MIR>
__global__ void __launch_bounds__(gemm_threads<MODE, MIR>(), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                   const __grid_constant__ CUtensorMap tAl,
                   const __grid_constant__ CUtensorMap tBl, const __grid_constant__ KParams p) {
  using C = Cfg<BN, KT, MODE>;
  constexpr int CL = C::CL;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;

  // Layout: stages | epilogue staging (1024-aligned) | barriers.
  uint8_t* bar_area = smem + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES;
  const uint32_t bar0 = sbase + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES;
  // barrier addresses
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
  const uint32_t fin_bar = bar0 + 8u * (2 * C::STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * (2 * C::STAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * (2 * C::STAGES + 5) + 8);
  // Ring of the run-time tile order (CTA pairs).  Pair c's first unit is c; its
  // unit of iteration it >= 1 is drawn from the counter (indices past the first
  // ncl units) and sits in ring slot (it - 1) % RING, with a "full" barrier in
  // both CTAs.  The leader's producer writes it once it has issued the first stage
  // of unit it - 1.  A slot is rewritten RING units later, and by then every reader
  // has moved on: when the leader's producer issues a stage of unit it, the MMA has
  // consumed unit it - 4 or later (at most 8 stages in flight, at least 2 per unit),
  // which needed both CTAs' loads of it - 4 and the epilogues' release of the
  // accumulator of it - 6; each of those roles reads a unit's slot before working on
  // it, and RING exceeds 6.
  constexpr int RING = 8;
  static_assert(C::STAGES <= 8, "the ring's slack assumes at most 8 stages");
  constexpr uint32_t ring_off = 8u * (2 * C::STAGES + 5) + 16u;
  static_assert(ring_off + 16u * RING <= static_cast<uint32_t>(C::BAR_BYTES), "barrier area");
  volatile long long* ring_u = reinterpret_cast<volatile long long*>(bar_area + ring_off);
  const uint32_t ring_u0 = bar0 + ring_off;
  auto rfull_bar = [&](int r) { return bar0 + ring_off + 8u * (RING + r); };
  // Compiled into the mirrored-store instances only (the fp32 products with
  // direct stores); the other instances keep the fixed order and the code of it.
  constexpr bool DYN = MIR && (MODE == 2) && (DASH_DYN_SCHED != 0);
  const bool dyn = DYN && (p.sched != nullptr);
  constexpr bool SPLIT = gemm_split<MODE, MIR>();
  constexpr int EXP_A = (MODE == 2 ? 2 : 1) * C::KPS * C::A_BYTES * C::NPART_A;
  constexpr int EXP_B = (MODE == 2 ? 2 : 1) * C::KPS * C::B_BYTES * C::NPART_B;
  static_assert(!SPLIT || EXP_A + EXP_B == C::EXPECT_BYTES, "split of the stage bytes");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Cluster of CL CTAs: rank within the cluster, cluster index and count.
  const uint32_t crank = (CL > 1) ? cluster_ctarank() : 0u;
  const bool leader = (crank == 0);  // in MODE 2 the leader issues the pair's MMAs
  const long long cid = blockIdx.x / CL;
  const long long ncl = gridDim.x / CL;
  constexpr uint16_t kMask = (1u << CL) - 1u;

  // Unit of iteration it >= 1 of this pair in the run-time order: the leader's
  // producer draws it (publish, from a counter value drawn one unit earlier) into
  // both CTAs' rings; the other roles read it (take).  The peer's copy arrives by
  // st.async, which completes on the peer's barrier; the peer's producer arms that
  // barrier for the 8 bytes (arm).  A unit of -1 ends the loops.
  auto publish = [&](long long it, unsigned long long t, long long& u) {
    const int r = static_cast<int>((it - 1) % RING);
    bool conflict = false;
    const long long d = resolve_unit(p.sched, p.sched_id, p.total_units - ncl, ncl, t, conflict);
    if (conflict) atomicExch(&g_dash_error, DEV_ERR_CONFLICT);
    u = d < 0 ? -1 : ncl + d;
    ring_u[r] = u;
    mbar_arrive(rfull_bar(r));
    st_async_b64(mapa_shared(ring_u0 + 8u * static_cast<uint32_t>(r), crank | 1u), u,
                 mapa_shared(rfull_bar(r), crank | 1u));
  };
  auto take = [&](long long it, bool arm, long long& u) -> bool {
    const int r = static_cast<int>((it - 1) % RING);
    if (arm) mbar_arrive_expect_tx(rfull_bar(r), 8u);
    if (!mbar_wait(rfull_bar(r), static_cast<uint32_t>(((it - 1) / RING) & 1), abort_flag))
      return false;
    u = ring_u[r];
    return true;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), SPLIT ? 2 : 1);
      // Released by the MMA warp (in a pair, the leader's).
      mbar_init(empty_bar(s), 1);
    }
    // One arrival per use: the leader's producer (leader), the peer's producer
    // arming it for the st.async (peer).
    for (int r = 0; r < RING; ++r) mbar_init(rfull_bar(r), 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      // Eight epilogue warps per CTA; in MODE 2 the leader's accumulator is freed
      // by the epilogues of both CTAs.
      mbar_init(tempty_bar(a), MODE == 2 ? 16 : 8);
    }
    mbar_init(fin_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tA);
    tma_prefetch_desc(&tB);
    if (C::NPART_A == 2) tma_prefetch_desc(&tAl);
    if (C::NPART_B == 2) tma_prefetch_desc(&tBl);
  }
  if (warp == 1) {
    if (MODE == 2)
      tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    else
      tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  }
  tc_fence_before();
  // Barriers must be initialised in every CTA before any peer signals into it.
  if (CL > 1)
    cluster_sync();
  else
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
      // Pair kernels: the boxes of this CTA's part of the tile at (vm0, vn0) of
      // block vz (A rows, its half of B), per k-block and operand part, handed to
      // `op` with the map and the coordinates the loads use (the other-major view
      // for a mirrored k-block).
      auto for_boxes = [&](int vz, int vm0, int vn0, int kb, int part, auto&& op) {
        const int k0 = kb * C::BK;
        const bool amir = p.sym_in && (k0 >> 8) < (vm0 >> 8);
        const bool bmir = p.sym_in_b && (k0 >> 8) > (vn0 >> 8);
        const CUtensorMap* ma = amir ? &p.tAm : (part ? &tAl : &tA);
        const CUtensorMap* mb = bmir ? (part ? &p.tBlm : &p.tBm) : (part ? &tBl : &tB);
        if (part < C::NPART_A) {
          if (!(p.a_mn ^ amir)) {
            op(ma, 0, 0, k0, vm0, vz);
          } else {
#pragma unroll
            for (int i = 0; i < C::A_BOXES_MN; ++i)
              op(ma, 0, i * C::MN_BOX_BYTES, vm0 + i * C::MN_ATOM, k0, vz);
          }
        }
        const int nb = vn0 + static_cast<int>(crank) * C::B_ROWS;  // this CTA's half of N
        if (!(p.b_mn ^ bmir)) {
          op(mb, 1, 0, k0, nb, vz);
        } else {
#pragma unroll
          for (int i = 0; i < C::B_BOXES_MN; ++i)
            op(mb, 1, i * C::MN_BOX_BYTES, nb + i * C::MN_ATOM, k0, vz);
        }
      };
      // Leader, run-time order: the unit of the next iteration, published once this
      // iteration's first stage is issued, from a counter draw made one unit earlier,
      // so that neither producer waits for the counter.
      long long u_next = -1;
      unsigned long long pend = 0;
      if (dyn && leader) pend = atomicAdd(p.sched, 1ull);
      for (long long it = 0; ok; ++it) {
        long long u = cid + it * ncl;
        if (dyn && it > 0) {
          if (leader) {
            u = u_next;
          } else if (!take(it, true, u)) {
            ok = false;
            break;
          }
          if (u < 0) break;
        } else if (!dyn && u >= p.total_units) {
          break;
        }
        long long blk;
        int m0, n0;
        decode_unit<CL>(u, p, crank, blk, m0, n0, BN);
        const int z = static_cast<int>(blk);
        for (int kb0 = 0; kb0 < p.nkb; kb0 += C::KPS) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint32_t fb = full_bar(stage);
          if (MODE != 2 || leader) {
            mbar_arrive_expect_tx(fb, SPLIT ? EXP_A : C::EXPECT_BYTES);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          }
          // In a pair, every load is counted on the leader's barrier.
          if (MODE == 2) fb = leader ? fb : mapa_shared(fb, crank & ~1u);
          for (int j = 0; j < C::KPS; ++j)
          for (int part = 0; part < C::NPART_B; ++part) {
            const int kb = kb0 + j;
            const int k0 = kb * C::BK;
            const uint32_t s0 = sbase + stage * C::STAGE_BYTES + j * C::SUB_BYTES;
            const uint32_t sA = s0 + part * C::LO_A;
            const uint32_t sB = s0 + C::A_BYTES + part * C::LO_B;
            const bool loadA = part < C::NPART_A;  // KT 3 has one A part
            const CUtensorMap* ma = part ? &tAl : &tA;
            const CUtensorMap* mb = part ? &tBl : &tB;
            if (MODE == 2) {
              // Symmetric operands: a k-block left of A's (below B's) diagonal tile is
              // read as the transpose of the stored tile, i.e. in the other major.
              for_boxes(z, m0, n0, kb, part, [&](const CUtensorMap* m, int isB, int off, int x,
                                                 int y, int zz) {
                if (SPLIT && isB) return;
                tma_load_3d_pair((isB ? sB : sA) + off, m, fb, x, y, zz);
              });
              continue;
            }
            if (!loadA) {
            } else if (!p.a_mn) {
              tma_load_3d(sA, ma, fb, k0, m0, z);
            } else {
#pragma unroll
              for (int i = 0; i < C::A_BOXES_MN; ++i)
                tma_load_3d(sA + i * C::MN_BOX_BYTES, ma, fb, m0 + i * C::MN_ATOM, k0, z);
            }
            if (!p.b_mn) {
              tma_load_3d(sB, mb, fb, k0, n0, z);
            } else {
#pragma unroll
              for (int i = 0; i < C::B_BOXES_MN; ++i)
                tma_load_3d(sB + i * C::MN_BOX_BYTES, mb, fb, n0 + i * C::MN_ATOM, k0, z);
            }
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (dyn && leader && kb0 == 0) {
            // The next iteration's unit, once this unit's first stage is on its way:
            // the peer's producer and the other roles find it well before they need it.
            publish(it + 1, pend, u_next);
            if (u_next >= 0) pend = atomicAdd(p.sched, 1ull);
          }
        }
      }
      if (!ok) {
        // Wait for the copies this CTA's barriers count so none lands after exit.
        for (int s = 0; s < C::STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && (MODE != 2 || leader)) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (long long it = 0; ok; ++it) {
        long long u = cid + it * ncl;
        if (dyn && it > 0) {
          if (!take(it, false, u)) {
            ok = false;
            break;
          }
          if (u < 0) break;
        } else if (!dyn && u >= p.total_units) {
          break;
        }
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // The pair tile's position, for the operand-major choice of symmetric operands.
        long long ublk;
        int um0 = 0, un0 = 0;
        if (p.sym_any) decode_unit<CL>(u, p, 0u, ublk, um0, un0, BN);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb0 = 0; kb0 < p.nkb; kb0 += C::KPS) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int j = 0; j < C::KPS; ++j) {
          const int kb = kb0 + j;
          const uint32_t sA = sbase + stage * C::STAGE_BYTES + j * C::SUB_BYTES;
          const uint32_t sB = sA + C::A_BYTES;
          const int k0 = kb * C::BK;
          const int amn = p.a_mn ^ ((p.sym_in && (k0 >> 8) < (um0 >> 8)) ? 1 : 0);
          const int bmn = p.b_mn ^ ((p.sym_in_b && (k0 >> 8) > (un0 >> 8)) ? 1 : 0);
          const uint32_t idesc =
              p.sym_any ? (p.idesc0 | (static_cast<uint32_t>(amn) << 15) |
                          (static_cast<uint32_t>(bmn) << 16))
                       : p.idesc;
#pragma unroll
          for (int kk = 0; kk < C::NSUB; ++kk) {
            const uint64_t da =
                amn ? smem_desc(sA + kk * C::UK * 128, C::MN_BOX_BYTES, C::MN_SBO, C::MN_LAYOUT)
                    : smem_desc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t db =
                bmn ? smem_desc(sB + kk * C::UK * 128, C::MN_BOX_BYTES, C::MN_SBO, C::MN_LAYOUT)
                    : smem_desc_sw128(sB + kk * 32, 16, 1024);
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            uint64_t dal = 0, dbl = 0;
            if (C::NPART_A == 2)
              dal = amn ? smem_desc(sA + C::LO_A + kk * C::UK * 128, C::MN_BOX_BYTES, C::MN_SBO,
                                    C::MN_LAYOUT)
                        : smem_desc_sw128(sA + C::LO_A + kk * 32, 16, 1024);
            if (C::NPART_B == 2)
              dbl = bmn ? smem_desc(sB + C::LO_B + kk * C::UK * 128, C::MN_BOX_BYTES, C::MN_SBO,
                                    C::MN_LAYOUT)
                        : smem_desc_sw128(sB + C::LO_B + kk * 32, 16, 1024);
            if (MODE == 2) {
              if (KT == 0) {
                mma_f16_pair(d_tmem, da, db, idesc, accum);
              } else if (KT == 3) {
                // The small part first, then the large one, into the same sum.
                mma_f16_pair(d_tmem, da, dbl, idesc, accum);
                mma_f16_pair(d_tmem, da, db, idesc, 1u);
              } else if (KT == 1) {
                mma_tf32_pair(d_tmem, da, db, idesc, accum);
              } else {
                mma_tf32_pair(d_tmem, dal, db, idesc, accum);
                mma_tf32_pair(d_tmem, da, dbl, idesc, 1u);
                mma_tf32_pair(d_tmem, da, db, idesc, 1u);
              }
            } else {
              if (KT == 0) {
                mma_f16(d_tmem, da, db, p.idesc, accum);
              } else if (KT == 3) {
                mma_f16(d_tmem, da, dbl, p.idesc, accum);
                mma_f16(d_tmem, da, db, p.idesc, 1u);
              } else if (KT == 1) {
                mma_tf32(d_tmem, da, db, p.idesc, accum);
              } else {
                mma_tf32(d_tmem, dal, db, p.idesc, accum);
                mma_tf32(d_tmem, da, dbl, p.idesc, 1u);
                mma_tf32(d_tmem, da, db, p.idesc, 1u);
              }
            }
          }
          }  // k-blocks of the stage
          // The stage is free once every CTA whose shared memory fed it is done.
          if (MODE == 2)
            mma_commit_pair_mc(empty_bar(stage), kMask);
          else
            mma_commit(empty_bar(stage));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (MODE == 2)
          mma_commit_pair_mc(tfull_bar(acc), kMask);  // both CTAs hold half the rows
        else
          mma_commit(tfull_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA issued above must be complete before TMEM is released.
      if (MODE == 2)
        mma_commit_pair(fin_bar);
      else
        mma_commit(fin_bar);
      mbar_wait_drain(fin_bar, 0);
    }
  } else if (SPLIT && warp == 10) {
    if (lane == 0) {
      // ---------------------------------------------------------- B producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (long long u = cid; ok && u < p.total_units; u += ncl) {
        long long blk;
        int m0, n0;
        decode_unit<CL>(u, p, crank, blk, m0, n0, BN);
        const int z = static_cast<int>(blk);
        for (int kb0 = 0; kb0 < p.nkb; kb0 += C::KPS) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint32_t fb = full_bar(stage);
          if (leader) {
            mbar_arrive_expect_tx(fb, EXP_B);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          }
          fb = leader ? fb : mapa_shared(fb, crank & ~1u);
          for (int j = 0; j < C::KPS; ++j)
          for (int part = 0; part < C::NPART_B; ++part) {
            const int kb = kb0 + j;
            const int k0 = kb * C::BK;
            const uint32_t s0 = sbase + stage * C::STAGE_BYTES + j * C::SUB_BYTES;
            const uint32_t sB = s0 + C::A_BYTES + part * C::LO_B;
            const bool bmir = p.sym_in_b && (k0 >> 8) > (n0 >> 8);
            const CUtensorMap* mb = bmir ? (part ? &p.tBlm : &p.tBm) : (part ? &tBl : &tB);
            const int nb = n0 + static_cast<int>(crank) * C::B_ROWS;
            if (!(p.b_mn ^ bmir)) {
              tma_load_3d_pair(sB, mb, fb, k0, nb, z);
            } else {
#pragma unroll
              for (int i = 0; i < C::B_BOXES_MN; ++i)
                tma_load_3d_pair(sB + i * C::MN_BOX_BYTES, mb, fb, nb + i * C::MN_ATOM, k0, z);
            }
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < C::STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // Eight warps: two per TMEM lane quarter, each owning half of the columns.
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;
    constexpr int HALF = BN / 2;
    uint8_t* wst = smem + C::STAGES * C::STAGE_BYTES + (warp - 2) * C::EPI_WARP_BYTES;
    const uint32_t wst_s = sbase + C::STAGES * C::STAGE_BYTES + (warp - 2) * C::EPI_WARP_BYTES;
    const int row = q * 32 + lane;
    const long long dd = static_cast<long long>(p.dim) * p.dim;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (long long it = 0;; ++it) {
      long long u = cid + it * ncl;
      if (dyn && it > 0) {
        // Lane 0 reads the unit and hands it to the warp.
        long long uu = 0;
        int got = 1;
        if (lane == 0) got = take(it, false, uu) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        uu = __shfl_sync(0xffffffffu, uu, 0);
        if (!got || uu < 0) break;
        u = uu;
      } else if (!dyn && u >= p.total_units) {
        break;
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) break;
      tc_fence_after();
      long long blk;
      int m0, n0;
      decode_unit<CL>(u, p, crank, blk, m0, n0, BN);
      const int rg = m0 + row;
      const int r0w = m0 + q * 32;  // first row of this warp
      const int nh = n0 + h * HALF;
      const long long rbase = blk * dd + static_cast<long long>(rg) * p.dim;
      const TileEpi te = tile_epi(p.epi, blk);
      float rsum = 0.0f;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * BN + h * HALF);
      // Two register sets: the TMEM load of chunk c+1 is in flight while chunk c
      // is processed.
      uint32_t ra[16], rb[16];
      tmem_ld16(taddr, ra);
      if (p.staged) {
        // Rounds of R chunks: 64 columns for one output, 32 for two (4 KB).
        const int R = (p.epi.nout == 1) ? 4 : 2;
        const int U = 2 * R;
#pragma unroll 1
        for (int c = 0; c < HALF / 16; c += 2) {
          tmem_wait_ld(ra);
          tmem_ld16(taddr + (c + 1) * 16, rb);
          const int ca = nh + c * 16, cb = ca + 16;
          if (c % R == 0) {
            // The previous round's stores must have read the buffer.
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
          }
          float fa[16], fb[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) fa[j] = __uint_as_float(ra[j]);
          epilogue16s(p.epi, te, rg, ca, rbase + ca, fa, rsum, chunk_on_diag(r0w, ca), wst, lane,
                      c % R, U);
          tmem_wait_ld(rb);
          if (c + 2 < HALF / 16) tmem_ld16(taddr + (c + 2) * 16, ra);
#pragma unroll
          for (int j = 0; j < 16; ++j) fb[j] = __uint_as_float(rb[j]);
          epilogue16s(p.epi, te, rg, cb, rbase + cb, fb, rsum, chunk_on_diag(r0w, cb), wst, lane,
                      (c + 1) % R, U);
          if ((c + 2) % R == 0)
            flush_round_tma(p, wst_s, lane, U, r0w, blk, nh + (c + 2 - R) * 16);
        }
      } else {
        // A computed tile above the diagonal of a symmetric output: also stored
        // transposed into its mirror (outputs flagged mirror).
        // (Compiled only into the MIR instances, so the others keep their registers.)
        const bool mir = MIR && p.sym_out && (m0 >> 8) != (n0 >> 8);
#pragma unroll 1
        for (int c = 0; c < HALF / 16; c += 2) {
          tmem_wait_ld(ra);
          tmem_ld16(taddr + (c + 1) * 16, rb);
          const int ca = nh + c * 16, cb = ca + 16;
          epilogue16(p.epi, te, rg, ca, rbase + ca, ra, rsum, chunk_on_diag(r0w, ca), mir, p.dim);
          tmem_wait_ld(rb);
          if (c + 2 < HALF / 16) tmem_ld16(taddr + (c + 2) * 16, ra);
          epilogue16(p.epi, te, rg, cb, rbase + cb, rb, rsum, chunk_on_diag(r0w, cb), mir, p.dim);
        }
      }
      if (p.epi.resid_acc != nullptr) {
        // A symmetric output stores one of each mirrored pair of off-diagonal tiles.
        if (p.sym_out && (m0 >> 8) != (n0 >> 8)) rsum *= 2.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, off);
        if (lane == 0) atomicAdd(p.epi.resid_acc + blk * p.epi.resid_stride, rsum);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (MODE == 2)
          mbar_arrive_remote(mapa_shared(tempty_bar(acc), crank & ~1u));
        else
          mbar_arrive(tempty_bar(acc));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // Staged tiles: every TMA store has landed before the CTA exits.
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // No CTA may leave while a peer can still signal into it or use its TMEM.
  if (CL > 1) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (MODE == 2)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- accurate 3xTF32
// The tensor core's fp32 accumulation truncates: every MMA instruction aligns its
// products and the running sum to their largest exponent, drops the bits below
// (toward zero) and rounds the result toward zero.  Over a long K the losses add
// up with one sign, a relative bias of order (K/8) 2^-24, which ill-conditioned
// iterations amplify.  This variant of the pair kernel for 3xTF32 keeps the bias
// at the level of a few instructions: the MMA warp starts a fresh TMEM partial
// accumulator every ACC_SUB sub-steps (one sub-step = the three MMAs of one K = 8
// slice), and eight reducer warps -- two per TMEM lane quarter, 64 columns each --
// add the partials into fp32 registers with round-to-nearest (two columns per
// packed add.rn.f32x2, which halves the reducers' add issue).  Pair tiles are
// 256 x 128, so TMEM holds three partial buffers and a fourth, final buffer: at a
// tile's end the reducers store their sums there and go on with the next tile's
// partials, while four epilogue warps (one per lane quarter) read the final buffer
// and run the fused epilogue.  The MMA therefore never waits for a tile's stores.
#ifndef DASH_ACC_SUB
#define DASH_ACC_SUB 2
#endif
constexpr int ACC_SUB = DASH_ACC_SUB;  // K = 8 sub-steps per TMEM partial
constexpr int ACC_BN = 128;            // pair tile 256 x 128
constexpr int ACC_NPB = 3;             // TMEM partial buffers (3 x 128 columns) + final
constexpr int ACC_REDUCERS = 8;        // reducer warps per CTA
constexpr int ACC_EPI = 4;             // epilogue warps per CTA
constexpr int ACC_THREADS = 32 * (2 + ACC_REDUCERS + ACC_EPI);

template <int KT>
__global__ void __launch_bounds__(ACC_THREADS, 1)
    gemm_tc_acc_kernel(const __grid_constant__ CUtensorMap tA,
                       const __grid_constant__ CUtensorMap tB,
                       const __grid_constant__ CUtensorMap tAl,
                       const __grid_constant__ CUtensorMap tBl, const __grid_constant__ KParams p) {
  constexpr int BN = ACC_BN;
  using C = Cfg<BN, KT, 2>;
  constexpr int CL = 2;
  constexpr int NPB = ACC_NPB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;
  // Layout: stages | epilogue staging (1024-aligned) | barriers.
  uint8_t* bar_area = smem + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES;
  const uint32_t bar0 = sbase + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto pfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto pempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + NPB + a); };
  // The final buffer: filled by this CTA's reducers, emptied by its epilogue warps.
  const uint32_t ffull_bar = bar0 + 8u * (2 * C::STAGES + 2 * NPB);
  const uint32_t fempty_bar = ffull_bar + 8u;
  const uint32_t fin_bar = fempty_bar + 8u;
  constexpr int NBAR = 2 * C::STAGES + 2 * NPB + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * NBAR + 8);
  static_assert(8 * NBAR + 16 <= C::BAR_BYTES, "barrier area");
  constexpr uint32_t TMEM_ACC_COLS = (NPB + 1) * BN;
  static_assert(TMEM_ACC_COLS == 512, "partial and final buffers fill TMEM");
  constexpr uint32_t FINAL_COL = NPB * BN;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = (crank == 0);
  const long long cid = blockIdx.x / CL;
  const long long ncl = gridDim.x / CL;
  constexpr uint16_t kMask = 3;
  const int ngroups = p.nkb * C::NSUB / ACC_SUB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < NPB; ++a) {
      mbar_init(pfull_bar(a), 1);
      mbar_init(pempty_bar(a), 2 * ACC_REDUCERS);  // the reducer warps of both CTAs
    }
    mbar_init(ffull_bar, ACC_REDUCERS);
    mbar_init(fempty_bar, ACC_EPI);
    mbar_init(fin_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tA);
    tma_prefetch_desc(&tB);
    tma_prefetch_desc(&tAl);
    tma_prefetch_desc(&tBl);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), TMEM_ACC_COLS);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (long long u = cid; u < p.total_units && ok; u += ncl) {
        long long blk;
        int m0, n0;
        decode_unit<CL>(u, p, crank, blk, m0, n0, BN);
        const int z = static_cast<int>(blk);
        for (int kb0 = 0; kb0 < p.nkb; kb0 += C::KPS) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint32_t fb = full_bar(stage);
          if (leader) {
            mbar_arrive_expect_tx(fb, C::EXPECT_BYTES);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          }
          fb = leader ? fb : mapa_shared(fb, 0);
          for (int j = 0; j < C::KPS; ++j) {
          const int kb = kb0 + j;
          const int k0 = kb * C::BK;
          const bool amir = p.sym_in && (k0 >> 8) < (m0 >> 8);
          const bool bmir = p.sym_in_b && (k0 >> 8) > (n0 >> 8);
          for (int part = 0; part < C::NPART; ++part) {
            const uint32_t sA = sbase + stage * C::STAGE_BYTES + j * C::SUB_BYTES +
                                part * (C::A_BYTES + C::B_BYTES);
            const uint32_t sB = sA + C::A_BYTES;
            const CUtensorMap* ma = amir ? (part ? &p.tAlm : &p.tAm) : (part ? &tAl : &tA);
            const CUtensorMap* mb = bmir ? (part ? &p.tBlm : &p.tBm) : (part ? &tBl : &tB);
            if (!(p.a_mn ^ amir)) {
              tma_load_3d_pair(sA, ma, fb, k0, m0, z);
            } else {
#pragma unroll
              for (int i = 0; i < C::A_BOXES_MN; ++i)
                tma_load_3d_pair(sA + i * C::MN_BOX_BYTES, ma, fb, m0 + i * C::MN_ATOM, k0, z);
            }
            const int nb = n0 + static_cast<int>(crank) * C::B_ROWS;
            if (!(p.b_mn ^ bmir)) {
              tma_load_3d_pair(sB, mb, fb, k0, nb, z);
            } else {
#pragma unroll
              for (int i = 0; i < C::B_BOXES_MN; ++i)
                tma_load_3d_pair(sB + i * C::MN_BOX_BYTES, mb, fb, nb + i * C::MN_ATOM, k0, z);
            }
          }
          }  // k-blocks of the stage
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < C::STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      long long gidx = 0;  // partials issued so far: buffer gidx % NPB
      int nsub = 0;        // sub-steps issued into the current partial
      uint32_t d_tmem = 0;
      bool ok = true;
      for (long long u = cid; u < p.total_units && ok; u += ncl) {
        long long ublk;
        int um0 = 0, un0 = 0;
        if (p.sym_any) decode_unit<CL>(u, p, 0u, ublk, um0, un0, BN);
        for (int kb0 = 0; kb0 < p.nkb && ok; kb0 += C::KPS) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int j = 0; j < C::KPS && ok; ++j) {
          const int kb = kb0 + j;
          const uint32_t sA = sbase + stage * C::STAGE_BYTES + j * C::SUB_BYTES;
          const uint32_t sB = sA + C::A_BYTES;
          const uint32_t lo_off = C::A_BYTES + C::B_BYTES;
          const int k0 = kb * C::BK;
          const int amn = p.a_mn ^ ((p.sym_in && (k0 >> 8) < (um0 >> 8)) ? 1 : 0);
          const int bmn = p.b_mn ^ ((p.sym_in_b && (k0 >> 8) > (un0 >> 8)) ? 1 : 0);
          const uint32_t idesc =
              p.sym_any ? (p.idesc0 | (static_cast<uint32_t>(amn) << 15) |
                          (static_cast<uint32_t>(bmn) << 16))
                       : p.idesc;
#pragma unroll
          for (int kk = 0; kk < C::NSUB; ++kk) {
            const int buf = static_cast<int>(gidx % NPB);
            if (nsub == 0) {
              const uint32_t par = static_cast<uint32_t>((gidx / NPB) & 1);
              if (!mbar_wait(pempty_bar(buf), par ^ 1u, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
            }
            const uint64_t da =
                amn ? smem_desc(sA + kk * C::UK * 128, C::MN_BOX_BYTES, C::MN_SBO, C::MN_LAYOUT)
                    : smem_desc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t db =
                bmn ? smem_desc(sB + kk * C::UK * 128, C::MN_BOX_BYTES, C::MN_SBO, C::MN_LAYOUT)
                    : smem_desc_sw128(sB + kk * 32, 16, 1024);
            const uint64_t dal =
                amn ? smem_desc(sA + lo_off + kk * C::UK * 128, C::MN_BOX_BYTES, C::MN_SBO,
                                C::MN_LAYOUT)
                    : smem_desc_sw128(sA + lo_off + kk * 32, 16, 1024);
            const uint64_t dbl =
                bmn ? smem_desc(sB + lo_off + kk * C::UK * 128, C::MN_BOX_BYTES, C::MN_SBO,
                                C::MN_LAYOUT)
                    : smem_desc_sw128(sB + lo_off + kk * 32, 16, 1024);
            mma_tf32_pair(d_tmem, dal, db, idesc, nsub ? 1u : 0u);  // fresh partial
            mma_tf32_pair(d_tmem, da, dbl, idesc, 1u);
            mma_tf32_pair(d_tmem, da, db, idesc, 1u);
            if (++nsub == ACC_SUB) {
              mma_commit_pair_mc(pfull_bar(buf), kMask);
              nsub = 0;
              ++gidx;
            }
          }
          }  // k-blocks of the stage
          if (!ok) break;
          mma_commit_pair_mc(empty_bar(stage), kMask);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      mma_commit_pair(fin_bar);
      mbar_wait_drain(fin_bar, 0);
    }
  } else if (warp < 2 + ACC_REDUCERS) {
    // ------------------------------------------------- reducers
    // Warp w: TMEM lane quarter w & 3, column group (w - 2) >> 2 of COLS columns.
    constexpr int COLS = BN / (ACC_REDUCERS / 4);
    const int q = warp & 3;
    const int cq = (warp - 2) >> 2;
    long long gidx = 0;
    uint32_t tcount = 0;
    bool ok = true;
    for (long long u = cid; u < p.total_units && ok; u += ncl, ++tcount) {
      // Running sums as packed fp32 pairs: one add.rn.f32x2 per two columns.
      uint64_t sum[COLS / 2];
#pragma unroll
      for (int j = 0; j < COLS / 2; ++j) sum[j] = 0ull;
      for (int kg = 0; kg < ngroups; ++kg, ++gidx) {
        const int buf = static_cast<int>(gidx % NPB);
        const uint32_t par = static_cast<uint32_t>((gidx / NPB) & 1);
        if (!mbar_wait(pfull_bar(buf), par, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(buf * BN + cq * COLS);
#pragma unroll
        for (int c = 0; c < COLS / 16; c += 2) {
          uint32_t ra[16], rb[16];
          tmem_ld16(taddr + c * 16, ra);
          tmem_ld16(taddr + (c + 1) * 16, rb);
          tmem_wait_ld(ra);
          tmem_fence_regs(rb);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            f32x2_add_rn(sum[c * 8 + j], f32x2_pack(ra[2 * j], ra[2 * j + 1]));
            f32x2_add_rn(sum[(c + 1) * 8 + j], f32x2_pack(rb[2 * j], rb[2 * j + 1]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(pempty_bar(buf), 0));
      }
      if (!ok) break;
      // The tile's sums go to the final buffer once the epilogue warps have read
      // the previous tile's.
      if (!mbar_wait(fempty_bar, (tcount & 1u) ^ 1u, abort_flag)) break;
      tc_fence_after();
      const uint32_t tfin = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(FINAL_COL + cq * COLS);
#pragma unroll
      for (int c = 0; c < COLS / 16; ++c) {
        uint32_t r[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) f32x2_unpack(sum[c * 8 + j], r[2 * j], r[2 * j + 1]);
        tmem_st16(tfin + c * 16, r);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ffull_bar);
    }
  } else {
    // ------------------------------------------------- epilogue
    // Warp w reads its TMEM lane quarter (w & 3) of the final buffer: 32 rows of the
    // CTA tile, all BN columns.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const long long dd = static_cast<long long>(p.dim) * p.dim;
    uint32_t tcount = 0;
    for (long long u = cid; u < p.total_units; u += ncl, ++tcount) {
      if (!mbar_wait(ffull_bar, tcount & 1u, abort_flag)) break;
      tc_fence_after();
      long long blk;
      int m0, n0;
      decode_unit<CL>(u, p, crank, blk, m0, n0, BN);
      const int rg = m0 + row;
      const int r0w = m0 + q * 32;
      const long long rbase = blk * dd + static_cast<long long>(rg) * p.dim;
      const TileEpi te = tile_epi(p.epi, blk);
      const bool mir = p.sym_out && (m0 >> 8) != (n0 >> 8);  // see the plain kernel
      float rsum = 0.0f;
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(FINAL_COL);
      // Off the MMA's critical path: one TMEM load in flight at a time.
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t ra[16];
        tmem_ld16(taddr + c * 16, ra);
        tmem_wait_ld(ra);
        if (c + 1 == BN / 16) {
          // Every load of the final buffer has completed: hand it back.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(fempty_bar);
        }
        const int ca = n0 + c * 16;
        epilogue16(p.epi, te, rg, ca, rbase + ca, ra, rsum, chunk_on_diag(r0w, ca), mir, p.dim);
      }
      if (p.epi.resid_acc != nullptr) {
        if (p.sym_out && (m0 >> 8) != (n0 >> 8)) rsum *= 2.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, off);
        if (lane == 0) atomicAdd(p.epi.resid_acc + blk * p.epi.resid_stride, rsum);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_ACC_COLS);
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Tensor map over a stack of nblocks row-major dim x dim matrices, box
// (box_inner elements along the contiguous axis) x box_outer rows, 128B swizzle.
static bool make_tmap(CUtensorMap* m, const void* base, int esize, int dim, long long nblocks,
                      uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  const CUtensorMapDataType dt =
      esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(dim),
                        static_cast<cuuint64_t>(nblocks)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(dim) * esize,
                           static_cast<cuuint64_t>(dim) * dim * esize};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(m, dt, 3, const_cast<void*>(base), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n;
  }
  return cache[dev];
}

// Tile counters of the run-time order, 4096 per device.  Launch v (v = 1, 2, ...
// in issue order, over all streams) uses counter v mod 4096 and tags it with v; its
// last draw clears the tag (resolve_unit), so the counter needs no reset between
// launches and a captured launch can be replayed.
constexpr int SCHED_SLOTS = 4096;
__device__ unsigned long long g_gemm_sched[SCHED_SLOTS];

static bool sched_slot(unsigned long long** w, uint32_t* id) {
  static std::atomic<unsigned long long*> base[64];
  static std::atomic<uint32_t> seq{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  unsigned long long* b = base[dev].load();
  if (b == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_gemm_sched) != cudaSuccess) return false;
    b = static_cast<unsigned long long*>(ptr);
    base[dev].store(b);
  }
  uint32_t v = seq.fetch_add(1u) + 1u;
  if (v == 0u) v = seq.fetch_add(1u) + 1u;
  *w = b + (v % SCHED_SLOTS);
  *id = v;
  return true;
}

// Kernel entry of a configuration (ACC: the accurate 3xTF32 pair variant).
template <int BN, int KT, int MODE, bool ACC, bool MIR>
struct KernelOf {
  static constexpr int THREADS = ACC ? ACC_THREADS : gemm_threads<MODE, MIR>();
  static auto get() {
    if constexpr (ACC)
      return gemm_tc_acc_kernel<KT>;
    else
      return gemm_tc_kernel<BN, KT, MODE, MIR>;
  }
};

// Largest number of clusters of this kernel that can be resident at once.
template <int BN, int KT, int MODE, bool ACC = false, bool MIR = false>
static int max_active_clusters() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    using C = Cfg<BN, KT, MODE>;
    constexpr int CL = C::CL;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(CL * 256, 1, 1);
    cfg.blockDim = dim3(KernelOf<BN, KT, MODE, ACC, MIR>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, KernelOf<BN, KT, MODE, ACC, MIR>::get(), &cfg) !=
        cudaSuccess)
      n = 0;
    cache[dev] = n > 0 ? n : -1;
  }
  return cache[dev];
}

template <int BN, int KT, int MODE, bool ACC = false, bool MIR = false>
static dash_status run_gemm(const GemmLaunch& g, cudaStream_t st) {
  using C = Cfg<BN, KT, MODE>;
  constexpr int CL = C::CL;
  CUtensorMap tA, tB, tAl, tBl;
  const int a_mn = g.transA ? 1 : 0;
  const int b_mn = g.transB ? 0 : 1;
  const uint32_t a_in = a_mn ? C::MN_ATOM : C::BK, a_out = a_mn ? C::BK : 128;
  const uint32_t b_in = b_mn ? C::MN_ATOM : C::BK, b_out = b_mn ? C::BK : BN / CL;
  // The TMA swizzle must produce the layout the MMA descriptor names.
  const CUtensorMapSwizzle mn_swz =
      C::H16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
  const CUtensorMapSwizzle a_swz = a_mn ? mn_swz : CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapSwizzle b_swz = b_mn ? mn_swz : CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_tmap(&tA, g.A, C::EB, g.dim, g.nblocks, a_in, a_out, a_swz)) return DASH_ERR_CUDA;
  if (!make_tmap(&tB, g.B, C::EB, g.dim, g.nblocks, b_in, b_out, b_swz)) return DASH_ERR_CUDA;
  tAl = tA;
  tBl = tB;
  if (C::NPART_A == 2 && !make_tmap(&tAl, g.A_lo, C::EB, g.dim, g.nblocks, a_in, a_out, a_swz))
    return DASH_ERR_CUDA;
  if (C::NPART_B == 2 && !make_tmap(&tBl, g.B_lo, C::EB, g.dim, g.nblocks, b_in, b_out, b_swz))
    return DASH_ERR_CUDA;
  KParams p;
  p.dim = g.dim;
  p.tiles_m = g.dim / 128;
  p.tiles_n = g.dim / BN;
  p.total_tiles = g.nblocks * p.tiles_m * p.tiles_n;
  p.total_units = p.total_tiles / CL;
  p.nkb = g.dim / C::BK;
  const uint32_t fmt = (g.kind == KIND_BF16 || g.kind == KIND_BF16_SPLITB)
                           ? 1u
                           : ((g.kind == KIND_F16 || g.kind == KIND_F16_SPLITB) ? 0u : 2u);
  p.idesc = make_idesc(fmt, a_mn, b_mn, C::MMA_M, BN);
  p.idesc0 = make_idesc(fmt, 0, 0, C::MMA_M, BN);
  p.a_mn = a_mn;
  p.b_mn = b_mn;
  p.epi = g.epi;
  // Symmetric-half iterates: CTA-pair tiles of the plain kernels only.
  const bool sym_ok = (MODE == 2 && (KT != 2 || ACC));
  p.sym_in = (sym_ok && g.sym_in) ? 1 : 0;
  p.sym_in_b = (sym_ok && g.sym_in_b) ? 1 : 0;
  p.sym_any = p.sym_in | p.sym_in_b;
  p.sym_out = (sym_ok && g.sym_out) ? 1 : 0;
  p.t256 = g.dim / 256;
  if (p.sym_out) {
    // CTA tiles: 2 per pair tile, 256 / BN pair tiles per upper 256 x 256 tile.
    p.total_tiles = g.nblocks * p.t256 * (p.t256 + 1) / 2 * (256 / BN) * CL;
    p.total_units = p.total_tiles / CL;
  }
  if (p.sym_any) {
    // The other-major view of each operand over the same memory.
    const uint32_t am_in = !a_mn ? C::MN_ATOM : C::BK, am_out = !a_mn ? C::BK : 128;
    const uint32_t bm_in = !b_mn ? C::MN_ATOM : C::BK, bm_out = !b_mn ? C::BK : BN / CL;
    if (!make_tmap(&p.tAm, g.A, C::EB, g.dim, g.nblocks, am_in, am_out,
                   !a_mn ? mn_swz : CU_TENSOR_MAP_SWIZZLE_128B))
      return DASH_ERR_CUDA;
    if (!make_tmap(&p.tBm, g.B, C::EB, g.dim, g.nblocks, bm_in, bm_out,
                   !b_mn ? mn_swz : CU_TENSOR_MAP_SWIZZLE_128B))
      return DASH_ERR_CUDA;
    p.tAlm = p.tAm;
    p.tBlm = p.tBm;
    if (C::NPART_A == 2 && !make_tmap(&p.tAlm, g.A_lo, C::EB, g.dim, g.nblocks, am_in, am_out,
                                      !a_mn ? mn_swz : CU_TENSOR_MAP_SWIZZLE_128B))
      return DASH_ERR_CUDA;
    if (C::NPART_B == 2 && !make_tmap(&p.tBlm, g.B_lo, C::EB, g.dim, g.nblocks, bm_in, bm_out,
                                      !b_mn ? mn_swz : CU_TENSOR_MAP_SWIZZLE_128B))
      return DASH_ERR_CUDA;
  }
  p.staged = (DASH_STAGED_EPILOGUE && C::EPI_BYTES > 0 && g.epi.nout >= 1 && g.epi.nout <= 2) ? 1 : 0;
  for (int o = 0; o < g.epi.nout && p.staged; ++o) {
    const EpiOut& O = g.epi.out[o];
    if ((O.fmt != FMT_F16 && O.fmt != FMT_BF16) ||
        (reinterpret_cast<uintptr_t>(O.hi) & 15u) != 0)
      p.staged = 0;
  }
  if (p.staged) {
    // Boxes of 32 rows x 64 columns (one output, 128-byte swizzle) or x 32
    // columns (two outputs, 64-byte swizzle), matching the staging layout.
    const bool one = (g.epi.nout == 1);
    for (int o = 0; o < g.epi.nout; ++o)
      if (!make_tmap(&p.tO[o], g.epi.out[o].hi, 2, g.dim, g.nblocks, one ? 64 : 32, 32,
                     one ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
        return DASH_ERR_CUDA;
  }
  // Run-time tile order for the mirrored-store pair instances (the accumulate and
  // the roots' fp32 results).  Timed launch by launch in the benchmark step (CUDA
  // events, interleaved rounds on several boxes), those launches were 8-16% faster
  // with it every time; the other products gained nothing consistent, and carrying
  // the ring's code slowed them, so they keep the fixed order.
  p.sched = nullptr;
  p.sched_id = 0u;
  if (MODE == 2 && MIR && !ACC && DASH_DYN_SCHED && !p.staged && p.total_units < (1LL << 31) &&
      !sched_slot(&p.sched, &p.sched_id))
    return DASH_ERR_CUDA;
  if (cudaFuncSetAttribute(KernelOf<BN, KT, MODE, ACC, MIR>::get(),
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_BYTES) != cudaSuccess)
    return DASH_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return DASH_ERR_CUDA;
  // Persistent grid: one CTA per SM, or as many clusters as can be co-resident.
  long long slots = sms / CL;
  if (CL > 1) {
    const int mac = max_active_clusters<BN, KT, MODE, ACC, MIR>();
    if (mac <= 0) return DASH_ERR_CUDA;
    if (mac < slots) slots = mac;
  }
  const long long nclusters = p.total_units < slots ? p.total_units : slots;
  const int rec = trace_begin(st);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * CL), 1, 1);
  cfg.blockDim = dim3(KernelOf<BN, KT, MODE, ACC, MIR>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, KernelOf<BN, KT, MODE, ACC, MIR>::get(), tA, tB, tAl, tBl, p);
  if (err == cudaSuccess) err = cudaGetLastError();
  if (rec >= 0) {
    const double bb = static_cast<double>(g.dim) * g.dim * g.nblocks;
    // A symmetric output computes and writes only the (T + 1) / 2T of C on or above
    // the diagonal (T = dim / 256): those are the flops and output bytes it costs.
    const double frac = p.sym_out ? (p.t256 + 1.0) / (2.0 * p.t256) : 1.0;
    double bytes = bb * C::EB * (C::NPART_A + C::NPART_B);
    for (int o = 0; o < g.epi.nout; ++o) bytes += frac * bb * fmt_bytes(g.epi.out[o].fmt);
    if (g.epi.E_hi != nullptr) bytes += frac * bb * fmt_bytes(g.epi.E_fmt);
    const bool bf = (g.kind == KIND_BF16 || g.kind == KIND_BF16_SPLITB);
    const int kind = KT == 2 ? DASH_TRACE_GEMM_3XTF32
                             : (KT == 1 ? DASH_TRACE_GEMM_TF32
                                        : (bf ? DASH_TRACE_GEMM_BF16 : DASH_TRACE_GEMM_F16));
    // Tensor-core flops as issued: a pair-B product issues two 16-bit MMAs per slice
    // (3xTF32 counts its fp32 product once against a third of the TF32 rate).
    trace_end(rec, st, kind, frac * 2.0 * bb * g.dim * (KT == 3 ? 2 : 1), bytes);
  }
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

dash_status launch_gemm(const GemmLaunch& g, cudaStream_t st) {
  if (g.nblocks <= 0) return DASH_OK;
  if (g.dim % 128 != 0 || g.dim < 128 || g.dim > 2048) return DASH_ERR_INVALID_ARG;
  const bool wide = (g.dim % 256) == 0;
  // An fp32 output of a symmetric-half launch that is completed below the
  // diagonal by transposed stores (the pair kernels' mirror instances).
  bool mir = false;
  for (int o = 0; o < g.epi.nout; ++o) mir = mir || (g.epi.out[o].mirror && g.sym_out);

  switch (g.kind) {
    // B a multiple of 256: CTA pairs on 256 x 256 tiles (cta_group::2); otherwise
    // one CTA per 128 x 128 tile.
    case KIND_F16:
    case KIND_BF16:
      if (wide && mir) return run_gemm<256, 0, 2, false, true>(g, st);
      return wide ? run_gemm<256, 0, 2>(g, st) : run_gemm<128, 0, 0>(g, st);
    case KIND_F16_SPLITB:
    case KIND_BF16_SPLITB:
      return wide ? run_gemm<256, 3, 2>(g, st) : run_gemm<128, 3, 0>(g, st);
    case KIND_TF32:
      if (wide && mir) return run_gemm<256, 1, 2, false, true>(g, st);
      return wide ? run_gemm<256, 1, 2>(g, st) : run_gemm<128, 1, 0>(g, st);
    case KIND_TF32X3:
      // fp32-accurate products: partial sums reduced with round-to-nearest.
      return wide ? run_gemm<ACC_BN, 2, 2, true>(g, st) : run_gemm<128, 2, 0>(g, st);
    default:
      return DASH_ERR_INVALID_ARG;
  }
}

}  // namespace dash
