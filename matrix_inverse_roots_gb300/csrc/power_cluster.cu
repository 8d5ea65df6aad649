// Half-precision multi-vector power iteration with every block read from HBM
// once per call: a thread-block cluster works on two blocks at a time, keeps their
// 16-bit copies in L2 for all the products, and exchanges the vector slabs through
// distributed shared memory ([pt] Metodologia 2, the multi-power iteration;
// Principais Contribuicoes item 4, the half-precision iteration).
//
// A block of order B = 128 C is handled by a cluster of C CTAs.  CTA r owns rows
// 128 r .. 128 r + 127 (one slab) of every product W = (sigma A + sigma ridge I) V D,
// D = diag(1 / ||previous column||), with the rounding points of the one-product-
// per-launch kernel: the 16-bit copy of sigma A, 16-bit vectors between products,
// fp32 accumulation and fp32 column sums of the stored values.
//
// Two lanes.  One block's products form a chain: product k + 1 needs every CTA's
// part of W_k.  Each cluster therefore runs two blocks ("lanes") and the MMA warp
// alternates between them, so that one lane's epilogue and exchange overlap the
// other lane's MMAs.  Lane 1 starts half a block after lane 0, so that the two
// lanes change blocks at different times.  Per lane: a TMEM accumulator, one V^T
// buffer (32 x B, 16-bit, the swizzled layout the MMA reads).  The cluster's blocks
// take turns in three scratch slots in global memory for their 16-bit copies: when
// a lane finishes a block, the slot it frees is refilled with the other lane's next
// block while that lane still has half a block to run.
//   warps 6..9   converters: the cluster's blocks in order, fp32 -> sigma A in 16
//                bits, each into its slot once the block three back has left it.
//   warp 0       TMA producer: the slab's 128 x 64 tiles from the slot, in the
//                order the MMA warp consumes them.
//   warp 1       MMA issuer: per product four M = 128, N = 32, K = 16 MMAs per
//                k-block into the lane's accumulator, B = the lane's V^T.
//   warps 2..5   epilogue, one slab row per thread: scale, ridge term, the new
//                rows of V^T in 16 bits into this CTA's buffer, fp32 column sums.
//                Once every CTA has finished the product's MMAs (an mbarrier each
//                CTA arrives on remotely), threads 1 .. C-1 each bulk-copy the
//                slab's 32 x 128 part of V^T and the column sums into one other CTA
//                (cp.async.bulk shared::cluster, completing on the receiver's
//                mbarrier).  After the last product rank 0 writes
//                lambda = max_c (v.w / v.v) / sigma and the start vectors of the
//                lane's next block are loaded (TMA, from the (32, B) transposed copy).
// Every wait is bounded; every branch after a wait is taken by all threads of a
// role (a barrier with an AND vote); a time-out sets the device flag, the CTA
// drains its copies and MMAs, frees TMEM and returns.
#include <atomic>

#include "dash_common.cuh"
#include "dash_internal.h"

namespace dash {

int power_cluster_read_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_dash_error, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_dash_error, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

namespace {

constexpr int PC_BM = 128;                    // slab rows per CTA
constexpr int PC_BK = 64;                     // 16-bit elements per 128-byte row
constexpr int PC_NV = 32;
constexpr int PC_MAX_CL = 8;                  // portable cluster size: B <= 1024
constexpr int PC_A_BYTES = PC_BM * 128;       // 16 KB A tile
constexpr int PC_STAGES = 5;
constexpr int PC_VT_TILE = PC_NV * 128;       // one k-block of V^T: 32 rows of 128 B
constexpr int PC_PART = 2 * PC_NV;            // column sums per CTA: s0 | s1
constexpr int PC_PART_BYTES = PC_PART * 4;    // 256
constexpr int PC_EPI_WARPS = 4;
constexpr int PC_EPI_THREADS = 32 * PC_EPI_WARPS;
constexpr int PC_CONV_WARPS = 4;
constexpr int PC_CONV_THREADS = 32 * PC_CONV_WARPS;
constexpr int PC_THREADS = 32 * (2 + PC_EPI_WARPS + PC_CONV_WARPS);
constexpr int PC_CONV0 = 32 * (2 + PC_EPI_WARPS);  // first converter thread
constexpr int PC_UNROLL = 8;                  // 32-byte converter loads in flight per thread
constexpr int PC_SLOTS = 3;                   // scratch slots per cluster
// barriers: full, empty per stage; per lane vfull, lamfull, tfull, tempty, mdone;
// per slot ready, sfree; fin
constexpr int PC_LANE_BARS = 5;
constexpr int PC_NBAR = 2 * PC_STAGES + 2 * PC_LANE_BARS + 2 * PC_SLOTS + 1;
constexpr int PC_BAR_AREA = 256;
static_assert(PC_NBAR * 8 + 16 <= PC_BAR_AREA, "barrier area");
constexpr int PC_TMEM_COLS = 64;              // two 32-column accumulators
// Named barriers (id 0 is __syncthreads).
constexpr int PC_BAR_EPI = 1;
constexpr int PC_BAR_CONV = 2;

// Shared memory: A stages | V^T lane 0 | V^T lane 1 | column sums
// [lane][parity][MAX_CL][64] | scales [lane][32] | reduction [4][64] | barriers.
size_t pc_smem_bytes(int dim) {
  const size_t vt = static_cast<size_t>(dim / PC_BK) * PC_VT_TILE;
  return 1024 + static_cast<size_t>(PC_STAGES) * PC_A_BYTES + 2 * vt +
         4 * PC_MAX_CL * PC_PART_BYTES + 2 * PC_NV * 4 + PC_EPI_WARPS * PC_PART_BYTES +
         PC_BAR_AREA;
}

struct PcParams {
  const float* A;        // (nblocks, dim, dim) fp32
  const float* sigma;    // (nblocks) power-of-two scale of each block
  uint16_t* scratch;     // (ncl * PC_SLOTS, dim, dim) 16-bit slots
  float* lambda;         // (nblocks)
  long long nblocks;
  int dim;
  int cl;                // CTAs per cluster = dim / 128
  int nv;
  int iters;
  float ridge;
  uint32_t idesc;
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

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier that also returns the AND of every participating thread's `v`, so
// that all of them take the same branch after a bounded wait (a thread leaving a
// loop that the others stay in would leave them at the next barrier forever).
__device__ __forceinline__ bool named_and(int id, int n, bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return out != 0;
}

// Byte offset of element (c, g) of V^T (32 x dim, 16-bit) in a buffer laid out as
// dim / 64 k-block tiles of 32 rows x 128 bytes with the 128-byte swizzle (16-byte
// chunk index XOR row mod 8), the layout a TMA load with 128B swizzle produces and
// the MMA's B descriptor reads.
__device__ __forceinline__ uint32_t vt_off(int c, int g) {
  const uint32_t bc = static_cast<uint32_t>(g & 63) * 2u;
  return static_cast<uint32_t>(g >> 6) * PC_VT_TILE + static_cast<uint32_t>(c) * 128u +
         (bc ^ (static_cast<uint32_t>(c & 7) << 4));
}


// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from this
// CTA's shared memory to shared memory of a CTA of the cluster (shared::cluster
// address from mapa_shared), completing on that CTA's mbarrier `bar`.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes,
                                                     uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Make this thread's generic-proxy global writes visible to a later TMA load.
__device__ __forceinline__ void fence_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The order in which the cluster's lane-products run.  Lane L holds the cluster's
// blocks j = 2 i + L (i = 0, 1, ...); its products are (i, k), k < iters.  Lane 1
// starts once lane 0 has run iters / 2 products, and from then on the two lanes
// alternate while both have products left, so that their block changes are half a
// block apart: a slot freed by one lane's block is refilled while the other lane
// still has half a block to run.  Producer, MMA warp and epilogue each walk this
// same sequence.
struct LaneSeq {
  // Per-lane fields as scalars (an array indexed by the lane would live in local
  // memory).
  long long nb0, nb1;  // blocks per lane
  long long i0, i1;    // current block of each lane
  int k0, k1;          // current product of each lane
  long long done0;     // products lane 0 has run
  int next;
  int iters;
  __device__ void init(long long nclust_blocks, int it) {
    nb0 = (nclust_blocks + 1) / 2;
    nb1 = nclust_blocks / 2;
    i0 = i1 = 0;
    k0 = k1 = 0;
    done0 = 0;
    next = 0;
    iters = it;
  }
  __device__ bool more(int l) const { return l ? (i1 < nb1) : (i0 < nb0); }
  __device__ bool avail(int l) const {
    return more(l) && (l == 0 || done0 >= iters / 2 || !more(0));
  }
  // The next lane-product; false when both lanes are done.
  __device__ bool step(int& lane, long long& bi, int& kk) {
    int l = next;
    if (!avail(l)) l ^= 1;
    if (!avail(l)) return false;
    lane = l;
    if (l == 0) {
      bi = i0;
      kk = k0;
      if (++k0 == iters) {
        k0 = 0;
        ++i0;
      }
      ++done0;
    } else {
      bi = i1;
      kk = k1;
      if (++k1 == iters) {
        k1 = 0;
        ++i1;
      }
    }
    next = l ^ 1;
    return true;
  }
};

template <bool BF>
__global__ void __launch_bounds__(PC_THREADS, 1)
    power_cluster_kernel(const __grid_constant__ CUtensorMap tS, const __grid_constant__ CUtensorMap tV,
                         const __grid_constant__ PcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;
  // The layout is the same in every CTA, so mapa_shared finds a peer's copy.
  const int dim = p.dim;
  const int C = p.cl;
  const int iters = p.iters;
  const uint32_t vt_bytes = static_cast<uint32_t>(dim / PC_BK) * PC_VT_TILE;
  const uint32_t off_vt = PC_STAGES * PC_A_BYTES;
  const uint32_t off_part = off_vt + 2 * vt_bytes;
  const uint32_t off_sc = off_part + 4 * PC_MAX_CL * PC_PART_BYTES;
  const uint32_t off_red = off_sc + 2 * PC_NV * 4;
  const uint32_t off_bar = off_red + PC_EPI_WARPS * PC_PART_BYTES;
  auto vt_buf = [&](int l) { return sbase + off_vt + static_cast<uint32_t>(l) * vt_bytes; };
  auto part_off = [&](int l, int par, int q) {
    return off_part + static_cast<uint32_t>((l * 2 + par) * PC_MAX_CL + q) * PC_PART_BYTES;
  };
  float* sc_s = reinterpret_cast<float*>(smem + off_sc);   // [lane][32]
  float* red = reinterpret_cast<float*>(smem + off_red);   // [4][64]
  const uint32_t bar0 = sbase + off_bar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (PC_STAGES + s); };
  auto lane_bar = [&](int l, int t) { return bar0 + 8u * (2 * PC_STAGES + l * PC_LANE_BARS + t); };
  enum { VFULL = 0, LAMFULL = 1, TFULL = 2, TEMPTY = 3, MDONE = 4 };
  auto slot_bar = [&](int s, int t) {
    return bar0 + 8u * (2 * PC_STAGES + 2 * PC_LANE_BARS + s * 2 + t);
  };
  enum { READY = 0, SFREE = 1 };
  const uint32_t fin_bar = bar0 + 8u * (2 * PC_STAGES + 2 * PC_LANE_BARS + 2 * PC_SLOTS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_bar + 8 * PC_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_bar + 8 * PC_NBAR + 8);

  const int warp = threadIdx.x >> 5;
  const int lane_id = threadIdx.x & 31;
  const int r = static_cast<int>(cluster_ctarank());
  const long long cid = blockIdx.x / C;
  const long long ncl = gridDim.x / C;
  const int nkb = dim / PC_BK;
  // This cluster's blocks: j-th = cid + j ncl; lane l takes those with j % 2 == l,
  // and block j's 16-bit copy lives in slot j % PC_SLOTS (its (j / PC_SLOTS)-th use).
  const long long nmine = (cid < p.nblocks) ? (p.nblocks - cid + ncl - 1) / ncl : 0;
  auto block_of = [&](int l, long long i) { return cid + ncl * (2 * i + l); };
  auto slot_index = [&](long long j) { return cid * PC_SLOTS + j % PC_SLOTS; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < PC_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int l = 0; l < 2; ++l) {
      mbar_init(lane_bar(l, VFULL), 1);
      mbar_init(lane_bar(l, LAMFULL), 1);
      mbar_init(lane_bar(l, TFULL), 1);
      mbar_init(lane_bar(l, TEMPTY), PC_EPI_WARPS);
      mbar_init(lane_bar(l, MDONE), C);
    }
    for (int s = 0; s < PC_SLOTS; ++s) {
      mbar_init(slot_bar(s, READY), 1);
      mbar_init(slot_bar(s, SFREE), 1);
    }
    mbar_init(fin_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane_id == 0) {
    tma_prefetch_desc(&tS);
    tma_prefetch_desc(&tV);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), PC_TMEM_COLS);
  tc_fence_before();
  // Every CTA's barriers are initialised before any CTA of the cluster uses them.
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane_id == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      LaneSeq seq;
      seq.init(nmine, iters);
      int l, k;
      long long i;
      while (ok && seq.step(l, i, k)) {
        // A block's first product waits for its 16-bit copy.
        const long long j = 2 * i + l;
        if (k == 0 && !mbar_wait(slot_bar(static_cast<int>(j % PC_SLOTS), READY),
                                 static_cast<uint32_t>((j / PC_SLOTS) & 1), abort_flag))
          break;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, PC_A_BYTES);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          tma_load_3d(sbase + stage * PC_A_BYTES, &tS, fb, kb * PC_BK, r * PC_BM,
                      static_cast<int>(slot_index(j)));
          if (++stage == PC_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < PC_STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane_id == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      long long n0 = 0, n1 = 0;  // lane-products issued per lane
      bool ok = true;
      LaneSeq seq;
      seq.init(nmine, iters);
      int l, k;
      long long i;
      while (ok && seq.step(l, i, k)) {
        const uint32_t par = static_cast<uint32_t>((l ? n1 : n0) & 1);
        if (!mbar_wait(lane_bar(l, VFULL), par, abort_flag) ||
            !mbar_wait(lane_bar(l, TEMPTY), par ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem_base + static_cast<uint32_t>(l * PC_NV);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sbase + stage * PC_A_BYTES;
          const uint32_t sV = vt_buf(l) + static_cast<uint32_t>(kb) * PC_VT_TILE;
#pragma unroll
          for (int kk = 0; kk < PC_BK / 16; ++kk) {
            const uint64_t da = smem_desc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t dv = smem_desc_sw128(sV + kk * 32, 16, 1024);
            mma_f16(acc, da, dv, p.idesc, (kb | kk) ? 1u : 0u);
          }
          mma_commit(empty_bar(stage));
          if (++stage == PC_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(lane_bar(l, TFULL));
        // The block's last product has read its slot: the converters may refill it.
        if (k == iters - 1) mma_commit(slot_bar(static_cast<int>((2 * i + l) % PC_SLOTS), SFREE));
        if (l) ++n1; else ++n0;
      }
      mma_commit(fin_bar);
      mbar_wait_drain(fin_bar, 0);
    }
  } else if (warp < 2 + PC_EPI_WARPS) {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int ew = warp - 2;             // epilogue warp index
    const int et = threadIdx.x - 64;     // 0 .. 127
    const int g = r * PC_BM + q * 32 + lane_id;  // block row of this thread
    // Start vectors of lane l's block i into its V^T buffer (16 TMA tiles).
    auto issue_v0 = [&](int l, long long i) {
      const uint32_t vb = lane_bar(l, VFULL);
      mbar_arrive_expect_tx(vb, vt_bytes);
      for (int kb = 0; kb < nkb; ++kb)
        tma_load_3d(vt_buf(l) + static_cast<uint32_t>(kb) * PC_VT_TILE, &tV, vb, kb * PC_BK, 0,
                    static_cast<int>(block_of(l, i)));
    };
    if (et == 0) {
      if (nmine >= 1) issue_v0(0, 0);
      if (nmine >= 2) issue_v0(1, 0);
    }
    long long n0 = 0, n1 = 0;  // lane-products finished per lane
    bool ok = true;
    LaneSeq seq;
    seq.init(nmine, iters);
    int l, k;
    long long i;
    while (ok && seq.step(l, i, k)) {
      const long long blk = block_of(l, i);
      const float sig = p.sigma[blk];
      const float rb = p.ridge * sig;  // the copy holds sigma A: ridge term sigma ridge
      const bool last = (k == iters - 1);
      const uint32_t par = static_cast<uint32_t>((l ? n1 : n0) & 1);
      const bool got = mbar_wait(lane_bar(l, TFULL), par, abort_flag) &&
                       mbar_wait(lane_bar(l, VFULL), par, abort_flag);
      if (!named_and(PC_BAR_EPI, PC_EPI_THREADS, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r0[16], r1[16];
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(l * PC_NV);
      tmem_ld16(taddr, r0);
      tmem_ld16(taddr + 16, r1);
      tmem_wait_ld(r0);
      tmem_fence_regs(r1);
      tc_fence_before();
      __syncwarp();
      if (lane_id == 0) mbar_arrive(lane_bar(l, TEMPTY));  // accumulator copied to registers
      // This CTA's MMAs of the product are done (TFULL): tell every CTA of the cluster,
      // thread 32 + q telling rank q (in parallel, while threads 0 .. 31 compute the
      // column scales).
      if (et >= 32 && et < 32 + C)
        mbar_arrive_cluster(mapa_shared(lane_bar(l, MDONE), static_cast<uint32_t>(et - 32)));
      // 1 / ||column c of V_k||, from the column sums of all CTAs (1 on the first
      // product, 0 for unused columns), computed once per product.
      if (et < PC_NV) {
        float s = 0.0f;
        if (et < p.nv) {
          if (k == 0) {
            s = 1.0f;
          } else {
            float n2 = 0.0f;
            for (int qq = 0; qq < C; ++qq)
              n2 += reinterpret_cast<const float*>(smem + part_off(l, k & 1, qq))[et];
            s = 1.0f / sqrtf(n2);
          }
        }
        sc_s[l * PC_NV + et] = s;
      }
      named_sync(PC_BAR_EPI, PC_EPI_THREADS);
      // W's row g; this thread's row of V_{k+1} replaces its row of V_k in place (no
      // other CTA reads this buffer, and this CTA's MMAs of product k are done).  The
      // 32 values are loaded together and stored together.
      uint16_t* vrow = reinterpret_cast<uint16_t*>(smem + off_vt + static_cast<uint32_t>(l) * vt_bytes);
      uint16_t vh[PC_NV];
#pragma unroll
      for (int c = 0; c < PC_NV; ++c) vh[c] = vrow[vt_off(c, g) >> 1];
      float t[PC_NV];
      if (last) {
        // The final column sums v.v and v.w, one after the other (one array live).
#pragma unroll
        for (int c = 0; c < PC_NV; ++c) {
          const float v = h16_to_f<BF>(vh[c]) * sc_s[l * PC_NV + c];
          t[c] = v * v;
        }
        red[ew * PC_PART + 32 + lane_id] = butterfly_colsum(t, lane_id);
#pragma unroll
        for (int c = 0; c < PC_NV; ++c) {
          const float scc = sc_s[l * PC_NV + c];
          const float v = h16_to_f<BF>(vh[c]) * scc;
          const float acc = __uint_as_float(c < 16 ? r0[c] : r1[c - 16]);
          t[c] = v * fmaf(rb, v, acc * scc);
        }
      } else {
#pragma unroll
        for (int c = 0; c < PC_NV; ++c) {
          const float scc = sc_s[l * PC_NV + c];
          const float v = h16_to_f<BF>(vh[c]) * scc;
          const float acc = __uint_as_float(c < 16 ? r0[c] : r1[c - 16]);
          vh[c] = f_to_h16<BF>(fmaf(rb, v, acc * scc));
          const float wr = h16_to_f<BF>(vh[c]);  // the next product sees the stored value
          t[c] = wr * wr;
        }
#pragma unroll
        for (int c = 0; c < PC_NV; ++c) vrow[vt_off(c, g) >> 1] = vh[c];
      }
      red[ew * PC_PART + lane_id] = butterfly_colsum(t, lane_id);
      named_sync(PC_BAR_EPI, PC_EPI_THREADS);
      const int np = (k + 1) & 1;  // column sums of V_{k+1} (or the final sums)
      if (et < (last ? PC_PART : PC_NV)) {
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < PC_EPI_WARPS; ++w) tot += red[w * PC_PART + et];
        reinterpret_cast<float*>(smem + part_off(l, np, r))[et] = tot;
      }
      fence_async_shared();  // rows of V^T and column sums: read next by bulk copies
      // Every CTA must have finished the product's MMAs before its buffer is written.
      bool md = true;
      if (et == 0) md = mbar_wait_cluster(lane_bar(l, MDONE), par, abort_flag);
      if (!named_and(PC_BAR_EPI, PC_EPI_THREADS, md)) {
        ok = false;
        break;
      }
      // Thread et = d (1 <= d < C) sends to cluster rank (r + d) mod C; thread 0 arms
      // this CTA's own barrier for what the peers send.
      if (et < C) {
        const uint32_t psrc = sbase + part_off(l, np, r);
        const uint32_t qr = static_cast<uint32_t>((r + et) % C);
        if (!last) {
          if (et == 0) {
            mbar_arrive_expect_tx(lane_bar(l, VFULL),
                                  static_cast<uint32_t>(C - 1) * (2 * PC_VT_TILE + PC_PART_BYTES));
          } else {
            // This CTA's 32 x 128 part of V_{k+1} (two k-block tiles) and its sums.
            const uint32_t vsrc = vt_buf(l) + static_cast<uint32_t>(2 * r) * PC_VT_TILE;
            const uint32_t rbar = mapa_shared(lane_bar(l, VFULL), qr);
            bulk_copy_to_cluster(mapa_shared(vsrc, qr), vsrc, 2 * PC_VT_TILE, rbar);
            bulk_copy_to_cluster(mapa_shared(psrc, qr), psrc, PC_PART_BYTES, rbar);
          }
        } else {
          if (et == 0)
            mbar_arrive_expect_tx(lane_bar(l, LAMFULL), static_cast<uint32_t>(C - 1) * PC_PART_BYTES);
          else
            bulk_copy_to_cluster(mapa_shared(psrc, qr), psrc, PC_PART_BYTES,
                                 mapa_shared(lane_bar(l, LAMFULL), qr));
        }
      }
      if (l) ++n1; else ++n0;
      if (last) {
        // lambda of the block from the final column sums of all CTAs.
        const bool fin = mbar_wait(lane_bar(l, LAMFULL), static_cast<uint32_t>(i & 1), abort_flag);
        if (!named_and(PC_BAR_EPI, PC_EPI_THREADS, fin)) {
          ok = false;
          break;
        }
        if (et == 0 && r == 0) {
          float best = -INFINITY;
          for (int c = 0; c < p.nv; ++c) {
            float num = 0.0f, den = 0.0f;
            for (int qq = 0; qq < C; ++qq) {
              const float* pp = reinterpret_cast<const float*>(smem + part_off(l, np, qq));
              num += pp[c];
              den += pp[32 + c];
            }
            best = fmaxf(best, num / den);
          }
          p.lambda[blk] = best / sig;  // a power-of-two scale divides out exactly
        }
        named_sync(PC_BAR_EPI, PC_EPI_THREADS);
        // The lane's next block: its start vectors (this CTA's MMAs of the block are
        // done, and no CTA sends into this buffer before this CTA's next MMAs).
        if (et == 0 && seq.more(l)) issue_v0(l, i + 1);
      }
    }
  } else {
    // -------------------------------------------------------------- converters
    const int ct = threadIdx.x - PC_CONV0;  // 0 .. 127
    const int cpr = dim / 8;                // 8-element chunks per row
    const int nch = PC_BM * cpr;            // chunks in the slab
    for (long long j = 0; j < nmine; ++j) {
      {
        const int sl = static_cast<int>(j % PC_SLOTS);
        const long long blk = cid + ncl * j;
        const float* src = p.A + (blk * dim + static_cast<long long>(r) * PC_BM) * dim;
        // The slot's previous block (three back) has been read by all its products.
        const bool got = mbar_wait(slot_bar(sl, SFREE),
                                   static_cast<uint32_t>((j / PC_SLOTS) & 1) ^ 1u, abort_flag);
        if (!named_and(PC_BAR_CONV, PC_CONV_THREADS, got)) break;
        const float sig = p.sigma[blk];
        uint16_t* dst = p.scratch + (slot_index(j) * dim + static_cast<long long>(r) * PC_BM) * dim;
        for (int i0 = ct; i0 < nch; i0 += PC_CONV_THREADS * PC_UNROLL) {
          float4 x[PC_UNROLL][2];
#pragma unroll
          for (int u = 0; u < PC_UNROLL; ++u) {
            const int ii = i0 + u * PC_CONV_THREADS;
            if (ii < nch) {
              const float4* s4 = reinterpret_cast<const float4*>(
                  src + static_cast<long long>(ii / cpr) * dim + (ii % cpr) * 8);
              x[u][0] = __ldcs(s4);
              x[u][1] = __ldcs(s4 + 1);
            }
          }
#pragma unroll
          for (int u = 0; u < PC_UNROLL; ++u) {
            const int ii = i0 + u * PC_CONV_THREADS;
            if (ii < nch) {
              uint4 o;
              o.x = static_cast<uint32_t>(f_to_h16<BF>(x[u][0].x * sig)) |
                    (static_cast<uint32_t>(f_to_h16<BF>(x[u][0].y * sig)) << 16);
              o.y = static_cast<uint32_t>(f_to_h16<BF>(x[u][0].z * sig)) |
                    (static_cast<uint32_t>(f_to_h16<BF>(x[u][0].w * sig)) << 16);
              o.z = static_cast<uint32_t>(f_to_h16<BF>(x[u][1].x * sig)) |
                    (static_cast<uint32_t>(f_to_h16<BF>(x[u][1].y * sig)) << 16);
              o.w = static_cast<uint32_t>(f_to_h16<BF>(x[u][1].z * sig)) |
                    (static_cast<uint32_t>(f_to_h16<BF>(x[u][1].w * sig)) << 16);
              *reinterpret_cast<uint4*>(dst + static_cast<long long>(ii / cpr) * dim + (ii % cpr) * 8) = o;
            }
          }
        }
        fence_async_global();  // the slot is read next by TMA
        named_sync(PC_BAR_CONV, PC_CONV_THREADS);
        if (ct == 0) mbar_arrive(slot_bar(sl, READY));
      }
    }
  }

  tc_fence_before();
  // No CTA leaves while a peer may still send into its shared memory.
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, PC_TMEM_COLS);
  }
}

}  // namespace

bool power_cluster_supported(int dim) {
  return dim >= PC_BM && dim % PC_BM == 0 && dim / PC_BM <= PC_MAX_CL;
}

size_t power_cluster_slot_bytes(int dim) { return static_cast<size_t>(dim) * dim * 2; }

// Clusters of dim / 128 CTAs of this kernel that fit on the current device at once
// (0 on error), cached per device, cluster size and format.
int power_cluster_max_clusters(int dim, int bf16) {
  static std::atomic<int> cache[64][2 * (PC_MAX_CL + 1)];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int C = dim / PC_BM;
  std::atomic<int>& oc = cache[dev][2 * C + (bf16 ? 1 : 0)];
  const int known = oc.load();
  if (known > 0) return known;
  auto kern = bf16 ? power_cluster_kernel<true> : power_cluster_kernel<false>;
  const size_t smem = pc_smem_bytes(dim);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C), 1, 1);
  cfg.blockDim = dim3(PC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return 0;
  oc.store(n);
  return n;
}

dash_status launch_power_cluster(const float* A, int bf16, float ridge, const float* sigma,
                                 int dim, long long nblocks, const uint16_t* Vt, int nv,
                                 int iters, uint16_t* scratch, int ncl, float* lambda,
                                 cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  if (!power_cluster_supported(dim) || ncl < 1 || nv < 1 || nv > PC_NV || iters < 1)
    return DASH_ERR_INVALID_ARG;
  CUtensorMap tS, tV;
  if (!map_3d_u16(&tS, scratch, dim, dim, static_cast<uint64_t>(ncl) * PC_SLOTS, PC_BK, PC_BM))
    return DASH_ERR_CUDA;
  if (!map_3d_u16(&tV, Vt, dim, PC_NV, static_cast<uint64_t>(nblocks), PC_BK, PC_NV))
    return DASH_ERR_CUDA;
  PcParams p;
  p.A = A;
  p.sigma = sigma;
  p.scratch = scratch;
  p.lambda = lambda;
  p.nblocks = nblocks;
  p.dim = dim;
  p.cl = dim / PC_BM;
  p.nv = nv;
  p.iters = iters;
  p.ridge = ridge;
  p.idesc = make_idesc(bf16 ? 1u : 0u, 0, 0, PC_BM, PC_NV);
  auto kern = bf16 ? power_cluster_kernel<true> : power_cluster_kernel<false>;
  const size_t smem = pc_smem_bytes(dim);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DASH_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * p.cl), 1, 1);
  cfg.blockDim = dim3(PC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int rec = trace_begin(st);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kern, tS, tV, p);
  const double bb = static_cast<double>(dim) * dim * nblocks;
  // Algorithmic bytes: A read once in fp32, the start vectors, lambda.
  trace_end(rec, st, DASH_TRACE_POWER, 2.0 * bb * nv * iters,
            4.0 * bb + static_cast<double>(nblocks) * (2.0 * dim * PC_NV + 8.0));
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

}  // namespace dash
