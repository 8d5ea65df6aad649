// Host-side interfaces between the C-ABI layer (dash_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dashroot.h"

namespace dash {

// One output of a fused epilogue:
//   D = mult[blk] * (alpha * C + gamma * I + eps * E)   stored in format fmt.
// (mult may be null = 1; E is the launch's optional extra matrix.)
// mirror (FMT_F32 outputs of a sym_out launch): each computed 256-tile above the
// diagonal is also stored transposed into its mirror below the diagonal, so the
// output holds the whole symmetric matrix.
struct EpiOut {
  void* hi;
  void* lo;
  const float* mult;
  float alpha, gamma, eps;
  int fmt;
  int mirror = 0;
};

struct EpiParams {
  EpiOut out[3];
  int nout;
  const void* E_hi;  // optional matrix read by the epilogue (same stacking as C)
  const void* E_lo;
  int E_fmt;
  float* resid_acc;        // if set: resid_acc[blk * resid_stride] += sum (C - I)^2
  long long resid_stride;
  int resid_plus_e;        // residual of C + E instead of C (identity-shifted iterates)
  const int* pad_valid;    // if set: rows / cols >= pad_valid[blk] become the identity's
};

// C[k] = op(A[k]) op(B[k]) for k < nblocks, fused with the epilogue.
struct GemmLaunch {
  int kind;  // KIND_*
  int dim;
  long long nblocks;
  const void* A;
  const void* A_lo;
  int transA;
  const void* B;
  const void* B_lo;
  int transB;
  EpiParams epi;
  // Symmetric-half iterates (honoured for CTA-pair tiles, B a multiple of 256):
  // sym_in -- A (sym_in_b: B) symmetric, only its 256-tiles on or above the
  // diagonal are read; sym_out -- only C's 256-tiles on or above the diagonal are
  // computed.
  int sym_in = 0;
  int sym_in_b = 0;
  int sym_out = 0;
};

dash_status launch_gemm(const GemmLaunch& g, cudaStream_t st);

// Element-wise affine map of a stack:  x = (src + ridge I) * inv_s[blk]  (inv_s
// may be null = 1), then each output D = mult[blk] * (alpha x + gamma I) and,
// if resid_acc is set, resid_acc[blk * resid_stride] += sum (x - I)^2.
struct AffOut {
  void* hi;
  void* lo;
  const float* mult;
  float alpha, gamma;
  int fmt;
};

struct AffParams {
  const void* src_hi;
  const void* src_lo;
  int src_fmt;
  float ridge;
  const float* inv_s;
  AffOut out[3];
  int nout;
  float* resid_acc;
  long long resid_stride;
  int dim;
  long long nblocks;
};

dash_status launch_affine(const AffParams& p, cudaStream_t st);

// inv_s[k] = 1 / s[k], s_m14[k] = s[k]^{-1/4}.
dash_status launch_scale_factors(const float* s, float* inv_s, float* s_m14, long long n,
                                 cudaStream_t st);

// out[i] = sqrt(acc[i]) * mul.
dash_status launch_sqrt_scale(const float* acc, float* out, long long n, float mul,
                              cudaStream_t st);

// acc[k] += sum over block k of (A + ridge I)^2 (acc zeroed by the caller).
dash_status launch_frob_acc(const float* A, float ridge, int dim, long long nblocks, float* acc,
                            cudaStream_t st);

// One power-iteration product W = (A + ridge I) V for every block, on the tensor
// cores in 3xTF32 (A and V split into TF32 hi/lo in shared memory).  V is read as
// Vin[blk][row][c] / sqrt(in_nrm2[blk][c]) (in_nrm2 null = unscaled), row stride 32.
// Not last: writes W and acc0[blk][c] += sum_r W^2.
// Last: acc0[blk][c] += sum_r v w, acc1[blk][c] += sum_r v v (W not written).
// Weight-shaped (rows, cols, leading dimension ld) <-> row-block-major (b, b)
// blocks, element size esize (2 or 4); vr / vc (nullable) get each block's extent.
dash_status launch_pack_blocks(const void* M, int esize, long long rows, long long cols,
                               long long ld, int b, void* out, int32_t* vr, int32_t* vc,
                               cudaStream_t st);
dash_status launch_unpack_blocks(const void* blocks, int esize, long long rows, long long cols,
                                 long long ld, int b, void* M, cudaStream_t st);

// out[i] = a[i] - b[i].
dash_status launch_sub(const float* a, const float* b, float* out, long long n, cudaStream_t st);

// n items of `elems` floats: dst[j] = src[idx[j]] (scatter 0) or dst[idx[j]] = src[j]
// (scatter 1), j < n; idx is a device array of n indices.  16-byte aligned pointers
// when elems is a multiple of 4.
dash_status launch_copy_items(const float* src, float* dst, const int32_t* idx, int scatter,
                              long long elems, long long n, cudaStream_t st);

// One half-precision power product on (nblocks, dim, dim) 16-bit A (bf16 != 0:
// bfloat16, else fp16); vectors transposed, (nblocks, 32, dim) 16-bit.  When
// blk_scale is given, block k of Ah holds sigma_k A_k and its ridge term is
// sigma_k ridge.
dash_status launch_power_step_half(const void* Ah, int bf16, float ridge, const float* blk_scale,
                                   int dim, long long nblocks, const uint16_t* Vt_in, int nv,
                                   const float* in_nrm2, uint16_t* Vt_out, float* acc0,
                                   float* acc1, int last, cudaStream_t st);

// The whole half-precision power iteration (iters products and lambda) with each
// block read from A once: clusters of dim / 128 CTAs, each running two blocks at a
// time ("lanes"), their 16-bit copies sigma A kept in `scratch` (3 ncl slots of dim^2
// 16-bit elements) for all products.  Vt (nblocks, 32, dim) 16-bit: the start
// vectors transposed (launch_pad_vectors_t); lambda[k] = max_c (v.w / v.v) /
// sigma[k] after the last product.
bool power_cluster_supported(int dim);  // dim a multiple of 128, at most 1024
size_t power_cluster_slot_bytes(int dim);
int power_cluster_max_clusters(int dim, int bf16);  // 0 on error
dash_status launch_power_cluster(const float* A, int bf16, float ridge, const float* sigma,
                                 int dim, long long nblocks, const uint16_t* Vt, int nv,
                                 int iters, uint16_t* scratch, int ncl, float* lambda,
                                 cudaStream_t st);

// 3-D tensor map over 16-bit elements (inner, outer, nblk), 128B swizzle.
bool map_3d_u16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t nblk,
                uint32_t box_inner, uint32_t box_outer);

// V0 (nblocks, dim, nv) fp32 -> Vt (nblocks, 32, dim) 16-bit, rows c >= nv zero.
dash_status launch_pad_vectors_t(const float* V0, int nv, int dim, long long nblocks, int bf16,
                                 uint16_t* Vt, cudaStream_t st);

dash_status launch_power_step_tc(const float* A, float ridge, int dim, long long nblocks,
                                 const float* Vin, int nv, const float* in_nrm2, float* Wout,
                                 float* acc0, float* acc1, int last, cudaStream_t st);

// V (nblocks, dim, 32) = V0 (nblocks, dim, nv) with columns nv..31 zero.
dash_status launch_pad_vectors(const float* V0, int nv, int dim, long long nblocks, float* V,
                               cudaStream_t st);

// lambda[k] = max_{c < nv} num[k][c] / den[k][c], divided by blk_scale[k] when given.
dash_status launch_power_finish(const float* num, const float* den, int nv, long long nblocks,
                                const float* blk_scale, float* lambda, cudaStream_t st);

// sigma[k] = 2^-e with max(max_i |A_k[i][i]|, |ridge|) in [2^(e-1), 2^e), e clamped to
// [-126, 126]; 1 for a zero or non-finite maximum.  For a symmetric positive
// semidefinite block every |sigma A_k[i][j]| <= 1, so a 16-bit copy neither
// overflows nor loses its large entries to underflow, and the scale is exact.
dash_status launch_diag_pow2_scale(const float* A, float ridge, int dim, long long nblocks,
                                   float* sigma, cudaStream_t st);

// Kernel trace hooks (no-ops unless dash_trace_start was called).
int trace_begin(cudaStream_t st);
void trace_end(int rec, cudaStream_t st, int kind, double flops, double bytes);

// Bounded-wait self-test: a wait on a barrier nothing arrives on.
dash_status launch_wait_selftest(int limit_us, cudaStream_t st);

int gemm_read_clear_error();
int power_tc_read_clear_error();
int power_cluster_read_clear_error();
int elementwise_read_clear_error();

int device_sm_count();

}  // namespace dash
