// Memory-bound kernels of the preconditioner step: the element-wise prologue
// that scales a block and writes the first iterates in operand format, the
// Frobenius reduction, per-block scale factors, and the multi-vector power
// iteration.  All are HBM-bound: 16-byte vector accesses along rows, warp-shuffle
// reductions, one atomic per CTA and block for the per-block sums.
#include <cmath>

#include "dash_common.cuh"
#include "dash_internal.h"

namespace dash {

int elementwise_read_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_dash_error, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_dash_error, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Block-wide sum of v over 256 threads; result valid in thread 0.
__device__ __forceinline__ float block_sum256(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.0f;
  if (threadIdx.x < 32) {
    s = (l < 8) ? red[l] : 0.0f;
    s = warp_sum(s);
  }
  __syncthreads();
  return s;
}

constexpr int EW_THREADS = 256;
constexpr int EW_VEC_PER_THREAD = 8;

// grid.x: chunks of one block, grid.y: blocks (strided over nblocks).
__global__ void __launch_bounds__(EW_THREADS) affine_kernel(const __grid_constant__ AffParams p) {
  __shared__ float red[8];
  const long long dd = static_cast<long long>(p.dim) * p.dim;
  const long long n4 = dd / 4;
  for (long long blk = blockIdx.y; blk < p.nblocks; blk += gridDim.y) {
    const float inv_s = (p.inv_s != nullptr) ? p.inv_s[blk] : 1.0f;
    float mult[3];
#pragma unroll
    for (int o = 0; o < 3; ++o)
      mult[o] = (o < p.nout && p.out[o].mult != nullptr) ? p.out[o].mult[blk] : 1.0f;
    float rsum = 0.0f;
    for (long long v = static_cast<long long>(blockIdx.x) * EW_THREADS + threadIdx.x; v < n4;
         v += static_cast<long long>(gridDim.x) * EW_THREADS) {
      const long long e = blk * dd + 4 * v;
      const int row = static_cast<int>((4 * v) / p.dim);
      const int col0 = static_cast<int>((4 * v) % p.dim);
      float x[4];
      load4(p.src_fmt, p.src_hi, p.src_lo, e, x);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool diag = (row == col0 + j);
        x[j] = (x[j] + (diag ? p.ridge : 0.0f)) * inv_s;
        if (p.resid_acc != nullptr) {
          const float d = x[j] - (diag ? 1.0f : 0.0f);
          rsum = fmaf(d, d, rsum);
        }
      }
#pragma unroll
      for (int o = 0; o < 3; ++o) {
        if (o < p.nout) {
          float d[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float t = p.out[o].alpha * x[j];
            if (row == col0 + j) t += p.out[o].gamma;
            d[j] = t * mult[o];
          }
          store4(p.out[o].fmt, p.out[o].hi, p.out[o].lo, e, d);
        }
      }
    }
    if (p.resid_acc != nullptr) {
      const float s = block_sum256(rsum, red);
      if (threadIdx.x == 0) atomicAdd(p.resid_acc + blk * p.resid_stride, s);
    }
  }
}

static dim3 ew_grid(int dim, long long nblocks) {
  const long long n4 = static_cast<long long>(dim) * dim / 4;
  long long gx = (n4 + EW_THREADS * EW_VEC_PER_THREAD - 1) / (EW_THREADS * EW_VEC_PER_THREAD);
  if (gx < 1) gx = 1;
  const long long gy = nblocks < 65535 ? nblocks : 65535;
  return dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
}

dash_status launch_affine(const AffParams& p, cudaStream_t st) {
  if (p.nblocks <= 0) return DASH_OK;
  const int rec = trace_begin(st);
  affine_kernel<<<ew_grid(p.dim, p.nblocks), EW_THREADS, 0, st>>>(p);
  const cudaError_t err = cudaGetLastError();
  if (rec >= 0) {
    const double bb = static_cast<double>(p.dim) * p.dim * p.nblocks;
    double bytes = bb * fmt_bytes(p.src_fmt);
    for (int o = 0; o < p.nout; ++o) bytes += bb * fmt_bytes(p.out[o].fmt);
    trace_end(rec, st, DASH_TRACE_ELEMENTWISE, 0.0, bytes);
  }
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

__global__ void scale_factors_kernel(const float* s, float* inv_s, float* s_m14, long long n) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const double v = static_cast<double>(s[i]);
  inv_s[i] = static_cast<float>(1.0 / v);
  s_m14[i] = static_cast<float>(pow(v, -0.25));
}

dash_status launch_scale_factors(const float* s, float* inv_s, float* s_m14, long long n,
                                 cudaStream_t st) {
  if (n <= 0) return DASH_OK;
  const int rec = trace_begin(st);
  scale_factors_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(s, inv_s, s_m14, n);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_REDUCE, 0.0, 12.0 * n);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

__global__ void sqrt_scale_kernel(const float* acc, float* out, long long n, float mul) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) out[i] = sqrtf(acc[i]) * mul;
}

dash_status launch_sqrt_scale(const float* acc, float* out, long long n, float mul,
                              cudaStream_t st) {
  if (n <= 0) return DASH_OK;
  const int rec = trace_begin(st);
  sqrt_scale_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(acc, out, n, mul);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_REDUCE, 0.0, 8.0 * n);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

__global__ void __launch_bounds__(EW_THREADS)
    frob_kernel(const float* A, float ridge, int dim, long long nblocks, float* acc) {
  __shared__ float red[8];
  const long long dd = static_cast<long long>(dim) * dim;
  const long long n4 = dd / 4;
  for (long long blk = blockIdx.y; blk < nblocks; blk += gridDim.y) {
    float s = 0.0f;
    for (long long v = static_cast<long long>(blockIdx.x) * EW_THREADS + threadIdx.x; v < n4;
         v += static_cast<long long>(gridDim.x) * EW_THREADS) {
      const float4 a = *reinterpret_cast<const float4*>(A + blk * dd + 4 * v);
      const int row = static_cast<int>((4 * v) / dim);
      const int col0 = static_cast<int>((4 * v) % dim);
      float x[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float t = x[j] + ((row == col0 + j) ? ridge : 0.0f);
        s = fmaf(t, t, s);
      }
    }
    s = block_sum256(s, red);
    if (threadIdx.x == 0) atomicAdd(acc + blk, s);
  }
}

dash_status launch_frob_acc(const float* A, float ridge, int dim, long long nblocks, float* acc,
                            cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  const int rec = trace_begin(st);
  frob_kernel<<<ew_grid(dim, nblocks), EW_THREADS, 0, st>>>(A, ridge, dim, nblocks, acc);
  const cudaError_t err = cudaGetLastError();
  const double bb = static_cast<double>(dim) * dim * nblocks;
  trace_end(rec, st, DASH_TRACE_REDUCE, 2.0 * bb, 4.0 * bb);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

// ---------------------------------------------------------------- power iteration
// W = (A + ridge I) V for every block, V being B x 32 (n_v <= 32 used columns,
// stored with a row stride of 32; the previous step's column norms are applied
// as W = (A V_raw) D + ridge V_raw D, D = diag(1/||column||)).
// One CTA owns R = min(B, 512) rows of one block (rows a multiple of R/8 apart
// share a thread), R/2 threads, each with an 8 rows x 8 vectors register tile.
// A and V stream through shared memory in 16-column chunks with cp.async,
// double-buffered.  Per column of A a thread does 8 scalar shared loads
// (conflict-free: its warp's 8 rows are consecutive and the staged row stride is
// 20 words) and two float4 loads of V for 64 FMAs.
constexpr int PW_NV = 32;
constexpr int PW_KC = 16;
constexpr int PW_STRIDE = 20;  // words per staged row of A (16 used, 16-byte aligned)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all_but_one() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__global__ void __launch_bounds__(256)
    power_step_kernel(const float* A, float ridge, int dim, long long nblocks, const float* Vin,
                      int vin_stride, int nv, const float* in_nrm2, float* Wout, float* acc0,
                      float* acc1, int last, int rows) {
  extern __shared__ __align__(16) float pw_smem[];
  float* As = pw_smem;                                    // [2][rows][PW_STRIDE]
  float* Vs = pw_smem + 2 * rows * PW_STRIDE;             // [2][PW_KC][PW_NV]
  __shared__ float vscale[PW_NV];
  __shared__ float red0[8][PW_NV];
  __shared__ float red1[8][PW_NV];

  const long long blk = blockIdx.y;
  const int r0 = blockIdx.x * rows;
  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;  // rows / 2
  const int groups = rows / 8;      // row groups; group g owns rows g + groups * i
  const int cg = tid & 3;           // vector columns 8cg .. 8cg+7
  const int g = tid >> 2;
  const long long dd = static_cast<long long>(dim) * dim;
  const float* Ab = A + blk * dd + static_cast<long long>(r0) * dim;
  const float* Vb = Vin + blk * static_cast<long long>(dim) * PW_NV;
  (void)vin_stride;

  if (tid < PW_NV) {
    float sc = 0.0f;
    if (tid < nv) sc = (in_nrm2 != nullptr) ? 1.0f / sqrtf(in_nrm2[blk * PW_NV + tid]) : 1.0f;
    vscale[tid] = sc;
  }
  __syncthreads();

  // Stage chunk kc into buffer b: A rows r0..r0+rows-1 and V rows kc..kc+15,
  // columns kc..kc+15 of A; all with 16-byte cp.async.
  auto stage = [&](int b, int kc) {
    float* Ad = As + b * rows * PW_STRIDE;
    const int nvec = rows * (PW_KC / 4);
    for (int f = tid; f < nvec; f += nthreads) {
      const int r = f >> 2, q = f & 3;
      cp_async16(Ad + r * PW_STRIDE + 4 * q, Ab + static_cast<long long>(r) * dim + kc + 4 * q);
    }
    float* Vd = Vs + b * PW_KC * PW_NV;
    for (int f = tid; f < PW_KC * PW_NV / 4; f += nthreads)
      cp_async16(Vd + 4 * f, Vb + static_cast<long long>(kc) * PW_NV + 4 * f);
    cp_async_commit();
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  const int nchunks = dim / PW_KC;
  stage(0, 0);
  for (int ch = 0; ch < nchunks; ++ch) {
    const int b = ch & 1;
    if (ch + 1 < nchunks) {
      stage(b ^ 1, (ch + 1) * PW_KC);
      cp_async_wait_all_but_one();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    const float* Ac = As + b * rows * PW_STRIDE;
    const float* Vc = Vs + b * PW_KC * PW_NV;
#pragma unroll
    for (int k = 0; k < PW_KC; ++k) {
      float a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = Ac[(g + groups * i) * PW_STRIDE + k];
      const float4 v0 = *reinterpret_cast<const float4*>(Vc + k * PW_NV + 8 * cg);
      const float4 v1 = *reinterpret_cast<const float4*>(Vc + k * PW_NV + 8 * cg + 4);
      const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], v[j], acc[i][j]);
    }
    __syncthreads();
  }

  // Ridge term, output and per-column statistics.
  float s0[8], s1[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    s0[j] = 0.0f;
    s1[j] = 0.0f;
  }
  float sc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) sc[j] = vscale[8 * cg + j];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = r0 + g + groups * i;
    const float* vr = Vb + static_cast<long long>(row) * PW_NV + 8 * cg;
    const float4 va = *reinterpret_cast<const float4*>(vr);
    const float4 vb = *reinterpret_cast<const float4*>(vr + 4);
    const float vraw[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
    float w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float v = vraw[j] * sc[j];
      w[j] = fmaf(ridge, v, acc[i][j] * sc[j]);
      if (last) {
        s0[j] = fmaf(v, w[j], s0[j]);
        s1[j] = fmaf(v, v, s1[j]);
      } else {
        s0[j] = fmaf(w[j], w[j], s0[j]);
      }
    }
    if (!last) {
      float* o = Wout + blk * static_cast<long long>(dim) * PW_NV +
                 static_cast<long long>(row) * PW_NV + 8 * cg;
      *reinterpret_cast<float4*>(o) = make_float4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<float4*>(o + 4) = make_float4(w[4], w[5], w[6], w[7]);
    }
  }
  // Lanes cg, cg+4, ..., cg+28 hold the same columns.
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      s0[j] += __shfl_xor_sync(0xffffffffu, s0[j], off);
      s1[j] += __shfl_xor_sync(0xffffffffu, s1[j], off);
    }
  }
  const int w = tid >> 5, l = tid & 31;
  const int nwarps = nthreads >> 5;
  if (l < 4) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      red0[w][8 * l + j] = s0[j];
      red1[w][8 * l + j] = s1[j];
    }
  }
  __syncthreads();
  if (tid < PW_NV && tid < nv) {
    float a = 0.f, b = 0.f;
    for (int i = 0; i < nwarps; ++i) {
      a += red0[i][tid];
      b += red1[i][tid];
    }
    atomicAdd(acc0 + blk * PW_NV + tid, a);
    if (last) atomicAdd(acc1 + blk * PW_NV + tid, b);
  }
}

// V[blk][r][c] = V0[blk][r][c] for c < nv, 0 for nv <= c < 32.
__global__ void pad_vectors_kernel(const float* V0, int nv, long long rows_total, float* V) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows_total * PW_NV) return;
  const long long r = i >> 5;
  const int c = static_cast<int>(i & 31);
  V[i] = (c < nv) ? V0[r * nv + c] : 0.0f;
}

dash_status launch_pad_vectors(const float* V0, int nv, int dim, long long nblocks, float* V,
                               cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  const long long n = static_cast<long long>(dim) * nblocks * PW_NV;
  const int rec = trace_begin(st);
  pad_vectors_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
      V0, nv, static_cast<long long>(dim) * nblocks, V);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_ELEMENTWISE, 0.0, 4.0 * static_cast<double>(dim) * nblocks * (nv + 32));
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

static int power_rows(int dim) {
  if (dim % 512 == 0) return 512;
  if (dim % 256 == 0) return 256;
  return 128;
}

dash_status launch_power_step(const float* A, float ridge, int dim, long long nblocks,
                              const float* Vin, int vin_stride, int nv, const float* in_nrm2,
                              float* Wout, float* acc0, float* acc1, int last, cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  if (nblocks > 65535) return DASH_ERR_INVALID_ARG;
  const int rows = power_rows(dim);
  const size_t smem = (2 * static_cast<size_t>(rows) * PW_STRIDE + 2 * PW_KC * PW_NV) * 4;
  if (cudaFuncSetAttribute(power_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DASH_ERR_CUDA;
  dim3 grid(dim / rows, static_cast<unsigned>(nblocks), 1);
  const int rec = trace_begin(st);
  power_step_kernel<<<grid, rows / 2, smem, st>>>(A, ridge, dim, nblocks, Vin, vin_stride, nv,
                                                  in_nrm2, Wout, acc0, acc1, last, rows);
  const cudaError_t err = cudaGetLastError();
  const double bb = static_cast<double>(dim) * dim * nblocks;
  const double vb = static_cast<double>(dim) * nblocks * 4.0;
  trace_end(rec, st, DASH_TRACE_POWER, 2.0 * bb * nv, 4.0 * bb + vb * (32 + (last ? 0 : 32)));
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

__global__ void power_finish_kernel(const float* num, const float* den, int nv, long long nblocks,
                                    float* lambda) {
  const long long k = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= nblocks) return;
  float best = -INFINITY;
  for (int c = 0; c < nv; ++c) best = fmaxf(best, num[k * PW_NV + c] / den[k * PW_NV + c]);
  lambda[k] = best;
}

dash_status launch_power_finish(const float* num, const float* den, int nv, long long nblocks,
                                float* lambda, cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  const int rec = trace_begin(st);
  power_finish_kernel<<<static_cast<unsigned>((nblocks + 127) / 128), 128, 0, st>>>(num, den, nv,
                                                                                    nblocks, lambda);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_REDUCE, 0.0, 8.0 * 32 * nblocks);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

}  // namespace dash
