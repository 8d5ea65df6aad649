// Memory-bound kernels of the preconditioner step: the element-wise prologue
// that scales a block and writes the first iterates in operand format, the
// Frobenius reduction, per-block scale factors, and the bookkeeping kernels of
// the multi-vector power iteration.  All are HBM-bound: 16-byte vector accesses along rows, warp-shuffle
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
      // The element index within the block is below dim^2 <= 2^22: 32-bit arithmetic
      // (a 64-bit division per vector made this loop issue-bound).
      const unsigned q = static_cast<unsigned>(4 * v);
      const int row = static_cast<int>(q / static_cast<unsigned>(p.dim));
      const int col0 = static_cast<int>(q - static_cast<unsigned>(row) * static_cast<unsigned>(p.dim));
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
      const unsigned q = static_cast<unsigned>(4 * v);  // below dim^2 <= 2^22
      const int row = static_cast<int>(q / static_cast<unsigned>(dim));
      const int col0 = static_cast<int>(q - static_cast<unsigned>(row) * static_cast<unsigned>(dim));
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
// The products themselves run on the tensor cores (power_tc.cu); here are the
// start-vector layout change and the final Rayleigh-quotient maximum.
constexpr int PW_NV = 32;

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

// One CTA per chunk of PT_ROWS rows of a block: it reads the chunk's start vectors
// (rows of nv floats, consecutive threads on consecutive floats), transposes them in
// shared memory and writes 32 rows of PT_ROWS 16-bit values (128 contiguous bytes
// each) of Vt.
constexpr int PT_ROWS = 64;

__global__ void __launch_bounds__(256)
    pad_vectors_t_kernel(const float* V0, int nv, int dim, long long nblocks, int bf16,
                         uint16_t* Vt) {
  __shared__ float t[PW_NV][PT_ROWS + 1];
  const int r0 = static_cast<int>(blockIdx.x) * PT_ROWS;
  for (long long b = blockIdx.y; b < nblocks; b += gridDim.y) {
    const float* src = V0 + (b * dim + r0) * nv;
    for (int i = threadIdx.x; i < PT_ROWS * PW_NV; i += blockDim.x) {
      const int rr = i / PW_NV, c = i % PW_NV;
      t[c][rr] = (c < nv) ? src[rr * nv + c] : 0.0f;
    }
    __syncthreads();
    uint16_t* dst = Vt + b * PW_NV * dim + r0;
    for (int i = threadIdx.x; i < PW_NV * PT_ROWS; i += blockDim.x) {
      const int c = i / PT_ROWS, rr = i % PT_ROWS;
      const float x = t[c][rr];
      dst[static_cast<long long>(c) * dim + rr] =
          bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
    }
    __syncthreads();
  }
}

dash_status launch_pad_vectors_t(const float* V0, int nv, int dim, long long nblocks, int bf16,
                                 uint16_t* Vt, cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  if (dim % PT_ROWS != 0 || nv < 1 || nv > PW_NV) return DASH_ERR_INVALID_ARG;
  const int rec = trace_begin(st);
  const dim3 grid(static_cast<unsigned>(dim / PT_ROWS),
                  static_cast<unsigned>(nblocks < 65535 ? nblocks : 65535), 1);
  pad_vectors_t_kernel<<<grid, 256, 0, st>>>(V0, nv, dim, nblocks, bf16, Vt);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_ELEMENTWISE, 0.0,
            static_cast<double>(dim) * nblocks * (4.0 * nv + 2.0 * PW_NV));
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

// ---------------------------------------------------------------- block packing
// A weight-shaped (rows, cols) matrix with leading dimension ld <-> its
// row-block-major stack of b x b blocks (block i * nbc + j holds rows i*b.. and
// columns j*b..), zero-padded beyond the matrix.  Copies of the raw 16- or 32-bit
// words.  Each thread moves one 16-byte vector of V words when cols and ld are
// multiples of V and both buffers are 16-byte aligned (a vector then never straddles
// the matrix edge, since b is a multiple of V too); otherwise one word.
template <typename T, int V>
__global__ void pack_blocks_kernel(const T* M, long long rows, long long cols, long long ld, int b,
                                   long long nbc, long long nb, T* out, int32_t* vr, int32_t* vc) {
  for (long long k = blockIdx.z; k < nb; k += gridDim.z) {
    const long long bi = k / nbc, bj = k - (k / nbc) * nbc;
    const long long r0 = bi * b, c0 = bj * b;
    for (int r = blockIdx.y; r < b; r += gridDim.y) {
      const long long gr = r0 + r;
      T* orow = out + (k * b + r) * static_cast<long long>(b);
      for (int c = (blockIdx.x * blockDim.x + threadIdx.x) * V; c < b;
           c += gridDim.x * blockDim.x * V) {
        const long long gc = c0 + c;
        if (V > 1) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (gr < rows && gc < cols) v = *reinterpret_cast<const uint4*>(M + gr * ld + gc);
          *reinterpret_cast<uint4*>(orow + c) = v;
        } else {
          orow[c] = (gr < rows && gc < cols) ? M[gr * ld + gc] : T(0);
        }
      }
    }
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
      if (vr) vr[k] = static_cast<int32_t>(rows - r0 < b ? rows - r0 : b);
      if (vc) vc[k] = static_cast<int32_t>(cols - c0 < b ? cols - c0 : b);
    }
  }
}

template <typename T, int V>
__global__ void unpack_blocks_kernel(const T* blocks, long long rows, long long cols, long long ld,
                                     int b, long long nbc, T* M) {
  for (long long gr = blockIdx.y; gr < rows; gr += gridDim.y) {
    const long long bi = gr / b;
    const long long r = gr - bi * b;
    for (long long gc = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * V;
         gc < cols; gc += static_cast<long long>(gridDim.x) * blockDim.x * V) {
      const long long bj = gc / b;
      const T* src = blocks + ((bi * nbc + bj) * b + r) * b + (gc - bj * b);
      if (V > 1)
        *reinterpret_cast<uint4*>(M + gr * ld + gc) = *reinterpret_cast<const uint4*>(src);
      else
        M[gr * ld + gc] = *src;
    }
  }
}

static bool vec16_ok(const void* p, const void* q, long long cols, long long ld, int v) {
  return ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(q)) & 15u) == 0 &&
         cols % v == 0 && ld % v == 0;
}

dash_status launch_pack_blocks(const void* M, int esize, long long rows, long long cols,
                               long long ld, int b, void* out, int32_t* vr, int32_t* vc,
                               cudaStream_t st) {
  const long long nbr = (rows + b - 1) / b, nbc = (cols + b - 1) / b, nb = nbr * nbc;
  if (nb <= 0) return DASH_OK;
  const int v = 16 / esize;
  const bool vec = vec16_ok(M, out, cols, ld, v);
  const int per_thread = vec ? v : 1;
  dim3 grid(static_cast<unsigned>((b / per_thread + 127) / 128), b < 65535 ? b : 65535,
            static_cast<unsigned>(nb < 65535 ? nb : 65535));
  const int rec = trace_begin(st);
  if (esize == 2) {
    const uint16_t* m = static_cast<const uint16_t*>(M);
    uint16_t* o = static_cast<uint16_t*>(out);
    if (vec)
      pack_blocks_kernel<uint16_t, 8><<<grid, 128, 0, st>>>(m, rows, cols, ld, b, nbc, nb, o, vr, vc);
    else
      pack_blocks_kernel<uint16_t, 1><<<grid, 128, 0, st>>>(m, rows, cols, ld, b, nbc, nb, o, vr, vc);
  } else {
    const uint32_t* m = static_cast<const uint32_t*>(M);
    uint32_t* o = static_cast<uint32_t*>(out);
    if (vec)
      pack_blocks_kernel<uint32_t, 4><<<grid, 128, 0, st>>>(m, rows, cols, ld, b, nbc, nb, o, vr, vc);
    else
      pack_blocks_kernel<uint32_t, 1><<<grid, 128, 0, st>>>(m, rows, cols, ld, b, nbc, nb, o, vr, vc);
  }
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_PACK, 0.0,
            static_cast<double>(esize) * (static_cast<double>(rows) * cols +
                                          static_cast<double>(nb) * b * b));
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

dash_status launch_unpack_blocks(const void* blocks, int esize, long long rows, long long cols,
                                 long long ld, int b, void* M, cudaStream_t st) {
  const long long nbc = (cols + b - 1) / b;
  if (rows <= 0 || cols <= 0) return DASH_OK;
  const int v = 16 / esize;
  const bool vec = vec16_ok(blocks, M, cols, ld, v);
  const int per_thread = vec ? v : 1;
  const long long gx = (cols / per_thread + 127) / 128;
  dim3 grid(static_cast<unsigned>(gx < 65535 ? gx : 65535),
            static_cast<unsigned>(rows < 65535 ? rows : 65535), 1);
  const int rec = trace_begin(st);
  if (esize == 2) {
    const uint16_t* s = static_cast<const uint16_t*>(blocks);
    uint16_t* m = static_cast<uint16_t*>(M);
    if (vec)
      unpack_blocks_kernel<uint16_t, 8><<<grid, 128, 0, st>>>(s, rows, cols, ld, b, nbc, m);
    else
      unpack_blocks_kernel<uint16_t, 1><<<grid, 128, 0, st>>>(s, rows, cols, ld, b, nbc, m);
  } else {
    const uint32_t* s = static_cast<const uint32_t*>(blocks);
    uint32_t* m = static_cast<uint32_t*>(M);
    if (vec)
      unpack_blocks_kernel<uint32_t, 4><<<grid, 128, 0, st>>>(s, rows, cols, ld, b, nbc, m);
    else
      unpack_blocks_kernel<uint32_t, 1><<<grid, 128, 0, st>>>(s, rows, cols, ld, b, nbc, m);
  }
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_PACK, 0.0, 2.0 * esize * static_cast<double>(rows) * cols);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

__global__ void sub_kernel(const float* a, const float* b, float* out, long long n) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) out[i] = a[i] - b[i];
}

dash_status launch_sub(const float* a, const float* b, float* out, long long n, cudaStream_t st) {
  if (n <= 0) return DASH_OK;
  const int rec = trace_begin(st);
  sub_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(a, b, out, n);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_REDUCE, 0.0, 12.0 * n);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

// Item j of n items of `elems` floats each: dst[j] = src[idx[j]] (gather) or
// dst[idx[j]] = src[j] (scatter).  grid.y walks the items, grid.x the 16-byte
// vectors of one item (single floats when elems is not a multiple of 4).
__global__ void __launch_bounds__(EW_THREADS)
    copy_items_kernel(const float* src, float* dst, const int32_t* idx, int scatter,
                      long long elems, long long n) {
  for (long long j = blockIdx.y; j < n; j += gridDim.y) {
    const long long k = idx[j];
    const float* s = src + (scatter ? j : k) * elems;
    float* d = dst + (scatter ? k : j) * elems;
    if ((elems & 3) == 0) {
      const long long nv = elems >> 2;
      for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < nv;
           v += static_cast<long long>(gridDim.x) * blockDim.x)
        reinterpret_cast<float4*>(d)[v] = reinterpret_cast<const float4*>(s)[v];
    } else {
      for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
           v < elems; v += static_cast<long long>(gridDim.x) * blockDim.x)
        d[v] = s[v];
    }
  }
}

dash_status launch_copy_items(const float* src, float* dst, const int32_t* idx, int scatter,
                              long long elems, long long n, cudaStream_t st) {
  if (n <= 0 || elems <= 0) return DASH_OK;
  const long long nv = (elems & 3) == 0 ? elems / 4 : elems;
  long long gx = (nv + EW_THREADS - 1) / EW_THREADS;
  if (gx > 64) gx = 64;
  // About 8 CTAs per SM over the whole launch.
  long long gy = (static_cast<long long>(device_sm_count()) * 8 + gx - 1) / gx;
  if (gy > n) gy = n;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const int rec = trace_begin(st);
  copy_items_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), EW_THREADS, 0,
                      st>>>(src, dst, idx, scatter, elems, n);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_ELEMENTWISE, 0.0, 8.0 * static_cast<double>(elems) * n);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

// One CTA per block (grid-strided): the largest |diagonal entry| and |ridge|, turned
// into the power of two that brings it into [1/2, 1).
__global__ void __launch_bounds__(EW_THREADS)
    diag_pow2_kernel(const float* A, float ridge, int dim, long long nblocks, float* sigma) {
  __shared__ float red[EW_THREADS / 32];
  const long long dd = static_cast<long long>(dim) * dim;
  for (long long blk = blockIdx.x; blk < nblocks; blk += gridDim.x) {
    float m = fabsf(ridge);
    for (int i = threadIdx.x; i < dim; i += EW_THREADS)
      m = fmaxf(m, fabsf(A[blk * dd + static_cast<long long>(i) * (dim + 1)]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float mx = red[0];
      for (int w = 1; w < EW_THREADS / 32; ++w) mx = fmaxf(mx, red[w]);
      // mx = f 2^e, f in [1/2, 1): the biased exponent field E of a normal mx is e + 126.
      const uint32_t E = (__float_as_uint(mx) >> 23) & 0xffu;
      float s = 1.0f;
      if (E != 0xffu && mx > 0.0f) {
        int e = static_cast<int>(E) - 126;  // a subnormal mx (E = 0) clamps below
        e = e < -126 ? -126 : (e > 126 ? 126 : e);
        s = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, a normal float
      }
      sigma[blk] = s;
    }
    __syncthreads();
  }
}

dash_status launch_diag_pow2_scale(const float* A, float ridge, int dim, long long nblocks,
                                   float* sigma, cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  const long long cap = static_cast<long long>(device_sm_count()) * 16;
  const long long grid = nblocks < cap ? nblocks : (cap > 0 ? cap : 1);
  const int rec = trace_begin(st);
  diag_pow2_kernel<<<static_cast<unsigned>(grid), EW_THREADS, 0, st>>>(A, ridge, dim, nblocks, sigma);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_REDUCE, 0.0, 4.0 * dim * nblocks + 4.0 * nblocks);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

__global__ void power_finish_kernel(const float* num, const float* den, int nv, long long nblocks,
                                    const float* blk_scale, float* lambda) {
  const long long k = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= nblocks) return;
  float best = -INFINITY;
  for (int c = 0; c < nv; ++c) best = fmaxf(best, num[k * PW_NV + c] / den[k * PW_NV + c]);
  // A power-of-two scale divides out exactly.
  lambda[k] = (blk_scale != nullptr) ? best / blk_scale[k] : best;
}

dash_status launch_power_finish(const float* num, const float* den, int nv, long long nblocks,
                                const float* blk_scale, float* lambda, cudaStream_t st) {
  if (nblocks <= 0) return DASH_OK;
  const int rec = trace_begin(st);
  power_finish_kernel<<<static_cast<unsigned>((nblocks + 127) / 128), 128, 0, st>>>(
      num, den, nv, nblocks, blk_scale, lambda);
  const cudaError_t err = cudaGetLastError();
  trace_end(rec, st, DASH_TRACE_REDUCE, 0.0, 8.0 * 32 * nblocks);
  return err == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

// ---------------------------------------------------------------- wait self-test
// One thread waits, with the given limit, on an mbarrier that nothing arrives
// on; when the limit runs out it records DEV_ERR_TIMEOUT and returns -- the
// same path every pipeline wait of the library takes.
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(b, 0)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicExch(&g_dash_error, DEV_ERR_TIMEOUT);
      return;
    }
  }
}

dash_status launch_wait_selftest(int limit_us, cudaStream_t st) {
  wait_selftest_kernel<<<1, 1, 0, st>>>(static_cast<unsigned long long>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

}  // namespace dash
