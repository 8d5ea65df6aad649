// C-ABI entry points of dashroot: argument checks, workspace carving, chunking
// over the block stack, and the launch sequences of the four hot-path steps.
// The arithmetic lives in gemm_tc.cu (dense products, fused epilogues) and
// elementwise.cu (prologues, reductions, power iteration).
#include <cmath>
#include <limits>
#include <cstring>
#include <vector>

#include "dash_common.cuh"
#include "dash_internal.h"
#include "dashroot.h"

using namespace dash;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dim(int B) { return B >= 128 && B <= 2048 && (B % 128) == 0; }

bool valid_prec(int prec) { return prec >= DASH_FP32_3XTF32 && prec <= DASH_BF16; }

// Splits a root solver's prec argument into the arithmetic and the format of X
// (DASH_ROOT_TF32: X rounded to TF32).  False for an unknown flag or precision.
bool root_prec(int& prec, int& xfmt) {
  if (prec & ~(0xff | DASH_ROOT_TF32)) return false;
  xfmt = (prec & DASH_ROOT_TF32) ? FMT_TF32 : FMT_F32;
  prec &= 0xff;
  return valid_prec(prec);
}

int prec_fmt(int prec) {
  switch (prec) {
    case DASH_FP32_3XTF32: return FMT_SPLIT;
    case DASH_TF32: return FMT_TF32;
    case DASH_FP16: return FMT_F16;
    default: return FMT_BF16;
  }
}

int prec_kind(int prec) {
  switch (prec) {
    case DASH_FP32_3XTF32: return KIND_TF32X3;
    case DASH_TF32: return KIND_TF32;
    case DASH_FP16: return KIND_F16;
    default: return KIND_BF16;
  }
}

// Bytes one B x B operand-format matrix takes (both halves for the split format).
size_t operand_bytes(int prec, int B) {
  const size_t e = (prec == DASH_FP32_3XTF32) ? 8 : (prec == DASH_TF32 ? 4 : 2);
  return e * static_cast<size_t>(B) * B;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A stack of nblocks operand-format matrices inside the workspace.
struct Buf {
  void* hi = nullptr;
  void* lo = nullptr;
};

struct Carver {
  char* p;
  size_t left;
  bool ok = true;
  Carver(void* ws, size_t bytes) : p(static_cast<char*>(ws)), left(bytes) {}
  void* take(size_t bytes) {
    bytes = round256(bytes);
    if (bytes > left || p == nullptr) {
      ok = false;
      return nullptr;
    }
    void* r = p;
    p += bytes;
    left -= bytes;
    return r;
  }
  Buf take_buf(int prec, int B, long long nblk) {
    Buf b;
    const size_t elems = static_cast<size_t>(B) * B * nblk;
    if (prec == DASH_FP32_3XTF32) {
      b.hi = take(elems * 4);
      b.lo = take(elems * 4);
    } else {
      b.hi = take(elems * (prec == DASH_TF32 ? 4 : 2));
    }
    return b;
  }
  // A 16-bit precision's buffer with room for a lo part (the pair formats).
  Buf take_pair16(int B, long long nblk) {
    Buf b;
    const size_t elems = static_cast<size_t>(B) * B * nblk;
    b.hi = take(elems * 2);
    b.lo = take(elems * 2);
    return b;
  }
};

bool is_half(int prec) { return prec == DASH_FP16 || prec == DASH_BF16; }

// Per-block bytes of the operand buffers, rounded the way the carver rounds
// them when a chunk holds nblk blocks (used to size chunks).
size_t bufs_bytes(int prec, int B, long long nblk, int nbufs) {
  const size_t elems = static_cast<size_t>(B) * B * nblk;
  size_t one = (prec == DASH_FP32_3XTF32) ? 2 * round256(elems * 4)
                                          : round256(elems * (prec == DASH_TF32 ? 4 : 2));
  return one * nbufs;
}

// Largest chunk (<= N blocks) whose operand buffers fit in `avail` bytes.
long long fit_chunk(int prec, int B, long long N, int nbufs, size_t avail) {
  if (nbufs == 0) return N;
  const size_t per = operand_bytes(prec, B) * nbufs;
  long long c = static_cast<long long>(avail / per);
  if (c > N) c = N;
  while (c > 0 && bufs_bytes(prec, B, c, nbufs) > avail) --c;
  return c;
}

template <typename T>
T* offset_blocks(T* p, long long blocks, int B, size_t esize) {
  return reinterpret_cast<T*>(reinterpret_cast<char*>(p) +
                              static_cast<size_t>(blocks) * B * B * esize);
}

template <typename T>
const T* offset_blocks(const T* p, long long blocks, int B, size_t esize) {
  return reinterpret_cast<const T*>(reinterpret_cast<const char*>(p) +
                                    static_cast<size_t>(blocks) * B * B * esize);
}

#define DASH_TRY(expr)                \
  do {                                \
    dash_status _s = (expr);          \
    if (_s != DASH_OK) return _s;     \
  } while (0)

EpiParams epi_none() {
  EpiParams e;
  std::memset(&e, 0, sizeof(e));
  return e;
}

EpiOut eout(const Buf& b, int fmt, float alpha, float gamma, float eps = 0.0f,
            const float* mult = nullptr) {
  EpiOut o;
  o.hi = b.hi;
  o.lo = b.lo;
  o.mult = mult;
  o.alpha = alpha;
  o.gamma = gamma;
  o.eps = eps;
  o.fmt = fmt;
  return o;
}

// Sets the epilogue's E operand to the buffer b (in format fmt).
void with_e(EpiParams& e, const Buf& b, int fmt) {
  e.E_hi = b.hi;
  e.E_lo = b.lo;
  e.E_fmt = fmt;
}

EpiOut eout_f32(float* p, float alpha, float gamma, float eps, const float* mult) {
  Buf b;
  b.hi = p;
  return eout(b, FMT_F32, alpha, gamma, eps, mult);
}

AffOut aout(const Buf& b, int fmt, float alpha, float gamma, const float* mult = nullptr) {
  AffOut o;
  o.hi = b.hi;
  o.lo = b.lo;
  o.mult = mult;
  o.alpha = alpha;
  o.gamma = gamma;
  o.fmt = fmt;
  return o;
}

AffParams aff_from(const void* src_hi, const void* src_lo, int src_fmt, int B, long long n) {
  AffParams a;
  std::memset(&a, 0, sizeof(a));
  a.src_hi = src_hi;
  a.src_lo = src_lo;
  a.src_fmt = src_fmt;
  a.dim = B;
  a.nblocks = n;
  return a;
}

// One GEMM launch C = X * Y over nc blocks in precision prec.
// sym: 0 plain; 1 symmetric operands (only their tiles on or above the diagonal
// are read); 2 also a symmetric result (only those tiles computed and stored);
// 3 a symmetric result from operands read whole (X Y^T with Y = X, or X^T X);
// 4 X symmetric (read from its upper tiles), Y and the result whole.
// Modes 1-4 take effect for B a multiple of 256 (CTA-pair kernels).
// pairB: Y is a 16-bit pair (FMT_F16X2 / FMT_BF16X2) of the 16-bit precision prec.
dash_status gemm(int prec, int B, long long nc, const Buf& X, int tX, const Buf& Y, int tY,
                 const EpiParams& e, cudaStream_t st, int sym = 0, bool pairB = false) {
  GemmLaunch g;
  g.sym_in = (sym == 1 || sym == 2 || sym == 4) ? 1 : 0;
  g.sym_in_b = (sym == 1 || sym == 2) ? 1 : 0;
  g.sym_out = (sym == 2 || sym == 3) ? 1 : 0;
  g.kind = prec_kind(prec);
  if (pairB) g.kind = (prec == DASH_BF16) ? KIND_BF16_SPLITB : KIND_F16_SPLITB;
  g.dim = B;
  g.nblocks = nc;
  g.A = X.hi;
  g.A_lo = X.lo;
  g.transA = tX;
  g.B = Y.hi;
  g.B_lo = Y.lo;
  g.transB = tY;
  g.epi = e;
  return launch_gemm(g, st);
}

// Whether a root solver may keep its iterates as symmetric halves: every iterate
// is a polynomial in the symmetric A, so each product of two is symmetric.  The
// CTA-pair kernels (B a multiple of 256) honour it in every precision.  Used by
// Coupled Newton and Chebyshev; Newton-Denman-Beavers keeps full products.
#ifndef DASH_SYM_HALVES
#define DASH_SYM_HALVES 1  // build-time: 0 computes every product whole
#endif
int sym_mode(int prec, int B) {
  (void)prec;
  return (DASH_SYM_HALVES && B % 256 == 0) ? 2 : 0;
}

// Small per-call arrays shared by the root solvers.
struct RootSmall {
  float* inv_s;
  float* s_m14;
  float* racc;
};

size_t root_small_bytes(long long N, long long nres) {
  return round256(N * 4) * 2 + round256(static_cast<size_t>(nres > 0 ? nres : 1) * 4);
}

dash_status common_root_checks(const float* A, const float* scale, long long N, int B, int iters,
                               int prec, const float* X, const void* ws) {
  if (N < 0 || !valid_dim(B) || !valid_prec(prec) || iters < 1) return DASH_ERR_INVALID_ARG;
  if (N == 0) return DASH_OK;
  if (!A || !scale || !X || !aligned16(A) || !aligned16(X) || !aligned16(scale))
    return DASH_ERR_INVALID_ARG;
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return DASH_ERR_INVALID_ARG;
  return DASH_OK;
}

constexpr int CN_BUFS = 7;
// The two M iterates of a 16-bit Coupled Newton carry a lo part: two more arrays.
int cn_bufs(int prec) { return is_half(prec) ? CN_BUFS + 2 : CN_BUFS; }

// M-update products of a 16-bit Coupled Newton of K iterations that read M as a
// 16-bit pair (hi + lo); the last three read it plain.  The root is sensitive to
// the rounding of M in proportion to how much the remaining iterations amplify
// its small eigenvalues (about (5/4)^4 per iteration), so only the early updates
// need M's extra bits.
#ifndef DASH_CN_PAIR_TAIL
#define DASH_CN_PAIR_TAIL 4  // M-updates at the end of the iteration that read M plain, + 1
#endif
int cn_pair_updates(int prec, int K) {
  return is_half(prec) ? (K > DASH_CN_PAIR_TAIL ? K - DASH_CN_PAIR_TAIL : 0) : 0;
}
constexpr int NDB_BUFS = 6;
constexpr int CHEB_BUFS = 4;
constexpr int APPLY_BUFS = 4;

}  // namespace

// ============================================================================ API

extern "C" {

const char* dash_status_string(int s) {
  switch (s) {
    case DASH_OK: return "DASH_OK";
    case DASH_ERR_INVALID_ARG: return "DASH_ERR_INVALID_ARG: invalid argument";
    case DASH_ERR_UNSUPPORTED: return "DASH_ERR_UNSUPPORTED: unsupported configuration";
    case DASH_ERR_CUDA: return "DASH_ERR_CUDA: CUDA runtime or launch error";
    case DASH_ERR_WORKSPACE_TOO_SMALL: return "DASH_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case DASH_ERR_TIMEOUT: return "DASH_ERR_TIMEOUT: a device-side wait timed out";
    case DASH_ERR_CONFLICT:
      return "DASH_ERR_CONFLICT: too many product launches in flight across streams";
    default: return "unknown dash_status";
  }
}

const char* dash_version(void) { return "dashroot 0.1 sm_103a"; }

dash_status dash_device_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return DASH_ERR_CUDA;
  const int a = gemm_read_clear_error();
  const int b = elementwise_read_clear_error();
  const int c = power_tc_read_clear_error();
  const int d = power_cluster_read_clear_error();
  if (a < 0 || b < 0 || c < 0 || d < 0) return DASH_ERR_CUDA;
  if (a == DASH_ERR_TIMEOUT || b == DASH_ERR_TIMEOUT || c == DASH_ERR_TIMEOUT ||
      d == DASH_ERR_TIMEOUT)
    return DASH_ERR_TIMEOUT;
  if (a == DASH_ERR_CONFLICT) return DASH_ERR_CONFLICT;
  return DASH_OK;
}

dash_status dash_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return DASH_ERR_INVALID_ARG;
  return launch_wait_selftest(limit_us, static_cast<cudaStream_t>(stream));
}

int64_t dash_op_matmuls(int op, int param) {
  switch (op) {
    case DASH_OP_ACCUMULATE: return 2;  // one per factor, L and R
    case DASH_OP_INV_ROOT_CN: return param <= 1 ? 0 : 4LL * param - 4;
    case DASH_OP_INV_ROOT_NDB: return param <= 1 ? 1 : 6LL * param - 6;
    case DASH_OP_INV_ROOT_CHEB: return param <= 1 ? 0 : param - 1;
    case DASH_OP_PRECONDITION_APPLY: return 2;
    default: return 0;
  }
}

dash_status dash_workspace_size(int op, int64_t N, int B, int prec, int param, size_t* bytes) {
  prec &= ~DASH_ROOT_TF32;  // moves a rounding step only: same workspace
  if (!bytes || N < 0 || !valid_dim(B) || !valid_prec(prec)) return DASH_ERR_INVALID_ARG;
  size_t s = 0;
  switch (op) {
    case DASH_OP_ACCUMULATE:
      // fp32 gradients are split into TF32 hi/lo (prec DASH_FP32_3XTF32); others need none.
      s = (prec == DASH_FP32_3XTF32) ? bufs_bytes(DASH_FP32_3XTF32, B, N, 1) : 0;
      break;
    case DASH_OP_SPECTRAL_SCALE:
      if (prec == DASH_FP16 || prec == DASH_BF16)  // the half-precision power modes
        s = round256(static_cast<size_t>(N) * B * B * 2) +
            2 * round256(static_cast<size_t>(N) * B * 32 * 2) + 3 * round256(N * 32 * 4) +
            round256(N * 4) + 256;
      else
        s = 2 * round256(static_cast<size_t>(N) * B * 32 * 4) + 3 * round256(N * 32 * 4) + 256;
      break;
    case DASH_OP_INV_ROOT_CN:
      s = root_small_bytes(N, N * (param > 0 ? param : 1)) + bufs_bytes(prec, B, N, cn_bufs(prec));
      break;
    case DASH_OP_INV_ROOT_NDB:
      s = root_small_bytes(N, 2 * N * (param > 0 ? param : 1)) + bufs_bytes(prec, B, N, NDB_BUFS);
      break;
    case DASH_OP_INV_ROOT_CHEB:
      s = root_small_bytes(N, 0) + bufs_bytes(prec, B, N, CHEB_BUFS);
      break;
    case DASH_OP_PRECONDITION_APPLY:
      s = bufs_bytes(prec, B, N, APPLY_BUFS);
      break;
    case DASH_OP_LAMBDA_MIN: {
      // The shifted stack, 1/c_k and mu_k, and spectral_scale's workspace.
      size_t sc = 0;
      DASH_TRY(dash_workspace_size(DASH_OP_SPECTRAL_SCALE, N, B, prec, param, &sc));
      s = round256(static_cast<size_t>(N) * B * B * 4) + 2 * round256(N * 4) + round256(sc) + 256;
      break;
    }
    default:
      return DASH_ERR_INVALID_ARG;
  }
  *bytes = s;
  return DASH_OK;
}

dash_status dash_gemm(const void* A, const void* A_lo, int trans_a, const void* Bm,
                      const void* B_lo, int trans_b, int64_t N, int B, int prec, float* C,
                      void* stream) {
  if (N < 0 || !valid_dim(B) || !valid_prec(prec)) return DASH_ERR_INVALID_ARG;
  if (N == 0) return DASH_OK;
  if (!A || !Bm || !C || !aligned16(A) || !aligned16(Bm) || !aligned16(C))
    return DASH_ERR_INVALID_ARG;
  if (prec == DASH_FP32_3XTF32 && (!A_lo || !B_lo || !aligned16(A_lo) || !aligned16(B_lo)))
    return DASH_ERR_INVALID_ARG;
  Buf X, Y;
  X.hi = const_cast<void*>(A);
  X.lo = const_cast<void*>(A_lo);
  Y.hi = const_cast<void*>(Bm);
  Y.lo = const_cast<void*>(B_lo);
  EpiParams e = epi_none();
  e.nout = 1;
  e.out[0] = eout_f32(C, 1.0f, 0.0f, 0.0f, nullptr);
  return gemm(prec, B, N, X, trans_a, Y, trans_b, e, static_cast<cudaStream_t>(stream));
}

dash_status dash_gemm_ex(const void* A, const void* A_lo, int trans_a, const void* Bm,
                         const void* B_lo, int trans_b, int64_t N, int B, int prec, int sym,
                         float* C, void* stream) {
  if (N < 0 || !valid_dim(B) || !valid_prec(prec) || sym < 0 || sym > 4)
    return DASH_ERR_INVALID_ARG;
  if (N == 0) return DASH_OK;
  if (!A || !Bm || !C || !aligned16(A) || !aligned16(Bm) || !aligned16(C))
    return DASH_ERR_INVALID_ARG;
  if (prec == DASH_FP32_3XTF32 && (!A_lo || !B_lo || !aligned16(A_lo) || !aligned16(B_lo)))
    return DASH_ERR_INVALID_ARG;
  const bool pair = is_half(prec) && B_lo != nullptr;
  if (pair && !aligned16(B_lo)) return DASH_ERR_INVALID_ARG;
  Buf X, Y;
  X.hi = const_cast<void*>(A);
  X.lo = const_cast<void*>(A_lo);
  Y.hi = const_cast<void*>(Bm);
  Y.lo = const_cast<void*>(B_lo);
  EpiParams e = epi_none();
  e.nout = 1;
  e.out[0] = eout_f32(C, 1.0f, 0.0f, 0.0f, nullptr);
  return gemm(prec, B, N, X, trans_a, Y, trans_b, e, static_cast<cudaStream_t>(stream), sym, pair);
}

// ---------------------------------------------------------------- accumulate

dash_status shampoo_accumulate(const void* G, int gdt, int64_t Ng, int B, float beta, float* F,
                               const int32_t* valid_rows, const int32_t* valid_cols, void* ws,
                               size_t ws_bytes, void* stream) {
  if (Ng < 0 || !valid_dim(B) || !(gdt == DASH_DT_F32 || gdt == DASH_DT_BF16 || gdt == DASH_DT_F16))
    return DASH_ERR_INVALID_ARG;
  if (!(beta >= 0.0f && beta <= 1.0f)) return DASH_ERR_INVALID_ARG;
  if (Ng == 0) return DASH_OK;
  if (!G || !F || !aligned16(G) || !aligned16(F)) return DASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int gprec = (gdt == DASH_DT_F32) ? DASH_FP32_3XTF32 : (gdt == DASH_DT_BF16 ? DASH_BF16 : DASH_FP16);
  long long chunk = Ng;
  Buf split;
  if (gdt == DASH_DT_F32) {
    if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return DASH_ERR_INVALID_ARG;
    chunk = fit_chunk(gprec, B, Ng, 1, ws ? ws_bytes : 0);
    if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
    Carver cv(ws, ws_bytes);
    split = cv.take_buf(gprec, B, chunk);
    if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  }
  const size_t gsz = (gdt == DASH_DT_F32) ? 4 : 2;
  // G G^T and G^T G are symmetric, and so is every factor: for B a multiple of 256
  // only the 256-tiles on or above the diagonal are computed (reading those of the
  // old F); the epilogue also stores each one transposed into its mirror below.
  const int SO = (B % 256 == 0) ? 3 : 0;
  for (long long c0 = 0; c0 < Ng; c0 += chunk) {
    const long long nc = (Ng - c0 < chunk) ? Ng - c0 : chunk;
    Buf g;
    const void* gsrc = offset_blocks(static_cast<const char*>(G), c0, B, gsz);
    if (gdt == DASH_DT_F32) {
      AffParams a = aff_from(gsrc, nullptr, FMT_F32, B, nc);
      a.nout = 1;
      a.out[0] = aout(split, FMT_SPLIT, 1.0f, 0.0f);
      DASH_TRY(launch_affine(a, st));
      g = split;
    } else {
      g.hi = const_cast<void*>(gsrc);
    }
    float* FL = offset_blocks(F, c0, B, 4);
    float* FR = offset_blocks(F, Ng + c0, B, 4);
    EpiParams e = epi_none();
    e.nout = 1;
    e.E_fmt = FMT_F32;
    // L_j = beta L_j + (1 - beta) G G^T
    e.out[0] = eout_f32(FL, 1.0f - beta, 0.0f, beta, nullptr);
    e.out[0].mirror = 1;
    e.E_hi = FL;
    e.pad_valid = valid_rows ? valid_rows + c0 : nullptr;
    DASH_TRY(gemm(gprec, B, nc, g, 0, g, 1, e, st, SO));
    // R_j = beta R_j + (1 - beta) G^T G
    e.out[0] = eout_f32(FR, 1.0f - beta, 0.0f, beta, nullptr);
    e.out[0].mirror = 1;
    e.E_hi = FR;
    e.pad_valid = valid_cols ? valid_cols + c0 : nullptr;
    DASH_TRY(gemm(gprec, B, nc, g, 1, g, 0, e, st, SO));
  }
  return DASH_OK;
}

// ---------------------------------------------------------------- scaling

dash_status spectral_scale(const float* A, float ridge, int64_t N, int B, int mode, int n_vec,
                           int power_iters, const float* V0, float* lambda_out, void* ws,
                           size_t ws_bytes, void* stream) {
  if (N < 0 || !valid_dim(B)) return DASH_ERR_INVALID_ARG;
  const bool half = (mode == DASH_SCALE_POWER_F16 || mode == DASH_SCALE_POWER_BF16);
  if (mode != DASH_SCALE_POWER && mode != DASH_SCALE_FROBENIUS && !half)
    return DASH_ERR_INVALID_ARG;
  if ((mode == DASH_SCALE_POWER || half) &&
      (n_vec < 1 || n_vec > 32 || power_iters < 1 || !V0))
    return DASH_ERR_INVALID_ARG;
  if (N == 0) return DASH_OK;
  if (!A || !lambda_out || !aligned16(A)) return DASH_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (mode == DASH_SCALE_FROBENIUS) {
    Carver cv(ws, ws_bytes);
    float* acc = static_cast<float*>(cv.take(static_cast<size_t>(N) * 4));
    if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
    if (cudaMemsetAsync(acc, 0, static_cast<size_t>(N) * 4, st) != cudaSuccess) return DASH_ERR_CUDA;
    DASH_TRY(launch_frob_acc(A, ridge, B, N, acc, st));
    return launch_sqrt_scale(acc, lambda_out, N, 1.0f, st);
  }
  if (half && power_cluster_supported(B)) {
    // Half precision, B <= 1024: the whole iteration in one launch, each block read
    // once (clusters of B / 128 CTAs, two blocks per cluster at a time, their 16-bit
    // copies kept in L2 for all products).  Needs three 16-bit block slots per
    // cluster; a workspace too small for three takes the one-launch-per-product path
    // below.
    const int bf = (mode == DASH_SCALE_POWER_BF16) ? 1 : 0;
    Carver cv(ws, ws_bytes);
    float* sigma = static_cast<float*>(cv.take(static_cast<size_t>(N) * 4));
    uint16_t* Vt = static_cast<uint16_t*>(cv.take(static_cast<size_t>(N) * 32 * B * 2));
    const size_t slot = power_cluster_slot_bytes(B);
    const long long nslots = cv.ok ? static_cast<long long>(cv.left / slot) : 0;
    if (nslots >= 3) {
      long long ncl = power_cluster_max_clusters(B, bf);
      if (ncl < 1) return DASH_ERR_CUDA;
      if (ncl > (N + 1) / 2) ncl = (N + 1) / 2;
      if (ncl > nslots / 3) ncl = nslots / 3;
      uint16_t* scratch = static_cast<uint16_t*>(cv.take(static_cast<size_t>(ncl) * 3 * slot));
      if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
      // sigma: each block's 16-bit copy holds sigma A with sigma an exact power of
      // two, so that it keeps fp16's range whatever the factor's magnitude.
      DASH_TRY(launch_diag_pow2_scale(A, ridge, B, N, sigma, st));
      DASH_TRY(launch_pad_vectors_t(V0, n_vec, B, N, bf, Vt, st));
      return launch_power_cluster(A, bf, ridge, sigma, B, N, Vt, n_vec, power_iters, scratch,
                                  static_cast<int>(ncl), lambda_out, st);
    }
  }
  if (half) {
    // Half precision: a 16-bit copy of each block, vectors transposed (32, B), one
    // launch per product.
    const int bf = (mode == DASH_SCALE_POWER_BF16) ? 1 : 0;
    const size_t per_blk = static_cast<size_t>(B) * B * 2 + 2 * static_cast<size_t>(B) * 32 * 2 +
                           3 * 32 * 4 + 4;
    long long chunk = static_cast<long long>(ws_bytes / per_blk);
    if (chunk > N) chunk = N;
    if (chunk > 65535) chunk = 65535;
    while (chunk > 0) {
      const size_t need = round256(static_cast<size_t>(chunk) * B * B * 2) +
                          2 * round256(static_cast<size_t>(chunk) * B * 32 * 2) +
                          3 * round256(static_cast<size_t>(chunk) * 32 * 4) +
                          round256(static_cast<size_t>(chunk) * 4);
      if (need <= ws_bytes) break;
      --chunk;
    }
    if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
    Carver cv(ws, ws_bytes);
    void* Ah = cv.take(static_cast<size_t>(chunk) * B * B * 2);
    uint16_t* Vt[2];
    Vt[0] = static_cast<uint16_t*>(cv.take(static_cast<size_t>(chunk) * B * 32 * 2));
    Vt[1] = static_cast<uint16_t*>(cv.take(static_cast<size_t>(chunk) * B * 32 * 2));
    float* nrm[2];
    nrm[0] = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * 32 * 4));
    nrm[1] = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * 32 * 4));
    float* den = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * 32 * 4));
    float* sigma = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * 4));
    if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
    const size_t acc_bytes = static_cast<size_t>(chunk) * 32 * 4;
    for (long long c0 = 0; c0 < N; c0 += chunk) {
      const long long nc = (N - c0 < chunk) ? N - c0 : chunk;
      // Each block is stored as sigma A with sigma an exact power of two, so that the
      // 16-bit copy keeps fp16's range whatever the factor's magnitude; lambda of
      // sigma (A + ridge I) is divided by sigma at the end.
      DASH_TRY(launch_diag_pow2_scale(offset_blocks(A, c0, B, 4), ridge, B, nc, sigma, st));
      AffParams a = aff_from(offset_blocks(A, c0, B, 4), nullptr, FMT_F32, B, nc);
      a.inv_s = sigma;
      a.nout = 1;
      Buf hb;
      hb.hi = Ah;
      a.out[0] = aout(hb, bf ? FMT_BF16 : FMT_F16, 1.0f, 0.0f);
      DASH_TRY(launch_affine(a, st));
      DASH_TRY(launch_pad_vectors_t(V0 + static_cast<size_t>(c0) * B * n_vec, n_vec, B, nc, bf,
                                    Vt[1], st));
      const uint16_t* vin = Vt[1];
      const float* in_n = nullptr;
      int cur = 0;
      for (int it = 0; it < power_iters; ++it) {
        const int last = (it == power_iters - 1);
        if (cudaMemsetAsync(nrm[cur], 0, acc_bytes, st) != cudaSuccess) return DASH_ERR_CUDA;
        if (last && cudaMemsetAsync(den, 0, acc_bytes, st) != cudaSuccess) return DASH_ERR_CUDA;
        DASH_TRY(launch_power_step_half(Ah, bf, ridge, sigma, B, nc, vin, n_vec, in_n, Vt[cur],
                                        nrm[cur], den, last, st));
        vin = Vt[cur];
        in_n = nrm[cur];
        cur ^= 1;
      }
      DASH_TRY(launch_power_finish(nrm[cur ^ 1], den, n_vec, nc, sigma, lambda_out + c0, st));
    }
    return DASH_OK;
  }
  // Power iteration, chunked so each chunk's vectors fit in the workspace.
  const size_t per_blk = 2 * static_cast<size_t>(B) * 32 * 4 + 3 * 32 * 4;
  long long chunk = static_cast<long long>(ws_bytes / per_blk);
  if (chunk > N) chunk = N;
  if (chunk > 65535) chunk = 65535;
  while (chunk > 0) {
    const size_t need = 2 * round256(static_cast<size_t>(chunk) * B * 32 * 4) +
                        3 * round256(static_cast<size_t>(chunk) * 32 * 4);
    if (need <= ws_bytes) break;
    --chunk;
  }
  if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
  Carver cv(ws, ws_bytes);
  float* V[2];
  V[0] = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * B * 32 * 4));
  V[1] = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * B * 32 * 4));
  float* nrm[2];
  nrm[0] = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * 32 * 4));
  nrm[1] = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * 32 * 4));
  float* den = static_cast<float*>(cv.take(static_cast<size_t>(chunk) * 32 * 4));
  if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  const size_t acc_bytes = static_cast<size_t>(chunk) * 32 * 4;
  for (long long c0 = 0; c0 < N; c0 += chunk) {
    const long long nc = (N - c0 < chunk) ? N - c0 : chunk;
    const float* Ac = offset_blocks(A, c0, B, 4);
    // Start vectors into the 32-column layout the product kernel streams.
    DASH_TRY(launch_pad_vectors(V0 + static_cast<size_t>(c0) * B * n_vec, n_vec, B, nc, V[1], st));
    const float* vin = V[1];
    const float* in_n = nullptr;
    int cur = 0;
    for (int it = 0; it < power_iters; ++it) {
      const int last = (it == power_iters - 1);
      if (cudaMemsetAsync(nrm[cur], 0, acc_bytes, st) != cudaSuccess) return DASH_ERR_CUDA;
      if (last && cudaMemsetAsync(den, 0, acc_bytes, st) != cudaSuccess) return DASH_ERR_CUDA;
      DASH_TRY(launch_power_step_tc(Ac, ridge, B, nc, vin, n_vec, in_n, V[cur], nrm[cur], den,
                                    last, st));
      vin = V[cur];
      in_n = nrm[cur];
      cur ^= 1;
    }
    // After the loop the last step's numerators sit in nrm[cur ^ 1].
    DASH_TRY(launch_power_finish(nrm[cur ^ 1], den, n_vec, nc, nullptr, lambda_out + c0, st));
  }
  return DASH_OK;
}

// ---------------------------------------------------------------- Coupled Newton

dash_status inv_root_cn(const float* A, float ridge, const float* scale, int64_t N, int B,
                        int iters, int prec, float* X, float* resid_out, void* ws,
                        size_t ws_bytes, void* stream) {
  int xfmt = FMT_F32;
  if (!root_prec(prec, xfmt)) return DASH_ERR_INVALID_ARG;
  DASH_TRY(common_root_checks(A, scale, N, B, iters, prec, X, ws));
  if (N == 0) return DASH_OK;
  if (resid_out && !aligned16(resid_out)) return DASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int K = iters;
  const int fmt = prec_fmt(prec);
  const int S = sym_mode(prec, B);  // symmetric-half iterates
  // 16-bit precisions (build-time modes, see gemm): the T^2 and T^4 products and the
  // M-update run whole (but in the two iterations below), the X product keeps
  // symmetric halves.  A product kept
  // as its upper 256-tiles is symmetrised by a tile mask, which turns the
  // antisymmetric part of a product of two rounded, not exactly commuting, iterates
  // (of order u ||M|| at 16 bits) into a symmetric error of the same size.  An
  // antisymmetric error moves eigenvalues only at second order; a symmetric one
  // moves them at first order, and M's smallest eigenvalues (about 1e-6 of the
  // largest on ill-conditioned factors) are what the root amplifies.  T comes from
  // the (not exactly symmetric) M-update, so T, T^2, T^4 and M are all read whole;
  // X only carries the result, whose absolute errors of order u |X| are harmless.
#ifndef DASH_CN16_TSYM
#define DASH_CN16_TSYM 0
#endif
#ifndef DASH_CN16_XSYM
#define DASH_CN16_XSYM 2
#endif
#ifndef DASH_CN16_MSYM
#define DASH_CN16_MSYM 0
#endif
  const int ST = (S && is_half(prec)) ? DASH_CN16_TSYM : S;
  const int SX = (S && is_half(prec)) ? DASH_CN16_XSYM : S;
  // Per-iteration modes of the T^2 / T^4 products and the M-update in 16-bit
  // precisions.  Whole products are needed while an error in M is amplified by the
  // iterations that follow.  Two iterations keep halves:
  //   k = 0: T_0 = (5I - A_s)/4 is exactly symmetric, so its squares keep halves;
  //     the M-update (T_0^4 rounded does not commute with M_0) stays whole, reading
  //     T^4 from its upper tiles (mode 4).
  //   k = K - 2, the last M-update: its error reaches X only through T_{K-1}, one
  //     factor of the final product, with no later iteration to amplify it (M is
  //     plain there, K - 2 >= jp).
  // Measured on rank-deficient factors (CN FP16, 10 iterations, B = 1024, against
  // the float64 oracle): every M-chain product whole 3.1e-3; this schedule 3.3e-3;
  // halves in all of the last three iterations 5.8e-3.
  auto t_mode = [&](int k) {
    if (!(S && is_half(prec))) return ST;
    return (k == 0 || k == K - 2) ? S : ST;
  };
  auto m_mode = [&](int k) {
    if (!(S && is_half(prec))) return S;
    if (k == K - 2) return S;
    return (k == 0) ? 4 : DASH_CN16_MSYM;
  };
  Carver cv(ws, ws_bytes);
  RootSmall sm;
  sm.inv_s = static_cast<float*>(cv.take(N * 4));
  sm.s_m14 = static_cast<float*>(cv.take(N * 4));
  sm.racc = static_cast<float*>(cv.take(static_cast<size_t>(N) * K * 4));
  if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  const int nbufs = (K >= 2) ? cn_bufs(prec) : 0;
  const long long chunk = fit_chunk(prec, B, N, nbufs, cv.left);
  if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
  // 16-bit precisions: M_k is a 16-bit pair for the first jp M-updates.
  const int jp = cn_pair_updates(prec, K);
  // 3xTF32 runs the identity-shifted form of the same iteration (see inv_root_ndb):
  // the T buffers hold D = T - I, D2 = T^2 - I and D4 = T^4 - I, and
  //   X T = X + X D,  T^2 - I = D D + 2D,  T^4 - I = D2 D2 + 2 D2,  T^4 M = M + D4 M,
  // each large term added exactly in the epilogue (E operand).
  const bool shift = (prec == DASH_FP32_3XTF32);
  const int pfmt = (prec == DASH_BF16) ? FMT_BF16X2 : FMT_F16X2;
  Buf bx[2], bm[2], bT, bT2, bT4;
  if (K >= 2) {
    bx[0] = cv.take_buf(prec, B, chunk);
    bx[1] = cv.take_buf(prec, B, chunk);
    bm[0] = is_half(prec) ? cv.take_pair16(B, chunk) : cv.take_buf(prec, B, chunk);
    bm[1] = is_half(prec) ? cv.take_pair16(B, chunk) : cv.take_buf(prec, B, chunk);
    bT = cv.take_buf(prec, B, chunk);
    bT2 = cv.take_buf(prec, B, chunk);
    bT4 = cv.take_buf(prec, B, chunk);
    if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  }
  DASH_TRY(launch_scale_factors(scale, sm.inv_s, sm.s_m14, N, st));
  if (resid_out &&
      cudaMemsetAsync(sm.racc, 0, static_cast<size_t>(N) * K * 4, st) != cudaSuccess)
    return DASH_ERR_CUDA;

  for (long long c0 = 0; c0 < N; c0 += chunk) {
    const long long nc = (N - c0 < chunk) ? N - c0 : chunk;
    const float* Ac = offset_blocks(A, c0, B, 4);
    float* Xc = offset_blocks(X, c0, B, 4);
    const float* inv_s = sm.inv_s + c0;
    const float* m14 = sm.s_m14 + c0;
    float* racc = resid_out ? sm.racc + c0 * K : nullptr;
    // Prologue: M_0 = A_s, T_0 = (5I - A_s)/4, X_1 = T_0; residual of M_0.
    AffParams a = aff_from(Ac, nullptr, FMT_F32, B, nc);
    a.ridge = ridge;
    a.inv_s = inv_s;
    a.resid_acc = racc;
    a.resid_stride = K;
    if (K == 1) {
      a.nout = 1;
      Buf xb;
      xb.hi = Xc;
      a.out[0] = aout(xb, xfmt, -0.25f, 1.25f, m14);
      DASH_TRY(launch_affine(a, st));
      continue;
    }
    a.nout = 2;
    a.out[0] = aout(bm[0], jp > 0 ? pfmt : fmt, 1.0f, 0.0f);
    a.out[1] = aout(bT, fmt, -0.25f, shift ? 0.25f : 1.25f);
    if (shift) {
      a.nout = 3;  // X_1 = T_0 = I + D_0 gets its own buffer
      a.out[2] = aout(bx[0], fmt, -0.25f, 1.25f);
    }
    DASH_TRY(launch_affine(a, st));
    // T_k and the scratch that takes T_k^2 and then T_{k+1} trade buffers every
    // iteration.  X_1 = T_0 is not copied: it is read from T_0's buffer, which
    // becomes scratch only after the first X product has consumed it.
    Buf tk = bT, tsp = bT2, xk = shift ? bx[0] : bT;
    int mc = 0, xn = shift ? 1 : 0;
    const float e1 = shift ? 1.0f : 0.0f, e2 = shift ? 2.0f : 0.0f;
    for (int k = 0; k < K; ++k) {
      if (k == K - 1) {
        // X_K = X_{K-1} T_{K-1}, scaled by s^{-1/4}, into the caller's fp32 output.
        EpiParams e = epi_none();
        e.nout = 1;
        Buf xb;
        xb.hi = Xc;
        e.out[0] = eout(xb, xfmt, 1.0f, 0.0f, e1, m14);
        e.out[0].mirror = 1;  // halves: the tiles below the diagonal by transposition
        if (shift) with_e(e, xk, fmt);
        DASH_TRY(gemm(prec, B, nc, xk, 0, tk, 0, e, st, SX));
        break;
      }
      if (k >= 1) {
        EpiParams e = epi_none();
        e.nout = 1;
        e.out[0] = eout(bx[xn], fmt, 1.0f, 0.0f, e1);
        if (shift) with_e(e, xk, fmt);
        DASH_TRY(gemm(prec, B, nc, xk, 0, tk, 0, e, st, SX));
        xk = bx[xn];
        xn ^= 1;
      }
      EpiParams ea = epi_none();
      ea.nout = 1;
      ea.out[0] = eout(tsp, fmt, 1.0f, 0.0f, e2);
      if (shift) with_e(ea, tk, fmt);
      DASH_TRY(gemm(prec, B, nc, tk, 0, tk, 0, ea, st, t_mode(k)));
      EpiParams eb = epi_none();
      eb.nout = 1;
      eb.out[0] = eout(bT4, fmt, 1.0f, 0.0f, e2);
      if (shift) with_e(eb, tsp, fmt);
      DASH_TRY(gemm(prec, B, nc, tsp, 0, tsp, 0, eb, st, t_mode(k)));
      // M_{k+1} = T^4 M_k; the same epilogue forms T_{k+1} (into the scratch, free
      // once T^4 is formed) and the residual of M_{k+1}.
      EpiParams em = epi_none();
      em.nout = 2;
      em.out[0] = eout(bm[mc ^ 1], (k + 1 < jp) ? pfmt : fmt, 1.0f, 0.0f, e1);
      em.out[1] = eout(tsp, fmt, -0.25f, shift ? 0.25f : 1.25f, shift ? -0.25f : 0.0f);
      if (shift) {
        with_e(em, bm[mc], fmt);
        em.resid_plus_e = 1;
      }
      em.resid_acc = racc ? racc + (k + 1) : nullptr;
      em.resid_stride = K;
      // 16-bit: T^4 and M read whole, M and T written whole (see ST above).
      DASH_TRY(gemm(prec, B, nc, bT4, 0, bm[mc], 0, em, st, m_mode(k), k < jp));
      mc ^= 1;
      const Buf t = tk;
      tk = tsp;
      tsp = t;
    }
  }
  if (resid_out)
    DASH_TRY(launch_sqrt_scale(sm.racc, resid_out, N * K, 1.0f / std::sqrt(static_cast<float>(B)), st));
  return DASH_OK;
}

// ---------------------------------------------------------------- Newton-Denman-Beavers

dash_status inv_root_ndb(const float* A, float ridge, const float* scale, int64_t N, int B,
                         int iters, int prec, float* X, float* resid_out, void* ws,
                         size_t ws_bytes, void* stream) {
  int xfmt = FMT_F32;
  if (!root_prec(prec, xfmt)) return DASH_ERR_INVALID_ARG;
  DASH_TRY(common_root_checks(A, scale, N, B, iters, prec, X, ws));
  if (N == 0) return DASH_OK;
  if (resid_out && !aligned16(resid_out)) return DASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int K = iters;
  const int fmt = prec_fmt(prec);
  // No symmetric-half iterates here: forcing each product of the coupled iteration
  // symmetric breaks the Y = A Z balance its left / right products keep, and on
  // ill-conditioned blocks (scaled condition ~1e6) the iteration then diverges --
  // in plain float32 as well -- where the full products converge.
  const int S = 0, SI = 0;
  // 3xTF32 runs the identity-shifted form of the same iteration: the buffer of T
  // holds D = T - I, and Y T = Y + Y D, T Z = Z + D Z add the large term exactly in
  // the epilogue (E operand).  The products then only carry the iterates' deviation
  // from identity scaling, so the tensor core's truncating accumulation and the
  // TF32 split act on small numbers; and D keeps full relative precision where T
  // would lose it next to its unit diagonal.
  const bool shift = (prec == DASH_FP32_3XTF32);
  const float gT = shift ? 0.5f : 1.5f;  // gamma of T (or D) = (3I - P) / 2 (- I)
  Carver cv(ws, ws_bytes);
  RootSmall sm;
  sm.inv_s = static_cast<float*>(cv.take(N * 4));
  sm.s_m14 = static_cast<float*>(cv.take(N * 4));
  sm.racc = static_cast<float*>(cv.take(static_cast<size_t>(N) * 2 * K * 4));
  if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  const long long chunk = fit_chunk(prec, B, N, NDB_BUFS, cv.left);
  if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
  Buf pool[NDB_BUFS];
  for (int i = 0; i < NDB_BUFS; ++i) pool[i] = cv.take_buf(prec, B, chunk);
  if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  DASH_TRY(launch_scale_factors(scale, sm.inv_s, sm.s_m14, N, st));
  if (resid_out &&
      cudaMemsetAsync(sm.racc, 0, static_cast<size_t>(N) * 2 * K * 4, st) != cudaSuccess)
    return DASH_ERR_CUDA;

  for (long long c0 = 0; c0 < N; c0 += chunk) {
    const long long nc = (N - c0 < chunk) ? N - c0 : chunk;
    const float* Ac = offset_blocks(A, c0, B, 4);
    float* Xc = offset_blocks(X, c0, B, 4);
    Buf Xout;
    Xout.hi = Xc;
    const float* inv_s = sm.inv_s + c0;
    const float* m14 = sm.s_m14 + c0;
    float* racc = resid_out ? sm.racc + c0 * 2 * K : nullptr;
    const long long rstride = 2LL * K;
    // Buffer roles are indices into pool; `used` marks buffers holding live data.
    int iC = 0, iT = 1, iZ = 2;
    // Stage-1 prologue: C = A_s, T_0 = (3I - A_s)/2, Z_1 = T_0, residual of C.
    AffParams a = aff_from(Ac, nullptr, FMT_F32, B, nc);
    a.ridge = ridge;
    a.inv_s = inv_s;
    a.resid_acc = racc;
    a.resid_stride = rstride;
    a.nout = 3;
    a.out[0] = aout(pool[iC], fmt, 1.0f, 0.0f);
    a.out[1] = aout(pool[iT], fmt, -0.5f, gT);
    a.out[2] = aout(pool[iZ], fmt, -0.5f, 1.5f);
    DASH_TRY(launch_affine(a, st));

    for (int stage = 0; stage < 2; ++stage) {
      // Live: C (= Y_0) in iC, T_0 in iT, Z_1 = T_0 in iZ.
      int iY = iC;
      auto free_buf = [&](int a0, int a1, int a2) {
        for (int i = 0; i < NDB_BUFS; ++i)
          if (i != a0 && i != a1 && i != a2) return i;
        return -1;
      };
      float* racc_s = racc ? racc + stage * K : nullptr;
      const bool keepY = (stage == 0);
      for (int k = 0; k < K; ++k) {
        const bool lastk = (k == K - 1);
        if (k >= 1) {
          // P = Z_k Y_k -> T_k = (3I - P)/2 (D_k = T_k - I) and the residual of P.
          EpiParams ep = epi_none();
          ep.nout = 1;
          ep.out[0] = eout(pool[iT], fmt, -0.5f, gT);
          ep.resid_acc = racc_s ? racc_s + k : nullptr;
          ep.resid_stride = rstride;
          DASH_TRY(gemm(prec, B, nc, pool[iZ], 0, pool[iY], 0, ep, st, S));
        }
        if (!lastk) {
          const int iYn = free_buf(iY, iZ, iT);
          EpiParams ey = epi_none();
          ey.nout = 1;
          ey.out[0] = eout(pool[iYn], fmt, 1.0f, 0.0f, shift ? 1.0f : 0.0f);
          if (shift) with_e(ey, pool[iY], fmt);  // Y + Y D
          DASH_TRY(gemm(prec, B, nc, pool[iY], 0, pool[iT], 0, ey, st, S));
          iY = iYn;
          if (k >= 1) {
            const int iZn = free_buf(iY, iZ, iT);
            EpiParams ez = epi_none();
            ez.nout = 1;
            ez.out[0] = eout(pool[iZn], fmt, 1.0f, 0.0f, shift ? 1.0f : 0.0f);
            if (shift) with_e(ez, pool[iZ], fmt);  // Z + D Z
            DASH_TRY(gemm(prec, B, nc, pool[iT], 0, pool[iZ], 0, ez, st, S));
            iZ = iZn;
          }
          continue;
        }
        // Last iteration of the stage.
        if (keepY) {
          // Y_K = Y_{K-1} T_{K-1}; its epilogue starts stage 2 on C' = Y_K:
          // C' (kept), T'_0 = (3I - C')/2, Z'_1 = T'_0, residual of C'.
          // With one iteration per stage, stage 2's answer is Z'_1 itself.
          const int iCn = free_buf(iY, iT, -1);
          const int iTn = free_buf(iY, iT, iCn);
          int iZn = -1;
          for (int i = 0; i < NDB_BUFS; ++i)
            if (i != iY && i != iT && i != iCn && i != iTn) {
              iZn = i;
              break;
            }
          EpiParams ey = epi_none();
          ey.resid_acc = racc ? racc + K : nullptr;
          ey.resid_stride = rstride;
          // Shifted: C' = Y + Y D, so every output adds (a multiple of) E = Y.
          const float e1 = shift ? 1.0f : 0.0f, eh = shift ? -0.5f : 0.0f;
          if (shift) {
            with_e(ey, pool[iY], fmt);
            ey.resid_plus_e = 1;
          }
          if (K == 1) {
            ey.nout = 1;
            ey.out[0] = eout(Xout, xfmt, -0.5f, 1.5f, eh, m14);
            // residual of C' = product itself
            DASH_TRY(gemm(prec, B, nc, pool[iY], 0, pool[iT], 0, ey, st, SI));
          } else {
            ey.nout = 3;
            ey.out[0] = eout(pool[iCn], fmt, 1.0f, 0.0f, e1);
            ey.out[1] = eout(pool[iTn], fmt, -0.5f, gT, eh);
            ey.out[2] = eout(pool[iZn], fmt, -0.5f, 1.5f, eh);
            DASH_TRY(gemm(prec, B, nc, pool[iY], 0, pool[iT], 0, ey, st, S));
          }
          iC = iCn;
          iT = iTn;
          iZ = iZn;
        } else {
          // Z_K = T_{K-1} Z_{K-1}, scaled by s^{-1/4}, into the caller's output.
          EpiParams ez = epi_none();
          ez.nout = 1;
          ez.out[0] = eout(Xout, xfmt, 1.0f, 0.0f, shift ? 1.0f : 0.0f, m14);
          if (shift) with_e(ez, pool[iZ], fmt);  // Z + D Z
          DASH_TRY(gemm(prec, B, nc, pool[iT], 0, pool[iZ], 0, ez, st, SI));
        }
      }
      if (stage == 0 && K == 1) break;  // stage 2 finished inside stage 1's epilogue
    }
  }
  if (resid_out)
    DASH_TRY(launch_sqrt_scale(sm.racc, resid_out, N * 2 * K,
                               1.0f / std::sqrt(static_cast<float>(B)), st));
  return DASH_OK;
}

// ---------------------------------------------------------------- Chebyshev / Clenshaw

dash_status dash_select_tiers(const float* lam_max, const float* lam_min, int64_t n,
                              const dash_tier* tiers, int ntiers, int32_t* choice) {
  if (n < 0 || ntiers < 1 || !tiers) return DASH_ERR_INVALID_ARG;
  for (int t = 0; t < ntiers; ++t) {
    const dash_tier& T = tiers[t];
    if (T.solver < DASH_SOLVER_CN || T.solver > DASH_SOLVER_CHEB || !valid_prec(T.prec) ||
        T.iters < 1 || !(T.u > 0.0) || !(T.gate > 0.0))
      return DASH_ERR_INVALID_ARG;
  }
  if (n == 0) return DASH_OK;
  if (!lam_max || !lam_min || !choice) return DASH_ERR_INVALID_ARG;
  for (int64_t k = 0; k < n; ++k) {
    const double hi = lam_max[k], lo = lam_min[k];
    // No usable estimate unless both are positive (NaN compares false): inf, the
    // last (most accurate) tier.
    double kappa = std::numeric_limits<double>::infinity();
    if (lo > 0.0 && hi > 0.0) kappa = hi / lo;
    int32_t pick = ntiers - 1;
    if (!std::isnan(kappa)) {
      for (int t = 0; t < ntiers; ++t) {
        if (kappa * tiers[t].u / 4.0 <= tiers[t].gate) {
          pick = t;
          break;
        }
      }
    }
    choice[k] = pick;
  }
  return DASH_OK;
}

dash_status dash_cheb_coeffs(int degree, double lo, double hi, double* c) {
  if (degree < 1 || degree > 64 || !(lo > 0.0) || !(hi > lo) || !std::isfinite(hi) || !c)
    return DASH_ERR_INVALID_ARG;
  // Coefficients of the degree-d interpolant of x^{-1/4} at the first-kind
  // Chebyshev points of [lo, hi], in the Chebyshev basis of t in [-1, 1].
  const int d = degree;
  const double pi = 3.14159265358979323846;
  for (int j = 0; j <= d; ++j) {
    double acc = 0.0;
    for (int i = 0; i <= d; ++i) {
      const double th = pi * (i + 0.5) / (d + 1);
      const double x = 0.5 * (hi - lo) * std::cos(th) + 0.5 * (hi + lo);
      acc += std::pow(x, -0.25) * std::cos(j * th);
    }
    c[j] = 2.0 * acc / (d + 1);
  }
  c[0] *= 0.5;
  return DASH_OK;
}

dash_status inv_root_cheb(const float* A, float ridge, const float* scale, int64_t N, int B,
                          int degree, double lo, double hi, int prec, float* X, void* ws,
                          size_t ws_bytes, void* stream) {
  int xfmt = FMT_F32;
  if (!root_prec(prec, xfmt)) return DASH_ERR_INVALID_ARG;
  DASH_TRY(common_root_checks(A, scale, N, B, 1, prec, X, ws));
  if (degree < 1 || degree > 64 || !(lo > 0.0) || !(hi > lo) || !std::isfinite(hi))
    return DASH_ERR_INVALID_ARG;
  if (N == 0) return DASH_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int d = degree;
  const int fmt = prec_fmt(prec);
  const int S = sym_mode(prec, B);  // symmetric-half iterates
  std::vector<double> c(d + 1);
  DASH_TRY(dash_cheb_coeffs(d, lo, hi, c.data()));
  const double aS = 2.0 / (hi - lo), gS = -(hi + lo) / (hi - lo);

  Carver cv(ws, ws_bytes);
  float* inv_s = static_cast<float*>(cv.take(N * 4));
  float* s_m14 = static_cast<float*>(cv.take(N * 4));
  cv.take(4);
  if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  const int nbufs = (d >= 2) ? CHEB_BUFS : 0;
  const long long chunk = fit_chunk(prec, B, N, nbufs, cv.left);
  if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
  Buf bS, bb[3];
  if (d >= 2) {
    bS = cv.take_buf(prec, B, chunk);
    for (int i = 0; i < 3; ++i) bb[i] = cv.take_buf(prec, B, chunk);
    if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  }
  DASH_TRY(launch_scale_factors(scale, inv_s, s_m14, N, st));
  for (long long c0 = 0; c0 < N; c0 += chunk) {
    const long long nc = (N - c0 < chunk) ? N - c0 : chunk;
    const float* Ac = offset_blocks(A, c0, B, 4);
    float* Xc = offset_blocks(X, c0, B, 4);
    const float* m14 = s_m14 + c0;
    AffParams a = aff_from(Ac, nullptr, FMT_F32, B, nc);
    a.ridge = ridge;
    a.inv_s = inv_s + c0;
    if (d == 1) {
      // P = c_0 I + c_1 S.
      Buf xb;
      xb.hi = Xc;
      a.nout = 1;
      a.out[0] = aout(xb, xfmt, static_cast<float>(c[1] * aS),
                      static_cast<float>(c[0] + c[1] * gS), m14);
      DASH_TRY(launch_affine(a, st));
      continue;
    }
    // S and b_{d-1} = c_{d-1} I + 2 c_d S.
    a.nout = 2;
    a.out[0] = aout(bS, fmt, static_cast<float>(aS), static_cast<float>(gS));
    a.out[1] = aout(bb[0], fmt, static_cast<float>(2.0 * c[d] * aS),
                    static_cast<float>(c[d - 1] + 2.0 * c[d] * gS));
    DASH_TRY(launch_affine(a, st));
    Buf xb;
    xb.hi = Xc;
    if (d == 2) {
      EpiParams e = epi_none();
      e.nout = 1;
      e.out[0] = eout(xb, xfmt, 1.0f, static_cast<float>(c[0] - c[2]), 0.0f, m14);
      e.out[0].mirror = 1;
      DASH_TRY(gemm(prec, B, nc, bS, 0, bb[0], 0, e, st, S));
      continue;
    }
    // b_{d-2} = 2 S b_{d-1} + (c_{d-2} - c_d) I
    int i1 = 0, i2 = -1, i0 = 1;  // b_{j+1}, b_{j+2}, b_j
    {
      EpiParams e = epi_none();
      e.nout = 1;
      e.out[0] = eout(bb[i0], fmt, 2.0f, static_cast<float>(c[d - 2] - c[d]));
      DASH_TRY(gemm(prec, B, nc, bS, 0, bb[i1], 0, e, st, S));
      i2 = i1;
      i1 = i0;
    }
    for (int j = d - 3; j >= 1; --j) {
      i0 = 3 - i1 - i2;
      EpiParams e = epi_none();
      e.nout = 1;
      e.out[0] = eout(bb[i0], fmt, 2.0f, static_cast<float>(c[j]), -1.0f);
      e.E_hi = bb[i2].hi;
      e.E_lo = bb[i2].lo;
      e.E_fmt = fmt;
      DASH_TRY(gemm(prec, B, nc, bS, 0, bb[i1], 0, e, st, S));
      i2 = i1;
      i1 = i0;
    }
    // P = S b_1 + c_0 I - b_2
    EpiParams e = epi_none();
    e.nout = 1;
    e.out[0] = eout(xb, xfmt, 1.0f, static_cast<float>(c[0]), -1.0f, m14);
    e.out[0].mirror = 1;
    e.E_hi = bb[i2].hi;
    e.E_lo = bb[i2].lo;
    e.E_fmt = fmt;
    // All products keep symmetric halves (E is read only where it was written);
    // the caller's X is completed below the diagonal by the mirrored stores.
    DASH_TRY(gemm(prec, B, nc, bS, 0, bb[i1], 0, e, st, S));
  }
  return DASH_OK;
}

// ---------------------------------------------------------------- per-block solver selection

namespace {

// Bytes spectral_scale needs for n blocks in `mode` (0 for Frobenius).
size_t scale_ws_bytes(int mode, long long n, int B, int n_vec) {
  size_t b = 0;
  const int prec = (mode == DASH_SCALE_POWER_F16)    ? DASH_FP16
                   : (mode == DASH_SCALE_POWER_BF16) ? DASH_BF16
                                                     : DASH_FP32_3XTF32;
  if (dash_workspace_size(DASH_OP_SPECTRAL_SCALE, n, B, prec, n_vec, &b) != DASH_OK) return 0;
  return b;
}

// Workspace of one solve of n blocks by tier t (its solver's full one-pass size).
size_t tier_ws_bytes(const dash_tier& t, long long n, int B) {
  const int op = t.solver == DASH_SOLVER_CN    ? DASH_OP_INV_ROOT_CN
                 : t.solver == DASH_SOLVER_NDB ? DASH_OP_INV_ROOT_NDB
                                               : DASH_OP_INV_ROOT_CHEB;
  size_t b = 0;
  if (dash_workspace_size(op, n, B, t.prec, t.iters, &b) != DASH_OK) return 0;
  return b;
}

dash_status solve_tier(const dash_tier& t, const float* A, float ridge, const float* lam, long long n,
                       int B, double lo, double hi, float* X, void* ws, size_t ws_bytes,
                       cudaStream_t st) {
  switch (t.solver) {
    case DASH_SOLVER_CN:
      return inv_root_cn(A, ridge, lam, n, B, t.iters, t.prec, X, nullptr, ws, ws_bytes, st);
    case DASH_SOLVER_NDB:
      return inv_root_ndb(A, ridge, lam, n, B, t.iters, t.prec, X, nullptr, ws, ws_bytes, st);
    default:
      return inv_root_cheb(A, ridge, lam, n, B, t.iters, lo, hi, t.prec, X, ws, ws_bytes, st);
  }
}

bool valid_tiers(const dash_tier* tiers, int ntiers) {
  if (!tiers || ntiers < 1) return false;
  for (int t = 0; t < ntiers; ++t) {
    const dash_tier& T = tiers[t];
    if (T.solver < DASH_SOLVER_CN || T.solver > DASH_SOLVER_CHEB || !valid_prec(T.prec) ||
        T.iters < 1 || !(T.u > 0.0) || !(T.gate > 0.0) ||
        (T.solver == DASH_SOLVER_CHEB && T.iters > 64))
      return false;
  }
  return true;
}

}  // namespace

dash_status spectral_lambda_min(const float* A, float ridge, const float* lam_max, int64_t N, int B,
                                int mode, int n_vec, int power_iters, const float* V0,
                                float* lam_min_out, void* ws, size_t ws_bytes, void* stream) {
  if (N < 0 || !valid_dim(B)) return DASH_ERR_INVALID_ARG;
  if (mode != DASH_SCALE_POWER && mode != DASH_SCALE_POWER_F16 && mode != DASH_SCALE_POWER_BF16)
    return DASH_ERR_INVALID_ARG;
  if (n_vec < 1 || n_vec > 32 || power_iters < 1 || !V0) return DASH_ERR_INVALID_ARG;
  if (N == 0) return DASH_OK;
  if (!A || !lam_max || !lam_min_out || !aligned16(A) || !aligned16(V0))
    return DASH_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t blk = static_cast<size_t>(B) * B * 4;
  // Per chunk of c blocks: the shifted stack, 1/c_k, mu_k, and spectral_scale's workspace.
  auto need = [&](long long c) {
    return round256(c * blk) + 2 * round256(c * 4) + round256(scale_ws_bytes(mode, c, B, n_vec));
  };
  long long chunk = N;
  while (chunk > 0 && need(chunk) > ws_bytes) chunk = (chunk > 64) ? chunk * 3 / 4 : chunk - 1;
  if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
  Carver cv(ws, ws_bytes);
  float* S = static_cast<float*>(cv.take(chunk * blk));
  float* inv_c = static_cast<float*>(cv.take(chunk * 4));
  float* mu = static_cast<float*>(cv.take(chunk * 4));
  const size_t sws = cv.left;
  void* sw = cv.take(sws > 256 ? sws - 256 : 0);
  if (!cv.ok || !sw) return DASH_ERR_WORKSPACE_TOO_SMALL;
  for (long long c0 = 0; c0 < N; c0 += chunk) {
    const long long nc = (N - c0 < chunk) ? N - c0 : chunk;
    // S_k = c_k I - (A_k + ridge I) = c_k (I - (A_k + ridge I) / c_k), c_k = lam_max[k].
    DASH_TRY(launch_scale_factors(lam_max + c0, inv_c, mu, nc, st));  // mu: scratch here
    AffParams a = aff_from(offset_blocks(A, c0, B, 4), nullptr, FMT_F32, B, nc);
    a.ridge = ridge;
    a.inv_s = inv_c;
    a.nout = 1;
    Buf sb;
    sb.hi = S;
    a.out[0] = aout(sb, FMT_F32, -1.0f, 1.0f, lam_max + c0);
    DASH_TRY(launch_affine(a, st));
    DASH_TRY(spectral_scale(S, 0.0f, nc, B, mode, n_vec, power_iters,
                            V0 + static_cast<size_t>(c0) * B * n_vec, mu, sw, sws - 256, st));
    DASH_TRY(launch_sub(lam_max + c0, mu, lam_min_out + c0, nc, st));
  }
  return DASH_OK;
}

dash_status dash_auto_workspace_size(int64_t N, int B, const dash_tier* tiers, int ntiers,
                                     size_t* bytes) {
  if (!bytes || N < 0 || !valid_dim(B) || !valid_tiers(tiers, ntiers)) return DASH_ERR_INVALID_ARG;
  size_t worst = 0;
  for (int t = 0; t < ntiers; ++t) {
    const size_t w = tier_ws_bytes(tiers[t], N, B);
    if (w > worst) worst = w;
  }
  const size_t blk = static_cast<size_t>(B) * B * 4;
  // Index list, gathered scales, gathered blocks and their roots, the solver's workspace.
  *bytes = round256(N * 4) + round256(N * 4) + 2 * round256(N * blk) + round256(worst);
  return DASH_OK;
}

dash_status inv_root_auto(const float* A, float ridge, const float* lam_max, const float* lam_min,
                          int64_t N, int B, const dash_tier* tiers, int ntiers, double cheb_lo,
                          double cheb_hi, float* X, int32_t* choice_out, void* ws,
                          size_t ws_bytes, void* stream) {
  if (N < 0 || !valid_dim(B) || !valid_tiers(tiers, ntiers)) return DASH_ERR_INVALID_ARG;
  for (int t = 0; t < ntiers; ++t)
    if (tiers[t].solver == DASH_SOLVER_CHEB &&
        (!(cheb_lo > 0.0) || !(cheb_hi > cheb_lo) || !std::isfinite(cheb_hi)))
      return DASH_ERR_INVALID_ARG;
  if (N == 0) return DASH_OK;
  if (!A || !lam_max || !lam_min || !X || !aligned16(A) || !aligned16(X) || !aligned16(lam_max))
    return DASH_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The one synchronisation: both estimates come back to the host for the tier rule.
  std::vector<float> hmax(N), hmin(N);
  if (cudaMemcpyAsync(hmax.data(), lam_max, N * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(hmin.data(), lam_min, N * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return DASH_ERR_CUDA;
  std::vector<int32_t> choice(N);
  DASH_TRY(dash_select_tiers(hmax.data(), hmin.data(), N, tiers, ntiers, choice.data()));
  if (choice_out) std::memcpy(choice_out, choice.data(), N * sizeof(int32_t));
  const size_t blk = static_cast<size_t>(B) * B * 4;
  for (int t = 0; t < ntiers; ++t) {
    std::vector<int32_t> idx;
    for (int64_t k = 0; k < N; ++k)
      if (choice[k] == t) idx.push_back(static_cast<int32_t>(k));
    const long long n = static_cast<long long>(idx.size());
    if (n == 0) continue;
    if (idx.back() - idx.front() + 1 == n) {
      // One contiguous range: solve in place, no copies.
      const long long a = idx.front();
      DASH_TRY(solve_tier(tiers[t], offset_blocks(A, a, B, 4), ridge, lam_max + a, n, B, cheb_lo,
                          cheb_hi, offset_blocks(X, a, B, 4), ws, ws_bytes, st));
      continue;
    }
    // Gather the tier's blocks (and scales) into a sub-stack, solve, scatter the roots.
    Carver cv(ws, ws_bytes);
    int32_t* didx = static_cast<int32_t*>(cv.take(n * 4));
    float* dlam = static_cast<float*>(cv.take(n * 4));
    if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
    long long chunk = n;
    while (chunk > 0 && 2 * round256(chunk * blk) + round256(tier_ws_bytes(tiers[t], chunk, B)) >
                            cv.left)
      chunk = (chunk > 64) ? chunk * 3 / 4 : chunk - 1;
    if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
    float* At = static_cast<float*>(cv.take(chunk * blk));
    float* Xt = static_cast<float*>(cv.take(chunk * blk));
    const size_t sws = cv.left;
    void* sw = cv.take(sws > 256 ? sws - 256 : 0);
    if (!cv.ok || !sw) return DASH_ERR_WORKSPACE_TOO_SMALL;
    if (cudaMemcpyAsync(didx, idx.data(), n * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return DASH_ERR_CUDA;
    DASH_TRY(launch_copy_items(lam_max, dlam, didx, 0, 1, n, st));
    for (long long c0 = 0; c0 < n; c0 += chunk) {
      const long long nc = (n - c0 < chunk) ? n - c0 : chunk;
      DASH_TRY(launch_copy_items(A, At, didx + c0, 0, static_cast<long long>(B) * B, nc, st));
      DASH_TRY(solve_tier(tiers[t], At, ridge, dlam + c0, nc, B, cheb_lo, cheb_hi, Xt, sw,
                          sws - 256, st));
      DASH_TRY(launch_copy_items(Xt, X, didx + c0, 1, static_cast<long long>(B) * B, nc, st));
    }
    // The next tier's index upload reuses didx; it is ordered after these kernels
    // on the stream (a copy from pageable host memory also waits for the stream).
  }
  return DASH_OK;
}

// ---------------------------------------------------------------- apply

// The preconditioned direction U = L^{-1/4} G R^{-1/4}; with W, the second product's
// epilogue also takes the weight step W <- W - lr U in place (E = W), and U is
// written only when asked for.
static dash_status apply_impl(const void* G, int gdt, const float* Froot, int64_t Ng, int B,
                              int prec, float* U, float* W, float lr, void* ws, size_t ws_bytes,
                              void* stream) {
  // DASH_ROOT_TF32 (with DASH_TF32 only): Froot is read as it is.
  const bool roots_ready = (prec == (DASH_TF32 | DASH_ROOT_TF32));
  if (roots_ready) prec = DASH_TF32;
  if (Ng < 0 || !valid_dim(B) || !valid_prec(prec) ||
      !(gdt == DASH_DT_F32 || gdt == DASH_DT_BF16 || gdt == DASH_DT_F16))
    return DASH_ERR_INVALID_ARG;
  if (Ng == 0) return DASH_OK;
  if (!G || !Froot || !aligned16(G) || !aligned16(Froot)) return DASH_ERR_INVALID_ARG;
  if ((!U && !W) || (U && !aligned16(U)) || (W && !aligned16(W))) return DASH_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int fmt = prec_fmt(prec);
  // TF32-rounded roots need no operand buffers of their own: G and T only.
  const long long chunk = fit_chunk(prec, B, Ng, roots_ready ? 2 : APPLY_BUFS, ws_bytes);
  if (chunk < 1) return DASH_ERR_WORKSPACE_TOO_SMALL;
  Carver cv(ws, ws_bytes);
  Buf bG = cv.take_buf(prec, B, chunk);
  Buf bT = cv.take_buf(prec, B, chunk);
  Buf bL, bR;
  if (!roots_ready) {
    bL = cv.take_buf(prec, B, chunk);
    bR = cv.take_buf(prec, B, chunk);
  }
  if (!cv.ok) return DASH_ERR_WORKSPACE_TOO_SMALL;
  const int gfmt = (gdt == DASH_DT_F32) ? FMT_F32 : (gdt == DASH_DT_BF16 ? FMT_BF16 : FMT_F16);
  const size_t gsz = (gdt == DASH_DT_F32) ? 4 : 2;
  for (long long c0 = 0; c0 < Ng; c0 += chunk) {
    const long long nc = (Ng - c0 < chunk) ? Ng - c0 : chunk;
    AffParams a = aff_from(offset_blocks(static_cast<const char*>(G), c0, B, gsz), nullptr, gfmt, B, nc);
    a.nout = 1;
    a.out[0] = aout(bG, fmt, 1.0f, 0.0f);
    DASH_TRY(launch_affine(a, st));
    Buf opL = bL, opR = bR;
    if (roots_ready) {
      // TF32-rounded roots are the TF32 operands themselves.
      opL.hi = const_cast<float*>(offset_blocks(Froot, c0, B, 4));
      opR.hi = const_cast<float*>(offset_blocks(Froot, Ng + c0, B, 4));
    } else {
      a = aff_from(offset_blocks(Froot, c0, B, 4), nullptr, FMT_F32, B, nc);
      a.nout = 1;
      a.out[0] = aout(bL, fmt, 1.0f, 0.0f);
      DASH_TRY(launch_affine(a, st));
      a = aff_from(offset_blocks(Froot, Ng + c0, B, 4), nullptr, FMT_F32, B, nc);
      a.nout = 1;
      a.out[0] = aout(bR, fmt, 1.0f, 0.0f);
      DASH_TRY(launch_affine(a, st));
    }
    EpiParams e = epi_none();
    e.nout = 1;
    e.out[0] = eout(bT, fmt, 1.0f, 0.0f);
    DASH_TRY(gemm(prec, B, nc, opL, 0, bG, 0, e, st));
    e.nout = 0;
    if (W) {
      float* Wc = offset_blocks(W, c0, B, 4);
      e.out[e.nout++] = eout_f32(Wc, -lr, 0.0f, 1.0f, nullptr);
      e.E_hi = Wc;
      e.E_fmt = FMT_F32;
    }
    if (U) e.out[e.nout++] = eout_f32(offset_blocks(U, c0, B, 4), 1.0f, 0.0f, 0.0f, nullptr);
    DASH_TRY(gemm(prec, B, nc, bT, 0, opR, 0, e, st));
  }
  return DASH_OK;
}

dash_status precondition_apply(const void* G, int gdt, const float* Froot, int64_t Ng, int B,
                               int prec, float* U, void* ws, size_t ws_bytes, void* stream) {
  if (!U && Ng > 0) return DASH_ERR_INVALID_ARG;
  return apply_impl(G, gdt, Froot, Ng, B, prec, U, nullptr, 0.0f, ws, ws_bytes, stream);
}

dash_status precondition_update(const void* G, int gdt, const float* Froot, int64_t Ng, int B,
                                int prec, float lr, float* W, float* U, void* ws,
                                size_t ws_bytes, void* stream) {
  if (!W && Ng > 0) return DASH_ERR_INVALID_ARG;
  if (!std::isfinite(lr)) return DASH_ERR_INVALID_ARG;
  return apply_impl(G, gdt, Froot, Ng, B, prec, U, W, lr, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- block packing

static int dt_size(int dt) {
  return dt == DASH_DT_F32 ? 4 : (dt == DASH_DT_BF16 || dt == DASH_DT_F16) ? 2 : 0;
}

dash_status pack_blocks(const void* M, int dt, int64_t rows, int64_t cols, int64_t ld, int B,
                        void* blocks, int32_t* valid_rows, int32_t* valid_cols, void* stream) {
  const int es = dt_size(dt);
  if (es == 0 || rows < 0 || cols < 0 || ld < cols || !valid_dim(B)) return DASH_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return DASH_OK;
  if (!M || !blocks || (reinterpret_cast<uintptr_t>(M) % es) ||
      (reinterpret_cast<uintptr_t>(blocks) % es) ||
      (valid_rows && (reinterpret_cast<uintptr_t>(valid_rows) & 3u)) ||
      (valid_cols && (reinterpret_cast<uintptr_t>(valid_cols) & 3u)))
    return DASH_ERR_INVALID_ARG;
  return launch_pack_blocks(M, es, rows, cols, ld, B, blocks, valid_rows, valid_cols,
                            static_cast<cudaStream_t>(stream));
}

dash_status unpack_blocks(const void* blocks, int dt, int64_t rows, int64_t cols, int64_t ld,
                          int B, void* M, void* stream) {
  const int es = dt_size(dt);
  if (es == 0 || rows < 0 || cols < 0 || ld < cols || !valid_dim(B)) return DASH_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return DASH_OK;
  if (!M || !blocks || (reinterpret_cast<uintptr_t>(M) % es) ||
      (reinterpret_cast<uintptr_t>(blocks) % es))
    return DASH_ERR_INVALID_ARG;
  return launch_unpack_blocks(blocks, es, rows, cols, ld, B, M, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
