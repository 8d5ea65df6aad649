/*
 * dashroot: the batched block-preconditioner step of DASH-style Shampoo on
 * NVIDIA GB300 (sm_103a).
 *
 * Method source: "DASH: Faster Shampoo via Batched Block Preconditioning and
 * Efficient Inverse-Root Solvers" (arXiv 2602.02016), as summarised by
 *   [pt]  gist.science/pt technical summary ("Definicao do Problema",
 *         "Metodologia" 1-2, "Principais Contribuicoes", "Resultados")
 *   [tg]  tgviewer.app, Telegram channel quant_prune_distill, post 646
 *   [abs] arxivdaily.com, the authors' abstract
 * The pages name the operations below and their properties but print no
 * formulas; each entry point states the reading it implements.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Stacks.  A stack of N square blocks of order B is one contiguous row-major
 *   (N, B, B) array; block k starts B*B elements after block k-1 ([pt]
 *   Metodologia 1, "Empilhamento de Tensores 3D": blocks stacked into an
 *   (N, B, B) tensor and processed together).  B must be a multiple of 128 with
 *   128 <= B <= 2048.  N >= 0; N == 0 is a no-op returning DASH_OK.
 * Memory.  Every pointer is caller-owned DEVICE memory unless stated
 *   otherwise, 16-byte aligned (else DASH_ERR_INVALID_ARG).  Inputs are const
 *   and are never written.  Outputs must not overlap inputs or the workspace,
 *   except where an argument says "in place".
 * Execution.  Work is enqueued on the caller's CUDA stream (a cudaStream_t
 *   passed as void*, NULL = legacy default stream) and runs asynchronously.
 *   No entry point allocates device memory or synchronises the stream.
 * Workspace.  Entry points that take (ws, ws_bytes) use that caller-owned
 *   device scratch; dash_workspace_size gives the size that lets a call
 *   process all N blocks in one pass.  A smaller workspace is accepted as long
 *   as it holds the per-call arrays plus one block's iterates: the call then
 *   walks the stack in chunks of as many blocks as fit.  Too small for one
 *   block: DASH_ERR_WORKSPACE_TOO_SMALL.  The workspace needs 256-byte
 *   alignment.
 * Precision.  dash_prec selects the tensor-core arithmetic of the dense
 *   B x B x B products: DASH_FP32_3XTF32 (each fp32 operand split into two
 *   TF32 parts, three TF32 products per tile, fp32-level accuracy),
 *   DASH_TF32, DASH_FP16 and DASH_BF16 (operands and stored iterates in that
 *   format).  All accumulation is fp32; every epilogue computes in fp32.
 * Errors.  Argument errors are detected on the host before anything is
 *   enqueued.  CUDA launch errors return DASH_ERR_CUDA.  A device-side wait
 *   that exceeds its time limit never traps: the kernel records
 *   DASH_ERR_TIMEOUT in a device flag and returns; dash_device_status reads
 *   and clears that flag.  Non-finite numbers are not errors: they propagate
 *   into the outputs and residuals.
 * Concurrency.  Calls on one stream run in order.  Calls on different streams may
 *   overlap, with their own workspaces, as long as fewer than 4096 of the
 *   library's matrix-product launches (at most a few dozen per call) are in
 *   flight at once: the products that write symmetric fp32 results (the
 *   accumulate, the roots) hand out their tiles from one of 4096 counters per
 *   device, tagged with the launch.  A launch that finds its counter taken by a
 *   later launch stops and records DASH_ERR_CONFLICT for dash_device_status; its
 *   outputs are then incomplete.  Launches captured in a CUDA graph may be
 *   replayed.
 */
#ifndef DASHROOT_H
#define DASHROOT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DASH_OK = 0,
  DASH_ERR_INVALID_ARG = 1,
  DASH_ERR_UNSUPPORTED = 2,
  DASH_ERR_CUDA = 3,
  DASH_ERR_WORKSPACE_TOO_SMALL = 4,
  DASH_ERR_TIMEOUT = 5,
  DASH_ERR_CONFLICT = 6
} dash_status;

typedef enum {
  DASH_FP32_3XTF32 = 0,
  DASH_TF32 = 1,
  DASH_FP16 = 2,
  DASH_BF16 = 3
} dash_prec;

/* Flag OR-ed into the prec argument (no counterpart on the pages: it only moves
 * a rounding step).
 *   inv_root_cn / inv_root_ndb / inv_root_cheb: X is written rounded to TF32
 *     (round to nearest, ties away from zero; fp32 container), the operand form
 *     of DASH_TF32 products.  The solver's arithmetic is unchanged.
 *   precondition_apply / precondition_update, with DASH_TF32 only: Froot
 *     already holds TF32-rounded roots (e.g. written with this flag) and the
 *     products read it as it is, without the conversion pass they otherwise
 *     make over both roots (results identical on such roots).
 * Anywhere else: DASH_ERR_INVALID_ARG. */
#define DASH_ROOT_TF32 0x100

typedef enum { DASH_DT_F32 = 0, DASH_DT_BF16 = 1, DASH_DT_F16 = 2 } dash_dtype;

/* Inverse-root solvers, for per-block solver selection. */
typedef enum { DASH_SOLVER_CN = 0, DASH_SOLVER_NDB = 1, DASH_SOLVER_CHEB = 2 } dash_solver;

/* One tier of per-block solver selection: a solver, its precision and iteration
 * count (degree for Chebyshev), the unit roundoff u its iterates are stored at,
 * and the relative error gate it is held to. */
typedef struct {
  int solver;  /* dash_solver */
  int prec;    /* dash_prec */
  int iters;   /* >= 1 */
  double u;    /* > 0 */
  double gate; /* > 0 */
} dash_tier;

typedef enum {
  DASH_SCALE_POWER = 0,
  DASH_SCALE_FROBENIUS = 1,
  DASH_SCALE_POWER_F16 = 2,
  DASH_SCALE_POWER_BF16 = 3
} dash_scale_mode;

typedef enum {
  DASH_OP_ACCUMULATE = 0,
  DASH_OP_SPECTRAL_SCALE = 1,
  DASH_OP_INV_ROOT_CN = 2,
  DASH_OP_INV_ROOT_NDB = 3,
  DASH_OP_INV_ROOT_CHEB = 4,
  DASH_OP_PRECONDITION_APPLY = 5,
  DASH_OP_LAMBDA_MIN = 6
} dash_op;

/*
 * shampoo_accumulate -- EMA update of the stacked Shampoo factors.
 * Source: [tg] second paragraph (Shampoo keeps L and R built from gradient
 * products and raises them to the -1/4 power), [tg] block-diagonal paragraph
 * (L and R of all blocks stacked in one tensor), [pt] Metodologia 1.
 * Reading: for every gradient block j < Ng
 *     F[j]      <- beta F[j]      + (1 - beta) G_j G_j^T      (L_j)
 *     F[Ng + j] <- beta F[Ng + j] + (1 - beta) G_j^T G_j      (R_j)
 * then rows and columns >= valid_rows[j] of L_j (>= valid_cols[j] of R_j) are
 * reset to the identity's (0 off the diagonal, 1 on it) -- the treatment of a
 * zero-padded gradient block.
 *   G           (Ng, B, B) gradient blocks, dtype gdt (DASH_DT_BF16 runs
 *               bf16 tensor-core products, exact products with fp32
 *               accumulation; DASH_DT_F32 runs 3xTF32).
 *   F           (2*Ng, B, B) fp32 factors, updated IN PLACE.  Factors are
 *               symmetric: for B a multiple of 256 only the 256 x 256 tiles on or
 *               above the diagonal are computed (reading only those of the old
 *               F), and each tile below is then written as the transpose of its
 *               mirror (SYRK-style: 10 of 16 tiles at B = 1024).  With bf16 / fp16
 *               gradients the result is exactly symmetric; with fp32 gradients
 *               (3xTF32) the diagonal tiles, computed whole, are symmetric to
 *               rounding.  Other B compute every element.
 *   valid_rows, valid_cols  (Ng,) int32 device arrays, or NULL (= B).
 *   ws/ws_bytes workspace; only DASH_DT_F32 needs one (see dash_workspace_size).
 */
dash_status shampoo_accumulate(const void* G, int gdt, int64_t Ng, int B, float beta,
                               float* F, const int32_t* valid_rows,
                               const int32_t* valid_cols, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * spectral_scale -- per-block scale s_k for the iterative root solvers.
 * Source: [pt] Metodologia 2, "Multi-Power-Iteration para Escalonamento"
 * (lambda_max from up to 32 start vectors run in parallel), [tg] paragraph on
 * scaling (Rayleigh-quotient estimate instead of the Frobenius norm), [pt]
 * Definicao do Problema item 3 (Frobenius scaling).
 *   mode DASH_SCALE_POWER: with V = V0[k] (B x n_vec, row-major, fp32), take
 *     power_iters products W = (A_k + ridge I) V; after every product but the
 *     last, normalise each column of W to unit 2-norm and continue with it;
 *     after the last, lambda_out[k] = max_j (v_j . w_j) / (v_j . v_j).
 *     1 <= n_vec <= 32, power_iters >= 1, V0 (N, B, n_vec) fp32.
 *   mode DASH_SCALE_POWER_F16 / _BF16: the same iteration in half precision
 *     ([pt] Principais Contribuicoes item 4, the half-precision power iteration
 *     among the contributions): sigma_k A_k is rounded once to fp16 / bf16, each product
 *     takes 16-bit A and 16-bit vectors with fp32 accumulation, the ridge term
 *     (sigma_k ridge), the column normalisation and the Rayleigh quotients are
 *     fp32, the vectors are stored in the 16-bit format between products, and the
 *     result is divided by sigma_k.  sigma_k is the power of two that brings
 *     max(max_i |A_k[i][i]|, |ridge|) into [1/2, 1); it is exact, so a block whose
 *     16-bit copy would neither overflow nor underflow gets the same lambda as
 *     with sigma_k = 1, and a positive semidefinite block (|A_ij| <= max_i A_ii)
 *     stays within fp16's range whatever its magnitude.  For B <= 1024, B a
 *     multiple of 128, the whole iteration is one launch that reads each fp32
 *     block once and keeps its 16-bit copy in L2 (thread-block clusters; it needs
 *     three 16-bit block slots of workspace besides the vectors, which
 *     dash_workspace_size covers); otherwise, or with less workspace, each product
 *     is one launch over a 16-bit copy of the whole stack.  Both round the same
 *     values to the same formats; their fp32 sums run in different orders.
 *   mode DASH_SCALE_FROBENIUS: lambda_out[k] = ||A_k + ridge I||_F
 *     (n_vec, power_iters, V0 ignored; may be 0 / NULL).
 *   A (N, B, B) fp32 symmetric blocks; lambda_out (N,) fp32.
 * Arithmetic: POWER runs the products on the tensor cores in 3xTF32 (fp32-level
 *   accuracy) with fp32 column sums; the half modes as stated; FROBENIUS fp32
 *   partial sums.
 * Workspace: dash_workspace_size(DASH_OP_SPECTRAL_SCALE, N, B, prec, n_vec) with
 *   prec DASH_FP16 / DASH_BF16 for the half modes (it then includes the 16-bit
 *   copy of sigma A, 2 B^2 bytes per block, and sigma, 4 bytes per block), any
 *   other prec for POWER and FROBENIUS.
 */
dash_status spectral_scale(const float* A, float ridge, int64_t N, int B, int mode,
                           int n_vec, int power_iters, const float* V0,
                           float* lambda_out, void* ws, size_t ws_bytes, void* stream);

/*
 * inv_root_cn -- Coupled Newton inverse 4th root of every block.
 * Source: [pt] Definicao do Problema item 2 and [tg] list item 1 (Coupled
 * Newton, a matmul-only iteration for matrix roots).  Reading (coupled inverse
 * p-th root iteration, p = 4): A_s = (A_k + ridge I) / scale[k];
 *   X_0 = I, M_0 = A_s;  T_i = (5I - M_i)/4;  X_{i+1} = X_i T_i;
 *   M_{i+1} = (T_i^2)^2 M_i;   X[k] = scale[k]^{-1/4} X_iters.
 * 4*iters - 4 products per block for iters >= 2, none for iters = 1 (iteration 0
 * needs no X product, the last no M update).  Every iterate is a polynomial in
 * the symmetric A_s, so for B a multiple of 256 a product may compute and store
 * only its 256 x 256 tiles on or above the diagonal (10 of 16 at B = 1024); X's
 * tiles below the diagonal are written as their mirrors' transposes.  A's tiles
 * below the diagonal then do not affect X, so A must be symmetric, as a factor is.
 * Arithmetic by precision:
 *   DASH_FP32_3XTF32: the identity-shifted form of the same iteration (T stored
 *     as D = T - I; X T = X + X D, T^2 = I + D D + 2D, ..., each large term added
 *     exactly in fp32), products with round-to-nearest partial sums, every
 *     product in symmetric halves.
 *   DASH_FP16 / DASH_BF16: M is carried as a 16-bit pair (hi + lo, about 22 bits
 *     in fp16) through all but the last three M updates (two products per slice);
 *     the T^2, T^4 and M products are computed whole (a symmetric-half product
 *     would turn the antisymmetric part of their rounding into error in M's
 *     smallest eigenvalues), except in the first iteration (T_0 exactly
 *     symmetric: T^2, T^4 in halves) and the last M update (its error meets X
 *     in one factor only: all three in halves); the X product in halves.
 *   DASH_TF32: plain, every product in symmetric halves.
 *   A (N, B, B) fp32; scale (N,) fp32 > 0 (e.g. from spectral_scale);
 *   iters >= 1; prec any dash_prec; X (N, B, B) fp32 output;
 *   resid_out (N, iters) fp32 or NULL: resid_out[k*iters + i] =
 *   ||M_i - I||_F / sqrt(B), the residual ||X_i^4 A_s - I|| of iterate i.
 */
dash_status inv_root_cn(const float* A, float ridge, const float* scale, int64_t N, int B,
                        int iters, int prec, float* X, float* resid_out, void* ws,
                        size_t ws_bytes, void* stream);

/*
 * inv_root_ndb -- Newton-Denman-Beavers inverse 4th root of every block.
 * Source: [pt] Metodologia 2, NDB bullet (yields square root and inverse
 * square root together; first iteration trimmed; three products per step,
 * fewer in practice), [tg] list item 2.  Reading (matmul-only Newton-Schulz
 * form of Denman-Beavers): one stage on C runs Y_0 = C, Z_0 = I,
 *   T_i = (3I - Z_i Y_i)/2, Y_{i+1} = Y_i T_i, Z_{i+1} = T_i Z_i;
 * stage 1 on C = A_s keeps Y (~A_s^{1/2}); stage 2 on C = that Y keeps Z
 * (~A_s^{-1/4}); X[k] = scale[k]^{-1/4} Z.  iters counts iterations PER STAGE;
 * 6*iters - 6 products per block for iters >= 2 (one for iters = 1).
 *   resid_out (N, 2, iters) fp32 or NULL: ||Z_i Y_i - I||_F / sqrt(B) per stage.
 *   Other arguments as inv_root_cn.  Half precision runs but the pages report
 *   it unstable ([pt] Resultados, Precisao).  Every product is computed whole.
 *   DASH_FP32_3XTF32 runs the identity-shifted form (T stored as D = T - I;
 *   Y T = Y + Y D, T Z = Z + D Z, the large term added exactly in fp32) with
 *   round-to-nearest partial sums.
 */
dash_status inv_root_ndb(const float* A, float ridge, const float* scale, int64_t N, int B,
                         int iters, int prec, float* X, float* resid_out, void* ws,
                         size_t ws_bytes, void* stream);

/*
 * inv_root_cheb -- Chebyshev/Clenshaw inverse 4th root of every block.
 * Source: [pt] Metodologia 2, Chebyshev bullet (Clenshaw's algorithm to
 * approximate matrix powers).  Reading: p = degree-d interpolant of x^{-1/4}
 * at the d+1 first-kind Chebyshev points of [lo, hi] (coefficients computed on
 * the host in double); S = (2 A_s - (lo+hi) I)/(hi - lo);
 *   b_{d+1} = b_{d+2} = 0, b_j = c_j I + 2 S b_{j+1} - b_{j+2},
 *   P = c_0 I + S b_1 - b_2,  X[k] = scale[k]^{-1/4} P.
 * d - 1 products per block.  1 <= degree <= 64, 0 < lo < hi.  For B a multiple
 * of 256 every product keeps symmetric halves as in inv_root_cn.
 */
/*
 * dash_select_tiers -- per-block solver selection by a condition estimate (host
 * code, no GPU needed).  Source: [pt] Significancia e Alegacoes, item Direcoes
 * Futuras (choosing the solver per block from its condition number, named as
 * future work).  Reading: kappa_k = lam_max[k] / lam_min[k] in double (+inf
 * unless both values are positive, NaN included); choice[k] = the first tier t, in the
 * given order (cheapest first), with kappa_k * u_t / 4 <= gate_t, else the last
 * tier.  (Storing the scaled block at roundoff u moves its smallest eigenvalue,
 * about 1/kappa, by about kappa u relative, and its inverse 4th root by a quarter
 * of that.)
 *   lam_max, lam_min (n,) and choice (n,) are caller-owned HOST arrays; tiers
 *   (ntiers >= 1) likewise.  DASH_ERR_INVALID_ARG for n < 0, null pointers (when
 *   n > 0) or a tier with an unknown solver or precision, iters < 1, u <= 0 or
 *   gate <= 0.
 */
dash_status dash_select_tiers(const float* lam_max, const float* lam_min, int64_t n,
                              const dash_tier* tiers, int ntiers, int32_t* choice);

/*
 * spectral_lambda_min -- a lambda_min estimate per block, for per-block solver
 * selection.  Source: [pt] Significancia e Alegacoes, item Direcoes Futuras
 * (solver choice from each block's condition number).  Reading: the power
 * iteration of spectral_scale (mode DASH_SCALE_POWER, _POWER_F16 or _POWER_BF16,
 * same n_vec, power_iters and V0 conventions) on the shifted block
 * c_k I - (A_k + ridge I), c_k = lam_max[k], gives mu_k, and
 * lam_min_out[k] = c_k - mu_k.  The shifted block's eigenvalues are c_k - lambda_i;
 * a Rayleigh quotient never exceeds the largest, so (up to rounding)
 * lam_min_out[k] >= lambda_min(A_k + ridge I): the estimate errs toward a
 * better-conditioned block.
 *   A (N, B, B) fp32 symmetric; lam_max (N,) fp32 > 0 (e.g. spectral_scale's
 *   output); lam_min_out (N,) fp32.
 * Workspace: dash_workspace_size(DASH_OP_LAMBDA_MIN, N, B, prec, n_vec) (prec
 *   DASH_FP16 / DASH_BF16 for the half modes) holds the shifted stack (4 B^2 bytes
 *   per block) and spectral_scale's workspace for all N blocks; a smaller one walks
 *   the stack in chunks.
 */
dash_status spectral_lambda_min(const float* A, float ridge, const float* lam_max, int64_t N,
                                int B, int mode, int n_vec, int power_iters, const float* V0,
                                float* lam_min_out, void* ws, size_t ws_bytes, void* stream);

/*
 * inv_root_auto -- inverse 4th roots with the solver chosen per block.  Source:
 * [pt] Significancia e Alegacoes, item Direcoes Futuras.  Reading: block k's tier
 * is dash_select_tiers(lam_max, lam_min, tiers)[k]; the blocks of each tier are
 * solved by that tier's solver (Coupled Newton or NDB with `iters` iterations,
 * Chebyshev of degree `iters` on [cheb_lo, cheb_hi]) in its precision, scaled by
 * lam_max exactly as inv_root_cn / _ndb / _cheb scale, and written to X[k].
 *   A (N, B, B) fp32; lam_max, lam_min (N,) fp32 device arrays (spectral_scale,
 *   spectral_lambda_min); tiers (ntiers >= 1, cheapest first) HOST array as for
 *   dash_select_tiers; X (N, B, B) fp32 output; choice_out (N,) int32 HOST array
 *   or NULL: receives each block's tier.
 * Synchronisation: unlike every other entry point, this one reads lam_max and
 *   lam_min back to the host and so synchronises `stream`, once; a tier whose
 *   blocks are not one contiguous range is gathered into a sub-stack of the
 *   workspace, solved and scattered back, and uploading its index list waits for
 *   the stream again.  A tier that is one contiguous range is solved in place.
 * Workspace: dash_auto_workspace_size (the worst case: every block in one
 *   gathered tier); a smaller one walks each gathered tier in chunks.
 * Errors: as dash_select_tiers for the tiers; DASH_ERR_INVALID_ARG for a
 *   Chebyshev tier with degree > 64 or a bad interval.
 */
dash_status inv_root_auto(const float* A, float ridge, const float* lam_max,
                          const float* lam_min, int64_t N, int B, const dash_tier* tiers,
                          int ntiers, double cheb_lo, double cheb_hi, float* X,
                          int32_t* choice_out, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes of inv_root_auto on N blocks of order B with these tiers. */
dash_status dash_auto_workspace_size(int64_t N, int B, const dash_tier* tiers, int ntiers,
                                     size_t* bytes);

/*
 * dash_cheb_coeffs -- the host-side coefficients inv_root_cheb uses (host code,
 * no GPU needed): c[0..degree] of the degree-d interpolant of x^{-1/4} at the d+1
 * first-kind Chebyshev points of [lo, hi], in the Chebyshev basis of
 * t = (2x - lo - hi)/(hi - lo), computed in double.  c (degree + 1) is
 * caller-owned host memory.  Same argument limits as inv_root_cheb;
 * DASH_ERR_INVALID_ARG otherwise.
 */
dash_status dash_cheb_coeffs(int degree, double lo, double hi, double* c);

dash_status inv_root_cheb(const float* A, float ridge, const float* scale, int64_t N, int B,
                          int degree, double lo, double hi, int prec, float* X, void* ws,
                          size_t ws_bytes, void* stream);

/*
 * precondition_apply -- the preconditioned update U_j = L_j^{-1/4} G_j R_j^{-1/4}.
 * Source: [tg] second paragraph (the -1/4 powers of L and R precondition the
 * gradient).  Froot (2*Ng, B, B) fp32 holds the roots in the factor order of
 * shampoo_accumulate (L roots, then R roots).  G (Ng, B, B) of dtype gdt;
 * U (Ng, B, B) fp32 output.  Two products per block in precision prec.
 */
dash_status precondition_apply(const void* G, int gdt, const float* Froot, int64_t Ng,
                               int B, int prec, float* U, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * precondition_update -- the weight step along the preconditioned direction,
 * W_j <- W_j - lr * L_j^{-1/4} G_j R_j^{-1/4}, fused into the second product of
 * precondition_apply (its epilogue reads W_j and writes the stepped W_j in place).
 * Source: [tg] second paragraph (the preconditioned gradient) for U; the pages
 * give no optimizer update rule, and the reading taken is the plain step
 * W - lr U.  W (Ng, B, B) fp32 weights in the block layout of G, updated IN
 * PLACE (padded rows / columns of a block stay as they are: U is zero there);
 * U (Ng, B, B) fp32 or NULL: when given, also receives U.  lr finite.  Workspace
 * as for precondition_apply (DASH_OP_PRECONDITION_APPLY).
 */
dash_status precondition_update(const void* G, int gdt, const float* Froot, int64_t Ng,
                                int B, int prec, float lr, float* W, float* U, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * pack_blocks / unpack_blocks -- a weight-shaped matrix <-> its stack of B x B
 * blocks.  Source: [pt] Metodologia 1 ("Empilhamento de Tensores 3D": gradient
 * blocks G_ij stacked into (N, B, B)).  M is row-major (rows, cols) with leading
 * dimension ld >= cols, dtype dt (DASH_DT_F32, DASH_DT_BF16, DASH_DT_F16;
 * element-aligned); blocks is (nbr * nbc, B, B) of the same dtype with
 * nbr = ceil(rows / B), nbc = ceil(cols / B), enumerated row-block-major: block
 * i * nbc + j holds rows i*B.. and columns j*B.. of M.
 *   pack_blocks zero-fills each block beyond the matrix and, when valid_rows /
 *   valid_cols (int32, nbr * nbc) are given, writes each block's valid extent
 *   min(B, rows - i*B) / min(B, cols - j*B) -- the arrays shampoo_accumulate
 *   takes.  unpack_blocks writes back the valid part only.  rows or cols = 0 is
 *   a no-op.  Bit copies: no conversion.
 */
dash_status pack_blocks(const void* M, int dt, int64_t rows, int64_t cols, int64_t ld, int B,
                        void* blocks, int32_t* valid_rows, int32_t* valid_cols, void* stream);
dash_status unpack_blocks(const void* blocks, int dt, int64_t rows, int64_t cols, int64_t ld,
                          int B, void* M, void* stream);

/*
 * dash_gemm -- the batched tensor-core product the solvers are built from,
 * exposed for tests and roofline measurement (no counterpart on the pages).
 * C[k] = op(A[k]) op(B[k]) for k < N, op = transpose when trans_* != 0.
 * Operands are already in the format of prec: fp32 containers for TF32 (the
 * tensor core reads their TF32 part), fp32 hi and lo arrays for
 * DASH_FP32_3XTF32 (A_lo / B_lo; C = hi*hi + hi*lo + lo*hi), 16-bit arrays
 * for DASH_FP16 / DASH_BF16 (A_lo, B_lo ignored).  C (N, B, B) fp32.
 */
dash_status dash_gemm(const void* A, const void* A_lo, int trans_a, const void* Bm,
                      const void* B_lo, int trans_b, int64_t N, int B, int prec, float* C,
                      void* stream);

/*
 * dash_gemm_ex -- dash_gemm with the two operand forms the root solvers use, for
 * tests (no counterpart on the pages).
 *   sym 0: as dash_gemm.  sym 1: A and B symmetric; only their 256 x 256 tiles on
 *   or above the diagonal are read (a tile below is taken as its mirror's
 *   transpose).  sym 2: as 1, and only C's tiles on or above the diagonal are
 *   computed and written (C symmetric by construction).  sym 3: A and B read whole,
 *   only C's tiles on or above the diagonal computed and written.  sym 4: A
 *   symmetric and read from its upper tiles as in 1, B read whole, C whole.
 *   Modes 1-4 apply for B a multiple of 256 and act as 0 otherwise.
 *   With prec DASH_FP16 / DASH_BF16, a non-NULL B_lo makes B a 16-bit pair:
 *   C = A B + A B_lo, both products in that 16-bit type (A_lo ignored).
 */
dash_status dash_gemm_ex(const void* A, const void* A_lo, int trans_a, const void* Bm,
                         const void* B_lo, int trans_b, int64_t N, int B, int prec, int sym,
                         float* C, void* stream);

/*
 * spectral_scale_noalloc -- spectral_scale for callers that cannot allocate
 * device memory when they run (work being captured into a CUDA graph, hooks
 * inside another framework's memory manager, fixed-budget or real-time loops).
 * The pages have no counterpart: it is spectral_scale with its scratch taken
 * from a static device array of DASH_NOALLOC_SCRATCH_BYTES (32 MiB) built into
 * the library, which every GPU that loads the library keeps until the process
 * exits.  Arguments and results are those of spectral_scale without ws/ws_bytes.
 *   Limit: one pass over all N blocks must fit the array, i.e.
 *   dash_workspace_size(DASH_OP_SPECTRAL_SCALE, N, B, prec, n_vec) <= 32 MiB,
 *   with prec DASH_FP16 / DASH_BF16 for the half modes.  With 32 vectors that is
 *     DASH_SCALE_POWER            N <= 127 at B = 1024 (1012 at 128, 63 at 2048);
 *     DASH_SCALE_POWER_F16 / BF16 N <= 15 at B = 1024 (677 at 128, 3 at 2048),
 *       because these modes also keep a 16-bit copy of every block there;
 *     DASH_SCALE_FROBENIUS        4*N bytes.
 *   Larger requests return DASH_ERR_WORKSPACE_TOO_SMALL before anything is
 *   enqueued.
 *   No cudaMalloc, cudaFree or other allocating call is made.  The first call on
 *   each device looks up the array's device address (cudaGetSymbolAddress), so
 *   make that first call before any stream capture.
 *   All calls share the one array and it keeps the previous call's contents
 *   (the call clears what it accumulates before use); calls that may overlap
 *   on the GPU -- different streams, or different host threads -- race on it
 *   and must be serialised by the caller.
 */
#define DASH_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
dash_status spectral_scale_noalloc(const float* A, float ridge, int64_t N, int B, int mode,
                                   int n_vec, int power_iters, const float* V0,
                                   float* lambda_out, void* stream);

/* Workspace bytes for op on N blocks of order B (param: iters for CN/NDB,
 * degree for Chebyshev, n_vec for spectral_scale; gdt for accumulate/apply is
 * taken from prec: pass DASH_FP32_3XTF32 for fp32 gradients). */
dash_status dash_workspace_size(int op, int64_t N, int B, int prec, int param,
                                size_t* bytes);

/* Dense B x B x B products one call of op issues per block (the matmul
 * counts stated above). */
int64_t dash_op_matmuls(int op, int param);

/*
 * Kernel trace, for benchmarks (no counterpart on the pages).  While a trace
 * is active, every kernel the library launches is bracketed by a pair of CUDA
 * events recorded on the stream it is launched on, with the kernel's class and
 * its algorithmic work.  dash_trace_start(capacity) begins a trace of up to
 * capacity launches (events are created once and reused; further launches are
 * not recorded); dash_trace_count() gives the number recorded so far;
 * dash_trace_read(i, ...) waits for record i's end event and returns its class
 * (dash_trace_kind), algorithmic flops (2 B^3 per block for a product, any
 * precision), algorithmic bytes and device milliseconds; dash_trace_stop() ends
 * the trace.  Host-side state, one trace per process; not thread-safe against
 * concurrent library calls on other threads.
 */
typedef enum {
  DASH_TRACE_GEMM_F16 = 0,
  DASH_TRACE_GEMM_BF16 = 1,
  DASH_TRACE_GEMM_TF32 = 2,
  DASH_TRACE_GEMM_3XTF32 = 3,
  DASH_TRACE_ELEMENTWISE = 4,
  DASH_TRACE_POWER = 5,
  DASH_TRACE_REDUCE = 6,
  DASH_TRACE_PACK = 7
} dash_trace_kind;

dash_status dash_trace_start(int capacity);
int dash_trace_count(void);
dash_status dash_trace_read(int i, int* kind, double* flops, double* bytes, float* ms);
dash_status dash_trace_stop(void);

/* Reads and clears the device-side error flags of the current device
 * (DASH_OK, DASH_ERR_TIMEOUT, or DASH_ERR_CONFLICT: see "Concurrency" above).
 * Synchronises the device. */
dash_status dash_device_status(void);

/* Failure-detection self-test (no counterpart on the pages): enqueues one
 * kernel whose bounded device wait, on a barrier nothing arrives on, runs out
 * after limit_us microseconds (1 .. 1e6).  It takes the same time-out path as
 * every pipeline wait of the library: the kernel records DASH_ERR_TIMEOUT and
 * returns, so the next dash_device_status() reports DASH_ERR_TIMEOUT and the
 * CUDA context stays usable.  Nothing else is touched. */
dash_status dash_selftest_wait_timeout(int limit_us, void* stream);

const char* dash_status_string(int status);

/* Library version, e.g. "dashroot 0.1 sm_103a". */
const char* dash_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DASHROOT_H */
