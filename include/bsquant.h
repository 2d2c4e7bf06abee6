/*
 * bsquant.h -- C ABI of the MX quantizer: real values -> block-scaled codes in
 * the layouts the block-scaled GEMM (bsgemm.h) consumes.
 *
 * Operation ("GEMM + RoPE + MXFP8 Projection (SM100)", section "Equations":
 * MXFP8 quantize -- an E8M0 scale per block with E4M3 data; "GEMM + Amax
 * (SM100)", sections "Parameters" and "Support surface and constraints", for
 * the E5M2 and packed E2M1 element formats and the scale atom layout):
 *
 *   for every row r of every batch l and every block b of sf_vec_size
 *   consecutive elements along the row:
 *     amax  = max |X[l, r, b*sfv .. b*sfv + sfv - 1]|
 *     e     = floor(log2 amax) - emax     (emax: E4M3 8, E5M2 15, E2M1 2),
 *             clamped to [-127, 127]
 *     SF    = e + 127                      (E8M0 byte)
 *     code  = X / 2^e rounded to the nearest value of the element format,
 *             ties to the even code, magnitudes past the largest finite value
 *             saturated to it, the sign kept
 *   An all-zero block gets SF 127; a block holding a NaN or an infinity gets
 *   SF 0xFF (E8M0 NaN) and the format's NaN code everywhere (E4M3 and E5M2
 *   0x7F; E2M1 has no NaN, so 0).  The pages name the operation but not the
 *   scale choice: this rule (the block maximum mapped into the element
 *   format's top binade) is the reading this library uses.
 *
 * Layouts:
 *   X      (L, rows, cols) fp32 or bf16, cols contiguous: element (l, r, k)
 *          at (l*rows + r)*cols + k.  Device memory, 16-byte aligned.
 *   codes  (L, rows, cols) FP8 bytes, or (L, rows, cols/2) packed E2M1 with
 *          element 2i in the low nibble of byte i -- the GEMM's A or B.
 *          Device memory, 16-byte aligned.
 *   SF     the GEMM's physical atom tensor (L, ceil(rows/128),
 *          ceil(cols/(4*sfv)), 32, 4, 4) of E8M0 bytes; row r = 128*t + 32*m1
 *          + m0 and block kb = 4*kt + kin at [l, t, kt, m0, m1, kin].  Every
 *          byte is written: padding positions (rows >= rows, blocks >=
 *          cols/sfv) get 127.  Device memory, 16-byte aligned.
 *
 * Columnwise (direction BSG_QUANT_COLWISE; "GEMM + RoPE + MXFP8 Projection
 * (SM100)", sections "Overview" and "Equations": MXFP8_S, blocks along the
 * tokens, the non-contiguous dimension): the same rule with each block 32
 * consecutive ROWS of one column.
 *   X      as above.  cols a multiple of 16, rows a multiple of 32.
 *   codes  (L, rows, cols) FP8 bytes in X's layout.  Read by the GEMM with
 *          rows as K and cols as M (or N), this is its m-major A (n-major
 *          B): strides (1, cols, cols*rows).
 *   SF     the GEMM's atom tensor for that operand: (L, ceil(cols/128),
 *          ceil(rows/128), 32, 4, 4); the scale of column c, block b sits
 *          where the GEMM reads row mn = c, K-block kb = b.  Padding
 *          positions (columns >= cols, blocks >= rows/32) get 127.  (The
 *          page prints its S-direction scales as a plain (tokens/32, ...,
 *          D) array; these are the same bytes in the atom layout the GEMM
 *          consumes.)
 *   E4M3 or E5M2 codes and sf_vec_size 32 only (the GEMM's MN-major
 *   operands are FP8): E2M1 or sf_vec_size 16 is BSG_ERR_UNSUPPORTED, rows
 *   not a multiple of 32 BSG_ERR_UNSUPPORTED, cols not a multiple of 16
 *   BSG_ERR_ALIGNMENT.
 *
 * Ownership: the caller owns X, codes and SF.  bsg_quantize allocates
 * nothing, never synchronises and enqueues one kernel on `stream` (a
 * cudaStream_t, NULL for the legacy default stream).
 *
 * Errors: every check happens before the launch and returns a bsg_status
 * (bsgemm.h); nothing aborts.  BSG_ERR_INVALID_ARG for an empty or oversized
 * shape or an unknown dtype, BSG_ERR_UNSUPPORTED for FP8 with sfv 16 or cols
 * not a multiple of sf_vec_size, BSG_ERR_ALIGNMENT for a pointer that is not
 * 16-byte aligned, BSG_ERR_ARCH off an sm_103 device, BSG_ERR_CUDA for a
 * failed CUDA call.
 */
#ifndef BSQUANT_H_
#define BSQUANT_H_

#include <stddef.h>
#include <stdint.h>

#include "bsgemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Direction of the scale blocks ("GEMM + RoPE + MXFP8 Projection (SM100)",
 * "Overview": rowwise (D-direction) and columnwise (S-direction)). */
typedef enum {
  BSG_QUANT_ROWWISE = 0,  /* blocks along each row (the contiguous cols) */
  BSG_QUANT_COLWISE = 1   /* blocks down each column (32 consecutive rows) */
} bsg_quant_direction;

typedef struct {
  int64_t rows, cols, L;  /* X is (L, rows, cols), cols contiguous */
  bsg_dtype in_dtype;     /* BSG_F32 or BSG_BF16 */
  bsg_dtype out_dtype;    /* BSG_E4M3, BSG_E5M2 or BSG_E2M1 (rowwise only) */
  int sf_vec_size;        /* 32; or 16 for BSG_E2M1 */
  int direction;          /* bsg_quant_direction; 0 (rowwise) for zero-initialised requests */
} bsg_quant_problem;

/* Host-only validation of a request against the rules above. */
bsg_status bsg_quant_check(const bsg_quant_problem* q);

/* Bytes of the code tensor and of the (padded) scale atom tensor. */
bsg_status bsg_quant_sizes(const bsg_quant_problem* q, size_t* code_bytes, size_t* sf_bytes);

/* Quantize X into codes and SF in the request's direction (one launch on
 * `stream`). */
bsg_status bsg_quantize(const bsg_quant_problem* q, const void* X, void* codes, void* sf,
                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSQUANT_H_ */
