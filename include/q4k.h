/*
 * q4k.h -- the second codec of libmxfp4.so: GGUF Q4_K weights, f32 activations,
 * on the GPU.  Status codes, pointer rules and stream semantics are those of
 * mxfp4.h (MXFP4_STATUS_*; device pointers 16-byte aligned; work enqueued on
 * `stream`, nothing enqueued on a refusal).
 *
 * Layout ("rlx-cpu 0.2.17 src/gguf_matmul.rs": the block layout its Q4_K block
 * dot reads, q4k_dot_q8_block_avx2 with q4k_scale_min_x86).  A [rows, cols]
 * matrix, cols a multiple of 256, is rows x cols/256 super-blocks of 144 bytes,
 * row-major.  A super-block holds 256 consecutive elements of a row:
 *   bytes 0-1    d, IEEE binary16, little-endian
 *   bytes 2-3    dmin, binary16
 *   bytes 4-15   the 6-bit scale sc_j and min m_j of its eight 32-element
 *                sub-blocks j: for j < 4 the low six bits of bytes 4+j (sc) and
 *                8+j (m); for j >= 4 the low / high nibble of byte 12+(j-4)
 *                give the low four bits of sc / m and the top two bits of
 *                bytes 4+(j-4) / 8+(j-4) their high two bits
 *   bytes 16-143 codes q: byte 16 + 32 s + l (s < 4, l < 32) holds element
 *                64 s + l in its low nibble (sub-block 2 s) and element
 *                64 s + 32 + l in its high nibble (sub-block 2 s + 1)
 * Element value: w = d * sc_j * q - dmin * m_j, as the exact arm of the page's
 * decode GEMV computes it (gguf_matmul_bt_m1_parallel: each super-block
 * dequantised to f32 on the fly, activations kept in f32): both products exact
 * in FP32, one FP32 rounding of the difference.
 */
#ifndef Q4K_H
#define Q4K_H

#include "mxfp4.h"

#ifdef __cplusplus
extern "C" {
#endif

/* rows * cols/256 * 144, or 0 when cols % 256 != 0 or a size is not positive. */
size_t q4k_nbytes(int rows, int cols);

/* Whole matrix to FP32: out[r*cols + c] = w[r][c] (the element values above,
 * bit for bit).  w: q4k_nbytes(rows, cols) bytes; out: rows*cols floats. */
int q4k_dequant(const void* w, int rows, int cols, float* out, cudaStream_t stream);

/* y[r] = sum_c w[r][c] * x[c] in FP32 on the CUDA cores: each element decoded to
 * its FP32 value and multiplied into FP32 sums (two chains per 32-bit code
 * word, four sums per lane by super-block mod 4, then a fixed warp tree).
 * Error bound: |y - exact| <= 1e-5 * sum_c |w[r][c] x[c]| for rows up to 32768
 * columns.  Deterministic: the order of every sum depends on the shape only.
 * x: [cols] floats, y: [rows] floats.  (The page's exact arm, m == 1.) */
int q4k_mv(const void* w, int rows, int cols, const float* x, float* y, cudaStream_t stream);

/* Y[t*rows + r] = sum_c w[r][c] * X[t*cols + c], t < nb: each code word decoded
 * once for up to 8 tokens per pass over the weights; per token the result
 * equals q4k_mv on that token bit for bit.  X: [nb, cols], Y: [nb, rows]
 * (the page's gguf_matmul_bt_m1_rows_generic idea: each block decoded once and
 * reused across the batch). */
int q4k_mm(const void* w, int rows, int cols, const float* X, int nb, float* Y,
           cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4K_H */
