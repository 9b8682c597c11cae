/*
 * mxfp4_oracle.h -- the CPU oracle for the MXFP4 dequant / matvec / small-batch
 * matmul / routed-expert path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously-correct
 * statement of what the GPU library computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library, and it never calls it.
 *
 * Conventions (all from "cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs"):
 *   - A [rows, cols] MXFP4 matrix is one byte buffer: the code plane
 *     (rows*cols/2 bytes) followed by the scale plane (rows*cols/32 bytes).
 *     (PEROP struct MxP: sbase = rows*cols/8 words; kernel mxfp4_mv.)
 *   - Group g of row r holds elements c = 32g .. 32g+31.  Its codes are four
 *     little-endian u32 words at word index (r*gpr + g)*4 + k, and nibble j of
 *     word k (bits 4j..4j+3) is element 32g + 8k + j.  (mxfp4_mv's group walk.)
 *   - Its E8M0 scale is byte (r*gpr + g) of the scale plane, i.e. byte i&3 of
 *     word sbase + (i>>2), little-endian.  (PEROP fn mx_scale.)
 *   - Arithmetic: every element decoded scalar by scalar to float; every product
 *     and every sum in double.  (The f64 reference of the page's device tests.)
 *
 * Every function is extern "C" so that Python's ctypes can call it.
 */
#ifndef MXFP4_ORACLE_H
#define MXFP4_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* E2M1 code (low 4 bits of n) -> float.  Magnitudes 0,0.5,1,1.5,2,3,4,6 for
 * n&7 = 0..7; bit 3 is the sign, so code 8 is -0.0.  (DECODE fn mx_e2m1.) */
float mxo_e2m1(unsigned n);

/* E8M0 scale byte -> float 2^(k-127); k = 0 gives the subnormal 2^-127 and
 * k = 255 gives NaN.  (DECODE fn mx_e8m0.) */
float mxo_e8m0(unsigned k);

/* Exact page length rows*cols*17/32 (codes + scales), 0 when cols % 32 != 0 or
 * a size is not positive.  (MoeBankCodec::lens; tests bank_codec_lengths.) */
size_t mxo_nbytes_exact(int rows, int cols);

/* Code nibble of element (r, c) and scale byte of group (r, g). */
unsigned mxo_code_at(const uint8_t* w, int rows, int cols, int r, int c);
unsigned mxo_scale_at(const uint8_t* w, int rows, int cols, int r, int g);

/* Decoded element w[r][c] = e2m1(code) * e8m0(scale), rounded to float (the
 * product is exact: the magnitude has at most two significant bits and the
 * scale is a power of two). */
float mxo_weight_at(const uint8_t* w, int rows, int cols, int r, int c);

/* Whole matrix -> out[r*cols + c]. */
void mxo_dequant(const uint8_t* w, int rows, int cols, float* out);

/* y[t*(r1-r0) + (r-r0)] = sum_c w[r][c] * x[t*cols + c] in double, and
 * l1[...] = sum_c |w[r][c] * x[t*cols + c]|, for tokens t < nb and rows
 * r0 <= r < r1.  nb = 1 is mxfp4_mv; nb > 1 is mxfp4_mm.  (PEROP kernels
 * mxfp4_mv / mxfp4_mm; host entry matmat: out[t*rows + r].) */
void mxo_matmat(const uint8_t* w, int rows, int cols, const float* x, int nb,
                int r0, int r1, double* y, double* l1);

/* Same as mxo_matmat over a list of (token, row) samples:
 * y[i], l1[i] for t = tok[i], r = row[i]. */
void mxo_matmat_samples(const uint8_t* w, int rows, int cols, const float* x,
                        const int32_t* tok, const int32_t* row, int n,
                        double* y, double* l1);

/* float -> bfloat16 -> float, round to nearest even; Inf and NaN pass
 * through.  (GLOBAL fn mxg_bf16.) */
float mxo_bf16_rne(float v);
void mxo_round_bf16(const float* in, float* out, size_t n);

/* SiLU in double: g / (1 + exp(-g)).  (dsv4_global_gate_up_mxfp4 tail.) */
double mxo_silu(double g);
/* d silu / d g, used only to propagate error bounds. */
double mxo_silu_grad(double g);

/* Routed-expert gate/up stage.  Expert e's gate and up matrices are
 * [inter, hidden] MXFP4 buffers at byte offset e * stride_bytes of their banks.
 * For pair p = t*top_k + j (token t, slot j) with expert e = ids[p] and every
 * row r < inter:
 *   g = gate_e[r] . x_t,  u = up_e[r] . x_t   (double),
 *   act = silu(g) * u                          (double),
 * written at [p*inter + r] together with the L1 bounds of g and u.
 * A pair whose expert id is out of range gets NaN everywhere.
 * (dsv4_global_gate_up_mxfp4 in its f32 form: no BF16 rounding, no limit,
 * no pre-weighting; cortiq-engine 0.8.77 moe_fast.rs gate_up_block.) */
void mxo_moe_gate_up(const uint8_t* gate_bank, const uint8_t* up_bank,
                     size_t stride_bytes, int n_experts, int hidden, int inter,
                     const float* x, int n_tokens, int top_k,
                     const int32_t* ids, double* g, double* u, double* l1g,
                     double* l1u, double* act);

/* Routed-expert down stage on a given float activation act[p*inter + c]:
 *   o_p[r] = down_e[r] . act_p                        (double, per pair),
 *   out[t*hidden + r] = sum_j route_w[t*top_k + j] * o_{t*top_k+j}[r],
 * summed over slots j in order, with
 *   l1_out[t*hidden + r] = sum_j |route_w| * sum_c |down_e[r][c] * act_p[c]|.
 * A pair whose expert id is out of range gets NaN in o_pairs / l1_pairs and
 * contributes nothing to out.  o_pairs / l1_pairs may be NULL.  (dsv4_global_down_mxfp4, generic f32 mode;
 * moe_fast.rs down_block; rlx-cpu gguf_matmul.rs grouped_moe_unpermute_out.) */
void mxo_moe_down(const uint8_t* down_bank, size_t stride_bytes, int n_experts,
                  int hidden, int inter, const float* act, int n_tokens,
                  int top_k, const int32_t* ids, const float* route_w,
                  double* o_pairs, double* l1_pairs, double* out,
                  double* l1_out);

/* The whole layer in double (the act is never rounded):
 *   out[t] = sum_j w_tj * down_e(silu(gate_e x_t) * (up_e x_t)).
 * bound_l1[t*hidden + r] = sum_j |w_tj| sum_c |down_e[r][c] a_c| and
 * bound_prop[...] = sum_j |w_tj| sum_c |down_e[r][c]| *
 *                   (|silu'(g_c)| L1g_c |u_c| + |silu(g_c)| L1u_c),
 * the two terms an implementation with relative-to-L1 error eps in each dot
 * product must stay within (times eps). */
void mxo_moe_forward(const uint8_t* gate_bank, const uint8_t* up_bank,
                     const uint8_t* down_bank, size_t gu_stride_bytes,
                     size_t down_stride_bytes, int n_experts, int hidden,
                     int inter, const float* x, int n_tokens, int top_k,
                     const int32_t* ids, const float* route_w, double* out,
                     double* bound_l1, double* bound_prop);

/* The layer in the general form of the page's global-bank kernels
 * (GLOBAL dsv4_global_gate_up_mxfp4 / dsv4_global_down_mxfp4 with their
 * flags; the expert slots and cold experts of its global-bank MoE test).
 *
 * Expert ids map to bank slots: slot = slot_of[e] when slot_of is given (a
 * negative entry marks a cold expert, one not resident in the bank; the page
 * writes u32::MAX), else slot = e.  A pair whose id is outside [0, n_experts)
 * or whose slot is outside [0, n_slots) is invalid; invalid and cold pairs
 * contribute nothing; the cold ones are listed, in increasing pair order, in
 * cold_pairs (n_cold of them).  Banks hold n_slots experts at the strides.
 *
 * Per valid pair p = t*top_k + j with slot s and route weight w:
 *   g = gate_s . x_t, u = up_s . x_t                   (double)
 *   bf16 mode: g = bf16(g), u = bf16(u)                 (mxg_bf16 of the float)
 *   limit > 0: u = clamp(u, -limit, limit), g = min(g, limit)
 *   a = silu(g) * u; bf16 mode: a = bf16(w * a)         (route weight folded in)
 *   o_p = down_s . a                                    (double)
 *   out[t] = sum_j w_j o_p (generic) or bf16(sum_j o_p) (bf16 mode), slots in order.
 * bound[t*hidden + r]: what an implementation may differ by when each FP32 dot
 * product carries up to eps = 1e-5 of its L1 norm, each bf16 rounding may land
 * one bf16 spacing away (the rounded values' neighbours), the limit clamps are
 * 1-Lipschitz (and remove the error of a value clamped with more than its error
 * to spare) and L = the largest |silu'| on [g - Eg, g + Eg]:
 *   Eg = eps L1g (+ sp(|g| + eps L1g)), Eu likewise
 *   Ea = |w'| ((|silu(g)| + L Eg) Eu + L |u| Eg + 2^-21 |silu(g) u|)
 *        (+ sp(|w silu(g) u| + that)), w' = w in bf16 mode, else 1
 *   Eo = sum_c |down| Ea_c + eps sum_c |down a|
 *   generic: bound = sum_j |w_j| Eo_j + eps sum_j |w_j o_j|
 *   bf16:    bound = sum_j Eo_j + eps sum_j |o_j| + sp(|out| + that)
 * where sp(v) is the bf16 spacing at |v| (2^(floor(log2|v|) - 7)). */
void mxo_moe_forward_ex(const uint8_t* gate_bank, const uint8_t* up_bank,
                        const uint8_t* down_bank, size_t gu_stride_bytes,
                        size_t down_stride_bytes, int n_slots, int hidden, int inter,
                        const float* x, int n_tokens, int top_k, const int32_t* ids,
                        const int32_t* slot_of, int n_experts, const float* route_w,
                        int bf16_mode, float limit, double* out, double* bound,
                        int32_t* cold_pairs, int* n_cold);

/* Routing plan by counting sort (rlx-cpu gguf_matmul.rs grouped_moe_sort_plan):
 * offsets[e] .. offsets[e+1] index the pairs of expert e in pair_of[], in
 * increasing pair order.  Returns the number of pairs with an invalid id (they
 * are left out of the plan). */
int mxo_moe_plan(const int32_t* ids, int n_pairs, int n_experts,
                 int32_t* offsets, int32_t* pair_of);

/* ---- The second codec: GGUF Q4_K ("rlx-cpu 0.2.17 src/gguf_matmul.rs",
 * q4k_dot_q8_block_avx2 and q4k_scale_min_x86, and the exact arm of
 * gguf_matmul_bt_m1_parallel).  A super-block holds 256 elements in 144 bytes:
 * d (IEEE binary16, bytes 0-1, little-endian), dmin (binary16, bytes 2-3), the
 * packed 6-bit scales and mins of its eight 32-element sub-blocks (bytes 4-15)
 * and 128 bytes of 4-bit codes (bytes 16-143).  Bytes 16 + 32 s + l (s < 4,
 * l < 32) hold element 64 s + l in the low nibble (sub-block 2 s) and element
 * 64 s + 32 + l in the high nibble (sub-block 2 s + 1).  A [rows, cols] matrix
 * (cols a multiple of 256) is rows x cols/256 blocks, row-major.  Element value
 * (the exact arm's on-the-fly f32 dequantisation): w = d*sc*q - dmin*m, the two
 * products exact in float and one float rounding of their difference. */

/* rows * cols/256 * 144, or 0 when cols % 256 != 0 or a size is not positive. */
size_t mxo_q4k_nbytes(int rows, int cols);

/* IEEE binary16 bits -> float (subnormals, infinities and NaN included). */
float mxo_f16(unsigned bits);

/* Scale and min of sub-block j (0..7) from the block's 12 packed bytes (the
 * page's q4k_scale_min_x86). */
void mxo_q4k_scale_min(const uint8_t* scales12, int j, unsigned* sc, unsigned* m);

/* Decoded element w[r][c] as a float, and the whole matrix -> out[r*cols + c]. */
float mxo_q4k_weight_at(const uint8_t* w, int rows, int cols, int r, int c);
void mxo_q4k_dequant(const uint8_t* w, int rows, int cols, float* out);

/* y[t*(r1-r0) + (r-r0)] = sum_c w[r][c] * x[t*cols + c] in double (w the decoded
 * floats), l1 = sum_c |w[r][c] x[t*cols + c]|, for tokens t < nb and rows
 * r0 <= r < r1. */
void mxo_q4k_matmat(const uint8_t* w, int rows, int cols, const float* x, int nb, int r0,
                    int r1, double* y, double* l1);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_ORACLE_H */
