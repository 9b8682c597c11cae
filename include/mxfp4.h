/*
 * mxfp4.h -- C ABI of libmxfp4.so: fused MXFP4 dequantisation with matrix-vector,
 * small-batch and large-batch matrix products and the two routed-expert (MoE)
 * passes, as hand-written CUDA kernels for sm_103a (GB300).
 *
 * Source of the operations: the docs.rs page "cortiq-engine 0.8.40
 * src/gpu_wgpu/mxfp4.rs" (const DECODE, const PEROP kernels mxfp4_mv /
 * mxfp4_mm, const GLOBAL kernels dsv4_global_gate_up_mxfp4 /
 * dsv4_global_down_mxfp4, host fn matmat), with the expert grouping of
 * "rlx-cpu 0.2.17 src/gguf_matmul.rs" (grouped_moe_sort_plan,
 * grouped_moe_unpermute_out).
 *
 * ---------------------------------------------------------------------------
 * Weight format (one [rows, cols] matrix, cols % 32 == 0, gpr = cols / 32):
 *   bytes [0, rows*cols/2)               code plane: for row r and group g, four
 *                                        little-endian u32 words at word index
 *                                        (r*gpr + g)*4 + k; nibble j (bits
 *                                        4j..4j+3) of word k is element
 *                                        c = 32g + 8k + j.  (PEROP mxfp4_mv.)
 *   bytes [rows*cols/2, +rows*gpr)       scale plane: E8M0 byte r*gpr + g.
 *                                        (PEROP fn mx_scale, struct MxP sbase.)
 *   then padding up to mxfp4_nbytes(rows, cols) (never read as data).
 * Decode: E2M1 code n -> +-{0, .5, 1, 1.5, 2, 3, 4, 6}[n & 7], bit 3 = sign
 * (code 8 = -0.0); E8M0 byte k -> 2^(k-127), k = 0 -> 2^-127 (subnormal, kept),
 * k = 255 -> NaN; element = code value * scale.  (DECODE mx_e2m1 / mx_e8m0.)
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  Except the
 *     host-buffer wrapper mxfp4_matmat_host, the library allocates nothing and
 *     copies nothing between host and device.
 *   - Weight pointers must be 16-byte aligned and hold mxfp4_nbytes(rows, cols)
 *     bytes; float pointers must be 16-byte aligned.
 *   - Work is enqueued on `stream` (0 = the legacy default stream); calls are
 *     asynchronous (no device synchronisation) unless stated otherwise.
 *   - Return value: an MXFP4_STATUS_* code.  On any non-zero code nothing was
 *     enqueued, except MXFP4_STATUS_LAUNCH_FAILED, which reports the CUDA error
 *     left by a launch (mxfp4_last_cuda_error() gives the cudaError_t).  There
 *     is no CPU fallback.  (The page's matmat returns false for every refusal.)
 *   - Results are deterministic: the same inputs give the same bits, run after
 *     run (no floating-point atomics).
 * ---------------------------------------------------------------------------
 */
#ifndef MXFP4_H
#define MXFP4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MXFP4_STATUS_OK = 0,
    MXFP4_STATUS_INVALID_ARGUMENT = 1, /* shape, count or id out of range    */
    MXFP4_STATUS_BAD_POINTER = 2,      /* NULL or misaligned pointer         */
    MXFP4_STATUS_LAUNCH_FAILED = 3,    /* CUDA reported an error             */
    MXFP4_STATUS_WORKSPACE_TOO_SMALL = 4
};

/* Human-readable name of a status code (static storage, never NULL). */
const char* mxfp4_status_string(int status);

/* cudaError_t recorded by the last MXFP4_STATUS_LAUNCH_FAILED on this thread. */
int mxfp4_last_cuda_error(void);

/* Reads the library's device fault word into *faults (0 = none) and clears it
 * if `reset` is non-zero.  A kernel that waits on its own asynchronous copies
 * gives up after a bounded number of polls instead of hanging the GPU; it then
 * sets this word and returns early, leaving its outputs incomplete.
 * Synchronises the current device. */
int mxfp4_device_faults(int* faults, int reset);

/* Launch overlap for mxfp4_mv and mxfp4_mm (up to MXFP4_MM_SMALL_MAX tokens),
 * off by default, process-wide.  The pages have no counterpart: this is a
 * property of a stream of launches on one GPU.  When enabled (enable != 0)
 * these calls use programmatic dependent launch: the kernel may start while
 * the previous kernel in the stream is still running and already stream the
 * weight buffer `w` (code and scale planes); it reads X and writes Y only
 * after that kernel has completed.  Enable it only if no work still running
 * in the stream writes the weight buffers (weights that stay fixed during
 * decoding).  Results are bit-identical either way.  Returns MXFP4_STATUS_OK. */
int mxfp4_set_launch_overlap(int enable);

/* Library version as major*10000 + minor*100 + patch. */
int mxfp4_version(void);

/* Bytes a [rows, cols] weight buffer must hold: rows*cols*17/32 (code plane +
 * scale plane, the page's MoeBankCodec::lens / tests bank_codec_lengths length)
 * rounded up to a multiple of 16 so that every row can be read with 16-byte
 * loads.  0 if rows < 1, cols < 32 or cols % 32 != 0. */
size_t mxfp4_nbytes(int rows, int cols);

/* Standalone decode: out[r*cols + c] = element (r, c) as float, bit-exact
 * (E2M1 value times E8M0 scale is exact in float; NaN for k = 255).
 * out: [rows*cols] floats.  (DECODE; the page's tests decode the whole matrix
 * with cortiq_core::mxfp4::dequant as their reference.) */
int mxfp4_dequant(const void* w, int rows, int cols, float* out, cudaStream_t stream);

/* Matrix-vector product, one token: y[r] = sum_c W[r][c] * x[c].  Each group's
 * 32 decoded weights (exact in f16) are dotted with x on the tensor cores
 * (mma.sync; x split into f16 halves hi + lo of x * 2^p, so every product is
 * exact), the group sum is scaled by its E8M0 factor and 2^-p in FP32 and
 * added to one of the row's four FP32 sums (groups by index mod 4), which are
 * added in order at the end.  x: [cols] floats, y: [rows] floats.  Error
 * bound: |y - exact| <= 1e-5 * sum_c |W[r][c] x[c]| + 2^-39 * max_c |x[c]| *
 * sum_c |W[r][c]| (a NaN scale makes the row NaN).  The second term comes from
 * the f16 subnormal spacing under hi and lo: elements below about 2^-38 of the
 * largest |x| are lost, which matters only for an x spanning more than ~2^30
 * whose large elements meet small weights (mxfp4_mm_fp32 has no such term).
 * Deterministic: the order of every sum depends on the shape only.  (PEROP
 * mxfp4_mv.) */
int mxfp4_mv(const void* w, int rows, int cols, const float* x, float* y,
             cudaStream_t stream);

/* Batched product: Y[t*rows + r] = sum_c W[r][c] * X[t*cols + c], t < nb.
 * X: [nb, cols] row-major floats, Y: [nb, rows] (the page's matmat output
 * layout).  Dispatch on nb:
 *   nb <= MXFP4_MM_SMALL_MAX: the small-batch path -- each weight group is
 *     decoded once and applied to up to 8 tokens per pass over the weights
 *     (PEROP mxfp4_mm: one decode shared by up to 8 tokens; shapes whose
 *     eight-token fragments do not fit in shared memory take passes of 4,
 *     with the same results); the arithmetic of
 *     mxfp4_mv, so per token the result equals mxfp4_mv on that token bit
 *     for bit, whatever the rest of the batch (the page's device test:
 *     "the batch equal to the matvec per token bit for bit").
 *   nb >  MXFP4_MM_SMALL_MAX: the tensor-core path of mxfp4_mm_bf16 (below):
 *     X is rounded to bfloat16 first.  The weights and X are converted to
 *     bfloat16 once ("rlx-cpu 0.2.17 src/gguf_matmul.rs": dense after
 *     dequant, as mxfp4_mm_bf16_ws) into a device workspace the library keeps
 *     per (device, stream): allocated on the stream (stream-ordered) by the
 *     first call that needs it, grown by later ones, never while the stream is
 *     being captured into a graph, and kept while the context lives (one
 *     made before a device reset is dropped, not reused)
 *     (mxfp4_mm_bf16_workspace_bytes(rows, cols, nb) bytes).  Without one (a
 *     capture before any eager call on that stream, or an allocation failure)
 *     the conversion runs inside the GEMM (mxfp4_mm_bf16); the results are the
 *     same bit for bit either way. */
#define MXFP4_MM_SMALL_MAX 64
int mxfp4_mm(const void* w, int rows, int cols, const float* X, int nb, float* Y,
             cudaStream_t stream);

/* The same product in plain FP32 on the CUDA cores, any nb >= 1: per group the
 * decoded values dotted with x in FP32 (two FMA chains), scaled, the row's
 * group partials reduced across a warp; chunks of 8 tokens share each decode.
 * Same error bound as mxfp4_mv.  Per token the result is bit-identical to this
 * function with nb = 1 on that token (same group walk, same reduction tree). */
int mxfp4_mm_fp32(const void* w, int rows, int cols, const float* X, int nb, float* Y,
                  cudaStream_t stream);

/* Large-batch (prefill) product on the tensor cores: W decoded exactly to
 * bfloat16, X rounded to nearest-even bfloat16 (GLOBAL fn mxg_bf16), products
 * accumulated in FP32.  Same shapes and layouts as mxfp4_mm, any nb >= 1.
 * Error bound against the product of W and bf16(X): 2e-2 * sum_c |W bf16(X)|
 * (tighter in practice).  The decoded weight is exact in bfloat16 for every
 * scale byte (scale bytes 0 and 1 give bfloat16 subnormals, which the tensor
 * cores keep). */
int mxfp4_mm_bf16(const void* w, int rows, int cols, const float* X, int nb, float* Y,
                  cudaStream_t stream);

/* Bytes of the workspace mxfp4_mm_bf16_ws needs: a bfloat16 copy of W
 * (rows*cols*2, rounded up to 256) followed by one of X (nb*cols*2).
 * 0 for an invalid shape or nb < 1. */
size_t mxfp4_mm_bf16_workspace_bytes(int rows, int cols, int nb);

/* The same product as mxfp4_mm_bf16 computed densely after dequantisation
 * ("rlx-cpu 0.2.17 src/gguf_matmul.rs" gguf_matmul_bt_cached: dequantise the
 * weights once, then a dense GEMM): W is decoded exactly to bfloat16 and X
 * rounded to nearest-even bfloat16 into `workspace` (device, owned by the
 * caller, 16-byte aligned, >= mxfp4_mm_bf16_workspace_bytes bytes, rewritten
 * by every call), then a tensor-core GEMM accumulates in FP32.  Same result
 * contract and error bound as mxfp4_mm_bf16.  MXFP4_STATUS_WORKSPACE_TOO_SMALL
 * (nothing launched) if workspace_bytes is short. */
int mxfp4_mm_bf16_ws(const void* w, int rows, int cols, const float* X, int nb, float* Y,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* p2-style host entry (the page's fn matmat): X and Y are HOST buffers, the
 * weight stays resident on the device.  Copies X to x_dev, runs mxfp4_mm
 * (mxfp4_mv when nb == 1), copies the result back to Y and synchronises the
 * stream.  x_dev: >= nb*cols floats, y_dev: >= nb*rows floats (device, owned by
 * the caller).  Pinned host memory gives asynchronous copies. */
int mxfp4_matmat_host(const void* w, int rows, int cols, const float* X_host, int nb,
                      float* Y_host, float* x_dev, float* y_dev, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Routed experts.  Banks: expert e's gate and up matrices ([inter, hidden]) are
 * at byte offset e * mxfp4_nbytes(inter, hidden) of gate_bank / up_bank, its
 * down matrix ([hidden, inter]) at e * mxfp4_nbytes(hidden, inter) of
 * down_bank.  Pairs: p = t*top_k + j for token t < n_tokens and slot
 * j < top_k; expert_ids[p] and route_w[p] are the routing choice and weight
 * (the page's gg_sel / gd_wt in their [batch, slots] layout).
 * -------------------------------------------------------------------------- */

/* Workspace bytes the two passes need: the routing plan, the per-pair down
 * outputs, and the tensor-core passes' split copies of the vectors (each token's
 * x and each pair's act row as f16 hi/lo fragments with one power of two per
 * vector, made once per pass and read by every segment of the vector's expert).
 * The same workspace serves one layer at a time (gate/up, then down). */
size_t mxfp4_moe_workspace_bytes(int n_experts, int n_tokens, int top_k, int hidden,
                                 int inter);

/* Gate/up pass: builds the routing plan (counting sort of the pairs by expert,
 * rlx-cpu grouped_moe_sort_plan) into `workspace`, then for every touched
 * expert reads its gate and up matrices ONCE for all of its pairs and writes
 *   act[p*inter + r] = silu(g) * u,  g = gate_e[r] . x_t,  u = up_e[r] . x_t,
 * silu(g) = g / (1 + exp(-g)), FP32 (dsv4_global_gate_up_mxfp4 without BF16
 * rounding, limit or pre-weighting).  x: [n_tokens, hidden]; act:
 * [n_tokens*top_k, inter].  Pairs with an out-of-range expert id are skipped
 * (their act rows are left untouched) and counted in the plan's error word,
 * readable with mxfp4_moe_plan_errors.  The plan stays valid for
 * mxfp4_moe_down only while expert_ids and workspace are unchanged. */
int mxfp4_moe_gate_up(const void* gate_bank, const void* up_bank, int n_experts,
                      int hidden, int inter, const float* x, int n_tokens, int top_k,
                      const int32_t* expert_ids, float* act, void* workspace,
                      size_t ws_bytes, cudaStream_t stream);

/* Down pass + weighted combine, reusing the plan left in `workspace` by
 * mxfp4_moe_gate_up: per touched expert, its down matrix is read once for all
 * its pairs, o_p[r] = down_e[r] . act_p (FP32, kept in the workspace), then
 *   y[t*hidden + r] = sum_j route_w[t*top_k + j] * o_{t*top_k + j}[r]
 * summed over j in slot order (dsv4_global_down_mxfp4's generic f32 mode, which
 * fuses the combine; rlx-cpu grouped_moe_unpermute_out).  A pair with an
 * invalid id contributes nothing.  y: [n_tokens, hidden].  Both passes' dot
 * products carry mxfp4_mv's error bound, with x the token's x (gate/up) or the
 * pair's act row (down). */
int mxfp4_moe_down(const void* down_bank, int n_experts, int hidden, int inter,
                   const float* act, int n_tokens, int top_k, const int32_t* expert_ids,
                   const float* route_w, float* y, void* workspace, size_t ws_bytes,
                   cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * The general form of the two passes: the flags of the page's global-bank
 * kernels (GLOBAL dsv4_global_gate_up_mxfp4 / dsv4_global_down_mxfp4) and the
 * expert slots of its global-bank MoE (the expert -> slot remap, with cold
 * experts left out of the bank).
 *
 * Banks hold n_slots experts (slot s at s * mxfp4_nbytes(...) as above).  Expert
 * ids lie in [0, n_experts); slot_of[id] (device, int32[n_experts], nullable:
 * then slot = id and n_experts must equal n_slots) gives the id's bank slot,
 * a negative entry marking a COLD expert (not resident; the page's u32::MAX
 * remap).  Pairs routed to a cold expert are skipped by both passes and
 * listed in the workspace (mxfp4_moe_cold_pairs) so that the caller can run
 * them elsewhere; pairs with an id outside [0, n_experts) or a slot at or past
 * n_slots are skipped and counted (mxfp4_moe_plan_errors).  The workspace size
 * is mxfp4_moe_workspace_bytes(n_slots, n_tokens, top_k, hidden, inter).
 *
 * mode MXFP4_MOE_MODE_F32: act = silu(g) * u and y[t] = sum_j w_tj o_tj in
 *   FP32, as mxfp4_moe_gate_up / mxfp4_moe_down.
 * mode MXFP4_MOE_MODE_V41 (the DeepSeek-V4.1 path: the kernels' flag _p0):
 *   g and u are rounded to bfloat16 (round to nearest even, GLOBAL fn
 *   mxg_bf16), act = bf16(w_tj * silu(g) * u) -- the route weight folded into
 *   the act -- and y[t] = bf16(sum_j o_tj) with o = down . act.
 * swiglu_limit > 0 (either mode): u is clamped to [-limit, limit] and g to at
 *   most limit before SiLU; 0 turns the clamp off; NaN is refused.
 * A shared expert is one more slot of every token: give it a bank slot, an id
 * and route weight 1 (the page's frame routes its shared slot so).
 * Error bound: see the oracle's mxo_moe_forward_ex (FP32 dot products within
 * 1e-5 of their L1 norms, each bf16 rounding at most one bf16 step away). */
#define MXFP4_MOE_MODE_F32 0
#define MXFP4_MOE_MODE_V41 1
int mxfp4_moe_gate_up_ex(const void* gate_bank, const void* up_bank, int n_slots, int hidden,
                         int inter, const float* x, int n_tokens, int top_k,
                         const int32_t* expert_ids, const int32_t* slot_of, int n_experts,
                         const float* route_w, int mode, float swiglu_limit, float* act,
                         void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Down pass + combine for mxfp4_moe_gate_up_ex's plan (same workspace, same
 * routing): route_w is read in MXFP4_MOE_MODE_F32 only (may be NULL in V41). */
int mxfp4_moe_down_ex(const void* down_bank, int n_slots, int hidden, int inter, const float* act,
                      int n_tokens, int top_k, const float* route_w, int mode, float* y,
                      void* workspace, size_t ws_bytes, cudaStream_t stream);

/* The same two passes on a SEGMENTED bank: the bank's n_segments *
 * segment_slots slots live in n_segments separate buffers (segments, at most
 * 16), slot s at local index s % segment_slots of segment s / segment_slots,
 * each segment holding its slots back to back at the same stride as a
 * one-buffer bank (the page's global bank: binding arrays of 8 or 16 segment
 * buffers, gg_sel's flat slot split into segment and local index).
 * gate_segments / up_segments / down_segments are HOST arrays of n_segments
 * DEVICE pointers (16-byte aligned), read during the call.  Every other
 * argument, the workspace and the results are those of the _ex passes with
 * n_slots = n_segments * segment_slots. */
int mxfp4_moe_gate_up_seg(const void* const* gate_segments, const void* const* up_segments,
                          int n_segments, int segment_slots, int hidden, int inter, const float* x,
                          int n_tokens, int top_k, const int32_t* expert_ids,
                          const int32_t* slot_of, int n_experts, const float* route_w, int mode,
                          float swiglu_limit, float* act, void* workspace, size_t ws_bytes,
                          cudaStream_t stream);
int mxfp4_moe_down_seg(const void* const* down_segments, int n_segments, int segment_slots,
                       int hidden, int inter, const float* act, int n_tokens, int top_k,
                       const float* route_w, int mode, float* y, void* workspace, size_t ws_bytes,
                       cudaStream_t stream);

/* The plan's cold pairs (p = t*top_k + j, increasing): their count in *n_cold
 * and the first min(count, capacity) indices copied to pairs_host (host).
 * Synchronises the stream. */
int mxfp4_moe_cold_pairs(const void* workspace, size_t ws_bytes, int n_slots, int n_tokens,
                         int top_k, int* n_cold, int32_t* pairs_host, int capacity,
                         cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * The routed-expert layer without a workspace.  The source pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory when they run the layer -- for example a serving process whose
 * device memory all belongs to its own pool allocator, or a loop that must not
 * call cudaMalloc once running because an allocation can block the device and
 * stall its other streams.
 *
 * It runs mxfp4_moe_gate_up and then mxfp4_moe_down (same kernels, same
 * results) with the routing plan, the activation act and the per-pair down
 * outputs kept in one file-scope device array of MXFP4_MOE_NOALLOC_SCRATCH_BYTES
 * bytes, which every GPU that loads the library holds until the process exits.
 * It allocates nothing.  The caller passes inputs and the output
 * y [n_tokens, hidden] only.
 *   - Size limit: mxfp4_moe_workspace_bytes(n_experts, n_tokens, top_k, hidden,
 *     inter) rounded up to 256, plus n_tokens*top_k*inter*4 bytes for act, must
 *     not exceed MXFP4_MOE_NOALLOC_SCRATCH_BYTES; larger problems are refused
 *     with MXFP4_STATUS_WORKSPACE_TOO_SMALL (use the workspace entry points).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is cached per device together
 *     with the id of the context it belongs to; after the device's context is
 *     destroyed and created again (cudaDeviceReset), the next call looks it up
 *     again, so make that call outside stream capture as well.
 *   - Every call uses the same array and the array keeps the previous call's
 *     contents; each call rewrites all of the scratch it reads, so nothing has
 *     to start at zero.  Calls that overlap on the GPU (other streams, other
 *     host threads) race on the array: serialise them.
 *   - Out-of-range expert ids are skipped as in mxfp4_moe_gate_up /
 *     mxfp4_moe_down; their count is not reported by this entry point. */
#define MXFP4_MOE_NOALLOC_SCRATCH_BYTES (16u << 20)
int mxfp4_moe_layer_noalloc(const void* gate_bank, const void* up_bank, const void* down_bank,
                            int n_experts, int hidden, int inter, const float* x, int n_tokens,
                            int top_k, const int32_t* expert_ids, const float* route_w, float* y,
                            cudaStream_t stream);

/* Copies the plan's count of out-of-range expert ids to *n_invalid (host) and
 * synchronises the stream.  For tests and debugging; the passes themselves
 * never synchronise. */
int mxfp4_moe_plan_errors(const void* workspace, size_t ws_bytes, int* n_invalid,
                          cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_H */
