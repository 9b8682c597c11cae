// kernels.h -- host-side launchers of the libmxfp4.so kernels (internal).
// The C ABI in mxfp4_api.cu validates every argument before calling these.
#pragma once

#include <cstddef>
#include <cstdint>
#include <functional>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mxk {

// Standalone decode of a whole matrix to float (bit-exact).
cudaError_t launch_dequant(const uint8_t* w, int rows, int cols, float* out, cudaStream_t s);

// FP32 small-batch product (nb = 1 is the matvec).  Per token bit-identical
// whatever nb is.
cudaError_t launch_matmat_fp32(const uint8_t* w, int rows, int cols, const float* X, int nb,
                               float* Y, cudaStream_t s);

// mma.sync product for up to 4 tokens per pass over the weights (split-f16
// activations, per-group FP32 scaling); cudaErrorNotSupported, with nothing
// launched, for shapes it cannot take.  Per token the same arithmetic for any nb.
cudaError_t launch_mv_tc(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                         cudaStream_t s);

// Programmatic dependent launch for the mv_tc kernels (process-wide switch).
void set_launch_overlap(bool on);
bool launch_overlap();

// mma.sync small-batch product (split-f16 activations, FP32 accumulate);
// cudaErrorNotSupported, with nothing launched, for shapes it cannot take.
cudaError_t launch_mm_tc(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                         cudaStream_t s);

// tcgen05 product with X rounded to bfloat16 (prefill.cu).
cudaError_t launch_mm_tcgen05(const uint8_t* w, int rows, int cols, const float* X, int nb,
                              float* Y, cudaStream_t s);

// Dense after dequant: W and X to bf16 in the workspace, then a TMA-fed tcgen05
// GEMM (prefill.cu).
size_t dense_ws_bytes(int rows, int cols, int nb);
cudaError_t launch_mm_dense(const uint8_t* w, int rows, int cols, const float* X, int nb,
                            float* Y, void* ws, cudaStream_t s);

// Tail of the gate/up pass ("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs",
// dsv4_global_gate_up_mxfp4): bf16 != 0 rounds gate and up to bfloat16, folds
// the pair's route weight into the act and rounds the act too (the V4.1
// mode); limit > 0 clamps up to [-limit, limit] and gate to at most limit.
struct MoeAct {
    const float* route_w;   // [pairs]; read in the bf16 mode only
    float limit;
    int bf16;
};

#ifdef __CUDACC__
__device__ __forceinline__ float moe_bf16(float v) {
    return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)))
                           << 16);
}

// act of pair `pair` from its gate and up dot products g and u (FP32).
__device__ __forceinline__ float moe_act(float g, float u, const MoeAct& epi, int pair) {
    if (epi.bf16) {
        g = moe_bf16(g);
        u = moe_bf16(u);
    }
    if (epi.limit > 0.0f) {
        const float lim = epi.limit;
        u = u < -lim ? -lim : (u > lim ? lim : u);
        g = g < lim ? g : lim;
    }
    float a = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
    if (epi.bf16) a = moe_bf16(__fmul_rn(__ldg(epi.route_w + pair), a));
    return a;
}
#endif

// An expert bank: its slots held in up to kMaxSegments separate buffers
// (segments) of seg_slots slots each, slot s at local index s % seg_slots of
// segment s / seg_slots, `stride` bytes per slot.  A bank in one buffer is
// one segment of all its slots.
constexpr int kMaxSegments = 16;
struct Bank {
    const uint8_t* seg[kMaxSegments];
    int n_seg;
    int seg_slots;
    size_t stride;
    __host__ __device__ const uint8_t* slot(int s) const {
        const int q = s / seg_slots;
        return seg[q] + static_cast<size_t>(s - q * seg_slots) * stride;
    }
};
inline Bank one_segment_bank(const uint8_t* base, int n_slots, size_t stride) {
    Bank b{};
    b.seg[0] = base;
    b.n_seg = 1;
    b.seg_slots = n_slots;
    b.stride = stride;
    return b;
}

// Routed experts.  The workspace layout is owned by moe.cu.  n_slots is the
// number of experts in the banks; ids map to slots through slot_of (nullable:
// slot = id; a negative entry marks a cold expert, whose pairs are skipped and
// listed), ids outside [0, n_ids) and slots outside [0, n_slots) are invalid.
size_t moe_workspace_bytes(int n_slots, int n_tokens, int top_k, int hidden, int inter);
cudaError_t launch_moe_gate_up(const Bank& gate, const Bank& up, int n_slots, int hidden,
                               int inter, const float* x, int n_tokens, int top_k,
                               const int32_t* ids, const int32_t* slot_of, int n_ids,
                               MoeAct epi, float* act, void* ws, cudaStream_t s);
// bf16 != 0: y = bf16(sum over the token's slots of o), the route weights being
// in the acts already; else y = sum of route_w * o.
cudaError_t launch_moe_down(const Bank& down, int n_slots, int hidden, int inter,
                            const float* act, int n_tokens, int top_k, const float* route_w,
                            int bf16, float* y, void* ws, cudaStream_t s);
cudaError_t moe_plan_errors(const void* ws, int* n_invalid, cudaStream_t s);
// The plan's cold pairs (increasing pair order): their count, and up to `cap`
// of them copied to host memory; synchronises the stream.
cudaError_t moe_cold_pairs(const void* ws, int n_slots, int n_pairs, int* n_cold,
                           int32_t* pairs_host, int cap, cudaStream_t s);

// Tensor-core expert passes (moe_tc.cu) over the plan arrays of moe.cu.  Each
// first splits its vectors (x by token for gate/up, act by pair for down) into
// the B-fragment blocks the pass copies per segment, in `frag`
// (moe_frag_bytes(n_vectors, cols) bytes, 16-byte aligned), then runs the pass.
// The gate/up pass calls `before` (the routing plan's launch) first.
// cudaErrorNotSupported, with nothing launched, for shapes they cannot take.
size_t moe_frag_bytes(int n_vec, int cols);
cudaError_t launch_moe_tc_gate_up(const Bank& gate, const Bank& up, int n_experts, int inter,
                                  int hidden, int top_k, const float* x, int n_tokens,
                                  uint8_t* frag, const std::function<cudaError_t()>& before,
                                  int32_t* hdr, const int32_t* offsets, const int32_t* touched,
                                  const int32_t* pair_of, MoeAct epi, float* act, cudaStream_t s);
cudaError_t launch_moe_tc_down(const Bank& down, int n_experts, int hidden, int inter,
                               const float* act, int n_pairs, uint8_t* frag, int32_t* hdr,
                               const int32_t* offsets, const int32_t* touched,
                               const int32_t* pair_of, float* o_pairs, cudaStream_t s);

// Device fault words (set when a bounded wait gives up); read and optionally clear.
cudaError_t read_fault_matvec(int* value, bool reset);
cudaError_t read_fault_mma(int* value, bool reset);
cudaError_t read_fault_prefill(int* value, bool reset);
cudaError_t read_fault_mvtc(int* value, bool reset);
cudaError_t read_fault_moetc(int* value, bool reset);

// Records a CUDA error for mxfp4_last_cuda_error() (this thread).
void record_cuda_error(int err);

// Unique id of the calling thread's current context (0 if the driver cannot
// say): an address cached under one context is not used under another.
unsigned long long current_context_id();

// A value computed once per device and then reused: kernel attributes (the
// dynamic shared-memory limit), SM counts and occupancies belong to a device,
// so a value obtained with one device current is never reused on another.
// `compute` runs with the device current, under the memo's lock.
class PerDevice {
  public:
    template <class F>
    int get(F&& compute) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMax) return compute();
        std::lock_guard<std::mutex> lock(mu_);
        if (!done_[dev]) {
            val_[dev] = compute();
            done_[dev] = true;
        }
        return val_[dev];
    }

  private:
    static constexpr int kMax = 64;
    std::mutex mu_;
    bool done_[kMax] = {};
    int val_[kMax] = {};
};

// Bytes of one [rows, cols] buffer, padded to 16.
inline size_t padded_nbytes(int rows, int cols) {
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) / 32 * 17;
    return (n + 15) / 16 * 16;
}

}  // namespace mxk
