// kernels.h -- host-side launchers of the libmxfp4.so kernels (internal).
// The C ABI in mxfp4_api.cu validates every argument before calling these.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>

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

// Routed experts.  The workspace layout is owned by moe.cu.
size_t moe_workspace_bytes(int n_experts, int n_tokens, int top_k, int hidden, int inter);
cudaError_t launch_moe_gate_up(const uint8_t* gate_bank, const uint8_t* up_bank, int n_experts,
                               int hidden, int inter, const float* x, int n_tokens, int top_k,
                               const int32_t* ids, float* act, void* ws, cudaStream_t s);
cudaError_t launch_moe_down(const uint8_t* down_bank, int n_experts, int hidden, int inter,
                            const float* act, int n_tokens, int top_k, const int32_t* ids,
                            const float* route_w, float* y, void* ws, cudaStream_t s);
cudaError_t moe_plan_errors(const void* ws, int* n_invalid, cudaStream_t s);

// Tensor-core expert passes (moe_tc.cu) over the plan arrays of moe.cu;
// cudaErrorNotSupported, with nothing launched, for shapes they cannot take.
cudaError_t launch_moe_tc_gate_up(const uint8_t* gate_bank, const uint8_t* up_bank, size_t stride,
                                  int n_experts, int inter, int hidden, int top_k, const float* x,
                                  const int32_t* hdr, const int32_t* offsets,
                                  const int32_t* touched, const int32_t* pair_of, float* act,
                                  cudaStream_t s);
cudaError_t launch_moe_tc_down(const uint8_t* down_bank, size_t stride, int n_experts, int hidden,
                               int inter, const float* act, const int32_t* hdr,
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
