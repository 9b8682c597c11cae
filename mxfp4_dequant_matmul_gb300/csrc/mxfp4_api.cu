// mxfp4_api.cu -- the extern "C" boundary of libmxfp4.so (declared in
// include/mxfp4.h).  Every entry point validates its arguments on the host,
// refuses with a status code (launching nothing) when they are wrong, and
// otherwise enqueues kernels on the caller's stream.  The refusal rules follow
// "cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs" host fn matmat (b == 0,
// rows == 0, cols % 32 != 0 or short buffers are refused), without its CPU
// fallback.
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/mxfp4.h"
#include "kernels.h"

namespace {

thread_local int g_last_cuda_error = 0;

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MXFP4_STATUS_OK;
    g_last_cuda_error = static_cast<int>(e);
    return MXFP4_STATUS_LAUNCH_FAILED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// rows >= 1, cols >= 32 and a multiple of 32, rows*cols small enough that every
// byte offset fits comfortably in 63 bits and every row index in an int.
int check_shape(int rows, int cols) {
    if (rows < 1 || cols < 32 || cols % 32 != 0) return MXFP4_STATUS_INVALID_ARGUMENT;
    if (static_cast<long long>(rows) * cols > (1LL << 46)) return MXFP4_STATUS_INVALID_ARGUMENT;
    return MXFP4_STATUS_OK;
}

int check_ptr(const void* p) {
    return (p == nullptr || !aligned16(p)) ? MXFP4_STATUS_BAD_POINTER : MXFP4_STATUS_OK;
}

#define MXFP4_TRY(expr)                            \
    do {                                           \
        const int _st = (expr);                    \
        if (_st != MXFP4_STATUS_OK) return _st;    \
    } while (0)

int check_product(const void* w, int rows, int cols, const float* X, int nb, const float* Y) {
    MXFP4_TRY(check_shape(rows, cols));
    if (nb < 1 || nb > (1 << 24)) return MXFP4_STATUS_INVALID_ARGUMENT;
    MXFP4_TRY(check_ptr(w));
    MXFP4_TRY(check_ptr(X));
    MXFP4_TRY(check_ptr(Y));
    return MXFP4_STATUS_OK;
}

const uint8_t* u8(const void* p) { return static_cast<const uint8_t*>(p); }

// The workspace of mxfp4_mm's large batches (weights and activations in bf16,
// dense after dequant), one per (device, stream): used only in that stream's
// order, so concurrent streams never share one.  Grown by stream-ordered
// allocation (the old one freed after the work already queued on the stream);
// never allocated while the stream is being captured into a graph; kept for the
// life of the context (an entry made under another context, before a device
// reset, is dropped: its memory went with that context).  nullptr when none can
// be had: the caller then takes the path that needs no workspace (the same
// results bit for bit).
void* stream_workspace(cudaStream_t s, size_t need) {
    struct Entry {
        void* ptr;
        size_t bytes;
        unsigned long long ctx;
    };
    static std::mutex mu;
    static std::map<std::pair<int, cudaStream_t>, Entry> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    const unsigned long long ctx = mxk::current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    Entry& e = cache[{dev, s}];
    if (e.ptr != nullptr && (ctx == 0 || e.ctx != ctx)) e = Entry{nullptr, 0, 0};
    if (e.ptr != nullptr && e.bytes >= need) return e.ptr;
    if (ctx == 0) return nullptr;
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess || st != cudaStreamCaptureStatusNone) {
        (void)cudaGetLastError();
        return nullptr;
    }
    void* p = nullptr;
    if (cudaMallocAsync(&p, need, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (e.ptr != nullptr) (void)cudaFreeAsync(e.ptr, s);
    e = Entry{p, need, ctx};
    return p;
}

}  // namespace

void mxk::record_cuda_error(int err) { g_last_cuda_error = err; }

extern "C" {

const char* mxfp4_status_string(int status) {
    switch (status) {
        case MXFP4_STATUS_OK: return "ok";
        case MXFP4_STATUS_INVALID_ARGUMENT: return "invalid argument";
        case MXFP4_STATUS_BAD_POINTER: return "null or misaligned pointer";
        case MXFP4_STATUS_LAUNCH_FAILED: return "CUDA launch failed";
        case MXFP4_STATUS_WORKSPACE_TOO_SMALL: return "workspace too small";
        default: return "unknown status";
    }
}

int mxfp4_last_cuda_error(void) { return g_last_cuda_error; }

int mxfp4_version(void) { return 100; }

int mxfp4_set_launch_overlap(int enable) {
    mxk::set_launch_overlap(enable != 0);
    return MXFP4_STATUS_OK;
}

int mxfp4_device_faults(int* faults, int reset) {
    if (faults == nullptr) return MXFP4_STATUS_BAD_POINTER;
    int a = 0, b = 0, c = 0, f = 0, h = 0;
    cudaError_t e = mxk::read_fault_matvec(&a, reset != 0);
    if (e == cudaSuccess) e = mxk::read_fault_mma(&b, reset != 0);
    if (e == cudaSuccess) e = mxk::read_fault_prefill(&c, reset != 0);
    if (e == cudaSuccess) e = mxk::read_fault_mvtc(&f, reset != 0);
    if (e == cudaSuccess) e = mxk::read_fault_moetc(&h, reset != 0);
    if (e != cudaSuccess) return from_cuda(e);
    *faults = a | (b << 1) | (c << 2) | (f << 3) | (h << 4);
    return MXFP4_STATUS_OK;
}

size_t mxfp4_nbytes(int rows, int cols) {
    if (check_shape(rows, cols) != MXFP4_STATUS_OK) return 0;
    return mxk::padded_nbytes(rows, cols);
}

int mxfp4_dequant(const void* w, int rows, int cols, float* out, cudaStream_t stream) {
    MXFP4_TRY(check_shape(rows, cols));
    MXFP4_TRY(check_ptr(w));
    MXFP4_TRY(check_ptr(out));
    return from_cuda(mxk::launch_dequant(u8(w), rows, cols, out, stream));
}

int mxfp4_mv(const void* w, int rows, int cols, const float* x, float* y, cudaStream_t stream) {
    MXFP4_TRY(check_product(w, rows, cols, x, 1, y));
    // the same kernel order as mxfp4_mm, so that a batch equals its matvecs
    cudaError_t e = mxk::launch_mv_tc(u8(w), rows, cols, x, 1, y, stream);
    if (e != cudaErrorNotSupported) return from_cuda(e);
    (void)cudaGetLastError();
    e = mxk::launch_mm_tc(u8(w), rows, cols, x, 1, y, stream);
    if (e != cudaErrorNotSupported) return from_cuda(e);
    (void)cudaGetLastError();
    return from_cuda(mxk::launch_matmat_fp32(u8(w), rows, cols, x, 1, y, stream));
}

int mxfp4_mm_fp32(const void* w, int rows, int cols, const float* X, int nb, float* Y,
                  cudaStream_t stream) {
    MXFP4_TRY(check_product(w, rows, cols, X, nb, Y));
    return from_cuda(mxk::launch_matmat_fp32(u8(w), rows, cols, X, nb, Y, stream));
}

int mxfp4_mm_bf16(const void* w, int rows, int cols, const float* X, int nb, float* Y,
                  cudaStream_t stream) {
    MXFP4_TRY(check_product(w, rows, cols, X, nb, Y));
    return from_cuda(mxk::launch_mm_tcgen05(u8(w), rows, cols, X, nb, Y, stream));
}

size_t mxfp4_mm_bf16_workspace_bytes(int rows, int cols, int nb) {
    if (check_shape(rows, cols) != MXFP4_STATUS_OK || nb < 1) return 0;
    return mxk::dense_ws_bytes(rows, cols, nb);
}

int mxfp4_mm_bf16_ws(const void* w, int rows, int cols, const float* X, int nb, float* Y,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    MXFP4_TRY(check_product(w, rows, cols, X, nb, Y));
    MXFP4_TRY(check_ptr(workspace));
    if (workspace_bytes < mxk::dense_ws_bytes(rows, cols, nb))
        return MXFP4_STATUS_WORKSPACE_TOO_SMALL;
    return from_cuda(mxk::launch_mm_dense(u8(w), rows, cols, X, nb, Y, workspace, stream));
}

int mxfp4_mm(const void* w, int rows, int cols, const float* X, int nb, float* Y,
             cudaStream_t stream) {
    MXFP4_TRY(check_product(w, rows, cols, X, nb, Y));
    if (nb <= MXFP4_MM_SMALL_MAX) {
        cudaError_t e = mxk::launch_mv_tc(u8(w), rows, cols, X, nb, Y, stream);
        if (e != cudaErrorNotSupported) return from_cuda(e);
        (void)cudaGetLastError();
        e = mxk::launch_mm_tc(u8(w), rows, cols, X, nb, Y, stream);
        if (e != cudaErrorNotSupported) return from_cuda(e);
        (void)cudaGetLastError();
        return from_cuda(mxk::launch_matmat_fp32(u8(w), rows, cols, X, nb, Y, stream));
    }
    // dense after dequant through the stream's workspace when it can be had,
    // else the conversion inside the GEMM (bit-identical results)
    if (void* ws = stream_workspace(stream, mxk::dense_ws_bytes(rows, cols, nb))) {
        const cudaError_t e = mxk::launch_mm_dense(u8(w), rows, cols, X, nb, Y, ws, stream);
        if (e != cudaErrorNotSupported) return from_cuda(e);
        (void)cudaGetLastError();
    }
    return from_cuda(mxk::launch_mm_tcgen05(u8(w), rows, cols, X, nb, Y, stream));
}

int mxfp4_matmat_host(const void* w, int rows, int cols, const float* X_host, int nb,
                      float* Y_host, float* x_dev, float* y_dev, cudaStream_t stream) {
    MXFP4_TRY(check_product(w, rows, cols, x_dev, nb, y_dev));
    if (X_host == nullptr || Y_host == nullptr) return MXFP4_STATUS_BAD_POINTER;
    const size_t xb = static_cast<size_t>(nb) * cols * sizeof(float);
    const size_t yb = static_cast<size_t>(nb) * rows * sizeof(float);
    cudaError_t e = cudaMemcpyAsync(x_dev, X_host, xb, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return from_cuda(e);
    const int st = nb == 1 ? mxfp4_mv(w, rows, cols, x_dev, y_dev, stream)
                           : mxfp4_mm(w, rows, cols, x_dev, nb, y_dev, stream);
    if (st != MXFP4_STATUS_OK) return st;
    e = cudaMemcpyAsync(Y_host, y_dev, yb, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(cudaStreamSynchronize(stream));
}

size_t mxfp4_moe_workspace_bytes(int n_experts, int n_tokens, int top_k, int hidden, int inter) {
    if (n_experts < 1 || n_tokens < 1 || top_k < 1 || hidden < 32 || inter < 32) return 0;
    return mxk::moe_workspace_bytes(n_experts, n_tokens, top_k, hidden, inter);
}

namespace {

int check_moe(int n_experts, int hidden, int inter, int n_tokens, int top_k, const void* ws,
              size_t ws_bytes) {
    if (n_experts < 1 || n_experts > (1 << 20) || n_tokens < 1 || top_k < 1 ||
        static_cast<long long>(n_tokens) * top_k > (1 << 22))
        return MXFP4_STATUS_INVALID_ARGUMENT;
    MXFP4_TRY(check_shape(inter, hidden));   // gate / up: [inter, hidden]
    MXFP4_TRY(check_shape(hidden, inter));   // down: [hidden, inter]
    if (static_cast<long long>(n_experts) * inter * hidden > (1LL << 46))
        return MXFP4_STATUS_INVALID_ARGUMENT;
    MXFP4_TRY(check_ptr(ws));
    if (ws_bytes < mxk::moe_workspace_bytes(n_experts, n_tokens, top_k, hidden, inter))
        return MXFP4_STATUS_WORKSPACE_TOO_SMALL;
    return MXFP4_STATUS_OK;
}

}  // namespace

int mxfp4_moe_gate_up(const void* gate_bank, const void* up_bank, int n_experts, int hidden,
                      int inter, const float* x, int n_tokens, int top_k,
                      const int32_t* expert_ids, float* act, void* workspace, size_t ws_bytes,
                      cudaStream_t stream) {
    MXFP4_TRY(check_moe(n_experts, hidden, inter, n_tokens, top_k, workspace, ws_bytes));
    MXFP4_TRY(check_ptr(gate_bank));
    MXFP4_TRY(check_ptr(up_bank));
    MXFP4_TRY(check_ptr(x));
    MXFP4_TRY(check_ptr(act));
    if (expert_ids == nullptr || (reinterpret_cast<uintptr_t>(expert_ids) & 3u))
        return MXFP4_STATUS_BAD_POINTER;
    const size_t stride = mxk::padded_nbytes(inter, hidden);
    return from_cuda(mxk::launch_moe_gate_up(
        mxk::one_segment_bank(u8(gate_bank), n_experts, stride),
        mxk::one_segment_bank(u8(up_bank), n_experts, stride), n_experts, hidden, inter, x,
        n_tokens, top_k, expert_ids, nullptr, n_experts, mxk::MoeAct{nullptr, 0.0f, 0}, act,
        workspace, stream));
}

int mxfp4_moe_down(const void* down_bank, int n_experts, int hidden, int inter, const float* act,
                   int n_tokens, int top_k, const int32_t* expert_ids, const float* route_w,
                   float* y, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    MXFP4_TRY(check_moe(n_experts, hidden, inter, n_tokens, top_k, workspace, ws_bytes));
    MXFP4_TRY(check_ptr(down_bank));
    MXFP4_TRY(check_ptr(act));
    MXFP4_TRY(check_ptr(y));
    if (expert_ids == nullptr || (reinterpret_cast<uintptr_t>(expert_ids) & 3u) ||
        route_w == nullptr || (reinterpret_cast<uintptr_t>(route_w) & 3u))
        return MXFP4_STATUS_BAD_POINTER;
    return from_cuda(mxk::launch_moe_down(
        mxk::one_segment_bank(u8(down_bank), n_experts, mxk::padded_nbytes(hidden, inter)),
        n_experts, hidden, inter, act, n_tokens, top_k, route_w, 0, y, workspace, stream));
}

namespace {

bool ptr4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_mode(int mode, float swiglu_limit) {
    if (mode != MXFP4_MOE_MODE_F32 && mode != MXFP4_MOE_MODE_V41) return MXFP4_STATUS_INVALID_ARGUMENT;
    if (!(swiglu_limit == swiglu_limit) || swiglu_limit > 3.0e38f) return MXFP4_STATUS_INVALID_ARGUMENT;
    return MXFP4_STATUS_OK;
}

}  // namespace

namespace {

// A bank given as segment base pointers (host array of device pointers).
int make_bank(const void* const* segs, int n_segments, int segment_slots, size_t stride,
              mxk::Bank* out) {
    if (segs == nullptr) return MXFP4_STATUS_BAD_POINTER;
    if (n_segments < 1 || n_segments > mxk::kMaxSegments || segment_slots < 1)
        return MXFP4_STATUS_INVALID_ARGUMENT;
    mxk::Bank b{};
    for (int i = 0; i < n_segments; ++i) {
        MXFP4_TRY(check_ptr(segs[i]));
        b.seg[i] = static_cast<const uint8_t*>(segs[i]);
    }
    b.n_seg = n_segments;
    b.seg_slots = segment_slots;
    b.stride = stride;
    *out = b;
    return MXFP4_STATUS_OK;
}

int gate_up_general(const mxk::Bank& gate, const mxk::Bank& up, int n_slots, int hidden,
                    int inter, const float* x, int n_tokens, int top_k, const int32_t* expert_ids,
                    const int32_t* slot_of, int n_experts, const float* route_w, int mode,
                    float swiglu_limit, float* act, void* workspace, size_t ws_bytes,
                    cudaStream_t stream) {
    MXFP4_TRY(check_moe(n_slots, hidden, inter, n_tokens, top_k, workspace, ws_bytes));
    MXFP4_TRY(check_mode(mode, swiglu_limit));
    if (n_experts < 1 || n_experts > (1 << 24)) return MXFP4_STATUS_INVALID_ARGUMENT;
    if (slot_of == nullptr && n_experts != n_slots) return MXFP4_STATUS_INVALID_ARGUMENT;
    MXFP4_TRY(check_ptr(x));
    MXFP4_TRY(check_ptr(act));
    if (!ptr4(expert_ids) || (slot_of != nullptr && !ptr4(slot_of)) ||
        (mode == MXFP4_MOE_MODE_V41 && !ptr4(route_w)))
        return MXFP4_STATUS_BAD_POINTER;
    const mxk::MoeAct epi{route_w, swiglu_limit > 0.0f ? swiglu_limit : 0.0f,
                          mode == MXFP4_MOE_MODE_V41 ? 1 : 0};
    return from_cuda(mxk::launch_moe_gate_up(gate, up, n_slots, hidden, inter, x, n_tokens, top_k,
                                             expert_ids, slot_of, n_experts, epi, act, workspace,
                                             stream));
}

int down_general(const mxk::Bank& down, int n_slots, int hidden, int inter, const float* act,
                 int n_tokens, int top_k, const float* route_w, int mode, float* y,
                 void* workspace, size_t ws_bytes, cudaStream_t stream) {
    MXFP4_TRY(check_moe(n_slots, hidden, inter, n_tokens, top_k, workspace, ws_bytes));
    MXFP4_TRY(check_mode(mode, 0.0f));
    MXFP4_TRY(check_ptr(act));
    MXFP4_TRY(check_ptr(y));
    if (mode == MXFP4_MOE_MODE_F32 && !ptr4(route_w)) return MXFP4_STATUS_BAD_POINTER;
    return from_cuda(mxk::launch_moe_down(down, n_slots, hidden, inter, act, n_tokens, top_k,
                                          route_w, mode == MXFP4_MOE_MODE_V41 ? 1 : 0, y,
                                          workspace, stream));
}

}  // namespace

int mxfp4_moe_gate_up_ex(const void* gate_bank, const void* up_bank, int n_slots, int hidden,
                         int inter, const float* x, int n_tokens, int top_k,
                         const int32_t* expert_ids, const int32_t* slot_of, int n_experts,
                         const float* route_w, int mode, float swiglu_limit, float* act,
                         void* workspace, size_t ws_bytes, cudaStream_t stream) {
    MXFP4_TRY(check_ptr(gate_bank));
    MXFP4_TRY(check_ptr(up_bank));
    MXFP4_TRY(check_shape(inter, hidden));
    if (n_slots < 1) return MXFP4_STATUS_INVALID_ARGUMENT;
    const size_t stride = mxk::padded_nbytes(inter, hidden);
    return gate_up_general(mxk::one_segment_bank(u8(gate_bank), n_slots, stride),
                           mxk::one_segment_bank(u8(up_bank), n_slots, stride), n_slots, hidden,
                           inter, x, n_tokens, top_k, expert_ids, slot_of, n_experts, route_w,
                           mode, swiglu_limit, act, workspace, ws_bytes, stream);
}

int mxfp4_moe_down_ex(const void* down_bank, int n_slots, int hidden, int inter, const float* act,
                      int n_tokens, int top_k, const float* route_w, int mode, float* y,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
    MXFP4_TRY(check_ptr(down_bank));
    MXFP4_TRY(check_shape(hidden, inter));
    if (n_slots < 1) return MXFP4_STATUS_INVALID_ARGUMENT;
    return down_general(
        mxk::one_segment_bank(u8(down_bank), n_slots, mxk::padded_nbytes(hidden, inter)), n_slots,
        hidden, inter, act, n_tokens, top_k, route_w, mode, y, workspace, ws_bytes, stream);
}

int mxfp4_moe_gate_up_seg(const void* const* gate_segments, const void* const* up_segments,
                          int n_segments, int segment_slots, int hidden, int inter, const float* x,
                          int n_tokens, int top_k, const int32_t* expert_ids,
                          const int32_t* slot_of, int n_experts, const float* route_w, int mode,
                          float swiglu_limit, float* act, void* workspace, size_t ws_bytes,
                          cudaStream_t stream) {
    MXFP4_TRY(check_shape(inter, hidden));
    if (segment_slots < 1 || n_segments < 1 || n_segments > mxk::kMaxSegments ||
        static_cast<long long>(n_segments) * segment_slots > (1 << 20))
        return MXFP4_STATUS_INVALID_ARGUMENT;
    const size_t stride = mxk::padded_nbytes(inter, hidden);
    mxk::Bank gate{}, up{};
    MXFP4_TRY(make_bank(gate_segments, n_segments, segment_slots, stride, &gate));
    MXFP4_TRY(make_bank(up_segments, n_segments, segment_slots, stride, &up));
    return gate_up_general(gate, up, n_segments * segment_slots, hidden, inter, x, n_tokens, top_k,
                           expert_ids, slot_of, n_experts, route_w, mode, swiglu_limit, act,
                           workspace, ws_bytes, stream);
}

int mxfp4_moe_down_seg(const void* const* down_segments, int n_segments, int segment_slots,
                       int hidden, int inter, const float* act, int n_tokens, int top_k,
                       const float* route_w, int mode, float* y, void* workspace, size_t ws_bytes,
                       cudaStream_t stream) {
    MXFP4_TRY(check_shape(hidden, inter));
    if (segment_slots < 1 || n_segments < 1 || n_segments > mxk::kMaxSegments ||
        static_cast<long long>(n_segments) * segment_slots > (1 << 20))
        return MXFP4_STATUS_INVALID_ARGUMENT;
    mxk::Bank down{};
    MXFP4_TRY(make_bank(down_segments, n_segments, segment_slots,
                        mxk::padded_nbytes(hidden, inter), &down));
    return down_general(down, n_segments * segment_slots, hidden, inter, act, n_tokens, top_k,
                        route_w, mode, y, workspace, ws_bytes, stream);
}

int mxfp4_moe_cold_pairs(const void* workspace, size_t ws_bytes, int n_slots, int n_tokens,
                         int top_k, int* n_cold, int32_t* pairs_host, int capacity,
                         cudaStream_t stream) {
    if (n_slots < 1 || n_tokens < 1 || top_k < 1 ||
        static_cast<long long>(n_tokens) * top_k > (1 << 22) || capacity < 0)
        return MXFP4_STATUS_INVALID_ARGUMENT;
    if (workspace == nullptr || n_cold == nullptr || !aligned16(workspace) ||
        (capacity > 0 && pairs_host == nullptr))
        return MXFP4_STATUS_BAD_POINTER;
    if (ws_bytes < mxk::moe_workspace_bytes(n_slots, n_tokens, top_k, 32, 32))
        return MXFP4_STATUS_WORKSPACE_TOO_SMALL;
    return from_cuda(mxk::moe_cold_pairs(workspace, n_slots, n_tokens * top_k, n_cold, pairs_host,
                                         capacity, stream));
}

int mxfp4_moe_plan_errors(const void* workspace, size_t ws_bytes, int* n_invalid,
                          cudaStream_t stream) {
    if (workspace == nullptr || n_invalid == nullptr || !aligned16(workspace))
        return MXFP4_STATUS_BAD_POINTER;
    if (ws_bytes < 16) return MXFP4_STATUS_WORKSPACE_TOO_SMALL;
    return from_cuda(mxk::moe_plan_errors(workspace, n_invalid, stream));
}

}  // extern "C"
