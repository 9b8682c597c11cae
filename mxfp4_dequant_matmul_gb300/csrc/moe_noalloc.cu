// moe_noalloc.cu -- the routed-expert layer for callers that cannot allocate
// device memory.
//
// Some callers of this library have no way to hand it a workspace: a serving
// process that gave all of its device memory to its own pool allocator at
// start-up (and owns no cudaMalloc it may call afterwards), or a real-time
// loop that must not allocate once running because cudaMalloc can block the
// device and stall every other stream.  For them the layer's scratch -- the
// routing plan, the gate/up activation and the per-pair down outputs -- lives
// in one file-scope device array of fixed size, which every GPU that loads the
// library holds until the process exits.  The entry point allocates nothing:
// no cudaMalloc, no cudaFree, no allocating library routine.
//
// The array's name in host code is a host-side stand-in, not a device
// address, so the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the kernels.
// The address belongs to the context that loaded the library's module: if the
// device's context is destroyed and made again (cudaDeviceReset), the next
// call sees a new context id and looks the address up again.
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "../../include/mxfp4.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = MXFP4_MOE_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_moe_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mu;
void* g_addr[kMaxDevices] = {};
unsigned long long g_addr_ctx[kMaxDevices] = {};

// Device address of g_moe_scratch on the current device: looked up on the
// first call per device (and again after the device's context was replaced),
// then cached.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // 0 before the runtime has made a context current: then the lookup below
    // runs (and makes it current), and the next call caches under its id
    const unsigned long long ctx = mxk::current_context_id();
    std::lock_guard<std::mutex> lock(g_addr_mu);
    if (g_addr[dev] == nullptr || ctx == 0 || ctx != g_addr_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_moe_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
        g_addr_ctx[dev] = ctx;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool shape_ok(int rows, int cols) {
    return rows >= 1 && cols >= 32 && cols % 32 == 0 &&
           static_cast<long long>(rows) * cols <= (1LL << 46);
}

}  // namespace

// Unique id of the calling thread's current context (0 if the driver cannot
// say): an address cached under one context is not used under another.
unsigned long long mxk::current_context_id() {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
        ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

extern "C" int mxfp4_moe_layer_noalloc(const void* gate_bank, const void* up_bank,
                                       const void* down_bank, int n_experts, int hidden,
                                       int inter, const float* x, int n_tokens, int top_k,
                                       const int32_t* expert_ids, const float* route_w, float* y,
                                       cudaStream_t stream) {
    if (n_experts < 1 || n_experts > (1 << 20) || n_tokens < 1 || top_k < 1 ||
        static_cast<long long>(n_tokens) * top_k > (1 << 22) || !shape_ok(inter, hidden) ||
        !shape_ok(hidden, inter) ||
        static_cast<long long>(n_experts) * inter * hidden > (1LL << 46))
        return MXFP4_STATUS_INVALID_ARGUMENT;
    if (!gate_bank || !up_bank || !down_bank || !x || !y || !aligned16(gate_bank) ||
        !aligned16(up_bank) || !aligned16(down_bank) || !aligned16(x) || !aligned16(y) ||
        !expert_ids || !route_w || !aligned4(expert_ids) || !aligned4(route_w))
        return MXFP4_STATUS_BAD_POINTER;

    // Scratch layout: [routing plan + per-pair down outputs | act], act 256-B aligned.
    const size_t plan_bytes = mxk::moe_workspace_bytes(n_experts, n_tokens, top_k, hidden, inter);
    const size_t act_offset = (plan_bytes + 255) / 256 * 256;
    const size_t act_bytes = static_cast<size_t>(n_tokens) * top_k * inter * sizeof(float);
    if (act_offset + act_bytes > kScratchBytes) return MXFP4_STATUS_WORKSPACE_TOO_SMALL;

    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e == cudaSuccess) {
        float* act = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + act_offset);
        const size_t gu_stride = mxk::padded_nbytes(inter, hidden);
        e = mxk::launch_moe_gate_up(
            mxk::one_segment_bank(static_cast<const uint8_t*>(gate_bank), n_experts, gu_stride),
            mxk::one_segment_bank(static_cast<const uint8_t*>(up_bank), n_experts, gu_stride),
            n_experts, hidden, inter, x, n_tokens, top_k, expert_ids, nullptr, n_experts,
            mxk::MoeAct{nullptr, 0.0f, 0}, act, scratch, stream);
        if (e == cudaSuccess)
            e = mxk::launch_moe_down(
                mxk::one_segment_bank(static_cast<const uint8_t*>(down_bank), n_experts,
                                      mxk::padded_nbytes(hidden, inter)),
                n_experts, hidden, inter, act, n_tokens, top_k, route_w, 0, y, scratch, stream);
    }
    if (e != cudaSuccess) {
        mxk::record_cuda_error(static_cast<int>(e));
        return MXFP4_STATUS_LAUNCH_FAILED;
    }
    return MXFP4_STATUS_OK;
}
