// matvec.cu -- standalone MXFP4 decode, and the FP32 matrix-vector /
// small-batch product on the CUDA cores (sm_103a).
//
// Product ("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs", PEROP kernels
// mxfp4_mv and mxfp4_mm, host fn matmat): Y[t*rows + r] = W[r,:] . X[t,:].
// The group walk is matmat_core.cuh's; here the grid is laid out as
// x = blocks of kWarps*R rows, y = chunks of NB tokens (the page's z = token
// chunk), and the row sums are written after a warp butterfly.
#include "matmat_core.cuh"
#include "kernels.h"

namespace mxk {
namespace {

// Standalone decode: thread i owns code word i (8 consecutive elements of the
// flattened row-major matrix, because words and elements are both row-major)
// and group i/4's scale.
__global__ void __launch_bounds__(256) k_dequant(const uint32_t* __restrict__ words,
                                                 size_t n_words,
                                                 const uint8_t* __restrict__ scales,
                                                 float4* __restrict__ out) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_words;
         i += stride) {
        const uint32_t word = __ldg(words + i);
        const float s = e8m0_to_f32(__ldg(scales + (i >> 2)));
        float v[8];
        e2m1x8_to_f32(word, v);
        // E2M1 value times a power of two: exact in float (no flush to zero).
        out[2 * i] = make_float4(__fmul_rn(v[0], s), __fmul_rn(v[1], s), __fmul_rn(v[2], s),
                                 __fmul_rn(v[3], s));
        out[2 * i + 1] = make_float4(__fmul_rn(v[4], s), __fmul_rn(v[5], s),
                                     __fmul_rn(v[6], s), __fmul_rn(v[7], s));
    }
}

template <int R, int NB>
__global__ void __launch_bounds__(kThreads) k_matmat(const uint8_t* __restrict__ w, int rows,
                                                     int cols, const float* __restrict__ X,
                                                     int nb, float* __restrict__ Y) {
    extern __shared__ float4 smem4[];
    float* xs = reinterpret_cast<float*>(smem4);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t0 = blockIdx.y * NB;
    const int nbt = min(NB, nb - t0);
    const long row_w = static_cast<long>(blockIdx.x) * (kWarps * R) + warp * R;

    const uint8_t* const wm[1] = {w};
    const float* xt[NB];
#pragma unroll
    for (int t = 0; t < NB; ++t)
        xt[t] = t < nbt ? X + static_cast<size_t>(t0 + t) * cols : nullptr;

    float acc[1][R][NB];
    zero(acc);
    cta_group_walk<R, NB, 1>(wm, rows, cols, row_w, xt, xs, acc);
    warp_allreduce(acc);

#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int t = 0; t < NB; ++t)
            if (lane == ((i * NB + t) & 31) && row_w + i < rows && t < nbt)
                Y[static_cast<size_t>(t0 + t) * rows + row_w + i] = acc[0][i][t];
}

// ---------------------------------------------------------------------------
// Streaming product for the case where all NB tokens' x fit in shared memory
// (staged once per CTA).  Persistent warps: warp j of the grid takes the row
// blocks j, j + (warps in grid), ...; each row block of R rows is walked in
// batches of U groups per lane (32*U groups), and the code words and scale
// bytes of the NEXT batch are loaded into registers before the current batch
// is decoded and multiplied, so every warp keeps its next loads in flight
// while it computes.  Lane l still takes groups l, l+32, l+64, ... of a row in
// increasing order and each token sees group_dots' arithmetic, so the results
// are bit-identical to the chunked kernel's.
template <int U, int R>
struct Batch {
    uint4 code[U][R];
    uint32_t sc[U][R];
};

template <int R, int NB, int U>
__global__ void __launch_bounds__(kThreads, 2) k_stream(const uint8_t* __restrict__ w, int rows,
                                                        int cols, const float* __restrict__ X,
                                                        int nb, float* __restrict__ Y) {
    extern __shared__ float4 smem4[];
    float* xs = reinterpret_cast<float*>(smem4);   // [NB][gpr][kXPad]
    const int gpr = cols / kGroup;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t0 = blockIdx.y * NB;
    const int nbt = min(NB, nb - t0);
    const uint8_t* scales = w + static_cast<size_t>(rows) * cols / 2;
    const long n_rb = (rows + R - 1) / R;
    const int n_gb = (gpr + 32 * U - 1) / (32 * U);
    const long stride = static_cast<long>(gridDim.x) * kWarps;

    auto load = [&](long rb, int gb, Batch<U, R>& b) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int g = gb * 32 * U + u * 32 + lane;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const long row = rb * R + i;
                if (g < gpr && row < rows) {
                    b.code[u][i] = ldg_stream(group_codes(w, gpr, row, g));
                    b.sc[u][i] = group_scale_byte(scales, gpr, row, g);
                } else {
                    b.code[u][i] = make_uint4(0u, 0u, 0u, 0u);
                    b.sc[u][i] = 0u;
                }
            }
        }
    };

    long rb = static_cast<long>(blockIdx.x) * kWarps + warp;
    int gb = 0;
    Batch<U, R> A, B;
    if (rb < n_rb) load(rb, 0, A);   // in flight while x is staged

    for (int i = threadIdx.x; i < NB * gpr * 8; i += kThreads) {
        const int t = i / (gpr * 8);
        const int rem = i - t * gpr * 8;
        const int g = rem >> 3, q = rem & 7;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < nbt)
            v = __ldg(reinterpret_cast<const float4*>(X + static_cast<size_t>(t0 + t) * cols +
                                                      static_cast<size_t>(g) * kGroup) + q);
        *reinterpret_cast<float4*>(xs + (t * gpr + g) * kXPad + q * 4) = v;
    }
    __syncthreads();

    float acc[R][NB];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int t = 0; t < NB; ++t) acc[i][t] = 0.0f;

    // One batch: prefetch the next into `nxt`, then multiply `cur`.
    auto step = [&](Batch<U, R>& cur, Batch<U, R>& nxt) -> bool {
        long rb2 = rb;
        int gb2 = gb + 1;
        if (gb2 == n_gb) {
            gb2 = 0;
            rb2 += stride;
        }
        if (rb2 < n_rb) load(rb2, gb2, nxt);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int g = gb * 32 * U + u * 32 + lane;
            if (g < gpr) {
                const float* xp[NB];
#pragma unroll
                for (int t = 0; t < NB; ++t) xp[t] = xs + (t * gpr + g) * kXPad;
                float dots[R][NB];
                group_dots<R, NB>(cur.code[u], xp, dots);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const float s = e8m0_to_f32(cur.sc[u][i]);
#pragma unroll
                    for (int t = 0; t < NB; ++t) acc[i][t] = __fmaf_rn(s, dots[i][t], acc[i][t]);
                }
            }
        }
        if (gb == n_gb - 1) {
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int t = 0; t < NB; ++t) {
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        acc[i][t] = __fadd_rn(acc[i][t], __shfl_xor_sync(0xffffffffu, acc[i][t], off));
                    const long row = rb * R + i;
                    if (lane == ((i * NB + t) & 31) && row < rows && t < nbt)
                        Y[static_cast<size_t>(t0 + t) * rows + row] = acc[i][t];
                    acc[i][t] = 0.0f;
                }
        }
        rb = rb2;
        gb = gb2;
        return rb < n_rb;
    };

    if (rb < n_rb) {
        while (step(A, B) && step(B, A)) {
        }
    }
}

// ---------------------------------------------------------------------------
// Matvec with the weights landed in shared memory by bulk copies.  Each warp
// owns a ring of S stages; a stage holds one row block of R rows (its code
// bytes, contiguous in the buffer, and a 16-byte aligned cover of its scale
// bytes) and is filled by two cp.async.bulk copies that complete on the
// stage's mbarrier.  The warp processes its row blocks j, j + (warps in grid),
// ... in order and refills a stage as soon as all lanes are done with it, so
// S row blocks per warp are always on their way from HBM, with no registers
// held for them.  Arithmetic and lane-to-group mapping are those of the other
// product kernels (bit-identical results).
__device__ int g_fault_matvec;   // set when a bounded wait gives up

constexpr uint32_t kWaitLimit = 1u << 22;

__host__ __device__ constexpr uint32_t round16(uint32_t v) { return (v + 15u) & ~15u; }

template <int R>
__host__ __device__ constexpr uint32_t bulk_stage_bytes(int cols) {
    return static_cast<uint32_t>(R) * static_cast<uint32_t>(cols) / 2 +
           round16(static_cast<uint32_t>(R) * static_cast<uint32_t>(cols / kGroup) + 32u);
}

template <int R, int S>
__global__ void __launch_bounds__(kThreads, 2) k_mv_bulk(const uint8_t* __restrict__ w, int rows,
                                                         int cols, const float* __restrict__ x,
                                                         float* __restrict__ y) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int gpr = cols / kGroup;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t code_stage = static_cast<uint32_t>(R) * cols / 2;
    const uint32_t stage_bytes = bulk_stage_bytes<R>(cols);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + warp * S;
    float* xs = reinterpret_cast<float*>(smem + 1024);
    uint8_t* ring = smem + 1024 + static_cast<size_t>(gpr) * kXPad * sizeof(float) +
                    static_cast<size_t>(warp) * S * stage_bytes;
    const size_t plane = static_cast<size_t>(rows) * cols / 2;
    const long n_rb = (rows + R - 1) / R;
    const long stride = static_cast<long>(gridDim.x) * kWarps;
    const long rb0 = static_cast<long>(blockIdx.x) * kWarps + warp;
    const uint64_t policy = l2_evict_first();

    // The 16-byte aligned cover of a row block's scale bytes.
    auto scale_cover = [&](long r0, int nr, size_t& lo, uint32_t& bytes) {
        lo = (static_cast<size_t>(r0) * gpr) & ~static_cast<size_t>(15);
        const size_t hi = (static_cast<size_t>(r0 + nr) * gpr + 15) & ~static_cast<size_t>(15);
        bytes = static_cast<uint32_t>(hi - lo);
    };
    auto issue = [&](long rb, int st) {   // lane 0 only
        const long r0 = rb * R;
        const int nr = static_cast<int>(min(static_cast<long>(R), rows - r0));
        const uint32_t cb = static_cast<uint32_t>(nr) * cols / 2;
        size_t lo;
        uint32_t sb;
        scale_cover(r0, nr, lo, sb);
        uint8_t* dst = ring + st * stage_bytes;
        mbar_arrive_expect_tx(&bars[st], cb + sb);
        bulk_g2s(dst, w + static_cast<size_t>(r0) * cols / 2, cb, &bars[st], policy);
        bulk_g2s(dst + code_stage, w + plane + lo, sb, &bars[st], policy);
    };

    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < S; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
#pragma unroll
        for (int st = 0; st < S; ++st)
            if (rb0 + st * stride < n_rb) issue(rb0 + st * stride, st);
    }
    // x into shared memory while the first stages are in flight (eight loads in
    // flight per thread before their stores)
    for (int base = threadIdx.x; base < gpr * 8; base += 8 * kThreads) {
        float4 v[8];
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            const int i = base + k8 * kThreads;
            if (i < gpr * 8)
                v[k8] = __ldg(reinterpret_cast<const float4*>(x) + i);
        }
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            const int i = base + k8 * kThreads;
            if (i < gpr * 8) *reinterpret_cast<float4*>(xs + (i >> 3) * kXPad + (i & 7) * 4) = v[k8];
        }
    }
    __syncthreads();

    int k = 0;
    for (long rb = rb0; rb < n_rb; rb += stride, ++k) {
        const int st = k % S;
        if (!mbar_wait(&bars[st], static_cast<uint32_t>(k / S) & 1u, kWaitLimit)) {
            if (lane == 0) atomicOr(&g_fault_matvec, 1);
            return;
        }
        const long r0 = rb * R;
        const int nr = static_cast<int>(min(static_cast<long>(R), rows - r0));
        size_t lo;
        uint32_t sb;
        scale_cover(r0, nr, lo, sb);
        const uint8_t* codes = ring + st * stage_bytes;
        const uint8_t* sc = codes + code_stage + (static_cast<size_t>(r0) * gpr - lo);
        float acc[R];
#pragma unroll
        for (int i = 0; i < R; ++i) acc[i] = 0.0f;
        for (int g = lane; g < gpr; g += 32) {
            uint4 code[R];
#pragma unroll
            for (int i = 0; i < R; ++i)
                code[i] = i < nr ? *reinterpret_cast<const uint4*>(
                                       codes + static_cast<size_t>(i) * cols / 2 + g * kGroupBytes)
                                 : make_uint4(0u, 0u, 0u, 0u);
            const float* xp[1] = {xs + g * kXPad};
            float dots[R][1];
            group_dots<R, 1>(code, xp, dots);
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const float s = i < nr ? e8m0_to_f32(sc[i * gpr + g]) : 0.0f;
                acc[i] = __fmaf_rn(s, dots[i][0], acc[i]);
            }
        }
        __syncwarp();   // every lane is done with this stage
        if (lane == 0 && rb + S * stride < n_rb) {
            fence_proxy_async_smem();
            issue(rb + S * stride, st);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                acc[i] = __fadd_rn(acc[i], __shfl_xor_sync(0xffffffffu, acc[i], off));
            if (lane == i && i < nr) y[r0 + i] = acc[i];
        }
    }
}

// Per-device opt-in to more than 48 KB of dynamic shared memory.
template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 152;
    return sms;
}

template <int R, int NB, int U>
cudaError_t launch_stream(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                          cudaStream_t s) {
    const int gpr = cols / kGroup;
    const size_t smem = static_cast<size_t>(NB) * gpr * kXPad * sizeof(float);
    auto kernel = k_stream<R, NB, U>;
    cudaError_t e = allow_smem(kernel, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const long n_rb = (rows + R - 1) / R;
    const long want = (n_rb + kWarps - 1) / kWarps;
    const long cap = static_cast<long>(per_sm) * sm_count();
    const dim3 grid(static_cast<unsigned>(want < cap ? want : cap), (nb + NB - 1) / NB);
    kernel<<<grid, kThreads, smem, s>>>(w, rows, cols, X, nb, Y);
    return cudaGetLastError();
}

constexpr int kBulkR = 2;
constexpr int kBulkS = 2;

size_t bulk_smem_bytes(int cols) {
    return 1024 + static_cast<size_t>(cols / kGroup) * kXPad * sizeof(float) +
           static_cast<size_t>(kWarps) * kBulkS * bulk_stage_bytes<kBulkR>(cols);
}

cudaError_t launch_mv_bulk(const uint8_t* w, int rows, int cols, const float* x, float* y,
                           cudaStream_t s) {
    const size_t smem = bulk_smem_bytes(cols);
    auto kernel = k_mv_bulk<kBulkR, kBulkS>;
    cudaError_t e = allow_smem(kernel, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const long n_rb = (rows + kBulkR - 1) / kBulkR;
    const long want = (n_rb + kWarps - 1) / kWarps;
    const long cap = static_cast<long>(per_sm) * sm_count();
    kernel<<<static_cast<unsigned>(want < cap ? want : cap), kThreads, smem, s>>>(w, rows, cols, x,
                                                                                 y);
    return cudaGetLastError();
}

template <int R, int NB>
cudaError_t launch(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                   cudaStream_t s) {
    const dim3 grid((rows + kWarps * R - 1) / (kWarps * R), (nb + NB - 1) / NB);
    k_matmat<R, NB><<<grid, kThreads, kStageBytes, s>>>(w, rows, cols, X, nb, Y);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequant(const uint8_t* w, int rows, int cols, float* out, cudaStream_t s) {
    const size_t n_words = static_cast<size_t>(rows) * cols / 8;
    const uint8_t* scales = w + static_cast<size_t>(rows) * cols / 2;
    const size_t blocks_needed = (n_words + 255) / 256;
    const size_t cap = 152u * 16u;
    const unsigned blocks = static_cast<unsigned>(blocks_needed < cap ? blocks_needed : cap);
    k_dequant<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(w), n_words, scales,
                                     reinterpret_cast<float4*>(out));
    return cudaGetLastError();
}

// Largest staged x (bytes) for which the streaming kernel is used.
constexpr size_t kStreamSmemMax = 96 * 1024;

cudaError_t launch_matmat_fp32(const uint8_t* w, int rows, int cols, const float* X, int nb,
                               float* Y, cudaStream_t s) {
    const int gpr = cols / kGroup;
    if (nb == 1 && bulk_smem_bytes(cols) <= 110 * 1024)
        return launch_mv_bulk(w, rows, cols, X, Y, s);
    if (nb == 1 && static_cast<size_t>(gpr) * kXPad * sizeof(float) <= kStreamSmemMax) {
        if (gpr <= 32) return launch_stream<2, 1, 1>(w, rows, cols, X, nb, Y, s);
        if (gpr <= 64) return launch_stream<2, 1, 2>(w, rows, cols, X, nb, Y, s);
        if (gpr <= 96) return launch_stream<2, 1, 3>(w, rows, cols, X, nb, Y, s);
        return launch_stream<2, 1, 4>(w, rows, cols, X, nb, Y, s);
    }
    if (nb == 1) return launch<4, 1>(w, rows, cols, X, nb, Y, s);
    if (nb == 2) return launch<4, 2>(w, rows, cols, X, nb, Y, s);
    if (nb <= 4) return launch<2, 4>(w, rows, cols, X, nb, Y, s);
    return launch<2, 8>(w, rows, cols, X, nb, Y, s);
}

cudaError_t read_fault_matvec(int* value, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_fault_matvec, sizeof(int));
    if (e != cudaSuccess || !reset) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_matvec, &zero, sizeof(int));
}

}  // namespace mxk
