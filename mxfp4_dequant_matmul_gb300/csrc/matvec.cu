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

template <int R, int NB, bool BF16X>
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
    cta_group_walk<R, NB, 1, BF16X>(wm, rows, cols, row_w, xt, xs, acc);
    warp_allreduce(acc);

#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int t = 0; t < NB; ++t)
            if (lane == ((i * NB + t) & 31) && row_w + i < rows && t < nbt)
                Y[static_cast<size_t>(t0 + t) * rows + row_w + i] = acc[0][i][t];
}

template <int R, int NB, bool BF16X>
cudaError_t launch(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                   cudaStream_t s) {
    const dim3 grid((rows + kWarps * R - 1) / (kWarps * R), (nb + NB - 1) / NB);
    k_matmat<R, NB, BF16X><<<grid, kThreads, kStageBytes, s>>>(w, rows, cols, X, nb, Y);
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

cudaError_t launch_matmat_fp32(const uint8_t* w, int rows, int cols, const float* X, int nb,
                               float* Y, cudaStream_t s) {
    if (nb == 1) return launch<4, 1, false>(w, rows, cols, X, nb, Y, s);
    if (nb == 2) return launch<4, 2, false>(w, rows, cols, X, nb, Y, s);
    if (nb <= 4) return launch<2, 4, false>(w, rows, cols, X, nb, Y, s);
    return launch<2, 8, false>(w, rows, cols, X, nb, Y, s);
}

// Placeholder for the tensor-core product: the same walk on bf16-rounded x.
// Every product of a bf16 value and a decoded weight is exact in FP32, so this
// has the tensor-core path's numerics (exact products, FP32 sums).
cudaError_t launch_mm_bf16(const uint8_t* w, int rows, int cols, const float* X, int nb,
                           float* Y, cudaStream_t s) {
    return launch<2, 8, true>(w, rows, cols, X, nb, Y, s);
}

}  // namespace mxk
