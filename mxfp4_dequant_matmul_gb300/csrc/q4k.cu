// q4k.cu -- the second codec: GGUF Q4_K weights with f32 activations (layout
// and element values in include/q4k.h; "rlx-cpu 0.2.17 src/gguf_matmul.rs",
// the exact arm of gguf_matmul_bt_m1_parallel and its Q4_K block dot).
//
// Work: one warp per row, eight 144-byte super-blocks per step (their loads in
// flight together, their headers unpacked by the lanes together), lane l taking
// the 32-bit code word at bytes 16 + 4 l of each: the low nibbles of its four bytes are
// elements 64 s + 4 (l % 8) + b of sub-block 2 s (s = l / 8), the high nibbles
// the same positions + 32 of sub-block 2 s + 1.  The word's nibbles are spread
// into bytes (two logic operations), each byte lands in the mantissa of 2^23
// (one byte permute), one subtraction of 2^23 gives q and one FMA rounds
// d sc q - dmin m once, as the exact arm does (two elements per packed FP32x2
// operation); the FP32 products with x then go into two
// chains (even and odd elements) per word, four sums per lane by super-block
// index mod 4, ((S0 + S1) + S2) + S3 and a fixed warp tree.  Up to eight tokens
// share each decoded word.
#include <cstdint>

#include <cuda_fp16.h>

#include "../../include/q4k.h"
#include "kernels.h"

namespace {

constexpr int kQK = 256;
constexpr int kBlk = 144;
constexpr int kWarpsQ = 8;
constexpr int kUnrollQ = 8;   // super-blocks per step: their loads in flight together

__device__ __forceinline__ uint4 ldg_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// A super-block's factors for this lane's two sub-blocks j = 2 s and j + 1:
// a = d sc, b = dmin m (both exact in FP32).
struct Factors {
    float a0, b0, a1, b1;
};
__device__ __forceinline__ Factors block_factors(const uint4 hdr, int s) {
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
    // bytes 4..15: hdr.y = bytes 4..7, hdr.z = 8..11, hdr.w = 12..15
    const int k = (2 * s) & 3;   // the two sub-blocks' index within their half
    uint32_t sc[2], mn[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t y = (hdr.y >> (8 * (k + i))) & 0xFFu;
        const uint32_t z = (hdr.z >> (8 * (k + i))) & 0xFFu;
        const uint32_t w = (hdr.w >> (8 * (k + i))) & 0xFFu;
        if (s < 2) {
            sc[i] = y & 63u;
            mn[i] = z & 63u;
        } else {
            sc[i] = (w & 0x0Fu) | ((y >> 6) << 4);
            mn[i] = (w >> 4) | ((z >> 6) << 4);
        }
    }
    Factors f;
    f.a0 = d * static_cast<float>(sc[0]);
    f.b0 = dmin * static_cast<float>(mn[0]);
    f.a1 = d * static_cast<float>(sc[1]);
    f.b1 = dmin * static_cast<float>(mn[1]);
    return f;
}

// The 8 element values of a code word: v[b] = low nibble of byte b (first
// sub-block), v[4 + b] = high nibble (second).  q lands in the low mantissa
// bits of 2^23 (one byte permute), one subtraction of 2^23 gives q exactly and
// fma(a, q, -b) rounds the exact a q - b once; with an infinite or NaN d or dmin
// (finite = false) q is taken as a float and a q as a product, as the
// definition does.
__device__ __forceinline__ void word_values(uint32_t word, const Factors& f, bool finite,
                                            float (&v)[8]) {
    const uint32_t lo = word & 0x0F0F0F0Fu, hi = (word >> 4) & 0x0F0F0F0Fu;
    const uint32_t magic = 0x4B000000u;
    if (finite) {
        // two elements per packed FP32x2 operation (each lane of it rounds as
        // the scalar operation would)
        const float2 a0 = make_float2(f.a0, f.a0), a1 = make_float2(f.a1, f.a1);
        const float2 nb0 = make_float2(-f.b0, -f.b0), nb1 = make_float2(-f.b1, -f.b1);
        const float2 n23 = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
        for (int b = 0; b < 4; b += 2) {
            // bytes b, b+1 of lo / hi into byte 0, bytes 1-3 from magic (0x00, 0x00, 0x4B)
            const float2 ql = make_float2(__uint_as_float(__byte_perm(lo, magic, 0x7650u + b)),
                                          __uint_as_float(__byte_perm(lo, magic, 0x7651u + b)));
            const float2 qh = make_float2(__uint_as_float(__byte_perm(hi, magic, 0x7650u + b)),
                                          __uint_as_float(__byte_perm(hi, magic, 0x7651u + b)));
            // q = (2^23 + q) - 2^23 exactly; a q - b rounded once by the FMA
            const float2 wl = __ffma2_rn(a0, __fadd2_rn(ql, n23), nb0);
            const float2 wh = __ffma2_rn(a1, __fadd2_rn(qh, n23), nb1);
            v[b] = wl.x;
            v[b + 1] = wl.y;
            v[4 + b] = wh.x;
            v[4 + b + 1] = wh.y;
        }
    } else {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float ql = static_cast<float>((lo >> (8 * b)) & 0xFFu);
            const float qh = static_cast<float>((hi >> (8 * b)) & 0xFFu);
            v[b] = __fsub_rn(__fmul_rn(f.a0, ql), f.b0);
            v[4 + b] = __fsub_rn(__fmul_rn(f.a1, qh), f.b1);
        }
    }
}

template <int NB>
__global__ void __launch_bounds__(kWarpsQ * 32)
    k_q4k_mm(const uint8_t* __restrict__ w, int rows, int cols, const float* __restrict__ X,
             int nb, float* __restrict__ Y) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = blockIdx.y * NB;
    const int nbt = min(NB, nb - t0);
    const int bpr = cols / kQK;
    const int s = lane >> 3;
    const int e_lo = 64 * s + 4 * (lane & 7);   // this lane's first low-nibble element
    const float* xt[NB];
#pragma unroll
    for (int t = 0; t < NB; ++t) xt[t] = X + static_cast<size_t>(t0 + min(t, nbt - 1)) * cols;
    // rows dealt to the warps in turn (a grid of one wave)
    for (int row = blockIdx.x * kWarpsQ + warp; row < rows;
         row += static_cast<int>(gridDim.x) * kWarpsQ) {
        const uint8_t* rb = w + static_cast<size_t>(row) * bpr * kBlk;
        float acc[NB][4];
#pragma unroll
        for (int t = 0; t < NB; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

        for (int b0 = 0; b0 < bpr; b0 += kUnrollQ) {
            // the step's eight headers are read and unpacked by the lanes together:
            // lane l takes super-block b0 + l / 4 and its sub-blocks 2 (l % 4) and
            // 2 (l % 4) + 1; the lanes of sub-blocks 2 s, 2 s + 1 then fetch theirs
            // from lane 4 u + s for super-block b0 + u
            const uint4 hdr = ldg_u4(rb + static_cast<size_t>(min(b0 + (lane >> 2), bpr - 1)) * kBlk);
            uint32_t code[kUnrollQ];
#pragma unroll
            for (int u = 0; u < kUnrollQ; ++u) {
                const int b = min(b0 + u, bpr - 1);   // (past the row's end: a repeat, unused)
                code[u] = ldg_u32(rb + static_cast<size_t>(b) * kBlk + 16 + 4 * lane);
            }
            const Factors fl = block_factors(hdr, lane & 3);
            const bool finite = __all_sync(0xffffffffu, isfinite(fl.a0) && isfinite(fl.b0) &&
                                                            isfinite(fl.a1) && isfinite(fl.b1));
#pragma unroll
            for (int u = 0; u < kUnrollQ; ++u) {
                const int b = b0 + u;
                Factors f;
                f.a0 = __shfl_sync(0xffffffffu, fl.a0, 4 * u + s);
                f.b0 = __shfl_sync(0xffffffffu, fl.b0, 4 * u + s);
                f.a1 = __shfl_sync(0xffffffffu, fl.a1, 4 * u + s);
                f.b1 = __shfl_sync(0xffffffffu, fl.b1, 4 * u + s);
                // (past the row's end: the last block again, its sum not added,
                // so that the control flow stays the same for every lane)
                float v[8];
                word_values(code[u], f, finite, v);
#pragma unroll
                for (int t = 0; t < NB; ++t) {
                    if (NB > 1 && t >= nbt) break;
                    const float* xb = xt[t] + static_cast<size_t>(min(b, bpr - 1)) * kQK + e_lo;
                    const float4 xl = __ldg(reinterpret_cast<const float4*>(xb));
                    const float4 xh = __ldg(reinterpret_cast<const float4*>(xb + 32));
                    // packed products: chain .x takes the even elements, .y the odd
                    float2 c = __fmul2_rn(make_float2(v[0], v[1]), make_float2(xl.x, xl.y));
                    c = __ffma2_rn(make_float2(v[2], v[3]), make_float2(xl.z, xl.w), c);
                    c = __ffma2_rn(make_float2(v[4], v[5]), make_float2(xh.x, xh.y), c);
                    c = __ffma2_rn(make_float2(v[6], v[7]), make_float2(xh.z, xh.w), c);
                    if (b < bpr) acc[t][u & 3] = __fadd_rn(acc[t][u & 3], __fadd_rn(c.x, c.y));
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            if (NB > 1 && t >= nbt) break;
            float v = __fadd_rn(__fadd_rn(__fadd_rn(acc[t][0], acc[t][1]), acc[t][2]), acc[t][3]);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) Y[static_cast<size_t>(t0 + t) * rows + row] = v;
        }
    }
}

// Thread per (row, super-block, code word): its 8 element values.
__global__ void k_q4k_dequant(const uint8_t* __restrict__ w, int rows, int cols,
                              float* __restrict__ out) {
    const int bpr = cols / kQK;
    const size_t n_words = static_cast<size_t>(rows) * bpr * 32;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_words;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int lane = static_cast<int>(i & 31);
        const size_t blk = i >> 5;   // row * bpr + b
        const uint8_t* p = w + blk * kBlk;
        const uint4 hdr = ldg_u4(p);
        const uint32_t code = ldg_u32(p + 16 + 4 * lane);
        const int s = lane >> 3;
        float v[8];
        const Factors f = block_factors(hdr, s);
        word_values(code, f, isfinite(f.a0) && isfinite(f.b0) && isfinite(f.a1) && isfinite(f.b1),
                    v);
        const size_t row = blk / bpr, b = blk - row * bpr;
        float* o = out + row * cols + b * kQK + 64 * s + 4 * (lane & 7);
        *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(o + 32) = make_float4(v[4], v[5], v[6], v[7]);
    }
}

template <int NB>
cudaError_t launch_q4k(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                       cudaStream_t s) {
    // one wave: as many CTAs as the SMs hold at once, each warp taking rows in turn
    static mxk::PerDevice memo;
    const int per_wave = memo.get([] {
        int dev = 0, sms = 0, per_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_q4k_mm<NB>, kWarpsQ * 32,
                                                          0) != cudaSuccess)
            return 0;
        return sms * per_sm;
    });
    const int need = (rows + kWarpsQ - 1) / kWarpsQ;
    const int gx = per_wave > 0 && per_wave < need ? per_wave : need;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>((nb + NB - 1) / NB));
    k_q4k_mm<NB><<<grid, kWarpsQ * 32, 0, s>>>(w, rows, cols, X, nb, Y);
    return cudaGetLastError();
}

bool aligned16_q(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_q4k(const void* w, int rows, int cols, const void* a, const void* b) {
    if (rows < 1 || cols < kQK || cols % kQK != 0 ||
        static_cast<long long>(rows) * cols > (1LL << 46))
        return MXFP4_STATUS_INVALID_ARGUMENT;
    if (w == nullptr || a == nullptr || b == nullptr || !aligned16_q(w) || !aligned16_q(a) ||
        !aligned16_q(b))
        return MXFP4_STATUS_BAD_POINTER;
    return MXFP4_STATUS_OK;
}

int status_of(cudaError_t e) {
    if (e == cudaSuccess) return MXFP4_STATUS_OK;
    mxk::record_cuda_error(static_cast<int>(e));
    return MXFP4_STATUS_LAUNCH_FAILED;
}

}  // namespace

extern "C" {

size_t q4k_nbytes(int rows, int cols) {
    if (rows < 1 || cols < kQK || cols % kQK != 0) return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(cols / kQK) * kBlk;
}

int q4k_dequant(const void* w, int rows, int cols, float* out, cudaStream_t stream) {
    const int st = check_q4k(w, rows, cols, out, out);
    if (st != MXFP4_STATUS_OK) return st;
    const size_t n_words = static_cast<size_t>(rows) * (cols / kQK) * 32;
    const unsigned blocks = static_cast<unsigned>(
        n_words / 256 + 1 > 152u * 16u ? 152u * 16u : n_words / 256 + 1);
    k_q4k_dequant<<<blocks, 256, 0, stream>>>(static_cast<const uint8_t*>(w), rows, cols, out);
    return status_of(cudaGetLastError());
}

int q4k_mv(const void* w, int rows, int cols, const float* x, float* y, cudaStream_t stream) {
    const int st = check_q4k(w, rows, cols, x, y);
    if (st != MXFP4_STATUS_OK) return st;
    return status_of(launch_q4k<1>(static_cast<const uint8_t*>(w), rows, cols, x, 1, y, stream));
}

int q4k_mm(const void* w, int rows, int cols, const float* X, int nb, float* Y,
           cudaStream_t stream) {
    const int st = check_q4k(w, rows, cols, X, Y);
    if (st != MXFP4_STATUS_OK) return st;
    if (nb < 1 || nb > (1 << 24)) return MXFP4_STATUS_INVALID_ARGUMENT;
    const uint8_t* wb = static_cast<const uint8_t*>(w);
    if (nb == 1) return status_of(launch_q4k<1>(wb, rows, cols, X, nb, Y, stream));
    if (nb == 2) return status_of(launch_q4k<2>(wb, rows, cols, X, nb, Y, stream));
    if (nb <= 4) return status_of(launch_q4k<4>(wb, rows, cols, X, nb, Y, stream));
    return status_of(launch_q4k<8>(wb, rows, cols, X, nb, Y, stream));
}

}  // extern "C"
