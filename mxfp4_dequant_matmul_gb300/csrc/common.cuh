// common.cuh -- device-side MXFP4 decode and small helpers shared by the
// kernels of libmxfp4.so (sm_103a).
//
// Format ("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs", const DECODE and
// const PEROP): a [rows, cols] matrix is a code plane of rows*cols/2 bytes --
// group g of row r is 16 bytes at byte (r*gpr + g)*16, four little-endian u32
// words, nibble j of word k being element 32g + 8k + j -- followed by a scale
// plane with one E8M0 byte per group at byte rows*cols/2 + r*gpr + g.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace mxk {

constexpr int kGroup = 32;        // elements per scale group
constexpr int kGroupBytes = 16;   // code bytes per group

// E8M0 byte -> float (DECODE fn mx_e8m0): the bits k << 23 give 2^(k-127);
// k = 0 gives the subnormal 2^-127 (bits 0x00400000), k = 255 gives NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t k) {
    uint32_t bits = (k == 0u) ? 0x00400000u : (k << 23);
    bits = (k == 255u) ? 0x7FC00000u : bits;
    return __uint_as_float(bits);
}

// Two f16 halves of a register -> two floats (exact widening).
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
    return make_float2(lo, hi);
}

// The four bytes of a code word (8 E2M1 codes) -> four f16x2 registers with
// the hardware E2M1 pair conversion: byte b holds codes 2b (low nibble) and
// 2b+1 (high nibble), which land in the low and high half of result b.  Every
// E2M1 value (0, +-0.5 .. +-6, -0 for code 8) is exact in f16.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// One code word -> its 8 element values as floats (exact).
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float (&v)[8]) {
    uint32_t h[4];
    e2m1x8_to_f16x2x4(w, h);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const float2 f = f16x2_to_f32x2(h[b]);
        v[2 * b] = f.x;
        v[2 * b + 1] = f.y;
    }
}

// Group dot products: for each of R rows (its 16 code bytes in code[i]) and
// each of NB tokens (32 floats of x at xp[t], 16-byte aligned) the sum of the
// 32 decoded codes times x, in FP32: two FMA chains, one over the even and one
// over the odd elements (one packed pair FMA feeds both), then even + odd.
// Every token sees exactly this sequence whatever R and NB are, which is what
// makes the batched product equal the matvec bit for bit.
template <int R, int NB>
__device__ __forceinline__ void group_dots(const uint4 (&code)[R], const float* const (&xp)[NB],
                                           float (&out)[R][NB]) {
    float2 d[R][NB];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int t = 0; t < NB; ++t) d[i][t] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float2 xv[NB][4];
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            const float4 xa = *reinterpret_cast<const float4*>(xp[t] + 8 * k);
            const float4 xb = *reinterpret_cast<const float4*>(xp[t] + 8 * k + 4);
            xv[t][0] = make_float2(xa.x, xa.y);
            xv[t][1] = make_float2(xa.z, xa.w);
            xv[t][2] = make_float2(xb.x, xb.y);
            xv[t][3] = make_float2(xb.z, xb.w);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const uint32_t word = k == 0 ? code[i].x : k == 1 ? code[i].y : k == 2 ? code[i].z
                                                                                 : code[i].w;
            uint32_t h[4];
            e2m1x8_to_f16x2x4(word, h);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float2 v = f16x2_to_f32x2(h[b]);
#pragma unroll
                for (int t = 0; t < NB; ++t) d[i][t] = __ffma2_rn(v, xv[t][b], d[i][t]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int t = 0; t < NB; ++t) out[i][t] = __fadd_rn(d[i][t].x, d[i][t].y);
}

// Device pointer arithmetic on the two planes.
__device__ __forceinline__ const uint4* group_codes(const uint8_t* w, size_t gpr, size_t row,
                                                    size_t g) {
    return reinterpret_cast<const uint4*>(w + (row * gpr + g) * kGroupBytes);
}

__device__ __forceinline__ uint32_t group_scale_byte(const uint8_t* scales, size_t gpr,
                                                     size_t row, size_t g) {
    return __ldg(scales + row * gpr + g);
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    // Weights are read once per call: do not keep them in L1.
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// --- shared-memory addresses, mbarriers and 1-D bulk copies -----------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// if it did not complete within `limit` polls (the caller records a fault and
// gives up instead of hanging the GPU).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
    const uint32_t a = smem_u32(bar);
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// Asynchronous global -> shared copy of `bytes` (multiple of 16, both
// addresses 16-byte aligned) completing on `bar`'s transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read exactly once (weights): evict first.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy for data that many CTAs read again: evict last.
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// mma.sync m16n8k16, f16 inputs, FP32 accumulator d += A B.  Lane (g = lane / 4,
// t = lane % 4) holds A rows g (a0, a2) and g + 8 (a1, a3) at K 2t, 2t + 1 (a0,
// a1) and 2t + 8, 2t + 9 (a2, a3), B column g at K 2t, 2t + 1 (b0) and 2t + 8,
// 2t + 9 (b1), and D rows g, g + 8, columns 2t, 2t + 1.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with a zero accumulator in.
__device__ __forceinline__ void mma16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

// Four 8 x 16-byte matrices: lane (g, t) gets word t of row g of matrix i in
// r[i]; lanes 8i .. 8i + 7 give the row addresses of matrix i.
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a)
                 : "memory");
}

// Two 8 x 16-byte matrices: lane (g, t) gets word t of row g of matrix i in
// r_i; lanes 8i .. 8i + 7 give the row addresses of matrix i.
__device__ __forceinline__ void ldsm_x2(uint32_t a, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(a)
                 : "memory");
}

// One arrival on an mbarrier (no transaction bytes).
__device__ __forceinline__ void mbar_arrive_m(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace mxk
