// prefill.cu -- large-batch MXFP4 product on the 5th-generation tensor cores
// (tcgen05 + TMEM, sm_103a).
//
// Y[t*rows + r] = sum_c W[r][c] * bf16(X[t][c]): the weights decoded exactly to
// bfloat16 (an E2M1 value times a power of two always fits), the activations
// rounded to nearest-even bfloat16 ("cortiq-engine 0.8.40
// src/gpu_wgpu/mxfp4.rs", GLOBAL fn mxg_bf16), products accumulated in FP32.
// This is the dense contraction of the prefill (many tokens share each weight;
// "rlx-cpu 0.2.17 src/gguf_matmul.rs" gguf_matmul_bt_cached: dequantise once,
// then a dense GEMM).
//
// One CTA computes a tile of 128 tokens (the MMA's M, operand A = bf16(X)) by
// 256 weight rows (N, operand B = decoded W), stepping K by 64 (one 128-byte
// swizzle atom of bf16).  All 16 warps produce: each k-step they load X (f32)
// and W (codes + scale bytes) for the next step into registers, convert the
// current step into bfloat16 tiles in shared memory (K-major, 128-byte
// swizzle), and thread 0 issues four tcgen05.mma (K = 16 each) into a 128 x 256
// FP32 accumulator in tensor memory; tcgen05.commit frees the stage when the
// MMAs have read it.  The epilogue reads the accumulator with tcgen05.ld and
// writes Y.  Every wait is bounded; a CTA that gives up sets the fault word,
// still frees its tensor memory and returns.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace mxk {
namespace {

constexpr int kPM = 128;            // tokens per tile (MMA M)
constexpr int kPN = 256;            // weight rows per tile (MMA N)
constexpr int kPK = 64;             // K per step (one 128-byte bf16 swizzle atom)
constexpr int kPStages = 3;
constexpr int kPThreads = 512;
constexpr int kAChunks = kPM * kPK / 8 / kPThreads;   // 16-byte bf16 chunks of A per thread
constexpr int kBChunks = kPN * kPK / 8 / kPThreads;   // and of B
constexpr uint32_t kATileBytes = kPM * kPK * 2;   // 16 KB
constexpr uint32_t kBTileBytes = kPN * kPK * 2;   // 32 KB
constexpr uint32_t kPStageBytes = kATileBytes + kBTileBytes;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kPWaitLimit = 1u << 24;

__device__ int g_fault_prefill;

// --- tcgen05 helpers ----------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);   // start address
    d |= static_cast<uint64_t>(1) << 16;                   // leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
    return d;
}

// Instruction descriptor: dense, D = F32, A = B = BF16, both K-major, N, M.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Two floats -> bf16x2, round to nearest even, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Raw inputs of one k-step held by one thread: kAChunks chunks of 8
// activations and kBChunks code words (8 weights each) with their scale bytes.
struct Raw {
    float4 x[kAChunks][2];
    uint32_t code[kBChunks];
    uint32_t sc[kBChunks];
};

__global__ void __launch_bounds__(kPThreads, 1) k_prefill(const uint8_t* __restrict__ w, int rows,
                                                          int cols, const float* __restrict__ X,
                                                          int nb, float* __restrict__ Y) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment of the tiles (the swizzle pattern repeats every 1024 B)
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bars[kPStages + 1];   // stage free, + accumulator done
    __shared__ uint32_t tmem_base;
    __shared__ int ok_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.x * kPN;      // weight rows of this tile
    const int t0 = blockIdx.y * kPM;      // tokens of this tile
    const int gpr = cols / kGroup;
    const int n_steps = (cols + kPK - 1) / kPK;
    const uint8_t* scales = w + static_cast<size_t>(rows) * cols / 2;

    if (warp == 0) tmem_alloc(&tmem_base, kTmemCols);
    if (tid == 0) {
        for (int i = 0; i <= kPStages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    auto load = [&](int s, Raw& raw) {
        const int k0 = s * kPK;
#pragma unroll
        for (int i = 0; i < kAChunks; ++i) {
            const int c = tid + kPThreads * i;
            const int m = c >> 3, j = c & 7;
            const int t = t0 + m, k = k0 + 8 * j;
            if (t < nb && k < cols) {
                const float4* src =
                    reinterpret_cast<const float4*>(X + static_cast<size_t>(t) * cols + k);
                raw.x[i][0] = __ldg(src);
                raw.x[i][1] = __ldg(src + 1);
            } else {
                raw.x[i][0] = make_float4(0.f, 0.f, 0.f, 0.f);
                raw.x[i][1] = raw.x[i][0];
            }
        }
#pragma unroll
        for (int i = 0; i < kBChunks; ++i) {
            const int c = tid + kPThreads * i;
            const int n = c >> 3, j = c & 7;
            const int r = r0 + n, g = 2 * s + (j >> 2);
            if (r < rows && g < gpr) {
                raw.code[i] = __ldg(reinterpret_cast<const uint32_t*>(
                                        w + (static_cast<size_t>(r) * gpr + g) * kGroupBytes) +
                                    (j & 3));
                raw.sc[i] = __ldg(scales + static_cast<size_t>(r) * gpr + g);
            } else {
                raw.code[i] = 0u;
                raw.sc[i] = 127u;   // 1.0 times code 0: an exact zero
            }
        }
    };
    auto store = [&](const Raw& raw, int st) {
        const uint32_t a_base = smem_u32(smem + st * kPStageBytes);
        const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
        for (int i = 0; i < kAChunks; ++i) {
            const int c = tid + kPThreads * i;
            const int m = c >> 3, j = c & 7;
            const float4 a = raw.x[i][0], b = raw.x[i][1];
            sts128(a_base + m * 128 + ((j ^ (m & 7)) << 4), pack_bf16x2(a.x, a.y),
                   pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
        }
#pragma unroll
        for (int i = 0; i < kBChunks; ++i) {
            const int c = tid + kPThreads * i;
            const int n = c >> 3, j = c & 7;
            const float s = e8m0_to_f32(raw.sc[i]);
            float v[8];
            e2m1x8_to_f32(raw.code[i], v);
            // value times a power of two: exact in float and in bfloat16
            sts128(b_base + n * 128 + ((j ^ (n & 7)) << 4),
                   pack_bf16x2(__fmul_rn(v[0], s), __fmul_rn(v[1], s)),
                   pack_bf16x2(__fmul_rn(v[2], s), __fmul_rn(v[3], s)),
                   pack_bf16x2(__fmul_rn(v[4], s), __fmul_rn(v[5], s)),
                   pack_bf16x2(__fmul_rn(v[6], s), __fmul_rn(v[7], s)));
        }
    };

    constexpr uint32_t idesc = idesc_bf16(kPM, kPN);
    bool ok = true;
    Raw A, B;
    load(0, A);
    for (int s = 0; s < n_steps; ++s) {
        Raw& cur = (s & 1) ? B : A;
        Raw& nxt = (s & 1) ? A : B;
        const int st = s % kPStages;
        if (s + 1 < n_steps) load(s + 1, nxt);
        // the stage is free once the MMAs of step s - kPStages have read it
        if (tid == 0) {
            ok_flag = s < kPStages ||
                      mbar_wait(&bars[st], static_cast<uint32_t>((s / kPStages - 1) & 1),
                                kPWaitLimit);
        }
        __syncthreads();
        if (!ok_flag) {
            ok = false;
            break;
        }
        store(cur, st);
        fence_proxy_async_smem();   // generic-proxy stores -> visible to the tensor core
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a_base = smem_u32(smem + st * kPStageBytes);
            const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
            for (int kk = 0; kk < kPK / 16; ++kk)
                umma_bf16(tmem, sw128_desc(a_base + kk * 32), sw128_desc(b_base + kk * 32), idesc,
                          (s > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&bars[st]);
            if (s == n_steps - 1) umma_commit(&bars[kPStages]);
        }
    }

    // epilogue: wait for the accumulator, then TMEM -> registers -> Y
    if (tid == 0) ok_flag = ok && mbar_wait(&bars[kPStages], 0u, kPWaitLimit);
    __syncthreads();
    if (ok_flag) {
        tc_fence_after();
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
        constexpr int kColsPerWarp = kPN / (kPThreads / 128);
        const int col0 = (warp >> 2) * kColsPerWarp;
        const int t = t0 + quarter * 32 + lane;
#pragma unroll 1
        for (int cc = 0; cc < kColsPerWarp; cc += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + col0 + cc, v);
            const int rbase = r0 + col0 + cc;
            if (t < nb) {
                float* dst = Y + static_cast<size_t>(t) * rows + rbase;
                if (rbase + 32 <= rows && (rows & 3) == 0) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + i) =
                            make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                        __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (rbase + i < rows) dst[i] = __uint_as_float(v[i]);
                }
            }
        }
    } else if (tid == 0) {
        atomicOr(&g_fault_prefill, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Version with the loads off the converting threads: warp 0 streams the raw
// tiles with TMA -- X as f32 (64 columns x 128 tokens), the codes (32 bytes x
// 256 rows) and, every 8 k-steps, the scale bytes of 16 groups (16 bytes x 256
// rows) -- into rings in shared memory; warps 2..15 convert a raw stage into
// the two bf16 operand tiles (128-byte swizzle) of a converted stage; warp 1
// issues the four tcgen05.mma of each converted stage and frees it with
// tcgen05.commit.  Needs cols % 512 == 0 (the scale plane's row stride is a
// multiple of 16 bytes) and 16-byte aligned X.
constexpr int kRawStages = 2;
constexpr int kConvStages = 2;
constexpr int kConvWarps = 14;
constexpr uint32_t kRawXBytes = kPM * kPK * 4;      // 32 KB f32
constexpr uint32_t kRawWBytes = kPN * kPK / 2;      // 8 KB codes
constexpr uint32_t kRawStageBytes = kRawXBytes + kRawWBytes;
constexpr uint32_t kScBlockBytes = kPN * 16;        // 16 groups x 256 rows
constexpr int kStepsPerSc = 8;                      // k-steps per scale block (2 groups each)

struct P2Layout {
    uint32_t conv, raw, sc, total;
};
__host__ __device__ constexpr P2Layout p2_layout() {
    return P2Layout{0, kConvStages * kPStageBytes,
                    kConvStages * kPStageBytes + kRawStages * kRawStageBytes,
                    kConvStages * kPStageBytes + kRawStages * kRawStageBytes + 2 * kScBlockBytes +
                        1024};
}

__device__ __forceinline__ void tma2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                      uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_p(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kPThreads, 1)
    k_prefill2(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
               const __grid_constant__ CUtensorMap smap, int rows, int cols, int nb,
               float* __restrict__ Y) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr P2Layout L = p2_layout();
    // raw_full/raw_free [kRawStages], conv_full/conv_free [kConvStages],
    // sc_full/sc_free [2], done
    __shared__ uint64_t bars[2 * kRawStages + 2 * kConvStages + 4 + 1];
    uint64_t* raw_full = bars;
    uint64_t* raw_free = raw_full + kRawStages;
    uint64_t* conv_full = raw_free + kRawStages;
    uint64_t* conv_free = conv_full + kConvStages;
    uint64_t* sc_full = conv_free + kConvStages;
    uint64_t* sc_free = sc_full + 2;
    uint64_t* done = sc_free + 2;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_word;
    volatile int* abort_flag = &abort_word;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.x * kPN;      // weight rows of this tile
    const int t0 = blockIdx.y * kPM;      // tokens of this tile
    const int n_steps = (cols + kPK - 1) / kPK;
    int issued_steps = 0, issued_blocks = 0;   // (producer) copies started

    if (warp == 0) tmem_alloc(&tmem_base, kTmemCols);
    if (tid == 0) {
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_free[i], kConvWarps);
        }
        for (int i = 0; i < kConvStages; ++i) {
            mbar_init(&conv_full[i], kConvWarps);
            mbar_init(&conv_free[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sc_full[i], 1);
            mbar_init(&sc_free[i], kConvWarps);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_fault_prefill, 1);
    };

    if (warp == 0) {
        // --- TMA producer
        if (lane == 0) {
            const uint64_t policy = l2_evict_first();
            for (int s = 0; s < n_steps && !*abort_flag; ++s) {
                const int rs = s % kRawStages;
                if (s >= kRawStages &&
                    !mbar_wait(&raw_free[rs], static_cast<uint32_t>(s / kRawStages - 1) & 1u,
                               kPWaitLimit)) {
                    fail();
                    break;
                }
                if (s % kStepsPerSc == 0) {   // a new block of scale bytes
                    const int b = s / kStepsPerSc, sb = b & 1;
                    if (b >= 2 && !mbar_wait(&sc_free[sb], static_cast<uint32_t>(b / 2 - 1) & 1u,
                                             kPWaitLimit)) {
                        fail();
                        break;
                    }
                    mbar_arrive_expect_tx(&sc_full[sb], kScBlockBytes);
                    tma2d(smem_u32(smem + L.sc + sb * kScBlockBytes), &smap, b * 16, r0,
                          &sc_full[sb], policy);
                    issued_blocks = b + 1;
                }
                const uint32_t raw = smem_u32(smem + L.raw + rs * kRawStageBytes);
                mbar_arrive_expect_tx(&raw_full[rs], kRawStageBytes);
                tma2d(raw, &xmap, s * kPK, t0, &raw_full[rs], policy);
                tma2d(raw + kRawXBytes, &wmap, s * (kPK / 2), r0, &raw_full[rs], policy);
                issued_steps = s + 1;
            }
        }
    } else if (warp == 1) {
        // --- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kPM, kPN);
            for (int s = 0; s < n_steps && !*abort_flag; ++s) {
                const int cs = s % kConvStages;
                if (!mbar_wait(&conv_full[cs], static_cast<uint32_t>(s / kConvStages) & 1u,
                               kPWaitLimit)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_u32(smem + L.conv + cs * kPStageBytes);
                const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
                for (int kk = 0; kk < kPK / 16; ++kk)
                    umma_bf16(tmem, sw128_desc(a_base + kk * 32), sw128_desc(b_base + kk * 32),
                              idesc, (s > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&conv_free[cs]);
                if (s == n_steps - 1) umma_commit(done);
            }
        }
    } else {
        // --- converters: raw stage -> bf16 operand tiles
        const int ct = tid - 64;   // 0 .. kConvWarps * 32 - 1
        constexpr int kCT = kConvWarps * 32;
        for (int s = 0; s < n_steps && !*abort_flag; ++s) {
            const int rs = s % kRawStages, cs = s % kConvStages, sb = (s / kStepsPerSc) & 1;
            bool ok = mbar_wait(&raw_full[rs], static_cast<uint32_t>(s / kRawStages) & 1u,
                                kPWaitLimit);
            ok = ok && mbar_wait(&sc_full[sb], static_cast<uint32_t>(s / (2 * kStepsPerSc)) & 1u,
                                 kPWaitLimit);
            ok = ok && (s < kConvStages ||
                        mbar_wait(&conv_free[cs], static_cast<uint32_t>(s / kConvStages - 1) & 1u,
                                  kPWaitLimit));
            if (!ok) {
                fail();
                break;
            }
            const uint8_t* raw = smem + L.raw + rs * kRawStageBytes;
            const uint8_t* scb = smem + L.sc + sb * kScBlockBytes;
            const uint32_t a_base = smem_u32(smem + L.conv + cs * kPStageBytes);
            const uint32_t b_base = a_base + kATileBytes;
            // A: 1024 chunks (token m, 8 columns j) of f32 -> bf16
            for (int c = ct; c < kPM * kPK / 8; c += kCT) {
                const int m = c >> 3, j = c & 7;
                const float4* src = reinterpret_cast<const float4*>(raw + (m * kPK + 8 * j) * 4);
                const float4 a = src[0], b = src[1];
                sts128(a_base + m * 128 + ((j ^ (m & 7)) << 4), pack_bf16x2(a.x, a.y),
                       pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
            }
            // B: 2048 chunks (row n, code word j) -> 8 decoded weights in bf16
            for (int c = ct; c < kPN * kPK / 8; c += kCT) {
                const int n = c >> 3, j = c & 7;
                const uint32_t code =
                    *reinterpret_cast<const uint32_t*>(raw + kRawXBytes + n * (kPK / 2) + 4 * j);
                const float sc = e8m0_to_f32(scb[n * 16 + (s % kStepsPerSc) * 2 + (j >> 2)]);
                float v[8];
                e2m1x8_to_f32(code, v);
                // a value times a power of two: exact in float and in bfloat16
                sts128(b_base + n * 128 + ((j ^ (n & 7)) << 4),
                       pack_bf16x2(__fmul_rn(v[0], sc), __fmul_rn(v[1], sc)),
                       pack_bf16x2(__fmul_rn(v[2], sc), __fmul_rn(v[3], sc)),
                       pack_bf16x2(__fmul_rn(v[4], sc), __fmul_rn(v[5], sc)),
                       pack_bf16x2(__fmul_rn(v[6], sc), __fmul_rn(v[7], sc)));
            }
            fence_proxy_async_smem();   // generic-proxy stores -> visible to the tensor core
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_p(&raw_free[rs]);
                mbar_arrive_p(&conv_full[cs]);
                if (s % kStepsPerSc == kStepsPerSc - 1 || s == n_steps - 1) mbar_arrive_p(&sc_free[sb]);
            }
        }
    }

    // --- epilogue: wait for the accumulator, then TMEM -> registers -> Y
    __syncthreads();
    if (tid == 0 && !*abort_flag && !mbar_wait(done, 0u, kPWaitLimit)) fail();
    __syncthreads();
    if (!*abort_flag) {
        tc_fence_after();
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
        constexpr int kColsPerWarp = kPN / (kPThreads / 128);
        const int col0 = (warp >> 2) * kColsPerWarp;
        const int t = t0 + quarter * 32 + lane;
#pragma unroll 1
        for (int cc = 0; cc < kColsPerWarp; cc += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + col0 + cc, v);
            const int rbase = r0 + col0 + cc;
            if (t < nb) {
                float* dst = Y + static_cast<size_t>(t) * rows + rbase;
                if (rbase + 32 <= rows && (rows & 3) == 0) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + i) =
                            make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                        __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (rbase + i < rows) dst[i] = __uint_as_float(v[i]);
                }
            }
        }
    } else {
        // a CTA that gave up: let every copy it started land before it exits
        // (thread 0 is the producer; waits on completed phases return at once)
        if (tid == 0) {
            for (int i = issued_steps - kRawStages; i < issued_steps; ++i)
                if (i >= 0)
                    mbar_wait(&raw_full[i % kRawStages],
                              static_cast<uint32_t>(i / kRawStages) & 1u, kPWaitLimit);
            for (int b = issued_blocks - 2; b < issued_blocks; ++b)
                if (b >= 0)
                    mbar_wait(&sc_full[b & 1], static_cast<uint32_t>(b / 2) & 1u, kPWaitLimit);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_p() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool map2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner,
           uint64_t outer, uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn_p();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

cudaError_t launch_prefill2(const uint8_t* w, int rows, int cols, const float* X, int nb,
                            float* Y, cudaStream_t s) {
    const int gpr = cols / kGroup;
    if (gpr % 16 != 0 || (reinterpret_cast<uintptr_t>(X) & 15) != 0) return cudaErrorNotSupported;
    CUtensorMap xmap, wmap, smap;
    const uint8_t* scales = w + static_cast<size_t>(rows) * cols / 2;
    if (!map2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, X, cols, nb,
               static_cast<uint64_t>(cols) * 4, kPK, kPM) ||
        !map2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, cols / 2, rows, cols / 2, kPK / 2, kPN) ||
        !map2d(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, scales, gpr, rows, gpr, 16, kPN))
        return cudaErrorNotSupported;
    constexpr P2Layout l = p2_layout();
    static PerDevice memo;
    const cudaError_t attr_err = static_cast<cudaError_t>(memo.get([] {
        return static_cast<int>(cudaFuncSetAttribute(
            k_prefill2, cudaFuncAttributeMaxDynamicSharedMemorySize,
            static_cast<int>(p2_layout().total)));
    }));
    if (attr_err != cudaSuccess) return attr_err;
    const dim3 grid((rows + kPN - 1) / kPN, (nb + kPM - 1) / kPM);
    k_prefill2<<<grid, kPThreads, l.total, s>>>(xmap, wmap, smap, rows, cols, nb, Y);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Dense after dequant ("rlx-cpu 0.2.17 src/gguf_matmul.rs" gguf_matmul_bt_cached:
// dequantise once, then a dense GEMM): W is decoded to bfloat16 and X rounded
// to bfloat16 into a caller's workspace by two elementwise kernels, then a
// plain tcgen05 GEMM streams both operands with TMA (128-byte swizzle, the
// layout the MMA descriptors read) through a 4-stage ring; warp 0 issues the
// copies, warp 1 the MMAs, every warp reads the accumulator back.

// Both operands of the dense product in one launch: items [0, nw) are code
// words of W (8 elements, exact in bfloat16: E2M1 value times E8M0 scale), items
// [nw, nw + nx4) are four activations of X, rounded to nearest-even bfloat16.
__global__ void __launch_bounds__(256) k_to_bf16(const uint8_t* __restrict__ w, int rows, int cols,
                                                 uint4* __restrict__ wout,
                                                 const float4* __restrict__ x, size_t nx4,
                                                 uint2* __restrict__ xout) {
    // the GEMM may launch now and set itself up; it reads these outputs only
    // after this grid has completed (griddepcontrol.wait)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int wpr = cols / 8;   // code words per row
    const int gpr = cols / kGroup;
    const size_t nw = static_cast<size_t>(rows) * wpr;
    const uint8_t* scales = w + static_cast<size_t>(rows) * cols / 2;
    const uint32_t* words = reinterpret_cast<const uint32_t*>(w);
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nw + nx4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        if (i < nw) {
            const size_t r = i / wpr;
            const int q = static_cast<int>(i - r * wpr);
            const float sc = e8m0_to_f32(__ldg(scales + r * gpr + q / 4));
            float v[8];
            e2m1x8_to_f32(__ldg(words + i), v);
            wout[i] = make_uint4(pack_bf16x2(__fmul_rn(v[0], sc), __fmul_rn(v[1], sc)),
                                 pack_bf16x2(__fmul_rn(v[2], sc), __fmul_rn(v[3], sc)),
                                 pack_bf16x2(__fmul_rn(v[4], sc), __fmul_rn(v[5], sc)),
                                 pack_bf16x2(__fmul_rn(v[6], sc), __fmul_rn(v[7], sc)));
        } else {
            const float4 a = __ldg(x + (i - nw));
            xout[i - nw] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
        }
    }
}

constexpr int kGStages = 4;

__device__ __forceinline__ void tma2d_g(uint32_t dst, const CUtensorMap* map, int x, int y,
                                        uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_g(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Persistent: CTA c takes tiles c, c + grid, ... (tile = TN weight rows x 128
// tokens, token tiles fastest).  Warp 0 streams both operands of every tile
// through the stage ring, warp 1 issues the MMAs into one of two 256-column
// TMEM accumulators (tile j into j % 2), and warps 8..15 read a finished
// accumulator back and store it while the next tile's MMAs run.
constexpr int kEpiWarp0 = 8;                       // first epilogue warp
constexpr int kEpiWarps = kPThreads / 32 - kEpiWarp0;   // 8: two per TMEM lane quarter

template <int TN>
__global__ void __launch_bounds__(kPThreads, 1)
    k_gemm_bf16(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                int rows, int cols, int nb, float* __restrict__ Y) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t full[kGStages], empty[kGStages], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_word;
    volatile int* abort_flag = &abort_word;
    constexpr uint32_t kBBytes = TN * kPK * 2, kStage = kATileBytes + kBBytes;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int n_steps = (cols + kPK - 1) / kPK;
    const int n_tt = (nb + kPM - 1) / kPM;
    const int n_tiles = (rows + TN - 1) / TN * n_tt;
    int issued = 0;   // (producer) stages started, over all tiles

    if (warp == 0) tmem_alloc(&tmem_base, 2 * kTmemCols);
    if (tid == 0) {
        for (int i = 0; i < kGStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kEpiWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // the operands are written by the conversion launch before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_fault_prefill, 1);
    };

    if (warp == 0 && lane == 0) {
        // --- TMA producer: A tile (128 tokens x 64) and B tile (TN rows x 64)
        uint64_t policy;   // every tile is read by many CTAs: keep both operands in L2
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
        for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
            const int r0 = (tile / n_tt) * TN, t0 = (tile % n_tt) * kPM;
            for (int s = 0; s < n_steps && !*abort_flag; ++s, ++issued) {
                const int st = issued % kGStages;
                if (issued >= kGStages &&
                    !mbar_wait(&empty[st], static_cast<uint32_t>(issued / kGStages - 1) & 1u,
                               kPWaitLimit)) {
                    fail();
                    break;
                }
                const uint32_t a = smem_u32(smem + st * kStage);
                mbar_arrive_expect_tx(&full[st], kStage);
                tma2d_g(a, &amap, s * kPK, t0, &full[st], policy);
                tma2d_g(a + kATileBytes, &bmap, s * kPK, r0, &full[st], policy);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // --- MMA issuer
        constexpr uint32_t idesc = idesc_bf16(kPM, TN);
        int used = 0;   // stages consumed, over all tiles
        int j = 0;      // this CTA's tile count
        for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x, ++j) {
            const int ab = j & 1;
            if (j >= 2 && !mbar_wait(&acc_empty[ab], static_cast<uint32_t>((j >> 1) - 1) & 1u,
                                     kPWaitLimit)) {
                fail();
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + ab * kTmemCols;
            for (int s = 0; s < n_steps; ++s, ++used) {
                const int st = used % kGStages;
                if (!mbar_wait(&full[st], static_cast<uint32_t>(used / kGStages) & 1u,
                               kPWaitLimit)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_u32(smem + st * kStage);
                const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
                for (int kk = 0; kk < kPK / 16; ++kk)
                    umma_bf16(d, sw128_desc(a_base + kk * 32), sw128_desc(b_base + kk * 32), idesc,
                              (s > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&empty[st]);
            }
            if (*abort_flag) break;
            umma_commit(&acc_full[ab]);
        }
    } else if (warp >= kEpiWarp0) {
        // --- epilogue: accumulator j % 2 -> Y, then hand it back
        const int ew = warp - kEpiWarp0;
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int half = ew >> 2;                // columns half*TN/2 ..
        constexpr int kCols = TN / 2;            // 128 or 112
        int j = 0;
        for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x, ++j) {
            const int ab = j & 1;
            if (!mbar_wait(&acc_full[ab], static_cast<uint32_t>(j >> 1) & 1u, kPWaitLimit)) {
                fail();
                break;
            }
            tc_fence_after();
            const int r0 = (tile / n_tt) * TN, t0 = (tile % n_tt) * kPM;
            const int t = t0 + quarter * 32 + lane;
            const uint32_t src = tmem + ab * kTmemCols + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 half * kCols;
#pragma unroll 1
            for (int cc = 0; cc < kCols; cc += 8) {
                uint32_t v[8];
                tmem_ld8(src + cc, v);
                const int rbase = r0 + half * kCols + cc;
                if (t < nb) {
                    float* dst = Y + static_cast<size_t>(t) * rows + rbase;
                    if (rbase + 8 <= rows && (rows & 3) == 0) {
                        *reinterpret_cast<float4*>(dst) =
                            make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]),
                                        __uint_as_float(v[2]), __uint_as_float(v[3]));
                        *reinterpret_cast<float4*>(dst + 4) =
                            make_float4(__uint_as_float(v[4]), __uint_as_float(v[5]),
                                        __uint_as_float(v[6]), __uint_as_float(v[7]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (rbase + i < rows) dst[i] = __uint_as_float(v[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_g(&acc_empty[ab]);
        }
    }

    __syncthreads();
    if (*abort_flag && tid == 0) {
        // a CTA that gave up: let the copies it started land before it exits
        for (int i = issued - kGStages; i < issued; ++i)
            if (i >= 0)
                mbar_wait(&full[i % kGStages], static_cast<uint32_t>(i / kGStages) & 1u,
                          kPWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_g() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A [outer][inner] bf16 matrix as a 2-D tensor map, tiles of 64 x box_outer
// elements (128-byte rows, 128-byte swizzle).
bool bf16_map(CUtensorMap* map, const void* base, int inner, int outer, uint32_t box_outer) {
    auto fn = encode_fn_g();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
    const cuuint32_t box[2] = {kPK, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

int grid_for(size_t n, int per_thread_items) {
    const size_t blocks = (n / per_thread_items + 255) / 256;
    return static_cast<int>(blocks < 4096 ? (blocks > 0 ? blocks : 1) : 4096);
}

}  // namespace

cudaError_t launch_mm_tcgen05(const uint8_t* w, int rows, int cols, const float* X, int nb,
                              float* Y, cudaStream_t s) {
    {
        const cudaError_t e2 = launch_prefill2(w, rows, cols, X, nb, Y, s);
        if (e2 != cudaErrorNotSupported) return e2;
        (void)cudaGetLastError();
    }
    const size_t smem = static_cast<size_t>(kPStages) * kPStageBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(k_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid((rows + kPN - 1) / kPN, (nb + kPM - 1) / kPM);
    k_prefill<<<grid, kPThreads, smem, s>>>(w, rows, cols, X, nb, Y);
    return cudaGetLastError();
}

size_t dense_ws_bytes(int rows, int cols, int nb) {
    const size_t wb = (static_cast<size_t>(rows) * cols * 2 + 255) / 256 * 256;
    return wb + static_cast<size_t>(nb) * cols * 2;
}

cudaError_t launch_mm_dense(const uint8_t* w, int rows, int cols, const float* X, int nb,
                            float* Y, void* ws, cudaStream_t s) {
    uint8_t* wb = static_cast<uint8_t*>(ws);
    uint8_t* xb = wb + (static_cast<size_t>(rows) * cols * 2 + 255) / 256 * 256;
    // weight rows per tile: 256, or 224 when that fills whole waves better
    // (rounds of tiles over the SMs x rows per tile)
    const int n_tt = (nb + kPM - 1) / kPM;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 1;
    auto tiles_of = [&](int tn) { return static_cast<long>((rows + tn - 1) / tn) * n_tt; };
    auto cost = [&](int tn) { return (tiles_of(tn) + sms - 1) / sms * tn; };
    const int tn = cost(224) < cost(256) ? 224 : 256;
    CUtensorMap amap, bmap;
    if (!bf16_map(&amap, xb, cols, nb, kPM) || !bf16_map(&bmap, wb, cols, rows, tn))
        return cudaErrorNotSupported;
    const size_t nw = static_cast<size_t>(rows) * cols / 8;
    const size_t nx4 = static_cast<size_t>(nb) * cols / 4;
    k_to_bf16<<<grid_for(nw + nx4, 4), 256, 0, s>>>(w, rows, cols, reinterpret_cast<uint4*>(wb),
                                                    reinterpret_cast<const float4*>(X), nx4,
                                                    reinterpret_cast<uint2*>(xb));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    static PerDevice memo;
    const size_t smem = static_cast<size_t>(kGStages) * kPStageBytes + 1024;   // (tn <= 256)
    const cudaError_t attr_err = static_cast<cudaError_t>(memo.get([smem] {
        cudaError_t a = cudaFuncSetAttribute(k_gemm_bf16<256>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (a == cudaSuccess)
            a = cudaFuncSetAttribute(k_gemm_bf16<224>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
        return static_cast<int>(a);
    }));
    if (attr_err != cudaSuccess) return attr_err;
    const long tiles = tiles_of(tn);
    const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);
    // programmatic dependent launch: set-up (barriers, TMEM) under the
    // conversion's tail, the first copy after it has completed
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t el =
        tn == 224 ? cudaLaunchKernelEx(&cfg, k_gemm_bf16<224>, amap, bmap, rows, cols, nb, Y)
                  : cudaLaunchKernelEx(&cfg, k_gemm_bf16<256>, amap, bmap, rows, cols, nb, Y);
    if (el != cudaSuccess) return el;
    return cudaGetLastError();
}

cudaError_t read_fault_prefill(int* value, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_fault_prefill, sizeof(int));
    if (e != cudaSuccess || !reset) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_prefill, &zero, sizeof(int));
}

}  // namespace mxk
