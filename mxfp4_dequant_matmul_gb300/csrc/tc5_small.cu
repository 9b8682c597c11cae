// tc5_small.cu -- small-batch MXFP4 product on the 5th-generation tensor cores,
// with the decoded weights as the tensor-memory operand (sm_103a).
//
// Y[t*rows + r] = sum_c W[r][c] X[t][c] for up to 8 tokens per pass
// ("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs", PEROP kernel mxfp4_mm: one
// decode of each weight group serves every token of the pass).
//
// A CTA takes a tile of 128 weight rows and a slice of the groups (the K
// dimension; the CTAs of a thread-block cluster split the groups and add their
// partial sums through distributed shared memory).  Per group (32 elements):
//   * a decoder warp per 32-row quarter reads its rows' 16 code bytes from a
//     TMA-filled shared-memory stage, converts the E2M1 codes to f16 (exact,
//     the hardware pair conversion) and stores them with tcgen05.st as the A
//     operand (128 rows x K = 32) of the group's slot in tensor memory;
//   * one thread issues two tcgen05.mma (M = 128, N = 16, K = 16) with that A
//     and, as B, the activations of the pass from shared memory: column n < 8
//     is token n's hi half, column 8 + n its lo half (hi = f16(x 2^p),
//     lo = f16(x 2^p - hi), one power of two p per token for the CTA's slice);
//     every product is exact and the accumulator is FP32;
//   * an epilogue warp per quarter reads the 16 accumulator columns back with
//     tcgen05.ld, and adds scale * (hi + lo) to each token's FP32 row sum.
// Eight slots (A + accumulator) rotate through tensor memory so that decode,
// MMA and epilogue of different groups overlap; mbarriers order them, and every
// wait is bounded.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace mxk {
namespace {

constexpr int kRowsT = 128;                 // rows per tile (MMA M)
constexpr int kNT = 16;                     // MMA N: 8 tokens x (hi, lo)
constexpr int kTok = 8;                     // tokens per pass
constexpr int kStageGroups = 8;             // groups per code stage (128 bytes per row)
constexpr int kStages5 = 4;                 // code stages
constexpr int kStageBytes5 = kRowsT * 128;  // 16 KB
constexpr int kSlots = 8;                   // (A, accumulator) slots in tensor memory
constexpr int kSlotCols = 32;               // A: 16 columns (K = 32 f16), D: 16 columns
constexpr uint32_t kTmemCols5 = kSlots * kSlotCols;   // 256
constexpr int kWarps5 = 10;                 // 0-3 decode, 4-7 epilogue, 8 TMA, 9 MMA
constexpr int kThreads5 = kWarps5 * 32;
constexpr uint32_t kWait5 = 1u << 24;

__device__ int g_fault_tc5;

// --- PTX helpers ---------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc5(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc5(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tcf_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tcf_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major operand in shared memory, 128-byte swizzle, 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t sw128_desc5(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor: D = F32, A = B = F16, K-major, N = 16, M = 128.
constexpr uint32_t kIdescF16 = (1u << 4) | (static_cast<uint32_t>(kNT >> 3) << 17) |
                               (static_cast<uint32_t>(kRowsT >> 4) << 24);

// D (tensor memory) += A (tensor memory) x B (shared memory).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(kIdescF16), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit5(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive5(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank5() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync5() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
__device__ __forceinline__ float ld_cluster5(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ float exp2i5(int e) {
    if (e >= -126 && e <= 127) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    if (e > 127) return __uint_as_float(0x7F800000u);
    if (e >= -149) return __uint_as_float(1u << (e + 149));
    return 0.0f;
}
__device__ __forceinline__ float scale2_5(float x, int p) {
    const int p1 = p / 2, p2 = p - p1;
    return __fmul_rn(__fmul_rn(x, exp2i5(p1)), exp2i5(p2));
}
__device__ __forceinline__ uint32_t pack_f16x2_5(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Shared memory layout (offsets from a 1024-byte aligned base).
struct T5Layout {
    uint32_t btile, stages, sc, sc_pitch, part, bars, misc, total;
};
__host__ __device__ inline T5Layout t5_layout(int ng) {
    T5Layout l;
    l.btile = 0;                                                   // [ceil(ng/2)][2 KB]
    l.stages = l.btile + static_cast<uint32_t>((ng + 1) / 2) * 2048;
    l.stages = (l.stages + 1023u) & ~1023u;
    l.sc = l.stages + kStages5 * kStageBytes5;                      // [128][sc_pitch]
    l.sc_pitch = (static_cast<uint32_t>(ng) + 15u) & ~15u;
    l.part = l.sc + kRowsT * l.sc_pitch;                           // [128][8] f32
    l.part = (l.part + 15u) & ~15u;
    l.bars = l.part + kRowsT * kTok * 4;                           // mbarriers
    l.bars = (l.bars + 7u) & ~7u;
    l.misc = l.bars + (2 * kStages5 + 3 * kSlots) * 8;             // tmem addr, flags, p
    l.total = l.misc + 128 + 1024;                                 // + alignment slack
    return l;
}

template <int CL>
__global__ void __launch_bounds__(kThreads5, 1)
    k_tc5_small(const __grid_constant__ CUtensorMap tmap, const uint8_t* __restrict__ w, int rows,
                int cols, const float* __restrict__ X, int nb, float* __restrict__ Y, int max_ng) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const T5Layout L = t5_layout(max_ng);
    uint8_t* btile = smem + L.btile;
    uint8_t* stages = smem + L.stages;
    uint8_t* sc_s = smem + L.sc;
    float* part = reinterpret_cast<float*>(smem + L.part);
    uint64_t* code_full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* code_free = code_full + kStages5;
    uint64_t* a_full = code_free + kStages5;
    uint64_t* d_full = a_full + kSlots;
    uint64_t* slot_free = d_full + kSlots;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
    int* pexp = reinterpret_cast<int*>(smem + L.misc + 8);             // [8] per-token 2^p
    unsigned* tmax = reinterpret_cast<unsigned*>(smem + L.misc + 40);  // [8] max |x| bits

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = CL > 1 ? cluster_rank5() : 0u;
    const int tile = blockIdx.x / CL;
    const int row0 = tile * kRowsT;
    const int t0 = blockIdx.y * kTok;
    const int nbt = min(kTok, nb - t0);
    const int gpr = cols / kGroup;
    const int g_lo = static_cast<int>(static_cast<long>(rank) * gpr / CL);
    const int g_hi = static_cast<int>(static_cast<long>(rank + 1) * gpr / CL);
    const int ng = g_hi - g_lo;
    const int n_st = (ng + kStageGroups - 1) / kStageGroups;
    const size_t plane = static_cast<size_t>(rows) * cols / 2;

    // --- set-up: barriers, tensor memory, first code stages
    if (tid == 0) {
        for (int i = 0; i < kStages5; ++i) {
            mbar_init(&code_full[i], 1);
            mbar_init(&code_free[i], 4);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&a_full[i], 4);
            mbar_init(&d_full[i], 1);
            mbar_init(&slot_free[i], 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (tid < kTok) tmax[tid] = 0u;
    if (warp == 0) tmem_alloc5(tmem_slot, kTmemCols5);
    tcf_before();
    __syncthreads();
    tcf_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t policy = l2_evict_first();

    auto issue_stage = [&](int s) {   // one TMA tile: 128 rows x 128 code bytes
        const int st = s % kStages5;
        mbar_arrive_expect_tx(&code_full[st], kStageBytes5);
        const int x = (g_lo + s * kStageGroups) * kGroupBytes;
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
                smem_u32(stages + st * kStageBytes5)),
            "l"(&tmap), "r"(x), "r"(row0), "r"(smem_u32(&code_full[st])), "l"(policy)
            : "memory");
    };
    if (warp == 8 && lane == 0)
        for (int s = 0; s < kStages5 && s < n_st; ++s) issue_stage(s);

    // --- scale bytes of the tile's rows and this CTA's groups
    {
        const int nrow = min(kRowsT, rows - row0);
        for (int base = tid; base < nrow * ng; base += 8 * kThreads5) {
            uint32_t v[8];
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
                const int i = base + k8 * kThreads5;
                v[k8] = 0u;
                if (i < nrow * ng) {
                    const int r = i / ng, j = i - r * ng;
                    v[k8] = __ldg(w + plane + static_cast<size_t>(row0 + r) * gpr + g_lo + j);
                }
            }
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
                const int i = base + k8 * kThreads5;
                if (i < nrow * ng) {
                    const int r = i / ng, j = i - r * ng;
                    sc_s[r * L.sc_pitch + j] = static_cast<uint8_t>(v[k8]);
                }
            }
        }
    }

    // --- activations: per-token largest |x| over this CTA's slice, then the B
    // tiles.  B tile for group pair g2: rows n (n < 8: token n hi, else token
    // n - 8 lo), 64 f16 per row (group 2*g2 then 2*g2 + 1), 128-byte swizzle.
    for (int i = tid; i < kTok * ng * 8; i += kThreads5) {
        const int t = i / (ng * 8), rem = i - t * ng * 8;
        float m = 0.0f;
        if (t < nbt) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(
                X + static_cast<size_t>(t0 + t) * cols + static_cast<size_t>(g_lo) * kGroup) + rem);
            m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        }
        if (m > 0.0f && m <= 3.402823466e38f) atomicMax(&tmax[t], __float_as_uint(m));
    }
    __syncthreads();
    if (tid < kTok) {
        const float m = __uint_as_float(tmax[tid]);
        // puts the token's largest |x| in [2^14, 2^15); capped so 2^-p stays normal
        pexp[tid] = m > 0.0f ? min(14 - ilogbf(m), 126) : 0;
    }
    __syncthreads();
    for (int i = tid; i < ((ng + 1) / 2) * kTok * 8; i += kThreads5) {
        // one 16-byte chunk c of token t in pair g2: elements 8*(c%4) .. of group 2*g2 + c/4
        const int g2 = i / (kTok * 8), rem = i - g2 * kTok * 8;
        const int t = rem >> 3, c = rem & 7;
        const int g = 2 * g2 + (c >> 2);
        float v[8];
        if (t < nbt && g < ng) {
            const float4* src = reinterpret_cast<const float4*>(
                X + static_cast<size_t>(t0 + t) * cols + static_cast<size_t>(g_lo + g) * kGroup +
                8 * (c & 3));
            const float4 a = __ldg(src), b = __ldg(src + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = 0.0f;
        }
        const int p = pexp[t];
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a0 = scale2_5(v[2 * k], p), a1 = scale2_5(v[2 * k + 1], p);
            hi[k] = pack_f16x2_5(a0, a1);
            const float h0 = __half2float(__ushort_as_half(static_cast<unsigned short>(hi[k] & 0xFFFFu)));
            const float h1 = __half2float(__ushort_as_half(static_cast<unsigned short>(hi[k] >> 16)));
            lo[k] = pack_f16x2_5(__fsub_rn(a0, h0), __fsub_rn(a1, h1));
        }
        uint8_t* tb = btile + g2 * 2048;
        const int rh = t, rl = t + 8;
        *reinterpret_cast<uint4*>(tb + rh * 128 + ((c ^ (rh & 7)) << 4)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(tb + rl * 128 + ((c ^ (rl & 7)) << 4)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    fence_proxy_async_smem();   // B tiles (generic stores) -> tensor-core reads
    tcf_before();
    __syncthreads();
    tcf_after();

    // --- roles
    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_fault_tc5, 1);
    };
    if (warp < 4) {
        // decoder for rows 32*warp .. +31
        const int q = warp;
        const int r = q * 32 + lane;
        for (int j = 0; j < ng && !*abort_flag; ++j) {
            const int s = j / kStageGroups, st = s % kStages5, jj = j % kStageGroups;
            if (jj == 0 && !mbar_wait(&code_full[st], static_cast<uint32_t>(s / kStages5) & 1u, kWait5)) {
                fail();
                break;
            }
            const int slot = j % kSlots;
            if (j >= kSlots &&
                !mbar_wait(&slot_free[slot], static_cast<uint32_t>(j / kSlots - 1) & 1u, kWait5)) {
                fail();
                break;
            }
            const uint4 code = *reinterpret_cast<const uint4*>(stages + st * kStageBytes5 + r * 128 +
                                                               ((jj ^ (r & 7)) << 4));
            uint32_t a[16];
            const uint32_t words[4] = {code.x, code.y, code.z, code.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t h[4];
                e2m1x8_to_f16x2x4(words[k], h);
                a[4 * k] = h[0];
                a[4 * k + 1] = h[1];
                a[4 * k + 2] = h[2];
                a[4 * k + 3] = h[3];
            }
            tmem_st16(tmem + (static_cast<uint32_t>(q * 32) << 16) + slot * kSlotCols, a);
            tcf_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive5(&a_full[slot]);
                if (jj == kStageGroups - 1 || j == ng - 1) mbar_arrive5(&code_free[st]);
            }
        }
    } else if (warp < 8) {
        // epilogue for rows 32*(warp-4) .. +31
        const int q = warp - 4;
        const int r = q * 32 + lane;
        float acc[kTok];
#pragma unroll
        for (int t = 0; t < kTok; ++t) acc[t] = 0.0f;
        for (int j = 0; j < ng && !*abort_flag; ++j) {
            const int slot = j % kSlots;
            if (!mbar_wait(&d_full[slot], static_cast<uint32_t>(j / kSlots) & 1u, kWait5)) {
                fail();
                break;
            }
            tcf_after();
            uint32_t d[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + slot * kSlotCols + 16, d);
            tcf_before();
            __syncwarp();
            if (lane == 0) mbar_arrive5(&slot_free[slot]);
            const float s = e8m0_to_f32(sc_s[r * L.sc_pitch + j]);
#pragma unroll
            for (int t = 0; t < kTok; ++t)
                acc[t] = __fmaf_rn(s, __fadd_rn(__uint_as_float(d[t]), __uint_as_float(d[t + 8])),
                                   acc[t]);
        }
#pragma unroll
        for (int t = 0; t < kTok; ++t) part[r * kTok + t] = __fmul_rn(acc[t], exp2i5(-pexp[t]));
    } else if (warp == 8) {
        // TMA producer: refill each code stage once its 4 decoders are done
        if (lane == 0) {
            for (int s = kStages5; s < n_st && !*abort_flag; ++s) {
                const int st = s % kStages5;
                if (!mbar_wait(&code_free[st], static_cast<uint32_t>(s / kStages5 - 1) & 1u, kWait5)) {
                    fail();
                    break;
                }
                issue_stage(s);
            }
        }
    } else {
        // MMA issuer
        if (lane == 0) {
            for (int j = 0; j < ng && !*abort_flag; ++j) {
                const int slot = j % kSlots;
                if (!mbar_wait(&a_full[slot], static_cast<uint32_t>(j / kSlots) & 1u, kWait5)) {
                    fail();
                    break;
                }
                tcf_after();
                const uint32_t bbase = smem_u32(btile + (j >> 1) * 2048) + (j & 1) * 64;
                const uint32_t a_col = tmem + slot * kSlotCols;
                const uint32_t d_col = a_col + 16;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    umma_ts(d_col, a_col + kk * 8, sw128_desc5(bbase + kk * 32), kk);
                umma_commit5(&d_full[slot]);
            }
        }
    }
    tcf_before();
    __syncthreads();

    // --- add the cluster's partial sums (rank order); CTA k writes its share of rows
    if (CL > 1) cluster_sync5();
    {
        const int r_lo = static_cast<int>(rank) * kRowsT / CL;
        const int r_hi = static_cast<int>(rank + 1) * kRowsT / CL;
        for (int i = r_lo * kTok + tid; i < r_hi * kTok; i += kThreads5) {
            const int lr = i / kTok, t = i - lr * kTok;
            float s = part[i];
            if (CL > 1) {
                s = ld_cluster5(part + i, 0);
                for (uint32_t k = 1; k < static_cast<uint32_t>(CL); ++k)
                    s = __fadd_rn(s, ld_cluster5(part + i, k));
            }
            const int row = row0 + lr;
            if (row < rows && t < nbt && !*abort_flag)
                Y[static_cast<size_t>(t0 + t) * rows + row] = s;
        }
    }
    if (CL > 1) cluster_sync5();
    if (warp == 0) {
        tcf_after();
        tmem_dealloc5(tmem, kTmemCols5);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn5() {
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

template <int CL>
cudaError_t launch5(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                    cudaStream_t s) {
    const int gpr = cols / kGroup;
    const int max_ng = (gpr + CL - 1) / CL;
    const T5Layout l = t5_layout(max_ng);
    if (l.total > 227 * 1024) return cudaErrorNotSupported;
    auto fn = encode_fn5();
    if (fn == nullptr) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols) / 2, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) / 2};
    const cuuint32_t box[2] = {128, kRowsT};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    auto kernel = k_tc5_small<CL>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(l.total));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(((rows + kRowsT - 1) / kRowsT) * CL),
                       static_cast<unsigned>((nb + kTok - 1) / kTok));
    cfg.blockDim = dim3(kThreads5);
    cfg.dynamicSmemBytes = l.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, map, w, rows, cols, X, nb, Y, max_ng);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

#ifndef MXFP4_TC5_CLUSTER
#define MXFP4_TC5_CLUSTER 0
#endif

}  // namespace

// tcgen05 small-batch product; cudaErrorNotSupported (nothing launched) when
// the shape does not fit.  The cluster size (the split of the groups, hence
// the summation order) depends on the shape only.
cudaError_t launch_mm_tc5(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                          cudaStream_t s) {
    int cl = MXFP4_TC5_CLUSTER;
    if (cl == 0) {
        // enough CTAs to cover the GPU: row tiles x split of the groups
        const int tiles = (rows + kRowsT - 1) / kRowsT;
        cl = tiles >= 96 ? 1 : tiles >= 48 ? 2 : 4;
    }
    switch (cl) {
        case 1: return launch5<1>(w, rows, cols, X, nb, Y, s);
        case 2: return launch5<2>(w, rows, cols, X, nb, Y, s);
        case 8: return launch5<8>(w, rows, cols, X, nb, Y, s);
        default: return launch5<4>(w, rows, cols, X, nb, Y, s);
    }
}

cudaError_t read_fault_tc5(int* value, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_fault_tc5, sizeof(int));
    if (e != cudaSuccess || !reset) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_tc5, &zero, sizeof(int));
}

}  // namespace mxk
