// tc5_small.cu -- small-batch MXFP4 product on the 5th-generation tensor cores,
// with the decoded weights as the tensor-memory operand (sm_103a).
//
// Y[t*rows + r] = sum_c W[r][c] X[t][c] for up to 8 tokens per pass
// ("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs", PEROP kernel mxfp4_mm: one
// decode of each weight group serves every token of the pass).
//
// A CTA takes a tile of 128 weight rows and a slice of the groups (the K
// dimension; the CTAs of a thread-block cluster split the groups and add their
// partial sums through distributed shared memory).
//   * Decoder warps (two per 32-row quarter of tensor memory, taking batches of
//     four groups in turn) read their rows' code bytes from TMA-filled
//     shared-memory stages, convert the E2M1 codes to f16 (the hardware pair
//     conversion, exact), multiply them by 2^(k - kmax) -- k the group's scale
//     byte, kmax the largest scale byte of the row in the slice, so the product
//     stays exact in f16 for scale spreads up to 23 binades -- and store them
//     with tcgen05.st as the A operand (128 rows x K = 32 per group) in a ring
//     of tensor-memory slots.
//   * One thread issues two tcgen05.mma (M = 128, N = 16, K = 16) per group,
//     all accumulating into one FP32 tile in tensor memory; B is the pass's
//     activations in shared memory: column n < 8 is token n's hi half, column
//     8 + n its lo half (hi = f16(x 2^p), lo = f16(x 2^p - hi), one power of two
//     p per token for the slice).  Every product is exact.
//   * At the end the accumulator is read once (tcgen05.ld), hi + lo added and
//     scaled by 2^(kmax - 127) 2^-p; a row with a NaN scale byte gives NaN.
// mbarriers order the stages and slots, and every wait is bounded.
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
constexpr int kBatch = 4;                   // groups per decoder batch
constexpr int kSlots = 6;                   // A batch slots in tensor memory
constexpr int kSlotCols = kBatch * 16;      // 16 columns (K = 32 f16) per group
constexpr uint32_t kDCol = kSlots * kSlotCols;   // accumulator: 16 columns after the slots
constexpr uint32_t kTmemCols5 = 512;
constexpr int kWarps5 = 10;                 // 0-7 decode (0-3 also epilogue), 8 TMA, 9 MMA
constexpr int kThreads5 = kWarps5 * 32;
constexpr uint32_t kWait5 = 1u << 24;
constexpr int kMaxGroups5 = 140;            // groups per CTA slice (shared memory bound)
constexpr int kMaxChunks = (kTok * kMaxGroups5 * 4 + kThreads5 - 1) / kThreads5;
constexpr int kMaxScChunks = (kRowsT * ((kMaxGroups5 + 30) / 16) + kThreads5 - 1) / kThreads5;

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
    uint32_t btile, stages, sc, sc_pitch, part, kref, bars, misc, total;
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
    l.kref = l.part + kRowsT * kTok * 4;                           // [128] kmax, [128] NaN flag
    l.bars = l.kref + 2 * kRowsT;                                  // mbarriers
    l.bars = (l.bars + 7u) & ~7u;
    l.misc = l.bars + (2 * kStages5 + 2 * kSlots + 1) * 8;         // tmem addr, flags, p
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
    uint64_t* a_free = a_full + kSlots;
    uint64_t* done_bar = a_free + kSlots;
    uint8_t* kref_s = smem + L.kref;
    uint8_t* nan_s = kref_s + kRowsT;
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
            mbar_init(&code_free[i], 8);   // both decoder warps of every quarter
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&a_full[i], 4);      // the batch's decoder warp of every quarter
            mbar_init(&a_free[i], 1);      // tcgen05.commit
        }
        mbar_init(done_bar, 1);
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

    // --- activations: every thread loads its 8-element chunks of the slice at
    // once (one round trip), the per-token largest |x| picks the power of two
    // p, then the chunks become the B tiles.  B tile for group pair g2: rows n
    // (n < 8: token n hi, else token n - 8 lo), 64 f16 per row (group 2*g2 then
    // 2*g2 + 1), 128-byte swizzle.
    {
        // scale bytes of the tile's rows and this CTA's groups: row r's ng bytes,
        // read as the aligned 16-byte words that cover them (the buffer is padded
        // to 16 bytes, so no word leaves it); loads issued before the activations'
        const int nrow = min(kRowsT, rows - row0);
        const int nch_row = (ng + 30) / 16;   // words covering ng bytes at any alignment
        uint4 sv[kMaxScChunks];
#pragma unroll
        for (int u = 0; u < kMaxScChunks; ++u) {
            const int i = tid + u * kThreads5;
            const int r = i / nch_row, c = i - r * nch_row;
            sv[u] = make_uint4(0u, 0u, 0u, 0u);
            if (r < nrow) {
                const size_t s0 = plane + static_cast<size_t>(row0 + r) * gpr + g_lo;
                const size_t addr = (s0 & ~static_cast<size_t>(15)) + 16 * static_cast<size_t>(c);
                if (addr < s0 + ng) sv[u] = ldg_stream(reinterpret_cast<const uint4*>(w + addr));
            }
        }
        // chunk i (8 elements): token t = i % 8, element block e8 = i / 8 of the
        // slice; kThreads5 is a multiple of 8, so each thread keeps one token
        const int t = tid & 7;
        const int n_e8 = ng * 4;
        const bool t_ok = t < nbt;
        float xv[kMaxChunks][8];
#pragma unroll
        for (int u = 0; u < kMaxChunks; ++u) {
            const int e8 = (tid >> 3) + u * (kThreads5 / 8);
            if (e8 < n_e8 && t_ok) {
                const float4* src = reinterpret_cast<const float4*>(
                    X + static_cast<size_t>(t0 + t) * cols + static_cast<size_t>(g_lo) * kGroup +
                    8 * e8);
                const float4 a = __ldg(src), b = __ldg(src + 1);
                xv[u][0] = a.x; xv[u][1] = a.y; xv[u][2] = a.z; xv[u][3] = a.w;
                xv[u][4] = b.x; xv[u][5] = b.y; xv[u][6] = b.z; xv[u][7] = b.w;
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) xv[u][k] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < kMaxScChunks; ++u) {
            const int i = tid + u * kThreads5;
            const int r = i / nch_row, c = i - r * nch_row;
            if (r < nrow) {
                const int mis = static_cast<int>((plane + static_cast<size_t>(row0 + r) * gpr + g_lo) & 15);
                const int off = 16 * c - mis;   // position of the word's byte 0 in the row
                const uint32_t wv[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int j = off + k;
                    if (j >= 0 && j < ng)
                        sc_s[r * L.sc_pitch + j] = static_cast<uint8_t>(wv[k >> 2] >> (8 * (k & 3)));
                }
            }
        }
        if (tid < nrow)   // bytes past the row's groups read as 0 in the scan below
            for (int j = ng; j < static_cast<int>(L.sc_pitch); ++j) sc_s[tid * L.sc_pitch + j] = 0;
        float m = 0.0f;
#pragma unroll
        for (int u = 0; u < kMaxChunks; ++u)
#pragma unroll
            for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(xv[u][k]) <= 3.402823466e38f ? fabsf(xv[u][k]) : 0.0f);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (lane < 8 && m > 0.0f) atomicMax(&tmax[t], __float_as_uint(m));
        __syncthreads();
        if (tid < kTok) {
            const float mt = __uint_as_float(tmax[tid]);
            // puts the token's largest |x| in [2^14, 2^15); capped so 2^-p stays normal
            pexp[tid] = mt > 0.0f ? min(14 - ilogbf(mt), 126) : 0;
        }
        __syncthreads();
        const float pmul = exp2i5(pexp[t]);   // 2^p, a normal float for every p above
#pragma unroll
        for (int u = 0; u < kMaxChunks; ++u) {
            const int e8 = (tid >> 3) + u * (kThreads5 / 8);
            if (e8 < n_e8) {
                const int g = e8 >> 2, g2 = g >> 1;
                const int c = ((g & 1) << 2) | (e8 & 3);   // 16-byte chunk within the 128-byte row
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a0 = __fmul_rn(xv[u][2 * k], pmul);
                    const float a1 = __fmul_rn(xv[u][2 * k + 1], pmul);
                    hi[k] = pack_f16x2_5(a0, a1);
                    const float2 h = f16x2_to_f32x2(hi[k]);
                    lo[k] = pack_f16x2_5(__fsub_rn(a0, h.x), __fsub_rn(a1, h.y));
                }
                uint8_t* tb = btile + g2 * 2048;
                const int rh = t, rl = t + 8;
                *reinterpret_cast<uint4*>(tb + rh * 128 + ((c ^ (rh & 7)) << 4)) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(tb + rl * 128 + ((c ^ (rl & 7)) << 4)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        // the odd group of a ragged last pair: zero B columns
        if (ng & 1) {
            uint8_t* tb = btile + (ng >> 1) * 2048;
            for (int i = tid; i < 16 * 4; i += kThreads5) {
                const int n = i >> 2, c = 4 | (i & 3);
                *reinterpret_cast<uint4*>(tb + n * 128 + ((c ^ (n & 7)) << 4)) = make_uint4(0, 0, 0, 0);
            }
        }
    }
    __syncthreads();
    if (tid < kRowsT) {   // largest scale byte below 255 of the row, and any 255
        unsigned mx = 0u, nanf = 0u;
        for (int j = 0; j < static_cast<int>(L.sc_pitch) && tid < rows - row0; j += 4) {
            const unsigned v = *reinterpret_cast<const unsigned*>(sc_s + tid * L.sc_pitch + j);
            const unsigned is255 = __vcmpeq4(v, 0xFFFFFFFFu);
            nanf |= is255;
            mx = __vmaxu4(mx, v & ~is255);
        }
        mx = max(max(mx & 0xFFu, (mx >> 8) & 0xFFu), max((mx >> 16) & 0xFFu, mx >> 24));
        kref_s[tid] = static_cast<uint8_t>(mx);
        nan_s[tid] = nanf ? 1 : 0;
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
    const int n_batch = (ng + kBatch - 1) / kBatch;
    const int nrow = min(kRowsT, rows - row0);
    float corr[kTok];   // groups too far below the row's largest scale, summed exactly
    // one such group of row r on the CUDA cores: corr[t] += 2^(k-127) sum_e v_e x_te
    auto far_group = [&](const uint4 code, int k, int j, float (&c)[kTok]) {
        const uint32_t words[4] = {code.x, code.y, code.z, code.w};
        float v[32];
#pragma unroll
        for (int kw = 0; kw < 4; ++kw) {
            uint32_t hh[4];
            e2m1x8_to_f16x2x4(words[kw], hh);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = f16x2_to_f32x2(hh[e]);
                v[8 * kw + 2 * e] = f.x;
                v[8 * kw + 2 * e + 1] = f.y;
            }
        }
        const float sk = exp2i5(k - 127);
        for (int t = 0; t < nbt; ++t) {
            const float4* xs = reinterpret_cast<const float4*>(
                X + static_cast<size_t>(t0 + t) * cols + static_cast<size_t>(g_lo + j) * kGroup);
            float sum = 0.0f;
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                const float4 xv = __ldg(xs + e4);
                sum = __fmaf_rn(v[4 * e4], xv.x, sum);
                sum = __fmaf_rn(v[4 * e4 + 1], xv.y, sum);
                sum = __fmaf_rn(v[4 * e4 + 2], xv.z, sum);
                sum = __fmaf_rn(v[4 * e4 + 3], xv.w, sum);
            }
            c[t] = __fmaf_rn(sum, sk, c[t]);
        }
    };
    if (warp < 8) {
        // decoder: quarter q (rows 32q .. 32q+31), batches h, h+2, h+4, ...
        const int q = warp & 3, h = warp >> 2;
        const int r = q * 32 + lane;
        const int kmax = kref_s[r];
        for (int t = 0; t < kTok; ++t) corr[t] = 0.0f;
        for (int b = h; b < n_batch && !*abort_flag; b += 2) {
            const int s_idx = b / 2, st = s_idx % kStages5;
            if (!mbar_wait(&code_full[st], static_cast<uint32_t>(s_idx / kStages5) & 1u, kWait5)) {
                fail();
                break;
            }
            const int slot = b % kSlots;
            if (b >= kSlots &&
                !mbar_wait(&a_free[slot], static_cast<uint32_t>(b / kSlots - 1) & 1u, kWait5)) {
                fail();
                break;
            }
#pragma unroll
            for (int gg = 0; gg < kBatch; ++gg) {
                const int j = b * kBatch + gg;
                if (j < ng) {
                    const int jj = j % kStageGroups;
                    const uint4 code = *reinterpret_cast<const uint4*>(
                        stages + st * kStageBytes5 + r * 128 + ((jj ^ (r & 7)) << 4));
                    // 2^(k - kmax) as f16: every E2M1 value times it is exact in
                    // f16 down to k - kmax = -23; a group further below goes to
                    // the CUDA-core sum instead (and a NaN scale is flagged)
                    const int k = sc_s[r * L.sc_pitch + j];
                    const int dd = k == 255 ? -100 : k - kmax;
                    const uint32_t fb = dd >= -14 ? static_cast<uint32_t>(dd + 15) << 10
                                        : dd >= -23 ? 1u << (dd + 24)
                                                    : 0u;
                    if (dd < -23 && k != 255 && r < nrow)
                        far_group(code, k, j, corr);
                    const __half2 f2 = __halves2half2(__ushort_as_half(static_cast<unsigned short>(fb)),
                                                      __ushort_as_half(static_cast<unsigned short>(fb)));
                    uint32_t a[16];
                    const uint32_t words[4] = {code.x, code.y, code.z, code.w};
#pragma unroll
                    for (int kw = 0; kw < 4; ++kw) {
                        uint32_t hh[4];
                        e2m1x8_to_f16x2x4(words[kw], hh);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __half2 v = *reinterpret_cast<__half2*>(&hh[e]);
                            v = __hmul2(v, f2);
                            a[4 * kw + e] = *reinterpret_cast<uint32_t*>(&v);
                        }
                    }
                    tmem_st16(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                         slot * kSlotCols + gg * 16, a);
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tcf_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive5(&a_full[slot]);
                mbar_arrive5(&code_free[st]);
            }
        }
    } else if (warp == 8) {
        // TMA producer: refill each code stage once its 8 decoder warps are done
        if (lane == 0) {
            for (int s2 = kStages5; s2 < n_st && !*abort_flag; ++s2) {
                const int st = s2 % kStages5;
                if (!mbar_wait(&code_free[st], static_cast<uint32_t>(s2 / kStages5 - 1) & 1u, kWait5)) {
                    fail();
                    break;
                }
                issue_stage(s2);
            }
        }
    } else {
        // MMA issuer: every group's two MMAs accumulate into one tile
        if (lane == 0) {
            const uint64_t bdesc0 = sw128_desc5(smem_u32(btile));
            for (int b = 0; b < n_batch && !*abort_flag; ++b) {
                const int slot = b % kSlots;
                if (!mbar_wait(&a_full[slot], static_cast<uint32_t>(b / kSlots) & 1u, kWait5)) {
                    fail();
                    break;
                }
                tcf_after();
#pragma unroll
                for (int gg = 0; gg < kBatch; ++gg) {
                    const int j = b * kBatch + gg;
                    if (j >= ng) break;
                    // B: group j's 64 bytes in its pair tile, K halves 32 bytes apart
                    const uint64_t bd =
                        bdesc0 + static_cast<uint64_t>(((j >> 1) * 2048 + (j & 1) * 64) >> 4);
                    const uint32_t a_col = tmem + slot * kSlotCols + gg * 16;
                    umma_ts(tmem + kDCol, a_col, bd, j > 0 ? 1u : 0u);
                    umma_ts(tmem + kDCol, a_col + 8, bd + 2, 1u);
                }
                umma_commit5(&a_free[slot]);
                if (b == n_batch - 1) umma_commit5(done_bar);
            }
        }
    }
    if (warp >= 4 && warp < 8) {   // second decoder of each row hands over its sum
        const int r = (warp & 3) * 32 + lane;
#pragma unroll
        for (int t = 0; t < kTok; ++t) part[r * kTok + t] = corr[t];
    }
    tcf_before();
    __syncthreads();

    // --- epilogue: the accumulator, once, scaled back
    if (warp < 4) {
        const int q = warp;
        const int r = q * 32 + lane;
        bool ok = !*abort_flag && (n_batch == 0 || mbar_wait(done_bar, 0u, kWait5));
        uint32_t d[16];
        if (ok) {
            tcf_after();
            if (n_batch > 0) tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + kDCol, d);
        } else {
            fail();
        }
        const int kr = static_cast<int>(kref_s[r]) - 127;
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
            float v = 0.0f;
            if (n_batch > 0)
                v = scale2_5(__fadd_rn(__uint_as_float(d[t]), __uint_as_float(d[t + 8])),
                             kr - pexp[t]);
            v = __fadd_rn(v, __fadd_rn(corr[t], part[r * kTok + t]));
            if (nan_s[r]) v = __uint_as_float(0x7FC00000u);
            part[r * kTok + t] = v;
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
    if (l.total > 227 * 1024 || max_ng > kMaxGroups5) return cudaErrorNotSupported;
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
