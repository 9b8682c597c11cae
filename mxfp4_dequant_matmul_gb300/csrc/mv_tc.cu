// mv_tc.cu -- MXFP4 matvec and products with up to eight tokens per pass, the
// dot products on the tensor cores through mma.sync (sm_103a).
//
// Y[t*rows + r] = sum_c W[r][c] X[t][c]  ("cortiq-engine 0.8.40
// src/gpu_wgpu/mxfp4.rs", PEROP kernels mxfp4_mv and mxfp4_mm).
//
// Why the tensor cores for a matvec: at the HBM rate an SM must take in about
// 44 weight elements per clock, and decoding to FP32 and multiplying on the
// FP32 pipe costs about three instructions per element, more than the four
// issue slots per clock of an SM can give.  Here the E2M1 codes go through the
// hardware pair conversion to f16 (exact) and straight into the A operand of
// mma.sync m16n8k16; the activations are the B operand, each token's x split
// into f16 halves hi = f16(x 2^p) and lo = f16(x 2^p - hi) (p one power of two
// per token and K-slice, putting the slice's largest |x| in [2^14, 2^15)).
// Every product of an E2M1 value with an f16 is exact in the FP32 accumulator.
//
// Register layout: lane (g = lane / 4, t = lane % 4) reads code word t of rows
// g and g + 8 (and g + 16, g + 24) of a group; the four f16 pairs of that word
// are its A registers of the group's two MMAs per 16 rows.  B columns 2c, 2c + 1
// are (hi, lo) of column set c = s NT + n: token n of group slot s.  GP = 4 / NT
// consecutive groups share one accumulator, group j0 + s putting its x in the
// columns of slot s only (the other columns are zero, so its MMAs add exact
// zeros there): after the GP groups, D columns 2t, 2t + 1 of every row hold
// group j0 + t / NT's hi and lo dot products for token t % NT alone -- for
// every token count exactly the values a fresh accumulator per group gives.
// hi + lo is then taken back by 2^-p, multiplied by the group's E8M0 scale and
// added to one of four FP32 sums per row and token, r = group mod 4 (in group
// order), and the four are added as ((P0 + P1) + P2) + P3 at the end.  So the
// arithmetic per token is the same for one, two or four tokens: the batched
// product equals the matvec bit for bit.  Eight tokens take two column sets
// (tokens 0-3 and 4-7, one n8 MMA each) on the same decoded A fragments, one
// group per accumulator as with four tokens: each group is decoded once for
// all eight.  Any scale byte is handled exactly
// (255 gives NaN) and no partial sum overflows unless the result does.
//
// Data movement: a unit is 32 rows x 8 groups (32 rows x 128 code bytes), one
// TMA tile load (cp.async.bulk.tensor, 128-byte swizzle) into a ring of two
// to four stages per warp (as deep as shared memory allows).  A CTA owns up to
// 128 rows: its 16 warps take equal contiguous ranges of its (32-row unit,
// chunk) tasks, keep their sums in registers and store them as their pieces of
// a row unit; the pieces are added in chunk order.  When the activations of a whole row do not fit in shared memory, a
// cluster of CTAs splits the groups and adds its partial sums in rank order
// through distributed shared memory.  The order of every sum depends on the
// shape only, so results are deterministic and a token's result does not
// depend on the other tokens of its batch.
#include <cstdint>
#include <atomic>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace mxk {
namespace {

constexpr int kWarpsM = 16;
constexpr int kThreadsM = kWarpsM * 32;
// The CTA's tasks are always split into 16 ranges: the ranges fix the order of
// every sum.  Up to four tokens, each of the 16 warps takes one range with a
// ring of its own.  Eight tokens need twice the activation fragments in shared
// memory, so there is room for only 8 rings: the warps work in pairs, a pair
// taking two consecutive ranges in turn through one ring, each warp of the
// pair the 16-row half of every unit.  Every row's sums are the same in the
// same order either way, so a token's result does not depend on the token
// count.
constexpr int kRangesM = 16;
__host__ __device__ constexpr int rings_mv(int NT) { return NT == 8 ? 8 : kWarpsM; }
constexpr int kRowsU = 32;                  // rows per unit (two MMA row blocks)
constexpr int kChunkM = 8;                  // groups per unit (128 code bytes per row)
constexpr int kStageM = kRowsU * 128;       // one TMA tile, 4 KB
constexpr int kMinStagesM = 2;              // ring stages per warp (more when they fit)
constexpr int kMaxStagesM = 4;
#ifndef MXFP4_PRE_STAGES
#define MXFP4_PRE_STAGES 1
#endif
constexpr int kPreStagesM = MXFP4_PRE_STAGES;   // stages started before the wait (overlap)
static_assert(kPreStagesM >= 1 && kPreStagesM <= kMinStagesM, "early stages must fit every ring");
constexpr uint32_t kSmemMaxM = 227 * 1024;
constexpr int kMaxRuCta = 4;                // 32-row units per CTA
constexpr uint32_t kWaitM = 1u << 22;

// Groups per CTA slice (the B fragments take 128 * NT bytes per group).  The
// same for every NT, so that the split of the groups, hence the order of every
// sum, does not depend on the number of tokens.
constexpr int kGMax = 128;

__device__ int g_fault_mvtc;   // set when a bounded wait gives up

__device__ __forceinline__ uint32_t cluster_rank_m() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_m() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
__device__ __forceinline__ float ld_cluster_m(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ float exp2i_m(int e) {
    if (e >= -126 && e <= 127) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    if (e > 127) return __uint_as_float(0x7F800000u);
    if (e >= -149) return __uint_as_float(1u << (e + 149));
    return 0.0f;
}

// Two floats -> f16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2_m(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Shared memory (offsets from a 1024-byte aligned base).
struct MvLayout {
    uint32_t lut, xf, sc, sc_pitch, part, fin, misc, bars, ring, total;
};
__host__ __device__ inline MvLayout mv_layout(int NT, int ng_max, int ru_cta, int stages) {
    MvLayout l;
    l.lut = 0;                                                        // [256] f32
    l.xf = 1024;                                                      // [NT][ng][128] bytes
    l.sc = l.xf + static_cast<uint32_t>(ng_max) * 128 * NT;           // [rows][pitch] u8
    // an odd number of 16-byte words per row: eight rows' scale bytes of a unit
    // fall in eight different bank groups
    l.sc_pitch = (static_cast<uint32_t>(ng_max) + 15u) & ~15u;
    if ((l.sc_pitch / 16u) % 2u == 0u) l.sc_pitch += 16u;
    l.part = l.sc + static_cast<uint32_t>(ru_cta) * kRowsU * l.sc_pitch;   // [warp + ru][32][NT]
    l.part = (l.part + 15u) & ~15u;
    // [rows][NT]; zero during the units: its bytes 32 .. 47 are the B values of
    // the lanes that hold none
    l.fin = l.part + static_cast<uint32_t>(kRangesM + ru_cta - 1) * kRowsU * NT * 4;
    l.misc = l.fin + static_cast<uint32_t>(ru_cta) * kRowsU * NT * 4;   // tmax[8], flag, x barrier
    l.bars = l.misc + 48;   // [full, empty][rings][kMaxStagesM]
    l.ring = (l.bars + 2 * kWarpsM * kMaxStagesM * 8 + 1023u) & ~1023u;
    l.total = l.ring + static_cast<uint32_t>(rings_mv(NT) * stages) * kStageM + 1024;   // + align slack
    return l;
}

template <int NT, int CL>
__global__ void __launch_bounds__(kThreadsM, 1)
    k_mv_tc(const __grid_constant__ CUtensorMap tmap, const uint8_t* __restrict__ w, int rows,
            int cols, const float* __restrict__ X, int nb, float* __restrict__ Y, int ru_cta,
            int ng_max, int stages, int overlap) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const MvLayout L = mv_layout(NT, ng_max, ru_cta, stages);
    float* lut = reinterpret_cast<float*>(smem + L.lut);
    uint8_t* xf_b = smem + L.xf;
    uint8_t* sc_s = smem + L.sc;
    float* part = reinterpret_cast<float*>(smem + L.part);
    float* fin = reinterpret_cast<float*>(smem + L.fin);
    constexpr int kThr = kThreadsM;
    constexpr bool kPaired = NT == 8;                   // two warps per ring
    constexpr int kRpw = kRangesM / rings_mv(NT);       // ranges per ring
    unsigned* tmax = reinterpret_cast<unsigned*>(smem + L.misc);   // [8]
    int* not_plain = reinterpret_cast<int*>(smem + L.misc + 32);
    uint64_t* x_bar = reinterpret_cast<uint64_t*>(smem + L.misc + 40);   // the activations' copy

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int owner = kPaired ? warp >> 1 : warp;        // the ring this warp reads
    const int half = kPaired ? warp & 1 : 0;            // its 16-row half of a unit (pairs)
    const bool issuer = lane == 0 && half == 0;         // starts the ring's copies
    const uint32_t rank = CL > 1 ? cluster_rank_m() : 0u;
    const int range = blockIdx.x / CL;
    const int t0 = blockIdx.y * NT;
    const int nbt = min(NT, nb - t0);
    const int gpr = cols / kGroup;
    const int g_lo = static_cast<int>(static_cast<long>(rank) * gpr / CL);
    const int g_hi = static_cast<int>(static_cast<long>(rank + 1) * gpr / CL);
    const int ng = g_hi - g_lo;                          // >= 1 (CL <= gpr)
    const int n_c = (ng + kChunkM - 1) / kChunkM;
    const int n_ru_all = (rows + kRowsU - 1) / kRowsU;
    const int ru0 = range * ru_cta;
    const int n_ru = min(ru_cta, n_ru_all - ru0);        // >= 1 by the grid size
    const int row0 = ru0 * kRowsU;
    const size_t plane = static_cast<size_t>(rows) * cols / 2;

    // The CTA's (row unit, chunk) tasks, row unit major, in 16 contiguous ranges
    // as equal as the count allows (shape only).  With 16 warps, warp w takes
    // range w when the count divides evenly (consecutive warps then stream
    // neighbouring rows), else range (w mod 4) 4 + w / 4, so that each scheduler
    // (the warps w = s mod 4) holds a contiguous quarter of the tasks; with 8
    // warps, warp w takes ranges 2w and 2w + 1 one after the other.  A warp's
    // sums become the piece of its range for a row unit (slot range + row unit)
    // whenever its range leaves the unit or ends.
    const int n_tasks = n_ru * n_c;
    const int rg0 = kRpw > 1 ? owner * kRpw
                             : (n_tasks % kRangesM == 0 ? warp
                                                        : (warp & 3) * (kRangesM / 4) + (warp >> 2));
    const int t_lo = rg0 * n_tasks / kRangesM;
    const int n_units = (rg0 + kRpw) * n_tasks / kRangesM - t_lo;
    int rg = rg0;                                          // the range of the current unit
    int rg_end = (rg0 + 1) * n_tasks / kRangesM;           // its end (a task index)

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars) + owner * kMaxStagesM;
    uint64_t* empty = bars + kWarpsM * kMaxStagesM;      // (pairs) both warps done with a stage
    uint8_t* ring = smem + L.ring + static_cast<size_t>(owner) * stages * kStageM;
    const uint64_t policy = l2_evict_first();
    // the unit of row unit ru, chunk c into stage st (lane 0)
    auto issue_rc = [&](int ru, int c, int st) {
        const int x = (g_lo + c * kChunkM) * kGroupBytes;
        const int y = row0 + ru * kRowsU;
        mbar_arrive_expect_tx(&bars[st], kStageM);
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(ring + st * kStageM)),
            "l"(&tmap), "r"(x), "r"(y), "r"(smem_u32(&bars[st])), "l"(policy)
            : "memory");
    };
    // the next kernel of the stream may begin its own launch (it waits for this
    // one before touching anything this one writes)
    if (overlap) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid < NT) tmax[tid] = 0u;
    if (tid == 0) {
        *not_plain = 0;
        mbar_init(x_bar, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < ru_cta * kRowsU * NT / 4; i += kThr)
        reinterpret_cast<uint4*>(fin)[i] = make_uint4(0u, 0u, 0u, 0u);

    // --- prologue: scale bytes, weights, activations
    const int nrow = min(n_ru * kRowsU, rows - row0);
    // 16-byte words covering a row's ng scale bytes: exactly ng / 16 when the
    // rows' slices start on 16 bytes and fill whole words, else enough for any
    // alignment (ragged words are stored byte by byte below)
    const bool sc_whole = gpr % 16 == 0 && g_lo % 16 == 0 && ng % 16 == 0;
    const int nch_row = sc_whole ? ng / 16 : (ng + 30) / 16;
    constexpr int kScU = (kMaxRuCta * kRowsU * ((kGMax + 30) / 16) + kThr - 1) / kThr;
    uint4 sv[kScU];
#pragma unroll
    for (int u = 0; u < kScU; ++u) {
        const int i = tid + u * kThr;
        const int r = i / nch_row, c = i - r * nch_row;
        sv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (r < nrow) {
            const size_t s0 = plane + static_cast<size_t>(row0 + r) * gpr + g_lo;
            const size_t addr = (s0 & ~static_cast<size_t>(15)) + 16 * static_cast<size_t>(c);
            if (addr < s0 + ng) sv[u] = ldg_stream(reinterpret_cast<const uint4*>(w + addr));
        }
    }
    // The weights stream after the prologue's own loads, which would otherwise
    // wait behind them in the memory system -- unless the launch overlaps the
    // previous kernel of the stream (programmatic dependent launch): then the
    // weights, which that kernel does not write, start at once (behind the
    // scale bytes), and x (which it may write) is read only once it has
    // completed.  (unit k goes to stage k: never more units than the ring has
    // stages)
    auto start_weights = [&](int k0, int k1) {   // this ring's units k0 .. k1-1
        if (issuer) {
            if (k0 == 0) {
                for (int st = 0; st < stages; ++st) {
                    mbar_init(&bars[st], 1);
                    if (kPaired) mbar_init(&empty[st], 2);
                }
                fence_mbar_init();
            }
            for (int k = k0; k < k1 && k < stages && k < n_units; ++k) {
                const int task = t_lo + k, ru = task / n_c;
                issue_rc(ru, task - ru * n_c, k);
            }
        }
    };
    if (overlap) {
        start_weights(0, kPreStagesM);
        __syncthreads();   // tmax, not_plain and x_bar are set before any use below
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }

    // Activation items: item i = (n ng + j) 4 + w is word w (8 elements) of group
    // j of token n; group j of token n takes bytes (n ng + j) 128 of xf, first as
    // floats (eight tokens), then as its hi and lo halves.  Up to four tokens
    // each thread loads its items into registers (one round trip); eight tokens'
    // items (up to 8 a thread) come by one bulk copy per token.
    const int n4 = ng * 4;
    const int n_items = NT * n4;
    constexpr int kXU = (NT * kGMax * 4 + kThr - 1) / kThr;
    constexpr bool kBulkX = NT == 8;
    float xv[kXU][8];   // (eight tokens: filled from shared memory once the copies land)
    if constexpr (kBulkX) {
        if (tid == 0) {
            mbar_arrive_expect_tx(x_bar, static_cast<uint32_t>(nbt * ng * 128));
            uint64_t keep;   // x is read by every CTA of the row split: keep it in L2
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
            for (int n = 0; n < nbt; ++n)
                bulk_g2s(xf_b + static_cast<size_t>(n) * ng * 128,
                         X + static_cast<size_t>(t0 + n) * cols +
                             static_cast<size_t>(g_lo) * kGroup,
                         static_cast<uint32_t>(ng * 128), x_bar, keep);
        }
    } else {
        int tok = tid / n4, rem = tid - (tid / n4) * n4;
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            if (tid + u * kThr < n_items && tok < nbt) {
                const float4* src = reinterpret_cast<const float4*>(
                    X + static_cast<size_t>(t0 + tok) * cols + static_cast<size_t>(g_lo) * kGroup +
                    8 * rem);
                const float4 a = __ldg(src), b = __ldg(src + 1);
                xv[u][0] = a.x; xv[u][1] = a.y; xv[u][2] = a.z; xv[u][3] = a.w;
                xv[u][4] = b.x; xv[u][5] = b.y; xv[u][6] = b.z; xv[u][7] = b.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xv[u][e] = 0.0f;
            }
            for (rem += kThr; rem >= n4; rem -= n4) ++tok;
        }
    }
    start_weights(overlap ? kPreStagesM : 0, stages);   // after the prologue's loads
    // the ring's later units: fetched into L2 now, so that their ring loads,
    // issued as stages free up, find them there
    if (!kPaired && issuer)   // (eight tokens: measured slower with it)
        for (int k = stages; k < n_units; ++k) {
            const int task = t_lo + k, ru = task / n_c;
            asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                             &tmap),
                         "r"((g_lo + (task - ru * n_c) * kChunkM) * kGroupBytes),
                         "r"(row0 + ru * kRowsU)
                         : "memory");
        }
    if (!overlap) __syncthreads();   // (the same, once the loads are on their way)
    if (tid < 256) lut[tid] = e8m0_to_f32(static_cast<uint32_t>(tid));
    // "plain" scales: no byte 0 or 255 and none above kPlainMax, so that 2^(k-127)
    // is the float with bits k << 23 and the rows' sums can stay in the 2^p
    // domain without overflow (|sum| < 128*32 * 6 * 2^(kPlainMax-127) * 2^15)
    constexpr uint32_t kPlainMax = 200u;
    bool odd = false;
#pragma unroll
    for (int u = 0; u < kScU; ++u) {
        const int i = tid + u * kThr;
        const int r = i / nch_row, c = i - r * nch_row;
        if (r < nrow) {
            const int mis =
                static_cast<int>((plane + static_cast<size_t>(row0 + r) * gpr + g_lo) & 15);
            const int off = 16 * c - mis;   // row position of the word's byte 0
            const uint32_t wv[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
            if (mis == 0 && off + 16 <= ng) {   // the whole word lies in the row: one store
                *reinterpret_cast<uint4*>(sc_s + r * L.sc_pitch + off) = sv[u];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    odd |= (__vcmpeq4(wv[q], 0u) | __vcmpgtu4(wv[q], kPlainMax * 0x01010101u)) != 0u;
            } else {
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int j = off + k;
                    const uint32_t b = (wv[k >> 2] >> (8 * (k & 3))) & 0xFFu;
                    if (j >= 0 && j < ng) {
                        sc_s[r * L.sc_pitch + j] = static_cast<uint8_t>(b);
                        odd |= b == 0u || b > kPlainMax;
                    }
                }
            }
        }
    }
    if (__any_sync(0xffffffffu, odd) && lane == 0) atomicOr(not_plain, 1);

    // Each token gets one power of two p, putting the largest finite |x| of its
    // slice in [2^14, 2^15) (p = 0 for zeros; capped at 126 so that 2^-p stays
    // normal), and x 2^p is split into f16 halves hi = f16(x 2^p) and
    // lo = f16(x 2^p - hi): item i's go to bytes 16 w and 64 + 16 w of its
    // group's 128.
    if constexpr (kBulkX) {
        if (!mbar_wait(x_bar, 0u, kWaitM) && lane == 0) atomicOr(&g_fault_mvtc, 1);
        int tok = tid / n4, rem = tid - (tid / n4) * n4;
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            const int i = tid + u * kThr;
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[u][e] = 0.0f;
            if (i < n_items && tok < nbt) {
                const float4* f = reinterpret_cast<const float4*>(xf_b + static_cast<size_t>(i) * 32);
                const float4 a = f[0], b = f[1];
                xv[u][0] = a.x; xv[u][1] = a.y; xv[u][2] = a.z; xv[u][3] = a.w;
                xv[u][4] = b.x; xv[u][5] = b.y; xv[u][6] = b.z; xv[u][7] = b.w;
            }
            for (rem += kThr; rem >= n4; rem -= n4) ++tok;
        }
    }
    {
        float mloc[NT];   // this thread's largest finite |x| per token
#pragma unroll
        for (int q = 0; q < NT; ++q) mloc[q] = 0.0f;
        int tok = tid / n4, rem = tid - (tid / n4) * n4;
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            float m = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float a = fabsf(xv[u][e]);
                m = fmaxf(m, a <= 3.402823466e38f ? a : 0.0f);   // NaN and inf do not count
            }
#pragma unroll
            for (int q = 0; q < NT; ++q)
                if (q == tok) mloc[q] = fmaxf(mloc[q], m);
            for (rem += kThr; rem >= n4; rem -= n4) ++tok;
        }
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            const unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(mloc[q]));
            if (mb != 0u && lane == 0) atomicMax(&tmax[q], mb);
        }
    }
    __syncthreads();
    // 2^p of token q from its largest |x|
    auto p_of = [&](int q) {
        const float m = __uint_as_float(tmax[q]);
        const int e = static_cast<int>(__float_as_uint(m) >> 23);   // exponent field (m >= 0)
        return m > 0.0f ? (e == 0 ? 126 : min(141 - e, 126)) : 0;
    };
    {
        int tok = tid / n4, rem = tid - (tid / n4) * n4;
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            const int i = tid + u * kThr;
            const float (&e8)[8] = xv[u];
            if (i < n_items) {
                const float pm = __uint_as_float(static_cast<uint32_t>(p_of(tok) + 127) << 23);
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a0 = __fmul_rn(e8[2 * k], pm), a1 = __fmul_rn(e8[2 * k + 1], pm);
                    hi[k] = pack_f16x2_m(a0, a1);
                    const float2 h = f16x2_to_f32x2(hi[k]);
                    lo[k] = pack_f16x2_m(__fsub_rn(a0, h.x), __fsub_rn(a1, h.y));
                }
                uint4* blk = reinterpret_cast<uint4*>(xf_b + static_cast<size_t>(i >> 2) * 128);
                blk[i & 3] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                blk[4 + (i & 3)] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            for (rem += kThr; rem >= n4; rem -= n4) ++tok;
        }
    }
    __syncthreads();

    // --- this warp's units
    // NS column sets of one n8 MMA each: tokens 4 s .. 4 s + 3 in set s (eight
    // tokens), else one set holding all NT tokens
    constexpr int NS = NT == 8 ? 2 : 1;
    constexpr int NTS = NT / NS;   // tokens per column set
    constexpr int GP = 4 / NTS;    // groups sharing one accumulator
    constexpr int RQ = kPaired ? 2 : 4;   // rows per lane in a unit: g + 8q (+ 16 half)
    const int slot = t / NTS, tk = t % NTS;   // D columns 2t, 2t + 1: group slot, token in set
    const int rbase = 16 * half;              // this warp's first row in a unit
    // acc[s][q][i]: row rbase + g + 8q, token s NTS + tk, sum r = slot + GP i
    // (groups j, j mod 4 = r)
    float acc[NS][RQ][NTS];
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
        for (int q = 0; q < RQ; ++q)
#pragma unroll
            for (int i = 0; i < NTS; ++i) acc[s][q][i] = 0.0f;
    // hi + lo of a group carries the factor 2^p: undone before the scale, so
    // that no partial sum leaves the float range unless the result does; the
    // 2^p domain is kept only when it is not below the true one (p >= 0, the
    // token's |x| below 2^15), so that it adds no underflow either
    float pinv[NS];
    bool plain[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const int p_t = p_of(s * NTS + tk);
        pinv[s] = exp2i_m(-p_t);
        plain[s] = *not_plain == 0 && p_t >= 0;
    }
    // every lane's tokens in the 2^p domain (the usual case): a warp-uniform flag
    const bool all_plain = __all_sync(0xffffffffu, plain[0] && plain[NS - 1]) != 0;
    // B: lanes 8 NTS s .. 8 NTS s + 8 NTS - 1 hold the fragment of group slot s,
    // lane 8 n + 4 h + w of them word w's half h (hi, lo) of token n of the
    // column set (column set c: tokens c NTS ..), 16 bytes of group j's 128 of
    // that token
    const int b_slot = lane / (8 * NTS);
    uint32_t xf_lane[NS];
#pragma unroll
    for (int c = 0; c < NS; ++c)
        xf_lane[c] = smem_u32(xf_b) +
                     static_cast<uint32_t>((c * NTS + (lane % (8 * NTS)) / 8) * ng * 128 +
                                           (lane % 8) * 16);
    const uint32_t zero_lane = smem_u32(fin) + 32;
    const uint32_t sel0 = 0x4044u + (static_cast<uint32_t>(slot) << 8);   // byte slot -> byte 2
    // token n's four sums: P_r in lane (g, (r mod GP) NTS + n), entry r / GP; lane
    // (g, n) adds them in order and stores them as this warp's piece of row unit ru
    auto flush = [&](int ru) {
        float* pw = part + static_cast<size_t>(rg + ru) * kRowsU * NT;
#pragma unroll
        for (int s = 0; s < NS; ++s) {
#pragma unroll
            for (int q = 0; q < RQ; ++q) {
                float p[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    p[r] = __shfl_sync(0xffffffffu, acc[s][q][r / GP],
                                       (lane & ~3) | ((r % GP) * NTS + tk));
                float v = __fadd_rn(__fadd_rn(__fadd_rn(p[0], p[1]), p[2]), p[3]);
                // back from the 2^p domain (exact: a power of two, no overflow)
                if (plain[s]) v = __fmul_rn(v, pinv[s]);
                if (t < NTS)   // lane (g, t): token t of set s
                    pw[(rbase + g + 8 * q) * NT + s * NTS + t] = v;
#pragma unroll
                for (int i = 0; i < NTS; ++i) acc[s][q][i] = 0.0f;
            }
        }
    };
    bool failed = false;
    int k = 0, cur_ru = -1;
    // (row unit, chunk) of unit k and of unit k + stages, the next to be issued
    int u_ru = t_lo / n_c, u_c = t_lo - (t_lo / n_c) * n_c;
    int i_ru = (t_lo + stages) / n_c, i_c = (t_lo + stages) - ((t_lo + stages) / n_c) * n_c;
    int st = 0;           // k mod stages
    uint32_t phase = 0;   // (k / stages) mod 2
    const uint8_t* scr = sc_s;
    for (; k < n_units; ++k) {
        const int ru = u_ru, chunk = u_c;   // this unit's row unit and chunk
        if (++u_c == n_c) {
            u_c = 0;
            ++u_ru;
        }
        if (kRpw > 1) {
            // the unit starts the ring's next range: the last range's piece is done
            while (t_lo + k >= rg_end) {
                if (cur_ru >= 0) flush(cur_ru);
                cur_ru = -1;
                ++rg;
                rg_end = (rg + 1) * n_tasks / kRangesM;
            }
        }
        if (ru != cur_ru) {
            if (cur_ru >= 0) flush(cur_ru);
            cur_ru = ru;
            scr = sc_s + static_cast<size_t>(ru * kRowsU + rbase + g) * L.sc_pitch;
        }
        if (!mbar_wait(&bars[st], phase, kWaitM)) {
            failed = true;
            break;
        }
        const uint8_t* stg = ring + st * kStageM;
        // this lane's row of the tile (lane, or rbase + lane % 16 for a pair's
        // half), chunk 0 after the swizzle; chunk j is at that address ^ (j << 4)
        // (the tile is 1024-byte aligned; rbase is a multiple of 8)
        const int trow = kPaired ? rbase + (lane & 15) : lane;
        const uint32_t row_addr = smem_u32(stg) + trow * 128 + ((lane & 7) << 4);
        const int gc0 = chunk * kChunkM;   // first group of the unit in the slice
        const int ngc = min(kChunkM, ng - gc0);
        uint2 sb[RQ];   // the unit's 8 scale bytes of rows rbase + g + 8q
#pragma unroll
        for (int q = 0; q < RQ; ++q)
            sb[q] = *reinterpret_cast<const uint2*>(scr + q * 8 * L.sc_pitch + gc0);
        // B fragments of the unit's first group (group j at immediate offsets
        // from it)
        uint32_t xb[NS];
#pragma unroll
        for (int c = 0; c < NS; ++c) xb[c] = xf_lane[c] + static_cast<uint32_t>(gc0) * 128;
        // the unit's groups; FAST: a whole unit (8 groups) and every lane's token
        // in the 2^p domain, so that no guard and no table path is needed (the
        // same arithmetic as the general form for such units)
        auto run_unit = [&](auto fast_c) {
            constexpr bool FAST = decltype(fast_c)::value;
#pragma unroll
            for (int j0 = 0; j0 < kChunkM; j0 += GP) {
                if (FAST || j0 < ngc) {
                    float d0[NS][4], d1[NS][4];   // per column set: rows g, g+8 and g+16, g+24
#pragma unroll
                    for (int s = 0; s < GP; ++s) {
                        const int j = j0 + s;
                        if (FAST || j < ngc) {
                            // code word t of the lane's rows (128-byte swizzle: chunk j
                            // of row r sits at chunk j ^ (r & 7))
                            uint32_t cwd[4];
                            uint32_t h0[4], h1[4], h2[4], h3[4];
                            if constexpr (kPaired) {
                                ldsm_x2(row_addr ^ static_cast<uint32_t>(j << 4), cwd[0], cwd[1]);
                            } else {
                                ldsm_x4(row_addr ^ static_cast<uint32_t>(j << 4), cwd);
                                e2m1x8_to_f16x2x4(cwd[2], h2);
                                e2m1x8_to_f16x2x4(cwd[3], h3);
                            }
                            e2m1x8_to_f16x2x4(cwd[0], h0);
                            e2m1x8_to_f16x2x4(cwd[1], h1);
#pragma unroll
                            for (int c = 0; c < NS; ++c) {
                                const uint32_t ba = xb[c] + static_cast<uint32_t>(j * 128);
                                const uint4 b = lds128(GP == 1 || b_slot == s ? ba : zero_lane);
                                if (s == 0) {
                                    mma16816_z(d0[c], h0[0], h1[0], h0[1], h1[1], b.x, b.y);
                                    if (!kPaired) mma16816_z(d1[c], h2[0], h3[0], h2[1], h3[1], b.x, b.y);
                                } else {
                                    mma16816(d0[c], h0[0], h1[0], h0[1], h1[1], b.x, b.y);
                                    if (!kPaired) mma16816(d1[c], h2[0], h3[0], h2[1], h3[1], b.x, b.y);
                                }
                                mma16816(d0[c], h0[2], h1[2], h0[3], h1[3], b.z, b.w);
                                if (!kPaired) mma16816(d1[c], h2[2], h3[2], h2[3], h3[3], b.z, b.w);
                            }
                        }
                    }
                    // this lane's group: j0 + slot (its scale byte: byte (j0 & 3) + slot of
                    // word j0 / 4 of the unit's bytes)
                    if (FAST || j0 + slot < ngc) {
                        const uint32_t sel = sel0 + (static_cast<uint32_t>(j0 & 3) << 8);
                        uint32_t kw[RQ];
#pragma unroll
                        for (int q = 0; q < RQ; ++q)
                            kw[q] = __byte_perm(j0 < 4 ? sb[q].x : sb[q].y, 0u, sel);
                        const int i_acc = (j0 / GP) % NTS;   // r = (j0 + slot) mod 4 = slot + GP i
#pragma unroll
                        for (int c = 0; c < NS; ++c) {
                            float v[RQ];
                            v[0] = __fadd_rn(d0[c][0], d0[c][1]);
                            v[1] = __fadd_rn(d0[c][2], d0[c][3]);
                            if constexpr (RQ == 4) {
                                v[RQ - 2] = __fadd_rn(d1[c][0], d1[c][1]);
                                v[RQ - 1] = __fadd_rn(d1[c][2], d1[c][3]);
                            }
#pragma unroll
                            for (int q = 0; q < RQ; ++q) {
                                if (FAST || plain[c])   // the sums stay in the 2^p domain; 2^(k-127) from its bits
                                    acc[c][q][i_acc] =
                                        __fmaf_rn(__uint_as_float(kw[q] << 7), v[q], acc[c][q][i_acc]);
                                else                    // any byte: the table, and 2^-p applied first
                                    acc[c][q][i_acc] = __fmaf_rn(
                                        lut[kw[q] >> 16], __fmul_rn(v[q], pinv[c]), acc[c][q][i_acc]);
                            }
                        }
                    }
                }
            }
        };
        if (all_plain && ngc == kChunkM)
            run_unit(std::true_type{});
        else
            run_unit(std::false_type{});
        __syncwarp();   // every lane is done with the stage
        if constexpr (kPaired) {
            // the stage is free once both warps of the pair are done with it
            if (lane == 0) mbar_arrive_m(&empty[st]);
            if (issuer && k + stages < n_units) {
                if (!mbar_wait(&empty[st], phase, kWaitM)) {
                    failed = true;
                } else {
                    fence_proxy_async_smem();
                    issue_rc(i_ru, i_c, st);
                }
            }
            if (__shfl_sync(0xffffffffu, failed ? 1 : 0, 0)) break;
            if (k + stages < n_units && ++i_c == n_c) {
                i_c = 0;
                ++i_ru;
            }
        } else if (lane == 0 && k + stages < n_units) {
            fence_proxy_async_smem();
            issue_rc(i_ru, i_c, st);
            if (++i_c == n_c) {
                i_c = 0;
                ++i_ru;
            }
        }
        if (++st == stages) {   // unit k + 1: stage (k + 1) mod stages, phase bit of (k + 1) / stages
            st = 0;
            phase ^= 1u;
        }
    }
    if (failed) {
        if (lane == 0) atomicOr(&g_fault_mvtc, 1);
        // let this ring's copies in flight land before the CTA can exit
        if (issuer)
            for (int kq = k; kq < k + stages && kq < n_units; ++kq)
                mbar_wait(&bars[kq % stages], static_cast<uint32_t>(kq / stages) & 1u, kWaitM);
    }
    if (cur_ru >= 0) flush(cur_ru);
    __syncthreads();

    // --- add each row unit's pieces in chunk order: the ranges from the one
    // holding the unit's first task to the one holding its last (the range of
    // task T is (16 T + 15) / n_tasks), empty ones skipped
    for (int i = tid; i < n_ru * kRowsU * NT; i += kThr) {
        const int ru = i / (kRowsU * NT), rem = i - ru * kRowsU * NT;
        const int r_a = (kRangesM * ru * n_c + kRangesM - 1) / n_tasks;
        const int r_b = (kRangesM * ((ru + 1) * n_c - 1) + kRangesM - 1) / n_tasks;
        float s = 0.0f;
        bool first = true;
        for (int r = r_a; r <= r_b; ++r) {
            if (r * n_tasks / kRangesM < (r + 1) * n_tasks / kRangesM) {
                const float v = part[static_cast<size_t>(r + ru) * kRowsU * NT + rem];
                s = first ? v : __fadd_rn(s, v);
                first = false;
            }
        }
        const int tok = rem % NT;
        if (CL == 1) {
            const int row = row0 + ru * kRowsU + rem / NT;
            if (row < rows && tok < nbt) Y[static_cast<size_t>(t0 + tok) * rows + row] = s;
        } else {
            fin[i] = s;
        }
    }
    if (CL > 1) {
        // --- add over the cluster's CTAs in rank order; CTA k writes its share of rows
        cluster_sync_m();
        const int nr = n_ru * kRowsU;
        const int r_lo = static_cast<int>(rank) * nr / CL;
        const int r_hi = static_cast<int>(rank + 1) * nr / CL;
        for (int i = r_lo * NT + tid; i < r_hi * NT; i += kThr) {
            float v[CL];   // every rank's value requested before the first is used
#pragma unroll
            for (int q = 0; q < CL; ++q) v[q] = ld_cluster_m(fin + i, static_cast<uint32_t>(q));
            float s = v[0];
#pragma unroll
            for (int q = 1; q < CL; ++q) s = __fadd_rn(s, v[q]);
            const int row = row0 + i / NT, tok = i % NT;
            if (row < rows && tok < nbt) Y[static_cast<size_t>(t0 + tok) * rows + row] = s;
        }
        cluster_sync_m();   // no CTA leaves while another still reads its sums
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_m() {
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

std::atomic<bool> g_overlap{false};

int sm_count_m() {
    static PerDevice memo;
    const int n = memo.get([] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            v = 0;
        return v;
    });
    return n > 0 ? n : 1;
}

// CTAs (CL = 1) or clusters that one wave holds, probed with the largest
// layout (four tokens) for every NT, so that the row split does not depend on
// the number of tokens either.
template <int CL>
int resident_mv() {
    static PerDevice memo;
    return memo.get([] {
        int resident = 0;
        const MvLayout lmax = mv_layout(4, kGMax, kMaxRuCta, kMinStagesM);
        auto k4 = k_mv_tc<4, CL>;
        if (cudaFuncSetAttribute(k4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemMaxM)) != cudaSuccess)
            return 0;
        if (CL == 1) return sm_count_m();
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(CL * 64, 1);
        q.blockDim = dim3(kThreadsM);
        q.dynamicSmemBytes = lmax.total;
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = CL;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        q.attrs = a;
        q.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, k4, &q) == cudaSuccess && nc > 0) resident = nc;
        return resident;
    });
}

template <int NT, int CL>
cudaError_t launch_mv(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                      cudaStream_t s) {
    const int gpr = cols / kGroup;
    const int ng_max = (gpr + CL - 1) / CL;
    auto kernel = k_mv_tc<NT, CL>;
    const int resident = resident_mv<CL>();
    if (resident < 1) return cudaErrorNotSupported;
    {
        static PerDevice memo;
        const cudaError_t attr_err = static_cast<cudaError_t>(memo.get([&] {
            return static_cast<int>(cudaFuncSetAttribute(
                kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemMaxM)));
        }));
        if (attr_err != cudaSuccess) return attr_err;
    }
    const int n_ru_all = (rows + kRowsU - 1) / kRowsU;
    int ru_cta = (n_ru_all + resident - 1) / resident;
    ru_cta = ru_cta < 1 ? 1 : (ru_cta > kMaxRuCta ? kMaxRuCta : ru_cta);
    const int n_ranges = (n_ru_all + ru_cta - 1) / ru_cta;
    // as many ring stages as the shared memory holds (deeper rings keep more
    // weight bytes in flight; the arithmetic does not depend on the depth)
    const uint32_t fixed = mv_layout(NT, ng_max, ru_cta, 0).total;
    int stages = fixed < kSmemMaxM
                     ? static_cast<int>((kSmemMaxM - fixed) / (rings_mv(NT) * kStageM)) : 0;
    stages = stages > kMaxStagesM ? kMaxStagesM : stages;
    if (stages < kMinStagesM) return cudaErrorNotSupported;
    const MvLayout l = mv_layout(NT, ng_max, ru_cta, stages);
    auto fn = encode_fn_m();
    if (fn == nullptr) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols) / 2, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) / 2};
    const cuuint32_t box[2] = {128, kRowsU};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_ranges * CL),
                       static_cast<unsigned>((nb + NT - 1) / NT));
    cfg.blockDim = dim3(kThreadsM);
    cfg.dynamicSmemBytes = l.total;
    cfg.stream = s;
    const int overlap = launch_overlap() ? 1 : 0;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 2 : 1;
    cudaError_t e =
        cudaLaunchKernelEx(&cfg, kernel, map, w, rows, cols, X, nb, Y, ru_cta, ng_max, stages,
                           overlap);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int NT>
cudaError_t launch_mv_nt(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                         cudaStream_t s) {
    const int gpr = cols / kGroup;
    switch ((gpr + kGMax - 1) / kGMax) {
        case 1: return launch_mv<NT, 1>(w, rows, cols, X, nb, Y, s);
        case 2: return launch_mv<NT, 2>(w, rows, cols, X, nb, Y, s);
        case 3: return launch_mv<NT, 3>(w, rows, cols, X, nb, Y, s);
        case 4: return launch_mv<NT, 4>(w, rows, cols, X, nb, Y, s);
        case 5:
        case 6: return launch_mv<NT, 6>(w, rows, cols, X, nb, Y, s);
        case 7:
        case 8: return launch_mv<NT, 8>(w, rows, cols, X, nb, Y, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

// Tensor-core product, up to 4 tokens per pass over the weights (passes along
// the grid's y); cudaErrorNotSupported, with nothing launched, for shapes it
// cannot take.  A token's arithmetic is the same whatever nb is.
cudaError_t launch_mv_tc(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                         cudaStream_t s) {
    if (nb <= 1) return launch_mv_nt<1>(w, rows, cols, X, nb, Y, s);
    if (nb == 2) return launch_mv_nt<2>(w, rows, cols, X, nb, Y, s);
    if (nb <= 4) return launch_mv_nt<4>(w, rows, cols, X, nb, Y, s);
    // one decode per group for up to eight tokens; passes of four where the
    // eight tokens' fragments do not fit in shared memory
    const cudaError_t e = launch_mv_nt<8>(w, rows, cols, X, nb, Y, s);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
    return launch_mv_nt<4>(w, rows, cols, X, nb, Y, s);
}

void set_launch_overlap(bool on) { g_overlap.store(on); }
bool launch_overlap() { return g_overlap.load(); }

cudaError_t read_fault_mvtc(int* value, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_fault_mvtc, sizeof(int));
    if (e != cudaSuccess || !reset) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_mvtc, &zero, sizeof(int));
}

}  // namespace mxk
