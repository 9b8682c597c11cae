// mma_small.cu -- small-batch MXFP4 product on the tensor cores (sm_103a).
//
// Y[t*rows + r] = sum_c W[r][c] X[t][c] for up to 8 tokens per chunk
// ("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs", PEROP kernel mxfp4_mm: one
// decode of each weight group serves every token of the chunk).
//
// Why tensor cores: with 8 tokens the product needs 8 FMAs per weight element
// and the FP32 pipe caps the kernel far below the HBM rate.  Here the decoded
// E2M1 codes (exact in f16, from the hardware pair conversion) are the A
// operand of mma.sync m16n8k16 (16 weight rows per warp tile, the 8 columns
// are the 8 tokens).  Each token's activation is split into f16 halves
// hi = f16(x * 2^p) and lo = f16(x * 2^p - hi), one power of two p per
// (token, group) putting the group's largest |x| just under 2^15: hi + lo
// carries 22 significant bits of x * 2^p and every product with an E2M1 value
// is exact in the FP32 accumulator.  hi and lo of an element sit in two k-slots
// of the same MMA facing the same weight, so the tensor core adds them.  A
// group (32 elements) is four MMAs into two fresh accumulators (two chains of
// two, for latency), added; each thread then multiplies its four outputs by
// scale * 2^-p and accumulates in FP32.
//
// K-permutation: lane (q = lane/4, u = lane%4) owns the k-slots 2u, 2u+1,
// 2u+8, 2u+9 of every MMA; for MMA m of a group it puts elements 8u+2m and
// 8u+2m+1 of the group in slots 2u, 2u+1 (weights and hi of x) and the same
// two elements again in slots 2u+8, 2u+9 (weights and lo of x).  A lane's A
// registers are then the decoded code word u of rows q and q+8, and its B
// registers the hi/lo halves of elements 8u..8u+7 of token q: nothing moves
// between lanes.
//
// Data movement: the code plane is described by a 2-D tensor map (bytes x
// rows); one TMA tile load (cp.async.bulk.tensor, 16 rows x 128 bytes, 128-byte
// swizzle) fills one stage of a per-warp ring for each unit of 16 rows x 8
// groups, and the lanes read their code words back with conflict-free 4-byte
// shared loads.  The scale bytes of the CTA's rows and groups are copied into
// shared memory once, before the loop.
//
// Work split without a workspace: a cluster of CL CTAs owns a range of 16-row
// blocks; CTA rank k of the cluster takes the k-th slice of the groups (so it
// prepares x for that slice only); its warps take the (row block, chunk of
// groups) units of the CTA round-robin.  Unit partials are added in chunk
// order, then over the cluster's CTAs in rank order through distributed
// shared memory: a fixed order, so results are deterministic, and a token's
// result does not depend on the other tokens of the batch.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace mxk {
namespace {

constexpr int kWarpsT = 16;                // warps per CTA
constexpr int kThreadsT = kWarpsT * 32;
constexpr int kChunk = 8;                  // groups per unit (128 code bytes per row)
constexpr int kStages = 2;                 // ring stages per warp
constexpr int kStageBytes = 16 * 128;      // one TMA tile: 16 rows x 128 bytes
constexpr uint32_t kWaitLimitT = 1u << 22;

__device__ int g_fault_mma;   // set when a bounded wait gives up

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

__device__ __forceinline__ uint32_t map_shared(const void* p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
    return out;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// 2^e as a float for any integer e (subnormal or 0 below 2^-126, inf above 2^127).
__device__ __forceinline__ float exp2i(int e) {
    if (e >= -126 && e <= 127) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    if (e > 127) return __uint_as_float(0x7F800000u);
    if (e >= -149) return __uint_as_float(1u << (e + 149));
    return 0.0f;
}

// x * 2^p exactly (two steps so that no factor leaves the float range).
__device__ __forceinline__ float scale2(float x, int p) {
    const int p1 = p / 2, p2 = p - p1;
    return __fmul_rn(__fmul_rn(x, exp2i(p1)), exp2i(p2));
}

// Two floats -> f16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared memory (bytes): xfrag [ng_cta][2 halves][32 lanes] uint4 |
// pfac [ng_cta][8] f32 | part [units][16 rows][8 tokens] f32 |
// sc [rows of the cluster][sc_pitch] u8 | mbarriers [warps][stages] |
// rings [warps][stages][2048] (1024-byte aligned: the swizzle repeats every 1 KB).
struct TcLayout {
    uint32_t xfrag, pfac, part, sc, sc_pitch, bars, ring, total;
};

__host__ __device__ inline TcLayout tc_layout(int ng_cta, int units, int rows_pc) {
    TcLayout l;
    l.xfrag = 0;
    l.pfac = l.xfrag + static_cast<uint32_t>(ng_cta) * 32 * 32;
    l.part = l.pfac + static_cast<uint32_t>(ng_cta) * 8 * 4;
    l.sc = l.part + static_cast<uint32_t>(units) * 16 * 8 * 4;
    l.sc_pitch = (static_cast<uint32_t>(ng_cta) + 15u) & ~15u;
    l.bars = l.sc + static_cast<uint32_t>(rows_pc) * l.sc_pitch;
    l.bars = (l.bars + 127u) & ~127u;
    l.ring = l.bars + kWarpsT * kStages * 8;
    l.ring = (l.ring + 1023u) & ~1023u;
    l.total = l.ring + kWarpsT * kStages * kStageBytes + 1024;   // + slack to align the base
    return l;
}

template <int CL>
__global__ void __launch_bounds__(kThreadsT, 1)
    k_mma_small(const __grid_constant__ CUtensorMap tmap, const uint8_t* __restrict__ w, int rows,
                int cols, const float* __restrict__ X, int nb, float* __restrict__ Y, int max_ng,
                int max_units, int rows_pc) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const TcLayout L = tc_layout(max_ng, max_units, rows_pc);
    uint32_t* xfrag = reinterpret_cast<uint32_t*>(smem + L.xfrag);
    float* pfac = reinterpret_cast<float*>(smem + L.pfac);
    float* part = reinterpret_cast<float*>(smem + L.part);
    uint8_t* sc_s = smem + L.sc;

    const int gpr = cols / kGroup;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = lane >> 2, u = lane & 3;
    const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
    const int cl = blockIdx.x / CL;
    const int n_cl = gridDim.x / CL;
    const int t0 = blockIdx.y * 8;
    const int nbt = min(8, nb - t0);
    const size_t plane = static_cast<size_t>(rows) * cols / 2;
    (void)plane;

    const int n_rb = (rows + 15) / 16;
    const int rb_lo = static_cast<int>(static_cast<long>(cl) * n_rb / n_cl);
    const int rb_hi = static_cast<int>(static_cast<long>(cl + 1) * n_rb / n_cl);
    const int g_lo = static_cast<int>(static_cast<long>(rank) * gpr / CL);
    const int g_hi = static_cast<int>(static_cast<long>(rank + 1) * gpr / CL);
    const int ng = g_hi - g_lo;
    const int n_chunks = (ng + kChunk - 1) / kChunk;           // this CTA's
    const int nc_max = (max_ng + kChunk - 1) / kChunk;         // same in every CTA
    const int n_units = (rb_hi - rb_lo) * n_chunks;
    // partial slot of unit (local row block r, chunk c): r * nc_max + c

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars) + warp * kStages;
    uint8_t* ring = smem + L.ring + static_cast<size_t>(warp) * kStages * kStageBytes;
    const uint64_t policy = l2_evict_first();

    // Stage fill for unit `un` (this warp's), by lane 0: one TMA tile load of
    // 16 rows x 128 code bytes (rows past the end and bytes past the row read
    // as zero).
    auto issue = [&](int un, int st) {
        if (lane != 0) return;
        const int rb = rb_lo + un / n_chunks, c = un % n_chunks;
        const int x = (g_lo + c * kChunk) * kGroupBytes, y = rb * 16;
        mbar_arrive_expect_tx(&bars[st], kStageBytes);
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(ring + st * kStageBytes)),
            "l"(&tmap), "r"(x), "r"(y), "r"(smem_u32(&bars[st])), "l"(policy)
            : "memory");
    };

    // Weights start streaming before x is prepared.
    if (lane == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    __syncwarp();
    for (int k = 0; k < kStages; ++k) {
        const int un = warp + k * kWarpsT;
        if (un < n_units) issue(un, k);
    }

    // --- the scale bytes of this cluster's rows and this CTA's groups
    const int row_lo = rb_lo * 16;
    const int nrow = min((rb_hi - rb_lo) * 16, rows - row_lo);
    // (eight loads in flight per thread before their stores)
    for (int base = threadIdx.x; base < nrow * ng; base += 8 * kThreadsT) {
        uint32_t v[8];
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            const int i = base + k8 * kThreadsT;
            v[k8] = 0u;
            if (i < nrow * ng) {
                const int r = i / ng, j = i - r * ng;
                v[k8] = __ldg(w + plane + static_cast<size_t>(row_lo + r) * gpr + g_lo + j);
            }
        }
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            const int i = base + k8 * kThreadsT;
            if (i < nrow * ng) {
                const int r = i / ng, j = i - r * ng;
                sc_s[r * L.sc_pitch + j] = static_cast<uint8_t>(v[k8]);
            }
        }
    }

    // --- x for this CTA's groups: warp w prepares groups w, w+8, ...; lane
    // (q, u) takes token q, elements 8u..8u+7.  All of the warp's loads are
    // issued before any is used.
    constexpr int kMaxPrep = 8;   // groups per warp with their loads batched
    auto prep_group = [&](int j, const float4& a, const float4& b) {
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        // p puts the largest |x| of the group in [2^14, 2^15) (capped at 126 so
        // 2^-p stays normal; an all-zero or non-finite group keeps p = 0).
        const int p = (m > 0.0f && m <= 3.402823466e38f) ? min(14 - ilogbf(m), 126) : 0;
        uint32_t f[8];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const float a0 = scale2(v[2 * mm], p), a1 = scale2(v[2 * mm + 1], p);
            const uint32_t hi = pack_f16x2(a0, a1);
            const float h0 =
                __half2float(__ushort_as_half(static_cast<unsigned short>(hi & 0xFFFFu)));
            const float h1 = __half2float(__ushort_as_half(static_cast<unsigned short>(hi >> 16)));
            f[2 * mm] = hi;                                                      // b0 of MMA mm
            f[2 * mm + 1] = pack_f16x2(__fsub_rn(a0, h0), __fsub_rn(a1, h1));   // b1 of MMA mm
        }
        uint4* dst = reinterpret_cast<uint4*>(xfrag) + static_cast<size_t>(j) * 64 + lane;
        dst[0] = make_uint4(f[0], f[1], f[2], f[3]);
        dst[32] = make_uint4(f[4], f[5], f[6], f[7]);
        if (u == 0) pfac[j * 8 + q] = exp2i(-p);
    };
    auto load_x = [&](int j, float4& a, float4& b) {
        a = make_float4(0.f, 0.f, 0.f, 0.f);
        b = a;
        if (j < ng && q < nbt) {
            const float4* src = reinterpret_cast<const float4*>(
                X + static_cast<size_t>(t0 + q) * cols + static_cast<size_t>(g_lo + j) * kGroup +
                8 * u);
            a = __ldg(src);
            b = __ldg(src + 1);
        }
    };
    {
        float4 xa[kMaxPrep], xb[kMaxPrep];
#pragma unroll
        for (int jj = 0; jj < kMaxPrep; ++jj) load_x(warp + jj * kWarpsT, xa[jj], xb[jj]);
#pragma unroll
        for (int jj = 0; jj < kMaxPrep; ++jj)
            if (warp + jj * kWarpsT < ng) prep_group(warp + jj * kWarpsT, xa[jj], xb[jj]);
        for (int j = warp + kMaxPrep * kWarpsT; j < ng; j += kWarpsT) {
            float4 a, b;
            load_x(j, a, b);
            prep_group(j, a, b);
        }
    }
    __syncthreads();

    // --- this warp's units
    bool failed = false;
    int k = 0;
    for (int un = warp; un < n_units; un += kWarpsT, ++k) {
        const int st = k % kStages;
        if (!mbar_wait(&bars[st], static_cast<uint32_t>(k / kStages) & 1u, kWaitLimitT)) {
            failed = true;
            break;
        }
        const int c = un % n_chunks;
        const int gc = g_lo + c * kChunk;
        const int ngc = min(kChunk, g_hi - gc);
        const int rb = rb_lo + un / n_chunks;
        const uint8_t* stg = ring + st * kStageBytes;
        // scale bytes of rows q and q+8 for this unit's groups (garbage for rows
        // past the end, whose results are never written)
        const uint8_t* sc0 = sc_s + static_cast<size_t>(rb * 16 + q - row_lo) * L.sc_pitch + (gc - g_lo);
        const uint8_t* sc1 = sc0 + 8 * L.sc_pitch;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};   // (row q | q+8) x (token 2u | 2u+1)
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (j < ngc) {
                // 128-byte swizzle: chunk j of row r sits at chunk j ^ (r & 7)
                const int sw = ((j ^ q) & 7) * 16 + u * 4;
                const uint32_t w0 = *reinterpret_cast<const uint32_t*>(stg + q * 128 + sw);
                const uint32_t w1 = *reinterpret_cast<const uint32_t*>(stg + (q + 8) * 128 + sw);
                uint32_t h0[4], h1[4];
                e2m1x8_to_f16x2x4(w0, h0);
                e2m1x8_to_f16x2x4(w1, h1);
                const uint4* xf = reinterpret_cast<const uint4*>(xfrag) +
                                  static_cast<size_t>(gc - g_lo + j) * 64 + lane;
                const uint4 b01 = xf[0], b23 = xf[32];
                // two independent accumulation chains (elements 8u..8u+3 and
                // 8u+4..8u+7), added afterwards
                float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
                mma_16816(da, h0[0], h1[0], h0[0], h1[0], b01.x, b01.y);
                mma_16816(db, h0[2], h1[2], h0[2], h1[2], b23.x, b23.y);
                mma_16816(da, h0[1], h1[1], h0[1], h1[1], b01.z, b01.w);
                mma_16816(db, h0[3], h1[3], h0[3], h1[3], b23.z, b23.w);
                float d[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) d[e] = __fadd_rn(da[e], db[e]);
                const float s0 = e8m0_to_f32(sc0[j]), s1 = e8m0_to_f32(sc1[j]);
                const float p0 = pfac[(gc - g_lo + j) * 8 + 2 * u];
                const float p1 = pfac[(gc - g_lo + j) * 8 + 2 * u + 1];
                acc[0] = __fmaf_rn(__fmul_rn(s0, p0), d[0], acc[0]);
                acc[1] = __fmaf_rn(__fmul_rn(s0, p1), d[1], acc[1]);
                acc[2] = __fmaf_rn(__fmul_rn(s1, p0), d[2], acc[2]);
                acc[3] = __fmaf_rn(__fmul_rn(s1, p1), d[3], acc[3]);
            }
        }
        __syncwarp();   // all lanes are done with the stage
        if (un + kStages * kWarpsT < n_units) {
            fence_proxy_async_smem();
            issue(un + kStages * kWarpsT, st);
        }
        float* pu = part + static_cast<size_t>((un / n_chunks) * nc_max + c) * 128;
        pu[q * 8 + 2 * u] = acc[0];
        pu[q * 8 + 2 * u + 1] = acc[1];
        pu[(q + 8) * 8 + 2 * u] = acc[2];
        pu[(q + 8) * 8 + 2 * u + 1] = acc[3];
    }
    if (failed) {
        if (lane == 0) atomicOr(&g_fault_mma, 1);
        // let this warp's copies in flight land before the CTA can exit
        for (int kk = k; kk < k + kStages; ++kk) {
            const int un = warp + kk * kWarpsT;
            if (un < n_units)
                mbar_wait(&bars[kk % kStages], static_cast<uint32_t>(kk / kStages) & 1u,
                          kWaitLimitT);
        }
    }
    __syncthreads();

    // --- add the chunks of each row block (chunk order) into chunk 0's slot
    const int nrb = rb_hi - rb_lo;
    for (int i = threadIdx.x; i < nrb * 128; i += kThreadsT) {
        const int r = i >> 7, e = i & 127;
        float s = 0.0f;   // a CTA without groups contributes zeros
        if (n_chunks > 0) {
            s = part[static_cast<size_t>(r * nc_max) * 128 + e];
            for (int c = 1; c < n_chunks; ++c)
                s = __fadd_rn(s, part[static_cast<size_t>(r * nc_max + c) * 128 + e]);
        }
        part[static_cast<size_t>(r * nc_max) * 128 + e] = s;
    }
    if (CL > 1) cluster_sync(); else __syncthreads();

    // --- add over the cluster's CTAs (rank order); CTA k writes its share
    const int r_lo = static_cast<int>(static_cast<long>(rank) * nrb * 16 / CL);
    const int r_hi = static_cast<int>(static_cast<long>(rank + 1) * nrb * 16 / CL);
    for (int i = r_lo * 8 + threadIdx.x; i < r_hi * 8; i += kThreadsT) {
        const int lr = i >> 3, tt = i & 7;
        const size_t off = static_cast<size_t>((lr >> 4) * nc_max) * 128 + (lr & 15) * 8 + tt;
        float s = 0.0f;
        if (CL > 1) {
            for (uint32_t kk = 0; kk < static_cast<uint32_t>(CL); ++kk) {
                const float v = ld_cluster_f32(map_shared(part + off, kk));
                s = kk == 0 ? v : __fadd_rn(s, v);
            }
        } else {
            s = part[off];
        }
        const int row = rb_lo * 16 + lr;
        if (row < rows && tt < nbt) Y[static_cast<size_t>(t0 + tt) * rows + row] = s;
    }
    if (CL > 1) cluster_sync();   // no CTA leaves while another still reads its partials
}

// cuTensorMapEncodeTiled from the driver (looked up once; no link to libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// The code plane as a 2-D byte tensor [rows][cols/2], tiles of 16 rows x 128
// bytes, 128-byte swizzle.
cudaError_t code_plane_map(CUtensorMap* map, const uint8_t* w, int rows, int cols) {
    auto fn = encode_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols) / 2, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) / 2};
    const cuuint32_t box[2] = {128, 16};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int CL>
cudaError_t launch_cl(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                      cudaStream_t s) {
    int dev = 0, sms = 152;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 152;
    const int gpr = cols / kGroup;
    const int n_rb = (rows + 15) / 16;
    const int max_ng = (gpr + CL - 1) / CL;
    const int n_chunks = (max_ng + kChunk - 1) / kChunk;
    auto kernel = k_mma_small<CL>;

    CUtensorMap map;
    e = code_plane_map(&map, w, rows, cols);
    if (e != cudaSuccess) return cudaErrorNotSupported;

    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreadsT);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    int n_cl = sms / CL;
    if (n_cl > n_rb) n_cl = n_rb;
    if (n_cl < 1) n_cl = 1;
    int max_rb = 0;
    TcLayout l{};
    for (int pass = 0; pass < 2; ++pass) {
        max_rb = (n_rb + n_cl - 1) / n_cl;
        l = tc_layout(max_ng, max_rb * n_chunks, max_rb * 16);
        if (l.total > 227 * 1024) return cudaErrorNotSupported;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(l.total));
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(static_cast<unsigned>(n_cl * CL), 1);
        cfg.dynamicSmemBytes = l.total;
        if (pass == 1) break;
        int fit = 0;
        if (cudaOccupancyMaxActiveClusters(&fit, kernel, &cfg) != cudaSuccess || fit < 1) break;
        if (fit >= n_cl) break;
        n_cl = fit;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(n_cl * CL), (nb + 7) / 8);
    e = cudaLaunchKernelEx(&cfg, kernel, map, w, rows, cols, X, nb, Y, max_ng, max_rb * n_chunks,
                           max_rb * 16);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

#ifndef MXFP4_MMA_CLUSTER
#define MXFP4_MMA_CLUSTER 0   // 0: by shape; otherwise 1, 2, 4 or 8
#endif

}  // namespace

cudaError_t read_fault_mma(int* value, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_fault_mma, sizeof(int));
    if (e != cudaSuccess || !reset) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_mma, &zero, sizeof(int));
}

// Tensor-core small-batch product; cudaErrorNotSupported (nothing launched)
// when one cluster's partials do not fit in a CTA's shared memory.
cudaError_t launch_mm_tc(const uint8_t* w, int rows, int cols, const float* X, int nb, float* Y,
                         cudaStream_t s) {
    // The cluster size fixes the summation order, so it depends on the shape
    // only: a token gets the same bits whatever the batch around it.
    int cl = MXFP4_MMA_CLUSTER;
    if (cl == 0) cl = 8;
    switch (cl) {
        case 1: return launch_cl<1>(w, rows, cols, X, nb, Y, s);
        case 2: return launch_cl<2>(w, rows, cols, X, nb, Y, s);
        case 4: return launch_cl<4>(w, rows, cols, X, nb, Y, s);
        default: return launch_cl<8>(w, rows, cols, X, nb, Y, s);
    }
}

}  // namespace mxk
