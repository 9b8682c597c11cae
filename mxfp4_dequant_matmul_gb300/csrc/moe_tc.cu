// moe_tc.cu -- routed-expert passes on the tensor cores through mma.sync
// (sm_103a): act = SiLU(gate_e x) * (up_e x) for every routed pair, and
// o = down_e act ("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs" kernels
// dsv4_global_gate_up_mxfp4 and dsv4_global_down_mxfp4), grouped by expert as
// "rlx-cpu 0.2.17 src/gguf_matmul.rs" grouped_moe_sort_plan groups them.
//
// The arithmetic of a product is the one of mv_tc.cu: E2M1 codes through the
// hardware pair conversion into the A operand of mma.sync m16n8k16, each
// pair's vector split into f16 hi and lo (one power of two per pair putting
// its largest |x| in [2^14, 2^15)), two MMAs per group and 16 rows, then 2^-p
// and the group's scale in FP32 and the FP32 row sum.  A segment with n pairs
// uses NP = 1, 2 or 4 column sets (NP >= n) and lets GP = 4 / NP consecutive
// groups share one accumulator: B columns 2c, 2c + 1 are (hi, lo) of pair
// c % NP for group slot c / NP, group j0 + s putting its x in slot s's columns
// only, so that the D columns of lane t hold group j0 + t / NP of pair t % NP
// alone.  Lane t sums its slot's groups; the slots are added in order at the
// end of the warp's units.
//
// Work: a segment is (touched expert, up to four of its pairs, 128 rows of its
// gate and up matrices or 256 rows of its down matrix); persistent CTAs claim
// the segments of all touched experts in order from a counter in the
// workspace, two ahead of use.  The vectors' B fragments are made once per
// pass by k_moe_split (a block per vector in the workspace); for each segment a
// CTA copies the rows' scale bytes with one bulk copy per matrix and its pairs'
// fragment blocks with one bulk copy per pair, and its 16 warps stream
// (matrix, 32-row unit, chunk range) units of 32 rows x 8 groups through
// per-warp rings of TMA tile loads (a 3-D tensor map over the bank: bytes,
// rows, experts).  A warp keeps its sums in the 2^p domain when its units'
// scale bytes are all in 1..200 and the segment's pairs have p >= 0, else it
// applies 2^-p and the table scale per group.  Partial sums are added in chunk
// order; the gate/up pass applies SiLU(g) * u and writes act[pair][row], the
// down pass writes o[pair][row].  Every order and every choice of arithmetic
// depends on the shapes, the routing and the data only (not on which CTA takes
// a segment).
#include <cstdint>
#include <functional>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace mxk {
namespace {

constexpr int kWarpsE = 16;
constexpr int kThreadsE = kWarpsE * 32;
constexpr int kRowsUE = 32;                 // rows per unit (two MMA row blocks)
constexpr int kChunkE = 8;                  // groups per unit
constexpr int kStageE = kRowsUE * 128;      // one TMA tile, 4 KB
constexpr int kStagesE = 2;                 // ring stages per warp
// 32-row units per segment: 8 / NM (256 rows of one matrix, 128 rows of two), so
// that every warp has the same number of units per segment in both passes
__host__ __device__ constexpr int ru_seg(int NM) { return 8 / NM; }
constexpr int kTokSeg = 4;                  // pairs per segment
constexpr int kGMaxE = 128;                 // groups per row (B fragments in shared memory)
constexpr int kMaxExpertsE = 1024;
constexpr uint32_t kSmemMaxE = 227 * 1024;
constexpr uint32_t kWaitE = 1u << 22;
constexpr int kSplitThreads = 256;

// Bytes of one vector's fragment block: 16 header bytes (its power of two p as
// an int32, then zeros) and 128 bytes per group.
__host__ __device__ constexpr uint32_t frag_block(int gpr) {
    return 16u + static_cast<uint32_t>(gpr) * 128u;
}

__device__ int g_fault_moetc;   // set when a bounded wait gives up

__device__ __forceinline__ float exp2i_e(int e) {
    if (e >= -126 && e <= 127) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    if (e > 127) return __uint_as_float(0x7F800000u);
    if (e >= -149) return __uint_as_float(1u << (e + 149));
    return 0.0f;
}

__device__ __forceinline__ uint32_t pack_f16x2_e(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// The B fragments of vectors of `cols` floats (a token's x for the gate/up
// pass, a pair's act row for the down pass), made once per pass instead of once
// per segment that reads them.  Vector v becomes the block of frag_block(gpr)
// bytes at frag + v * frag_block(gpr):
//   bytes 0-15            p (int32), then zeros: the power of two that puts the
//                         vector's largest finite |x| in [2^14, 2^15) (p = 14 -
//                         floor(log2 m) from m's exponent field; a subnormal m
//                         takes the cap, 126, which keeps 2^-p normal; 0 for a
//                         vector of zeros)
//   16 + 128 j + 16 w     f16 hi of x * 2^p for elements 32 j + 8 w .. + 7 of
//                         group j, two to a 32-bit word
//   16 + 128 j + 64 + 16 w  f16 lo = f16(x * 2^p - hi) of the same elements
// so that lanes 8 q .. 8 q + 7 of a warp, reading 16 bytes each at 16 + 128 j +
// 16 (lane % 8) of pair q's block, hold B columns 2 q (hi) and 2 q + 1 (lo) of
// mma.sync m16n8k16 for group j.  A block of threads per vector (grid-stride),
// each thread holding its (at most kSplitItems) 8-element pieces in registers.
// wait_first: the vectors come from the previous kernel (wait for it before
// reading); else they are inputs already complete and the wait comes last, so
// that the pass launched after this kernel also sees the previous kernel done.
constexpr int kSplitItems = (kGMaxE * 4 + kSplitThreads - 1) / kSplitThreads;

__global__ void __launch_bounds__(kSplitThreads) k_moe_split(const float* __restrict__ vec,
                                                             int n_vec, int cols,
                                                             uint8_t* __restrict__ frag,
                                                             int wait_first) {
    __shared__ unsigned s_max[3];   // by vector index mod 3: one barrier per vector
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int gpr = cols / kGroup, n_items = gpr * 4;   // gpr <= kGMaxE
    const size_t vb = frag_block(gpr);
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) s_max[0] = 0u;
    __syncthreads();
    for (int v = blockIdx.x, it = 0; v < n_vec; v += gridDim.x, ++it) {
        unsigned* sm = &s_max[it % 3];
        // the next vector's slot: last read before the previous vector's barrier,
        // next written after this vector's
        if (threadIdx.x == 0) s_max[(it + 1) % 3] = 0u;
        const float4* src = reinterpret_cast<const float4*>(vec + static_cast<size_t>(v) * cols);
        float f[kSplitItems][8];
        float mx = 0.0f;
#pragma unroll
        for (int u = 0; u < kSplitItems; ++u) {
            const int i = threadIdx.x + u * kSplitThreads;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (i < n_items) {
                a = __ldg(src + 2 * i);
                b = __ldg(src + 2 * i + 1);
            }
            f[u][0] = a.x; f[u][1] = a.y; f[u][2] = a.z; f[u][3] = a.w;
            f[u][4] = b.x; f[u][5] = b.y; f[u][6] = b.z; f[u][7] = b.w;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float m = fabsf(f[u][k]);
                mx = fmaxf(mx, m <= 3.402823466e38f ? m : 0.0f);   // NaN and inf do not count
            }
        }
        const unsigned mb_w = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
        if (lane == 0 && mb_w != 0u) atomicMax(sm, mb_w);
        __syncthreads();
        const unsigned mb = *sm;
        const int e = static_cast<int>(mb >> 23);
        const int p = mb != 0u ? (e == 0 ? 126 : min(141 - e, 126)) : 0;
        const float pm = exp2i_e(p);
        uint8_t* blk = frag + static_cast<size_t>(v) * vb;
        if (threadIdx.x == 0) *reinterpret_cast<int4*>(blk) = make_int4(p, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kSplitItems; ++u) {
            const int i = threadIdx.x + u * kSplitThreads;
            if (i >= n_items) continue;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float f0 = __fmul_rn(f[u][2 * k], pm), f1 = __fmul_rn(f[u][2 * k + 1], pm);
                hi[k] = pack_f16x2_e(f0, f1);
                const float2 h = f16x2_to_f32x2(hi[k]);
                lo[k] = pack_f16x2_e(__fsub_rn(f0, h.x), __fsub_rn(f1, h.y));
            }
            uint4* d = reinterpret_cast<uint4*>(blk + 16 + 128 * (i >> 2) + 16 * (i & 3));
            d[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            d[4] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    }
    if (!wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Plan arrays written by the routing plan kernel (moe.cu).
struct PlanRef {
    int32_t* hdr;             // [1] = number of touched experts; [4], [5] = the
                              // pass's segment claim and finished-CTA counters
    const int32_t* offsets;   // [E + 1]
    const int32_t* touched;   // [touched]
    const int32_t* pair_of;   // pairs grouped by expert
};

// Shared memory (offsets from a 1024-byte aligned base).  Two scale buffers
// (the next segment's rows arrive while this one runs); the partial sums of a
// segment reuse its scale buffer once every warp is done with the scales.
struct ELayout {
    uint32_t xf, sc, sc_bytes, lut, misc, segst, bars, ring, total;
};
__host__ __device__ inline ELayout e_layout(int NM, int gpr, int n_experts) {
    ELayout l;
    l.xf = 0;                                                          // [4][frag_block(gpr)]
    l.sc = l.xf + kTokSeg * frag_block(gpr);                           // [2][NM][sc_bytes]
    l.sc_bytes = (static_cast<uint32_t>(ru_seg(NM) * kRowsUE) * gpr + 32u + 15u) & ~15u;
    const uint32_t part_bytes = kWarpsE * kRowsUE * kTokSeg * 4;      // [warps][32][4] f32
    const uint32_t buf = NM * l.sc_bytes > part_bytes ? NM * l.sc_bytes : part_bytes;
    l.sc_bytes = buf / NM;   // (>= the scale rows; the buffer also holds the partial sums)
    l.sc_bytes = (l.sc_bytes + 15u) & ~15u;
    l.lut = l.sc + 2 * NM * l.sc_bytes;                                // [256] f32
    l.misc = l.lut + 1024;   // -, pairs[2][4], lead[4], 16 zeros, -, meta[2][8]
    l.segst = l.misc + 192;                                           // [touched + 1] int
    l.bars = (l.segst + 4u * (static_cast<uint32_t>(n_experts) + 1u) + 7u) & ~7u;
    l.ring = (l.bars + (kWarpsE * kStagesE + 3) * 8 + 1023u) & ~1023u;
    l.total = l.ring + kWarpsE * kStagesE * kStageE + 1024;           // + alignment slack
    return l;
}

// The code planes of a bank's segments as 3-D byte tensors [slots][rows][cols/2]
// (one tensor map per segment; those past the bank's segment count unused).
struct BankMaps {
    CUtensorMap m[kMaxSegments];
};

// NM = 2: the gate/up pass (matrices gate, up; vector = the token's x),
// NM = 1: the down pass (matrix down; vector = the pair's act row).
template <int NM>
__global__ void __launch_bounds__(kThreadsE, 1)
    k_moe_tc(const __grid_constant__ BankMaps tm0, const __grid_constant__ BankMaps tm1,
             const Bank bank0, const Bank bank1, int rows, int cols, int top_k, int n_experts,
             const uint8_t* __restrict__ frag, PlanRef plan, MoeAct epi, float* __restrict__ out) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int gpr = cols / kGroup;
    const ELayout L = e_layout(NM, gpr, n_experts);
    const uint32_t vb = frag_block(gpr);   // one pair's fragment block in xf
    float* lut = reinterpret_cast<float*>(smem + L.lut);
    // per segment, double-buffered (buffer = the CTA's segment count mod 2, so
    // that the next segment's are set while this one runs): the pair ids
    int* spair = reinterpret_cast<int*>(smem + L.misc + 32);            // [2][4]
    int* lead = reinterpret_cast<int*>(smem + L.misc + 64);             // [2 buffers][2 matrices]
    const uint32_t zero16 = smem_u32(smem + L.misc + 80);               // 16 zero bytes
    int* segmeta = reinterpret_cast<int*>(smem + L.misc + 112);   // [2][u, e, b0, n_e, s, -, -, -]
    int* segst = reinterpret_cast<int*>(smem + L.segst);
    uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + L.bars);       // [2 buffers]
    uint64_t* xbar = sbar + 2;                                          // the fragment blocks
    uint64_t* ring_bars = sbar + 3;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const size_t plane = static_cast<size_t>(rows) * cols / 2;
    constexpr int kSegRows = ru_seg(NM) * kRowsUE;
    const int n_blocks = (rows + kSegRows - 1) / kSegRows;
    const int n_c = (gpr + kChunkE - 1) / kChunkE;
    const uint64_t policy = l2_evict_first();

    // launched dependent on the previous kernel of the layer (programmatic
    // dependent launch): let the next one be scheduled, set up, then wait for
    // the previous kernel's plan / activations before reading them
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid < 256) lut[tid] = e8m0_to_f32(static_cast<uint32_t>(tid));
    if (tid < 4) reinterpret_cast<uint32_t*>(smem + L.misc + 80)[tid] = 0u;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
        mbar_init(&sbar[0], 1);
        mbar_init(&sbar[1], 1);
        mbar_init(xbar, 1);
        for (int i = 0; i < kWarpsE * kStagesE; ++i) mbar_init(&ring_bars[i], 1);
        fence_mbar_init();
        // segments are claimed in order from a counter of the workspace (zeroed by
        // the plan and again by the last CTA of each pass), so that CTAs that
        // start late or run slow take fewer: this CTA's first two
        const int c0 = atomicAdd(plan.hdr + 4, 2);
        segmeta[4] = c0;
        segmeta[8 + 4] = c0 + 1;
    }
    // segst: the first segment of each touched expert (ceil(pairs / 4) x row
    // blocks each), a prefix sum over the touched experts, thread t taking
    // experts 2t and 2t + 1 (at most 1024 of them)
    const int n_touched = plan.hdr[1];
    int n_seg;
    {
        int* wtot = reinterpret_cast<int*>(smem + L.xf);   // [16] (xf is not in use yet)
        int eu[2], bu[2], nu[2], cu[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int u = 2 * tid + k;
            eu[k] = bu[k] = nu[k] = cu[k] = 0;
            if (u < n_touched) {
                eu[k] = __ldg(plan.touched + u);
                bu[k] = __ldg(plan.offsets + eu[k]);
                nu[k] = __ldg(plan.offsets + eu[k] + 1) - bu[k];
                cu[k] = (nu[k] + kTokSeg - 1) / kTokSeg * n_blocks;
            }
        }
        const int tsum = cu[0] + cu[1];
        int incl = tsum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane == 31) wtot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int v = lane < kWarpsE ? wtot[lane] : 0;
#pragma unroll
            for (int d = 1; d < kWarpsE; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, v, d);
                if (lane >= d) v += o;
            }
            __syncwarp();
            if (lane < kWarpsE) wtot[lane] = v;
        }
        __syncthreads();
        const int excl = (warp > 0 ? wtot[warp - 1] : 0) + incl - tsum;
        n_seg = wtot[kWarpsE - 1];
        if (tid == 0) segst[0] = 0;
        int lo = excl;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int u = 2 * tid + k;
            if (u < n_touched) {
                segst[u + 1] = lo + cu[k];
                // the meta slots of this CTA's first two segments
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int sq = segmeta[q * 8 + 4];
                    if (sq >= lo && sq < lo + cu[k]) {
                        segmeta[q * 8 + 0] = u;
                        segmeta[q * 8 + 1] = eu[k];
                        segmeta[q * 8 + 2] = bu[k];
                        segmeta[q * 8 + 3] = nu[k];
                    }
                }
            }
            lo += cu[k];
        }
    }
    __syncthreads();
    // (thread 0) the segment after next: claimed and looked up while this one
    // runs, each load issued in one phase and used in a later one, so that they
    // wait on nothing (claim; touched index and id; first pair and count)
    int la_s = n_seg, la_u = segmeta[8 + 4] < n_seg ? segmeta[8] : 0, la_e = 0, la_b0 = 0,
        la_b1 = 0;
    uint64_t* bars = ring_bars + warp * kStagesE;
    uint8_t* ring = smem + L.ring + static_cast<size_t>(warp) * kStagesE * kStageE;

    // A segment as this warp sees it.
    struct Seg {
        int e, sg, z, beg, npair, row0, nrow, n_ru, WK, m, my_ru, c_lo, n_units;
        bool active;
    };
    // segment s from its expert's entry in meta slot `slot`
    // this warp's share of a segment of n_ru row units: (active, row unit, first
    // chunk, chunk count); the full segments' once, the last row block's when met
    struct Share {
        bool active;
        int WK, my_ru, c_lo, n_units;
    };
    auto share_of = [&](int n_ru) {
        Share h;
        h.WK = min(n_c, kWarpsE / (NM * n_ru));
        h.active = warp < NM * n_ru * h.WK;
        const int qq = warp / NM;
        h.my_ru = qq % n_ru;
        const int kk = qq / n_ru;
        h.c_lo = h.active ? kk * n_c / h.WK : 0;
        h.n_units = h.active ? (kk + 1) * n_c / h.WK - h.c_lo : 0;
        return h;
    };
    const Share full_share = share_of(ru_seg(NM));
    auto seg_of = [&](int s, int slot) {
        Seg q{};
        if (s >= n_seg) return q;   // none: no units
        const int* m = segmeta + slot * 8;
        const int u = m[0], b0 = m[2], n_e = m[3];
        q.e = m[1];
        // the expert's bank segment and its plane in that segment (both banks of
        // a pass are split alike)
        q.sg = bank0.n_seg == 1 ? 0 : q.e / bank0.seg_slots;
        q.z = q.e - q.sg * bank0.seg_slots;
        const int rel = s - segst[u];
        const int ck = rel / n_blocks, b = rel - ck * n_blocks;
        q.beg = b0 + ck * kTokSeg;
        q.npair = min(kTokSeg, n_e - ck * kTokSeg);
        q.row0 = b * kSegRows;
        q.nrow = min(kSegRows, rows - q.row0);
        q.n_ru = (q.nrow + kRowsUE - 1) / kRowsUE;
        q.m = warp % NM;
        const Share h = q.n_ru == ru_seg(NM) ? full_share : share_of(q.n_ru);
        q.WK = h.WK;
        q.active = h.active;
        q.my_ru = h.my_ru;
        q.c_lo = h.c_lo;
        q.n_units = h.n_units;
        return q;
    };
    // this warp's unit k of segment q into stage st (lane 0): expert slot q.e is
    // plane q.e % seg_slots of its bank segment's tensor map
    auto issue = [&](const Seg& q, int k, int st) {
        const int x = (q.c_lo + k) * kChunkE * kGroupBytes;
        const int y = q.row0 + q.my_ru * kRowsUE;
        mbar_arrive_expect_tx(&bars[st], kStageE);
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(
                smem_u32(ring + st * kStageE)),
            "l"(q.m == 0 ? &tm0.m[q.sg] : &tm1.m[q.sg]), "r"(x), "r"(y), "r"(q.z),
            "r"(smem_u32(&bars[st])), "l"(policy)
            : "memory");
    };
    // the scale rows of segment q into buffer bi (thread 0): one bulk copy per matrix
    auto issue_scales = [&](const Seg& q, int bi) {
        uint32_t total = 0;
        uint32_t sz[NM];
        const uint8_t* a0[NM];
        for (int mm = 0; mm < NM; ++mm) {
            const Bank& bk = mm == 0 ? bank0 : bank1;
            const uint8_t* src = bk.seg[q.sg] + static_cast<size_t>(q.z) * bk.stride + plane +
                                 static_cast<size_t>(q.row0) * gpr;
            a0[mm] = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(src) &
                                                      ~static_cast<uintptr_t>(15));
            lead[bi * 2 + mm] = static_cast<int>(src - a0[mm]);
            sz[mm] = (static_cast<uint32_t>(lead[bi * 2 + mm] + q.nrow * gpr) + 15u) & ~15u;
            total += sz[mm];
        }
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&sbar[bi], total);
        for (int mm = 0; mm < NM; ++mm)
            bulk_g2s(smem + L.sc + (bi * NM + mm) * L.sc_bytes, a0[mm], sz[mm], &sbar[bi], policy);
    };

    // the fragment blocks of segment q's pairs (ids pr) into xf (thread 0): one
    // bulk copy per pair, kept in L2 (every segment of the pair's expert reads them)
    const uint64_t keep = l2_evict_last();
    auto issue_frags = [&](const Seg& q, const int* pr) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(q.npair) * vb);
        for (int k = 0; k < q.npair; ++k) {
            const size_t v = NM == 2 ? static_cast<size_t>(pr[k] / top_k) : static_cast<size_t>(pr[k]);
            bulk_g2s(smem + L.xf + k * vb, frag + v * vb, vb, xbar, keep);
        }
    };
    int kglob = 0;      // this warp's units consumed so far (ring phase)
    int issued = 0;     // this warp's units issued so far (lane 0): never more than kglob + stages
    int nseg_cta = 0;   // segments this CTA has taken so far (buffers and phases)
    bool failed = false;
    int s_cur = segmeta[4];
    Seg cur = seg_of(s_cur, 0);
    int sc_pend = -1;   // (thread 0) buffer of a scale copy not yet seen complete
    uint32_t sc_pend_par = 0;
    bool x_pend = false;   // (thread 32) a fragment copy not yet seen complete
    uint32_t x_pend_par = 0;
    if (tid == 0 && s_cur < n_seg) {
        issue_scales(cur, 0);
        sc_pend = 0;
    }
    if (tid == 32 && s_cur < n_seg) {
        int pr[kTokSeg];
        for (int k = 0; k < cur.npair; ++k) pr[k] = plan.pair_of[cur.beg + k];
        issue_frags(cur, pr);
        x_pend = true;
    }
    if (tid < kTokSeg) spair[tid] = tid < cur.npair ? plan.pair_of[cur.beg + tid] : 0;
    __syncthreads();

    for (int s = s_cur; s < n_seg; ++nseg_cta) {
        const int bi = nseg_cta & 1;
        const int s_nxt = segmeta[(bi ^ 1) * 8 + 4];
        const Seg nxt = seg_of(s_nxt, bi ^ 1);
        // the next unit of this warp's stream (this segment's, then the next one's)
        auto issue_next = [&]() {
            const int j = issued - kglob;
            if (j < cur.n_units)
                issue(cur, j, issued % kStagesE);
            else
                issue(nxt, j - cur.n_units, issued % kStagesE);
            ++issued;
        };
        const int stream_end = kglob + cur.n_units + nxt.n_units;

        // --- prologue, every warp for itself (no barrier: the last segment's
        // epilogue reads only its partial sums and pair ids, which nothing
        // before this segment's final barrier overwrites)
        const int* sp = spair + bi * kTokSeg;
        // the next segment's pair ids: requested now, stored after this one's
        // units (spair[bi ^ 1] may still be read by the last epilogue's stores)
        const int nxt_pair =
            warp == 1 && lane < nxt.npair ? plan.pair_of[nxt.beg + lane] : 0;   // lanes < 4
        int la_step = 0;   // (thread 0) 1: touched index and id looked up, 2: first pair and count
        if (tid == 0) la_s = atomicAdd(plan.hdr + 4, 1);
        // column sets of this segment: NP >= its pairs
        const int np = cur.npair <= 1 ? 1 : cur.npair <= 2 ? 2 : 4;
        // weights: fill the ring (some units may have been issued already)
        if (lane == 0) {
            fence_proxy_async_smem();
            while (issued < kglob + kStagesE && issued < stream_end) issue_next();
        }
        // this segment's fragment blocks (copied at the end of the last one) and
        // its scale rows (the lanes of a warp agree on the outcome)
        const bool landed = mbar_wait(xbar, static_cast<uint32_t>(nseg_cta) & 1u, kWaitE) &&
                            mbar_wait(&sbar[bi], static_cast<uint32_t>(nseg_cta >> 1) & 1u, kWaitE);
        failed = failed || !__all_sync(0xffffffffu, landed);
        if (tid == 0 && !failed) sc_pend = -1;
        if (tid == 32 && !failed) x_pend = false;
        const uint8_t* scm = smem + L.sc + (bi * NM + cur.m) * L.sc_bytes + lead[bi * 2 + cur.m];
        // "Plain" scale bytes (1 .. 200): 2^(k-127) is the float with bits k << 23
        // and the rows' sums may stay in the 2^p domain (|sum| below 128*32 * 6 *
        // 2^(200-127) * 2^15).  A warp with any other byte among its units' (lane
        // l: row 32 ru + l of its matrix over its chunk range) takes the table and
        // 2^-p per group.  Per byte b, in bit 7: b == 0 (the borrow of b - 1 with
        // b's own top bit clear) or b > 200 (top bit set and its low seven bits +
        // 55 reaching 128); no carry crosses a byte.
        bool odd = false;
        if (!failed && cur.active) {
            const int r = cur.my_ru * kRowsUE + lane;
            const int g0 = cur.c_lo * kChunkE;
            const int ng = min(gpr, (cur.c_lo + cur.n_units) * kChunkE) - g0;
            if (r < cur.nrow) {
                const uintptr_t a = reinterpret_cast<uintptr_t>(scm + r * gpr + g0);
                const uint32_t* wp = reinterpret_cast<const uint32_t*>(a & ~static_cast<uintptr_t>(3));
                const uint32_t sh = 8u * static_cast<uint32_t>(a & 3u);
                uint32_t flag = 0u, w0 = wp[0];
#pragma unroll 4
                for (int o = 0; o < ng; o += 4) {
                    const uint32_t w1 = wp[(o >> 2) + 1];
                    uint32_t w = __funnelshift_r(w0, w1, sh);
                    w0 = w1;
                    const int left = ng - o;   // bytes of the row left; past them: 1s
                    if (left < 4)
                        w = (w & (0xFFFFFFFFu >> (8 * (4 - left)))) | (0x01010101u << (8 * left));
                    flag |= ((w - 0x01010101u) & ~w) | (((w & 0x7F7F7F7Fu) + 0x37373737u) & w);
                }
                odd = (flag & 0x80808080u) != 0u;
            }
        }
        // pair q's power of two (the head of its fragment block; 0 for column
        // sets past the segment's pairs)
        auto p_of = [&](int q) {
            return q < cur.npair ? *reinterpret_cast<const int*>(smem + L.xf + q * vb) : 0;
        };
        // this warp's units in the 2^p domain: no odd scale byte, every pair's p >= 0
        bool fast = !__any_sync(0xffffffffu, odd);
#pragma unroll
        for (int q = 0; q < kTokSeg; ++q) fast = fast && p_of(q) >= 0;

        // --- this warp's units
        float acc[4] = {0.f, 0.f, 0.f, 0.f};   // rows g, g+8, g+16, g+24, this lane's groups
        const int slot = t / np, tok = t % np;   // D columns 2t, 2t + 1: group slot, pair
        const float pinv = exp2i_e(-p_of(tok));
        // B: lanes 8 np s .. 8 np s + 8 np - 1 hold the fragment of group slot s,
        // lanes 8 q .. 8 q + 7 of them pair q's (the last pair's for column sets
        // past the segment's pairs, whose D columns are not used)
        const int b_slot = lane / (8 * np);
        const int b_pair = min((lane % (8 * np)) >> 3, cur.npair - 1);
        const uint32_t xf_lane = smem_u32(smem + L.xf) + static_cast<uint32_t>(b_pair) * vb + 16u +
                                 static_cast<uint32_t>(lane & 7) * 16u;
        // the groups of a unit, GP to an accumulator
        auto unit_groups = [&](auto gp_c, auto fast_c, uint32_t row_addr, int gc0, int ngc,
                               const uint32_t (&sb)[4][2]) {
            constexpr int GP = decltype(gp_c)::value;
            constexpr bool FAST = decltype(fast_c)::value;
#pragma unroll
            for (int j0 = 0; j0 < kChunkE; j0 += GP) {
                if (j0 < ngc) {
                    float d0[4], d1[4];   // rows g, g+8 and g+16, g+24
#pragma unroll
                    for (int sl = 0; sl < GP; ++sl) {
                        const int j = j0 + sl;
                        if (j < ngc) {
                            uint32_t cwd[4];   // code word t of rows g, g+8, g+16, g+24
                            ldsm_x4(row_addr ^ static_cast<uint32_t>(j << 4), cwd);
                            uint32_t h0[4], h1[4], h2[4], h3[4];
                            e2m1x8_to_f16x2x4(cwd[0], h0);
                            e2m1x8_to_f16x2x4(cwd[1], h1);
                            e2m1x8_to_f16x2x4(cwd[2], h2);
                            e2m1x8_to_f16x2x4(cwd[3], h3);
                            const uint4 bf = lds128(
                                b_slot == sl ? xf_lane + static_cast<uint32_t>(gc0 + j) * 128u : zero16);
                            if (sl == 0) {
                                mma16816_z(d0, h0[0], h1[0], h0[1], h1[1], bf.x, bf.y);
                                mma16816_z(d1, h2[0], h3[0], h2[1], h3[1], bf.x, bf.y);
                            } else {
                                mma16816(d0, h0[0], h1[0], h0[1], h1[1], bf.x, bf.y);
                                mma16816(d1, h2[0], h3[0], h2[1], h3[1], bf.x, bf.y);
                            }
                            mma16816(d0, h0[2], h1[2], h0[3], h1[3], bf.z, bf.w);
                            mma16816(d1, h2[2], h3[2], h2[3], h3[3], bf.z, bf.w);
                        }
                    }
                    if (j0 + slot < ngc) {   // this lane's group j0 + slot
                        const int hw = j0 >> 2;
                        const float v[4] = {__fadd_rn(d0[0], d0[1]), __fadd_rn(d0[2], d0[3]),
                                            __fadd_rn(d1[0], d1[1]), __fadd_rn(d1[2], d1[3])};
                        if constexpr (FAST) {   // 2^(k-127) from its bits; 2^-p at the end
                            const uint32_t sel = 0x4044u + (static_cast<uint32_t>((j0 & 3) + slot) << 8);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                acc[q] = __fmaf_rn(__uint_as_float(__byte_perm(sb[q][hw], 0u, sel) << 7),
                                                   v[q], acc[q]);
                        } else {                // any byte: the table, and 2^-p first
                            const uint32_t sel = 0x4440u + static_cast<uint32_t>((j0 & 3) + slot);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                acc[q] = __fmaf_rn(lut[__byte_perm(sb[q][hw], 0u, sel)],
                                                   __fmul_rn(v[q], pinv), acc[q]);
                        }
                    }
                }
            }
        };
        int k = 0;
        for (; k < cur.n_units && !failed; ++k) {
            const int kg = kglob + k, st = kg % kStagesE;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&bars[st], static_cast<uint32_t>(kg / kStagesE) & 1u, kWaitE))) {
                failed = true;
                break;
            }
            const uint8_t* stg = ring + st * kStageE;
            // this lane's row (lane) of the tile, chunk 0 after the 128-byte swizzle;
            // chunk j is at that address ^ (j << 4) (the tile is 1024-byte aligned)
            const uint32_t row_addr = smem_u32(stg) + lane * 128 + ((lane & 7) << 4);
            const int gc0 = (cur.c_lo + k) * kChunkE;
            const int ngc = min(kChunkE, gpr - gc0);
            uint32_t sb[4][2];   // 8 scale bytes of rows g, g+8, g+16, g+24 (any alignment)
#pragma unroll
            for (int r4 = 0; r4 < 4; ++r4) {
                const uint32_t a = static_cast<uint32_t>((cur.my_ru * kRowsUE + g + 8 * r4) * gpr + gc0);
                const uint32_t* wp = reinterpret_cast<const uint32_t*>(
                    reinterpret_cast<uintptr_t>(scm + a) & ~static_cast<uintptr_t>(3));
                const uint32_t sh = 8u * (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(scm + a)) & 3u);
                const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2];
                sb[r4][0] = __funnelshift_r(w0, w1, sh);
                sb[r4][1] = __funnelshift_r(w1, w2, sh);
            }
            if (fast) {
                if (np == 1)
                    unit_groups(std::integral_constant<int, 4>{}, std::true_type{}, row_addr, gc0, ngc, sb);
                else if (np == 2)
                    unit_groups(std::integral_constant<int, 2>{}, std::true_type{}, row_addr, gc0, ngc, sb);
                else
                    unit_groups(std::integral_constant<int, 1>{}, std::true_type{}, row_addr, gc0, ngc, sb);
            } else {
                if (np == 1)
                    unit_groups(std::integral_constant<int, 4>{}, std::false_type{}, row_addr, gc0, ngc, sb);
                else if (np == 2)
                    unit_groups(std::integral_constant<int, 2>{}, std::false_type{}, row_addr, gc0, ngc, sb);
                else
                    unit_groups(std::integral_constant<int, 1>{}, std::false_type{}, row_addr, gc0, ngc, sb);
            }
            __syncwarp();   // every lane is done with the stage
            if (lane == 0 && issued < stream_end) {   // refill: this segment's or the next one's
                fence_proxy_async_smem();
                issue_next();
            }
            // (thread 0) the segment after next, one dependent step per unit
            if (tid == 0 && la_s < n_seg && la_step < 2) {
                if (la_step == 0) {
                    while (segst[la_u + 1] <= la_s) ++la_u;
                    la_e = __ldg(plan.touched + la_u);
                } else {
                    la_b0 = __ldg(plan.offsets + la_e);
                    la_b1 = __ldg(plan.offsets + la_e + 1);
                }
                ++la_step;
            }
        }
        if (failed) {
            // let this warp's copies in flight land before the CTA can exit
            for (int kq = kglob + k; kq < issued; ++kq)
                mbar_wait(&bars[kq % kStagesE], static_cast<uint32_t>(kq / kStagesE) & 1u, kWaitE);
        }
        kglob += cur.n_units;
        if (tid == 0) {   // the segment after next, for the next iteration
            if (la_s < n_seg) {
                if (la_step < 1) {
                    while (segst[la_u + 1] <= la_s) ++la_u;
                    la_e = __ldg(plan.touched + la_u);
                }
                if (la_step < 2) {
                    la_b0 = __ldg(plan.offsets + la_e);
                    la_b1 = __ldg(plan.offsets + la_e + 1);
                }
                segmeta[bi * 8 + 0] = la_u;
                segmeta[bi * 8 + 1] = la_e;
                segmeta[bi * 8 + 2] = la_b0;
                segmeta[bi * 8 + 3] = la_b1 - la_b0;
            }
            segmeta[bi * 8 + 4] = la_s;
        }
        // every warp is done with the scales and xf and past the last epilogue
        failed = __syncthreads_or(failed) != 0;
        if (warp == 1 && lane < kTokSeg) spair[(bi ^ 1) * kTokSeg + lane] = nxt_pair;
        int nxt_pr[kTokSeg];   // (warp 1) the next segment's pair ids
#pragma unroll
        for (int q = 0; q < kTokSeg; ++q) nxt_pr[q] = __shfl_sync(0xffffffffu, nxt_pair, q);
        // the next segment's scale rows go to the other buffer (thread 0), its
        // pairs' fragment blocks to xf (thread 32), side by side
        if (!failed && s_nxt < n_seg) {
            if (tid == 0) {
                issue_scales(nxt, bi ^ 1);
                sc_pend = bi ^ 1;
                sc_pend_par = static_cast<uint32_t>((nseg_cta + 1) >> 1) & 1u;
            } else if (tid == 32) {
                issue_frags(nxt, nxt_pr);
                x_pend = true;
                x_pend_par = static_cast<uint32_t>(nseg_cta + 1) & 1u;
            }
        }
        float* part = reinterpret_cast<float*>(smem + L.sc + bi * NM * L.sc_bytes);
        // pair n: the slots' sums in lanes (g, s np + n), added in slot order into lane (g, n)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float v = acc[q];
            for (int sl = 1; sl < 4 / np; ++sl)
                v = __fadd_rn(v, __shfl_sync(0xffffffffu, acc[q], (lane & ~3) | (sl * np + tok)));
            acc[q] = v;
        }
        if (fast) {   // back from the 2^p domain (a power of two: exact)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = __fmul_rn(acc[q], pinv);
        }
        if (cur.active && t < np) {   // lane (g, t) has pair t
            float* pw = part + static_cast<size_t>(warp) * kRowsUE * kTokSeg;
            pw[g * kTokSeg + t] = acc[0];
            pw[(g + 8) * kTokSeg + t] = acc[1];
            pw[(g + 16) * kTokSeg + t] = acc[2];
            pw[(g + 24) * kTokSeg + t] = acc[3];
        }
        __syncthreads();
        // --- chunk ranges in order (warp (kk * n_ru + ru) * NM + m), then the epilogue
        for (int i = tid; i < cur.n_ru * kRowsUE * kTokSeg; i += kThreadsE) {
            const int ru = i / (kRowsUE * kTokSeg), rem = i - ru * kRowsUE * kTokSeg;
            const int tok = rem % kTokSeg, row = cur.row0 + ru * kRowsUE + rem / kTokSeg;
            float v[NM];
#pragma unroll
            for (int mm = 0; mm < NM; ++mm) {
                float sacc = part[static_cast<size_t>(ru * NM + mm) * kRowsUE * kTokSeg + rem];
                for (int qq = 1; qq < cur.WK; ++qq)
                    sacc = __fadd_rn(sacc, part[static_cast<size_t>((qq * cur.n_ru + ru) * NM + mm) *
                                                    kRowsUE * kTokSeg + rem]);
                v[mm] = sacc;
            }
            if (row < rows && tok < cur.npair) {
                const size_t o = static_cast<size_t>(sp[tok]) * rows + row;
                if constexpr (NM == 2)
                    out[o] = moe_act(v[0], v[1], epi, sp[tok]);
                else
                    out[o] = v[0];
            }
        }
        if (failed) break;   // the same in every thread
        cur = nxt;
        s = s_nxt;
    }
    // a failed CTA may still have copies of a next segment in flight: wait for them
    if (failed) {
        __syncthreads();
        if (lane == 0)
            for (int kq = kglob; kq < issued; ++kq)
                mbar_wait(&bars[kq % kStagesE], static_cast<uint32_t>(kq / kStagesE) & 1u, kWaitE);
        if (tid == 0 && sc_pend >= 0) mbar_wait(&sbar[sc_pend], sc_pend_par, kWaitE);
        if (tid == 32 && x_pend) mbar_wait(xbar, x_pend_par, kWaitE);
    }
    if (failed && lane == 0) atomicOr(&g_fault_moetc, 1);
    // the last CTA to finish zeroes the claim counters for the next pass (every
    // CTA's claims come before its count)
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(plan.hdr + 5, 1) == static_cast<int>(gridDim.x) - 1) {
            __threadfence();
            plan.hdr[4] = 0;
            plan.hdr[5] = 0;
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_e() {
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

// The code planes of one bank segment as a 3-D byte tensor [slots][rows][cols/2]
// (the slot stride is the padded matrix size), tiles of 32 rows x 128 bytes.
bool bank_map(CUtensorMap* map, const uint8_t* bank, size_t stride, int n_experts, int rows,
              int cols) {
    auto fn = encode_fn_e();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols) / 2, static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(n_experts)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) / 2,
                                   static_cast<cuuint64_t>(stride)};
    const cuuint32_t box[3] = {128, kRowsUE, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(bank), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count_e() {
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

// Checks and tensor maps first (cudaErrorNotSupported with nothing launched),
// then `before` (the routing plan of the gate/up pass), the vectors' split and
// the pass, each launched dependent on the kernel before it.
template <int NM>
cudaError_t launch_e(const Bank& bank0, const Bank& bank1, int n_experts, int rows, int cols,
                     int top_k, const float* vec, int n_vec, uint8_t* frag,
                     const std::function<cudaError_t()>& before, PlanRef plan, MoeAct epi,
                     float* out, cudaStream_t s) {
    const int gpr = cols / kGroup;
    if (gpr > kGMaxE || n_experts > kMaxExpertsE) return cudaErrorNotSupported;
    const ELayout l = e_layout(NM, gpr, n_experts);
    if (l.total > kSmemMaxE) return cudaErrorNotSupported;
    auto kernel = k_moe_tc<NM>;
    {
        static PerDevice memo;
        const cudaError_t attr_err = static_cast<cudaError_t>(memo.get([&] {
            return static_cast<int>(cudaFuncSetAttribute(
                kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemMaxE)));
        }));
        if (attr_err != cudaSuccess) return attr_err;
    }
    BankMaps m0{}, m1{};
    for (int i = 0; i < bank0.n_seg; ++i)
        if (!bank_map(&m0.m[i], bank0.seg[i], bank0.stride, bank0.seg_slots, rows, cols))
            return cudaErrorNotSupported;
    if (NM == 2) {
        for (int i = 0; i < bank1.n_seg; ++i)
            if (!bank_map(&m1.m[i], bank1.seg[i], bank1.stride, bank1.seg_slots, rows, cols))
                return cudaErrorNotSupported;
    }
    cudaError_t e = cudaSuccess;
    if (before) {
        e = before();
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    const int sms = sm_count_e();
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(n_vec < 4 * sms ? n_vec : 4 * sms));
        cfg.blockDim = dim3(kSplitThreads);
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // the gate/up pass's x is an input (complete before the plan started);
        // the down pass's act comes from the previous kernel
        e = cudaLaunchKernelEx(&cfg, k_moe_split, vec, n_vec, cols, frag, NM == 1 ? 1 : 0);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(kThreadsE);
    cfg.dynamicSmemBytes = l.total;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, m0, m1, bank0, bank1, rows, cols, top_k, n_experts,
                           static_cast<const uint8_t*>(frag), plan, epi, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

size_t moe_frag_bytes(int n_vec, int cols) {
    return static_cast<size_t>(n_vec) * frag_block(cols / kGroup);
}

cudaError_t launch_moe_tc_gate_up(const Bank& gate, const Bank& up, int n_experts, int inter,
                                  int hidden, int top_k, const float* x, int n_tokens,
                                  uint8_t* frag, const std::function<cudaError_t()>& before,
                                  int32_t* hdr, const int32_t* offsets, const int32_t* touched,
                                  const int32_t* pair_of, MoeAct epi, float* act, cudaStream_t s) {
    return launch_e<2>(gate, up, n_experts, inter, hidden, top_k, x, n_tokens, frag, before,
                       PlanRef{hdr, offsets, touched, pair_of}, epi, act, s);
}

cudaError_t launch_moe_tc_down(const Bank& down, int n_experts, int hidden, int inter,
                               const float* act, int n_pairs, uint8_t* frag, int32_t* hdr,
                               const int32_t* offsets, const int32_t* touched,
                               const int32_t* pair_of, float* o_pairs, cudaStream_t s) {
    return launch_e<1>(down, down, n_experts, hidden, inter, 1, act, n_pairs, frag, nullptr,
                       PlanRef{hdr, offsets, touched, pair_of}, MoeAct{nullptr, 0.0f, 0}, o_pairs,
                       s);
}

cudaError_t read_fault_moetc(int* value, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_fault_moetc, sizeof(int));
    if (e != cudaSuccess || !reset) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_moetc, &zero, sizeof(int));
}

}  // namespace mxk
