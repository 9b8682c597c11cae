// matmat_core.cuh -- the CTA-level FP32 group walk shared by the matvec, the
// small-batch product and the two routed-expert passes.
//
// It restates the per-lane loop of "cortiq-engine 0.8.40
// src/gpu_wgpu/mxfp4.rs" PEROP kernels mxfp4_mv / mxfp4_mm: lane l of a warp
// takes groups g = l, l+32, ...; for each it decodes the 32 codes once, dots
// them with every token's x over the group (group_dots: FP32 FMA chains over
// the even and the odd elements), and adds scale * dot to the token's row
// partial.  A CTA
// of kWarps warps stages the tokens' x in shared memory chunk by chunk and
// each warp carries R rows of NM matrices, so one x read from shared memory
// feeds R*NM rows and one decode feeds NB tokens.  The order of operations
// seen by a token does not depend on R, NM, NB or the chunk size.
#pragma once

#include "common.cuh"

namespace mxk {

constexpr int kWarps = 8;                   // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kXPad = 36;                   // floats per staged group (32 + 4):
                                            // 16-B lane reads at 144-B stride
                                            // fall in distinct banks
constexpr int kStageGroups = 256;           // staged groups per chunk * NB
constexpr size_t kStageBytes = kStageGroups * kXPad * sizeof(float);

// acc[m][i][t] gets the row partial of this lane; call warp_allreduce after.
// wm[m]: base of matrix m (code plane first, scale plane after it);
// row_w: first row of this warp (rows >= `rows` are skipped);
// xt[t]: the token vectors (16-B aligned, `cols` floats), nullptr = zero;
// xs: kStageBytes of shared memory.  Must be called by all kThreads threads.
template <int R, int NB, int NM>
__device__ __forceinline__ void cta_group_walk(const uint8_t* const (&wm)[NM], int rows,
                                               int cols, long row_w,
                                               const float* const (&xt)[NB], float* xs,
                                               float (&acc)[NM][R][NB]) {
    constexpr int KCG = kStageGroups / NB;   // groups per chunk, a multiple of 32
    const int gpr = cols / kGroup;
    const int lane = threadIdx.x & 31;
    const size_t code_bytes = static_cast<size_t>(rows) * cols / 2;

    for (int gc = 0; gc < gpr; gc += KCG) {
        const int ng = min(KCG, gpr - gc);
        __syncthreads();   // the previous chunk (or previous use of xs) is done
        for (int i = threadIdx.x; i < NB * ng * 8; i += kThreads) {
            const int t = i / (ng * 8);
            const int rem = i - t * ng * 8;
            const int g = rem >> 3, q = rem & 7;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            const float* src = xt[0];
#pragma unroll
            for (int u = 1; u < NB; ++u)
                if (t == u) src = xt[u];
            if (src != nullptr) {
                v = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(gc + g) *
                                                                    kGroup) + q);
            }
            *reinterpret_cast<float4*>(xs + (t * KCG + g) * kXPad + q * 4) = v;
        }
        __syncthreads();

        for (int gl = lane; gl < ng; gl += 32) {
            const int g = gc + gl;
            uint4 code[NM * R];
            float s[NM * R];
#pragma unroll
            for (int m = 0; m < NM; ++m)
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const long row = row_w + i;
                    if (row < rows) {
                        code[m * R + i] = ldg_stream(group_codes(wm[m], gpr, row, g));
                        s[m * R + i] =
                            e8m0_to_f32(group_scale_byte(wm[m] + code_bytes, gpr, row, g));
                    } else {
                        code[m * R + i] = make_uint4(0u, 0u, 0u, 0u);
                        s[m * R + i] = 0.0f;
                    }
                }
            const float* xp[NB];
#pragma unroll
            for (int t = 0; t < NB; ++t) xp[t] = xs + (t * KCG + gl) * kXPad;
            float dots[NM * R][NB];
            group_dots<NM * R, NB>(code, xp, dots);
#pragma unroll
            for (int m = 0; m < NM; ++m)
#pragma unroll
                for (int i = 0; i < R; ++i)
#pragma unroll
                    for (int t = 0; t < NB; ++t)
                        acc[m][i][t] = __fmaf_rn(s[m * R + i], dots[m * R + i][t], acc[m][i][t]);
        }
    }
}

// Butterfly sum over the 32 lanes (same tree for every value).
template <int NM, int R, int NB>
__device__ __forceinline__ void warp_allreduce(float (&acc)[NM][R][NB]) {
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int t = 0; t < NB; ++t)
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    acc[m][i][t] = __fadd_rn(acc[m][i][t],
                                             __shfl_xor_sync(0xffffffffu, acc[m][i][t], off));
}

template <int NM, int R, int NB>
__device__ __forceinline__ void zero(float (&acc)[NM][R][NB]) {
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int t = 0; t < NB; ++t) acc[m][i][t] = 0.0f;
}

}  // namespace mxk
