// moe.cu -- routed-expert passes over MXFP4 expert banks (sm_103a).
//
// Sources: "cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs" kernels
// dsv4_global_gate_up_mxfp4 (act = silu(gate.x) * (up.x) per routed pair) and
// dsv4_global_down_mxfp4 (down . act, weighted by the route weight and summed
// over the token's slots); "rlx-cpu 0.2.17 src/gguf_matmul.rs"
// grouped_moe_sort_plan (counting sort of the routed pairs by expert) and
// grouped_moe_unpermute_out (back to token order); "cortiq-engine 0.8.77
// src/qtensor/moe_fast.rs" (gate and up read once for all of an expert's
// tokens; act laid out [pair, inter]).
//
// Unlike the page's kernels, which walk every routed slot of every token and
// so read an expert's weights once per pair, the work here is grouped by
// expert: each touched expert's gate, up and down matrices are read once per
// call, their decode shared by all of the expert's pairs.
//
// Pipeline (all stream-ordered, no inter-CTA waits):
//   k_moe_plan_s    one CTA: counts, offsets, touched-expert list, pair lists
//                   (shared-memory scans; k_moe_plan beyond 4096 experts)
//   gate/up pass    k_moe_tc<2> (moe_tc.cu, tensor cores), else k_moe_pass
//   down pass       k_moe_tc<1>, else k_moe_pass -> per-pair outputs
//   k_moe_combine   y[t] = sum_j w[t,j] * o[t*top_k + j], slots in order
#include <mutex>

#include "matmat_core.cuh"
#include "kernels.h"

namespace mxk {
namespace {

// Workspace layout (all offsets 16-byte aligned; o_pairs and the fragment
// blocks 256-byte aligned).
struct WsLayout {
    size_t hdr, offsets, touched, pair_of, pair_slot, cold, o_pairs, frag_x, frag_a, total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// (hdr, offsets, touched, pair_of, pair_slot and cold depend on n_slots and
// the pair count only)
WsLayout ws_layout(int n_slots, int n_tokens, int top_k, int hidden, int inter) {
    const int n_pairs = n_tokens * top_k;
    WsLayout l;
    // int32[8]: invalid pairs, touched experts, cold pairs, -, the tensor-core
    // passes' segment claim counter and finished-CTA counter, -, -
    l.hdr = 0;
    l.offsets = 32;                                       // int32[slots + 1]
    l.touched = align_up(l.offsets + 4 * (static_cast<size_t>(n_slots) + 1), 16);
    l.pair_of = align_up(l.touched + 4 * static_cast<size_t>(n_slots), 16);
    l.pair_slot = align_up(l.pair_of + 4 * static_cast<size_t>(n_pairs), 16);   // int32[pairs]
    l.cold = align_up(l.pair_slot + 4 * static_cast<size_t>(n_pairs), 16);      // int32[pairs]
    l.o_pairs = align_up(l.cold + 4 * static_cast<size_t>(n_pairs), 256);
    // the tensor-core passes' B-fragment blocks: of each token's x, of each pair's act
    l.frag_x = align_up(l.o_pairs + 4 * static_cast<size_t>(n_pairs) * hidden, 256);
    l.frag_a = align_up(l.frag_x + moe_frag_bytes(n_tokens, hidden), 256);
    l.total = l.frag_a + moe_frag_bytes(n_pairs, inter);
    return l;
}

struct Plan {
    int32_t* hdr;
    int32_t* offsets;
    int32_t* touched;
    int32_t* pair_of;
    int32_t* pair_slot;   // the pair's bank slot; -1 invalid, -2 cold
    int32_t* cold;        // cold pairs, increasing
    float* o_pairs;
    uint8_t* frag_x;
    uint8_t* frag_a;
};

Plan plan_view(void* ws, int n_slots, int n_tokens, int top_k, int hidden, int inter) {
    const WsLayout l = ws_layout(n_slots, n_tokens, top_k, hidden, inter);
    char* b = static_cast<char*>(ws);
    return Plan{reinterpret_cast<int32_t*>(b + l.hdr), reinterpret_cast<int32_t*>(b + l.offsets),
                reinterpret_cast<int32_t*>(b + l.touched),
                reinterpret_cast<int32_t*>(b + l.pair_of),
                reinterpret_cast<int32_t*>(b + l.pair_slot),
                reinterpret_cast<int32_t*>(b + l.cold),
                reinterpret_cast<float*>(b + l.o_pairs),
                reinterpret_cast<uint8_t*>(b + l.frag_x),
                reinterpret_cast<uint8_t*>(b + l.frag_a)};
}

constexpr int32_t kSlotInvalid = -1, kSlotCold = -2;

// The bank slot of pair p: slot_of[id] (or the id itself without a table);
// ids outside [0, n_ids) and slots at or past n_slots are invalid, a negative
// table entry marks a cold expert.
__device__ __forceinline__ int32_t resolve_slot(const int32_t* __restrict__ ids,
                                                const int32_t* __restrict__ slot_of, int n_ids,
                                                int n_slots, int p) {
    const int32_t e = __ldg(ids + p);
    if (e < 0 || e >= n_ids) return kSlotInvalid;
    const int32_t s = slot_of ? __ldg(slot_of + e) : e;
    if (s < 0) return kSlotCold;
    return s < n_slots ? s : kSlotInvalid;
}

// Warp 0 lists the cold pairs in increasing order (a ballot per 32 pairs) and
// stores their count; the pair slots are visible to the whole CTA.
__device__ __forceinline__ void list_cold(int n_pairs, Plan plan) {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    int base = 0;
    for (int p0 = 0; p0 < n_pairs; p0 += 32) {
        const int p = p0 + lane;
        const bool c = p < n_pairs && plan.pair_slot[p] == kSlotCold;
        const unsigned m = __ballot_sync(0xffffffffu, c);
        if (c) plan.cold[base + __popc(m & ((1u << lane) - 1u))] = p;
        base += __popc(m);
    }
    if (lane == 0) plan.hdr[2] = base;
}

// ---------------------------------------------------------------------------
// Routing plan, one CTA.  Thread s counts and then lists the pairs of slot s
// (stable: increasing pair index), as the counting sort of
// grouped_moe_sort_plan does; thread 0 prefix-sums the counts.
__global__ void __launch_bounds__(1024) k_moe_plan(const int32_t* __restrict__ ids, int n_pairs,
                                                   int n_experts, const int32_t* __restrict__ slot_of,
                                                   int n_ids, Plan plan) {
    __shared__ int s_invalid;
    if (threadIdx.x == 0) s_invalid = 0;
    __syncthreads();
    int bad = 0;
    for (int p = threadIdx.x; p < n_pairs; p += blockDim.x) {
        const int32_t sl = resolve_slot(ids, slot_of, n_ids, n_experts, p);
        plan.pair_slot[p] = sl;
        bad += sl == kSlotInvalid ? 1 : 0;
    }
    if (bad) atomicAdd(&s_invalid, bad);
    __syncthreads();
    list_cold(n_pairs, plan);
    for (int e = threadIdx.x; e < n_experts; e += blockDim.x) {
        int count = 0;
        for (int p = 0; p < n_pairs; ++p) count += (plan.pair_slot[p] == e) ? 1 : 0;
        plan.offsets[e + 1] = count;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0, touched = 0;
        plan.offsets[0] = 0;
        for (int e = 0; e < n_experts; ++e) {
            const int c = plan.offsets[e + 1];
            if (c > 0) plan.touched[touched++] = e;
            run += c;
            plan.offsets[e + 1] = run;
        }
        plan.hdr[0] = s_invalid;
        plan.hdr[1] = touched;
        plan.hdr[4] = 0;
        plan.hdr[5] = 0;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n_experts; e += blockDim.x) {
        int pos = plan.offsets[e];
        for (int p = 0; p < n_pairs; ++p)
            if (plan.pair_slot[p] == e) plan.pair_of[pos++] = p;
    }
}

// The same plan with the counts, offsets and touched flags in shared memory
// (up to kPlanSmemExperts slots) and the pairs' slots too (up to
// kPlanSmemPairs pairs; beyond, read back from the workspace): counts by
// shared atomics, offsets and the touched list by block-wide exclusive scans,
// then each warp lists the pairs of its touched slots in increasing order, 32
// pairs per ballot.  The arrays it writes are those of k_moe_plan.
constexpr int kPlanSmemExperts = 4096;
constexpr int kPlanSmemPairs = 6144;   // with 4096 slots: 40 KB, under the 48 KB default

__global__ void __launch_bounds__(1024) k_moe_plan_s(const int32_t* __restrict__ ids, int n_pairs,
                                                     int n_experts,
                                                     const int32_t* __restrict__ slot_of, int n_ids,
                                                     Plan plan) {
    extern __shared__ int s_dyn[];   // [n_experts] counts, then [n_pairs] slots (if they fit)
    int* s_cnt = s_dyn;
    int* s_ps = s_dyn + n_experts;
    __shared__ int s_wsum[2][32];
    __shared__ int s_invalid;
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
    // the expert pass may be scheduled now; it waits for this plan to complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const bool ps_smem = n_pairs <= kPlanSmemPairs;
    const int32_t* ps = ps_smem ? s_ps : plan.pair_slot;
    for (int e = tid; e < n_experts; e += nt) s_cnt[e] = 0;
    if (tid == 0) s_invalid = 0;
    __syncthreads();
    int bad = 0;
    for (int p = tid; p < n_pairs; p += nt) {
        const int32_t sl = resolve_slot(ids, slot_of, n_ids, n_experts, p);
        plan.pair_slot[p] = sl;
        if (ps_smem) s_ps[p] = sl;
        if (sl == kSlotInvalid)
            ++bad;
        else if (sl >= 0)
            atomicAdd(&s_cnt[sl], 1);
    }
    if (bad) atomicAdd(&s_invalid, bad);
    __syncthreads();
    if (w == 0) {   // the cold pairs, increasing
        int base = 0;
        for (int p0 = 0; p0 < n_pairs; p0 += 32) {
            const int p = p0 + lane;
            const bool c = p < n_pairs && ps[p] == kSlotCold;
            const unsigned m = __ballot_sync(0xffffffffu, c);
            if (c) plan.cold[base + __popc(m & ((1u << lane) - 1u))] = p;
            base += __popc(m);
        }
        if (lane == 0) plan.hdr[2] = base;
    }
    // thread tid takes experts [e0, e1): its count and touched sums, scanned
    // across the warp, then across the warps
    const int per = (n_experts + nt - 1) / nt;
    const int e0 = min(tid * per, n_experts), e1 = min(e0 + per, n_experts);
    int c_sum = 0, f_sum = 0;
    for (int e = e0; e < e1; ++e) {
        c_sum += s_cnt[e];
        f_sum += s_cnt[e] > 0 ? 1 : 0;
    }
    int c_inc = c_sum, f_inc = f_sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int c = __shfl_up_sync(0xffffffffu, c_inc, d);
        const int f = __shfl_up_sync(0xffffffffu, f_inc, d);
        if (lane >= d) {
            c_inc += c;
            f_inc += f;
        }
    }
    if (lane == 31) {
        s_wsum[0][w] = c_inc;
        s_wsum[1][w] = f_inc;
    }
    __syncthreads();
    if (w == 0) {
        const int nw = nt >> 5;
        int c = lane < nw ? s_wsum[0][lane] : 0, f = lane < nw ? s_wsum[1][lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int cu = __shfl_up_sync(0xffffffffu, c, d);
            const int fu = __shfl_up_sync(0xffffffffu, f, d);
            if (lane >= d) {
                c += cu;
                f += fu;
            }
        }
        s_wsum[0][lane] = c;   // inclusive over warps 0 .. lane
        s_wsum[1][lane] = f;
    }
    __syncthreads();
    int c_run = c_inc - c_sum + (w > 0 ? s_wsum[0][w - 1] : 0);
    int f_run = f_inc - f_sum + (w > 0 ? s_wsum[1][w - 1] : 0);
    for (int e = e0; e < e1; ++e) {
        const int c = s_cnt[e];
        plan.offsets[e] = c_run;
        if (c > 0) plan.touched[f_run++] = e;
        s_cnt[e] = c_run;   // from here on: the first position of expert e
        c_run += c;
    }
    if (tid == nt - 1) {   // its range ends at n_experts: the totals
        plan.offsets[n_experts] = c_run;
        plan.hdr[0] = s_invalid;
        plan.hdr[1] = f_run;
        plan.hdr[4] = 0;
        plan.hdr[5] = 0;
    }
    __syncthreads();
    const int n_planned = plan.offsets[n_experts];
    const int nw = nt >> 5;
    for (int e = w; e < n_experts; e += nw) {   // warp w lists slots w, w + nw, ...
        int pos = s_cnt[e];
        const int end = e + 1 < n_experts ? s_cnt[e + 1] : n_planned;
        for (int p0 = 0; p0 < n_pairs && pos < end; p0 += 32) {
            const int p = p0 + lane;
            const bool mine = p < n_pairs && ps[p] == e;
            const unsigned m = __ballot_sync(0xffffffffu, mine);
            if (mine) plan.pair_of[pos + __popc(m & ((1u << lane) - 1u))] = p;
            pos += __popc(m);
        }
    }
}

// ---------------------------------------------------------------------------
// One chunk of up to NB pairs of expert e against NM matrices; `rows` rows,
// `cols` columns.  Epilogue by pass.
enum class Pass { kGateUp, kDown };

template <Pass P, int R, int NB>
__device__ __forceinline__ void expert_chunk(const uint8_t* const (&wm)[P == Pass::kGateUp ? 2 : 1],
                                             int rows, int cols, long row_w,
                                             const int32_t* pairs, int n, int top_k,
                                             const float* vec_base, float* out, float* xs,
                                             const MoeAct& epi) {
    constexpr int NM = P == Pass::kGateUp ? 2 : 1;
    const int lane = threadIdx.x & 31;
    const float* xt[NB];
    int pr[NB];
#pragma unroll
    for (int t = 0; t < NB; ++t) {
        pr[t] = t < n ? pairs[t] : 0;
        // gate/up reads the token's x; down reads the pair's act row
        const size_t vrow = P == Pass::kGateUp ? static_cast<size_t>(pr[t] / top_k)
                                               : static_cast<size_t>(pr[t]);
        xt[t] = t < n ? vec_base + vrow * cols : nullptr;
    }
    float acc[NM][R][NB];
    zero(acc);
    cta_group_walk<R, NB, NM>(wm, rows, cols, row_w, xt, xs, acc);
    warp_allreduce(acc);
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int t = 0; t < NB; ++t)
            if (lane == ((i * NB + t) & 31) && row_w + i < rows && t < n) {
                const size_t o = static_cast<size_t>(pr[t]) * rows + row_w + i;
                if constexpr (P == Pass::kGateUp) {
                    out[o] = moe_act(acc[0][i][t], acc[1][i][t], epi, pr[t]);
                } else {
                    out[o] = acc[0][i][t];
                }
            }
}

// Persistent over units (touched expert u, row block rb), u-major.
template <Pass P, int R>
__global__ void __launch_bounds__(kThreads) k_moe_pass(const Bank bank0, const Bank bank1,
                                                       int rows, int cols,
                                                       int top_k, const float* __restrict__ vec,
                                                       Plan plan, MoeAct epi,
                                                       float* __restrict__ out) {
    extern __shared__ float4 smem4[];
    float* xs = reinterpret_cast<float*>(smem4);
    constexpr int NM = P == Pass::kGateUp ? 2 : 1;
    const int warp = threadIdx.x >> 5;
    const int n_touched = plan.hdr[1];
    const int rbn = (rows + kWarps * R - 1) / (kWarps * R);
    const int total = n_touched * rbn;
    for (int unit = blockIdx.x; unit < total; unit += gridDim.x) {
        const int u = unit / rbn, rb = unit - u * rbn;
        const int e = plan.touched[u];
        const int beg = plan.offsets[e], n_e = plan.offsets[e + 1] - beg;
        const long row_w = static_cast<long>(rb) * (kWarps * R) + warp * R;
        const uint8_t* wm[NM];
        wm[0] = bank0.slot(e);
        if constexpr (NM == 2) wm[1] = bank1.slot(e);
        const uint8_t* const(&wmc)[NM] = wm;
        for (int c = 0; c < n_e; c += 8) {
            const int n = min(8, n_e - c);
            const int32_t* pairs = plan.pair_of + beg + c;
            if (n == 1)
                expert_chunk<P, R, 1>(wmc, rows, cols, row_w, pairs, n, top_k, vec, out, xs,
                                        epi);
            else if (n == 2)
                expert_chunk<P, R, 2>(wmc, rows, cols, row_w, pairs, n, top_k, vec, out, xs,
                                        epi);
            else if (n <= 4)
                expert_chunk<P, R, 4>(wmc, rows, cols, row_w, pairs, n, top_k, vec, out, xs,
                                        epi);
            else
                expert_chunk<P, R, 8>(wmc, rows, cols, row_w, pairs, n, top_k, vec, out, xs,
                                        epi);
        }
    }
}

// y[t*hidden + r] = sum over slots j (in order) of w[t,j] * o[(t*top_k+j)*hidden + r];
// in the bf16 mode the route weights are in the acts already and the sum of
// the o's is rounded to bfloat16 (dsv4_global_down_mxfp4).  Pairs the plan left
// out (invalid or cold) add nothing.
__global__ void __launch_bounds__(256) k_moe_combine(const float* __restrict__ o_pairs,
                                                     const int32_t* __restrict__ pair_slot,
                                                     const float* __restrict__ route_w,
                                                     int bf16, int n_tokens, int top_k,
                                                     int hidden, float* __restrict__ y) {
    // launched dependent on the down pass: its per-pair outputs after it completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t n = static_cast<size_t>(n_tokens) * hidden;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t t = i / hidden, r = i - t * hidden;
        float acc = 0.0f;
        for (int j = 0; j < top_k; ++j) {
            const size_t p = t * top_k + j;
            if (pair_slot[p] < 0) continue;
            const float o = __ldg(o_pairs + p * hidden + r);
            acc = bf16 ? __fadd_rn(acc, o) : __fmaf_rn(__ldg(route_w + p), o, acc);
        }
        y[i] = bf16 ? moe_bf16(acc) : acc;
    }
}

// Persistent grid size for a kernel: resident CTAs per SM times the SM count.
int persistent_grid(const void* kernel, size_t smem) {
    static std::mutex mu;
    static int cache_dev[16] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
    static int cache_sms[16];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 16 && cache_dev[dev] == dev) {
            sms = cache_sms[dev];
        } else {
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                sms = 152;
            if (dev < 16) {
                cache_dev[dev] = dev;
                cache_sms[dev] = sms;
            }
        }
    }
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    return sms * per_sm;
}

constexpr int kRowsPerWarp = 2;

template <Pass P>
cudaError_t launch_pass(const Bank& bank0, const Bank& bank1, int n_experts, int rows, int cols,
                        int top_k, const float* vec, Plan plan, MoeAct epi, float* out,
                        cudaStream_t s) {
    auto kernel = k_moe_pass<P, kRowsPerWarp>;
    const long rbn = (rows + kWarps * kRowsPerWarp - 1) / (kWarps * kRowsPerWarp);
    const long max_units = static_cast<long>(n_experts) * rbn;
    const long cap = persistent_grid(reinterpret_cast<const void*>(kernel), kStageBytes);
    const unsigned grid = static_cast<unsigned>(max_units < cap ? max_units : cap);
    kernel<<<grid, kThreads, kStageBytes, s>>>(bank0, bank1, rows, cols, top_k, vec, plan, epi,
                                               out);
    return cudaGetLastError();
}

}  // namespace

size_t moe_workspace_bytes(int n_slots, int n_tokens, int top_k, int hidden, int inter) {
    return ws_layout(n_slots, n_tokens, top_k, hidden, inter).total;
}

cudaError_t launch_moe_gate_up(const Bank& gate, const Bank& up, int n_slots, int hidden,
                               int inter, const float* x, int n_tokens, int top_k,
                               const int32_t* ids, const int32_t* slot_of, int n_ids,
                               MoeAct epi, float* act, void* ws, cudaStream_t s) {
    const int n_pairs = n_tokens * top_k;
    const Plan plan = plan_view(ws, n_slots, n_tokens, top_k, hidden, inter);
    const std::function<cudaError_t()> launch_plan = [&]() -> cudaError_t {
        if (n_slots <= kPlanSmemExperts)
            k_moe_plan_s<<<1, 1024,
                           4 * (static_cast<size_t>(n_slots) +
                                static_cast<size_t>(n_pairs <= kPlanSmemPairs ? n_pairs : 0)),
                           s>>>(ids, n_pairs, n_slots, slot_of, n_ids, plan);
        else
            k_moe_plan<<<1, 1024, 0, s>>>(ids, n_pairs, n_slots, slot_of, n_ids, plan);
        return cudaGetLastError();
    };
    cudaError_t e = launch_moe_tc_gate_up(gate, up, n_slots, inter, hidden, top_k, x, n_tokens,
                                          plan.frag_x, launch_plan, plan.hdr, plan.offsets,
                                          plan.touched, plan.pair_of, epi, act, s);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();   // nothing launched: the plan and the FP32 pass
    e = launch_plan();
    if (e != cudaSuccess) return e;
    return launch_pass<Pass::kGateUp>(gate, up, n_slots, inter, hidden, top_k, x, plan, epi, act,
                                      s);
}

cudaError_t launch_moe_down(const Bank& down, int n_slots, int hidden, int inter,
                            const float* act, int n_tokens, int top_k, const float* route_w,
                            int bf16, float* y, void* ws, cudaStream_t s) {
    const int n_pairs = n_tokens * top_k;
    const Plan plan = plan_view(ws, n_slots, n_tokens, top_k, hidden, inter);
    cudaError_t e = launch_moe_tc_down(down, n_slots, hidden, inter, act, n_pairs, plan.frag_a,
                                       plan.hdr, plan.offsets, plan.touched, plan.pair_of,
                                       plan.o_pairs, s);
    if (e == cudaErrorNotSupported) {
        (void)cudaGetLastError();
        e = launch_pass<Pass::kDown>(down, down, n_slots, hidden, inter, top_k, act, plan,
                                     MoeAct{nullptr, 0.0f, 0}, plan.o_pairs, s);
    }
    if (e != cudaSuccess) return e;
    const size_t n = static_cast<size_t>(n_tokens) * hidden;
    const unsigned blocks = static_cast<unsigned>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_moe_combine, static_cast<const float*>(plan.o_pairs),
                           static_cast<const int32_t*>(plan.pair_slot), route_w, bf16, n_tokens,
                           top_k, hidden, y);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t moe_cold_pairs(const void* ws, int n_slots, int n_pairs, int* n_cold,
                           int32_t* pairs_host, int cap, cudaStream_t s) {
    const WsLayout l = ws_layout(n_slots, n_pairs, 1, 32, 32);
    const char* b = static_cast<const char*>(ws);
    int32_t n = 0;
    cudaError_t e = cudaMemcpyAsync(&n, b + l.hdr + 8, sizeof(n), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *n_cold = n;
    const int k = n < cap ? n : cap;
    if (k > 0 && pairs_host != nullptr) {
        e = cudaMemcpyAsync(pairs_host, b + l.cold, sizeof(int32_t) * static_cast<size_t>(k),
                            cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

cudaError_t moe_plan_errors(const void* ws, int* n_invalid, cudaStream_t s) {
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *n_invalid = v;
    return cudaSuccess;
}

}  // namespace mxk
