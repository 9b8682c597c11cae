// mxfp4_oracle.cpp -- CPU oracle (test infrastructure only; see the header).
//
// Plain C++17, scalar, double accumulation, no intrinsics, no threads: it must
// build and give the same answers on x86-64 and aarch64 hosts.  Each function
// says which part of "cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs" (or of the
// two prior-art pages) it restates.

#include "mxfp4_oracle.h"

#include <cmath>
#include <cstring>
#include <limits>
#include <vector>

namespace {

// E2M1 magnitudes by the low three code bits: exponent bits (e1 e0), mantissa
// bit m; value 2^(E-1) * (1 + m/2) for E >= 1 and m/2 for E = 0.
const float kE2M1Magnitude[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

inline size_t code_plane_bytes(int rows, int cols) {
    return static_cast<size_t>(rows) * static_cast<size_t>(cols) / 2;
}

inline int groups_per_row(int cols) { return cols / 32; }

// Little-endian u32 word `index` of the buffer, assembled byte by byte so that
// the host's own byte order never matters.
inline uint32_t le_word(const uint8_t* buf, size_t index) {
    const uint8_t* p = buf + 4 * index;
    return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
           (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24);
}

}  // namespace

// The functions below get C linkage from their declarations in the header.

// DECODE fn mx_e2m1: magnitude from the low three bits, bit 3 flips the sign
// (negating +0.0 gives -0.0, as the page's select(v, -v, ...) does).
float mxo_e2m1(unsigned n) {
    float mag = kE2M1Magnitude[n & 7u];
    return (n & 8u) ? -mag : mag;
}

// DECODE fn mx_e8m0: 2^(k-127); k = 255 is NaN; k = 0 is 2^-127 (subnormal).
float mxo_e8m0(unsigned k) {
    k &= 0xFFu;
    if (k == 255u) return std::numeric_limits<float>::quiet_NaN();
    return std::ldexp(1.0f, static_cast<int>(k) - 127);
}

// MoeBankCodec::lens / tests bank_codec_lengths: a [rows, cols] tensor is
// rows*cols/2 code bytes plus rows*cols/32 scale bytes = rows*cols*17/32.
size_t mxo_nbytes_exact(int rows, int cols) {
    if (rows <= 0 || cols <= 0 || cols % 32 != 0) return 0;
    return code_plane_bytes(rows, cols) + static_cast<size_t>(rows) * groups_per_row(cols);
}

// mxfp4_mv group walk: element c of row r is nibble j = i % 8 of word
// k = i / 8 of group g = c / 32 (i = c % 32); the group's words start at word
// (r*gpr + g)*4.
unsigned mxo_code_at(const uint8_t* w, int rows, int cols, int r, int c) {
    (void)rows;
    const int gpr = groups_per_row(cols);
    const int g = c / 32, i = c % 32, k = i / 8, j = i % 8;
    const size_t word = (static_cast<size_t>(r) * gpr + g) * 4 + k;
    return (le_word(w, word) >> (4 * j)) & 0xFu;
}

// PEROP fn mx_scale: scale index i = r*gpr + g; byte i of the scale plane,
// which starts right after the code plane.
unsigned mxo_scale_at(const uint8_t* w, int rows, int cols, int r, int g) {
    const int gpr = groups_per_row(cols);
    const size_t i = static_cast<size_t>(r) * gpr + g;
    return w[code_plane_bytes(rows, cols) + i];
}

float mxo_weight_at(const uint8_t* w, int rows, int cols, int r, int c) {
    return mxo_e2m1(mxo_code_at(w, rows, cols, r, c)) *
           mxo_e8m0(mxo_scale_at(w, rows, cols, r, c / 32));
}

void mxo_dequant(const uint8_t* w, int rows, int cols, float* out) {
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c)
            out[static_cast<size_t>(r) * cols + c] = mxo_weight_at(w, rows, cols, r, c);
}

// The page's f64 reference (tests fn reference): decode to float, multiply and
// sum in double; l1 is the sum of |products| (the magnitude the tolerance is
// relative to).
void mxo_matmat(const uint8_t* w, int rows, int cols, const float* x, int nb,
                int r0, int r1, double* y, double* l1) {
    const int nr = r1 - r0;
    for (int t = 0; t < nb; ++t) {
        const float* xt = x + static_cast<size_t>(t) * cols;
        for (int r = r0; r < r1; ++r) {
            double sum = 0.0, mag = 0.0;
            for (int c = 0; c < cols; ++c) {
                const double p = static_cast<double>(mxo_weight_at(w, rows, cols, r, c)) *
                                 static_cast<double>(xt[c]);
                sum += p;
                mag += std::fabs(p);
            }
            y[static_cast<size_t>(t) * nr + (r - r0)] = sum;
            l1[static_cast<size_t>(t) * nr + (r - r0)] = mag;
        }
    }
}

void mxo_matmat_samples(const uint8_t* w, int rows, int cols, const float* x,
                        const int32_t* tok, const int32_t* row, int n,
                        double* y, double* l1) {
    for (int s = 0; s < n; ++s) {
        const float* xt = x + static_cast<size_t>(tok[s]) * cols;
        const int r = row[s];
        double sum = 0.0, mag = 0.0;
        for (int c = 0; c < cols; ++c) {
            const double p = static_cast<double>(mxo_weight_at(w, rows, cols, r, c)) *
                             static_cast<double>(xt[c]);
            sum += p;
            mag += std::fabs(p);
        }
        y[s] = sum;
        l1[s] = mag;
    }
}

// GLOBAL fn mxg_bf16: keep the top 16 bits after adding 0x7FFF plus the lowest
// kept bit (round to nearest, ties to even); Inf/NaN unchanged.
float mxo_bf16_rne(float v) {
    uint32_t bits;
    std::memcpy(&bits, &v, 4);
    if ((bits & 0x7F800000u) == 0x7F800000u) return v;
    const uint32_t lsb = (bits >> 16) & 1u;
    bits = (bits + 0x7FFFu + lsb) & 0xFFFF0000u;
    float out;
    std::memcpy(&out, &bits, 4);
    return out;
}

void mxo_round_bf16(const float* in, float* out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = mxo_bf16_rne(in[i]);
}

// dsv4_global_gate_up_mxfp4 tail: act = (gate / (1 + exp(-gate))) * up.
double mxo_silu(double g) { return g / (1.0 + std::exp(-g)); }

double mxo_silu_grad(double g) {
    const double s = 1.0 / (1.0 + std::exp(-g));
    return s * (1.0 + g * (1.0 - s));
}

namespace {

// One dot product of row r of an MXFP4 matrix with a double or float vector.
template <typename T>
void row_dot(const uint8_t* w, int rows, int cols, int r, const T* v, double* sum,
             double* mag) {
    double s = 0.0, m = 0.0;
    for (int c = 0; c < cols; ++c) {
        const double p = static_cast<double>(mxo_weight_at(w, rows, cols, r, c)) *
                         static_cast<double>(v[c]);
        s += p;
        m += std::fabs(p);
    }
    *sum = s;
    *mag = m;
}

inline bool valid_expert(int32_t e, int n_experts) { return e >= 0 && e < n_experts; }

}  // namespace

void mxo_moe_gate_up(const uint8_t* gate_bank, const uint8_t* up_bank,
                     size_t stride_bytes, int n_experts, int hidden, int inter,
                     const float* x, int n_tokens, int top_k,
                     const int32_t* ids, double* g, double* u, double* l1g,
                     double* l1u, double* act) {
    const double nan = std::numeric_limits<double>::quiet_NaN();
    for (int t = 0; t < n_tokens; ++t) {
        const float* xt = x + static_cast<size_t>(t) * hidden;
        for (int j = 0; j < top_k; ++j) {
            const size_t p = static_cast<size_t>(t) * top_k + j;
            const int32_t e = ids[p];
            for (int r = 0; r < inter; ++r) {
                const size_t o = p * inter + r;
                if (!valid_expert(e, n_experts)) {
                    g[o] = u[o] = l1g[o] = l1u[o] = act[o] = nan;
                    continue;
                }
                const uint8_t* ge = gate_bank + static_cast<size_t>(e) * stride_bytes;
                const uint8_t* ue = up_bank + static_cast<size_t>(e) * stride_bytes;
                row_dot(ge, inter, hidden, r, xt, &g[o], &l1g[o]);
                row_dot(ue, inter, hidden, r, xt, &u[o], &l1u[o]);
                act[o] = mxo_silu(g[o]) * u[o];
            }
        }
    }
}

namespace {

// Down pass of one pair on a double or float activation, then the weighted
// top-k combine in slot order.
template <typename A>
void moe_down_impl(const uint8_t* down_bank, size_t stride_bytes, int n_experts,
                   int hidden, int inter, const A* act, int n_tokens, int top_k,
                   const int32_t* ids, const float* route_w, double* o_pairs,
                   double* l1_pairs, double* out, double* l1_out) {
    const double nan = std::numeric_limits<double>::quiet_NaN();
    for (int t = 0; t < n_tokens; ++t) {
        for (int r = 0; r < hidden; ++r) {
            out[static_cast<size_t>(t) * hidden + r] = 0.0;
            l1_out[static_cast<size_t>(t) * hidden + r] = 0.0;
        }
        for (int j = 0; j < top_k; ++j) {
            const size_t p = static_cast<size_t>(t) * top_k + j;
            const int32_t e = ids[p];
            const double wt = static_cast<double>(route_w[p]);
            for (int r = 0; r < hidden; ++r) {
                double o, m;
                if (valid_expert(e, n_experts)) {
                    const uint8_t* de = down_bank + static_cast<size_t>(e) * stride_bytes;
                    row_dot(de, hidden, inter, r, act + p * inter, &o, &m);
                } else {
                    o = m = nan;
                }
                if (o_pairs) o_pairs[p * hidden + r] = o;
                if (l1_pairs) l1_pairs[p * hidden + r] = m;
                // A pair routed to an out-of-range expert contributes nothing.
                if (!valid_expert(e, n_experts)) continue;
                out[static_cast<size_t>(t) * hidden + r] += wt * o;
                l1_out[static_cast<size_t>(t) * hidden + r] += std::fabs(wt) * m;
            }
        }
    }
}

}  // namespace

void mxo_moe_down(const uint8_t* down_bank, size_t stride_bytes, int n_experts,
                  int hidden, int inter, const float* act, int n_tokens,
                  int top_k, const int32_t* ids, const float* route_w,
                  double* o_pairs, double* l1_pairs, double* out,
                  double* l1_out) {
    moe_down_impl(down_bank, stride_bytes, n_experts, hidden, inter, act, n_tokens,
                  top_k, ids, route_w, o_pairs, l1_pairs, out, l1_out);
}

void mxo_moe_forward(const uint8_t* gate_bank, const uint8_t* up_bank,
                     const uint8_t* down_bank, size_t gu_stride_bytes,
                     size_t down_stride_bytes, int n_experts, int hidden,
                     int inter, const float* x, int n_tokens, int top_k,
                     const int32_t* ids, const float* route_w, double* out,
                     double* bound_l1, double* bound_prop) {
    const size_t n_act = static_cast<size_t>(n_tokens) * top_k * inter;
    std::vector<double> g(n_act), u(n_act), l1g(n_act), l1u(n_act), act(n_act), err(n_act);
    mxo_moe_gate_up(gate_bank, up_bank, gu_stride_bytes, n_experts, hidden, inter, x,
                    n_tokens, top_k, ids, g.data(), u.data(), l1g.data(), l1u.data(),
                    act.data());
    // Propagated size of a relative-to-L1 error in g and u, per act element.
    for (size_t i = 0; i < n_act; ++i)
        err[i] = std::fabs(mxo_silu_grad(g[i])) * l1g[i] * std::fabs(u[i]) +
                 std::fabs(mxo_silu(g[i])) * l1u[i];
    moe_down_impl(down_bank, down_stride_bytes, n_experts, hidden, inter, act.data(),
                  n_tokens, top_k, ids, route_w, nullptr, nullptr, out, bound_l1);
    // bound_prop: the same combine with |down| against the propagated errors.
    for (int t = 0; t < n_tokens; ++t) {
        for (int r = 0; r < hidden; ++r) {
            double acc = 0.0;
            for (int j = 0; j < top_k; ++j) {
                const size_t p = static_cast<size_t>(t) * top_k + j;
                const int32_t e = ids[p];
                if (!valid_expert(e, n_experts)) continue;   // contributes nothing
                const uint8_t* de = down_bank + static_cast<size_t>(e) * down_stride_bytes;
                double s = 0.0;
                for (int c = 0; c < inter; ++c)
                    s += std::fabs(static_cast<double>(mxo_weight_at(de, hidden, inter, r, c))) *
                         err[p * inter + c];
                acc += std::fabs(static_cast<double>(route_w[p])) * s;
            }
            bound_prop[static_cast<size_t>(t) * hidden + r] = acc;
        }
    }
}

// grouped_moe_sort_plan: count pairs per expert, prefix-sum the counts into
// offsets, then place each pair at its expert's next free slot (stable).
int mxo_moe_plan(const int32_t* ids, int n_pairs, int n_experts, int32_t* offsets,
                 int32_t* pair_of) {
    std::vector<int32_t> counts(static_cast<size_t>(n_experts), 0);
    int invalid = 0;
    for (int p = 0; p < n_pairs; ++p) {
        if (valid_expert(ids[p], n_experts)) ++counts[ids[p]];
        else ++invalid;
    }
    offsets[0] = 0;
    for (int e = 0; e < n_experts; ++e) offsets[e + 1] = offsets[e] + counts[e];
    std::vector<int32_t> next(offsets, offsets + n_experts);
    for (int p = 0; p < n_pairs; ++p)
        if (valid_expert(ids[p], n_experts)) pair_of[next[ids[p]]++] = p;
    return invalid;
}

