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

namespace {

// bf16 spacing at |v|: 2^(e - 7) with e the binade of |v| (normal range floor).
double bf16_spacing(double v) {
    const double a = std::fabs(v);
    int e = -126;
    if (a > 0.0 && std::isfinite(a)) e = std::ilogb(a) < -126 ? -126 : std::ilogb(a);
    return std::ldexp(1.0, e - 7);
}

// GLOBAL fn mxg_bf16 applied to the float value of v.
double bf16_of(double v) { return static_cast<double>(mxo_bf16_rne(static_cast<float>(v))); }

// The largest |silu'| on [z - r, z + r] (a Lipschitz constant of SiLU there):
// |silu'| is monotone between its extremes near -2.3994 (0.0998) and 2.3994
// (1.0998), so the endpoints and any extreme inside the interval decide it.
double silu_lipschitz(double z, double r) {
    const double lo = z - r, hi = z + r;
    double m = std::fmax(std::fabs(mxo_silu_grad(lo)), std::fabs(mxo_silu_grad(hi)));
    if (lo <= 2.4 && hi >= 2.39) m = std::fmax(m, 1.1);
    if (lo <= -2.39 && hi >= -2.4) m = std::fmax(m, 0.1);
    return m * 1.01;
}

}  // namespace

// The global-bank kernels with their flags: the gate/up tail (bf16 rounding of
// gate and up, the SwiGLU limit, the route weight folded into a bf16 act) and
// the down kernel (pre-weighted acts summed over the slots, the sum rounded to
// bf16), on a bank addressed through an expert -> slot table.
void mxo_moe_forward_ex(const uint8_t* gate_bank, const uint8_t* up_bank,
                        const uint8_t* down_bank, size_t gu_stride_bytes,
                        size_t down_stride_bytes, int n_slots, int hidden, int inter,
                        const float* x, int n_tokens, int top_k, const int32_t* ids,
                        const int32_t* slot_of, int n_experts, const float* route_w,
                        int bf16_mode, float limit, double* out, double* bound,
                        int32_t* cold_pairs, int* n_cold) {
    const double eps = 1e-5;
    const int n_pairs = n_tokens * top_k;
    std::vector<int> slot(static_cast<size_t>(n_pairs), -1);
    int cold = 0;
    for (int p = 0; p < n_pairs; ++p) {
        const int32_t e = ids[p];
        if (e < 0 || e >= n_experts) continue;            // invalid id
        const int32_t s = slot_of ? slot_of[e] : e;
        if (s < 0) {                                      // cold: not in the bank
            cold_pairs[cold++] = p;
            continue;
        }
        if (s < n_slots) slot[p] = s;                     // else invalid slot
    }
    *n_cold = cold;
    std::vector<double> a(static_cast<size_t>(inter)), ea(static_cast<size_t>(inter));
    std::vector<double> o(static_cast<size_t>(hidden)), eo(static_cast<size_t>(hidden));
    for (int t = 0; t < n_tokens; ++t) {
        const float* xt = x + static_cast<size_t>(t) * hidden;
        std::vector<double> acc(static_cast<size_t>(hidden), 0.0), eacc(acc), mag(acc);
        for (int j = 0; j < top_k; ++j) {
            const int p = t * top_k + j;
            if (slot[p] < 0) continue;
            const uint8_t* ge = gate_bank + static_cast<size_t>(slot[p]) * gu_stride_bytes;
            const uint8_t* ue = up_bank + static_cast<size_t>(slot[p]) * gu_stride_bytes;
            const uint8_t* de = down_bank + static_cast<size_t>(slot[p]) * down_stride_bytes;
            const double w = static_cast<double>(route_w[p]);
            const double wpre = bf16_mode ? std::fabs(w) : 1.0;
            for (int c = 0; c < inter; ++c) {
                double g, u, l1g, l1u;
                row_dot(ge, inter, hidden, c, xt, &g, &l1g);
                row_dot(ue, inter, hidden, c, xt, &u, &l1u);
                double eg = eps * l1g, eu = eps * l1u;
                if (bf16_mode) {   // a value eg off may round to a neighbour of bf16(g)
                    eg += bf16_spacing(std::fabs(g) + eg);
                    eu += bf16_spacing(std::fabs(u) + eu);
                    g = bf16_of(g);
                    u = bf16_of(u);
                }
                if (limit > 0.0f) {   // a value clamped with room to spare has no error left
                    const double lim = static_cast<double>(limit);
                    if (std::fabs(u) - lim > eu) eu = 0.0;
                    if (g - lim > eg) eg = 0.0;
                    u = u < -lim ? -lim : (u > lim ? lim : u);
                    g = g < lim ? g : lim;
                }
                const double sg = mxo_silu(g);
                double av = sg * u;
                const double lg = silu_lipschitz(g, eg);
                // (+ a few float roundings of the SiLU and the products)
                double e = wpre * ((std::fabs(sg) + lg * eg) * eu + lg * std::fabs(u) * eg +
                                   std::ldexp(std::fabs(av), -21));
                if (bf16_mode) {
                    av = w * av;
                    e += bf16_spacing(std::fabs(av) + e);
                    av = bf16_of(av);
                }
                a[static_cast<size_t>(c)] = av;
                ea[static_cast<size_t>(c)] = e;
            }
            for (int r = 0; r < hidden; ++r) {
                double sum = 0.0, l1 = 0.0, prop = 0.0;
                for (int c = 0; c < inter; ++c) {
                    const double dw = static_cast<double>(mxo_weight_at(de, hidden, inter, r, c));
                    sum += dw * a[static_cast<size_t>(c)];
                    l1 += std::fabs(dw * a[static_cast<size_t>(c)]);
                    prop += std::fabs(dw) * ea[static_cast<size_t>(c)];
                }
                const double eo_r = prop + eps * l1;
                if (bf16_mode) {
                    acc[static_cast<size_t>(r)] += sum;
                    eacc[static_cast<size_t>(r)] += eo_r;
                    mag[static_cast<size_t>(r)] += std::fabs(sum);
                } else {
                    acc[static_cast<size_t>(r)] += w * sum;
                    eacc[static_cast<size_t>(r)] += std::fabs(w) * eo_r;
                    mag[static_cast<size_t>(r)] += std::fabs(w * sum);
                }
            }
        }
        for (int r = 0; r < hidden; ++r) {
            const size_t i = static_cast<size_t>(t) * hidden + r;
            double y = acc[static_cast<size_t>(r)];
            double b = eacc[static_cast<size_t>(r)] + eps * mag[static_cast<size_t>(r)];
            if (bf16_mode) {
                b += bf16_spacing(std::fabs(y) + b);
                y = bf16_of(y);
            }
            out[i] = y;
            bound[i] = b;
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


// ---- GGUF Q4_K (the second codec) ----------------------------------------

namespace {
constexpr int kQK = 256;          // elements per super-block
constexpr int kQ4KBytes = 144;    // 2 + 2 + 12 + 128
}  // namespace

size_t mxo_q4k_nbytes(int rows, int cols) {
    if (rows <= 0 || cols <= 0 || cols % kQK != 0) return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(cols / kQK) * kQ4KBytes;
}

// IEEE 754 binary16: sign bit 15, exponent bits 10-14 (bias 15), fraction bits
// 0-9; exponent 0 is zero or subnormal (fraction * 2^-24), 31 is infinity or NaN.
float mxo_f16(unsigned bits) {
    const unsigned sign = (bits >> 15) & 1u, e = (bits >> 10) & 31u, f = bits & 1023u;
    float v;
    if (e == 0u) v = std::ldexp(static_cast<float>(f), -24);
    else if (e == 31u) v = f == 0u ? std::numeric_limits<float>::infinity()
                                   : std::numeric_limits<float>::quiet_NaN();
    else v = std::ldexp(static_cast<float>(1024u + f), static_cast<int>(e) - 25);
    return sign ? -v : v;
}

// q4k_scale_min_x86: sub-blocks 0-3 keep their 6-bit scale and min in the low six
// bits of bytes j and j + 4; sub-blocks 4-7 take their low four bits from the two
// nibbles of byte j + 4 and their high two bits from the top of bytes j - 4
// (scale) and j (min).
void mxo_q4k_scale_min(const uint8_t* q, int j, unsigned* sc, unsigned* m) {
    if (j < 4) {
        *sc = q[j] & 63u;
        *m = q[j + 4] & 63u;
    } else {
        *sc = (q[j + 4] & 0x0Fu) | ((q[j - 4] >> 6) << 4);
        *m = (q[j + 4] >> 4) | ((q[j] >> 6) << 4);
    }
}

float mxo_q4k_weight_at(const uint8_t* w, int rows, int cols, int r, int c) {
    (void)rows;
    const uint8_t* blk =
        w + (static_cast<size_t>(r) * (cols / kQK) + static_cast<size_t>(c / kQK)) * kQ4KBytes;
    const int e = c % kQK, s = e / 64, p = e % 64;
    const int j = 2 * s + (p >= 32 ? 1 : 0);                       // sub-block
    const uint8_t byte = blk[16 + 32 * s + (p % 32)];
    const unsigned q = p < 32 ? (byte & 0x0Fu) : (byte >> 4);
    unsigned sc = 0, m = 0;
    mxo_q4k_scale_min(blk + 4, j, &sc, &m);
    const float d = mxo_f16(static_cast<unsigned>(blk[0]) | (static_cast<unsigned>(blk[1]) << 8));
    const float dmin =
        mxo_f16(static_cast<unsigned>(blk[2]) | (static_cast<unsigned>(blk[3]) << 8));
    // d*sc*q and dmin*m are exact in float (at most 11+6+4 and 11+6 significant
    // bits); the difference rounds once (the build has contraction off)
    const float scaled = (d * static_cast<float>(sc)) * static_cast<float>(q);
    const float mins = dmin * static_cast<float>(m);
    return scaled - mins;
}

void mxo_q4k_dequant(const uint8_t* w, int rows, int cols, float* out) {
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c)
            out[static_cast<size_t>(r) * cols + c] = mxo_q4k_weight_at(w, rows, cols, r, c);
}

void mxo_q4k_matmat(const uint8_t* w, int rows, int cols, const float* x, int nb, int r0,
                    int r1, double* y, double* l1) {
    const int nr = r1 - r0;
    for (int t = 0; t < nb; ++t) {
        const float* xt = x + static_cast<size_t>(t) * cols;
        for (int r = r0; r < r1; ++r) {
            double sum = 0.0, mag = 0.0;
            for (int c = 0; c < cols; ++c) {
                const double p = static_cast<double>(mxo_q4k_weight_at(w, rows, cols, r, c)) *
                                 static_cast<double>(xt[c]);
                sum += p;
                mag += std::fabs(p);
            }
            y[static_cast<size_t>(t) * nr + (r - r0)] = sum;
            l1[static_cast<size_t>(t) * nr + (r - r0)] = mag;
        }
    }
}
