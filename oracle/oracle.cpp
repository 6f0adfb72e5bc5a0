/*
 * oracle.cpp -- plain, slow, single-threaded CPU reference of one decode step.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): used by tests, the smoke check and
 * the bench's CPU-baseline leg, never by the product path.
 *
 * Everything is written as the plain definition, in the accumulation type T
 * (float or double): bf16 weights are widened exactly, every dot product is
 * accumulated in index order, softmax subtracts the maximum, and the KV cache
 * holds bf16 values rounded to nearest-even. Sources per function below; the
 * pages themselves print no formulas, so the model details are the readings
 * stated in the design notes.
 */
#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <map>
#include <set>
#include <tuple>
#include <vector>

#include "../synth/synth.h"

namespace {

typedef std::tuple<int, int, int> TKey;

double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

/* round to bf16, nearest-even, from float (T = float) or double (T = double) */
uint16_t to_bf16(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
uint16_t to_bf16(double d) {
    /* exact round-to-nearest-even of a double to bf16: work on the double's
     * bits (52-bit mantissa) so there is no intermediate float rounding */
    if (std::isnan(d)) return 0x7fc0;
    uint64_t u;
    std::memcpy(&u, &d, 8);
    uint64_t sign = u >> 63;
    double a = std::fabs(d);
    if (a == 0.0) return (uint16_t)(sign << 15);
    int e;
    double m = std::frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    /* bf16 normal: 8 significant bits. scale so the kept bits are integral */
    if (e - 1 < -126) {
        /* subnormal range of bf16: quantum 2^-133 */
        double q = std::ldexp(a, 133);
        double r = std::nearbyint(q); /* default rounding mode: nearest-even */
        uint32_t bits = (uint32_t)r;  /* may carry into the smallest normal */
        return (uint16_t)((sign << 15) | bits);
    }
    double q = std::ldexp(m, 8); /* in [128, 256) */
    double r = std::nearbyint(q);
    if (r == 256.0) { r = 128.0; e += 1; }
    int exp_field = e - 1 + 127;
    if (exp_field >= 255) return (uint16_t)((sign << 15) | 0x7f80);
    uint32_t mant = (uint32_t)r - 128u;
    return (uint16_t)((sign << 15) | ((uint32_t)exp_field << 7) | mant);
}

template <class T> T bf(uint16_t h) { return (T)bf16_to_double(h); }

}  // namespace

/* Value of an FP8 E4M3 code, from the format's definition (OCP "Microscaling
 * Formats (MX) Specification" v1.0, the E4M3 element type): sign bit, 4
 * exponent bits of bias 7, 3 mantissa bits; exponent field 0 holds the
 * subnormals m * 2^-9; 0x7F and 0xFF are NaN; there are no infinities. */
double oracle_e4m3_value(uint8_t code) {
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
    const double v = e == 0 ? std::ldexp((double)m, -9) : std::ldexp(8.0 + m, e - 10);
    return s ? -v : v;
}

/* MX dequantisation (same specification): element j of row r is its E4M3
 * value times 2^(E - 127), E the E8M0 scale byte of its block of 32
 * consecutive elements of the row (scale 0xFF is NaN). codes [rows, cols],
 * scales [rows, cols / 32], out [rows, cols]. */
void oracle_mx_dequant(const uint8_t* codes, const uint8_t* scales, int32_t rows, int32_t cols, double* out) {
    const int32_t nb = cols / 32;
    for (int32_t r = 0; r < rows; ++r)
        for (int32_t j = 0; j < cols; ++j) {
            const uint8_t E = scales[(size_t)r * nb + j / 32];
            const double x = oracle_e4m3_value(codes[(size_t)r * cols + j]);
            out[(size_t)r * cols + j] = E == 0xFF ? std::numeric_limits<double>::quiet_NaN() : std::ldexp(x, (int)E - 127);
        }
}

struct oracle_model {
    oracle_cfg c;
    synth_dims d;
    uint64_t seed;
    int lazy;
    int gen_threads;
    std::map<TKey, std::vector<uint16_t>> w;
    std::set<TKey> pinned; /* caller-provided tensors, never released */
};

struct oracle_kv {
    int32_t L, B, max_pos, row;
    int32_t attn_kind, half; /* GQA: half = Hkv*hd (K then V); MLA: half = 0 */
    std::vector<uint16_t> data; /* [L][B][max_pos][row] */
    uint16_t* at(int l, int b, int p) { return &data[(((size_t)l * B + b) * max_pos + p) * row]; }
};

namespace {

synth_dims dims_of(const oracle_cfg& c) {
    synth_dims d;
    d.n_layers = c.n_layers; d.d_model = c.d_model; d.vocab = c.vocab; d.attn_kind = c.attn_kind;
    d.n_q_heads = c.n_q_heads; d.n_kv_heads = c.n_kv_heads; d.head_dim = c.head_dim;
    d.q_lora_rank = c.q_lora_rank; d.kv_lora_rank = c.kv_lora_rank; d.qk_nope_dim = c.qk_nope_dim;
    d.qk_rope_dim = c.qk_rope_dim; d.v_head_dim = c.v_head_dim;
    d.n_routed_experts = c.n_routed_experts; d.top_k = c.top_k; d.n_shared_experts = c.n_shared_experts;
    d.ffn_dim = c.ffn_dim; d.shared_ffn_dim = c.shared_ffn_dim;
    return d;
}

bool is_expert_kind(int kind) {
    return kind == SYNTH_GATE || kind == SYNTH_UP || kind == SYNTH_DOWN || kind == SYNTH_SH_GATE ||
           kind == SYNTH_SH_UP || kind == SYNTH_SH_DOWN;
}

const uint16_t* tensor(oracle_model* m, int kind, int layer, int expert) {
    TKey k(kind, layer, expert);
    auto it = m->w.find(k);
    if (it != m->w.end()) return it->second.data();
    int32_t rows, cols;
    float sigma, mean;
    if (synth_weight_spec(&m->d, kind, &rows, &cols, &sigma, &mean) != 0) return nullptr;
    std::vector<uint16_t> v((size_t)rows * cols);
    if (m->c.expert_format == 1 && is_expert_kind(kind)) {
        /* MXFP8 expert weights: the generator's E4M3 codes and E8M0 block
         * scales, dequantised; every value (at most 4 significant bits, scale
         * 2^-10 or 2^-9) is a bf16 number, so the bf16 store holds it exactly */
        std::vector<uint8_t> q((size_t)rows * cols), sc((size_t)rows * (cols / SYNTH_MX_BLOCK));
        synth_fill_e4m3(q.data(), q.size(), m->seed, synth_tensor_id(kind, layer, expert), 0, m->gen_threads);
        synth_fill_e8m0(sc.data(), sc.size(), m->seed, synth_tensor_id(kind + 6, layer, expert), 0);
        std::vector<double> deq(q.size());
        oracle_mx_dequant(q.data(), sc.data(), rows, cols, deq.data());
        for (size_t i = 0; i < deq.size(); ++i) v[i] = to_bf16(deq[i]);
    } else {
        synth_fill_bf16(v.data(), v.size(), m->seed, synth_tensor_id(kind, layer, expert), sigma, mean, 0,
                        m->gen_threads);
    }
    auto& slot = m->w[k];
    slot.swap(v);
    return slot.data();
}

void release_layer(oracle_model* m, int layer) {
    for (auto it = m->w.begin(); it != m->w.end();) {
        if (std::get<1>(it->first) == layer && !m->pinned.count(it->first))
            it = m->w.erase(it);
        else
            ++it;
    }
}

/* y[r] = sum_k W[r, k] x[k], W row-major bf16 [rows, cols]; index-order sums */
template <class T> void matvec(const uint16_t* W, int rows, int cols, const T* x, T* y) {
    for (int r = 0; r < rows; ++r) {
        const uint16_t* w = W + (size_t)r * cols;
        T acc = 0;
        for (int k = 0; k < cols; ++k) acc += bf<T>(w[k]) * x[k];
        y[r] = acc;
    }
}

/* RMSNorm: x * 1/sqrt(mean(x^2) + eps) * g */
template <class T> void rmsnorm(const T* x, const uint16_t* g, int n, T eps, T* out) {
    T ss = 0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    T r = (T)1 / std::sqrt(ss / (T)n + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * r * bf<T>(g[i]);
}

/* rotate-half RoPE on x[0..dim): pairs (i, i + dim/2), frequency theta^(-2i/dim);
 * frequency, angle, cos and sin in double, then cast to T */
template <class T> void rope(T* x, int dim, int pos, double theta) {
    int half = dim / 2;
    for (int i = 0; i < half; ++i) {
        double inv = std::pow(theta, -2.0 * (double)i / (double)dim);
        double ang = (double)pos * inv;
        T c = (T)std::cos(ang), s = (T)std::sin(ang);
        T a = x[i], b = x[i + half];
        x[i] = a * c - b * s;
        x[i + half] = b * c + a * s;
    }
}

template <class T> void softmax(const T* x, int n, T* out) {
    T mx = x[0];
    for (int i = 1; i < n; ++i) mx = std::max(mx, x[i]);
    T s = 0;
    for (int i = 0; i < n; ++i) { out[i] = std::exp(x[i] - mx); s += out[i]; }
    for (int i = 0; i < n; ++i) out[i] /= s;
}

template <class T> T silu(T z) { return z / ((T)1 + std::exp(-z)); }

/* router: softmax over all experts, top-k by probability (ties -> lower expert
 * index), selected probabilities renormalised to sum 1; margin = gap between
 * the k-th and (k+1)-th largest router logits */
template <class T> void topk(const T* logits, int n, int k, int32_t* idx, T* w, T* margin) {
    std::vector<T> p(n);
    softmax(logits, n, p.data());
    std::vector<int> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return p[a] > p[b]; });
    T s = 0;
    for (int j = 0; j < k; ++j) s += p[order[j]];
    for (int j = 0; j < k; ++j) { idx[j] = order[j]; w[j] = p[order[j]] / s; }
    if (margin) {
        if (k < n) {
            /* logits sorted the same way (softmax is monotone) */
            std::vector<int> lo(n);
            for (int i = 0; i < n; ++i) lo[i] = i;
            std::stable_sort(lo.begin(), lo.end(), [&](int a, int b) { return logits[a] > logits[b]; });
            *margin = logits[lo[k - 1]] - logits[lo[k]];
        } else {
            *margin = std::numeric_limits<T>::infinity();
        }
    }
}

/* attention of one query over n cached rows: softmax(q.K^T * scale) V */
template <class T>
void attend_rows(const T* q, const uint16_t* K, size_t kstride, const uint16_t* V, size_t vstride, int n, int hd,
                 T scale, T* out) {
    std::vector<T> s(n);
    for (int j = 0; j < n; ++j) {
        const uint16_t* k = K + (size_t)j * kstride;
        T acc = 0;
        for (int i = 0; i < hd; ++i) acc += q[i] * bf<T>(k[i]);
        s[j] = acc * scale;
    }
    std::vector<T> p(n);
    softmax(s.data(), n, p.data());
    for (int i = 0; i < hd; ++i) out[i] = 0;
    for (int j = 0; j < n; ++j) {
        const uint16_t* v = V + (size_t)j * vstride;
        for (int i = 0; i < hd; ++i) out[i] += p[j] * bf<T>(v[i]);
    }
}

/* y = sum of SwiGLU experts applied to xn: silu(Wg xn) * (Wu xn) -> Wd */
template <class T> void swiglu(const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int d, int f, const T* xn,
                               T* y) {
    std::vector<T> g(f), u(f), h(f);
    matvec(Wg, f, d, xn, g.data());
    matvec(Wu, f, d, xn, u.data());
    for (int j = 0; j < f; ++j) h[j] = silu(g[j]) * u[j];
    matvec(Wd, d, f, h.data(), y);
}

/* ---- one layer's attention block for one token (decode with cache) ---- */
template <class T>
void attention_token(oracle_model* m, oracle_kv* kv, int l, int b, int p, const T* xn, int absorbed, T* attn_out) {
    const oracle_cfg& c = m->c;
    const int d = c.d_model;
    if (c.attn_kind == 0) {
        const int Hq = c.n_q_heads, Hkv = c.n_kv_heads, hd = c.head_dim;
        std::vector<T> q((size_t)Hq * hd), k((size_t)Hkv * hd), v((size_t)Hkv * hd);
        matvec(tensor(m, SYNTH_WQ, l, 0), Hq * hd, d, xn, q.data());
        matvec(tensor(m, SYNTH_WK, l, 0), Hkv * hd, d, xn, k.data());
        matvec(tensor(m, SYNTH_WV, l, 0), Hkv * hd, d, xn, v.data());
        for (int h = 0; h < Hq; ++h) rope(&q[(size_t)h * hd], hd, p, c.rope_theta);
        for (int g = 0; g < Hkv; ++g) rope(&k[(size_t)g * hd], hd, p, c.rope_theta);
        uint16_t* row = kv->at(l, b, p);
        for (int i = 0; i < Hkv * hd; ++i) { row[i] = to_bf16(k[i]); row[Hkv * hd + i] = to_bf16(v[i]); }
        std::vector<T> o((size_t)Hq * hd);
        const T scale = (T)1 / std::sqrt((T)hd);
        const int group = Hq / Hkv;
        for (int h = 0; h < Hq; ++h) {
            int g = h / group;
            const uint16_t* K0 = kv->at(l, b, 0) + (size_t)g * hd;
            const uint16_t* V0 = kv->at(l, b, 0) + (size_t)Hkv * hd + (size_t)g * hd;
            attend_rows(&q[(size_t)h * hd], K0, kv->row, V0, kv->row, p + 1, hd, scale, &o[(size_t)h * hd]);
        }
        matvec(tensor(m, SYNTH_WO, l, 0), d, Hq * hd, o.data(), attn_out);
        return;
    }
    /* MLA */
    const int H = c.n_q_heads, ql = c.q_lora_rank, kl = c.kv_lora_rank;
    const int nope = c.qk_nope_dim, rd = c.qk_rope_dim, vd = c.v_head_dim, qh = nope + rd;
    std::vector<T> cq(ql), cqn(ql), q((size_t)H * qh), kva(kl + rd), ckv(kl);
    matvec(tensor(m, SYNTH_WDQ, l, 0), ql, d, xn, cq.data());
    rmsnorm(cq.data(), tensor(m, SYNTH_Q_NORM, l, 0), ql, (T)c.rms_eps, cqn.data());
    matvec(tensor(m, SYNTH_WUQ, l, 0), H * qh, ql, cqn.data(), q.data());
    for (int h = 0; h < H; ++h) rope(&q[(size_t)h * qh + nope], rd, p, c.rope_theta);
    matvec(tensor(m, SYNTH_WDKV, l, 0), kl + rd, d, xn, kva.data());
    rmsnorm(kva.data(), tensor(m, SYNTH_KV_NORM, l, 0), kl, (T)c.rms_eps, ckv.data());
    rope(&kva[kl], rd, p, c.rope_theta);
    uint16_t* row = kv->at(l, b, p);
    for (int i = 0; i < kl; ++i) row[i] = to_bf16(ckv[i]);
    for (int i = 0; i < rd; ++i) row[kl + i] = to_bf16(kva[kl + i]);
    const uint16_t* Wukv = tensor(m, SYNTH_WUKV, l, 0); /* per head: nope rows of W_uk, then vd rows of W_uv */
    const T scale = (T)1 / std::sqrt((T)qh);
    const int n = p + 1;
    std::vector<T> o((size_t)H * vd), s(n), pr(n);
    for (int h = 0; h < H; ++h) {
        const T* qn = &q[(size_t)h * qh];
        const T* qr = qn + nope;
        const uint16_t* Wuk = Wukv + (size_t)h * (nope + vd) * kl;
        const uint16_t* Wuv = Wuk + (size_t)nope * kl;
        T* oh = &o[(size_t)h * vd];
        if (!absorbed) {
            /* plain definition: decompress k_nope and v for every position */
            std::vector<T> cj(kl), kn(nope), vj(vd);
            for (int j = 0; j < n; ++j) {
                const uint16_t* r = kv->at(l, b, j);
                for (int i = 0; i < kl; ++i) cj[i] = bf<T>(r[i]);
                matvec(Wuk, nope, kl, cj.data(), kn.data());
                T acc = 0;
                for (int i = 0; i < nope; ++i) acc += qn[i] * kn[i];
                for (int i = 0; i < rd; ++i) acc += qr[i] * bf<T>(r[kl + i]);
                s[j] = acc * scale;
            }
            softmax(s.data(), n, pr.data());
            for (int i = 0; i < vd; ++i) oh[i] = 0;
            for (int j = 0; j < n; ++j) {
                const uint16_t* r = kv->at(l, b, j);
                for (int i = 0; i < kl; ++i) cj[i] = bf<T>(r[i]);
                matvec(Wuv, vd, kl, cj.data(), vj.data());
                for (int i = 0; i < vd; ++i) oh[i] += pr[j] * vj[i];
            }
        } else {
            /* absorbed: q_lat = W_uk^T q_nope; scores against the latent; W_uv after */
            std::vector<T> qlat(kl, 0), olat(kl, 0);
            for (int c2 = 0; c2 < kl; ++c2) {
                T acc = 0;
                for (int i = 0; i < nope; ++i) acc += qn[i] * bf<T>(Wuk[(size_t)i * kl + c2]);
                qlat[c2] = acc;
            }
            for (int j = 0; j < n; ++j) {
                const uint16_t* r = kv->at(l, b, j);
                T acc = 0;
                for (int i = 0; i < kl; ++i) acc += qlat[i] * bf<T>(r[i]);
                for (int i = 0; i < rd; ++i) acc += qr[i] * bf<T>(r[kl + i]);
                s[j] = acc * scale;
            }
            softmax(s.data(), n, pr.data());
            for (int j = 0; j < n; ++j) {
                const uint16_t* r = kv->at(l, b, j);
                for (int i = 0; i < kl; ++i) olat[i] += pr[j] * bf<T>(r[i]);
            }
            matvec(Wuv, vd, kl, olat.data(), oh);
        }
    }
    matvec(tensor(m, SYNTH_WO, l, 0), d, H * vd, o.data(), attn_out);
}

/* ---- feed-forward block for one token: routed experts + shared expert ---- */
template <class T>
void ffn_token(oracle_model* m, int l, const T* xn, T* y, int32_t* ridx, T* rw, T* rmargin) {
    const oracle_cfg& c = m->c;
    const int d = c.d_model;
    for (int i = 0; i < d; ++i) y[i] = 0;
    std::vector<T> ye(d);
    if (c.n_routed_experts > 0) {
        const int E = c.n_routed_experts, k = c.top_k;
        std::vector<T> logits(E), w(k);
        std::vector<int32_t> idx(k);
        T margin;
        matvec(tensor(m, SYNTH_ROUTER, l, 0), E, d, xn, logits.data());
        topk(logits.data(), E, k, idx.data(), w.data(), &margin);
        for (int j = 0; j < k; ++j) {
            int e = idx[j];
            swiglu(tensor(m, SYNTH_GATE, l, e), tensor(m, SYNTH_UP, l, e), tensor(m, SYNTH_DOWN, l, e), d, c.ffn_dim,
                   xn, ye.data());
            for (int i = 0; i < d; ++i) y[i] += w[j] * ye[i];
        }
        if (ridx) for (int j = 0; j < k; ++j) { ridx[j] = idx[j]; rw[j] = w[j]; }
        if (rmargin) *rmargin = margin;
    }
    if (c.n_shared_experts > 0) {
        swiglu(tensor(m, SYNTH_SH_GATE, l, 0), tensor(m, SYNTH_SH_UP, l, 0), tensor(m, SYNTH_SH_DOWN, l, 0), d,
               c.shared_ffn_dim, xn, ye.data());
        for (int i = 0; i < d; ++i) y[i] += ye[i];
    }
}

template <class T> void embed(oracle_model* m, int tok, T* x) {
    const uint16_t* E = tensor(m, SYNTH_EMBED, -1, 0) + (size_t)tok * m->c.d_model;
    for (int i = 0; i < m->c.d_model; ++i) x[i] = bf<T>(E[i]);
}

template <class T> void head(oracle_model* m, const T* x, double* logits) {
    const int d = m->c.d_model, V = m->c.vocab;
    std::vector<T> xf(d), lg(V);
    rmsnorm(x, tensor(m, SYNTH_FINAL_NORM, -1, 0), d, (T)m->c.rms_eps, xf.data());
    matvec(tensor(m, SYNTH_LM_HEAD, -1, 0), V, d, xf.data(), lg.data());
    for (int i = 0; i < V; ++i) logits[i] = (double)lg[i];
}

int argmax(const double* v, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

template <class T>
int decode_impl(oracle_model* m, oracle_kv* kv, const int32_t* tokens, const int32_t* positions, int B, int Tn,
                int absorbed, double* logits, int32_t* ridx, double* rw, double* rmargin, int32_t* accept) {
    const oracle_cfg& c = m->c;
    const int d = c.d_model, M = B * Tn, L = c.n_layers, k = c.top_k;
    std::vector<T> x((size_t)M * d), xn(d), ya(d), yf(d);
    for (int t = 0; t < M; ++t) embed(m, tokens[t], &x[(size_t)t * d]);
    std::vector<int32_t> li(k > 0 ? k : 1);
    std::vector<T> lw(k > 0 ? k : 1);
    /* layer-major order: within a layer, each sequence's tokens in order, so a
     * token's K/V is in the cache before the next token of that sequence
     * attends (causal within the step) */
    for (int l = 0; l < L; ++l) {
        for (int b = 0; b < B; ++b) {
            for (int t = 0; t < Tn; ++t) {
                const int mt = b * Tn + t, p = positions[b] + t;
                T* xt = &x[(size_t)mt * d];
                rmsnorm(xt, tensor(m, SYNTH_ATTN_NORM, l, 0), d, (T)c.rms_eps, xn.data());
                attention_token<T>(m, kv, l, b, p, xn.data(), absorbed, ya.data());
                for (int i = 0; i < d; ++i) xt[i] += ya[i];
                rmsnorm(xt, tensor(m, SYNTH_FFN_NORM, l, 0), d, (T)c.rms_eps, xn.data());
                T margin = 0;
                ffn_token<T>(m, l, xn.data(), yf.data(), li.data(), lw.data(), &margin);
                for (int i = 0; i < d; ++i) xt[i] += yf[i];
                if (c.n_routed_experts > 0) {
                    size_t o = ((size_t)l * M + mt);
                    if (ridx) for (int j = 0; j < k; ++j) ridx[o * k + j] = li[j];
                    if (rw) for (int j = 0; j < k; ++j) rw[o * k + j] = (double)lw[j];
                    if (rmargin) rmargin[o] = (double)margin;
                }
            }
        }
        if (m->lazy) release_layer(m, l);
    }
    std::vector<double> own;
    if (!logits && accept) { own.resize((size_t)M * c.vocab); logits = own.data(); }
    std::vector<double> lg((size_t)c.vocab);
    for (int mt = 0; mt < M; ++mt) head(m, &x[(size_t)mt * d], logits ? logits + (size_t)mt * c.vocab : lg.data());
    if (accept) {
        /* greedy verification: token t+1 of the block is accepted when it equals
         * the argmax (ties -> lower id) of the logits at block position t; the
         * acceptance length counts the accepted drafts plus the one token the
         * model always emits */
        for (int b = 0; b < B; ++b) {
            int a = 0;
            while (a < Tn - 1 && argmax(logits + (size_t)(b * Tn + a) * c.vocab, c.vocab) == tokens[b * Tn + a + 1]) ++a;
            accept[b] = a + 1;
        }
    }
    return 0;
}

/* brute force from position 0: K/V for all positions recomputed per layer,
 * explicit causal attention matrix, no cache object at all */
template <class T> int full_impl(oracle_model* m, const int32_t* tokens, int B, int P, double* logits) {
    const oracle_cfg& c = m->c;
    const int d = c.d_model, L = c.n_layers;
    for (int b = 0; b < B; ++b) {
        std::vector<T> X((size_t)P * d), XN((size_t)P * d), Y(d);
        for (int p = 0; p < P; ++p) embed(m, tokens[b * P + p], &X[(size_t)p * d]);
        for (int l = 0; l < L; ++l) {
            for (int p = 0; p < P; ++p)
                rmsnorm(&X[(size_t)p * d], tensor(m, SYNTH_ATTN_NORM, l, 0), d, (T)c.rms_eps, &XN[(size_t)p * d]);
            std::vector<T> O; /* [P][heads*vdim] */
            int odim;
            if (c.attn_kind == 0) {
                const int Hq = c.n_q_heads, Hkv = c.n_kv_heads, hd = c.head_dim, group = Hq / Hkv;
                odim = Hq * hd;
                std::vector<T> Q((size_t)P * Hq * hd), K((size_t)P * Hkv * hd), V((size_t)P * Hkv * hd);
                for (int p = 0; p < P; ++p) {
                    matvec(tensor(m, SYNTH_WQ, l, 0), Hq * hd, d, &XN[(size_t)p * d], &Q[(size_t)p * Hq * hd]);
                    matvec(tensor(m, SYNTH_WK, l, 0), Hkv * hd, d, &XN[(size_t)p * d], &K[(size_t)p * Hkv * hd]);
                    matvec(tensor(m, SYNTH_WV, l, 0), Hkv * hd, d, &XN[(size_t)p * d], &V[(size_t)p * Hkv * hd]);
                    for (int h = 0; h < Hq; ++h) rope(&Q[((size_t)p * Hq + h) * hd], hd, p, c.rope_theta);
                    for (int g = 0; g < Hkv; ++g) rope(&K[((size_t)p * Hkv + g) * hd], hd, p, c.rope_theta);
                }
                /* the cache stores bf16: round K and V the same way */
                for (auto& v : K) v = bf<T>(to_bf16(v));
                for (auto& v : V) v = bf<T>(to_bf16(v));
                O.assign((size_t)P * odim, 0);
                const T scale = (T)1 / std::sqrt((T)hd);
                std::vector<T> S((size_t)P * P);
                for (int h = 0; h < Hq; ++h) {
                    int g = h / group;
                    /* full score matrix, masked above the diagonal */
                    for (int i = 0; i < P; ++i)
                        for (int j = 0; j < P; ++j) {
                            T acc = 0;
                            for (int e = 0; e < hd; ++e)
                                acc += Q[((size_t)i * Hq + h) * hd + e] * K[((size_t)j * Hkv + g) * hd + e];
                            S[(size_t)i * P + j] = j <= i ? acc * scale : -std::numeric_limits<T>::infinity();
                        }
                    for (int i = 0; i < P; ++i) {
                        std::vector<T> pr(i + 1);
                        softmax(&S[(size_t)i * P], i + 1, pr.data());
                        for (int j = 0; j <= i; ++j)
                            for (int e = 0; e < hd; ++e)
                                O[(size_t)i * odim + h * hd + e] += pr[j] * V[((size_t)j * Hkv + g) * hd + e];
                    }
                }
            } else {
                const int H = c.n_q_heads, ql = c.q_lora_rank, kl = c.kv_lora_rank;
                const int nope = c.qk_nope_dim, rd = c.qk_rope_dim, vd = c.v_head_dim, qh = nope + rd;
                odim = H * vd;
                std::vector<T> Q((size_t)P * H * qh), C((size_t)P * kl), R((size_t)P * rd);
                std::vector<T> cq(ql), cqn(ql), kva(kl + rd);
                for (int p = 0; p < P; ++p) {
                    const T* xn = &XN[(size_t)p * d];
                    matvec(tensor(m, SYNTH_WDQ, l, 0), ql, d, xn, cq.data());
                    rmsnorm(cq.data(), tensor(m, SYNTH_Q_NORM, l, 0), ql, (T)c.rms_eps, cqn.data());
                    matvec(tensor(m, SYNTH_WUQ, l, 0), H * qh, ql, cqn.data(), &Q[(size_t)p * H * qh]);
                    for (int h = 0; h < H; ++h) rope(&Q[((size_t)p * H + h) * qh + nope], rd, p, c.rope_theta);
                    matvec(tensor(m, SYNTH_WDKV, l, 0), kl + rd, d, xn, kva.data());
                    rmsnorm(kva.data(), tensor(m, SYNTH_KV_NORM, l, 0), kl, (T)c.rms_eps, &C[(size_t)p * kl]);
                    rope(&kva[kl], rd, p, c.rope_theta);
                    for (int i = 0; i < rd; ++i) R[(size_t)p * rd + i] = kva[kl + i];
                }
                for (auto& v : C) v = bf<T>(to_bf16(v));
                for (auto& v : R) v = bf<T>(to_bf16(v));
                /* decompress K_nope and V for every position and head (plain MLA) */
                const uint16_t* Wukv = tensor(m, SYNTH_WUKV, l, 0);
                std::vector<T> KN((size_t)P * H * nope), VV((size_t)P * H * vd);
                for (int p = 0; p < P; ++p)
                    for (int h = 0; h < H; ++h) {
                        const uint16_t* Wuk = Wukv + (size_t)h * (nope + vd) * kl;
                        matvec(Wuk, nope, kl, &C[(size_t)p * kl], &KN[((size_t)p * H + h) * nope]);
                        matvec(Wuk + (size_t)nope * kl, vd, kl, &C[(size_t)p * kl], &VV[((size_t)p * H + h) * vd]);
                    }
                O.assign((size_t)P * odim, 0);
                const T scale = (T)1 / std::sqrt((T)qh);
                for (int h = 0; h < H; ++h)
                    for (int i = 0; i < P; ++i) {
                        std::vector<T> s(i + 1), pr(i + 1);
                        for (int j = 0; j <= i; ++j) {
                            T acc = 0;
                            for (int e = 0; e < nope; ++e)
                                acc += Q[((size_t)i * H + h) * qh + e] * KN[((size_t)j * H + h) * nope + e];
                            for (int e = 0; e < rd; ++e)
                                acc += Q[((size_t)i * H + h) * qh + nope + e] * R[(size_t)j * rd + e];
                            s[j] = acc * scale;
                        }
                        softmax(s.data(), i + 1, pr.data());
                        for (int j = 0; j <= i; ++j)
                            for (int e = 0; e < vd; ++e)
                                O[(size_t)i * odim + h * vd + e] += pr[j] * VV[((size_t)j * H + h) * vd + e];
                    }
            }
            for (int p = 0; p < P; ++p) {
                T* xt = &X[(size_t)p * d];
                matvec(tensor(m, SYNTH_WO, l, 0), d, odim, &O[(size_t)p * odim], Y.data());
                for (int i = 0; i < d; ++i) xt[i] += Y[i];
                std::vector<T> xn(d);
                rmsnorm(xt, tensor(m, SYNTH_FFN_NORM, l, 0), d, (T)c.rms_eps, xn.data());
                ffn_token<T>(m, l, xn.data(), Y.data(), nullptr, nullptr, nullptr);
                for (int i = 0; i < d; ++i) xt[i] += Y[i];
            }
        }
        for (int p = 0; p < P; ++p) head(m, &X[(size_t)p * d], logits + ((size_t)b * P + p) * c.vocab);
    }
    return 0;
}

bool cfg_ok(const oracle_cfg* c) {
    if (!c || c->n_layers < 1 || c->d_model < 1 || c->vocab < 1) return false;
    if (c->attn_kind == 0) {
        if (c->n_q_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 2 || c->head_dim % 2) return false;
        if (c->n_q_heads % c->n_kv_heads) return false;
    } else if (c->attn_kind == 1) {
        if (c->n_q_heads < 1 || c->q_lora_rank < 1 || c->kv_lora_rank < 1 || c->qk_nope_dim < 1 ||
            c->qk_rope_dim < 2 || c->qk_rope_dim % 2 || c->v_head_dim < 1)
            return false;
    } else {
        return false;
    }
    if (c->n_routed_experts < 0 || (c->n_routed_experts > 0 && (c->top_k < 1 || c->top_k > c->n_routed_experts)))
        return false;
    if (c->n_shared_experts < 0 || c->n_shared_experts > 1) return false;
    if (c->expert_format != 0 && c->expert_format != 1) return false;
    if (c->expert_format == 1 && (c->d_model % SYNTH_MX_BLOCK || c->ffn_dim % SYNTH_MX_BLOCK ||
                                  c->shared_ffn_dim % SYNTH_MX_BLOCK))
        return false;
    return true;
}

}  // namespace

extern "C" {

oracle_model* oracle_create(const oracle_cfg* cfg, uint64_t seed, int lazy, int gen_threads) {
    if (!cfg_ok(cfg)) return nullptr;
    oracle_model* m = new oracle_model();
    m->c = *cfg;
    m->d = dims_of(*cfg);
    m->seed = seed;
    m->lazy = lazy;
    m->gen_threads = gen_threads;
    return m;
}

void oracle_destroy(oracle_model* m) { delete m; }

int oracle_set_tensor(oracle_model* m, int32_t kind, int32_t layer, int32_t expert, const uint16_t* data, int64_t n) {
    int32_t rows, cols;
    float s, mu;
    if (!m || !data || synth_weight_spec(&m->d, kind, &rows, &cols, &s, &mu) != 0) return -1;
    if (n != (int64_t)rows * cols) return -1;
    TKey k(kind, layer, expert);
    m->w[k].assign(data, data + n);
    m->pinned.insert(k);
    return 0;
}

int64_t oracle_get_tensor(oracle_model* m, int32_t kind, int32_t layer, int32_t expert, uint16_t* out, int64_t cap) {
    int32_t rows, cols;
    float s, mu;
    if (!m || synth_weight_spec(&m->d, kind, &rows, &cols, &s, &mu) != 0) return -1;
    int64_t n = (int64_t)rows * cols;
    if (out) {
        if (cap < n) return -1;
        const uint16_t* t = tensor(m, kind, layer, expert);
        std::memcpy(out, t, (size_t)n * 2);
    }
    return n;
}

oracle_kv* oracle_kv_create(const oracle_model* m, int32_t batch, int32_t max_pos) {
    if (!m || batch < 1 || max_pos < 1) return nullptr;
    oracle_kv* kv = new oracle_kv();
    kv->L = m->c.n_layers;
    kv->B = batch;
    kv->max_pos = max_pos;
    kv->row = m->c.attn_kind == 0 ? 2 * m->c.n_kv_heads * m->c.head_dim : m->c.kv_lora_rank + m->c.qk_rope_dim;
    kv->attn_kind = m->c.attn_kind;
    kv->half = m->c.attn_kind == 0 ? m->c.n_kv_heads * m->c.head_dim : 0;
    kv->data.assign((size_t)kv->L * batch * max_pos * kv->row, 0);
    return kv;
}

void oracle_kv_destroy(oracle_kv* kv) { delete kv; }

int32_t oracle_kv_row_len(const oracle_kv* kv) { return kv ? kv->row : -1; }

int oracle_kv_prefill(oracle_kv* kv, uint64_t seed, int32_t ctx, int gen_threads) {
    if (!kv || ctx < 0 || ctx > kv->max_pos) return -1;
    if (ctx == 0) return 0;
    /* pre-filled entries are bf16 N(0, 1) draws, position-major per stream:
     * GQA has a K stream and a V stream of row length Hkv*hd, MLA one latent
     * stream of row length kv_lora + rope */
    const int nstreams = kv->attn_kind == 0 ? 2 : 1;
    const int rl = kv->attn_kind == 0 ? kv->half : kv->row;
    std::vector<uint16_t> tmp((size_t)ctx * rl);
    for (int l = 0; l < kv->L; ++l)
        for (int b = 0; b < kv->B; ++b)
            for (int s = 0; s < nstreams; ++s) {
                int kind = kv->attn_kind == 1 ? SYNTH_KV_LATENT : (s == 0 ? SYNTH_KV_K : SYNTH_KV_V);
                synth_fill_bf16(tmp.data(), tmp.size(), seed, synth_tensor_id(kind, l, b), 1.0f, 0.0f, 0,
                                gen_threads);
                for (int p = 0; p < ctx; ++p)
                    std::memcpy(kv->at(l, b, p) + s * rl, &tmp[(size_t)p * rl], (size_t)rl * 2);
            }
    return 0;
}

int oracle_kv_rows(const oracle_kv* kvc, int32_t layer, int32_t seq, int32_t pos0, int32_t n, uint16_t* out,
                   int write) {
    oracle_kv* kv = const_cast<oracle_kv*>(kvc);
    if (!kv || !out || layer < 0 || layer >= kv->L || seq < 0 || seq >= kv->B || pos0 < 0 || n < 0 ||
        pos0 + n > kv->max_pos)
        return -1;
    for (int p = 0; p < n; ++p) {
        if (write)
            std::memcpy(kv->at(layer, seq, pos0 + p), out + (size_t)p * kv->row, (size_t)kv->row * 2);
        else
            std::memcpy(out + (size_t)p * kv->row, kv->at(layer, seq, pos0 + p), (size_t)kv->row * 2);
    }
    return 0;
}

int oracle_decode(oracle_model* m, oracle_kv* kv, const int32_t* tokens, const int32_t* positions, int32_t B, int32_t T,
                  int precision, int mla_absorbed, double* logits, int32_t* route_idx, double* route_w,
                  double* route_margin, int32_t* accept) {
    if (!m || !kv || !tokens || !positions || B < 1 || T < 1 || B > kv->B) return -1;
    for (int b = 0; b < B; ++b)
        if (positions[b] < 0 || positions[b] + T > kv->max_pos) return -1;
    for (int i = 0; i < B * T; ++i)
        if (tokens[i] < 0 || tokens[i] >= m->c.vocab) return -1;
    if (precision == 64)
        return decode_impl<double>(m, kv, tokens, positions, B, T, mla_absorbed, logits, route_idx, route_w,
                                   route_margin, accept);
    if (precision == 32)
        return decode_impl<float>(m, kv, tokens, positions, B, T, mla_absorbed, logits, route_idx, route_w,
                                  route_margin, accept);
    return -1;
}

int oracle_full_recompute(oracle_model* m, const int32_t* tokens, int32_t B, int32_t P, int precision, double* logits) {
    if (!m || !tokens || !logits || B < 1 || P < 1) return -1;
    if (precision == 64) return full_impl<double>(m, tokens, B, P, logits);
    if (precision == 32) return full_impl<float>(m, tokens, B, P, logits);
    return -1;
}

void oracle_rmsnorm(const double* x, const uint16_t* gain, int32_t n, double eps, double* out) {
    rmsnorm<double>(x, gain, n, eps, out);
}
void oracle_rope(double* x, int32_t dim, int32_t pos, double theta) { rope<double>(x, dim, pos, theta); }
void oracle_softmax(const double* x, int32_t n, double* out) { softmax<double>(x, n, out); }
void oracle_topk(const double* logits, int32_t n, int32_t k, int32_t* idx, double* w, double* margin) {
    topk<double>(logits, n, k, idx, w, margin);
}
double oracle_silu(double z) { return silu<double>(z); }
void oracle_attend(const double* q, const uint16_t* K, const uint16_t* V, int32_t n, int32_t hd, double scale,
                   double* out) {
    attend_rows<double>(q, K, (size_t)hd, V, (size_t)hd, n, hd, scale, out);
}

}  // extern "C"
