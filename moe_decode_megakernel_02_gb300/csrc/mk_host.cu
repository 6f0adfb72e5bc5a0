// mk_host.cu -- C ABI of the decode megakernel (include/mk.h): validation,
// weight packing, scratch layout, paged KV cache and the cooperative launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/mk.h"
#include "mk_kernel.cuh"

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

#define CK(call)                                                                                        \
    do {                                                                                                \
        cudaError_t e_ = (call);                                                                        \
        if (e_ != cudaSuccess)                                                                          \
            return fail(e_ == cudaErrorMemoryAllocation ? MK_ERR_OOM : MK_ERR_CUDA, "%s: %s (%s:%d)", #call, \
                        cudaGetErrorString(e_), __FILE__, __LINE__);                                    \
    } while (0)

constexpr uint32_t MODEL_MAGIC = 0x4d4b4d44u;  // "MKMD"
constexpr uint32_t KV_MAGIC = 0x4d4b4b56u;     // "MKKV"

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// host-side fault injection: MK_FAULT names the failure to report
bool fault(const char* what) {
    const char* e = getenv("MK_FAULT");
    return e && strcmp(e, what) == 0;
}

uint64_t next_serial() {
    static std::atomic<uint64_t> n{0};
    return ++n;
}

}  // namespace

struct mk_model {
    uint32_t magic;
    mk_config cfg;
    int dev, sms, G;
    uint16_t* wblob = nullptr;
    size_t wbytes = 0;
    uint8_t* sblob = nullptr;
    size_t sbytes = 0;
    std::vector<mk::Layer> layers;
    mk::Layer* d_layers = nullptr;
    mk::Params base;  // everything except the per-step fields
    bool rfuse_ok;    // the router can be folded into the output projection
    bool qfuse_ok;    // MLA: the absorbed query can be computed by the QB CTAs
    bool ufuse_ok;    // MLA: the value up-projection can be computed by the combine CTAs
    unsigned* ctr = nullptr;
    size_t ctr_n = 0;
    unsigned* status = nullptr;
    int* dbg_idx = nullptr;
    float* dbg_w = nullptr;
    float* dbg_margin = nullptr;
    int last_M = 0;
    bool last_noalloc = false;  // the last step ran in the static scratch (its routing is not in dbg_*)
    // one launch per stage (mk_decode_step_unfused): token ids and positions
    // are copied into these, and a graph of the launches is kept per shape
    int* u_tok = nullptr;
    int* u_pos = nullptr;
    std::map<std::tuple<const void*, int, int, const void*, const void*>, cudaGraphExec_t> graphs;
    const int* last_amax = nullptr;  // argmax of the last step's rows (steps given an accept buffer)
    uint64_t steps = 0;
    uint64_t serial = 0;  // distinct per loaded model in this process
    // KV caches of this model not yet freed; a model freed while some are
    // alive gives up its device memory at once and its host record (which
    // the caches still read for their dimensions) when the last one goes
    int live_kv = 0;
    bool released = false;
    // MK_DEBUG: offsets of the 256-byte guards after each scratch region
    // (pattern 0xA5, written at load, checked by mk_step_status)
    std::vector<size_t> guards;
};

struct mk_kv {
    uint32_t magic;
    mk_model* m;
    int batch, max_ctx, pps;
    size_t page_elems, layer_elems;
    uint16_t* pool = nullptr;
    int* btab = nullptr;
    void* tmaps = nullptr;  // MLA: the latent and rope tensor maps of the pool (device memory)
    std::vector<int> h_btab;
};

namespace {

struct Dims {
    int L, d, V, gqa, Hq, Hkv, hd, ql, kl, nope, rd, vd, E, k, sh, ffn, sffn, Mx;
    int a_rows, o_in, qh;
    int f8;  // MXFP8 expert weights
};

Dims dims_of(const mk_config& c) {
    Dims d;
    d.L = c.n_layers; d.d = c.d_model; d.V = c.vocab; d.gqa = c.attn_kind == MK_ATTN_GQA;
    d.Hq = c.n_q_heads; d.Hkv = c.n_kv_heads; d.hd = c.head_dim;
    d.ql = c.q_lora_rank; d.kl = c.kv_lora_rank; d.nope = c.qk_nope_dim; d.rd = c.qk_rope_dim; d.vd = c.v_head_dim;
    d.E = c.n_routed_experts; d.k = c.top_k; d.sh = c.n_shared_experts; d.ffn = c.ffn_dim; d.sffn = c.shared_ffn_dim;
    d.Mx = c.max_batch * c.max_tokens_per_seq;
    d.qh = d.nope + d.rd;
    d.a_rows = d.gqa ? (d.Hq + 2 * d.Hkv) * d.hd : d.ql + d.kl + d.rd;
    d.o_in = d.gqa ? d.Hq * d.hd : d.Hq * d.vd;
    d.f8 = c.expert_format == MK_EXPERT_MXFP8;
    return d;
}

bool k_ok(int K) { return K == 128 || (K > 0 && K % 256 == 0 && (K <= 2048 || K % 1024 == 0 || K % 512 == 0)); }

// unit width for an expert of Fi intermediate dimensions on a d-wide model:
// about 384 KB of gate/up weights per unit; 0 if no width divides Fi
int unit_width(int Fi, int d) {
    const int target = 98304 / d;
    for (int F : {64, 48, 32, 16})
        if ((F <= target || F == 16) && Fi % F == 0) return F;
    return 0;
}

// gate/up K panel (as for every GEMV) and rows per tile dividing 2F
void unit_geometry(int d, int F, int& Kc, int& R, int& Rd) {
    Kc = d > 2048 ? (d % 1024 == 0 ? 1024 : (d % 512 == 0 ? 512 : 256)) : d;
    R = (mk::TILE_MAX / (2 * Kc)) / 8 * 8;
    if (R > 2 * F) R = 2 * F;
    while (R > 8 && (2 * F) % R) R -= 8;
    Rd = mk::SLOT_BYTES / (2 * F) / 128 * 128;  // down tiles fill a ring slot
    if (Rd > d) Rd = d;
}

// MXFP8 experts: units 64 wide (two 32-code scale blocks of a down row);
// gate/up tiles of R = 32768 / d whole rows (one K panel: 32 KB of codes)
// followed by their scales; down tiles of Rd rows x 64 codes (32 KB, at most
// d rows) followed by theirs
struct F8Geom {
    int F, R, Rd, tb_gu, tb_dn;
    size_t gu_bytes, dn_bytes;  // per expert
};
F8Geom f8_geometry(int d, int Fi) {
    F8Geom g;
    g.F = 64;
    g.R = 32768 / d;
    g.Rd = std::min(d, 32768 / g.F);
    g.tb_gu = g.R * d + g.R * (d / 32);
    g.tb_dn = g.Rd * g.F + g.Rd * (g.F / 32);
    g.gu_bytes = (size_t)(2 * Fi / g.R) * g.tb_gu;
    g.dn_bytes = (size_t)(Fi / g.F) * (d / g.Rd) * g.tb_dn;
    return g;
}

int validate(const mk_config* c) {
    if (!c) return fail(MK_ERR_INVALID_ARG, "cfg is NULL");
    if (c->n_layers < 1 || c->d_model < 1 || c->vocab < 1 || c->max_batch < 1 || c->max_tokens_per_seq < 1 ||
        c->max_ctx < 1)
        return fail(MK_ERR_INVALID_ARG, "non-positive dimension");
    if (c->kv_page_size != mk::PAGE) return fail(MK_ERR_UNSUPPORTED, "kv_page_size must be %d", mk::PAGE);
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f)) return fail(MK_ERR_INVALID_ARG, "rms_eps/rope_theta");
    const Dims d = dims_of(*c);
    if (d.Mx > mk::MAX_M) return fail(MK_ERR_UNSUPPORTED, "max_batch*max_tokens_per_seq > %d", mk::MAX_M);
    if (c->max_tokens_per_seq > 16) return fail(MK_ERR_UNSUPPORTED, "max_tokens_per_seq > 16");
    if (!k_ok(d.d) || d.d % 8) return fail(MK_ERR_UNSUPPORTED, "d_model must be 128 or a multiple of 256");
    if (c->attn_kind == MK_ATTN_GQA) {
        if (d.Hq < 1 || d.Hkv < 1 || d.Hq % d.Hkv) return fail(MK_ERR_INVALID_ARG, "GQA heads");
        if (d.hd != 64 && d.hd != 128) return fail(MK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
        if (d.Hq / d.Hkv * c->max_tokens_per_seq > 8)
            return fail(MK_ERR_UNSUPPORTED, "GQA: (q heads per kv head) * tokens per step must be <= 8");
        if (!k_ok(d.o_in)) return fail(MK_ERR_UNSUPPORTED, "n_q_heads*head_dim");
    } else if (c->attn_kind == MK_ATTN_MLA) {
        if (d.Hq != mk::MLA_H || d.kl != mk::MLA_KL || d.rd != mk::MLA_RD || d.nope != 128)
            return fail(MK_ERR_UNSUPPORTED, "MLA kernel implements 16 heads, kv_lora 512, rope 64, nope 128");
        if (d.vd < 8 || d.vd % 8 || !k_ok(d.ql) || !k_ok(d.o_in)) return fail(MK_ERR_UNSUPPORTED, "MLA dims");
    } else {
        return fail(MK_ERR_INVALID_ARG, "attn_kind");
    }
    if (d.E < 0 || d.E > mk::MAX_E) return fail(MK_ERR_UNSUPPORTED, "n_routed_experts > %d", mk::MAX_E);
    if (d.E > 0) {
        if (d.k < 1 || d.k > mk::MAX_K || d.k > d.E) return fail(MK_ERR_UNSUPPORTED, "top_k");
        if (d.ffn < 8 || d.ffn % 8 || !k_ok(d.ffn) || d.E % 8) return fail(MK_ERR_UNSUPPORTED, "expert ffn / count");
    }
    if (d.sh < 0 || d.sh > 1) return fail(MK_ERR_UNSUPPORTED, "n_shared_experts must be 0 or 1");
    if (d.sh && (d.sffn % 8 || !k_ok(d.sffn))) return fail(MK_ERR_UNSUPPORTED, "shared_ffn_dim");
    if (d.E == 0 && !d.sh) return fail(MK_ERR_UNSUPPORTED, "model needs routed or shared experts");
    if (d.E && !unit_width(d.ffn, d.d)) return fail(MK_ERR_UNSUPPORTED, "ffn_dim must be a multiple of 16");
    if (d.sh && !unit_width(d.sffn, d.d)) return fail(MK_ERR_UNSUPPORTED, "shared_ffn_dim must be a multiple of 16");
    if (d.V % 8) return fail(MK_ERR_UNSUPPORTED, "vocab must be a multiple of 8");
    if (c->expert_format != MK_EXPERT_BF16 && c->expert_format != MK_EXPERT_MXFP8)
        return fail(MK_ERR_INVALID_ARG, "expert_format");
    if (d.f8) {
        if (d.d != 512 && d.d != 1024 && d.d != 2048) return fail(MK_ERR_UNSUPPORTED, "MXFP8 experts: d_model 512, 1024 or 2048");
        if ((d.E && d.ffn % 64) || (d.sh && d.sffn % 64))
            return fail(MK_ERR_UNSUPPORTED, "MXFP8 experts: ffn_dim and shared_ffn_dim multiples of 64");
        static_assert(32768 + 1024 <= mk::SLOT_BYTES - 16, "an MXFP8 tile fits a ring slot");
    }
    return MK_OK;
}

int gemv_items_host(const mk::Gemv& g) { return g.n_rb * g.n_kc; }

// K panel of a matrix with K columns: the whole row up to 2048, else the
// largest of 1024 / 512 / 256 dividing K; narrower (down to 256) while Mx
// tokens' staged input rows would not fit the staging area at once (models
// loaded for many tokens per step: their stages then stage each panel once
// per run of items instead of re-staging token chunks for every tile)
int panel_width(int K, int Mx) {
    int Kc = K;
    if (K > 2048) Kc = K % 1024 == 0 ? 1024 : (K % 512 == 0 ? 512 : 256);
    while (Kc > 256 && !mk::stage_fits(Mx, Kc) && K % (Kc / 2) == 0) Kc /= 2;
    return Kc;
}

void make_gemv(mk::Gemv& g, const uint16_t* W, int N, int K, int in_kind, const float* src, int src_stride,
               const uint16_t* gain, int out_kind, float* dst, int dst_stride, int Mx, float* dst2 = nullptr) {
    std::memset(&g, 0, sizeof g);
    const int Kc = panel_width(K, Mx);
    int R = (mk::TILE_MAX / (2 * Kc)) / 8 * 8;
    if (R > N) R = N;
    g.W = W;
    g.N = N;
    g.K = K;
    g.Kc = Kc;
    g.R = R;
    g.n_kc = K / Kc;
    g.n_rb = (N + R - 1) / R;
    g.in_kind = in_kind;
    g.src = src;
    g.src_stride = src_stride;
    g.gain = gain;
    g.out_kind = out_kind;
    g.dst = dst;
    g.dst_stride = dst_stride;
    g.dst2 = dst2;
}

// canonical [rows][K] block -> rows [row0, row0+rows) of a packed [n_kc][N][Kc] matrix
int pack_rows(uint16_t* dst, int N, int K, int Kc, int row0, const void* src, int rows, size_t src_row_pitch,
              cudaStream_t s) {
    const int n_kc = K / Kc;
    for (int kc = 0; kc < n_kc; ++kc) {
        CK(cudaMemcpy2DAsync(dst + (size_t)kc * N * Kc + (size_t)row0 * Kc, (size_t)Kc * 2,
                             static_cast<const uint16_t*>(src) + (size_t)kc * Kc, src_row_pitch, (size_t)Kc * 2,
                             rows, cudaMemcpyDefault, s));
    }
    return MK_OK;
}

// SwiGLU expert as units of F intermediate dimensions (see mk::FfnKind):
// gate/up rows unit-major, [n_kc][2 Fi][Kc]; row 2F u + j is gate row uF + j
// (j < F) or up row uF + j - F
__global__ void pack_gu_units(uint16_t* __restrict__ dst, const uint16_t* __restrict__ gate,
                              const uint16_t* __restrict__ up, int Fi, int d, int F, int Kc) {
    const size_t per_kc = (size_t)2 * Fi * Kc, n8 = (size_t)(d / Kc) * per_kc / 8;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const size_t e = i * 8;
        const int kc = (int)(e / per_kc);
        const size_t rem = e - (size_t)kc * per_kc;
        const int row = (int)(rem / Kc), k = (int)(rem - (size_t)row * Kc);
        const int u = row / (2 * F), j = row - u * 2 * F;
        const uint16_t* src = j < F ? gate + (size_t)(u * F + j) * d : up + (size_t)(u * F + j - F) * d;
        *reinterpret_cast<uint4*>(dst + e) = *reinterpret_cast<const uint4*>(src + (size_t)kc * Kc + k);
    }
}

// MXFP8 gate/up tiles: tile t holds unit-major rows t R .. t R + R - 1 (row
// 2F u + j is gate row uF + j for j < F, else up row uF + j - F): their d
// codes each, then their d / 32 scale bytes each. One work item per 16-byte
// chunk of codes or per scale byte.
__global__ void pack_gu_f8(uint8_t* __restrict__ dst, const uint8_t* __restrict__ gq, const uint8_t* __restrict__ uq,
                           const uint8_t* __restrict__ gs, const uint8_t* __restrict__ us, int Fi, int d, int F, int R,
                           int tb) {
    const int cpr = d / 16 + d / 32;
    const size_t n = (size_t)2 * Fi * cpr;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int row = (int)(i / cpr), k = (int)(i - (size_t)row * cpr);
        const int u = row / (2 * F), j = row - u * 2 * F;
        const bool gate = j < F;
        const int sr = gate ? u * F + j : u * F + j - F;
        const int t = row / R, rr = row - t * R;
        uint8_t* tile = dst + (size_t)t * tb;
        if (k < d / 16) {
            *reinterpret_cast<uint4*>(tile + (size_t)rr * d + 16 * k) =
                *reinterpret_cast<const uint4*>((gate ? gq : uq) + (size_t)sr * d + 16 * k);
        } else {
            const int kk = k - d / 16;
            tile[(size_t)R * d + rr * (d / 32) + kk] = (gate ? gs : us)[(size_t)sr * (d / 32) + kk];
        }
    }
}

// MXFP8 down tiles: unit u, tile t: rows t Rd .. t Rd + Rd - 1 of the down
// matrix, their codes [uF, uF + F) each, then those codes' F / 32 scales each
__global__ void pack_dn_f8(uint8_t* __restrict__ dst, const uint8_t* __restrict__ q, const uint8_t* __restrict__ sc,
                           int Fi, int d, int F, int Rd, int tb) {
    const int nt = d / Rd, nu = Fi / F, cpr = F / 16 + F / 32;
    const size_t n = (size_t)nu * d * cpr;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t rid = i / cpr;
        const int k = (int)(i - rid * cpr);
        const int u = (int)(rid / d), r = (int)(rid - (size_t)u * d);
        const int t = r / Rd, rr = r - t * Rd;
        uint8_t* tile = dst + ((size_t)u * nt + t) * tb;
        if (k < F / 16) {
            *reinterpret_cast<uint4*>(tile + (size_t)rr * F + 16 * k) =
                *reinterpret_cast<const uint4*>(q + (size_t)r * Fi + (size_t)u * F + 16 * k);
        } else {
            const int kk = k - F / 16;
            tile[(size_t)Rd * F + rr * (F / 32) + kk] = sc[(size_t)r * (Fi / 32) + u * (F / 32) + kk];
        }
    }
}

// down matrix [d][Fi] -> per unit [nu][d][F]
__global__ void pack_dn_units(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src, int Fi, int d, int F) {
    const size_t n8 = (size_t)d * Fi / 8, per_u = (size_t)d * F;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const size_t e = i * 8;
        const int u = (int)(e / per_u);
        const size_t rem = e - (size_t)u * per_u;
        const int r = (int)(rem / F), f = (int)(rem - (size_t)r * F);
        *reinterpret_cast<uint4*>(dst + e) = *reinterpret_cast<const uint4*>(src + (size_t)r * Fi + (size_t)u * F + f);
    }
}

__global__ void transpose_heads(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, int H, int rows_in,
                                int head_stride_rows, int cols) {
    // in: per head h, a [rows_in][cols] block starting at row h*head_stride_rows
    // out: per head h, [cols][rows_in]
    const size_t n = (size_t)H * rows_in * cols;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int h = (int)(i / ((size_t)rows_in * cols));
        const size_t r = i - (size_t)h * rows_in * cols;
        const int c = (int)(r / rows_in), q = (int)(r - (size_t)c * rows_in);
        out[i] = in[((size_t)h * head_stride_rows + q) * cols + c];
    }
}

// W_uv per head and latent quarter, j-major: out[h][q][j][v] = W_uv[h][v][128 q + j]
// (from the canonical [H*(nope+vd)][kl] W_ukv, whose head h holds its W_uk
// rows, then its W_uv rows)
__global__ void pack_uv_quarters(uint16_t* __restrict__ out, const uint16_t* __restrict__ wukv, int H, int nope,
                                 int vd, int kl) {
    const size_t n = (size_t)H * vd * kl, per_h = (size_t)vd * kl, per_q = (size_t)128 * vd;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int h = (int)(i / per_h);
        const size_t r = i - h * per_h;
        const int q = (int)(r / per_q);
        const size_t r2 = r - q * per_q;
        const int j = (int)(r2 / vd), v = (int)(r2 - (size_t)j * vd);
        out[i] = wukv[((size_t)h * (nope + vd) + nope + v) * kl + (size_t)q * 128 + j];
    }
}

__global__ void kv_scatter(uint16_t* pool, const int* btab, int pps, size_t page_elems, int gqa, int Hkv, int hd,
                           int kl, int rd, int seq, int pos0, int n, int row, uint16_t* rows, int to_cache) {
    const size_t total = (size_t)n * row;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int p = (int)(i / row), j = (int)(i - (size_t)p * row);
        const int pos = pos0 + p;
        uint16_t* pg = pool + (size_t)btab[seq * pps + pos / mk::PAGE] * page_elems;
        const int pr = pos % mk::PAGE;
        size_t off;
        if (gqa) {
            const int isv = j >= Hkv * hd;
            const int jj = isv ? j - Hkv * hd : j;
            const int g = jj / hd, e = jj - g * hd;
            off = (size_t)g * 2 * mk::PAGE * hd + (size_t)isv * mk::PAGE * hd + (size_t)pr * hd + e;
        } else {
            off = j < kl ? (size_t)pr * kl + j : (size_t)mk::PAGE * kl + (size_t)pr * rd + (j - kl);
        }
        if (to_cache)
            pg[off] = rows[i];
        else
            rows[i] = pg[off];
    }
}

bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

long long wait_ns() {
    const char* e = getenv("MK_WAIT_NS");
    long long v = e ? atoll(e) : 0;
    return v > 0 ? v : 2000000000LL;
}

}  // namespace

extern "C" {

const char* mk_last_error(void) { return g_err.c_str(); }

// failures found in the library's other translation units (mk_synth.cu)
__attribute__((visibility("hidden"))) int mk_set_error_(int code, const char* msg) {
    g_err = msg;
    return code;
}
__attribute__((visibility("hidden"))) int mk_fault_oom_(void) {
    return fault("oom") ? fail(MK_ERR_OOM, "allocation refused (injected by MK_FAULT=oom)") : MK_OK;
}

int mk_load_weights(const mk_config* cfg, const mk_weight* table, int32_t n, void* stream, mk_model** out) {
    if (!out) return fail(MK_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    int rc = validate(cfg);
    if (rc) return rc;
    if (!table || n < 1) return fail(MK_ERR_INVALID_ARG, "empty weight table");
    if (fault("bad_arg")) return fail(MK_ERR_INVALID_ARG, "arguments rejected (injected by MK_FAULT=bad_arg)");
    if (fault("oom")) return fail(MK_ERR_OOM, "allocation refused (injected by MK_FAULT=oom)");
    cudaStream_t s = (cudaStream_t)stream;
    const Dims D = dims_of(*cfg);

    // ---- index the table ----
    std::map<std::tuple<int, int, int>, const void*> T;
    for (int i = 0; i < n; ++i) {
        const mk_weight& w = table[i];
        if (!w.data) return fail(MK_ERR_INVALID_ARG, "table[%d].data is NULL", i);
        auto key = std::make_tuple(w.kind, w.layer, w.expert);
        if (T.count(key)) return fail(MK_ERR_INVALID_ARG, "duplicate tensor kind %d layer %d expert %d", w.kind, w.layer, w.expert);
        T[key] = w.data;
    }
    auto need = [&](int kind, int layer, int expert, const void** p) -> int {
        auto it = T.find(std::make_tuple(kind, layer, expert));
        if (it == T.end()) return fail(MK_ERR_INVALID_ARG, "missing tensor kind %d layer %d expert %d", kind, layer, expert);
        *p = it->second;
        return MK_OK;
    };

    mk_model* m = new mk_model();
    m->magic = MODEL_MAGIC;
    m->serial = next_serial();
    m->cfg = *cfg;
    auto bail = [&](int code) {
        if (m->wblob) cudaFree(m->wblob);
        if (m->sblob) cudaFree(m->sblob);
        if (m->d_layers) cudaFree(m->d_layers);
        delete m;
        return code;
    };
    CK(cudaGetDevice(&m->dev));
    CK(cudaDeviceGetAttribute(&m->sms, cudaDevAttrMultiProcessorCount, m->dev));
    CK(cudaFuncSetAttribute(mk::megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mk::SMEM_TOTAL));
    int per_sm = 0;
    CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mk::megakernel, mk::NTHREADS, mk::SMEM_TOTAL));
    if (per_sm < 1) return bail(fail(MK_ERR_UNSUPPORTED, "megakernel does not fit on an SM"));
    m->G = m->sms < 255 ? m->sms : 255;

    // ---- packed weight layout ----
    const int L = D.L, d = D.d;
    struct Off { size_t a, qn, kvn, uq, ukT, uk, uv, uvq, o, router, gu, down, shgu, shdown, an, fn; };
    std::vector<Off> lo(L);
    size_t cur = 0;
    auto take = [&](size_t elems) { size_t o = cur; cur += align256(elems * 2) / 2; return o; };
    const size_t off_embed = take((size_t)D.V * d), off_lm = take((size_t)D.V * d), off_fn = take(d);
    for (int l = 0; l < L; ++l) {
        Off& o = lo[l];
        o.an = take(d);
        o.fn = take(d);
        o.a = take((size_t)D.a_rows * d);
        if (!D.gqa) {
            o.qn = take(D.ql);
            o.kvn = take(D.kl);
            o.uq = take((size_t)D.Hq * D.qh * D.ql);
            o.ukT = take((size_t)D.Hq * D.kl * D.nope);
            o.uk = take((size_t)D.Hq * D.nope * D.kl);
            o.uvq = take((size_t)D.Hq * D.vd * D.kl);
            o.uv = take((size_t)D.Hq * D.vd * D.kl);
        }
        o.o = take((size_t)d * D.o_in);
        // (MXFP8 experts: bytes of tiles, counted in 2-byte elements)
        if (D.E) {
            o.router = take((size_t)D.E * d);
            o.gu = take(D.f8 ? D.E * f8_geometry(d, D.ffn).gu_bytes / 2 : (size_t)D.E * 2 * D.ffn * d);
            o.down = take(D.f8 ? D.E * f8_geometry(d, D.ffn).dn_bytes / 2 : (size_t)D.E * d * D.ffn);
        }
        if (D.sh) {
            o.shgu = take(D.f8 ? f8_geometry(d, D.sffn).gu_bytes / 2 : (size_t)2 * D.sffn * d);
            o.shdown = take(D.f8 ? f8_geometry(d, D.sffn).dn_bytes / 2 : (size_t)d * D.sffn);
        }
    }
    m->wbytes = cur * 2;
    {
        cudaError_t e = cudaMalloc(&m->wblob, m->wbytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return bail(fail(MK_ERR_OOM, "weights: cudaMalloc(%zu) failed", m->wbytes));
        }
    }
    uint16_t* W = m->wblob;

    // ---- scratch layout (floats unless noted) ----
    const size_t Mx = D.Mx;
    const int Q8 = 8;
    size_t scur = 0;
    const bool dbg = getenv("MK_DEBUG") && atoi(getenv("MK_DEBUG")) > 0;
    auto stake = [&](size_t bytes) {
        const size_t o = scur;
        scur += align256(bytes);
        if (dbg) {  // a guard after the region
            m->guards.push_back(scur);
            scur += 256;
        }
        return o;
    };
    const size_t s_x = stake((size_t)(L + 1) * Mx * d * 4);
    const size_t s_a = stake((size_t)L * Mx * D.a_rows * 4);
    const size_t s_q = D.gqa ? 0 : stake((size_t)L * Mx * D.Hq * D.qh * 4);
    const size_t s_qlat = D.gqa ? 0 : stake((size_t)L * Mx * D.Hq * D.kl * 4);
    const size_t s_olat = D.gqa ? 0 : stake((size_t)L * Mx * D.Hq * D.kl * 4);
    const size_t s_o = stake((size_t)L * Mx * D.o_in * 4);
    const size_t s_rlog = D.E ? stake((size_t)L * Mx * mk::router_row(D.E) * 4) : 0;
    const size_t s_racc = D.E ? stake((size_t)L * mk::ROUTER_COPIES * Mx * mk::router_row(D.E) * 4) : 0;
    // expert units: per CTA, gate/up outputs and hidden values of at most one
    // expert's units for every token
    const size_t ubuf_stride = (size_t)3 * std::max(D.E ? D.ffn : 0, D.sh ? D.sffn : 0) * Mx;
    const size_t s_ubuf = stake((size_t)m->G * ubuf_stride * 4);
    const size_t part_rows = D.gqa ? (size_t)cfg->max_batch * D.Hkv * m->G * Q8 : (size_t)Mx * m->G * mk::MLA_H;
    const size_t s_part = stake(part_rows * (D.gqa ? D.hd : mk::MLA_KL) * 4);
    const size_t s_part_ml = stake(part_rows * 2 * 4);
    const int trace_cap = 8192;
    const bool tracing = getenv("MK_TRACE") && atoi(getenv("MK_TRACE")) > 0;
    const size_t s_trace = tracing ? stake((size_t)m->G * trace_cap * sizeof(mk::TraceRec)) : 0;
    const size_t s_trace_n = tracing ? stake((size_t)m->G * 4) : 0;
    const size_t s_newlat = stake(Mx * mk::MLA_D * 2);
    const size_t s_amax = stake(Mx * 4);
    const size_t s_rss = stake((size_t)(L + 1) * 3 * Mx * 4);  // row sums of squares of split-panel norms
    const size_t s_zero = stake(4096);
    const size_t ctr_n = (size_t)2 * (L + 1) * mk::NCTR;
    const size_t s_ctr = stake(ctr_n * 4);
    const size_t s_status = stake(64);
    const size_t s_dbgi = D.E ? stake((size_t)L * Mx * D.k * 4) : 0;
    const size_t s_dbgw = D.E ? stake((size_t)L * Mx * D.k * 4) : 0;
    const size_t s_dbgm = D.E ? stake((size_t)L * Mx * 4) : 0;
    const size_t s_utok = stake(Mx * 4), s_upos = stake((size_t)cfg->max_batch * 4);
    const int rope_dim = D.gqa ? D.hd : D.rd;
    const int npos = cfg->max_ctx + cfg->max_tokens_per_seq;
    const size_t s_rope = stake((size_t)npos * (rope_dim / 2) * 8);
    m->sbytes = scur;
    {
        cudaError_t e = cudaMalloc(&m->sblob, m->sbytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return bail(fail(MK_ERR_OOM, "scratch: cudaMalloc(%zu) failed", m->sbytes));
        }
    }
    CK(cudaMemsetAsync(m->sblob, 0, m->sbytes, s));
    for (size_t g : m->guards) CK(cudaMemsetAsync(m->sblob + g, 0xA5, 256, s));
    uint8_t* S = m->sblob;
    auto F = [&](size_t off) { return reinterpret_cast<float*>(S + off); };

    // ---- copy / pack every tensor ----
    const void* p;
    int r;
#define NEED(kind, layer, expert)                      \
    do {                                               \
        if ((r = need(kind, layer, expert, &p))) return bail(r); \
    } while (0)
#define PACK(dst, N, K, row0, src, rows)                                                              \
    do {                                                                                              \
        const int Kc_ = panel_width((K), (int)Mx);                                                      \
        if ((r = pack_rows(dst, N, K, Kc_, row0, src, rows, (size_t)(K) * 2, s))) return bail(r);     \
    } while (0)
    NEED(MK_W_EMBED, -1, 0);
    CK(cudaMemcpyAsync(W + off_embed, p, (size_t)D.V * d * 2, cudaMemcpyDefault, s));
    NEED(MK_W_LM_HEAD, -1, 0);
    PACK(W + off_lm, D.V, d, 0, p, D.V);
    NEED(MK_W_FINAL_NORM, -1, 0);
    CK(cudaMemcpyAsync(W + off_fn, p, (size_t)d * 2, cudaMemcpyDefault, s));
    uint16_t* tmp = nullptr;  // device staging for the MLA W_uk transpose
    if (!D.gqa) CK(cudaMalloc(&tmp, (size_t)D.Hq * (D.nope + D.vd) * D.kl * 2));
    uint16_t* etmp = nullptr;  // device staging of one expert (gate, up, down)
    CK(cudaMalloc(&etmp, (size_t)3 * std::max(D.E ? D.ffn : 0, D.sh ? D.sffn : 0) * d * 2));
    for (int l = 0; l < L; ++l) {
        const Off& o = lo[l];
        NEED(MK_W_ATTN_NORM, l, 0);
        CK(cudaMemcpyAsync(W + o.an, p, (size_t)d * 2, cudaMemcpyDefault, s));
        NEED(MK_W_FFN_NORM, l, 0);
        CK(cudaMemcpyAsync(W + o.fn, p, (size_t)d * 2, cudaMemcpyDefault, s));
        if (D.gqa) {
            NEED(MK_W_WQ, l, 0);
            PACK(W + o.a, D.a_rows, d, 0, p, D.Hq * D.hd);
            NEED(MK_W_WK, l, 0);
            PACK(W + o.a, D.a_rows, d, D.Hq * D.hd, p, D.Hkv * D.hd);
            NEED(MK_W_WV, l, 0);
            PACK(W + o.a, D.a_rows, d, (D.Hq + D.Hkv) * D.hd, p, D.Hkv * D.hd);
        } else {
            NEED(MK_W_WDQ, l, 0);
            PACK(W + o.a, D.a_rows, d, 0, p, D.ql);
            NEED(MK_W_WDKV, l, 0);
            PACK(W + o.a, D.a_rows, d, D.ql, p, D.kl + D.rd);
            NEED(MK_W_Q_NORM, l, 0);
            CK(cudaMemcpyAsync(W + o.qn, p, (size_t)D.ql * 2, cudaMemcpyDefault, s));
            NEED(MK_W_KV_NORM, l, 0);
            CK(cudaMemcpyAsync(W + o.kvn, p, (size_t)D.kl * 2, cudaMemcpyDefault, s));
            NEED(MK_W_WUQ, l, 0);
            PACK(W + o.uq, D.Hq * D.qh, D.ql, 0, p, D.Hq * D.qh);
            NEED(MK_W_WUKV, l, 0);
            CK(cudaMemcpyAsync(tmp, p, (size_t)D.Hq * (D.nope + D.vd) * D.kl * 2, cudaMemcpyDefault, s));
            transpose_heads<<<512, 256, 0, s>>>(tmp, W + o.ukT, D.Hq, D.nope, D.nope + D.vd, D.kl);
            CK(cudaGetLastError());
            CK(cudaMemcpy2DAsync(W + o.uk, (size_t)D.nope * D.kl * 2, tmp, (size_t)(D.nope + D.vd) * D.kl * 2,
                                 (size_t)D.nope * D.kl * 2, D.Hq, cudaMemcpyDeviceToDevice, s));
            pack_uv_quarters<<<512, 256, 0, s>>>(W + o.uvq, tmp, D.Hq, D.nope, D.vd, D.kl);
            CK(cudaGetLastError());
            // W_uv, head by head, into the K-panel layout of its GEMV (kv_lora
            // 512 splits into two panels of 256 on models loaded for many
            // tokens per step)
            for (int h = 0; h < D.Hq; ++h)
                if ((r = pack_rows(W + o.uv, D.Hq * D.vd, D.kl, panel_width(D.kl, (int)Mx), h * D.vd,
                                   tmp + (size_t)h * (D.nope + D.vd) * D.kl + (size_t)D.nope * D.kl, D.vd,
                                   (size_t)D.kl * 2, s)))
                    return bail(r);
        }
        NEED(MK_W_WO, l, 0);
        PACK(W + o.o, d, D.o_in, 0, p, d);
        // experts: gate, up and down go through a device copy, then into the
        // unit layout
        auto pack_expert = [&](int kgate, int kup, int kdown, int e, int Fi, uint16_t* gu, uint16_t* dn) -> int {
            const size_t n = (size_t)Fi * d;
            if (D.f8) {
                // codes of gate, up, down, then their scales, into the staging
                // buffer (6 n bytes hold them), then into the tiles
                uint8_t* b = reinterpret_cast<uint8_t*>(etmp);
                const int kinds[6] = {kgate, kup, kdown, kgate + 6, kup + 6, kdown + 6};
                const size_t offs[6] = {0, n, 2 * n, 3 * n, 3 * n + n / 32, 3 * n + 2 * n / 32};
                for (int i = 0; i < 6; ++i) {
                    if ((r = need(kinds[i], l, e, &p))) return r;
                    CK(cudaMemcpyAsync(b + offs[i], p, i < 3 ? n : n / 32, cudaMemcpyDefault, s));
                }
                const F8Geom g = f8_geometry(d, Fi);
                pack_gu_f8<<<1024, 256, 0, s>>>(reinterpret_cast<uint8_t*>(gu), b, b + n, b + 3 * n, b + 3 * n + n / 32,
                                               Fi, d, g.F, g.R, g.tb_gu);
                CK(cudaGetLastError());
                pack_dn_f8<<<1024, 256, 0, s>>>(reinterpret_cast<uint8_t*>(dn), b + 2 * n, b + 3 * n + 2 * n / 32, Fi, d,
                                               g.F, g.Rd, g.tb_dn);
                CK(cudaGetLastError());
                return MK_OK;
            }
            const int F = unit_width(Fi, d);
            int Kc, R, Rd;
            unit_geometry(d, F, Kc, R, Rd);
            if ((r = need(kgate, l, e, &p))) return r;
            CK(cudaMemcpyAsync(etmp, p, n * 2, cudaMemcpyDefault, s));
            if ((r = need(kup, l, e, &p))) return r;
            CK(cudaMemcpyAsync(etmp + n, p, n * 2, cudaMemcpyDefault, s));
            if ((r = need(kdown, l, e, &p))) return r;
            CK(cudaMemcpyAsync(etmp + 2 * n, p, n * 2, cudaMemcpyDefault, s));
            pack_gu_units<<<1024, 256, 0, s>>>(gu, etmp, etmp + n, Fi, d, F, Kc);
            CK(cudaGetLastError());
            pack_dn_units<<<1024, 256, 0, s>>>(dn, etmp + 2 * n, Fi, d, F);
            CK(cudaGetLastError());
            return MK_OK;
        };
        if (D.E) {
            NEED(MK_W_ROUTER, l, 0);
            PACK(W + o.router, D.E, d, 0, p, D.E);
            const size_t gu_es = D.f8 ? f8_geometry(d, D.ffn).gu_bytes / 2 : (size_t)2 * D.ffn * d;
            const size_t dn_es = D.f8 ? f8_geometry(d, D.ffn).dn_bytes / 2 : (size_t)d * D.ffn;
            for (int e = 0; e < D.E; ++e)
                if ((r = pack_expert(MK_W_GATE, MK_W_UP, MK_W_DOWN, e, D.ffn, W + o.gu + (size_t)e * gu_es,
                                     W + o.down + (size_t)e * dn_es)))
                    return bail(r);
        }
        if (D.sh && (r = pack_expert(MK_W_SH_GATE, MK_W_SH_UP, MK_W_SH_DOWN, 0, D.sffn, W + o.shgu, W + o.shdown)))
            return bail(r);
    }
#undef NEED
#undef PACK

    // ---- RoPE table (fp64 frequency, angle, cos, sin; stored fp32) ----
    {
        const int half = rope_dim / 2;
        std::vector<float2> rt((size_t)npos * half);
        for (int pos = 0; pos < npos; ++pos)
            for (int i = 0; i < half; ++i) {
                const double inv = std::pow((double)cfg->rope_theta, -2.0 * (double)i / (double)rope_dim);
                const double ang = (double)pos * inv;
                rt[(size_t)pos * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
        CK(cudaMemcpyAsync(S + s_rope, rt.data(), rt.size() * sizeof(float2), cudaMemcpyHostToDevice, s));
        CK(cudaStreamSynchronize(s));  // rt and tmp go out of scope
    }
    if (tmp) CK(cudaFree(tmp));
    CK(cudaFree(etmp));

    // ---- stage descriptors ----
    m->layers.resize(L);
    const int Mxi = (int)Mx;
    for (int l = 0; l < L; ++l) {
        const Off& o = lo[l];
        mk::Layer& Ld = m->layers[l];
        std::memset(&Ld, 0, sizeof Ld);
        float* x = F(s_x) + (size_t)l * Mx * d;
        float* xn = F(s_x) + (size_t)(l + 1) * Mx * d;
        float* a = F(s_a) + (size_t)l * Mx * D.a_rows;
        float* ob = F(s_o) + (size_t)l * Mx * D.o_in;
        Ld.x = x;
        Ld.xn = xn;
        Ld.a = a;
        Ld.a_stride = D.a_rows;
        Ld.o = ob;
        make_gemv(Ld.g[mk::G_A], W + o.a, D.a_rows, d, mk::IN_RMS, x, d, W + o.an, mk::OUT_STORE, a, D.a_rows, Mxi);
        if (!D.gqa) {
            float* q = F(s_q) + (size_t)l * Mx * D.Hq * D.qh;
            float* qlat = F(s_qlat) + (size_t)l * Mx * D.Hq * D.kl;
            float* olat = F(s_olat) + (size_t)l * Mx * D.Hq * D.kl;
            Ld.q = q;
            Ld.qlat = qlat;
            Ld.olat = olat;
            Ld.kv_norm = W + o.kvn;
            Ld.uk = W + o.uk;
            Ld.uvq = W + o.uvq;
            make_gemv(Ld.g[mk::G_QB], W + o.uq, D.Hq * D.qh, D.ql, mk::IN_RMS, a, D.a_rows, W + o.qn, mk::OUT_STORE,
                      q, D.Hq * D.qh, Mxi);
            make_gemv(Ld.g[mk::G_QLAT], W + o.ukT, D.Hq * D.kl, D.nope, mk::IN_COPY, q, D.Hq * D.qh, nullptr,
                      mk::OUT_STORE, qlat, D.Hq * D.kl, Mxi);
            Ld.g[mk::G_QLAT].grp_rows = D.kl;
            Ld.g[mk::G_QLAT].grp_stride = D.qh;
            make_gemv(Ld.g[mk::G_UV], W + o.uv, D.Hq * D.vd, D.kl, mk::IN_COPY, olat, D.Hq * D.kl, nullptr,
                      mk::OUT_STORE, ob, D.Hq * D.vd, Mxi);
            Ld.g[mk::G_UV].grp_rows = D.vd;
            Ld.g[mk::G_UV].grp_stride = D.kl;
        }
        make_gemv(Ld.g[mk::G_O], W + o.o, d, D.o_in, mk::IN_COPY, ob, D.o_in, nullptr, mk::OUT_RESID, x, d, Mxi, xn);
        Ld.ffn.gain = W + o.fn;
        auto set_kind = [&](mk::FfnKind& K, int Fi, const uint16_t* gu, const uint16_t* dn) {
            if (D.f8) {
                const F8Geom g = f8_geometry(d, Fi);
                K.qgu = reinterpret_cast<const uint8_t*>(gu);
                K.qdn = reinterpret_cast<const uint8_t*>(dn);
                K.qgu_es = (long long)g.gu_bytes;
                K.qdn_es = (long long)g.dn_bytes;
                K.qtb_gu = g.tb_gu;
                K.qtb_dn = g.tb_dn;
                K.Fi = Fi;
                K.F = g.F;
                K.nu = Fi / g.F;
                K.R = g.R;
                K.Rd = g.Rd;
                Ld.ffn.Kc = d;
                Ld.ffn.n_kc = 1;
                return;
            }
            K.gu = gu;
            K.dn = dn;
            K.gu_es = (long long)2 * Fi * d;
            K.dn_es = (long long)d * Fi;
            K.Fi = Fi;
            K.F = unit_width(Fi, d);
            K.nu = Fi / K.F;
            int Kc, R, Rd;
            unit_geometry(d, K.F, Kc, R, Rd);
            K.R = R;
            K.Rd = Rd;
            Ld.ffn.Kc = Kc;
            Ld.ffn.n_kc = d / Kc;
        };
        if (D.E) {
            float* rlog = F(s_rlog) + (size_t)l * Mx * mk::router_row(D.E);
            Ld.rlog = rlog;
            make_gemv(Ld.g[mk::G_ROUTER], W + o.router, D.E, d, mk::IN_RMS, x, d, W + o.fn, mk::OUT_STORE, rlog,
                      mk::router_row(D.E), Mxi);
            set_kind(Ld.ffn.k[0], D.ffn, W + o.gu, W + o.down);
        }
        if (D.sh) set_kind(Ld.ffn.k[1], D.sffn, W + o.shgu, W + o.shdown);
    }
    (void)Mxi;
    CK(cudaMalloc(&m->d_layers, sizeof(mk::Layer) * L));
    CK(cudaMemcpyAsync(m->d_layers, m->layers.data(), sizeof(mk::Layer) * L, cudaMemcpyHostToDevice, s));

    mk::Params& P = m->base;
    std::memset(&P, 0, sizeof P);
    P.L = L; P.d = d; P.V = D.V; P.attn = D.gqa ? 0 : 1; P.Hq = D.Hq; P.Hkv = D.Hkv; P.hd = D.hd;
    P.ql = D.ql; P.kl = D.kl; P.nope = D.nope; P.rd = D.rd; P.vd = D.vd; P.E = D.E; P.topk = D.k;
    P.has_sh = D.sh; P.ffn = D.ffn; P.sffn = D.sffn;
    P.f8 = D.f8;
    P.eps = cfg->rms_eps;
    P.attn_scale = D.gqa ? (float)(1.0 / std::sqrt((double)D.hd)) : (float)(1.0 / std::sqrt((double)D.qh));
    P.G = m->G;
    P.layers = m->d_layers;
    P.embed = W + off_embed;
    make_gemv(P.lm, W + off_lm, D.V, d, mk::IN_RMS, F(s_x) + (size_t)L * Mx * d, d, W + off_fn, mk::OUT_STORE,
              nullptr, D.V, (int)Mx);
    P.rope = reinterpret_cast<const float2*>(S + s_rope);
    P.rope_half = rope_dim / 2;
    P.rope_npos = npos;
    P.zeros = reinterpret_cast<const uint16_t*>(S + s_zero);
    P.newlat = reinterpret_cast<uint16_t*>(S + s_newlat);
    P.part = F(s_part);
    P.part_ml = F(s_part_ml);
    P.s_max = m->G;
    if (tracing) {
        P.trace = reinterpret_cast<mk::TraceRec*>(S + s_trace);
        P.trace_n = reinterpret_cast<unsigned*>(S + s_trace_n);
        P.trace_cap = trace_cap;
        P.trace_items = atoi(getenv("MK_TRACE")) > 2 ? 2 : atoi(getenv("MK_TRACE")) > 1 ? 1 : 0;
    }
    P.amax = reinterpret_cast<int*>(S + s_amax);
    P.ubuf = F(s_ubuf);
    P.ubuf_stride = (long long)ubuf_stride;
    // buffers accumulated with atomics (K split into panels) are cleared at the start of each step
    P.carry = m->layers[0].g[mk::G_O].n_kc > 1;
    int nz = 0;
    if (m->layers[0].g[mk::G_A].n_kc > 1) {
        P.zptr[nz] = F(s_a);
        P.zn[nz++] = (long long)L * Mx * D.a_rows;
    }
    if (P.carry) {
        P.zptr[nz] = F(s_x) + (size_t)Mx * d;
        P.zn[nz++] = (long long)L * Mx * d;
    }
    // outputs of the other projections that split K into panels
    if (!D.gqa && m->layers[0].g[mk::G_QB].n_kc > 1) {
        P.zptr[nz] = F(s_q);
        P.zn[nz++] = (long long)L * Mx * D.Hq * D.qh;
    }
    if (!D.gqa && (m->layers[0].g[mk::G_QLAT].n_kc > 1 || m->layers[0].g[mk::G_UV].n_kc > 1)) {
        if (m->layers[0].g[mk::G_QLAT].n_kc > 1) {
            P.zptr[nz] = F(s_qlat);
            P.zn[nz++] = (long long)L * Mx * D.Hq * D.kl;
        }
        if (m->layers[0].g[mk::G_UV].n_kc > 1) {
            P.zptr[nz] = F(s_o);
            P.zn[nz++] = (long long)L * Mx * D.o_in;
        }
    }
    if (D.E && m->layers[0].g[mk::G_ROUTER].n_kc > 1) {
        P.zptr[nz] = F(s_rlog);
        P.zn[nz++] = (long long)L * Mx * mk::router_row(D.E);
    }
    P.rss = F(s_rss);
    P.rss_mx = (int)Mx;
    P.zptr[nz] = P.rss;
    P.zn[nz++] = (long long)(L + 1) * 3 * Mx;
    // the router folded into the output projection: possible when that
    // projection has one K panel (its rows are final in the CTA that computes
    // them) and a CTA's rows of every token (twice) and its logit sums fit
    // the staging area
    {
        const mk::Gemv& go = m->layers[0].g[mk::G_O];
        const int items = gemv_items_host(go), per_cta = (items + m->G - 1) / m->G;
        const char* ev = getenv("MK_ROUTER_STAGE");
        m->rfuse_ok = D.E > 0 && go.n_kc == 1 && go.out_kind == mk::OUT_RESID && go.R % 8 == 0 && go.N % 8 == 0 &&
                      m->layers[0].g[mk::G_ROUTER].Kc % 8 == 0 &&
                      (2 * per_cta * go.R + mk::router_row(D.E)) * Mx <= mk::STAGE_FLOATS && !(ev && atoi(ev) > 0);
        P.rfuse = 0;  // per step
        P.racc = D.E ? F(s_racc) : nullptr;
    }
    // the absorbed query folded into QB: QB tiles of 16 rows that never
    // straddle a head's nope and rope rows, one K panel, and every CTA with
    // an item of A (those CTAs clear q_lat before QB adds into it)
    if (!D.gqa) {
        const mk::Gemv& gq = m->layers[0].g[mk::G_QB];
        const char* ev = getenv("MK_QLAT_STAGE");
        m->qfuse_ok = gq.n_kc == 1 && gq.R == 16 && D.nope % gq.R == 0 && D.qh % gq.R == 0 &&
                      gemv_items_host(m->layers[0].g[mk::G_A]) >= m->G && !(ev && atoi(ev) > 0);
        // the value up-projection folded into the combine: a slab of 128
        // latent dimensions x vd fits a ring slot, two values per thread
        const char* eu = getenv("MK_UV_STAGE");
        m->ufuse_ok = D.vd % 2 == 0 && D.vd <= 128 && 128 * D.vd * 2 <= mk::SLOT_BYTES &&
                      gemv_items_host(m->layers[0].g[mk::G_A]) >= m->G && !(eu && atoi(eu) > 0);
    } else {
        m->qfuse_ok = m->ufuse_ok = false;
    }
    // logits (split-K head) and the router accumulators are added per step
    static_assert(sizeof(P.zptr) / sizeof(P.zptr[0]) >= 9, "zero list: 7 buffers here + 2 per step");
    P.nz = nz;
    m->ctr = reinterpret_cast<unsigned*>(S + s_ctr);
    m->ctr_n = ctr_n;
    m->status = reinterpret_cast<unsigned*>(S + s_status);
    P.ctr = m->ctr;
    P.status = m->status;
    P.timeout_ns = wait_ns();
    P.debug = getenv("MK_DEBUG") && atoi(getenv("MK_DEBUG")) > 0;
    if (D.E) {
        m->dbg_idx = reinterpret_cast<int*>(S + s_dbgi);
        m->dbg_w = reinterpret_cast<float*>(S + s_dbgw);
        m->dbg_margin = reinterpret_cast<float*>(S + s_dbgm);
    }
    m->u_tok = reinterpret_cast<int*>(S + s_utok);
    m->u_pos = reinterpret_cast<int*>(S + s_upos);
    CK(cudaStreamSynchronize(s));
    *out = m;
    return MK_OK;
}

int mk_model_info(const mk_model* m, mk_info* out) {
    if (!m || m->magic != MODEL_MAGIC || !out) return fail(MK_ERR_INVALID_ARG, "bad model or out");
    out->weight_bytes = (int64_t)m->wbytes;
    out->scratch_bytes = (int64_t)m->sbytes;
    out->grid_ctas = m->G;
    out->threads_per_cta = mk::NTHREADS;
    out->smem_bytes = mk::SMEM_TOTAL;
    out->ring_slots = mk::NSLOT;
    out->slot_bytes = mk::SLOT_BYTES;
    out->sm_count = m->sms;
    return MK_OK;
}

// the two tensor maps of an MLA cache's pool (pages of 64 rows x 512 latent
// values, then 64 rows x 64 rope values, bf16): 4-D views [L][pages][64][512]
// and [L][pages][64][64] whose boxes of 32 rows x 64 values are the attention
// chunks' pieces, copied in the 128-byte swizzled order
static int mla_tensor_maps(mk_kv* kv, int L) {
    using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static Encode encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return fail(MK_ERR_CUDA, "kv: the driver has no cuTensorMapEncodeTiled");
        }
        encode = reinterpret_cast<Encode>(fn);
    }
    const cuuint64_t pages = kv->layer_elems / kv->page_elems;
    alignas(64) CUtensorMap maps[2];
    const cuuint32_t box[4] = {64, (cuuint32_t)mk::MLA_CH, 1, 1}, one[4] = {1, 1, 1, 1};
    const cuuint64_t dl[4] = {(cuuint64_t)mk::MLA_KL, (cuuint64_t)mk::PAGE, pages, (cuuint64_t)L};
    const cuuint64_t dr[4] = {(cuuint64_t)mk::MLA_RD, (cuuint64_t)mk::PAGE, pages, (cuuint64_t)L};
    const cuuint64_t sl[3] = {(cuuint64_t)mk::MLA_KL * 2, kv->page_elems * 2, kv->layer_elems * 2};
    const cuuint64_t sr[3] = {(cuuint64_t)mk::MLA_RD * 2, kv->page_elems * 2, kv->layer_elems * 2};
    CUresult r = encode(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, kv->pool, dl, sl, box, one,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
        r = encode(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, kv->pool + (size_t)mk::PAGE * mk::MLA_KL, dr, sr,
                   box, one, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "kv: cuTensorMapEncodeTiled failed (%d)", (int)r);
    static_assert(sizeof(CUtensorMap) == 128, "tensor maps are 128 bytes");
    if (cudaMalloc(&kv->tmaps, sizeof maps) != cudaSuccess) {
        cudaGetLastError();
        return fail(MK_ERR_OOM, "kv: tensor maps");
    }
    CK(cudaMemcpy(kv->tmaps, maps, sizeof maps, cudaMemcpyHostToDevice));
    return MK_OK;
}

int mk_alloc_kv(const mk_model* m, int32_t batch, int32_t max_ctx, mk_kv** out) {
    if (!out) return fail(MK_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!m || m->magic != MODEL_MAGIC) return fail(MK_ERR_INVALID_ARG, "bad model handle");
    if (batch < 1 || batch > m->cfg.max_batch) return fail(MK_ERR_INVALID_ARG, "batch out of range");
    if (max_ctx < 1 || max_ctx > m->cfg.max_ctx + m->cfg.max_tokens_per_seq)
        return fail(MK_ERR_INVALID_ARG, "max_ctx out of range");
    if (fault("oom")) return fail(MK_ERR_OOM, "allocation refused (injected by MK_FAULT=oom)");
    const Dims D = dims_of(m->cfg);
    mk_kv* kv = new mk_kv();
    kv->magic = KV_MAGIC;
    kv->m = const_cast<mk_model*>(m);
    kv->batch = batch;
    kv->max_ctx = max_ctx;
    kv->pps = (max_ctx + mk::PAGE - 1) / mk::PAGE;
    kv->page_elems = D.gqa ? (size_t)D.Hkv * 2 * mk::PAGE * D.hd : (size_t)mk::PAGE * mk::MLA_D;
    const size_t pages = (size_t)batch * kv->pps;
    kv->layer_elems = pages * kv->page_elems;
    const size_t bytes = kv->layer_elems * D.L * 2;
    cudaError_t e = cudaMalloc(&kv->pool, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete kv;
        return fail(MK_ERR_OOM, "kv: cudaMalloc(%zu) failed", bytes);
    }
    e = cudaMalloc(&kv->btab, pages * sizeof(int));
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFree(kv->pool);
        delete kv;
        return fail(MK_ERR_OOM, "kv block table");
    }
    CK(cudaMemset(kv->pool, 0, bytes));
    if (!D.gqa) {
        if (const int rc = mla_tensor_maps(kv, D.L)) {
            cudaFree(kv->pool);
            cudaFree(kv->btab);
            if (kv->tmaps) cudaFree(kv->tmaps);
            delete kv;
            return rc;
        }
    }
    kv->h_btab.resize(pages);
    for (int b = 0; b < batch; ++b)
        for (int j = 0; j < kv->pps; ++j) kv->h_btab[(size_t)b * kv->pps + j] = j * batch + b;
    CK(cudaMemcpy(kv->btab, kv->h_btab.data(), pages * sizeof(int), cudaMemcpyHostToDevice));
    kv->m->live_kv++;
    *out = kv;
    return MK_OK;
}

int32_t mk_kv_pages_per_seq(const mk_kv* kv) { return (kv && kv->magic == KV_MAGIC) ? kv->pps : -1; }

int mk_kv_set_block_table(mk_kv* kv, const int32_t* table) {
    if (!kv || kv->magic != KV_MAGIC || !table) return fail(MK_ERR_INVALID_ARG, "bad kv or table");
    const size_t pages = (size_t)kv->batch * kv->pps;
    std::vector<char> seen(pages, 0);
    for (size_t i = 0; i < pages; ++i) {
        if (table[i] < 0 || (size_t)table[i] >= pages || seen[table[i]])
            return fail(MK_ERR_INVALID_ARG, "block table entry %zu invalid or repeated", i);
        seen[table[i]] = 1;
    }
    std::memcpy(kv->h_btab.data(), table, pages * sizeof(int));
    CK(cudaMemcpy(kv->btab, table, pages * sizeof(int), cudaMemcpyHostToDevice));
    return MK_OK;
}

static int kv_copy(const mk_kv* kv, int32_t layer, int32_t seq, int32_t pos0, int32_t n, void* rows, void* stream,
                   int to_cache) {
    if (!kv || kv->magic != KV_MAGIC || !rows) return fail(MK_ERR_INVALID_ARG, "bad kv or rows");
    const Dims D = dims_of(kv->m->cfg);
    if (layer < 0 || layer >= D.L || seq < 0 || seq >= kv->batch || pos0 < 0 || n < 0 || pos0 + n > kv->max_ctx)
        return fail(MK_ERR_INVALID_ARG, "kv range out of bounds");
    if (n == 0) return MK_OK;
    const int row = D.gqa ? 2 * D.Hkv * D.hd : mk::MLA_D;
    const size_t bytes = (size_t)n * row * 2;
    cudaStream_t s = (cudaStream_t)stream;
    uint16_t* dev = static_cast<uint16_t*>(rows);
    const bool host = !is_device_ptr(rows);
    if (host) {
        CK(cudaMalloc(&dev, bytes));
        if (to_cache) CK(cudaMemcpyAsync(dev, rows, bytes, cudaMemcpyHostToDevice, s));
    }
    kv_scatter<<<256, 256, 0, s>>>(kv->pool + (size_t)layer * kv->layer_elems, kv->btab, kv->pps, kv->page_elems,
                                   D.gqa, D.Hkv, D.hd, D.kl, D.rd, seq, pos0, n, row, dev, to_cache);
    CK(cudaGetLastError());
    if (host) {
        if (!to_cache) CK(cudaMemcpyAsync(rows, dev, bytes, cudaMemcpyDeviceToHost, s));
        CK(cudaStreamSynchronize(s));
        CK(cudaFree(dev));
    }
    return MK_OK;
}

int mk_kv_write(mk_kv* kv, int32_t layer, int32_t seq, int32_t pos0, int32_t n, const void* rows, void* stream) {
    return kv_copy(kv, layer, seq, pos0, n, const_cast<void*>(rows), stream, 1);
}

int mk_kv_read(const mk_kv* kv, int32_t layer, int32_t seq, int32_t pos0, int32_t n, void* rows, void* stream) {
    return kv_copy(kv, layer, seq, pos0, n, rows, stream, 0);
}

// FFN CTA groups: gr CTAs run the router (one per router tile) and then,
// with the CTAs from gs on, the routed experts' units; CTAs [0, gs) run the
// shared expert's units; gs follows the two kinds' expected work, the routed
// unit count taken as the expected number of distinct experts of M tokens
// picking top_k of E uniformly at random
static void ffn_split(const mk_model* m, int M, bool rfuse, int& gs, int& gr) {
    const Dims D = dims_of(m->cfg);
    const mk::Layer& L0 = m->layers[0];
    gr = D.E && !rfuse ? std::min(gemv_items_host(L0.g[mk::G_ROUTER]), m->G / 4) : 0;
    if (!D.E) {
        gs = m->G;
        return;
    }
    if (!D.sh) {
        gs = 0;
        return;
    }
    // a unit's time grows with its token count (the weights stream once, the
    // arithmetic is per token): about 1 + 0.8 (t - 1) tile times for t tokens.
    // A routed expert's units take only its own tokens (M k / distinct on
    // average) when its input is one K panel, and the shared expert's run
    // once per token group (mk::shared_group).
    const auto cost = [](double t) { return 1.0 + 0.8 * (t - 1.0); };
    const double uniq = D.E * (1.0 - std::pow(1.0 - (double)D.k / D.E, (double)M));
    const int tgs = mk::shared_group(M, L0.ffn.n_kc, L0.ffn.Kc);
    const int ntg = (M + tgs - 1) / tgs;
    const double us = L0.ffn.k[1].nu * ntg * cost(M / (double)ntg);
    const double ur = uniq * L0.ffn.k[0].nu * cost(M > 1 && L0.ffn.n_kc == 1 ? M * D.k / uniq : M);
    const int avail = m->G;  // the router CTAs also take routed units after their router tile
    gs = (int)std::lround(avail * us / (us + ur));
    if (gs < 1) gs = 1;
    if (gs > avail - 1) gs = avail - 1;
}

// per step: the router folded into the output projection for two or more
// tokens (one token routes sooner with its own router stage, which overlaps
// the shared expert), and the FFN CTA groups
static void step_router(const mk_model* m, mk::Params& P) {
    P.rfuse = m->rfuse_ok && P.M >= 2;
    if (P.rfuse) {
        P.zptr[P.nz] = P.racc;
        P.zn[P.nz++] = (long long)P.L * mk::ROUTER_COPIES * P.M * mk::router_row(P.E);
    }
    ffn_split(m, P.M, P.rfuse, P.gs, P.gr);
}

// the step's parameters (everything but the launch-specific fields), after
// the argument checks every decode entry point shares
static int step_params(mk_model* m, mk_kv* kv, const int32_t* tokens, const int32_t* positions, int32_t batch,
                       int32_t T, float* logits, int32_t* accept, mk::Params& P) {
    if (!m || m->magic != MODEL_MAGIC) return fail(MK_ERR_INVALID_ARG, "bad model handle");
    if (!kv || kv->magic != KV_MAGIC) return fail(MK_ERR_INVALID_ARG, "bad kv handle");
    if (kv->m != m) return fail(MK_ERR_STATE, "kv cache belongs to another model");
    if (!tokens || !positions || !logits) return fail(MK_ERR_INVALID_ARG, "NULL tokens/positions/logits");
    if (batch < 1 || batch > kv->batch) return fail(MK_ERR_INVALID_ARG, "batch %d out of range", batch);
    if (T < 1 || T > m->cfg.max_tokens_per_seq) return fail(MK_ERR_INVALID_ARG, "T %d out of range", T);
    if (accept && T < 2) return fail(MK_ERR_INVALID_ARG, "accept needs T > 1");
    if (fault("bad_arg")) return fail(MK_ERR_INVALID_ARG, "arguments rejected (injected by MK_FAULT=bad_arg)");
    P = m->base;
    P.page_elems = (long long)kv->page_elems;
    P.pps = kv->pps;
    P.btab = kv->btab;
    P.kv_cap = kv->max_ctx;
    P.kv_batch = kv->batch;
    P.kv_pool = kv->pool;
    P.kv_layer_elems = (long long)kv->layer_elems;
    P.kv_tmaps = kv->tmaps;
    P.tokens = tokens;
    P.pos = positions;
    P.B = batch;
    P.T = T;
    P.M = batch * T;
    step_router(m, P);
    P.logits = logits;
    P.accept = accept;
    P.lm.dst = logits;
    if (P.lm.n_kc > 1) {
        P.zptr[P.nz] = logits;
        P.zn[P.nz++] = (long long)P.M * P.V;
    }
    P.dbg_idx = m->dbg_idx;
    P.dbg_w = m->dbg_w;
    P.dbg_margin = m->dbg_margin;
    // every token's c_q staged at once, one tile's outputs per thread
    P.qfuse = m->qfuse_ok && mk::stage_fits(P.M, P.ql) && P.M * m->layers[0].g[mk::G_QB].R <= mk::NCT;
    // the combine's items are per token: each reads its 32 KB slab of W_uv,
    // so for many tokens the separate stage (W_uv read once) is cheaper
    P.ufuse = m->ufuse_ok && P.M <= 16;
    return MK_OK;
}

int mk_decode_step(mk_model* m, mk_kv* kv, const int32_t* tokens, const int32_t* positions, int32_t batch,
                   int32_t T, float* logits, int32_t* accept, void* stream) {
    mk::Params P;
    if (const int rc = step_params(m, kv, tokens, positions, batch, T, logits, accept, P)) return rc;
    P.stall = getenv("MK_TEST_STALL") != nullptr;
    P.skip_sig = fault("skip_signal") ? 1 + mk::C_A : 0;
    P.parity = (int)(m->steps & 1);
    cudaStream_t s = (cudaStream_t)stream;
    void* args[] = {&P};
    CK(cudaLaunchCooperativeKernel((const void*)mk::megakernel, dim3(m->G), dim3(mk::NTHREADS), args,
                                   mk::SMEM_TOTAL, s));
    m->steps++;
    m->last_M = P.M;
    m->last_noalloc = false;
    m->last_amax = accept ? P.amax : nullptr;
    return MK_OK;
}

// the launches of one step run as one launch per stage: (staged, first, end)
// program positions; stages the model or this step does not have are left
// out, and stages that read only the same earlier results share a launch
static std::vector<std::tuple<int, int, int>> stage_windows(const mk_model* m, const mk::Params& P) {
    using namespace mk;
    std::vector<std::tuple<int, int, int>> w;
    w.emplace_back(2, 0, 0);  // set-up: embedding, accumulators zeroed
    const int L = P.L;
    const bool mla = P.attn == 1;
    auto win = [&](int l, int a, int b) { w.emplace_back(1, prog_index(P, l, a), prog_index(P, l, b)); };
    for (int l = 0; l < L; ++l) {
        win(l, S_A, S_A + 1);
        if (mla) {
            win(l, S_QB, S_APP + 1);  // the latent append reads only A's output
            if (!P.qfuse) win(l, S_QLAT, S_QLAT + 1);
        }
        win(l, S_ATTN, S_ATTN + 1);
        win(l, S_COMB, S_COMB + 1);
        if (mla && !P.ufuse) win(l, S_UV, S_UV + 1);
        win(l, S_O, S_O + 1);
        const bool router = P.E > 0 && !P.rfuse;
        if (router || P.carry) win(l, S_ROUTER, S_CARRY + 1);  // both read only O's output
        win(l, S_FFN, S_FFN + 1);
    }
    w.emplace_back(1, prog_index(P, L, S_LM), prog_index(P, L, S_LM + 1));
    if (P.accept) {  // acceptance reads every row's argmax: a launch of its own
        w.emplace_back(1, prog_index(P, L, S_AMAX), prog_index(P, L, S_AMAX + 1));
        w.emplace_back(1, prog_index(P, L, S_ACCEPT), prog_index(P, L, S_ACCEPT + 1));
    }
    (void)m;
    return w;
}

int mk_decode_step_unfused(mk_model* m, mk_kv* kv, const int32_t* tokens, const int32_t* positions, int32_t batch,
                           int32_t T, float* logits, int32_t* accept, void* stream) {
    mk::Params P;
    if (const int rc = step_params(m, kv, tokens, positions, batch, T, logits, accept, P)) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    // the graph reads the token ids and positions from the model's own
    // buffers, so one graph serves every call of the same shape
    CK(cudaMemcpyAsync(m->u_tok, tokens, (size_t)P.M * 4, cudaMemcpyDefault, s));
    CK(cudaMemcpyAsync(m->u_pos, positions, (size_t)batch * 4, cudaMemcpyDefault, s));
    P.tokens = m->u_tok;
    P.pos = m->u_pos;
    P.trace = nullptr;
    P.trace_n = nullptr;
    P.trace_items = 0;
    P.parity = 0;
    const auto key = std::make_tuple((const void*)kv, batch, T, (const void*)logits, (const void*)accept);
    auto it = m->graphs.find(key);
    if (it == m->graphs.end()) {
        cudaStream_t cs;
        CK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
        cudaGraph_t g = nullptr;
        CK(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal));
        int rc = MK_OK;
        for (const auto& wdw : stage_windows(m, P)) {
            mk::Params Q = P;
            Q.staged = std::get<0>(wdw);
            Q.st_lo = std::get<1>(wdw);
            Q.st_hi = std::get<2>(wdw);
            cudaLaunchConfig_t lc = {};
            lc.gridDim = dim3(m->G);
            lc.blockDim = dim3(mk::NTHREADS);
            lc.dynamicSmemBytes = mk::SMEM_TOTAL;
            lc.stream = cs;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            at[0].val.programmaticStreamSerializationAllowed = 1;
            lc.attrs = at;
            lc.numAttrs = 1;
            const cudaError_t e = cudaLaunchKernelEx(&lc, mk::megakernel, Q);
            if (e != cudaSuccess) {
                rc = fail(MK_ERR_CUDA, "staged launch: %s", cudaGetErrorString(e));
                break;
            }
        }
        const cudaError_t ee = cudaStreamEndCapture(cs, &g);
        cudaStreamDestroy(cs);
        if (rc) {
            if (g) cudaGraphDestroy(g);
            return rc;
        }
        if (ee != cudaSuccess) return fail(MK_ERR_CUDA, "stage graph capture: %s", cudaGetErrorString(ee));
        cudaGraphExec_t ex = nullptr;
        const cudaError_t ie = cudaGraphInstantiate(&ex, g, 0);
        cudaGraphDestroy(g);
        if (ie != cudaSuccess) return fail(MK_ERR_CUDA, "stage graph instantiate: %s", cudaGetErrorString(ie));
        it = m->graphs.emplace(key, ex).first;
    }
    CK(cudaGraphLaunch(it->second, s));
    m->last_M = P.M;
    m->last_noalloc = false;
    m->last_amax = accept ? P.amax : nullptr;
    return MK_OK;
}

// MK_DEBUG: every scratch guard still holds its pattern (one overwritten is
// restored and reported). MK_FAULT=corrupt_guard overwrites one first (host
// injection, to test the caller's handling of the report).
static int check_guards(mk_model* m) {
    if (m->guards.empty()) return MK_OK;
    if (fault("corrupt_guard")) CK(cudaMemset(m->sblob + m->guards[m->guards.size() / 2], 0, 4));
    unsigned char b[256];
    for (size_t i = 0; i < m->guards.size(); ++i) {
        CK(cudaMemcpy(b, m->sblob + m->guards[i], sizeof b, cudaMemcpyDeviceToHost));
        for (unsigned char v : b)
            if (v != 0xA5) {
                CK(cudaMemset(m->sblob + m->guards[i], 0xA5, 256));
                return fail(MK_ERR_STATE, "debug check failed (MK_DEBUG; scratch guard %zu of %zu overwritten)", i,
                            m->guards.size());
            }
    }
    return MK_OK;
}

int mk_step_status(mk_model* m, void* stream) {
    if (!m || m->magic != MODEL_MAGIC) return fail(MK_ERR_INVALID_ARG, "bad model handle");
    cudaStream_t s = (cudaStream_t)stream;
    CK(cudaStreamSynchronize(s));
    unsigned st[4];
    CK(cudaMemcpy(st, m->status, sizeof st, cudaMemcpyDeviceToHost));
    if (st[0] == 0 && st[1] == 0) return check_guards(m);
    // reset device state so the next step starts clean
    CK(cudaMemset(m->ctr, 0, m->ctr_n * sizeof(unsigned)));
    CK(cudaMemset(m->status, 0, 64));
    CK(cudaDeviceSynchronize());
    m->steps = 0;
    if (st[0] == mk::ST_TIMEOUT)
        return fail(MK_ERR_TIMEOUT, "device wait timed out (where=0x%x, cta=%u)", st[2], st[3]);
    if (st[0] == mk::ST_INVALID)
        return fail(MK_ERR_INVALID_ARG, "token id or position out of range for this step");
    if (st[0] == mk::ST_DEBUG)
        return fail(MK_ERR_STATE, "debug check failed (MK_DEBUG; where=0x%x, cta=%u)", st[2], st[3]);
    return fail(MK_ERR_CUDA, "device status %u", st[0]);
}

int mk_trace_read(mk_model* m, void* recs_out, int64_t bytes, int32_t* counts_out, void* stream) {
    if (!m || m->magic != MODEL_MAGIC || !counts_out) return fail(MK_ERR_INVALID_ARG, "bad arguments");
    if (!m->base.trace) return fail(MK_ERR_STATE, "tracing is off (set MK_TRACE=1 before mk_load_weights)");
    const size_t need = (size_t)m->G * m->base.trace_cap * sizeof(mk::TraceRec);
    if (!recs_out || bytes < (int64_t)need) return fail(MK_ERR_INVALID_ARG, "trace buffer needs %zu bytes", need);
    CK(cudaStreamSynchronize((cudaStream_t)stream));
    CK(cudaMemcpy(recs_out, m->base.trace, need, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(counts_out, m->base.trace_n, (size_t)m->G * 4, cudaMemcpyDeviceToHost));
    return MK_OK;
}

int mk_debug_routing(mk_model* m, int32_t* idx_out, float* w_out, float* margin_out, void* stream) {
    if (!m || m->magic != MODEL_MAGIC || !idx_out || !w_out) return fail(MK_ERR_INVALID_ARG, "bad arguments");
    if (!m->dbg_idx) return fail(MK_ERR_STATE, "model has no router");
    if (m->last_M == 0) return fail(MK_ERR_STATE, "no step has run on this model");
    if (m->last_noalloc)
        return fail(MK_ERR_STATE, "the last step ran through mk_decode_step_noalloc, which keeps no routing record");
    CK(cudaStreamSynchronize((cudaStream_t)stream));
    const size_t n = (size_t)m->cfg.n_layers * m->last_M * m->cfg.top_k;
    // the device buffers are laid out [L][M][k] and [L][M] for the last step's M
    CK(cudaMemcpy(idx_out, m->dbg_idx, n * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(w_out, m->dbg_w, n * 4, cudaMemcpyDeviceToHost));
    if (margin_out)
        CK(cudaMemcpy(margin_out, m->dbg_margin, (size_t)m->cfg.n_layers * m->last_M * 4, cudaMemcpyDeviceToHost));
    return MK_OK;
}

int mk_debug_scratch_read(mk_model* m, int64_t offset, int64_t bytes, void* host_out, void* stream) {
    if (!m || m->magic != MODEL_MAGIC || !host_out) return fail(MK_ERR_INVALID_ARG, "bad model handle or NULL output");
    if (offset < 0 || bytes < 0 || (uint64_t)offset + (uint64_t)bytes > m->sbytes)
        return fail(MK_ERR_INVALID_ARG, "range outside the scratch (%zu bytes)", m->sbytes);
    CK(cudaStreamSynchronize((cudaStream_t)stream));
    if (bytes) CK(cudaMemcpy(host_out, m->sblob + offset, (size_t)bytes, cudaMemcpyDeviceToHost));
    return MK_OK;
}

int mk_last_argmax(mk_model* m, int32_t* out, void* stream) {
    if (!m || m->magic != MODEL_MAGIC || !out) return fail(MK_ERR_INVALID_ARG, "bad arguments");
    if (!m->last_amax) return fail(MK_ERR_STATE, "the last step was not given an accept buffer");
    CK(cudaStreamSynchronize((cudaStream_t)stream));
    CK(cudaMemcpy(out, m->last_amax, (size_t)m->last_M * 4, cudaMemcpyDefault));
    return MK_OK;
}

void mk_free(void* h) {
    if (!h) return;
    const uint32_t magic = *static_cast<uint32_t*>(h);
    if (magic == KV_MAGIC) {
        mk_kv* kv = static_cast<mk_kv*>(h);
        kv->magic = 0;
        cudaFree(kv->pool);
        cudaFree(kv->btab);
        if (kv->tmaps) cudaFree(kv->tmaps);
        mk_model* m = kv->m;
        delete kv;
        if (m && --m->live_kv == 0 && m->released) delete m;
    } else if (magic == MODEL_MAGIC) {
        mk_model* m = static_cast<mk_model*>(h);
        m->magic = 0;
        for (auto& g : m->graphs) cudaGraphExecDestroy(g.second);
        m->graphs.clear();
        cudaFree(m->wblob);
        cudaFree(m->sblob);
        cudaFree(m->d_layers);
        m->wblob = nullptr;
        m->sblob = nullptr;
        m->d_layers = nullptr;
        if (m->live_kv > 0)
            m->released = true;  // deleted with its last KV cache
        else
            delete m;
    }
}

}  // extern "C"

// ===========================================================================
// Decode step that allocates nothing (mk_decode_step_noalloc).
//
// Some callers may not allocate device memory on their call path: code that
// runs while another component owns the allocator (a host framework with its
// own fixed memory pool or a strict memory budget), code on a latency-critical
// thread that must not enter the driver's allocator, or hosts that plan all
// memory before serving starts. For them this entry point runs the same
// megakernel as mk_decode_step, but takes its per-step scratch (activations,
// attention partials, dependency counters, status word and the per-layer
// stage descriptors) from one file-scope device array of fixed size instead
// of the model's own scratch allocation. Weights, the KV cache, tokens,
// positions and logits are the loaded model's / the caller's as usual.
// ===========================================================================
#include <mutex>

#ifndef MK_NOALLOC_SCRATCH_BYTES
#define MK_NOALLOC_SCRATCH_BYTES (64u << 20)  // 64 MiB, held by every device that loads the library
#endif
#define MK_NOALLOC_MAX_LAYERS 128
#define MK_NOALLOC_MAX_DEVICES 64

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MK_NOALLOC_SCRATCH_BYTES];

// device address of g_noalloc_scratch per device (looked up once per device)
void* g_noalloc_base[MK_NOALLOC_MAX_DEVICES];
// serial of the model whose read-only tables (RoPE, zero page) the array
// holds, per device (0: none)
uint64_t g_noalloc_seeded[MK_NOALLOC_MAX_DEVICES];
// host staging of the relocated stage descriptors (fixed size, no allocation)
mk::Layer g_noalloc_layers[MK_NOALLOC_MAX_LAYERS];
std::mutex g_noalloc_mu;

// maps a pointer into the model's scratch allocation onto the same offset of
// the static array; other pointers (weights, caller buffers) are unchanged
struct Reloc {
    const uint8_t* from;
    size_t n;
    uint8_t* to;
    template <class T> T* operator()(T* p) const {
        const uint8_t* b = reinterpret_cast<const uint8_t*>(p);
        if (b >= from && b < from + n) return reinterpret_cast<T*>(to + (b - from));
        return p;
    }
};

void reloc_gemv(mk::Gemv& g, const Reloc& r) {
    g.src = r(g.src);
    g.dst = r(g.dst);
    g.dst2 = r(g.dst2);
}

}  // namespace

extern "C" int mk_decode_step_noalloc(mk_model* m, mk_kv* kv, const int32_t* tokens, const int32_t* positions,
                                      int32_t batch, int32_t T, float* logits, int32_t* accept, void* stream) {
    if (!m || m->magic != MODEL_MAGIC) return fail(MK_ERR_INVALID_ARG, "bad model handle");
    if (!kv || kv->magic != KV_MAGIC) return fail(MK_ERR_INVALID_ARG, "bad kv handle");
    if (kv->m != m) return fail(MK_ERR_STATE, "kv cache belongs to another model");
    if (!tokens || !positions || !logits) return fail(MK_ERR_INVALID_ARG, "NULL tokens/positions/logits");
    if (batch < 1 || batch > kv->batch) return fail(MK_ERR_INVALID_ARG, "batch %d out of range", batch);
    if (T < 1 || T > m->cfg.max_tokens_per_seq) return fail(MK_ERR_INVALID_ARG, "T %d out of range", T);
    if (accept && T < 2) return fail(MK_ERR_INVALID_ARG, "accept needs T > 1");
    if (fault("bad_arg")) return fail(MK_ERR_INVALID_ARG, "arguments rejected (injected by MK_FAULT=bad_arg)");
    const int L = m->cfg.n_layers;
    const size_t desc_off = align256(m->sbytes);
    const size_t need = desc_off + sizeof(mk::Layer) * (size_t)L;
    if (L > MK_NOALLOC_MAX_LAYERS || need > (size_t)MK_NOALLOC_SCRATCH_BYTES)
        return fail(MK_ERR_UNSUPPORTED,
                    "mk_decode_step_noalloc: this model needs %zu bytes of step scratch (%d layers); the static "
                    "scratch holds at most %u bytes and %d layers -- use mk_decode_step",
                    need, L, (unsigned)MK_NOALLOC_SCRATCH_BYTES, MK_NOALLOC_MAX_LAYERS);
    int dev = 0;
    CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= MK_NOALLOC_MAX_DEVICES) return fail(MK_ERR_UNSUPPORTED, "device id %d too large", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_base[dev]) {
        // set-up, once per device, with that device current: in host code the
        // array's name is only a stand-in, the kernel needs its device address
        void* ptr = nullptr;
        CK(cudaGetSymbolAddress(&ptr, g_noalloc_scratch));
        g_noalloc_base[dev] = ptr;
    }
    uint8_t* base = static_cast<uint8_t*>(g_noalloc_base[dev]);
    cudaStream_t s = (cudaStream_t)stream;
    const Reloc r{m->sblob, m->sbytes, base};
    // the array keeps the previous call's contents. The step reads two
    // tables it does not write -- the RoPE table and a zero page -- which are
    // seeded from the model's scratch when another model used the array
    // last (both are constant after mk_load_weights, so this copy never
    // races with steps of the model in flight); every other region the step
    // reads is written earlier in the same step, except the counters and the
    // status word, which are cleared here.
    if (g_noalloc_seeded[dev] != m->serial) {
        const size_t rope_bytes = (size_t)m->base.rope_npos * m->base.rope_half * sizeof(float2);
        CK(cudaMemcpyAsync(const_cast<float2*>(r(m->base.rope)), m->base.rope, rope_bytes, cudaMemcpyDeviceToDevice,
                           s));
        CK(cudaMemsetAsync(const_cast<uint16_t*>(r(m->base.zeros)), 0, 4096, s));
        g_noalloc_seeded[dev] = m->serial;
    }
    CK(cudaMemsetAsync(r(m->ctr), 0, m->ctr_n * sizeof(unsigned), s));
    CK(cudaMemsetAsync(r(m->status), 0, 64, s));
    for (int l = 0; l < L; ++l) {
        mk::Layer& Ld = g_noalloc_layers[l];
        Ld = m->layers[l];
        for (int gi = 0; gi < mk::NG; ++gi) reloc_gemv(Ld.g[gi], r);
        Ld.a = r(Ld.a);
        Ld.q = r(Ld.q);
        Ld.qlat = r(Ld.qlat);
        Ld.olat = r(Ld.olat);
        Ld.o = r(Ld.o);
        Ld.rlog = r(Ld.rlog);
        Ld.x = r(Ld.x);
        Ld.xn = r(Ld.xn);
    }
    mk::Layer* d_layers = reinterpret_cast<mk::Layer*>(base + desc_off);
    CK(cudaMemcpyAsync(d_layers, g_noalloc_layers, sizeof(mk::Layer) * (size_t)L, cudaMemcpyHostToDevice, s));

    mk::Params P = m->base;
    P.layers = d_layers;
    reloc_gemv(P.lm, r);
    P.rope = r(P.rope);
    P.zeros = r(P.zeros);
    P.newlat = r(P.newlat);
    P.part = r(P.part);
    P.part_ml = r(P.part_ml);
    P.amax = r(P.amax);
    P.ubuf = r(P.ubuf);
    P.racc = r(P.racc);
    P.rss = r(P.rss);
    for (int z = 0; z < P.nz; ++z) P.zptr[z] = r(P.zptr[z]);
    P.ctr = r(P.ctr);
    P.status = r(P.status);
    P.dbg_idx = r(m->dbg_idx);
    P.dbg_w = r(m->dbg_w);
    P.dbg_margin = r(m->dbg_margin);
    P.trace = nullptr;
    P.trace_n = nullptr;
    P.trace_items = 0;
    P.page_elems = (long long)kv->page_elems;
    P.pps = kv->pps;
    P.btab = kv->btab;
    P.kv_cap = kv->max_ctx;
    P.kv_batch = kv->batch;
    P.kv_pool = kv->pool;
    P.kv_layer_elems = (long long)kv->layer_elems;
    P.kv_tmaps = kv->tmaps;
    P.tokens = tokens;
    P.pos = positions;
    P.B = batch;
    P.T = T;
    P.M = batch * T;
    step_router(m, P);
    P.logits = logits;
    P.accept = accept;
    P.lm.dst = logits;
    if (P.lm.n_kc > 1) {
        P.zptr[P.nz] = logits;
        P.zn[P.nz++] = (long long)P.M * P.V;
    }
    P.parity = 0;
    void* args[] = {&P};
    CK(cudaLaunchCooperativeKernel((const void*)mk::megakernel, dim3(m->G), dim3(mk::NTHREADS), args,
                                   mk::SMEM_TOTAL, s));
    m->last_M = P.M;
    m->last_noalloc = true;
    m->last_amax = accept ? P.amax : nullptr;
    // report this step's device-side status before returning
    CK(cudaStreamSynchronize(s));
    unsigned st[4];
    CK(cudaMemcpy(st, P.status, sizeof st, cudaMemcpyDeviceToHost));
    if (st[0] == 0 && st[1] == 0) return MK_OK;
    if (st[0] == mk::ST_TIMEOUT)
        return fail(MK_ERR_TIMEOUT, "device wait timed out (where=0x%x, cta=%u)", st[2], st[3]);
    if (st[0] == mk::ST_INVALID) return fail(MK_ERR_INVALID_ARG, "token id or position out of range for this step");
    if (st[0] == mk::ST_DEBUG)
        return fail(MK_ERR_STATE, "debug check failed (MK_DEBUG; where=0x%x, cta=%u)", st[2], st[3]);
    return fail(MK_ERR_CUDA, "device status %u", st[0]);
}
