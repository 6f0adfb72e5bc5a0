/*
 * synth_host.c -- host implementation of the generator defined in synth.h.
 * Built with -ffp-contract=off so that the fp32 multiply and add are never
 * fused (bit-identical to the device implementation on x86 and aarch64).
 */
#include "synth.h"
#include <pthread.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN_GAMMA 0x9e3779b97f4a7c15ULL

uint64_t synth_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

uint64_t synth_draw(uint64_t key, uint64_t j) { return synth_mix64(key + (j + 1) * GOLDEN_GAMMA); }

uint64_t synth_key(uint64_t seed, uint64_t tensor_id) { return synth_mix64(synth_mix64(seed) ^ tensor_id); }

uint64_t synth_tensor_id(int32_t kind, int32_t layer, int32_t expert) {
    return ((uint64_t)(uint32_t)kind << 48) | ((uint64_t)(uint32_t)(layer + 1) << 24) |
           (uint64_t)(uint32_t)expert;
}

static inline uint32_t sum16x4(uint64_t r) {
    return (uint32_t)(r & 0xffff) + (uint32_t)((r >> 16) & 0xffff) + (uint32_t)((r >> 32) & 0xffff) +
           (uint32_t)(r >> 48);
}

float synth_scale_const(float sigma) { return (float)((double)sigma / 65535.0); }

float synth_normal_f32(uint64_t key, uint64_t index, float c, float mean) {
    uint32_t s = sum16x4(synth_draw(key, 3 * index)) + sum16x4(synth_draw(key, 3 * index + 1)) +
                 sum16x4(synth_draw(key, 3 * index + 2));
    float v = (float)((int32_t)s - 393210) * c;
    if (mean != 0.0f) v = v + mean;
    return v;
}

uint16_t synth_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40); /* quiet NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint8_t synth_e4m3_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    const uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    const uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return 0x7f;                 /* NaN */
    if (a >= 0x43e80000u) return (uint8_t)(sign | 0x7e); /* |f| >= 464: saturate to 448 */
    if (a >= 0x3c800000u) {                           /* |f| >= 2^-6: normal E4M3 */
        const uint32_t r = a + 0x7ffffu + ((a >> 20) & 1u); /* keep 3 of 23 mantissa bits, ties to even */
        const uint32_t e = (r >> 23) - 127u + 7u, m = (r >> 20) & 7u;
        return (uint8_t)(sign | (e << 3) | m);
    }
    /* subnormal E4M3: multiples of 2^-9 (8 of them give the smallest normal) */
    float x, fa;
    memcpy(&fa, &a, 4);
    x = fa * 512.0f;                                  /* exact: a power-of-two scaling */
    uint32_t n = (uint32_t)x;
    const float fr = x - (float)n;                    /* exact: x < 8 */
    if (fr > 0.5f || (fr == 0.5f && (n & 1u))) ++n;
    return (uint8_t)(sign | n);
}

void synth_fill_e4m3(uint8_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t index0, int threads) {
    /* the bf16 fill's normal draws, one fp32 value at a time (no threads
     * needed at the sizes the CPU side generates) */
    (void)threads;
    const uint64_t key = synth_key(seed, tensor_id);
    const float c = synth_scale_const(SYNTH_F8_SIGMA);
    for (uint64_t i = 0; i < n; ++i) out[i] = synth_e4m3_rne(synth_normal_f32(key, index0 + i, c, 0.0f));
}

void synth_fill_e8m0(uint8_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t index0) {
    const uint64_t key = synth_key(seed, tensor_id);
    for (uint64_t i = 0; i < n; ++i) out[i] = (uint8_t)(117u + (uint32_t)(synth_draw(key, index0 + i) & 1u));
}

typedef struct {
    uint16_t* out;
    uint64_t lo, hi, key, index0;
    float c, mean;
} fill_job;

static void* fill_worker(void* p) {
    fill_job* j = (fill_job*)p;
    for (uint64_t i = j->lo; i < j->hi; ++i)
        j->out[i] = synth_bf16_rne(synth_normal_f32(j->key, j->index0 + i, j->c, j->mean));
    return 0;
}

void synth_fill_bf16(uint16_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id, float sigma, float mean,
                     uint64_t index0, int threads) {
    uint64_t key = synth_key(seed, tensor_id);
    float c = synth_scale_const(sigma);
    if (threads <= 0) {
        long nc = sysconf(_SC_NPROCESSORS_ONLN);
        threads = nc > 0 ? (int)nc : 1;
    }
    if (threads > 64) threads = 64;
    if (n < (1u << 16) || threads == 1) {
        fill_job j = {out, 0, n, key, index0, c, mean};
        fill_worker(&j);
        return;
    }
    pthread_t tid[64];
    int started[64];
    fill_job jobs[64];
    uint64_t per = (n + threads - 1) / threads;
    for (int t = 0; t < threads; ++t) {
        uint64_t lo = per * t, hi = lo + per > n ? n : lo + per;
        started[t] = 0;
        if (lo >= hi) continue;
        jobs[t] = (fill_job){out, lo, hi, key, index0, c, mean};
        if (pthread_create(&tid[t], 0, fill_worker, &jobs[t]) == 0)
            started[t] = 1;
        else
            fill_worker(&jobs[t]);
    }
    for (int t = 0; t < threads; ++t)
        if (started[t]) pthread_join(tid[t], 0);
}

int32_t synth_token(uint64_t seed, int64_t step, int32_t b, int32_t t, int32_t vocab) {
    uint64_t key = synth_key(seed, synth_tensor_id(SYNTH_TOKENS, -1, 0));
    uint64_t j = ((uint64_t)step << 20) + ((uint64_t)(uint32_t)b << 10) + (uint64_t)(uint32_t)t;
    return (int32_t)(synth_draw(key, j) % (uint64_t)(uint32_t)vocab);
}

int synth_weight_spec(const synth_dims* d, int32_t kind, int32_t* rows, int32_t* cols, float* sigma,
                      float* mean) {
    int32_t r = 0, c = 0;
    float s = 0.02f, m = 0.0f;
    int gqa = d->attn_kind == 0, mla = d->attn_kind == 1, moe = d->n_routed_experts > 0;
    int sh = d->n_shared_experts > 0;
    switch (kind) {
    case SYNTH_EMBED: case SYNTH_LM_HEAD: r = d->vocab; c = d->d_model; break;
    case SYNTH_FINAL_NORM: case SYNTH_ATTN_NORM: case SYNTH_FFN_NORM: r = 1; c = d->d_model; m = 1.0f; break;
    case SYNTH_WQ: if (!gqa) return -1; r = d->n_q_heads * d->head_dim; c = d->d_model; break;
    case SYNTH_WK: case SYNTH_WV: if (!gqa) return -1; r = d->n_kv_heads * d->head_dim; c = d->d_model; break;
    case SYNTH_WO:
        r = d->d_model;
        c = gqa ? d->n_q_heads * d->head_dim : d->n_q_heads * d->v_head_dim;
        break;
    case SYNTH_WDQ: if (!mla) return -1; r = d->q_lora_rank; c = d->d_model; break;
    case SYNTH_Q_NORM: if (!mla) return -1; r = 1; c = d->q_lora_rank; m = 1.0f; break;
    case SYNTH_WUQ: if (!mla) return -1; r = d->n_q_heads * (d->qk_nope_dim + d->qk_rope_dim); c = d->q_lora_rank; break;
    case SYNTH_WDKV: if (!mla) return -1; r = d->kv_lora_rank + d->qk_rope_dim; c = d->d_model; break;
    case SYNTH_KV_NORM: if (!mla) return -1; r = 1; c = d->kv_lora_rank; m = 1.0f; break;
    case SYNTH_WUKV: if (!mla) return -1; r = d->n_q_heads * (d->qk_nope_dim + d->v_head_dim); c = d->kv_lora_rank; break;
    case SYNTH_ROUTER: if (!moe) return -1; r = d->n_routed_experts; c = d->d_model; break;
    case SYNTH_GATE: case SYNTH_UP: if (!moe) return -1; r = d->ffn_dim; c = d->d_model; break;
    case SYNTH_DOWN: if (!moe) return -1; r = d->d_model; c = d->ffn_dim; break;
    case SYNTH_SH_GATE: case SYNTH_SH_UP: if (!sh) return -1; r = d->shared_ffn_dim; c = d->d_model; break;
    case SYNTH_SH_DOWN: if (!sh) return -1; r = d->d_model; c = d->shared_ffn_dim; break;
    case SYNTH_GATE_SCALE: case SYNTH_UP_SCALE: case SYNTH_DOWN_SCALE:
    case SYNTH_SH_GATE_SCALE: case SYNTH_SH_UP_SCALE: case SYNTH_SH_DOWN_SCALE:
        /* one E8M0 byte per block of 32 elements of the code tensor's rows */
        if (synth_weight_spec(d, kind - 6, &r, &c, 0, 0) != 0 || c % SYNTH_MX_BLOCK) return -1;
        c /= SYNTH_MX_BLOCK;
        break;
    default: return -1;
    }
    if (rows) *rows = r;
    if (cols) *cols = c;
    if (sigma) *sigma = s;
    if (mean) *mean = m;
    return 0;
}

int32_t synth_kv_row(const synth_dims* d, int32_t kind) {
    if (kind == SYNTH_KV_LATENT) return d->attn_kind == 1 ? d->kv_lora_rank + d->qk_rope_dim : -1;
    if (kind == SYNTH_KV_K || kind == SYNTH_KV_V) return d->attn_kind == 0 ? d->n_kv_heads * d->head_dim : -1;
    return -1;
}
