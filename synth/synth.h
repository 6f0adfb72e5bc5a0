/*
 * synth.h -- seeded synthetic inputs for the MoE decode step.
 *
 * This module is the ONE piece of code shared by the CPU oracle and the
 * harness that feeds the CUDA path. It holds no model arithmetic: it only
 * turns (seed, tensor id, element index) into numbers, and knows the shape and
 * scale of each synthetic tensor (the input recipe).
 *
 * Generator (stated once, implemented twice -- synth_host.c and synth_cuda.cu
 * -- from this definition, and checked bit-identical by a GPU test):
 *
 *   mix64(z)      : the SplitMix64 output finaliser (Steele, Lea & Flood,
 *                   "Fast splittable pseudorandom number generators",
 *                   OOPSLA 2014; the variant in Vigna's public splitmix64.c):
 *                     z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9
 *                     z = (z ^ (z >> 27)) * 0x94d049bb133111eb
 *                     return z ^ (z >> 31)
 *   draw(key, j)  : mix64(key + (j + 1) * 0x9e3779b97f4a7c15), i.e. the j-th
 *                   output of a SplitMix64 stream started at `key`.
 *   key(seed, id) : mix64(mix64(seed) ^ id)
 *   normal(key,i) : Irwin-Hall(12) approximation of N(0,1). Take the three
 *                   64-bit draws j = 3i, 3i+1, 3i+2, split each into four
 *                   16-bit fields, S = sum of the 12 fields (an integer in
 *                   [0, 786420]). value = float(S - 393210) * c, where
 *                   c = float(sigma / 65535.0) is rounded once from double,
 *                   then (optionally) + mean, each an IEEE fp32 operation with
 *                   round-to-nearest-even and no fused multiply-add; finally
 *                   rounded to bf16 with round-to-nearest-even.
 *   token(seed, step, b, t, V): draw(key(seed, TOKENS id), step*2^20 + b*2^10 + t) mod V
 *
 * MXFP8 expert weights (the microscaling format of the OCP "Microscaling
 * Formats (MX) Specification" v1.0: each block of 32 consecutive elements of
 * a row shares one E8M0 scale byte E, value 2^(E-127); the elements are FP8
 * E4M3 codes -- sign, 4 exponent bits of bias 7, 3 mantissa bits, subnormals
 * of quantum 2^-9, largest finite 448, codes 0x7F/0xFF NaN, no infinities):
 *   code(i)   = e4m3_rne(normal(key, i) with sigma 16): the same normal draw
 *               as a bf16 weight, rounded to E4M3 (nearest, ties to even;
 *               |value| >= 464 saturates to 448, NaN gives 0x7F) instead of
 *               bf16. |16 N| <= 96, so no draw saturates.
 *   scale(b)  = 117 + (draw(key(seed, scale tensor id), b) & 1): 2^-10 or
 *               2^-9, block b = row * (cols / 32) + column / 32.
 * The elements are then about N(0, 0.016..0.031), the bf16 recipe's scale.
 * The scale tensors have kinds of their own (GATE_SCALE .. SH_DOWN_SCALE).
 *
 * Recipe (the reading of "weights bf16 N(0, 0.02)" and "KV bf16 N(0, 1)"):
 * matrices and embeddings sigma = 0.02, mean 0; RMSNorm gains sigma = 0.02,
 * mean 1; pre-filled KV entries sigma = 1, mean 0. KV entries are indexed
 * position-major (index = pos * row_len + j) so a longer context extends a
 * shorter one.
 */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* tensor kinds (the "kind" field of a tensor id) */
enum synth_kind {
    SYNTH_EMBED = 1, SYNTH_LM_HEAD = 2, SYNTH_FINAL_NORM = 3,
    SYNTH_ATTN_NORM = 4, SYNTH_FFN_NORM = 5,
    /* GQA */
    SYNTH_WQ = 6, SYNTH_WK = 7, SYNTH_WV = 8, SYNTH_WO = 9,
    /* MLA */
    SYNTH_WDQ = 10, SYNTH_Q_NORM = 11, SYNTH_WUQ = 12, SYNTH_WDKV = 13,
    SYNTH_KV_NORM = 14, SYNTH_WUKV = 15,
    /* MoE */
    SYNTH_ROUTER = 16, SYNTH_GATE = 17, SYNTH_UP = 18, SYNTH_DOWN = 19,
    SYNTH_SH_GATE = 20, SYNTH_SH_UP = 21, SYNTH_SH_DOWN = 22,
    /* E8M0 block scales of the MXFP8 expert weights (kind of the codes + 6) */
    SYNTH_GATE_SCALE = 23, SYNTH_UP_SCALE = 24, SYNTH_DOWN_SCALE = 25,
    SYNTH_SH_GATE_SCALE = 26, SYNTH_SH_UP_SCALE = 27, SYNTH_SH_DOWN_SCALE = 28,
    /* non-weight streams */
    SYNTH_KV_K = 40, SYNTH_KV_V = 41, SYNTH_KV_LATENT = 42, SYNTH_TOKENS = 43
};

/* model dimensions, as far as the recipe needs them */
typedef struct synth_dims {
    int32_t n_layers, d_model, vocab, attn_kind; /* attn_kind 0 = GQA, 1 = MLA */
    int32_t n_q_heads, n_kv_heads, head_dim;
    int32_t q_lora_rank, kv_lora_rank, qk_nope_dim, qk_rope_dim, v_head_dim;
    int32_t n_routed_experts, top_k, n_shared_experts, ffn_dim, shared_ffn_dim;
} synth_dims;

uint64_t synth_mix64(uint64_t z);
uint64_t synth_draw(uint64_t key, uint64_t j);
uint64_t synth_key(uint64_t seed, uint64_t tensor_id);
/* tensor id of (kind, layer, expert); layer -1 for tensors outside the layer
 * stack; expert is the expert index, or the sequence index for KV streams */
uint64_t synth_tensor_id(int32_t kind, int32_t layer, int32_t expert);
float    synth_normal_f32(uint64_t key, uint64_t index, float c, float mean);
uint16_t synth_bf16_rne(float f);
float    synth_scale_const(float sigma);   /* float(sigma / 65535.0) */

/* fill out[0..n) with elements index0 .. index0+n-1 of tensor `tensor_id`
 * (bf16 bit patterns); uses up to `threads` host threads (<=0: all) */
void synth_fill_bf16(uint16_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id,
                     float sigma, float mean, uint64_t index0, int threads);

int32_t synth_token(uint64_t seed, int64_t step, int32_t b, int32_t t, int32_t vocab);

#define SYNTH_F8_SIGMA 16.0f      /* sigma of the normal draws behind E4M3 codes */
#define SYNTH_MX_BLOCK 32         /* elements per E8M0 scale */
/* fp32 -> FP8 E4M3 code, round to nearest even, saturating (see above) */
uint8_t synth_e4m3_rne(float f);
/* E4M3 codes of elements index0 .. index0+n-1 of tensor `tensor_id` */
void synth_fill_e4m3(uint8_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t index0, int threads);
/* E8M0 scale bytes of blocks index0 .. index0+n-1 of scale tensor `tensor_id` */
void synth_fill_e8m0(uint8_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t index0);

/* shape and scale of weight tensor (kind, layer, expert) under the recipe.
 * returns 0 and fills rows/cols/sigma/mean if the tensor exists for these
 * dims, -1 otherwise. 1-D tensors (norm gains) report rows = 1. */
int synth_weight_spec(const synth_dims* d, int32_t kind, int32_t* rows, int32_t* cols,
                      float* sigma, float* mean);

/* row length of one cached position for KV kind (SYNTH_KV_K / _V / _LATENT) */
int32_t synth_kv_row(const synth_dims* d, int32_t kind);

#ifdef __cplusplus
}
#endif
#endif
