/*
 * oracle.h -- C ABI of the CPU oracle for one MoE/dense transformer decode
 * (or speculative-verify) step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, import or
 * call this library; it exists so that tests, the smoke check and the bench's
 * CPU baseline have an independent, obviously-correct reference. It shares no
 * code with the CUDA path; its only shared dependency is the synthetic input
 * generator (synth/), which holds none of the model's arithmetic.
 *
 * What it computes (the plain definition, single thread, accumulation type
 * fp32 or fp64 chosen per call): embedding lookup; per layer RMSNorm, GQA or
 * MLA attention over a bf16 KV cache with rotate-half RoPE, output
 * projection and residual; RMSNorm, softmax router with top-k and
 * renormalised weights, routed and shared SwiGLU experts, residual; final
 * RMSNorm and LM head; optionally the expert weights in MXFP8 (E4M3 codes
 * with an E8M0 scale per 32 elements of a row, the OCP "Microscaling
 * Formats (MX) Specification" v1.0), dequantised exactly before the same
 * plain step (the pages state no weight precision). Sources: "TPU Megakernel Achieves 709 tokens/s on Kimi
 * K3" (kongchang.com), section "The Key Innovation" (all layers are MoE
 * layers with per-layer routing) and the MoE explainer after "Cross-Layer
 * Weight Prefetching" (a router picks a few experts per token); the myzaker
 * article, section on fusing hundreds of small kernels (decode re-reads the
 * weights for every token); the Inferact blog translation on tanhow.com,
 * paragraph on VMEM lifetimes (MLA KV cache); the myzaker article's
 * speculative-decoding paragraphs (draft tokens verified in one batch). Model
 * shapes and every detail the pages leave open follow the readings listed in
 * the design notes (router softmax then top-k then renormalise; rotate-half
 * RoPE with theta 1e4; contiguous GQA head groups; bf16 round-to-nearest-even
 * KV append; absorbed and unabsorbed MLA both provided).
 */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

typedef struct oracle_cfg {
    int32_t n_layers, d_model, vocab, attn_kind; /* 0 GQA, 1 MLA */
    int32_t n_q_heads, n_kv_heads, head_dim;
    int32_t q_lora_rank, kv_lora_rank, qk_nope_dim, qk_rope_dim, v_head_dim;
    int32_t n_routed_experts, top_k, n_shared_experts, ffn_dim, shared_ffn_dim;
    float rms_eps, rope_theta;
    /* 0: every weight bf16; 1: routed and shared expert weights MXFP8 (the
     * generator's E4M3 codes and E8M0 block scales, dequantised exactly) */
    int32_t expert_format;
} oracle_cfg;

typedef struct oracle_model oracle_model;
typedef struct oracle_kv oracle_kv;

/* Weights come from the synthetic generator with `seed`, produced on first
 * use. lazy != 0 releases a layer's tensors once the layer has been
 * processed (for models larger than host memory). gen_threads: host threads
 * the generator may use (the oracle's arithmetic is always single-threaded). */
oracle_model* oracle_create(const oracle_cfg* cfg, uint64_t seed, int lazy, int gen_threads);
void oracle_destroy(oracle_model* m);
/* Replace one weight tensor by caller data (bf16 bits, canonical [rows, cols]
 * row-major, copied). kind/layer/expert as in synth.h. Returns 0 or -1. */
int oracle_set_tensor(oracle_model* m, int32_t kind, int32_t layer, int32_t expert, const uint16_t* data,
                      int64_t n);
/* Copy a weight tensor out (generating it if needed). Returns element count or -1. */
int64_t oracle_get_tensor(oracle_model* m, int32_t kind, int32_t layer, int32_t expert, uint16_t* out,
                          int64_t cap);

/* KV cache: per layer and sequence a contiguous bf16 array of max_pos rows.
 * GQA row = [K: Hkv*hd | V: Hkv*hd]; MLA row = [c_kv: kv_lora | k_rope: rope]. */
oracle_kv* oracle_kv_create(const oracle_model* m, int32_t batch, int32_t max_pos);
void oracle_kv_destroy(oracle_kv* kv);
/* fill positions [0, ctx) of every layer and sequence from the generator */
int oracle_kv_prefill(oracle_kv* kv, uint64_t seed, int32_t ctx, int gen_threads);
int oracle_kv_rows(const oracle_kv* kv, int32_t layer, int32_t seq, int32_t pos0, int32_t n, uint16_t* out,
                   int write);
int32_t oracle_kv_row_len(const oracle_kv* kv);

/* One decode step. tokens [B*T] (row-major b, t), positions [B] = position of
 * each sequence's first token in this step. Outputs (any may be NULL):
 *   logits [B*T, V] (as double), route_idx [L, B*T, k], route_w [L, B*T, k],
 *   route_margin [L, B*T] (fp router-logit gap between k-th and (k+1)-th),
 *   accept [B] greedy acceptance length (T > 1: 1 + leading draft matches).
 * precision: 32 or 64. mla_absorbed: 0 decompresses K/V per head and
 * position (the plain definition), 1 uses the absorbed form.
 * Returns 0, or -1 on bad arguments. */
int oracle_decode(oracle_model* m, oracle_kv* kv, const int32_t* tokens, const int32_t* positions, int32_t B,
                  int32_t T, int precision, int mla_absorbed, double* logits, int32_t* route_idx,
                  double* route_w, double* route_margin, int32_t* accept);

/* Brute force: run tokens [B, P] from position 0 with no cache at all --
 * every layer recomputes K/V for all positions (rounded to bf16 like the
 * cache) and applies an explicit causal softmax(QK^T)V. logits [B, P, V]. */
int oracle_full_recompute(oracle_model* m, const int32_t* tokens, int32_t B, int32_t P, int precision,
                          double* logits);

/* Building blocks, exposed for pinning (all fp64 unless stated). */
double oracle_e4m3_value(uint8_t code);
void oracle_mx_dequant(const uint8_t* codes, const uint8_t* scales, int32_t rows, int32_t cols, double* out);
void oracle_rmsnorm(const double* x, const uint16_t* gain, int32_t n, double eps, double* out);
void oracle_rope(double* x, int32_t dim, int32_t pos, double theta);
void oracle_softmax(const double* x, int32_t n, double* out);
void oracle_topk(const double* logits, int32_t n, int32_t k, int32_t* idx, double* w, double* margin);
double oracle_silu(double z);
/* single-query GQA-style attention over n cached rows: q [hd], K/V [n, hd] bf16 */
void oracle_attend(const double* q, const uint16_t* K, const uint16_t* V, int32_t n, int32_t hd, double scale,
                   double* out);

#ifdef __cplusplus
}
#endif
#endif
