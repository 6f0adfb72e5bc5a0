/*
 * mk.h -- C ABI of the single-launch MoE decode megakernel for GB300 (sm_103a).
 *
 * One call of mk_decode_step runs one decode step (T = 1) or one speculative
 * verify step (T > 1) of a Mixture-of-Experts (or dense) transformer: every
 * layer -- RMSNorm, GQA or MLA attention over a paged bf16 KV cache, output
 * projection, softmax/top-k router, shared and routed SwiGLU experts,
 * residual updates -- then the final norm and the LM head, in ONE persistent
 * kernel launch. While one stage computes, a producer warp in every CTA keeps
 * streaming the weight tiles of the following stages (and layers) into a
 * shared-memory ring with TMA bulk copies, so HBM stays busy across layer
 * boundaries.
 *
 * Sources (the pages describe the method, not an interface; the interface is
 * this library's own):
 *  - all MoE layers of the model in a single kernel, no per-layer launches:
 *    "TPU Megakernel Achieves 709 tokens/s on Kimi K3" (kongchang.com),
 *    section "The Key Innovation: 92 MoE Layers in a Single Pallas Kernel";
 *  - weights of the next layer move while the current layer computes:
 *    same page, section "Cross-Layer Weight Prefetching"; the myzaker article,
 *    section on fusing hundreds of small kernels ("attention weights of layer
 *    N+1 already move while layer N runs its MoE");
 *  - decode is bound by moving weights from HBM, every token re-reads them:
 *    myzaker article, same section; tanhow.com translation of the Inferact
 *    blog, paragraph on the memory-bandwidth limit;
 *  - router picks a few experts per token, per layer: kongchang.com, MoE
 *    explainer after "Cross-Layer Weight Prefetching";
 *  - MLA KV cache: tanhow.com translation, paragraph on VMEM lifetimes;
 *  - speculative verification of draft tokens in one batch: myzaker article,
 *    DSpark paragraphs; paged KV (PagedAttention): myzaker article, section
 *    on the vLLM founders.
 *
 * Conventions for every entry point:
 *  - returns MK_OK (0) or a negative mk_status; the thread-local message of
 *    the last failure is available from mk_last_error();
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream);
 *  - pointers documented as "device" must be device (or managed) memory of
 *    the current device; "host or device" accepts either (copied with
 *    cudaMemcpyDefault);
 *  - the library never exits the process and never traps on the device.
 */
#ifndef MK_H
#define MK_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

#define MK_ABI_VERSION 2

typedef enum mk_status {
    MK_OK = 0,
    MK_ERR_INVALID_ARG = -1, /* bad pointer, size, shape, position or token id */
    MK_ERR_OOM = -2,         /* device allocation failed */
    MK_ERR_CUDA = -3,        /* a CUDA runtime call failed */
    MK_ERR_UNSUPPORTED = -4, /* configuration outside what the kernel implements */
    MK_ERR_TIMEOUT = -5,     /* a device-side wait exceeded its time limit; the step was abandoned */
    MK_ERR_STATE = -6        /* call out of order (e.g. kv from another model) */
} mk_status;

enum { MK_ATTN_GQA = 0, MK_ATTN_MLA = 1 };

/* Model shape. GQA uses n_q_heads/n_kv_heads/head_dim; MLA uses n_q_heads
 * plus the *_rank/*_dim fields. n_routed_experts = 0 gives a dense model whose
 * MLP is the shared expert (n_shared_experts = 1, shared_ffn_dim wide). */
typedef struct mk_config {
    int32_t n_layers, d_model, vocab, attn_kind;
    int32_t n_q_heads, n_kv_heads, head_dim;
    int32_t q_lora_rank, kv_lora_rank, qk_nope_dim, qk_rope_dim, v_head_dim;
    int32_t n_routed_experts, top_k, n_shared_experts, ffn_dim, shared_ffn_dim;
    int32_t max_batch, max_tokens_per_seq, max_ctx, kv_page_size;
    float rms_eps, rope_theta;
    int32_t expert_format;  /* mk_expert_format: how routed and shared expert weights are stored */
} mk_config;

/* Expert weight formats.
 *  MK_EXPERT_BF16  every weight bf16 (the default).
 *  MK_EXPERT_MXFP8 the gate, up and down weights of the routed and shared
 *      experts in the MXFP8 format of the OCP "Microscaling Formats (MX)
 *      Specification" v1.0: FP8 E4M3 elements (sign, 4 exponent bits of bias
 *      7, 3 mantissa bits, subnormals) with one E8M0 scale byte E (value
 *      2^(E-127)) per block of 32 consecutive elements of a row; the weight is
 *      element x scale. About half the bytes of bf16 experts (1 + 1/32 bytes
 *      per weight). The kernel takes the dequantised values exactly; scale
 *      byte 0xFF (NaN in the format) is not supported.
 *      Supported for d_model 512, 1024 or 2048 (one K panel per expert row),
 *      ffn_dim and shared_ffn_dim multiples of 64, any batch and tokens per
 *      step (each of an expert unit's tokens takes the unit's tiles in turn on
 *      the CUDA cores; the bf16 experts' tensor-core tiles for several tokens
 *      have no MXFP8 counterpart); other shapes give MK_ERR_UNSUPPORTED at
 *      load. */
enum mk_expert_format { MK_EXPERT_BF16 = 0, MK_EXPERT_MXFP8 = 1 };

/* Weight kinds. Canonical layouts are row-major [rows, cols] bf16:
 *  EMBED, LM_HEAD [vocab, d]; *_NORM gains [n];
 *  GQA: WQ [Hq*hd, d], WK/WV [Hkv*hd, d], WO [d, Hq*hd];
 *  MLA: WDQ [q_lora, d], Q_NORM [q_lora], WUQ [H*(nope+rope), q_lora] (per
 *       head: nope rows then rope rows), WDKV [kv_lora+rope, d] (latent rows
 *       then k_rope rows), KV_NORM [kv_lora], WUKV [H*(nope+v), kv_lora]
 *       (per head: W_uk rows then W_uv rows), WO [d, H*v];
 *  MoE: ROUTER [E, d]; per expert GATE/UP [ffn, d], DOWN [d, ffn];
 *  shared expert: SH_GATE/SH_UP [sffn, d], SH_DOWN [d, sffn].
 * With expert_format MK_EXPERT_MXFP8, GATE, UP, DOWN, SH_GATE, SH_UP and
 * SH_DOWN hold one E4M3 code byte per element (same shapes), and the *_SCALE
 * kinds their E8M0 scale bytes, [rows, cols / 32] (block b of row r scales
 * elements 32 b .. 32 b + 31 of that row). */
enum mk_weight_kind {
    MK_W_EMBED = 1, MK_W_LM_HEAD = 2, MK_W_FINAL_NORM = 3, MK_W_ATTN_NORM = 4, MK_W_FFN_NORM = 5,
    MK_W_WQ = 6, MK_W_WK = 7, MK_W_WV = 8, MK_W_WO = 9,
    MK_W_WDQ = 10, MK_W_Q_NORM = 11, MK_W_WUQ = 12, MK_W_WDKV = 13, MK_W_KV_NORM = 14, MK_W_WUKV = 15,
    MK_W_ROUTER = 16, MK_W_GATE = 17, MK_W_UP = 18, MK_W_DOWN = 19,
    MK_W_SH_GATE = 20, MK_W_SH_UP = 21, MK_W_SH_DOWN = 22,
    MK_W_GATE_SCALE = 23, MK_W_UP_SCALE = 24, MK_W_DOWN_SCALE = 25,
    MK_W_SH_GATE_SCALE = 26, MK_W_SH_UP_SCALE = 27, MK_W_SH_DOWN_SCALE = 28
};

/* One entry of the weight table: layer = -1 for EMBED/LM_HEAD/FINAL_NORM,
 * expert = routed expert index (0 otherwise); data = bf16 bits (or MXFP8
 * code / scale bytes) in the canonical layout, host or device memory, only
 * read during the call. */
typedef struct mk_weight {
    int32_t kind, layer, expert, reserved;
    const void* data;
} mk_weight;

typedef struct mk_model mk_model;
typedef struct mk_kv mk_kv;

/* Static facts about a loaded model (sizes in bytes). */
typedef struct mk_info {
    int64_t weight_bytes;      /* packed weights resident in HBM */
    int64_t scratch_bytes;     /* activations, partials, counters */
    int32_t grid_ctas;         /* persistent CTAs (one per SM) */
    int32_t threads_per_cta;
    int32_t smem_bytes;        /* dynamic shared memory per CTA */
    int32_t ring_slots, slot_bytes;
    int32_t sm_count;
} mk_info;

/* Validate `cfg`, allocate device memory for all weights and per-step
 * scratch, and copy every tensor of `table` (n entries; each required tensor
 * exactly once) into the library's packed layout. The caller keeps ownership
 * of its buffers. Errors: INVALID_ARG (bad/missing/duplicate tensor),
 * UNSUPPORTED (shape the kernel does not implement), OOM, CUDA.
 * Synchronises `stream` before returning.
 * Schedule: for steps of two or more tokens, when the attention output
 * projection has one K panel, the CTAs that compute it also accumulate the
 * router logits of their rows, and the step has no separate router stage.
 * With the environment variable MK_ROUTER_STAGE=1 set at this call, the
 * model always keeps the separate router stage (the schedule used
 * otherwise); results agree within rounding. Likewise, for MLA models and
 * steps of at most 16 tokens, the CTAs of the query up-projection also apply
 * the absorbed key projection, and the CTAs that merge the attention splits
 * also apply the value up-projection; MK_QLAT_STAGE=1 and MK_UV_STAGE=1 keep
 * those as stages of their own. */
int mk_load_weights(const mk_config* cfg, const mk_weight* table, int32_t n, void* stream, mk_model** out);

/* mk_load_weights over seeded synthetic weights generated in device memory:
 * every tensor the model of `cfg` has, element i of tensor (kind, layer,
 * expert) drawn by the input recipe's counter-based generator (SplitMix64
 * hash of (seed, tensor id, i), Irwin-Hall(12) normal draw, bf16 round to
 * nearest even; matrices and embeddings N(0, 0.02), RMSNorm gains
 * 1 + N(0, 0.02)). The same numbers a caller gets from the generator module
 * on the host, so a CPU reference can rebuild the model from (cfg, seed).
 * Holds a temporary device copy of all weights during the call (about the
 * size of mk_info.weight_bytes). Errors as mk_load_weights. Synchronises
 * `stream`. The pages use trained weights; the synthetic model stands in for
 * them with the stated shapes (workload descriptions of the deep MoE model:
 * bf16 weights drawn from N(0, 0.02)). With expert_format MK_EXPERT_MXFP8
 * the expert weights are the generator's E4M3 codes (the same normal draws
 * with sigma 16, rounded to E4M3 nearest even) and E8M0 block scales (117 or
 * 118: 2^-10 or 2^-9). */
int mk_load_synthetic(const mk_config* cfg, uint64_t seed, void* stream, mk_model** out);

/* Paged KV cache for `batch` sequences of up to `max_ctx` positions each
 * (must be <= cfg.max_ctx, batch <= cfg.max_batch). Pages hold
 * cfg.kv_page_size positions. The default block table interleaves the
 * sequences' pages (page j of sequence b is physical page j*batch + b).
 * Contents start as zeros. */
int mk_alloc_kv(const mk_model* m, int32_t batch, int32_t max_ctx, mk_kv** out);

/* Replace the block table: host array [batch][pages_per_seq] of distinct
 * physical page ids in [0, batch*pages_per_seq). Synchronous. */
int mk_kv_set_block_table(mk_kv* kv, const int32_t* table);
int32_t mk_kv_pages_per_seq(const mk_kv* kv);

/* Copy n positions [pos0, pos0+n) of sequence `seq`, layer `layer` between
 * the cache and `rows` (host or device; bf16 [n][row], row = [K heads | V
 * heads] (2*Hkv*hd) for GQA, [latent | k_rope] (kv_lora+rope) for MLA). The
 * row layout is the logical one; pages and the block table are hidden.
 * Asynchronous on `stream` when `rows` is device memory. */
int mk_kv_write(mk_kv* kv, int32_t layer, int32_t seq, int32_t pos0, int32_t n, const void* rows, void* stream);
int mk_kv_read(const mk_kv* kv, int32_t layer, int32_t seq, int32_t pos0, int32_t n, void* rows, void* stream);

/* One decode (T = 1) or verify (T > 1) step of `batch` sequences.
 *  tokens    device int32 [batch*T], token t of sequence b at b*T + t;
 *  positions device int32 [batch], position of each sequence's first token
 *            in this step; positions [0, positions[b]) of the cache must
 *            hold that sequence's context; the step writes K/V (or latents)
 *            for positions [positions[b], positions[b]+T);
 *  logits    device float [batch*T, vocab] (written);
 *  accept    device int32 [batch] or NULL: greedy acceptance length (1 + the
 *            number of leading draft tokens t+1 that equal the argmax of the
 *            logits at t; argmax ties go to the lower id). Needs T > 1.
 * Asynchronous: argument errors are returned immediately; errors found on
 * the device (token or position out of range, timeouts) are reported by the
 * next mk_step_status. */
int mk_decode_step(mk_model* m, mk_kv* kv, const int32_t* tokens, const int32_t* positions, int32_t batch,
                   int32_t T, float* logits, int32_t* accept, void* stream);

/* The same step as mk_decode_step, run as one kernel launch per stage
 * instead of one launch for the whole step: the comparison point for what a
 * single launch buys. The pages contrast a decode step of hundreds of small
 * kernels, whose boundaries stall the weight stream, with one fused program
 * (myzaker article, section on fusing hundreds of small kernels into one
 * program; tanhow.com translation of the Inferact blog, paragraph on kernel
 * boundaries, CUDA Graphs and programmatic dependent launch). Here each
 * stage (per layer: the attention projections, attention, its combine, the
 * output projection, the router, the experts; then the LM head) is its own
 * launch of the same kernel code, ordered by the stream instead of by
 * dependency counters, so no stage's weights move before the previous
 * stage has finished; the launches are replayed from a CUDA graph (captured
 * on the first call of each shape: kv, batch, T, logits and accept buffers)
 * with programmatic dependent launch between them. Same arguments, results
 * and error reporting as mk_decode_step; token ids and positions are copied
 * into the model's own buffers first (so the graph does not depend on
 * them). The first call of a shape captures into a private stream and must
 * not itself be made while `stream` is being captured. */
int mk_decode_step_unfused(mk_model* m, mk_kv* kv, const int32_t* tokens, const int32_t* positions, int32_t batch,
                           int32_t T, float* logits, int32_t* accept, void* stream);

/* mk_decode_step without any allocation on the call path. The pages have no
 * counterpart of this entry point: it is for callers that may not allocate
 * device memory while they run -- code inside a host framework that owns a
 * fixed memory pool or budget, or a latency-critical serving thread that
 * must stay out of the driver's allocator.
 * Same arguments and results as mk_decode_step. The step's scratch
 * (activations, attention partials, dependency counters, status word, stage
 * descriptors) lives in one static device array of 64 MiB that every device
 * which loads this library holds until the process exits; a model whose
 * step scratch (mk_info.scratch_bytes plus about 1.3 KB per layer) does not
 * fit, or that has more than 128 layers, is rejected with
 * MK_ERR_UNSUPPORTED. The first call on each device looks up the array's
 * device address. All calls share the array, which keeps the last call's contents;
 * each call clears what must start at zero (dependency counters, status
 * word) and, when another model used the array last, copies in the model's
 * constant tables (RoPE angles, a zero page). Calls that overlap on the GPU
 * (work of other streams or host threads still in flight) race on the
 * array. The model's own scratch is neither read nor written. The call
 * synchronises `stream` and returns the step's device status itself
 * (MK_OK, MK_ERR_TIMEOUT, MK_ERR_INVALID_ARG); afterwards mk_debug_routing
 * returns MK_ERR_STATE (this path keeps no routing record) and
 * mk_last_argmax reads the static array. */
int mk_decode_step_noalloc(mk_model* m, mk_kv* kv, const int32_t* tokens, const int32_t* positions, int32_t batch,
                           int32_t T, float* logits, int32_t* accept, void* stream);

/* Fault injection on the host (testing the caller's error handling; the GPU
 * is never made to fault): while the environment variable MK_FAULT is
 *   "oom"         mk_load_weights, mk_load_synthetic and mk_alloc_kv fail
 *                 with MK_ERR_OOM before they allocate anything;
 *   "bad_arg"     mk_load_weights, mk_decode_step and mk_decode_step_noalloc
 *                 reject their arguments with MK_ERR_INVALID_ARG;
 *   "skip_signal" mk_decode_step launches a step in which no CTA signals
 *                 the completion of layer 0's first projection: the
 *                 stages that read it wait until the wait limit (MK_WAIT_NS)
 *                 and the step reports MK_ERR_TIMEOUT through mk_step_status;
 *   "corrupt_guard" (debug mode, below) mk_step_status overwrites one scratch
 *                 guard before checking them and reports MK_ERR_STATE.
 * Each host failure sets mk_last_error() to a message naming MK_FAULT.
 *
 * Debug mode: with MK_DEBUG=1 when the model is loaded, every CTA writes a
 * 16-byte pattern into the unused end of each shared-memory ring slot and
 * after its input staging area at the start of a step and compares it when
 * it leaves; the producer checks every weight-tile copy against the slot
 * size before issuing it (an oversized one ends the step instead); the
 * expert units check that every entry of their token map is a token of the
 * step; and every scratch region of the model is followed by a 256-byte
 * guard (pattern 0xA5) that mk_step_status compares after the step (and
 * restores). A failed check reports MK_ERR_STATE through mk_step_status
 * (with the place in mk_last_error()); nothing traps. The guards cover the
 * model's own scratch (mk_decode_step, mk_decode_step_unfused), not the
 * static scratch of mk_decode_step_noalloc. While MK_FAULT is
 * "corrupt_guard", mk_step_status overwrites one guard before its check
 * (host injection: the report path without a device fault). */

/* Synchronise `stream` and return the device status of the last step
 * (MK_OK, MK_ERR_TIMEOUT, MK_ERR_INVALID_ARG, or MK_ERR_STATE for a failed
 * debug-mode check). A failed status resets the
 * model's device state so the next step can run.
 * Every wait inside the step (on another CTA's progress or on a copy into
 * shared memory) gives up after the limit set by the environment variable
 * MK_WAIT_NS (nanoseconds, read at mk_load_weights; default 2 s): the step
 * records MK_ERR_TIMEOUT and all CTAs leave, the context stays usable.
 * Testing that path: while the environment variable MK_TEST_STALL is set,
 * mk_decode_step makes CTA 0 first wait on a counter nothing signals. */
int mk_step_status(mk_model* m, void* stream);

/* Routing of the last step, as computed on the device: host arrays
 * idx [L][batch*T][k] (int32, in rank order: largest router logit first),
 * w [L][batch*T][k] (float, renormalised top-k weights) and, when margin_out
 * is not NULL, margin [L][batch*T] (float: the k-th largest router logit
 * minus the (k+1)-th, +inf when k equals the expert count; a parity check
 * accepts a different expert set only where this margin is small).
 * Synchronises `stream`. MoE models only. Errors: STATE when the model has
 * no router, no step ran yet, or the last step ran through
 * mk_decode_step_noalloc (which keeps no routing record). */
int mk_debug_routing(mk_model* m, int32_t* idx_out, float* w_out, float* margin_out, void* stream);

/* Copy `bytes` bytes at `offset` of the model's own per-step scratch
 * allocation (mk_info.scratch_bytes) to host memory `host_out`. A debugging
 * aid: tests use it to check that mk_decode_step_noalloc leaves the model's
 * scratch untouched. Synchronises `stream`. Errors: INVALID_ARG when the
 * range is outside the scratch. */
int mk_debug_scratch_read(mk_model* m, int64_t offset, int64_t bytes, void* host_out, void* stream);

/* Greedy argmax of every logits row of the last step that was given an
 * `accept` buffer (computed by the step itself; ties -> lower token id):
 * `out` int32 [batch*T], host or device memory. A speculative loop takes the
 * token after the accepted prefix of sequence b from row b*T + accept[b] - 1.
 * Synchronises `stream`. Errors: INVALID_ARG (NULL), STATE (the last step had
 * no accept buffer). */
int mk_last_argmax(mk_model* m, int32_t* out, void* stream);

int mk_model_info(const mk_model* m, mk_info* out);

/* Stage trace of the last step, recorded when the environment variable
 * MK_TRACE=1 was set at mk_load_weights. For each CTA (grid_ctas of them)
 * up to 8192 records of 32 bytes: {uint32 code = stage << 16 | layer,
 * uint32 items, int64 t_wait, int64 t_ready, int64 t_end} (device
 * %globaltimer ns: the CTA started waiting for the stage's inputs, they were
 * ready, its items were done). recs_out: host buffer of grid_ctas*8192*32
 * bytes; counts_out: host int32 [grid_ctas] records written. Synchronises
 * `stream`. Errors: STATE when tracing is off. */
int mk_trace_read(mk_model* m, void* recs_out, int64_t bytes, int32_t* counts_out, void* stream);

/* Free a model or a KV cache (NULL is a no-op). Either may be freed first:
 * a model freed while KV caches of it are alive releases its device memory
 * at once and rejects every later call; its caches keep their own memory
 * (mk_kv_read, mk_kv_write and mk_free still work on them) and the model's
 * small host record, which they read for its dimensions, is deleted with
 * the last of them. */
void mk_free(void* handle);

const char* mk_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
