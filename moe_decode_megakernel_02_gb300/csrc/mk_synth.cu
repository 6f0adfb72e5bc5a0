// mk_synth.cu -- mk_load_synthetic: a model of seeded synthetic weights,
// generated directly in device memory and loaded through mk_load_weights.
//
// The numbers come from the input generator module (synth/: the SplitMix64
// counter hash and Irwin-Hall(12) normal draws of the input recipe, linked
// into this library as it is -- it holds no model arithmetic). Weight kinds
// and their numbering are the same in both (mk_weight_kind == synth_kind).
#include <cuda_runtime.h>

#include <cstdio>
#include <vector>

#include "../../include/mk.h"
#include "../../synth/synth.h"

extern "C" int synth_fill_bf16_cuda(uint16_t* dev_out, uint64_t n, uint64_t seed, uint64_t tensor_id, float sigma,
                                    float mean, uint64_t index0, void* stream);
extern "C" int synth_fill_e4m3_cuda(uint8_t* dev_out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t index0,
                                    void* stream);
extern "C" int synth_fill_e8m0_cuda(uint8_t* dev_out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t index0,
                                    void* stream);

// the message of a failure found here goes through the same thread-local
// slot as the rest of the library's (mk_set_error_, defined in mk_host.cu)
extern "C" __attribute__((visibility("hidden"))) int mk_set_error_(int code, const char* msg);
// MK_ERR_OOM while MK_FAULT=oom (host-side fault injection), else MK_OK
extern "C" __attribute__((visibility("hidden"))) int mk_fault_oom_(void);

namespace {

// what a tensor holds: bf16 draws, E4M3 codes or E8M0 scale bytes
enum Fill { FILL_BF16, FILL_E4M3, FILL_E8M0 };

struct Spec {
    int kind, layer, expert;
    size_t elems, off;  // elements, byte offset
    float sigma, mean;
    Fill fill;
};

}  // namespace

extern "C" int mk_load_synthetic(const mk_config* cfg, uint64_t seed, void* stream, mk_model** out) {
    if (!out) return mk_set_error_(MK_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!cfg) return mk_set_error_(MK_ERR_INVALID_ARG, "cfg is NULL");
    if (cfg->n_layers < 1 || cfg->d_model < 1 || cfg->vocab < 1 || cfg->n_routed_experts < 0)
        return mk_set_error_(MK_ERR_INVALID_ARG, "non-positive dimension");
    if (const int rc = mk_fault_oom_()) return rc;
    const synth_dims d = {cfg->n_layers, cfg->d_model, cfg->vocab, cfg->attn_kind, cfg->n_q_heads,
                          cfg->n_kv_heads, cfg->head_dim, cfg->q_lora_rank, cfg->kv_lora_rank, cfg->qk_nope_dim,
                          cfg->qk_rope_dim, cfg->v_head_dim, cfg->n_routed_experts, cfg->top_k,
                          cfg->n_shared_experts, cfg->ffn_dim, cfg->shared_ffn_dim};
    // every tensor the recipe defines for these dimensions, 256-byte aligned
    // in one device buffer
    // (MXFP8 experts: the expert kinds are E4M3 codes, one byte each, and
    // their scale kinds E8M0 bytes)
    const bool f8 = cfg->expert_format == MK_EXPERT_MXFP8;
    auto is_expert = [](int k) {
        return k == SYNTH_GATE || k == SYNTH_UP || k == SYNTH_DOWN || k == SYNTH_SH_GATE || k == SYNTH_SH_UP ||
               k == SYNTH_SH_DOWN;
    };
    std::vector<Spec> specs;
    size_t total = 0;
    auto add = [&](int kind, int layer, int expert) {
        int32_t r = 0, c = 0;
        float sg = 0.f, mn = 0.f;
        if (synth_weight_spec(&d, kind, &r, &c, &sg, &mn) != 0) return;
        const size_t n = (size_t)r * c;
        const Fill f = !f8 ? FILL_BF16 : is_expert(kind) ? FILL_E4M3 : is_expert(kind - 6) ? FILL_E8M0 : FILL_BF16;
        specs.push_back({kind, layer, expert, n, total, sg, mn, f});
        total += (n * (f == FILL_BF16 ? 2 : 1) + 255) / 256 * 256;
    };
    auto add_expert = [&](int kind, int layer, int expert) {
        add(kind, layer, expert);
        if (f8) add(kind + 6, layer, expert);
    };
    for (int k : {SYNTH_EMBED, SYNTH_LM_HEAD, SYNTH_FINAL_NORM}) add(k, -1, 0);
    for (int l = 0; l < cfg->n_layers; ++l) {
        for (int k : {SYNTH_ATTN_NORM, SYNTH_FFN_NORM, SYNTH_WQ, SYNTH_WK, SYNTH_WV, SYNTH_WO, SYNTH_WDQ, SYNTH_Q_NORM,
                      SYNTH_WUQ, SYNTH_WDKV, SYNTH_KV_NORM, SYNTH_WUKV, SYNTH_ROUTER})
            add(k, l, 0);
        for (int k : {SYNTH_SH_GATE, SYNTH_SH_UP, SYNTH_SH_DOWN}) add_expert(k, l, 0);
        for (int e = 0; e < cfg->n_routed_experts; ++e)
            for (int k : {SYNTH_GATE, SYNTH_UP, SYNTH_DOWN}) add_expert(k, l, e);
    }
    uint8_t* buf = nullptr;
    if (cudaMalloc(&buf, total) != cudaSuccess) {
        cudaGetLastError();
        char msg[128];
        snprintf(msg, sizeof msg, "synthetic weights: cudaMalloc(%zu) failed", total);
        return mk_set_error_(MK_ERR_OOM, msg);
    }
    std::vector<mk_weight> table;
    table.reserve(specs.size());
    for (const Spec& s : specs) {
        const uint64_t tid = synth_tensor_id(s.kind, s.layer, s.expert);
        const int rc = s.fill == FILL_BF16
                           ? synth_fill_bf16_cuda(reinterpret_cast<uint16_t*>(buf + s.off), s.elems, seed, tid, s.sigma,
                                                  s.mean, 0, stream)
                       : s.fill == FILL_E4M3 ? synth_fill_e4m3_cuda(buf + s.off, s.elems, seed, tid, 0, stream)
                                             : synth_fill_e8m0_cuda(buf + s.off, s.elems, seed, tid, 0, stream);
        if (rc != 0) {
            cudaStreamSynchronize((cudaStream_t)stream);
            cudaFree(buf);
            return mk_set_error_(MK_ERR_CUDA, "synthetic weights: generator launch failed");
        }
        table.push_back(mk_weight{s.kind, s.layer, s.expert, 0, buf + s.off});
    }
    // mk_load_weights synchronises the stream before it returns, after its
    // last read of `buf`
    const int rc = mk_load_weights(cfg, table.data(), (int32_t)table.size(), stream, out);
    cudaStreamSynchronize((cudaStream_t)stream);
    cudaFree(buf);
    return rc;
}
