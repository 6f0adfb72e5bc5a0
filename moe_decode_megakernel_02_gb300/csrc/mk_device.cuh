// mk_device.cuh -- the persistent decode megakernel (sm_103a).
//
// One cooperative launch, one CTA per SM. Each CTA = 8 consumer warps + 1
// producer warp. The whole step (all layers, the LM head, verify acceptance)
// is a fixed program of stages; the work items of every stage are spread
// over the CTAs. Every CTA's producer warp walks the same program as its
// consumers and streams each weight tile / KV chunk its consumers will need
// into a shared-memory ring of NSLOT slots (3 by default) with TMA bulk copies
// (cp.async.bulk + mbarrier complete_tx). Weight tiles depend on no
// activation, so the producer runs ahead across stage and layer boundaries
// while the consumers wait for their inputs: this is the GPU form of the
// cross-layer weight prefetch ("TPU Megakernel Achieves 709 tokens/s on Kimi
// K3", section "Cross-Layer Weight Prefetching"; myzaker article: layer N+1's
// attention weights move while layer N computes its MoE). The only tiles that
// must wait are the routed experts', which are known once the router is done.
//
// Dependencies between stages are release/acquire counters in global memory
// (one per layer and stage, double-buffered by step parity); every wait gives
// up after a time limit, records MK_ERR_TIMEOUT and makes every CTA leave.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace mk {

// ---------------------------------------------------------------- shape ----
constexpr int NCW = 8;                    // consumer warps
constexpr int NCT = NCW * 32;             // consumer threads
constexpr int NTHREADS = NCT + 32;        // + one producer warp
// three ring slots: shared memory stays under the 196 KB carveout, which
// leaves L1 60 KB instead of 28 KB for the stack of the stage functions
// (measured: the one-token step 2 % faster than with four slots)
#ifndef MK_NSLOT
#define MK_NSLOT 3
#endif
#ifndef MK_STAGE_BYTES
#define MK_STAGE_BYTES 66048
#endif
constexpr int NSLOT = MK_NSLOT;           // ring slots
constexpr int SLOT_BYTES = 37888;         // one MLA chunk (32 padded latent rows + rope rows)
constexpr int TILE_MAX = 32768;           // GEMV weight tile
constexpr int STAGE_BYTES = MK_STAGE_BYTES;  // activation / query staging
constexpr int STAGE_FLOATS = STAGE_BYTES / 4;
// staged input rows are Kc + 8 floats apart: a tensor-core fragment load
// (8 token rows, 2 floats each) then touches every bank once per half warp
__host__ __device__ constexpr int stage_stride(int Kc) { return Kc + 8; }
__host__ __device__ constexpr bool stage_fits(int M, int Kc) { return M * stage_stride(Kc) <= STAGE_FLOATS; }
constexpr int RED_FLOATS = 1024;
constexpr int MT = 4;                     // tokens per register group in the GEMV
constexpr int MAX_M = 64;                 // batch * tokens per step
constexpr int MAX_E = 256;
// router logits accumulated by the output projection's CTAs go to one of
// ROUTER_COPIES copies (by CTA), so that few CTAs add into the same lines;
// a token's row holds E logits and the sum of squares, padded to 4 floats
constexpr int ROUTER_COPIES = 8;
__host__ __device__ constexpr int router_row(int E) { return (E + 4) & ~3; }
constexpr int MAX_K = 8;
constexpr int GQA_CH = 64;                // positions per GQA chunk (= one page)
constexpr int MLA_CH = 32;                // positions per MLA chunk (half a page)
constexpr int PAGE = 64;
// MLA: 16 heads, latent 512, rope 64 (checked on the host)
constexpr int MLA_H = 16, MLA_KL = 512, MLA_RD = 64, MLA_D = MLA_KL + MLA_RD;
constexpr int MLA_QS = 584;               // padded smem row stride of the queries (bf16 elements)
// an MLA chunk in shared memory: 9 boxes of MLA_CH positions x 64 bf16 (128
// bytes a row) -- the latent's 8 column blocks, then the rope -- each in the
// 128-byte swizzled order of the bulk tensor copy that fills it (the 16-byte
// piece j of a row sits at piece j ^ bits 7..9 of the row's address)
constexpr int MLA_BOX = MLA_CH * 128;
constexpr int MLA_TILE_BYTES = 9 * MLA_BOX;
static_assert(MLA_TILE_BYTES <= SLOT_BYTES - 16, "MLA chunk must fit a slot (and leave its debug canary alone)");
static_assert(64 * (256 * 2 + 16) <= SLOT_BYTES - 16 && 16 * (1024 * 2 + 16) <= SLOT_BYTES - 16 &&
                  8 * (2048 * 2 + 16) <= SLOT_BYTES - 16,
              "padded tensor-core tiles leave the slot's debug canary alone");
static_assert(SLOT_BYTES % 1024 == 0, "ring slots keep the 1024-byte alignment of the swizzled boxes");

enum InKind { IN_COPY = 0, IN_RMS = 1, IN_SWIGLU = 2 };
// OUT_ACC: += into a CTA-private buffer; OUT_ADD: every warp adds its share
// (a K slice) atomically into a zeroed CTA-private buffer, no barrier per tile
enum OutKind { OUT_STORE = 0, OUT_RESID = 1, OUT_SCALED = 2, OUT_ACC = 3, OUT_ADD = 4 };
enum StatusCode { ST_OK = 0, ST_INVALID = 1, ST_TIMEOUT = 5, ST_DEBUG = 6 };

// A matrix-vector stage: out[m][row] (+)= W[row, :] . f(in)[m, :]
// W is packed [n_kc][N][Kc] (K-panels; n_kc == 1 is plain row-major).
struct Gemv {
    const uint16_t* W;
    long long w_estride;          // elements between routed experts
    int N, K, Kc, R, n_kc, n_rb;  // rows, reduction length, panel width, rows per tile
    int in_kind;
    const float* src;             // input rows [M][src_stride]
    int src_stride;
    long long src_sstride;        // per routed slot (gate/up output of the slot)
    const uint16_t* gain;         // IN_RMS gain [K]
    int grp_rows, grp_stride;     // grouped input: rows [i*grp_rows, ...) read src + i*grp_stride
    int sw_off;                   // IN_SWIGLU: up values at +sw_off
    int out_kind;
    float* dst;
    int dst_stride;
    long long dst_sstride;        // per routed slot
    float* dst2;                  // OUT_RESID: next layer's residual
};

enum { G_A = 0, G_QB, G_QLAT, G_UV, G_O, G_ROUTER, NG };

// SwiGLU experts as units: unit u of an expert owns F of its Fi intermediate
// dimensions. Its gate and up rows (2F rows of the gate/up matrix, whose rows
// are stored unit-major: gate rows then up rows of unit 0, of unit 1, ...)
// and its F columns of the down matrix (stored per unit as [d][F]) are all a
// CTA needs to add the unit's share of the expert output to the residual:
// no exchange between CTAs inside the FFN.
struct FfnKind {
    const uint16_t* gu;       // [n_kc][2*Fi][Kc], rows unit-major (bf16 experts)
    const uint16_t* dn;       // [nu][d][F] (bf16 experts)
    long long gu_es, dn_es;   // elements between routed experts
    int Fi, F, nu;            // intermediate width, unit width, units per expert
    int R, Rd;                // gate/up rows per tile, down rows per tile
    // MXFP8 experts (gu, dn null): tiles of E4M3 codes, each followed by its
    // rows' E8M0 block scales (one per 32 codes of a row)
    const uint8_t* qgu;       // [2Fi/R] tiles: R rows x Kc codes, then R x Kc/32 scales (rows unit-major)
    const uint8_t* qdn;       // [nu][d/Rd] tiles: Rd rows x F codes, then Rd x F/32 scales
    long long qgu_es, qdn_es; // bytes between routed experts
    int qtb_gu, qtb_dn;       // bytes per gate/up tile, per down tile
};
struct Ffn {
    FfnKind k[2];             // [0] routed experts, [1] shared expert
    int Kc, n_kc;             // gate/up K panel
    const uint16_t* gain;     // FFN RMSNorm gain
};

struct Layer {
    Gemv g[NG];
    Ffn ffn;
    const uint16_t* kv_norm;  // MLA latent RMSNorm gain
    const uint16_t* uk;       // MLA: W_uk per head [H][nope][kl] (the absorbed query folded into QB)
    const uint16_t* uvq;      // MLA: W_uv per head and latent quarter [H][4][vd][kl/4] (UV folded into COMB)
    const float* a;           // GQA: q|k|v   MLA: c_q | latent | k_rope   [M][a_stride]
    const float* q;           // MLA: q_b output [M][H*(nope+rope)]
    const float* qlat;        // MLA: absorbed queries [M][H*kl]
    float* olat;              // MLA: combined latent attention output [M][H*kl]
    float* o;                 // attention output [M][Hq*hd | H*vd]
    float* rlog;              // router stage output: logits [M][router_row(E)]
    float* x;                 // residual entering the layer [M][d]
    float* xn;                // residual leaving the layer [M][d]
    int a_stride;
};

// counters per layer (and one extra "layer" L for the head)
enum { C_A = 0, C_QB, C_APP, C_QLAT, C_ATTN, C_COMB, C_UV, C_O, C_ROUTER, C_SHGU, C_CARRY, C_SHDOWN, C_DOWN,
       C_INIT, C_LM, C_AMAX, C_NRM0, C_NRM1, C_NRM2, C_GU0, NCTR = C_GU0 + MAX_E };

struct Params {
    int L, d, V, attn, Hq, Hkv, hd, ql, kl, nope, rd, vd, E, topk, has_sh, ffn, sffn;
    float eps, attn_scale;
    int G;                          // CTAs in the grid
    const Layer* layers;
    Gemv lm;
    const uint16_t* embed;
    const float2* rope;             // [npos][rope_half] (cos, sin)
    int rope_half, rope_npos;
    uint16_t* kv_pool;              // [L][pages][page_elems]
    long long kv_layer_elems;
    long long page_elems;           // elements of one page (per layer pool)
    int pps;                        // pages per sequence
    const int* btab;                // [kv_batch][pps]
    int kv_cap, kv_batch;           // positions per sequence, sequences in the cache
    const uint16_t* zeros;          // >= 2 KB of zero bytes
    // MLA caches: two tensor maps (CUtensorMap, 128 bytes each) in device
    // memory -- the latent [L][pages][64 rows][512] and the rope [L][pages]
    // [64 rows][64] of the pool, boxes of 32 rows x 64 bf16, 128-byte swizzle
    const void* kv_tmaps;
    uint16_t* newlat;               // MLA new latents [MAX_M][576] bf16
    float* part;                    // attention partials: unnormalised O rows
    float* part_ml;                 // attention partials: (running max, sum) per row
    int s_max;
    const int* tokens;
    const int* pos;
    int B, T, M;
    float* logits;
    int* accept;
    int* amax;
    float* zptr[10];
    long long zn[10];               // floats to zero at the start of the step
    int nz, carry;                  // carry: residual copied by items (split-K output projection)
    int gs, gr;                     // CTAs [0, gs): shared expert, [gs, G): routed experts ([G-gr, G) first run the router)
    int stall;                      // testing: CTA 0 first waits on a counter nothing signals (ends in a timeout)
    int skip_sig;                   // testing: 1 + the stage whose layer-0 signals the CTAs leave out (0: none)
    int debug;                      // shared-memory canaries and token-map checks (ST_DEBUG on a failure)
    int f8;                         // MXFP8 expert weights
    // one launch per stage (the unfused comparison path): 0 = the whole step
    // in this launch; 1 = program positions [st_lo, st_hi) only, 2 = the
    // step's set-up only (embedding, buffers zeroed). Launches are ordered by
    // the stream, so no dependency counter is waited on or signalled.
    int staged, st_lo, st_hi;
    int rfuse;                      // router logits accumulated by the output projection's CTAs (no router stage)
    int qfuse;                      // MLA: the absorbed query computed by the QB CTAs (no QLAT stage)
    int ufuse;                      // MLA: the value up-projection computed by the combine CTAs (no UV stage)
    float* racc;                    // their accumulators [L][ROUTER_COPIES][M][router_row(E)], zero at step start
    // sums of squares of the rows of RMSNorm inputs whose K panels are parts
    // of the row, summed once per stage by its CTAs (several tokens):
    // [L + 1][3 sites: A or LM, QB, router][rss_mx], zero at step start
    float* rss;
    int rss_mx;
    float* ubuf;                    // per CTA: expert-unit gate/up and hidden values when shared memory is short
    long long ubuf_stride;          // floats per CTA
    unsigned* ctr;                  // [2][L+1][NCTR]
    int parity;
    unsigned* status;               // [0] code [1] abort [2] where [3] cta
    long long timeout_ns;
    int* dbg_idx;                   // routing of the step (written by CTA 0): [L][M][k]
    float* dbg_w;
    float* dbg_margin;              // [L][M]: k-th minus (k+1)-th router logit (+inf when k = E)
    struct TraceRec* trace;         // optional stage trace [G][trace_cap]
    unsigned* trace_n;              // records written per CTA
    int trace_cap;
    int trace_items;                // also one record per GEMV work item
};

// one traced stage of one CTA (consumer side): when the CTA started waiting
// for the stage's inputs, when they were ready, when its items were done
struct TraceRec {
    unsigned code;  // stage << 16 | layer
    unsigned n;     // items this CTA processed
    long long t_wait, t_ready, t_end;
};

// ----------------------------------------------------------- smem layout ----
// one dependency of a stage: wait until counter (layer, which) >= target
struct Dep {
    int layer, which;
    unsigned target;
};

struct Misc {
    unsigned long long full[NSLOT];
    unsigned long long empty[NSLOT];
    Dep dep[3];                     // the next consumer wait (written and read by thread 0)
    int ndep;
    Gemv ug, pug;                   // expert-unit gate/up GEMV (consumers, producer)
    float uw[MAX_M];                // expert-unit routing weight per token
    // tokens of the current GEMV: gm of them, token i staged at row gt[i] of
    // the staging area (all tokens in order, except in a routed expert's
    // units, which take only the tokens routed to the expert)
    uint8_t gt[MAX_M];
    int gm;
    // 0: staging row = token id (all tokens staged, or a consecutive range);
    // otherwise a key of the token map (routed expert + 1, or 1024 + first
    // token of a shared-expert token group) and staging row i holds the
    // map's token gt[m0 + i] (the map's tokens gathered, m0 the first staged)
    int gather;
    long long tdbg[4];              // trace: clock64 marks of the expert-unit gate/up GEMV
    int abort;
    int n_slots, p_nslots;
    float rms[MAX_M];
    uint8_t slot_e[MAX_E];          // consumer: routed slot -> expert
    uint8_t p_slot_e[MAX_E];        // producer copy
    alignas(4) uint8_t used[MAX_E];    // tokens routed to each expert (consumers)
    alignas(4) uint8_t p_used[MAX_E];  // producer copy
    uint8_t ridx[MAX_M][MAX_K];
    float rw[MAX_M][MAX_K];
    float cw[256];                  // combine weights
    float bred[NCW];                // block reductions
};
constexpr int SMEM_RING = 0;
constexpr int SMEM_STAGE = NSLOT * SLOT_BYTES;
// 16 bytes between the staging area and the reduction area: a canary in
// debug mode (checked when the CTA leaves)
constexpr int SMEM_CANARY = SMEM_STAGE + STAGE_BYTES;
constexpr int SMEM_RED = SMEM_CANARY + 16;
constexpr int SMEM_MISC = SMEM_RED + RED_FLOATS * 4;
constexpr int SMEM_CTX = (SMEM_MISC + (int)sizeof(Misc) + 15) & ~15;
constexpr int CTX_BYTES = 160;  // per warp (checked against sizeof(Ctx))
// the current layer's descriptors, one copy for the consumers and one for
// the producer warp (they can be in different layers): gpu-scope acquires
// invalidate the L1, so descriptors read from global memory would cost an
// L2 round trip at every use
constexpr int LAYER_BYTES = ((int)sizeof(Layer) + 15) & ~15;
constexpr int SMEM_LAYER = SMEM_CTX + (NCW + 1) * CTX_BYTES;
constexpr int SMEM_PLAYER = SMEM_LAYER + LAYER_BYTES;
// a copy of the kernel parameters: read through a reference, the parameter
// block would be fetched like global data, again after every acquire
constexpr int SMEM_PARAMS = SMEM_PLAYER + LAYER_BYTES;
constexpr int SMEM_TOTAL = SMEM_PARAMS + (((int)sizeof(Params) + 15) & ~15);
static_assert(SMEM_TOTAL <= 232448, "shared memory per CTA exceeds 227 KB");

// ------------------------------------------------------------------ PTX ----
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ long long gtimer() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_release(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void mbar_init(unsigned long long* b, unsigned n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned long long* b, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// streamed data (weights, cached KV) is read once per step: load it with an
// evict-first L2 policy so it does not push code and activations out of L2
__device__ __forceinline__ unsigned long long l2_evict_first() {
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void bulk_g2s_pol(void* dst, const void* src, unsigned bytes, unsigned long long* bar,
                                             unsigned long long pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar)), "l"(pol)
        : "memory");
}
// start moving [src, src+bytes) from HBM into L2 (no completion to wait for):
// the smem ring holds only a few tiles per SM, too few bytes in flight to
// cover HBM latency under load; tiles prefetched into L2 further ahead fill
// the ring at L2 latency instead
__device__ __forceinline__ void l2_prefetch(const void* src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// the same with an evict-last policy: small vectors every step re-reads
// (norm gains, layer descriptors) stay in L2 while the weights stream past
__device__ __forceinline__ void l2_prefetch_keep(const void* src, unsigned bytes) {
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, unsigned long long* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar)), "l"(l2_evict_first())
        : "memory");
}
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory"); }

// 16 bytes from global memory (through L2, not L1: the data may have been
// written by other SMs moments ago) into shared memory, asynchronously; a
// thread issues all its pieces, then waits for them once
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// one box of a 4-D tensor map into shared memory, completing on `bar`
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int x, int y, int z, int w,
                                            unsigned long long* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(su32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(su32(bar))
        : "memory");
}
// the byte of the 16-byte piece holding bf16 element (row, k) of an MLA
// chunk whose boxes start at `base`, `bb` bytes apart (swizzled as above)
__device__ __forceinline__ const uint8_t* mla_piece(const uint8_t* base, int bb, int row, int k) {
    const uint8_t* r = base + (k >> 6) * bb + row * 128;
    return r + ((((unsigned)k >> 3 & 7u) ^ (su32(r) >> 7 & 7u)) << 4);
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(su32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(su32(p)));
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------- status ----
__device__ __noinline__ void raise_status(const Params& p, unsigned code, unsigned where) {
    if (atomicCAS(&p.status[0], 0u, code) == 0u) {
        p.status[2] = where;
        p.status[3] = blockIdx.x;
    }
    atomicExch(&p.status[1], 1u);
    __threadfence();
}

// one thread: wait until *c >= target (acquire); false on abort / timeout
// (polls with relaxed loads: every gpu-scope acquire invalidates the SM's L1;
// the fence after the last poll completes the acquire pattern)
__device__ __noinline__ bool wait_ge(const Params& p, const unsigned* c, unsigned target, unsigned where) {
    if (p.staged) return true;  // the inputs were written by earlier launches
    if (ld_relaxed(c) >= target) {
        fence_acq_rel();
        return true;
    }
    const long long t0 = gtimer();
    for (unsigned it = 0;; ++it) {
        if (ld_relaxed(c) >= target) {
            fence_acq_rel();
            return true;
        }
        if ((it & 31) == 31) {
            if (ld_relaxed(&p.status[1])) return false;
            if (gtimer() - t0 > p.timeout_ns) {
                raise_status(p, ST_TIMEOUT, where);
                return false;
            }
        }
    }
}

// a lane: wait for mbarrier phase `parity`; false on abort / timeout
__device__ __noinline__ bool mbar_wait(const Params& p, unsigned long long* b, unsigned parity, unsigned where) {
    if (mbar_test(b, parity)) return true;
    const long long t0 = gtimer();
    for (unsigned it = 0;; ++it) {
        if (mbar_test(b, parity)) return true;
        if ((it & 15) == 15) {
            if (ld_relaxed(&p.status[1])) return false;
            if (gtimer() - t0 > p.timeout_ns) {
                raise_status(p, ST_TIMEOUT, where);
                return false;
            }
        }
    }
}

__device__ __forceinline__ unsigned* ctr_of(const Params& p, int layer, int which) {
    return p.ctr + ((size_t)p.parity * (p.L + 1) + layer) * NCTR + which;
}

// ------------------------------------------------------------ schedule ----
// items [lo, hi) of a stage with n items for this CTA; `off` rotates which
// CTAs take the extra items from stage to stage.
__device__ __forceinline__ void my_range(const Params& p, int n, int off, int& lo, int& hi) {
    int v = (int)blockIdx.x + off;
    if (v >= p.G) v -= p.G;
    // 32-bit products (G <= 255 CTAs, n < 2^23 items): 64-bit division is a long software sequence
    lo = v * n / p.G;
    hi = (v + 1) * n / p.G;
}

// n items over the CTAs [c0, c0 + gc) only (empty range for the others)
__device__ __forceinline__ void my_range_sub(int n, int c0, int gc, int& lo, int& hi) {
    const int v = (int)blockIdx.x - c0;
    if (v < 0 || v >= gc) {
        lo = hi = 0;
        return;
    }
    lo = v * n / gc;
    hi = (v + 1) * n / gc;
}

__device__ __forceinline__ int gemv_items(const Gemv& g) { return g.n_rb * g.n_kc; }

// tokens per work item of the shared expert (M tokens, FFN input in n_kc K
// panels of Kc): 4 when every token's input fits the staging area at once,
// as many as fit when it does not (each group gathered), else all
__host__ __device__ __forceinline__ int shared_group(int M, int n_kc, int Kc) {
    if (M <= 1 || n_kc != 1) return M < 1 ? 1 : M;
    if (stage_fits(M, Kc)) return M > 4 ? 4 : M;
    return STAGE_FLOATS / stage_stride(Kc);
}

// attention splits: units = prefix chunks + 1 tail unit (the new positions)
__device__ __forceinline__ int gqa_target(const Params& p) {
    int t = p.G / (p.B * p.Hkv);
    return t < 1 ? 1 : t;
}
__device__ __forceinline__ int mla_target(const Params& p) {
    // splits per query row: one item per CTA; when that leaves CTAs idle
    // (B T does not divide the grid well), about three items per CTA
    const int rows = p.B * p.T;
    int t = p.G / rows;
    if (t < 4 && t * rows < p.G - p.G / 8) t = (3 * p.G) / rows;
    t = t > p.s_max ? p.s_max : t;
    return t < 1 ? 1 : t;
}
__device__ __forceinline__ int nch_of(const Params& p, int b, int ch) { return (p.pos[b] + ch - 1) / ch; }

__device__ int attn_items(const Params& p) {
    int n = 0;
    if (p.attn == 0) {
        const int tg = gqa_target(p);
        for (int b = 0; b < p.B; ++b) {
            int u = nch_of(p, b, GQA_CH) + 1;
            n += p.Hkv * (u < tg ? u : tg);
        }
    } else {
        const int tg = mla_target(p);
        for (int b = 0; b < p.B; ++b) {
            int u = nch_of(p, b, MLA_CH) + 1;
            n += p.T * (u < tg ? u : tg);
        }
    }
    return n;
}

struct AttnItem {
    int b, g, s, S, u_lo, u_hi, nch;
};
// decode item index -> (sequence, head group or token, split, unit range)
__device__ AttnItem attn_item(const Params& p, int i) {
    AttnItem it;
    const bool gqa = p.attn == 0;
    const int tg = gqa ? gqa_target(p) : mla_target(p);
    const int per = gqa ? p.Hkv : p.T;
    const int ch = gqa ? GQA_CH : MLA_CH;
    for (int b = 0; b < p.B; ++b) {
        int nch = nch_of(p, b, ch);
        int u = nch + 1;
        int S = u < tg ? u : tg;
        if (i < per * S) {
            it.b = b;
            it.g = i / S;
            it.s = i % S;
            it.S = S;
            it.nch = nch;
            it.u_lo = (int)((long long)it.s * u / S);
            it.u_hi = (int)((long long)(it.s + 1) * u / S);
            return it;
        }
        i -= per * S;
    }
    it.b = it.g = it.s = it.S = it.u_lo = it.u_hi = it.nch = 0;
    return it;
}

__device__ __forceinline__ const uint16_t* page_ptr(const Params& p, const uint16_t* pool, int b, int page_idx) {
    return pool + (size_t)p.btab[b * p.pps + page_idx] * p.page_elems;
}

// --------------------------------------------------------- producer ring ----
struct PRing {
    unsigned slot, phase;
};

// lane 0 acquires the next slot (waits for the consumers to free it) and
// announces `bytes`; returns the slot pointer (lane 0 only), or nullptr on abort
__device__ __forceinline__ uint8_t* prod_begin(const Params& p, uint8_t* smem, Misc& ms, PRing& r, unsigned bytes) {
    if (!mbar_wait(p, &ms.empty[r.slot], r.phase ^ 1u, 0x100u)) return nullptr;
    mbar_expect_tx(&ms.full[r.slot], bytes);
    return smem + SMEM_RING + r.slot * SLOT_BYTES;
}
// ring states are shared by the lanes of a warp (they live in shared memory):
// every lane reads the old value before any lane writes the new one
__device__ __forceinline__ void prod_next(PRing& r) {
    PRing n = r;
    if (++n.slot == NSLOT) {
        n.slot = 0;
        n.phase ^= 1u;
    }
    __syncwarp();
    r = n;
    __syncwarp();
}

// consumer ring state (identical in every consumer thread)
struct CRing {
    unsigned slot, phase;
};
__device__ __forceinline__ const uint8_t* cons_wait(const Params& p, uint8_t* smem, Misc& ms, CRing& r) {
    if (mbar_test(&ms.full[r.slot], r.phase)) return smem + SMEM_RING + r.slot * SLOT_BYTES;  // fast path
    if (!mbar_wait(p, &ms.full[r.slot], r.phase, 0x200u)) {
        ms.abort = 1;
        return nullptr;
    }
    return smem + SMEM_RING + r.slot * SLOT_BYTES;
}
__device__ __forceinline__ void cons_release(Misc& ms, CRing& r) {
    CRing n = r;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ms.empty[n.slot]);
    if (++n.slot == NSLOT) {
        n.slot = 0;
        n.phase ^= 1u;
    }
    __syncwarp();
    r = n;
    __syncwarp();
}

}  // namespace mk
