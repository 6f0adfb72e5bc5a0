// mk_kernel.cuh -- stage program of the decode megakernel (producer + consumers).
#pragma once
#include <new>

#include "mk_device.cuh"

namespace mk {

struct Deps {
    Dep d[3];
    int n;
};
__device__ __forceinline__ Deps deps0() {
    Deps d;
    d.n = 0;
    return d;
}
__device__ __forceinline__ Deps deps1(int l, int w, unsigned t) {
    Deps d;
    d.n = 1;
    d.d[0] = {l, w, t};
    return d;
}

// per-thread view of the run (consumer threads and the producer warp each
// keep an identical copy of the schedule state)
struct alignas(16) Ctx {
    const Params& p;
    uint8_t* smem;
    Misc& ms;
    int off;
    bool dead;
    CRing cr;
    PRing pr;
    // what the staging buffer currently holds
    const void* sk_src;
    const void* sk_gain;
    const void* rms_src;  // c.ms.rms holds the whole rows' sums of squares of this input
    int st_rank, st_np;   // plain GEMV stage: this CTA's rank among the np CTAs that have items
    int sk_off, sk_kc, sk_m0, sk_kind, sk_gather;
    int issued;  // producer: ring fills issued
    long long t_start;
    unsigned cur_code;  // trace: stage being run
    int pl, pst;                     // program position: layer, stage
    int n_down, n_shdown, n_carry;   // items the current layer's last stages signal
    __device__ Ctx(const Params& pp, uint8_t* s)
        : p(pp), smem(s), ms(*reinterpret_cast<Misc*>(s + SMEM_MISC)), off(0), dead(false) {
        cr.slot = 0;
        cr.phase = 0;
        pr.slot = 0;
        pr.phase = 0;
        sk_src = nullptr;
        sk_gain = nullptr;
        rms_src = nullptr;
        sk_off = sk_kc = sk_m0 = sk_kind = sk_gather = -1;
        issued = 0;
        pl = pst = 0;
        n_down = n_shdown = n_carry = 0;
        t_start = gtimer();
        if (pp.trace && threadIdx.x == 0) pp.trace_n[blockIdx.x] = 0;
    }
    __device__ float* stage() { return reinterpret_cast<float*>(smem + SMEM_STAGE); }
    __device__ float* red() { return reinterpret_cast<float*>(smem + SMEM_RED); }
    // this thread's side's copy of the current layer's descriptors
    __device__ const Layer& layer() const {
        return *reinterpret_cast<const Layer*>(smem + (threadIdx.x >= NCT ? SMEM_PLAYER : SMEM_LAYER));
    }
    __device__ void advance(int n) {
        const int o = (int)((off + (long long)n) % p.G);
        __syncwarp();
        off = o;
        __syncwarp();
    }
    __device__ void bump_issued() {
        const int v = issued + 1;
        __syncwarp();
        issued = v;
        __syncwarp();
    }
    __device__ void set_ring(const CRing& v) {
        __syncwarp();
        cr = v;
        __syncwarp();
    }
    __device__ void set_pos(int l, int st) {
        __syncwarp();
        pl = l;
        pst = st;
        __syncwarp();
    }
    __device__ void set_count(int& field, int v) {
        __syncwarp();
        field = v;
        __syncwarp();
    }
    __device__ void set_pring(const PRing& v, int iss) {
        __syncwarp();
        pr = v;
        issued = iss;
        __syncwarp();
    }
};

static_assert(sizeof(Ctx) <= CTX_BYTES, "Ctx must fit its shared-memory slot");

__device__ __forceinline__ int ctid() { return threadIdx.x; }

// consumer: the stage's dependencies travel through shared memory (thread 0
// writes them, thread 0 waits on them): stage functions are not inlined and
// a struct passed by reference would live in each thread's stack
__device__ __forceinline__ void set_deps(Ctx& c, const Deps& ds) {
    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i)
            if (i < ds.n) c.ms.dep[i] = ds.d[i];
        c.ms.ndep = ds.n;
    }
}

// consumer: thread 0 waits for the deps set by set_deps(), then every
// consumer thread passes a barrier (so their later reads of other CTAs' data
// are ordered after it)
__device__ bool cwait(Ctx& c, unsigned where) {
    if (threadIdx.x == 0 && !c.dead) {
        bool ok = true;
        const int n = c.ms.ndep;
        for (int i = 0; i < n && ok; ++i) {
            const Dep d = c.ms.dep[i];
            if (d.target > 0) ok = wait_ge(c.p, ctr_of(c.p, d.layer, d.which), d.target, where);
        }
        if (!ok) c.ms.abort = 1;
    }
    cbar();
    if (*(volatile int*)&c.ms.abort) c.dead = true;
    return !c.dead;
}

// consumer: all consumer threads' global writes done -> release `n` to a
// counter (the barrier orders the other threads' writes before thread 0's
// release, which is cumulative over them)
__device__ void csignal(Ctx& c, int layer, int which, unsigned n) {
    cbar();
    // (MK_FAULT=skip_signal: the CTAs leave out their releases of one stage
    // of layer 0, so that stage's readers run into their wait limit)
    const bool skip = c.p.skip_sig && layer == 0 && which == c.p.skip_sig - 1;
    if (threadIdx.x == 0 && n && !c.p.staged && !skip) red_release(ctr_of(c.p, layer, which), n);
    if (*(volatile int*)&c.ms.abort) c.dead = true;
}

// consumer-wide reductions (all 256 consumer threads call; uses Misc.bred)
__device__ float cblock_sum(Ctx& c, float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    cbar();
    if (lane == 0) c.ms.bred[warp] = v;
    cbar();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) t += c.ms.bred[w];
    return t;
}
__device__ float cblock_max(Ctx& c, float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    cbar();
    if (lane == 0) c.ms.bred[warp] = v;
    cbar();
    float t = -INFINITY;
#pragma unroll
    for (int w = 0; w < NCW; ++w) t = fmaxf(t, c.ms.bred[w]);
    return t;
}

// stage trace (consumer thread 0): wait start, inputs ready, stage done
__device__ __forceinline__ void trace_rec(Ctx& c, unsigned code, unsigned n, long long t0, long long t1) {
    if (!c.p.trace || threadIdx.x != 0) return;
    unsigned* cnt = c.p.trace_n + blockIdx.x;
    const unsigned i = atomicAdd(cnt, 1u);
    if (i >= (unsigned)c.p.trace_cap) return;
    TraceRec* r = c.p.trace + (size_t)blockIdx.x * c.p.trace_cap + i;
    r->code = code;
    r->n = n;
    r->t_wait = t0;
    r->t_ready = t1;
    r->t_end = gtimer();
}

// a trace record from any thread (per-warp records, MK_TRACE=3)
__device__ __forceinline__ void trace_rec_any(Ctx& c, unsigned code, unsigned n, long long t0, long long t1) {
    unsigned* cnt = c.p.trace_n + blockIdx.x;
    const unsigned i = atomicAdd(cnt, 1u);
    if (i >= (unsigned)c.p.trace_cap) return;
    TraceRec* r = c.p.trace + (size_t)blockIdx.x * c.p.trace_cap + i;
    r->code = code;
    r->n = n;
    r->t_wait = t0;
    r->t_ready = t1;
    r->t_end = gtimer();
}

// =============================================================== GEMV ====

// the global token row staged at staging row t (first staged entry m0)
__device__ __forceinline__ int staged_token(const Misc& ms, int m0, int t) {
    return ms.gather ? (int)ms.gt[m0 + t] : m0 + t;
}
// the staging row of token-map entry i when entries [0, ...) are staged
__device__ __forceinline__ int staging_row(const Misc& ms, int i) { return ms.gather ? i : (int)ms.gt[i]; }

// fill stage[t][0..Kc) with f(input) for tokens m0 .. m0+ms-1
// small inputs (at most two 8-float chunks per thread, K panel a multiple
// of 256 so a warp's chunks belong to one token): every global load is
// issued up front into registers, the values never leave registers between
// the sum of squares and the scaling, one barrier in between
__device__ __forceinline__ void stage_input_small(Ctx& c, const Gemv& g, const float* src, int grp_off, int k0, int m0,
                                                  int ms) {
    const Params& p = c.p;
    float* xs = c.stage();
    const int Kc = g.Kc, tid = ctid(), lane = tid & 31;
    const int total = ms * Kc, kind = g.in_kind, stride = g.src_stride;
    float4 va[2], vb[2];
    uint4 gw[2];
    int t_[2];
    bool ok[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int i = (tid + q * NCT) * 8;
        ok[q] = i < total;
        const int t = ok[q] ? i / Kc : 0, k = i - t * Kc;
        t_[q] = t;
        va[q] = vb[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        gw[q] = make_uint4(0u, 0u, 0u, 0u);
        if (ok[q]) {
            const float* r = src + (size_t)staged_token(c.ms, m0, t) * stride + grp_off + k0 + k;
            va[q] = __ldcg(reinterpret_cast<const float4*>(r));
            vb[q] = __ldcg(reinterpret_cast<const float4*>(r + 4));
            if (kind == IN_RMS) {
                gw[q] = __ldg(reinterpret_cast<const uint4*>(g.gain + k0 + k));
            } else if (kind == IN_SWIGLU) {
                const float4 ua = __ldcg(reinterpret_cast<const float4*>(r + g.sw_off));
                const float4 ub = __ldcg(reinterpret_cast<const float4*>(r + g.sw_off + 4));
                va[q] = make_float4(silu(va[q].x) * ua.x, silu(va[q].y) * ua.y, silu(va[q].z) * ua.z, silu(va[q].w) * ua.w);
                vb[q] = make_float4(silu(vb[q].x) * ub.x, silu(vb[q].y) * ub.y, silu(vb[q].z) * ub.z, silu(vb[q].w) * ub.w);
            }
        }
    }
    if (kind == IN_RMS) {
        float* acc = c.ms.rms;  // zeroed by restage() before its leading barrier
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float s2 = va[q].x * va[q].x;
            s2 = fmaf(va[q].y, va[q].y, s2);
            s2 = fmaf(va[q].z, va[q].z, s2);
            s2 = fmaf(va[q].w, va[q].w, s2);
            s2 = fmaf(vb[q].x, vb[q].x, s2);
            s2 = fmaf(vb[q].y, vb[q].y, s2);
            s2 = fmaf(vb[q].z, vb[q].z, s2);
            s2 = fmaf(vb[q].w, vb[q].w, s2);
#pragma unroll
            for (int o = 16; o; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
            if (lane == 0 && ok[q]) atomicAdd(&acc[t_[q]], s2);
        }
        cbar();
        const float invK = 1.0f / (float)g.K;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (!ok[q]) continue;
            const float r = 1.0f / sqrtf(acc[t_[q]] * invK + p.eps);
            const uint4 w = gw[q];
            va[q] = make_float4(va[q].x * bf_lo(w.x) * r, va[q].y * bf_hi(w.x) * r, va[q].z * bf_lo(w.y) * r,
                                va[q].w * bf_hi(w.y) * r);
            vb[q] = make_float4(vb[q].x * bf_lo(w.z) * r, vb[q].y * bf_hi(w.z) * r, vb[q].z * bf_lo(w.w) * r,
                                vb[q].w * bf_hi(w.w) * r);
        }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        if (!ok[q]) continue;
        const int i = (tid + q * NCT) * 8, t = i / Kc;
        float* d = xs + t * stage_stride(Kc) + (i - t * Kc);
        *reinterpret_cast<float4*>(d) = va[q];
        *reinterpret_cast<float4*>(d + 4) = vb[q];
    }
}

__device__ __noinline__ void stage_input(Ctx& c, const Gemv& g, const float* src, int grp_off, int kc, int m0, int ms) {
    const Params& p = c.p;
    float* xs = c.stage();
    const int Kc = g.Kc, k0 = kc * Kc, tid = ctid(), lane = tid & 31, warp = tid >> 5;
    const int total = ms * Kc;
    if (total <= 2 * NCT * 8 && (Kc & 255) == 0 && (g.in_kind != IN_RMS || g.n_kc == 1)) {
        stage_input_small(c, g, src, g.in_kind == IN_RMS ? 0 : grp_off, k0, m0, ms);
        return;
    }
    if (g.in_kind == IN_COPY || (g.in_kind == IN_RMS && g.n_kc == 1)) {
        // several tokens' rows: every 16-byte piece is in flight at once
        // (one L2 round trip instead of one per loop iteration), then the
        // RMSNorm, if any, works on the copy in shared memory
        const int off = g.in_kind == IN_RMS ? 0 : grp_off;
        const int SS = stage_stride(Kc);
        for (int i = tid * 4; i < total; i += NCT * 4) {
            const int t = i / Kc, k = i - t * Kc;
            cp_async16(xs + t * SS + k, src + (size_t)staged_token(c.ms, m0, t) * g.src_stride + off + k0 + k);
        }
        cp_async_wait_all();
        cbar();
        if (g.in_kind == IN_COPY) return;
        // c.ms.rms[] was zeroed by restage() before its leading barrier; a
        // warp's 128 consecutive floats never straddle a row (rows are
        // multiples of 128 floats), so `t` changes uniformly in the warp
        float* acc = c.ms.rms;
        float part = 0.f;
        int cur = -1;
        for (int i = tid * 4; i < total; i += NCT * 4) {
            const int t = i / Kc;
            const float4 v = *reinterpret_cast<const float4*>(xs + t * SS + (i - t * Kc));
            if (t != cur) {
                if (cur >= 0) {
#pragma unroll
                    for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                    if (lane == 0) atomicAdd(&acc[cur], part);
                }
                part = 0.f;
                cur = t;
            }
            part = fmaf(v.x, v.x, part);
            part = fmaf(v.y, v.y, part);
            part = fmaf(v.z, v.z, part);
            part = fmaf(v.w, v.w, part);
        }
        if (cur >= 0) {
#pragma unroll
            for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) atomicAdd(&acc[cur], part);
        }
        cbar();
        const float invK = 1.0f / (float)g.K;
#pragma unroll 4
        for (int i = tid * 4; i < total; i += NCT * 4) {
            const int t = i / Kc, k = i - t * Kc;
            const float r = 1.0f / sqrtf(acc[t] * invK + p.eps);
            const uint2 gw = __ldg(reinterpret_cast<const uint2*>(g.gain + k));
            float4* xp = reinterpret_cast<float4*>(xs + t * SS + k);
            float4 o = *xp;
            o.x = o.x * bf_lo(gw.x) * r;
            o.y = o.y * bf_hi(gw.x) * r;
            o.z = o.z * bf_lo(gw.y) * r;
            o.w = o.w * bf_hi(gw.y) * r;
            *xp = o;
        }
        return;
    }
    if (g.in_kind == IN_RMS) {
        // c.ms.rms[] was zeroed by restage() before its leading barrier.
        // Split panels (the K panel is part of the row): the sum of squares
        // runs over the whole row first, then the panel is scaled.
        float* acc = c.ms.rms;
        const int rowlen = g.K, tot = c.rms_src == src ? 0 : ms * rowlen;  // (0: summed by the stage's CTAs)
        const uint16_t* gain = g.gain;
        float part = 0.f;
        int cur = -1;
        // 4 loads per thread in flight per round trip (the rows were written
        // by other SMs moments ago: every load goes to L2)
        for (int i0 = tid * 4; i0 < tot; i0 += NCT * 4 * 4) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * NCT * 4, t = i / rowlen;
                v[u] = i < tot ? __ldcg(reinterpret_cast<const float4*>(
                                     src + (size_t)staged_token(c.ms, m0, t) * g.src_stride + i - t * rowlen))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * NCT * 4, t = i / rowlen;
                if (i >= tot) break;  // uniform in the warp
                // a warp's 128 consecutive floats never straddle a row (rows are
                // multiples of 128 floats), so `t` changes uniformly in the warp
                if (t != cur) {
                    if (cur >= 0) {
#pragma unroll
                        for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                        if (lane == 0) atomicAdd(&acc[cur], part);
                    }
                    part = 0.f;
                    cur = t;
                }
                part = fmaf(v[u].x, v[u].x, part);
                part = fmaf(v[u].y, v[u].y, part);
                part = fmaf(v[u].z, v[u].z, part);
                part = fmaf(v[u].w, v[u].w, part);
            }
        }
        if (cur >= 0) {
#pragma unroll
            for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) atomicAdd(&acc[cur], part);
        }
        cbar();
        const float invK = 1.0f / (float)g.K;
#pragma unroll 4
        for (int i = tid * 4; i < total; i += NCT * 4) {
            const int t = i / Kc, k = i - t * Kc;
            const float r = 1.0f / sqrtf(acc[t] * invK + p.eps);
            const float4 v =
                __ldcg(reinterpret_cast<const float4*>(src + (size_t)staged_token(c.ms, m0, t) * g.src_stride + k0 + k));
            const uint2 gw = __ldg(reinterpret_cast<const uint2*>(gain + k0 + k));
            float4 o;
            o.x = v.x * bf_lo(gw.x) * r;
            o.y = v.y * bf_hi(gw.x) * r;
            o.z = v.z * bf_lo(gw.y) * r;
            o.w = v.w * bf_hi(gw.y) * r;
            *reinterpret_cast<float4*>(xs + t * stage_stride(Kc) + k) = o;
        }
    } else {  // IN_SWIGLU: h = silu(gate) * up
#pragma unroll 4
        for (int i = tid * 4; i < total; i += NCT * 4) {
            const int t = i / Kc, k = i - t * Kc;
            const float* r = src + (size_t)staged_token(c.ms, m0, t) * g.src_stride + k0 + k;
            float4 gv = __ldcg(reinterpret_cast<const float4*>(r));
            float4 uv = __ldcg(reinterpret_cast<const float4*>(r + g.sw_off));
            float4 o;
            o.x = silu(gv.x) * uv.x;
            o.y = silu(gv.y) * uv.y;
            o.z = silu(gv.z) * uv.z;
            o.w = silu(gv.w) * uv.w;
            *reinterpret_cast<float4*>(xs + t * stage_stride(Kc) + k) = o;
        }
    }
}

// token m was routed to `expert` (its weight may still round to zero)
__device__ __forceinline__ bool routed_to(const Misc& ms, int m, int expert, int k) {
    for (int j = 0; j < k; ++j)
        if (ms.ridx[m][j] == expert) return true;
    return false;
}

__device__ __forceinline__ float route_weight(const Misc& ms, int m, int expert, int k) {
    for (int j = 0; j < k; ++j)
        if (ms.ridx[m][j] == expert) return ms.rw[m][j];
    return 0.f;
}

// one output value of a GEMV item
__device__ __forceinline__ void gemv_out(Ctx& c, const Gemv& g, int slot, int expert, int m, int row, float y) {
    if (g.out_kind == OUT_STORE) {
        float* d = g.dst + (size_t)slot * g.dst_sstride + (size_t)m * g.dst_stride + row;
        if (g.n_kc == 1)
            *d = y;
        else
            atomicAdd(d, y);
    } else if (g.out_kind == OUT_RESID) {
        float* d = g.dst + (size_t)m * g.dst_stride + row;
        if (g.n_kc == 1) {
            const float v = __ldcg(d) + y;
            *d = v;
            g.dst2[(size_t)m * g.dst_stride + row] = v;
        } else {
            atomicAdd(d, y);
        }
    } else if (g.out_kind == OUT_SCALED) {  // expert down projection added into the next residual
        const float w = expert < 0 ? 1.0f : route_weight(c.ms, m, expert, c.p.topk);
        if (w != 0.f) atomicAdd(g.dst + (size_t)m * g.dst_stride + row, w * y);
    } else {  // OUT_ACC: this thread owns the value
        g.dst[(size_t)m * g.dst_stride + row] += y;
    }
}

// 8 products of bf16 weights and fp32 inputs held in registers (no
// addressable local array: that would live in local memory)
__device__ __forceinline__ void fma8v(float& a, const uint4 w, const float4 x0, const float4 x1) {
    a = fmaf(bf_lo(w.x), x0.x, a);
    a = fmaf(bf_hi(w.x), x0.y, a);
    a = fmaf(bf_lo(w.y), x0.z, a);
    a = fmaf(bf_hi(w.y), x0.w, a);
    a = fmaf(bf_lo(w.z), x1.x, a);
    a = fmaf(bf_hi(w.z), x1.y, a);
    a = fmaf(bf_lo(w.w), x1.z, a);
    a = fmaf(bf_hi(w.w), x1.w, a);
}

// the same 8 products into two accumulators (halves the dependent chain)
__device__ __forceinline__ void fma8v2(float& a, float& b, const uint4 w, const float4 x0, const float4 x1) {
    a = fmaf(bf_lo(w.x), x0.x, a);
    b = fmaf(bf_hi(w.x), x0.y, b);
    a = fmaf(bf_lo(w.y), x0.z, a);
    b = fmaf(bf_hi(w.y), x0.w, b);
    a = fmaf(bf_lo(w.z), x1.x, a);
    b = fmaf(bf_hi(w.z), x1.y, b);
    a = fmaf(bf_lo(w.w), x1.z, a);
    b = fmaf(bf_hi(w.w), x1.w, b);
}

__device__ __forceinline__ void fma8(float& a, const uint4& w, const float (&x)[8]) {
    a = fmaf(bf_lo(w.x), x[0], a);
    a = fmaf(bf_hi(w.x), x[1], a);
    a = fmaf(bf_lo(w.y), x[2], a);
    a = fmaf(bf_hi(w.y), x[3], a);
    a = fmaf(bf_lo(w.z), x[4], a);
    a = fmaf(bf_hi(w.z), x[5], a);
    a = fmaf(bf_lo(w.w), x[6], a);
    a = fmaf(bf_hi(w.w), x[7], a);
}

// One warp's share of a weight tile: the warp owns rows [warp*RW, warp*RW+RW)
// of the tile (RW = rows/8) and its lanes split the K panel into 16-byte
// chunks; products against MTc staged tokens, a warp-shuffle reduction, and
// the warp writes its own outputs. No CTA-wide barrier per tile.
template <int MTc>
__device__ void gemv_warp_tile(Ctx& c, const Gemv& g, const uint8_t* tile, int nr, const float* xs, int mt0,
                               int mcount, int mbase, int slot, int expert, int r0) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // warp w owns rows [w RW, w RW + RW) of the tile, clipped to nr (tiles of
    // fewer than 8 rows leave some warps without rows)
    const int Kc = g.Kc, NC = Kc >> 3, RW = (nr + 7) >> 3, rw0 = warp * RW;
    const int RWv = max(0, min(RW, nr - rw0));  // this warp's rows
    const uint4* T4 = reinterpret_cast<const uint4*>(tile);
    // staged row of token mbase + m: the staging holds tokens from mbase - mt0 on
    int xrow[MTc];
#pragma unroll
    for (int m = 0; m < MTc; ++m)
        xrow[m] = m < mcount && !c.ms.gather ? (int)c.ms.gt[mbase + m] - (mbase - mt0) : mt0 + m;
    if (NC >= 32) {
        const int JC = NC >> 5;
        for (int r = 0; r < RWv; r += 4) {
            const int nrr = min(4, RWv - r);
            float acc[4][MTc];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int m = 0; m < MTc; ++m) acc[i][m] = 0.f;
            for (int j = 0; j < JC; ++j) {
                const int ch = lane + 32 * j;
                float xv[MTc][8];
#pragma unroll
                for (int m = 0; m < MTc; ++m) {
                    const float4 a = *reinterpret_cast<const float4*>(xs + (size_t)xrow[m] * stage_stride(Kc) + ch * 8);
                    const float4 b = *reinterpret_cast<const float4*>(xs + (size_t)xrow[m] * stage_stride(Kc) + ch * 8 + 4);
                    xv[m][0] = a.x; xv[m][1] = a.y; xv[m][2] = a.z; xv[m][3] = a.w;
                    xv[m][4] = b.x; xv[m][5] = b.y; xv[m][6] = b.z; xv[m][7] = b.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < nrr) {
                        const uint4 w = T4[(size_t)(rw0 + r + i) * NC + ch];
#pragma unroll
                        for (int m = 0; m < MTc; ++m) fma8(acc[i][m], w, xv[m]);
                    }
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int m = 0; m < MTc; ++m) acc[i][m] += __shfl_xor_sync(0xffffffffu, acc[i][m], o);
            // lane i*MTc + m writes value (row i, token m)
            float myv = 0.f;
            int mi = 4, mm = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int m = 0; m < MTc; ++m)
                    if (lane == i * MTc + m) {
                        myv = acc[i][m];
                        mi = i;
                        mm = m;
                    }
            if (mi < nrr && mm < mcount) gemv_out(c, g, slot, expert, mbase + mm, r0 + rw0 + r + mi, myv);
        }
    } else {
        // short rows (K = 128): 32/NC rows per pass, NC lanes per row
        const int G = 32 / NC, gi = lane / NC, ch = lane - gi * NC;
        for (int pass = 0; pass < (RWv + G - 1) / G; ++pass) {
            const int rl = pass * G + gi, row = rw0 + rl;
            const bool rv = rl < RWv;
            float acc[MTc];
            const uint4 w = rv ? T4[(size_t)row * NC + ch] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int m = 0; m < MTc; ++m) {
                float xv[8];
                const float4 a = *reinterpret_cast<const float4*>(xs + (size_t)xrow[m] * stage_stride(Kc) + ch * 8);
                const float4 b = *reinterpret_cast<const float4*>(xs + (size_t)xrow[m] * stage_stride(Kc) + ch * 8 + 4);
                xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
                xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
                acc[m] = 0.f;
                fma8(acc[m], w, xv);
            }
            for (int o = NC >> 1; o; o >>= 1)
#pragma unroll
                for (int m = 0; m < MTc; ++m) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
            float myv = 0.f;
#pragma unroll
            for (int m = 0; m < MTc; ++m)
                if (ch == m) myv = acc[m];
            if (rv && ch < mcount) gemv_out(c, g, slot, expert, mbase + ch, r0 + row, myv);
        }
    }
}

// (re)stage the input of item j when it differs from what the buffer holds;
// the staged input is identified by buffer, head group, K panel, token range
// and gain: every GEMV input buffer is written once per step
__device__ __forceinline__ bool restage(Ctx& c, const Gemv& g, const float* src, int grp_off, int kc, int m0,
                                        int ms) {
    if (c.sk_src == src && c.sk_off == grp_off && c.sk_kc == kc && c.sk_m0 == m0 && c.sk_kind == g.in_kind &&
        c.sk_gain == g.gain && c.sk_gather == c.ms.gather)
        return false;
    // nobody reads the RMS accumulators between stagings: zero them before
    // the barrier that ends every use of the previous contents
    if (g.in_kind == IN_RMS && ctid() < ms && c.rms_src != src) c.ms.rms[ctid()] = 0.f;
    cbar();
    stage_input(c, g, src, grp_off, kc, m0, ms);
    cbar();
    c.sk_src = src;
    c.sk_off = grp_off;
    c.sk_kc = kc;
    c.sk_m0 = m0;
    c.sk_kind = g.in_kind;
    c.sk_gain = g.gain;
    c.sk_gather = c.ms.gather;
    return true;
}

// inline bounded spin on a ring barrier (no calls: hot loops stay free of
// register spills); false on timeout or abort
__device__ __forceinline__ bool spin_wait(const Params& p, unsigned long long* bar, unsigned parity) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = gtimer();
    for (unsigned it = 1;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 63) == 0 && (gtimer() - t0 > p.timeout_ns || ld_relaxed(&p.status[1]))) return false;
    }
}

// end of the run of items that share the staged input (same K panel and,
// for grouped inputs, the same head group) starting at item j of panel kc0,
// row block rb0: items [j, jend) -- arithmetic only, no per-item divisions
__device__ __forceinline__ int run_end(int j, int j_hi, int n_rb, int rb0, int R, int grp_rows, int g0) {
    int rb_end = n_rb;  // the panel ends the run
    if (grp_rows) {
        const int gb = (g0 + 1) * grp_rows;  // first row of the next group
        rb_end = min(n_rb, (gb + R - 1) / R);
    }
    return min(j_hi, j + (rb_end - rb0));
}

// ---- split-K GEMV (M <= 8 tokens) ----
// Every lane handles 8 rows of a tile against ONE 16-byte chunk of the K
// panel, whose input values it keeps in registers for the whole run; per
// tile it does 8 shared-memory loads and 64*MR FMAs. A warp's lanes form
// 32/CPWP row groups of CPWP lanes (CPWP = 32, or 16 for K panels whose row
// slices are 12 or 16 chunks); the row slice of a warp is CPW <= CPWP
// chunks wide, and NKS warps (8, 4, 2 or 1) share the same rows with
// different K slices. The warp reduces its 8*MR partials across the CPWP
// lanes of a group (each halving step exchanges half of the values, so a
// lane ends with one sum instead of 8), writes them to its own slot in
// shared memory, and after one CTA barrier per chunk of up to MC tokens
// every output of the chunk sums the NKS warps' partials. Tokens come MR at
// a time; the tile's weights are read once per MR tokens.
//   Kc 2048: NKS 8, CPW 32 -> 8 rows    Kc 1024: NKS 4, CPW 32 -> 16 rows
//   Kc  768: NKS 8, CPW 12 -> 16 rows   Kc  512: NKS 2, CPW 32 -> 32 rows
//   Kc  256: NKS 1, CPW 32 -> 64 rows   Kc  128: NKS 1, CPW 16 -> 128 rows
__device__ __forceinline__ int ks_nks(int Kc) {
    return Kc == 2048 ? 8 : Kc == 1024 ? 4 : Kc == 768 ? 8 : Kc == 512 ? 2 : (Kc == 256 || Kc == 128) ? 1 : 0;
}

// reduce v[8][MR] across the CPWP lanes of a row group; afterwards a lane
// holds in v[0] the sum for local row 4*b1 + 2*b2 + b3 (bits CPWP/2,
// CPWP/4, CPWP/8 of its lane index)
template <int CPWP, int MR>
__device__ __forceinline__ void ks_reduce(float (&v)[8][MR]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int lvl = 0; lvl < 3; ++lvl) {
        const int o = CPWP >> (lvl + 1), half = 4 >> lvl;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k)
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                const float send = up ? v[k][m] : v[k + half][m];
                const float keep = up ? v[k + half][m] : v[k][m];
                v[k][m] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
    }
#pragma unroll
    for (int o = CPWP / 16; o >= 1; o >>= 1)
#pragma unroll
        for (int m = 0; m < MR; ++m) v[0][m] += __shfl_xor_sync(0xffffffffu, v[0][m], o);
}

template <int CPWP, int MR>
__device__ __forceinline__ void gemv_range_ks(Ctx& c, const Gemv& g, int slot, int expert, int j_lo, int j_hi) {
    const Params& p = c.p;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    constexpr int RG = 32 / CPWP, RWT = 8 * RG;  // row groups per warp, rows per warp tile
    const int M = c.ms.gm, Kc = g.Kc, NC = Kc >> 3, NKS = ks_nks(Kc), CPW = NC / NKS;
    const int ks = warp % NKS, rb = warp / NKS;
    const int rg = lane / CPWP, ch = lane % CPWP;
    const bool act = ch < CPW;
    const int chunk = ks * CPW + ch;
    const int lrow = rg + RG * ((lane & (CPWP / 2) ? 4 : 0) + (lane & (CPWP / 4) ? 2 : 0) + (lane & (CPWP / 8) ? 1 : 0));
    const bool writer = (lane & (CPWP / 8 - 1)) == 0;
    const int n_rb = g.n_rb, R = g.R, N = g.N, grp_rows = g.grp_rows, grp_stride = g.grp_stride;
    const int out_kind = g.out_kind, n_kc = g.n_kc, dst_stride = g.dst_stride;
    float* const dst = g.dst + (size_t)slot * g.dst_sstride;
    float* const dst2 = g.dst2;
    const float* src = g.src + (size_t)slot * g.src_sstride;
    Misc& ms = c.ms;
    uint8_t* const ring = c.smem + SMEM_RING;
    const float* const xs = c.stage();
    // tokens in chunks of MC (one CTA barrier and one final sum per chunk),
    // each chunk in groups of MR (partials written without a barrier);
    // partials [2][NCW][RWT * MC] in the first half of the reduction area
    constexpr int MC = (32 / RWT) > MR ? (32 / RWT) : MR;
    float* const part = c.red();
    const int ngrp = (M + MR - 1) / MR;
    CRing cr = c.cr;
    bool dead = c.dead, timed_out = false;
    int buf = 0;
    float4 xa[MR], xb[MR];
    int j = j_lo;
    while (j < j_hi) {
        // a run of items sharing the staged input (same K panel and head group)
        const int kc0 = j / n_rb, rb0 = j - kc0 * n_rb;
        const int g0 = grp_rows ? (rb0 * R) / grp_rows : 0;
        const int jend = run_end(j, j_hi, n_rb, rb0, R, grp_rows, g0);
        const long long ta = p.trace_items ? gtimer() : 0;
        restage(c, g, src, g0 * grp_stride, kc0, 0, M);
        const long long tb = p.trace_items ? gtimer() : 0;
        long long tc = tb;
        const int jrun = j;
        for (; j < jend; ++j) {
            const int rbk = rb0 + (j - jrun);  // same K panel for the whole run
            const int r0 = rbk * R, nr = min(R, N - r0);
            const uint8_t* tile = nullptr;
            if (!dead) {
                if (spin_wait(p, &ms.full[cr.slot], cr.phase))
                    tile = ring + cr.slot * SLOT_BYTES;
                else
                    dead = timed_out = true;
            }
            if (p.trace_items && j == jrun) tc = gtimer();
            for (int mc0 = 0; mc0 < M; mc0 += MC) {
                const int mcn = min(MC, M - mc0);
                for (int mb = mc0; mb < mc0 + mcn; mb += MR) {
                    if (j == jrun || ngrp > 1) {
#pragma unroll
                        for (int m = 0; m < MR; ++m) {
                            const bool ok = act && mb + m < M;
                            const float* xp = xs + (size_t)(ok ? staging_row(ms, mb + m) : 0) * stage_stride(Kc) + chunk * 8;
                            xa[m] = ok ? *reinterpret_cast<const float4*>(xp) : make_float4(0.f, 0.f, 0.f, 0.f);
                            xb[m] = ok ? *reinterpret_cast<const float4*>(xp + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    float v[8][MR];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int m = 0; m < MR; ++m) v[i][m] = 0.f;
                    if (tile) {
                        const uint4* T4 = reinterpret_cast<const uint4*>(tile) + chunk;
                        const int rw = rb * RWT + rg;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int r = rw + RG * i;
                            if (act && r < nr) {
                                const uint4 w = T4[(size_t)r * NC];
#pragma unroll
                                for (int m = 0; m < MR; ++m) fma8v(v[i][m], w, xa[m], xb[m]);
                            }
                        }
                    }
                    ks_reduce<CPWP, MR>(v);
                    if (writer) {
                        float* pw = part + (buf * NCW + warp) * RWT * MC + lrow * MC + (mb - mc0);
#pragma unroll
                        for (int m = 0; m < MR; ++m)
                            if (mb + m < mc0 + mcn) pw[m] = v[0][m];
                    }
                }
                if (mc0 + MC >= M) {
                    // the tile has been read: hand the slot back to the producer
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ms.empty[cr.slot]);
                }
                cbar();
                if (tile) {
                    for (int t = tid; t < nr * mcn; t += NCT) {
                        const int r = t / mcn, mi = t - r * mcn, m = mc0 + mi;
                        const int b = r / RWT, rl = r - b * RWT;
                        const float* q = part + ((buf * NCW + b * NKS) * RWT + rl) * MC + mi;
                        float y = q[0];
                        for (int k = 1; k < NKS; ++k) y += q[k * RWT * MC];
                        const int row = r0 + r;
                        float* d = dst + (size_t)m * dst_stride + row;
                        if (out_kind == OUT_STORE) {
                            if (n_kc == 1)
                                *d = y;
                            else
                                atomicAdd(d, y);
                        } else if (out_kind == OUT_RESID) {
                            if (n_kc == 1) {
                                const float nv = __ldcg(d) + y;
                                *d = nv;
                                dst2[(size_t)m * dst_stride + row] = nv;
                            } else {
                                atomicAdd(d, y);
                            }
                        } else if (out_kind == OUT_SCALED) {
                            const float w = expert < 0 ? 1.0f : route_weight(ms, m, expert, p.topk);
                            if (w != 0.f) atomicAdd(d, w * y);
                        } else {
                            *d += y;
                        }
                    }
                }
                buf ^= 1;
            }
            if (++cr.slot == NSLOT) {
                cr.slot = 0;
                cr.phase ^= 1u;
            }
        }
        // item trace: one record per run (staging time, first tile ready, run done)
        if (p.trace_items && threadIdx.x == 0) trace_rec(c, 0x80000000u | c.cur_code, (unsigned)(tb - ta), ta, tc);
    }
    if (timed_out) {
        ms.abort = 1;
        raise_status(p, ST_TIMEOUT, 0x210u);
    }
    c.set_ring(cr);
    if (dead) c.dead = true;
}

// ---- one-token GEMV with the input in registers ----
// A warp owns whole rows (rows warp, warp+8, ... of a tile) and its lanes
// split the K panel into 16-byte chunks; the lane's chunks of the input
// (lane + 32q, q < JC = Kc/256, at most 8 -> 64 floats) stay in registers for
// the run. Per tile the shared-memory traffic is the weights once, there is
// no CTA barrier, and the warps move on to the next tile independently.
// K panels of 128 elements (16 chunks): two rows per warp pass, 16 lanes each.
// The MT instances take 2 to 4 tokens (the token map's rows of the staging
// area): each tile once per token, the token's input reloaded each time.
__device__ __forceinline__ void rx_out(const Params& p, Misc& ms, int out_kind, int n_kc, float* d, float* d2, int expert,
                                       float y) {
    if (out_kind == OUT_STORE) {
        if (n_kc == 1)
            *d = y;
        else
            atomicAdd(d, y);
    } else if (out_kind == OUT_RESID) {
        if (n_kc == 1) {
            const float nv = __ldcg(d) + y;
            *d = nv;
            *d2 = nv;
        } else {
            atomicAdd(d, y);
        }
    } else if (out_kind == OUT_SCALED) {
        const float w = expert < 0 ? 1.0f : route_weight(ms, 0, expert, p.topk);
        if (w != 0.f) atomicAdd(d, w * y);
    } else {
        *d += y;
    }
}

// sums of RB per-lane values over the warp: after log2(RB) halving steps
// (each lane keeps half of its values and adds its partner's other half)
// and plain steps for the remaining lane bits, v[0] of every lane holds the
// full sum of value b = its lane bits 16, 8, 4 (high to low, as many as
// log2 RB) -- returned; lanes whose low 5 - log2(RB) bits are 0 are one
// writer per value
template <int RB>
__device__ __forceinline__ int rx_reduce(float (&v)[RB]) {
    const int lane = threadIdx.x & 31;
    int b = 0;
#pragma unroll
    for (int lvl = 0, n = RB; n > 1; ++lvl, n >>= 1) {
        const int o = 16 >> lvl, half = n / 2;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < RB / 2; ++k) {
            if (k < half) {
                const float send = up ? v[k] : v[k + half];
                const float keep = up ? v[k + half] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        if (up) b += half;
    }
    constexpr int LV = RB == 1 ? 0 : (RB == 2 ? 1 : (RB == 4 ? 2 : (RB == 8 ? 3 : 4)));
#pragma unroll
    for (int o = 16 >> LV; o >= 1; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    return b;
}

// 8 values per lane summed over each 16-lane half: halving over lane bits
// 8, 4, 2, then bit 1; returns the value index v[0] now holds
__device__ __forceinline__ int rx_reduce16(float (&v)[8]) {
    const int lane = threadIdx.x & 31;
    int k = 0;
#pragma unroll
    for (int lvl = 0, n = 8; n > 1; ++lvl, n >>= 1) {
        const int o = 8 >> lvl, half = n / 2;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < half) {
                const float send = up ? v[j] : v[j + half];
                const float keep = up ? v[j + half] : v[j];
                v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        if (up) k += half;
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    return k;
}

template <int JC, bool MT = false>
__device__ __forceinline__ void gemv_range_rx(Ctx& c, const Gemv& g, int slot, int expert, int j_lo, int j_hi) {
    const Params& p = c.p;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // JC chunks of 8 elements per lane (K panel = 256*JC); JC == 0: K panel 128
    constexpr bool wide = JC > 0;
    constexpr int NC = wide ? 32 * JC : 16;
    const int n_rb = g.n_rb, R = g.R, N = g.N, grp_rows = g.grp_rows, grp_stride = g.grp_stride;
    const int out_kind = g.out_kind, n_kc = g.n_kc, dst_stride = g.dst_stride;
    float* const dst = g.dst + (size_t)slot * g.dst_sstride;
    float* const dst2 = g.dst2;
    const float* src = g.src + (size_t)slot * g.src_sstride;
    Misc& ms = c.ms;
    uint8_t* const ring = c.smem + SMEM_RING;
    const float* const xs = c.stage();
    // tokens: MT (wide panels only) up to 4, each tile once per token and the
    // input reloaded per token; otherwise one, its input in registers for the run
    const int ntok = MT ? ms.gm : 1;
    CRing cr = c.cr;
    bool dead = c.dead, timed_out = false;
    constexpr int NX = wide ? JC : 1;
    float4 xa[NX], xb[NX];
    if (p.trace_items == 1 && threadIdx.x == 0) ms.tdbg[0] = clock64();
    int j = j_lo;
    while (j < j_hi) {
        const int kc0 = j / n_rb, rb0 = j - kc0 * n_rb;
        const int g0 = grp_rows ? (rb0 * R) / grp_rows : 0;
        const int jend = run_end(j, j_hi, n_rb, rb0, R, grp_rows, g0);
        if (p.trace_items == 1 && threadIdx.x == 0) ms.tdbg[1] = clock64();
        const long long ta = p.trace_items ? gtimer() : 0;
        restage(c, g, src, g0 * grp_stride, kc0, 0, ms.gather ? ms.gm : p.M);
        const long long tb = p.trace_items ? gtimer() : 0;
        long long tc = tb;
        const int ch0 = wide ? lane : (lane & 15);
        const auto load_x = [&](int tk) {
            const float* xt = xs + (size_t)staging_row(ms, tk) * stage_stride(g.Kc);
#pragma unroll
            for (int q = 0; q < NX; ++q) {
                const float* xp = xt + (ch0 + 32 * q) * 8;
                xa[q] = *reinterpret_cast<const float4*>(xp);
                xb[q] = *reinterpret_cast<const float4*>(xp + 4);
            }
        };
        load_x(0);
        const int jrun = j;
        for (; j < jend; ++j) {
            if constexpr (JC == 8) {
                // K panel 2048 (8 rows per tile, one per warp): two tiles per
                // iteration, both rows' loads and FMAs in flight together and
                // one reduction for the two sums
                if (j + 1 < jend && !dead) {
                    const int r0A = (rb0 + (j - jrun)) * R, nrA = min(R, N - r0A);
                    const int r0B = r0A + R, nrB = min(R, N - r0B);
                    CRing crB = cr;
                    if (++crB.slot == NSLOT) {
                        crB.slot = 0;
                        crB.phase ^= 1u;
                    }
                    if (!spin_wait(p, &ms.full[cr.slot], cr.phase) || !spin_wait(p, &ms.full[crB.slot], crB.phase)) {
                        dead = timed_out = true;
                    } else {
                        if (p.trace_items && j == jrun) tc = gtimer();
                        const uint4* wA = reinterpret_cast<const uint4*>(ring + cr.slot * SLOT_BYTES) + (size_t)warp * NC + lane;
                        const uint4* wB = reinterpret_cast<const uint4*>(ring + crB.slot * SLOT_BYTES) + (size_t)warp * NC + lane;
                        for (int tk = 0; tk < ntok; ++tk) {
                            if (MT) load_x(tk);
                            float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int q0 = 0; q0 < 8; q0 += 2) {
                                uint4 u[4];
                                u[0] = wA[32 * q0];
                                u[1] = wA[32 * (q0 + 1)];
                                u[2] = wB[32 * q0];
                                u[3] = wB[32 * (q0 + 1)];
                                fma8v2(a[0], a[1], u[0], xa[q0], xb[q0]);
                                fma8v2(a[2], a[3], u[1], xa[q0 + 1], xb[q0 + 1]);
                                fma8v2(b[0], b[1], u[2], xa[q0], xb[q0]);
                                fma8v2(b[2], b[3], u[3], xa[q0 + 1], xb[q0 + 1]);
                            }
                            float v[2] = {(a[0] + a[1]) + (a[2] + a[3]), (b[0] + b[1]) + (b[2] + b[3])};
                            const int which = rx_reduce<2>(v);  // lane 0: tile A, lane 16: tile B
                            if ((lane & 15) == 0) {
                                const int row = (which ? r0B : r0A) + warp + tk * dst_stride;
                                if (warp < (which ? nrB : nrA))
                                    rx_out(p, ms, out_kind, n_kc, dst + row, dst2 + row, expert, v[0]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&ms.empty[cr.slot]);
                        mbar_arrive(&ms.empty[crB.slot]);
                    }
                    cr = crB;
                    if (++cr.slot == NSLOT) {
                        cr.slot = 0;
                        cr.phase ^= 1u;
                    }
                    ++j;
                    continue;
                }
            }
            const int rb = rb0 + (j - jrun);
            const int r0 = rb * R, nr = min(R, N - r0);
            const uint8_t* tile = nullptr;
            if (!dead) {
                if (spin_wait(p, &ms.full[cr.slot], cr.phase))
                    tile = ring + cr.slot * SLOT_BYTES;
                else
                    dead = timed_out = true;
            }
            if (p.trace_items && j == jrun) tc = gtimer();
            if (tile) {
                const uint4* T4 = reinterpret_cast<const uint4*>(tile);
                if constexpr (wide) {
                    // RB rows of the warp at a time (rows warp*RB + b + 8*RB*k):
                    // all their loads and FMAs first, then one transposed
                    // reduction for the RB sums
                    constexpr int RB = JC >= 8 ? 1 : (JC >= 3 ? 2 : (JC == 2 ? 4 : 8));
                    for (int tk = 0; tk < ntok; ++tk) {
                    if (MT) load_x(tk);
                    for (int rbase = warp * RB; rbase < nr; rbase += 8 * RB) {
                        float v[RB];
#pragma unroll
                        for (int b = 0; b < RB; ++b) {
                            const int r = rbase + b;
                            float a[4] = {0.f, 0.f, 0.f, 0.f};
                            if (r < nr) {
                                const uint4* w0 = T4 + (size_t)r * NC + lane;
#pragma unroll
                                for (int q0 = 0; q0 < JC; q0 += 4) {
                                    uint4 w[4];
#pragma unroll
                                    for (int u = 0; u < 4; ++u)
                                        if (q0 + u < JC) w[u] = w0[32 * (q0 + u)];
#pragma unroll
                                    for (int u = 0; u < 4; ++u)
                                        if (q0 + u < JC)
                                            fma8v2(a[(2 * u) & 3], a[(2 * u + 1) & 3], w[u], xa[q0 + u], xb[q0 + u]);
                                }
                            }
                            v[b] = (a[0] + a[1]) + (a[2] + a[3]);
                        }
                        const int b = rx_reduce<RB>(v);
                        const int r = rbase + b;
                        const size_t o = (size_t)tk * dst_stride + r0 + r;
                        if ((lane & (32 / RB - 1)) == 0 && r < nr) rx_out(p, ms, out_kind, n_kc, dst + o, dst2 + o, expert, v[0]);
                    }
                    }
                } else {
                    // 16 chunks per row: lanes 0-15 row r, lanes 16-31 row r + 1,
                    // r = 2 warp + 16 k; all 8 passes first, then one reduction
                    const int half = lane >> 4, ch = lane & 15;
                    float v[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int rr = warp * 2 + half + 16 * k;
                        float a = 0.f, a1 = 0.f;
                        if (rr < nr) fma8v2(a, a1, T4[(size_t)rr * NC + ch], xa[0], xb[0]);
                        v[k] = a + a1;
                    }
                    // halving over lane bits 8, 4, 2 of the 16-lane half, then bit 1
                    const int k = rx_reduce16(v);
                    const int rr = warp * 2 + half + 16 * k;
                    if ((ch & 1) == 0 && rr < nr) rx_out(p, ms, out_kind, n_kc, dst + r0 + rr, dst2 + r0 + rr, expert, v[0]);
                    for (int r = warp * 2 + 128; r < nr; r += 16) {  // tiles of more than 128 rows
                        const int r2 = r + half;
                        float a = 0.f, a1 = 0.f;
                        if (r2 < nr) fma8v2(a, a1, T4[(size_t)r2 * NC + ch], xa[0], xb[0]);
                        a += a1;
#pragma unroll
                        for (int o = 8; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                        if (ch == 0 && r2 < nr) rx_out(p, ms, out_kind, n_kc, dst + r0 + r2, dst2 + r0 + r2, expert, a);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.empty[cr.slot]);
            if (++cr.slot == NSLOT) {
                cr.slot = 0;
                cr.phase ^= 1u;
            }
        }
        if (p.trace_items == 1 && threadIdx.x == 0) trace_rec(c, 0x80000000u | c.cur_code, (unsigned)(tb - ta), ta, tc);
        if (p.trace_items == 1 && threadIdx.x == 0) ms.tdbg[2] = clock64();
        if (p.trace_items == 2 && lane == 0)
            trace_rec_any(c, 0xC0000000u | ((unsigned)warp << 24) | c.cur_code, (unsigned)(tb - ta), ta, tc);
    }
    if (timed_out) {
        ms.abort = 1;
        raise_status(p, ST_TIMEOUT, 0x210u);
    }
    c.set_ring(cr);
    if (dead) c.dead = true;
}

// general path (any M, short K panels): input staged in shared memory
__device__ __forceinline__ void gemv_range_smem(Ctx& c, const Gemv& g, int slot, int expert, int j_lo, int j_hi) {
    const Params& p = c.p;
    const float* src = g.src + (size_t)slot * g.src_sstride;
    const int cap = STAGE_FLOATS / stage_stride(g.Kc);
    const int M = c.ms.gm;
    for (int j = j_lo; j < j_hi; ++j) {
        const int kc = j / g.n_rb, rb = j - kc * g.n_rb;
        const int r0 = rb * g.R, nr = min(g.R, g.N - r0);
        const int grp_off = g.grp_rows ? (r0 / g.grp_rows) * g.grp_stride : 0;
        const uint8_t* tile = nullptr;
        const long long ta = p.trace_items ? gtimer() : 0;
        long long tb = ta, tc = ta;
        for (int m0 = 0; m0 < M; m0 += cap) {
            const int ms = min(cap, M - m0);
            restage(c, g, src, grp_off, kc, m0, ms);
            if (p.trace_items) tb = gtimer();
            if (!tile && !c.dead) tile = cons_wait(p, c.smem, c.ms, c.cr);
            if (p.trace_items) tc = gtimer();
            if (tile) {
                for (int mt0 = 0; mt0 < ms; mt0 += MT) {
                    const int cnt = min(MT, ms - mt0);
                    if (cnt == 1)
                        gemv_warp_tile<1>(c, g, tile, nr, c.stage(), mt0, cnt, m0 + mt0, slot, expert, r0);
                    else if (cnt == 2)
                        gemv_warp_tile<2>(c, g, tile, nr, c.stage(), mt0, cnt, m0 + mt0, slot, expert, r0);
                    else
                        gemv_warp_tile<4>(c, g, tile, nr, c.stage(), mt0, cnt, m0 + mt0, slot, expert, r0);
                }
            }
        }
        cons_release(c.ms, c.cr);
        if (p.trace_items && threadIdx.x == 0) trace_rec(c, 0x80000000u | c.cur_code, (unsigned)(tb - ta), ta, tc);
    }
}

// ---- tensor-core GEMV (2 to 8 tokens, K panels of 2048 or 1024) ----
// Per tile of R = 8 NG rows: out[token][row] = sum_k x[token][k] W[row][k] as
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) with the tokens as the 16
// rows of A (at most 8 used) and 8 weight rows as the 8 columns of B. Warps
// split the tile into NG row groups x 8/NG K slices of 256: 16 k-steps per
// warp. Per k-step a lane converts its two pairs of staged input values into
// bf16 hi + lo fragments (x = hi + lo keeps ~16 mantissa bits; two MMAs per
// k-step; fragments are rebuilt per tile: kept for the whole run they would
// not fit the registers and spill to the stack). The producer copies
// these tiles row by row into rows Kc*2 + 16 bytes apart, so a warp's B
// fragment loads (8 rows x 4 lanes) touch 32 distinct banks. The warp frees
// the slot right after its MMAs, then the 8 warps' partial sums meet in the
// reduction area.
// tensor-core tiles: 2 to 8 tokens on K panels of 2048 / 1024 (R = 8 / 16
// rows), 2 to 64 tokens on K panels of 256 (R = 64 rows, the panels of models
// loaded for many tokens per step, gemv_range_mma_wide)
__device__ __forceinline__ bool mma_wide(const Gemv& g) { return g.Kc == 256 && g.R == 64; }
__device__ __forceinline__ bool mma_gemv(int ntok, const Gemv& g) {
    if (ntok < 2 || g.out_kind == OUT_SCALED) return false;
    if (mma_wide(g)) return ntok <= MAX_M;
    return ntok <= 8 && (g.Kc == 2048 || g.Kc == 1024) && g.R * g.Kc * 2 == TILE_MAX;
}
__device__ __forceinline__ uint32_t bf2_pack(float a, float b) {  // a: lower k index, low half
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int NG>
__device__ __forceinline__ void gemv_range_mma(Ctx& c, const Gemv& g, int slot, int j_lo, int j_hi) {
    const Params& p = c.p;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int gq = lane >> 2, t4 = lane & 3;
    constexpr int WK = NCW / NG, KS = 16;  // warps per row group, k-steps per warp
    const int ngw = warp / WK, kbase = (warp % WK) * KS * 16;
    const int M = c.ms.gm, Kc = g.Kc, SS = stage_stride(Kc), pitch = Kc * 2 + 16, R = g.R;
    const int n_rb = g.n_rb, N = g.N, grp_rows = g.grp_rows, grp_stride = g.grp_stride;
    const int out_kind = g.out_kind, n_kc = g.n_kc, dst_stride = g.dst_stride;
    float* const dst = g.dst + (size_t)slot * g.dst_sstride;
    float* const dst2 = g.dst2;
    const float* src = g.src + (size_t)slot * g.src_sstride;
    Misc& ms = c.ms;
    uint8_t* const ring = c.smem + SMEM_RING;
    const float* const xs = c.stage();
    float* const part = c.red();  // [warp][token 8][row 8] partial sums (lower half of the area)
    CRing cr = c.cr;
    bool dead = c.dead, timed_out = false;
    int j = j_lo;
    while (j < j_hi) {
        const int kc0 = j / n_rb, rb0 = j - kc0 * n_rb;
        const int g0 = grp_rows ? (rb0 * R) / grp_rows : 0;
        const int jend = run_end(j, j_hi, n_rb, rb0, R, grp_rows, g0);
        const long long ta = p.trace_items ? gtimer() : 0;
        restage(c, g, src, g0 * grp_stride, kc0, 0, ms.gather ? ms.gm : p.M);
        const long long tb = p.trace_items ? gtimer() : 0;
        long long tc = tb;
        // this warp's input: token gq (tokens >= M contribute zeros), k = kbase + 16 s + 2 t4 (+8)
        const bool xok = gq < M;
        const float* xr = xs + (size_t)(xok ? staging_row(ms, gq) : 0) * SS + kbase + 2 * t4;
        const int jrun = j;
        for (; j < jend; ++j) {
            const int r0 = (rb0 + (j - jrun)) * R, nr = min(R, N - r0);
            const uint8_t* tile = nullptr;
            if (!dead) {
                if (spin_wait(p, &ms.full[cr.slot], cr.phase))
                    tile = ring + cr.slot * SLOT_BYTES;
                else
                    dead = timed_out = true;
            }
            if (p.trace_items && j == jrun) tc = gtimer();
            float hsum[4] = {0.f, 0.f, 0.f, 0.f}, lsum[4] = {0.f, 0.f, 0.f, 0.f};
            if (tile) {
                const uint8_t* tr = tile + (size_t)(ngw * 8 + gq) * pitch + (size_t)kbase * 2 + 4 * t4;
#pragma unroll 4
                for (int s2 = 0; s2 < KS; ++s2) {
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(tr + 32 * s2);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(tr + 32 * s2 + 16);
                    const float2 u = xok ? *reinterpret_cast<const float2*>(xr + 16 * s2) : make_float2(0.f, 0.f);
                    const float2 v = xok ? *reinterpret_cast<const float2*>(xr + 16 * s2 + 8) : make_float2(0.f, 0.f);
                    const uint32_t h0 = bf2_pack(u.x, u.y), h1 = bf2_pack(v.x, v.y);
                    const uint32_t a_h[4] = {h0, 0u, h1, 0u};
                    const uint32_t a_l[4] = {bf2_pack(u.x - bf_lo(h0), u.y - bf_hi(h0)), 0u,
                                             bf2_pack(v.x - bf_lo(h1), v.y - bf_hi(h1)), 0u};
                    mma_bf16(hsum, a_h, b0, b1);
                    mma_bf16(lsum, a_l, b0, b1);
                }
            }
            // the warp has read its part of the tile: hand the slot back
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.empty[cr.slot]);
            if (++cr.slot == NSLOT) {
                cr.slot = 0;
                cr.phase ^= 1u;
            }
            if (out_kind == OUT_ADD) {  // (uniform) the warp's K slice straight into the buffer
                const int row = r0 + ngw * 8 + 2 * t4;
                if (tile && xok && row - r0 < nr) {
                    float* d = dst + (size_t)gq * dst_stride + row;
                    atomicAdd(d, hsum[0] + lsum[0]);
                    atomicAdd(d + 1, hsum[1] + lsum[1]);
                }
                continue;
            }
            // token gq, rows 2 t4 and 2 t4 + 1 of this warp's row group
            *reinterpret_cast<float2*>(part + (warp * 8 + gq) * 8 + 2 * t4) =
                make_float2(hsum[0] + lsum[0], hsum[1] + lsum[1]);
            cbar();
            if (tile) {
                for (int t = tid; t < M * R; t += NCT) {
                    const int m = t / R, r = t - m * R;
                    if (r >= nr) continue;
                    const int ng = r >> 3, rr = r & 7;
                    float y = 0.f;
#pragma unroll
                    for (int k = 0; k < WK; ++k) y += part[((ng * WK + k) * 8 + m) * 8 + rr];
                    const int row = r0 + r;
                    float* d = dst + (size_t)m * dst_stride + row;
                    if (out_kind == OUT_STORE) {
                        if (n_kc == 1)
                            *d = y;
                        else
                            atomicAdd(d, y);
                    } else if (out_kind == OUT_RESID) {
                        if (n_kc == 1) {
                            const float nv = __ldcg(d) + y;
                            *d = nv;
                            dst2[(size_t)m * dst_stride + row] = nv;
                        } else {
                            atomicAdd(d, y);
                        }
                    } else {  // OUT_ACC
                        *d += y;
                    }
                }
            }
            cbar();  // the partials have been read
        }
        if (p.trace_items && threadIdx.x == 0) trace_rec(c, 0x80000000u | c.cur_code, (unsigned)(tb - ta), ta, tc);
    }
    if (timed_out) {
        ms.abort = 1;
        raise_status(p, ST_TIMEOUT, 0x230u);
    }
    c.set_ring(cr);
    if (dead) c.dead = true;
}

// ---- tensor-core GEMV on K panels of 256 (64 rows per tile, up to 64 tokens) ----
// Each warp owns 8 rows and the whole panel (16 k-steps of mma.sync
// m16n8k16), the tokens in blocks of 16 (A's rows g and g + 8), so a warp's
// sums are final: no partials and no CTA barrier per tile. The B fragments
// (weights, rows 16 bytes apart as in gemv_range_mma) are read once per token
// block; the input fragments come from the staging area as there.
__device__ __forceinline__ void gemv_range_mma_wide(Ctx& c, const Gemv& g, int slot, int j_lo, int j_hi) {
    const Params& p = c.p;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gq = lane >> 2, t4 = lane & 3;
    const int M = c.ms.gm, Kc = g.Kc, SS = stage_stride(Kc), pitch = Kc * 2 + 16, R = g.R;
    const int n_rb = g.n_rb, N = g.N, grp_rows = g.grp_rows, grp_stride = g.grp_stride;
    const int out_kind = g.out_kind, n_kc = g.n_kc, dst_stride = g.dst_stride;
    float* const dst = g.dst + (size_t)slot * g.dst_sstride;
    float* const dst2 = g.dst2;
    const float* src = g.src + (size_t)slot * g.src_sstride;
    Misc& ms = c.ms;
    uint8_t* const ring = c.smem + SMEM_RING;
    const float* const xs = c.stage();
    CRing cr = c.cr;
    bool dead = c.dead, timed_out = false;
    int j = j_lo;
    while (j < j_hi) {
        const int kc0 = j / n_rb, rb0 = j - kc0 * n_rb;
        const int g0 = grp_rows ? (rb0 * R) / grp_rows : 0;
        const int jend = run_end(j, j_hi, n_rb, rb0, R, grp_rows, g0);
        const long long ta = p.trace_items ? gtimer() : 0;
        restage(c, g, src, g0 * grp_stride, kc0, 0, ms.gather ? ms.gm : p.M);
        const long long tb = p.trace_items ? gtimer() : 0;
        long long tc = tb;
        const int jrun = j;
        for (; j < jend; ++j) {
            const int r0 = (rb0 + (j - jrun)) * R, nr = min(R, N - r0);
            const uint8_t* tile = nullptr;
            if (!dead) {
                if (spin_wait(p, &ms.full[cr.slot], cr.phase))
                    tile = ring + cr.slot * SLOT_BYTES;
                else
                    dead = timed_out = true;
            }
            if (p.trace_items && j == jrun) tc = gtimer();
            if (tile) {
                const uint8_t* tr = tile + (size_t)(warp * 8 + gq) * pitch + 4 * t4;
                const int row = r0 + warp * 8 + 2 * t4;  // this lane's output rows: row, row + 1
                for (int mb = 0; mb < M; mb += 16) {
                    const int t0 = mb + gq, t1 = t0 + 8;
                    const bool ok0 = t0 < M, ok1 = t1 < M;
                    const float* x0 = xs + (size_t)(ok0 ? staging_row(ms, t0) : 0) * SS + 2 * t4;
                    const float* x1 = xs + (size_t)(ok1 ? staging_row(ms, t1) : 0) * SS + 2 * t4;
                    float hs[4] = {0.f, 0.f, 0.f, 0.f}, ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                    for (int s2 = 0; s2 < 16; ++s2) {
                        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(tr + 32 * s2);
                        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(tr + 32 * s2 + 16);
                        const float2 z = make_float2(0.f, 0.f);
                        const float2 u0 = ok0 ? *reinterpret_cast<const float2*>(x0 + 16 * s2) : z;
                        const float2 v0 = ok0 ? *reinterpret_cast<const float2*>(x0 + 16 * s2 + 8) : z;
                        const float2 u1 = ok1 ? *reinterpret_cast<const float2*>(x1 + 16 * s2) : z;
                        const float2 v1 = ok1 ? *reinterpret_cast<const float2*>(x1 + 16 * s2 + 8) : z;
                        const uint32_t hu0 = bf2_pack(u0.x, u0.y), hu1 = bf2_pack(u1.x, u1.y);
                        const uint32_t hv0 = bf2_pack(v0.x, v0.y), hv1 = bf2_pack(v1.x, v1.y);
                        const uint32_t a_h[4] = {hu0, hu1, hv0, hv1};
                        const uint32_t a_l[4] = {bf2_pack(u0.x - bf_lo(hu0), u0.y - bf_hi(hu0)),
                                                 bf2_pack(u1.x - bf_lo(hu1), u1.y - bf_hi(hu1)),
                                                 bf2_pack(v0.x - bf_lo(hv0), v0.y - bf_hi(hv0)),
                                                 bf2_pack(v1.x - bf_lo(hv1), v1.y - bf_hi(hv1))};
                        mma_bf16(hs, a_h, b0, b1);
                        mma_bf16(ls, a_l, b0, b1);
                    }
                    // hs[0..1]: token t0, rows row and row + 1; hs[2..3]: token t1
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int m = q < 2 ? t0 : t1, rr = row + (q & 1);
                        if ((q < 2 ? ok0 : ok1) && rr - r0 < nr) {
                            const float y = hs[q] + ls[q];
                            float* d = dst + (size_t)m * dst_stride + rr;
                            if (out_kind == OUT_STORE) {
                                if (n_kc == 1)
                                    *d = y;
                                else
                                    atomicAdd(d, y);
                            } else if (out_kind == OUT_RESID) {
                                if (n_kc == 1) {
                                    const float nv = __ldcg(d) + y;
                                    *d = nv;
                                    dst2[(size_t)m * dst_stride + rr] = nv;
                                } else {
                                    atomicAdd(d, y);
                                }
                            } else {  // OUT_ACC
                                *d += y;
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.empty[cr.slot]);
            if (++cr.slot == NSLOT) {
                cr.slot = 0;
                cr.phase ^= 1u;
            }
        }
        if (p.trace_items && threadIdx.x == 0) trace_rec(c, 0x80000000u | c.cur_code, (unsigned)(tb - ta), ta, tc);
    }
    if (timed_out) {
        ms.abort = 1;
        raise_status(p, ST_TIMEOUT, 0x240u);
    }
    c.set_ring(cr);
    if (dead) c.dead = true;
}

__device__ __noinline__ void gemv_mma(Ctx& c, const Gemv& g, int slot, int j_lo, int j_hi) {
    if (mma_wide(g))
        gemv_range_mma_wide(c, g, slot, j_lo, j_hi);
    else if (g.Kc == 2048)
        gemv_range_mma<1>(c, g, slot, j_lo, j_hi);
    else
        gemv_range_mma<2>(c, g, slot, j_lo, j_hi);
}

// consumer: GEMV work items [j_lo, j_hi) of one slot, two or more tokens:
// split-K path when every token's K panel is staged at once, shared-memory
// path otherwise. A function of
// its own: inlined next to the one-token path, the two would together need
// more registers than a thread has, and spills go to local memory.
__device__ __noinline__ void gemv_multi(Ctx& c, const Gemv& g, int slot, int expert, int j_lo, int j_hi) {
    const int M = c.ms.gm, nks = ks_nks(g.Kc);
    const bool narrow = g.Kc == 128 || g.Kc == 768;  // row slices of 16 / 12 chunks
    // split K (input in registers for the whole run, two tokens at a time)
    // when every token's K panel is staged at once
    const bool ks = M >= 2 && nks > 0 && g.R <= (8 / nks) * (narrow ? 16 : 8) && stage_fits(M, g.Kc);
    if (!ks)
        gemv_range_smem(c, g, slot, expert, j_lo, j_hi);
    else if (narrow)
        gemv_range_ks<16, 2>(c, g, slot, expert, j_lo, j_hi);
    else
        gemv_range_ks<32, 2>(c, g, slot, expert, j_lo, j_hi);
}

// consumer: GEMV work items [j_lo, j_hi) of one slot (one copy of the GEMV
// code for the plain stages and the expert units: every stage's code runs
// once per layer, and a smaller footprint keeps it in the instruction cache)
__device__ __noinline__ void cons_gemv(Ctx& c, const Gemv& g, int slot, int expert, int j_lo, int j_hi) {
    const int M = c.ms.gm, Kc = g.Kc;
    // K panels of 2048 and 1024: the register path also for 2 to 4 tokens
    // (each tile once per token)
    const bool mt = M >= 2 && M <= 4 && g.out_kind != OUT_SCALED;
    if (mma_gemv(M, g))
        gemv_mma(c, g, slot, j_lo, j_hi);
    else if (M == 1 && Kc == 2048)
        gemv_range_rx<8>(c, g, slot, expert, j_lo, j_hi);
    else if (mt && Kc == 2048)
        gemv_range_rx<8, true>(c, g, slot, expert, j_lo, j_hi);
    else if (M == 1 && Kc == 1024)
        gemv_range_rx<4>(c, g, slot, expert, j_lo, j_hi);
    else if (mt && Kc == 1024)
        gemv_range_rx<4, true>(c, g, slot, expert, j_lo, j_hi);
    else if (M == 1 && Kc == 768)
        gemv_range_rx<3>(c, g, slot, expert, j_lo, j_hi);
    else if (M == 1 && Kc == 512)
        gemv_range_rx<2>(c, g, slot, expert, j_lo, j_hi);
    else if (M == 1 && Kc == 256)
        gemv_range_rx<1>(c, g, slot, expert, j_lo, j_hi);
    else if (M == 1 && Kc == 128)
        gemv_range_rx<0>(c, g, slot, expert, j_lo, j_hi);
    else
        gemv_multi(c, g, slot, expert, j_lo, j_hi);
    if (*(volatile int*)&c.ms.abort) c.dead = true;
}

// producer: bulk-load the weight tiles of items [lo, hi) (one slot). All
// descriptor fields and the ring state live in registers for the loop.
// L2 prefetch of weight tiles [lo, hi) of one slot (one lane per tile)
__device__ __forceinline__ void prefetch_tiles(const Gemv& g, int expert, int lo, int hi) {
    const uint16_t* W = g.W + (expert >= 0 ? (size_t)expert * g.w_estride : 0);
    for (int j = lo + (int)(threadIdx.x & 31); j < hi; j += 32) {
        const int kc = j / g.n_rb, rb = j - kc * g.n_rb;
        const int r0 = rb * g.R, nr = min(g.R, g.N - r0);
        l2_prefetch(W + (size_t)kc * g.N * g.Kc + (size_t)r0 * g.Kc, (unsigned)nr * g.Kc * 2u);
    }
}

#ifndef MK_PF_TILES
#define MK_PF_TILES 8
#endif
#ifndef MK_UNIT_PF_BYTES
#define MK_UNIT_PF_BYTES (640 * 1024)
#endif
constexpr int PF_TILES = MK_PF_TILES;            // L2 prefetch distance beyond the ring, in tiles
constexpr int UNIT_PF_BYTES = MK_UNIT_PF_BYTES;  // expert units: L2 prefetch up front, per CTA

// producer: bulk-load the weight tiles of items [lo, hi) (one slot); tiles a
// tensor-core GEMV of `ntok` tokens reads (mma_gemv) are copied row by row
// into rows Kc*2 + 16 bytes apart. All descriptor fields and the ring state
// live in registers for the loop.
__device__ __noinline__ void prod_gemv(Ctx& c, const Gemv& g, int expert, int lo, int hi, int ntok) {
    const uint16_t* W = g.W + (expert >= 0 ? (size_t)expert * g.w_estride : 0);
    const int n_rb = g.n_rb, R = g.R, N = g.N, Kc = g.Kc;
    const Params& p = c.p;
    Misc& ms = c.ms;
    uint8_t* ring = c.smem + SMEM_RING;
    PRing pr = c.pr;
    int issued = c.issued;
    const int lane = threadIdx.x & 31;
    const bool leader = lane == 0;
    const bool pad = mma_gemv(ntok, g);
    const unsigned long long pol = l2_evict_first();
    // panel / row block of item j and of item j + PF_TILES, advanced per item;
    // the window's first tiles go towards L2 after the first copy is issued
    int kc = lo / n_rb, rb = lo - kc * n_rb;
    int kp = (lo + PF_TILES) / n_rb, rbp = lo + PF_TILES - kp * n_rb;
    for (int j = lo; j < hi; ++j) {
        const int r0 = rb * R, nr = min(R, N - r0);
        const unsigned bytes = (unsigned)nr * Kc * 2u;
        const uint16_t* src = W + (size_t)kc * N * Kc + (size_t)r0 * Kc;
        if (leader && j + PF_TILES < hi) {
            const int rp = rbp * R;
            l2_prefetch(W + (size_t)kp * N * Kc + (size_t)rp * Kc, (unsigned)min(R, N - rp) * Kc * 2u);
        }
        if (++rb == n_rb) {
            rb = 0;
            ++kc;
        }
        if (++rbp == n_rb) {
            rbp = 0;
            ++kp;
        }
        if (p.debug && (pad ? (unsigned)nr * (Kc * 2 + 16) : bytes) > (unsigned)(SLOT_BYTES - 16)) {
            // (debug mode: a tile that would overrun its ring slot)
            if (leader) raise_status(p, ST_DEBUG, 0x9210u);
            c.dead = true;
            break;
        }
        int ok = 1;
        if (leader) {
            if (spin_wait(p, &ms.empty[pr.slot], pr.phase ^ 1u)) {
                mbar_expect_tx(&ms.full[pr.slot], bytes);
                if (!pad) bulk_g2s_pol(ring + pr.slot * SLOT_BYTES, src, bytes, &ms.full[pr.slot], pol);
            } else {
                ok = 0;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (leader) raise_status(p, ST_TIMEOUT, 0x110u);
            c.dead = true;
            break;
        }
        if (pad)  // one copy per row (nr <= 64 rows: at most two per lane)
            for (int r = lane; r < nr; r += 32)
                bulk_g2s_pol(ring + pr.slot * SLOT_BYTES + (size_t)r * (Kc * 2 + 16), src + (size_t)r * Kc,
                             (unsigned)Kc * 2u, &ms.full[pr.slot], pol);
        __syncwarp();
        ++issued;
        prod_next(pr);
        if (j == lo) prefetch_tiles(g, expert, lo + 1, min(hi, lo + PF_TILES));
    }
    c.set_pring(pr, issued);
}

// consumers, output projection with the router folded in (one K panel, so
// this CTA's rows [R lo, R hi) of the new residual are final after its
// GEMV): their share of every token's router logits, sum_i Wr[e][i] g[i] x[i]
// (the 1/rms factor is applied by the reader), and of the sum of squares of
// x, added into this CTA's copy of the layer's accumulators (vector
// reductions, one per 4 floats). The accumulators start at zero (cleared at
// the start of the step) and are complete when every item of the output
// projection has been signalled.
__device__ __noinline__ void router_part(Ctx& c, int l, const Gemv& go, int lo, int hi) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const Gemv& gr = Ld.g[G_ROUTER];
    const int r_lo = lo * go.R, nr = min(go.N, hi * go.R) - r_lo;  // a multiple of 8
    const int E = p.E, M = p.M, tid = ctid(), Kc = gr.Kc, RS = router_row(E);
    // the staging area is reused as scratch; its recorded key stays that of
    // the output projection's input, a per-layer buffer no later GEMV reads
    float* xg = c.stage();            // [M][nr] x g
    float* xs = xg + M * nr;          // [M][nr] x
    float* sums = xs + M * nr;        // [M][RS]
    cbar();                           // this CTA's stores of the rows are visible to all its threads
    for (int i = tid; i < M * nr; i += NCT) {
        const int m = i / nr, r = i - m * nr;
        const float x = __ldcg(go.dst + (size_t)m * go.dst_stride + r_lo + r);
        xg[i] = x * bf2f(gr.gain[r_lo + r]);
        xs[i] = x;
    }
    for (int i = tid; i < M * RS; i += NCT) sums[i] = 0.f;
    cbar();
    // thread: expert e, 8-row groups sub, sub + 4, ...; tokens 8 at a time
    const int sub = tid & 3, ng = nr >> 3;
    for (int e0 = 0; e0 < E; e0 += NCT / 4) {
        const int e = e0 + (tid >> 2);
        for (int m0 = 0; m0 < M; m0 += 8) {
            float s[8], s2[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) s[t] = s2[t] = 0.f;
            if (e < E) {
                for (int q = sub; q < ng; q += 4) {
                    const int i = r_lo + 8 * q, kc = i / Kc;
                    const uint4 w = *reinterpret_cast<const uint4*>(gr.W + ((size_t)kc * E + e) * Kc + (i - kc * Kc));
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        if (m0 + t < M) {
                            const float4* xm = reinterpret_cast<const float4*>(xg + (m0 + t) * nr + 8 * q);
                            fma8v2(s[t], s2[t], w, xm[0], xm[1]);
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (m0 + t < M) {
                    float v = s[t] + s2[t];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    if (sub == 0 && e < E) sums[(m0 + t) * RS + e] = v;
                }
            }
        }
    }
    // sums of squares: warp w takes tokens w, w + NCW, ...
    const int lane = tid & 31;
    for (int m = tid >> 5; m < M; m += NCW) {
        float q = 0.f;
        for (int r = lane; r < nr; r += 32) {
            const float x = xs[m * nr + r];
            q = fmaf(x, x, q);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
        if (lane == 0) sums[m * RS + E] = q;
    }
    cbar();
    float* acc = p.racc + ((size_t)l * ROUTER_COPIES + blockIdx.x % ROUTER_COPIES) * M * RS;
    for (int i = 4 * tid; i < M * RS; i += 4 * NCT) {
        const float4 v = *reinterpret_cast<const float4*>(sums + i);
        asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(acc + i), "f"(v.x), "f"(v.y),
                     "f"(v.z), "f"(v.w)
                     : "memory");
    }
}

// consumer side of a GEMV stage: items [lo, hi) of g after the deps set by
// set_deps, then signal `sig` (the GEMV code, cons_gemv, is shared with the
// expert units).
// RMSNorm input whose K panels are parts of the row, several tokens: the
// stage's np CTAs (this one has rank `rank`) each sum the squares of one
// slice of the M x K input (128-float blocks, a few KB), add them into the
// step's per-row accumulators and meet at a counter; every CTA then holds
// the whole rows' sums and stages only its panels (instead of every CTA
// reading every row: 458 KB at 56 tokens x 2048)
__device__ __noinline__ void rms_prepass(Ctx& c, int l, const Gemv& g, int sig, int rank, int np) {
    const Params& p = c.p;
    const int site = sig == C_QB ? 1 : (sig == C_ROUTER ? 2 : 0);
    float* const acc = p.rss + ((size_t)l * 3 + site) * p.rss_mx;
    const int tid = ctid(), lane = tid & 31, warp = tid >> 5, K = g.K;
    const int nb = (p.M * K) >> 7, b0 = (int)((long long)rank * nb / np), b1 = (int)((long long)(rank + 1) * nb / np);
    for (int b = b0 + warp; b < b1; b += NCW) {
        const int i = (b << 7) + lane * 4, t = i / K;  // a block lies in one row (K is a multiple of 128)
        const float4 v = __ldcg(reinterpret_cast<const float4*>(g.src + (size_t)t * g.src_stride + (i - t * K)));
        float part = v.x * v.x;
        part = fmaf(v.y, v.y, part);
        part = fmaf(v.z, v.z, part);
        part = fmaf(v.w, v.w, part);
#pragma unroll
        for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) atomicAdd(acc + t, part);
    }
    // every CTA's additions are done before its arrival (the barrier orders the
    // other threads' atomics before thread 0's release, which is cumulative)
    cbar();
    unsigned* const arr = ctr_of(p, l, C_NRM0 + site);
    if (threadIdx.x == 0 && !c.dead) {
        red_release(arr, 1u);
        if (!wait_ge(p, arr, (unsigned)np, 0x1500u | (unsigned)(l << 16) | (unsigned)site)) c.ms.abort = 1;
    }
    cbar();
    if (*(volatile int*)&c.ms.abort) c.dead = true;
    if (tid < p.M) c.ms.rms[tid] = __ldcg(acc + tid);
    c.rms_src = g.src;  // (each warp's own state; restage's barrier orders the rms values)
}

__device__ __noinline__ void cons_mm(Ctx& c, int l, const Gemv& g, int sig, int lo, int hi) {
    c.cur_code = ((unsigned)sig << 16) | (unsigned)l;
    const long long t0 = gtimer();
    cwait(c, 0x1000u | (unsigned)(l << 16) | (unsigned)sig);
    const long long t1 = gtimer();
    const bool pre = c.p.rss && !c.p.staged && g.in_kind == IN_RMS && g.n_kc > 1 && c.p.M >= 2 && !c.dead;
    if (pre) rms_prepass(c, l, g, sig, c.st_rank, c.st_np);
    cons_gemv(c, g, 0, -1, lo, hi);
    c.rms_src = nullptr;
    if (sig == C_O && c.p.rfuse && !c.dead) router_part(c, l, g, lo, hi);
    if (sig == C_A && (c.p.qfuse || c.p.ufuse)) {
        // buffers of layer l that later stages add into with reductions: the
        // QB CTAs' absorbed queries (q_lat), the combine CTAs' value
        // up-projection (o); every CTA (each has A items) clears its share
        // before signalling A
        const int gt = (int)blockIdx.x * NCT + ctid(), gs = c.p.G * NCT;
        if (c.p.qfuse) {
            float4* q = reinterpret_cast<float4*>(const_cast<float*>(c.layer().qlat));
            const int n4 = c.p.M * MLA_H * MLA_KL / 4;
            for (int i = gt; i < n4; i += gs) q[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (c.p.ufuse) {
            float4* o = reinterpret_cast<float4*>(c.layer().o);
            const int n4 = c.p.M * MLA_H * c.p.vd / 4;
            for (int i = gt; i < n4; i += gs) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    csignal(c, l, sig, (unsigned)(hi - lo));
    trace_rec(c, ((unsigned)sig << 16) | (unsigned)l, (unsigned)(hi - lo), t0, t1);
}

// ---- the absorbed query folded into QB (MLA, all tokens' c_q staged) ----
// q_lat[h] = q_nope[h] . W_uk[h] is a sum over the 128 nope dimensions of
// head h. A QB tile of R nope rows of head h (R = 16) yields q_nope for those
// dimensions; the CTA multiplies them at once by the same R rows of W_uk[h]
// (a slab of R x 512, streamed into the ring right after the tile) and adds
// the product into q_lat with vector reductions. q_lat is cleared by the A
// stage, so the attention waits only for QB: one dependent stage fewer.
__device__ __noinline__ void qb_fused_cons(Ctx& c, int l, int lo, int hi) {
    const Params& p = c.p;
    c.cur_code = ((unsigned)C_QB << 16) | (unsigned)l;
    const long long t0 = gtimer();
    cwait(c, 0x1000u | (unsigned)(l << 16) | (unsigned)C_QB);
    const long long t1 = gtimer();
    const Layer& Ld = c.layer();
    const Gemv& g = Ld.g[G_QB];
    const int M = p.M, qh = p.nope + p.rd, R = g.R, tid = ctid();
    // [M][R] a nope tile's outputs, in the upper half of the reduction area
    // (the split-K GEMV uses the lower half)
    float* qv = c.red() + RED_FLOATS / 2;
    // every warp runs every iteration and every barrier (a warp that saw an
    // abort skips the work, not the barriers: its copy of `dead` may differ
    // from the other warps')
    for (int j = lo; j < hi; ++j) {
        const int r0 = j * R, h = r0 / qh, i0 = r0 - h * qh;
        if (i0 >= p.nope) {  // rope rows: the attention reads them from q
            cons_gemv(c, g, 0, -1, j, j + 1);
            continue;
        }
        // nope rows: the same GEMV with its outputs going to qv (only this
        // CTA reads them)
        if (tid == 0) {
            c.ms.ug = g;
            c.ms.ug.dst = qv - r0;
            c.ms.ug.dst_stride = R;
        }
        cbar();
        cons_gemv(c, c.ms.ug, 0, -1, j, j + 1);
        cbar();  // every warp's outputs of the tile are in qv
        const uint8_t* slab = c.dead ? nullptr : cons_wait(p, c.smem, c.ms, c.cr);
        if (slab) {
            // thread: latent columns 2 tid, 2 tid + 1 (512 = 2 NCT)
            const uint32_t* W = reinterpret_cast<const uint32_t*>(slab) + tid;
            float* ql = const_cast<float*>(Ld.qlat) + (size_t)h * MLA_KL + 2 * tid;
            for (int m = 0; m < M; ++m) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
                for (int r = 0; r < R; ++r) {
                    const uint32_t w = W[(size_t)r * (MLA_KL / 2)];
                    const float x = qv[m * R + r];
                    a0 = fmaf(x, bf_lo(w), a0);
                    a1 = fmaf(x, bf_hi(w), a1);
                }
                asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" ::"l"(ql + (size_t)m * MLA_H * MLA_KL),
                             "f"(a0), "f"(a1)
                             : "memory");
            }
        }
        cons_release(c.ms, c.cr);  // every warp's ring state advances alike
        if (*(volatile int*)&c.ms.abort) c.dead = true;
    }
    csignal(c, l, C_QB, (unsigned)(hi - lo));
    trace_rec(c, ((unsigned)C_QB << 16) | (unsigned)l, (unsigned)(hi - lo), t0, t1);
}

// producer side: each QB tile, and after a tile of nope rows its W_uk slab
__device__ __noinline__ void qb_fused_prod(Ctx& c, int lo, int hi) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const Gemv& g = Ld.g[G_QB];
    const int qh = p.nope + p.rd, R = g.R;
    for (int j = lo; j < hi && !c.dead; ++j) {
        prod_gemv(c, g, -1, j, j + 1, p.M);
        const int r0 = j * R, h = r0 / qh, i0 = r0 - h * qh;
        if (c.dead || i0 >= p.nope) continue;
        const unsigned bytes = (unsigned)R * MLA_KL * 2u;
        int ok = 1;
        if ((threadIdx.x & 31) == 0) {
            uint8_t* dst = prod_begin(p, c.smem, c.ms, c.pr, bytes);
            if (dst)
                bulk_g2s(dst, Ld.uk + ((size_t)h * p.nope + i0) * MLA_KL, bytes, &c.ms.full[c.pr.slot]);
            else
                ok = 0;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            c.dead = true;
            return;
        }
        c.bump_issued();
        prod_next(c.pr);
    }
}

// ============================================================ routing ====
// one more token routed to expert e (8-bit counts, added through their word)
__device__ __forceinline__ void count_token(uint8_t* cnt, int e) {
    atomicAdd(reinterpret_cast<unsigned*>(cnt + (e & ~3)), 1u << (8 * (e & 3)));
}

// routed expert units (slot-major, nu per slot) over gc CTAs by expected
// time: a unit of an expert with t tokens weighs 5 + 4 (t - 1). CTA ci takes
// the units whose start weight s satisfies ci W <= s gc < (ci + 1) W, a
// contiguous range [lo, hi). Every warp computes it alike (no shared state).
__device__ __forceinline__ int routed_first(const uint8_t* cnt, const uint8_t* slot_e, int nslots, int nu, long long T,
                                            int gc) {
    const int lane = threadIdx.x & 31;
    long long base = 0;  // start weight of the chunk's first slot
    for (int s0 = 0; s0 < nslots; s0 += 32) {
        const int s = s0 + lane;
        const int wu = s < nslots ? 5 + 4 * ((int)cnt[slot_e[s]] - 1) : 0;
        long long inc = (long long)wu * nu;  // inclusive scan of the slot weights
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        const long long S = base + inc - (long long)wu * nu;  // this slot's start
        // the slot holds the first unit at or past T when its last unit does
        const bool hit = s < nslots && (S + (long long)(nu - 1) * wu) * gc >= T;
        const unsigned b = __ballot_sync(0xffffffffu, hit);
        if (b) {
            const int src = __ffs(b) - 1;
            const long long Ss = __shfl_sync(0xffffffffu, S, src);
            const int w = __shfl_sync(0xffffffffu, wu, src);
            const long long need = T - Ss * gc;  // first u with (Ss + u w) gc >= T
            const int u = need <= 0 ? 0 : (int)((need + (long long)w * gc - 1) / ((long long)w * gc));
            return (s0 + src) * nu + u;
        }
        base += __shfl_sync(0xffffffffu, inc, 31);
    }
    return nslots * nu;
}

__device__ __forceinline__ void routed_range(const uint8_t* cnt, const uint8_t* slot_e, int nslots, int nu, int ci,
                                             int gc, int& lo, int& hi) {
    const int lane = threadIdx.x & 31;
    long long W = 0;
    for (int s = lane; s < nslots; s += 32) W += (long long)(5 + 4 * ((int)cnt[slot_e[s]] - 1)) * nu;
#pragma unroll
    for (int o = 16; o; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    if (ci < 0 || ci >= gc) {
        lo = hi = 0;
        return;
    }
    lo = routed_first(cnt, slot_e, nslots, nu, (long long)ci * W, gc);
    hi = routed_first(cnt, slot_e, nslots, nu, (long long)(ci + 1) * W, gc);
}
// softmax / top-k of the router logits of every token (ties -> lower id),
// union of the selected experts (sorted by id) -> routed slots.
// consumers: full routing into Misc; producer warp: slot list only.
template <bool PROD>
__device__ __forceinline__ bool route(Ctx& c, int l) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const int E = p.E, k = p.topk;
    const int tid = threadIdx.x, lane = tid & 31;
    uint8_t* used = PROD ? c.ms.p_used : c.ms.used;
    uint8_t* slot_e = PROD ? c.ms.p_slot_e : c.ms.slot_e;
    if constexpr (PROD) {
        int ok = 1;
        if (lane == 0) {
            ok = p.rfuse ? wait_ge(p, ctr_of(p, l, C_O), (unsigned)gemv_items(Ld.g[G_O]), 0x300u)
                         : wait_ge(p, ctr_of(p, l, C_ROUTER), (unsigned)gemv_items(Ld.g[G_ROUTER]), 0x300u);
            __threadfence();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        if (!ok) {
            c.dead = true;
            return false;
        }
        for (int e = lane; e < E; e += 32) used[e] = 0;
        __syncwarp();
    } else {
        const long long t0 = gtimer();
        set_deps(c, p.rfuse ? deps1(l, C_O, (unsigned)gemv_items(Ld.g[G_O]))
                            : deps1(l, C_ROUTER, (unsigned)gemv_items(Ld.g[G_ROUTER])));
        cwait(c, 0x400u);
        trace_rec(c, (0x40u << 16) | (unsigned)l, 0u, t0, gtimer());
        for (int e = tid; e < E; e += NCT) used[e] = 0;
        cbar();
    }
    const int warp = PROD ? 0 : (tid >> 5);
    const int nw = PROD ? 1 : NCW;
    for (int m = warp; m < p.M; m += nw) {
        float v[MAX_E / 32];
        const int RS = router_row(E);
        const float* lg = (p.rfuse ? p.racc + (size_t)l * ROUTER_COPIES * p.M * RS : Ld.rlog) + (size_t)m * RS;
#pragma unroll
        for (int i = 0; i < MAX_E / 32; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? __ldcg(lg + e) : -INFINITY;
        }
        if (p.rfuse) {
            // accumulated logits: the sum over the copies, times 1/rms of the
            // residual (mean square over d)
            // (each batch of loads issued together: one L2 round trip per batch)
            const size_t cs = (size_t)p.M * RS;
            float q[ROUTER_COPIES];
#pragma unroll
            for (int cp = 0; cp < ROUTER_COPIES; ++cp) q[cp] = __ldcg(lg + cp * cs + E);
            float ss = 0.f;
#pragma unroll
            for (int cp = 0; cp < ROUTER_COPIES; ++cp) ss += q[cp];
#pragma unroll
            for (int i = 0; i < MAX_E / 32; ++i) {
                if (32 * i < E) {
                    const int e = lane + 32 * i;
#pragma unroll
                    for (int cp = 1; cp < ROUTER_COPIES; ++cp) q[cp] = e < E ? __ldcg(lg + cp * cs + e) : 0.f;
#pragma unroll
                    for (int cp = 1; cp < ROUTER_COPIES; ++cp) v[i] += q[cp];
                }
            }
            const float sc = 1.0f / sqrtf(ss * (1.0f / (float)p.d) + p.eps);
#pragma unroll
            for (int i = 0; i < MAX_E / 32; ++i) v[i] *= sc;
        }
        if (E <= 64 && !__any_sync(0xffffffffu, v[0] != v[0] || v[1] != v[1])) {
            // up to 64 experts: each lane ranks its two logits against all
            // others (greater value, or equal value and lower id, ranks
            // first) -- independent shuffles instead of k dependent argmax
            // rounds; the selected experts are those of rank < k
            int rk[2] = {0, 0};
#pragma unroll 4
            for (int sl = 0; sl < 32; ++sl) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float ov = __shfl_sync(0xffffffffu, v[i], sl);
                    const int oe = sl + 32 * i;
#pragma unroll
                    for (int q = 0; q < 2; ++q) rk[q] += (ov > v[q] || (ov == v[q] && oe < lane + 32 * q)) ? 1 : 0;
                }
            }
            // renormalised top-k probabilities = softmax over the selected
            // logits; the largest logit (rank 0) is the largest of all
            float mx = fmaxf(v[0], v[1]);
#pragma unroll
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float ex[2], den = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const bool s = rk[q] < k && lane + 32 * q < E;
                ex[q] = s ? expf(v[q] - mx) : 0.f;
                den += ex[q];
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
            if (!PROD && blockIdx.x == 0 && p.dbg_margin) {
                // router margin of this token: the k-th largest logit minus
                // the (k+1)-th (the values of ranks k - 1 and k)
                float a = -INFINITY, b = -INFINITY;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (lane + 32 * q < E) {
                        if (rk[q] == k - 1) a = v[q];
                        if (rk[q] == k) b = v[q];
                    }
                }
#pragma unroll
                for (int o = 16; o; o >>= 1) {
                    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
                    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
                }
                if (lane == 0) p.dbg_margin[(size_t)l * p.M + m] = k < E ? a - b : INFINITY;
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int e = lane + 32 * q;
                if (rk[q] < k && e < E) {
                    count_token(used, e);
                    if constexpr (!PROD) {
                        c.ms.ridx[m][rk[q]] = (uint8_t)e;
                        c.ms.rw[m][rk[q]] = ex[q] / den;
                        if (blockIdx.x == 0 && p.dbg_idx) {
                            const size_t o = ((size_t)l * p.M + m) * k + rk[q];
                            p.dbg_idx[o] = e;
                            p.dbg_w[o] = ex[q] / den;
                        }
                    }
                }
            }
            continue;
        }
        float sel[MAX_K];
        int sid[MAX_K];
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < MAX_E / 32; ++i) {
                const int e = lane + 32 * i;
                if (e < E && (v[i] > bv || (v[i] == bv && e < bi))) {
                    bv = v[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (bi >= E) {  // NaN logits (only after a failed step): keep ids in range
                bi = j;
                bv = 0.f;
            }
            sel[j] = bv;
            sid[j] = bi;
#pragma unroll
            for (int i = 0; i < MAX_E / 32; ++i)
                if (lane + 32 * i == bi) v[i] = -INFINITY;
        }
        if (!PROD && blockIdx.x == 0 && p.dbg_margin) {
            // router margin: the k-th selected logit minus the largest one left
            float bv = -INFINITY;
#pragma unroll
            for (int i = 0; i < MAX_E / 32; ++i)
                if (lane + 32 * i < E) bv = fmaxf(bv, v[i]);
#pragma unroll
            for (int o = 16; o; o >>= 1) bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, o));
            if (lane == 0) p.dbg_margin[(size_t)l * p.M + m] = k < E ? sel[k - 1] - bv : INFINITY;
        }
        if (lane == 0) {
            // renormalised top-k probabilities = softmax over the selected logits
            float den = 0.f, w[MAX_K];
            for (int j = 0; j < k; ++j) {
                w[j] = expf(sel[j] - sel[0]);
                den += w[j];
            }
            for (int j = 0; j < k; ++j) {
                count_token(used, sid[j]);
                if constexpr (!PROD) {
                    c.ms.ridx[m][j] = (uint8_t)sid[j];
                    c.ms.rw[m][j] = w[j] / den;
                    if (blockIdx.x == 0 && p.dbg_idx) {
                        const size_t o = ((size_t)l * p.M + m) * k + j;
                        p.dbg_idx[o] = sid[j];
                        p.dbg_w[o] = w[j] / den;
                    }
                }
            }
        }
    }
    if constexpr (PROD) {
        __syncwarp();
    } else {
        cbar();
    }
    if (PROD || tid < 32) {
        int n = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const bool u = e < E && used[e];
            const unsigned b = __ballot_sync(0xffffffffu, u);
            if (u) slot_e[n + __popc(b & ((1u << lane) - 1u))] = (uint8_t)e;
            n += __popc(b);
        }
        if (lane == 0) {
            if (PROD)
                c.ms.p_nslots = n;
            else
                c.ms.n_slots = n;
        }
    }
    if constexpr (PROD) {
        __syncwarp();
    } else {
        cbar();
    }
    return true;
}

// ====================================================== GQA attention ====
// item (sequence b, kv head g, split s) over units [u_lo, u_hi): prefix
// chunks of 64 cached positions (from the ring) and, in the last split, the T
// new positions (computed here, appended to the cache, read from smem).
// Output: unnormalised partial (max, sum, o[hd]) per query row t*Gq + hh.

// reduce 32 values across the warp: lane i returns the sum of value i
__device__ __forceinline__ float reduce_scatter32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int o = 16 >> step;
        const int n = 16 >> step;
        const bool up = lane & o;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = up ? v[i] : v[i + n];
            const float keep = up ? v[i + n] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

template <int DPL>
struct GqaState {
    float m[8], l[8], o[8][DPL];
};

// one warp's share (rows [base, base+8)) of a block of K/V rows
template <int DPL, bool TAIL>
__device__ void gqa_rows(const Params& p, GqaState<DPL>& st, const float (&q)[8][DPL], int Q, const void* Kp,
                         const void* Vp, int base, int nvalid, int tailT, float* sc) {
    const int lane = threadIdx.x & 31, hd = p.hd, Gq = p.Hq / p.Hkv;
    // partial dot products of this lane's DPL dims for rows base..base+7
    for (int half = 0; half < (Q > 4 ? 2 : 1); ++half) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
        const int r0 = half * 4;  // query rows r0..r0+3 (Q > 4) or all rows (Q <= 4)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = base + j;
            if (row < nvalid) {
                float kv[DPL];
                if (TAIL) {
                    const float* K = reinterpret_cast<const float*>(Kp) + (size_t)row * hd + lane * DPL;
#pragma unroll
                    for (int e = 0; e < DPL; ++e) kv[e] = K[e];
                } else {
                    const uint16_t* K = reinterpret_cast<const uint16_t*>(Kp) + (size_t)row * hd + lane * DPL;
#pragma unroll
                    for (int e = 0; e < DPL; ++e) kv[e] = bf2f(K[e]);
                }
                if (Q <= 4) {
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        float a = 0.f;
#pragma unroll
                        for (int e = 0; e < DPL; ++e) a = fmaf(q[qq][e], kv[e], a);
                        v[j * 4 + qq] = a;
                    }
                } else {
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        float a = 0.f;
#pragma unroll
                        for (int e = 0; e < DPL; ++e) a = fmaf(q[r0 + qq][e], kv[e], a);
                        v[j * 4 + qq] = a;
                    }
                }
            }
        }
        const float s = reduce_scatter32(v);
        sc[half * 32 + lane] = s;
    }
    __syncwarp();
    // online softmax per query row over this warp's rows
#pragma unroll 1
    for (int qr = 0; qr < Q; ++qr) {
        const int t = qr / Gq;
        float sv[8];
        float mc = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = base + j;
            bool ok = row < nvalid && (!TAIL || row <= t);
            const int idx = Q <= 4 ? (j * 4 + qr) : ((qr >> 2) * 32 + j * 4 + (qr & 3));
            sv[j] = ok ? sc[idx] : -INFINITY;
            mc = fmaxf(mc, sv[j]);
        }
        if (mc == -INFINITY) continue;
        const float mn = fmaxf(st.m[qr], mc);
        const float corr = st.m[qr] == -INFINITY ? 0.f : expf(st.m[qr] - mn);
        float ps = 0.f;
        float acc[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = st.o[qr][e] * corr;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (sv[j] == -INFINITY) continue;
            const float pj = expf(sv[j] - mn);
            ps += pj;
            const int row = base + j;
            if (TAIL) {
                const float* V = reinterpret_cast<const float*>(Vp) + (size_t)row * hd + lane * DPL;
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[e] = fmaf(pj, V[e], acc[e]);
            } else {
                const uint16_t* V = reinterpret_cast<const uint16_t*>(Vp) + (size_t)row * hd + lane * DPL;
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[e] = fmaf(pj, bf2f(V[e]), acc[e]);
            }
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) st.o[qr][e] = acc[e];
        st.l[qr] = st.l[qr] * corr + ps;
        st.m[qr] = mn;
    }
    __syncwarp();
}

template <int DPL>
__device__ __forceinline__ void cons_attn_gqa(Ctx& c, int l, const AttnItem& it) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const int hd = p.hd, Gq = p.Hq / p.Hkv, T = p.T, Q = T * Gq, half = hd / 2;
    const int tid = ctid(), lane = tid & 31, warp = tid >> 5;
    const int b = it.b, g = it.g, pos0 = p.pos[b];
    const bool tail = it.u_hi == it.nch + 1;
    float* qs = c.stage();             // [Q][hd]
    float* tk = qs + Q * hd;           // [T][hd] new keys (bf16-rounded)
    float* tv = tk + T * hd;           // [T][hd]
    float* sc = tv + T * hd;           // [NCW][64]
    float* ws = sc + NCW * 64;         // [NCW][Q][2 + hd]
    cbar();
    c.sk_src = nullptr;
    const int a_stride = Ld.a_stride;
    for (int i = tid; i < Q * half; i += NCT) {
        const int qr = i / half, e = i - qr * half;
        const int t = qr / Gq, h = g * Gq + (qr - t * Gq);
        const float* qa = Ld.a + (size_t)(b * T + t) * a_stride + h * hd;
        const float2 cs = p.rope[(size_t)(pos0 + t) * p.rope_half + e];
        const float x0 = __ldcg(qa + e), x1 = __ldcg(qa + e + half);
        qs[qr * hd + e] = (x0 * cs.x - x1 * cs.y) * p.attn_scale;
        qs[qr * hd + e + half] = (x1 * cs.x + x0 * cs.y) * p.attn_scale;
    }
    if (tail) {
        uint16_t* pool = p.kv_pool + (size_t)l * p.kv_layer_elems;
        for (int i = tid; i < T * half; i += NCT) {
            const int t = i / half, e = i - t * half;
            const int pos = pos0 + t;
            const float* ka = Ld.a + (size_t)(b * T + t) * a_stride + p.Hq * hd + g * hd;
            const float* va = ka + p.Hkv * hd;
            const float2 cs = p.rope[(size_t)pos * p.rope_half + e];
            const float x0 = __ldcg(ka + e), x1 = __ldcg(ka + e + half);
            const uint16_t k0 = f2bf(x0 * cs.x - x1 * cs.y), k1 = f2bf(x1 * cs.x + x0 * cs.y);
            const uint16_t v0 = f2bf(__ldcg(va + e)), v1 = f2bf(__ldcg(va + e + half));
            tk[t * hd + e] = bf2f(k0);
            tk[t * hd + e + half] = bf2f(k1);
            tv[t * hd + e] = bf2f(v0);
            tv[t * hd + e + half] = bf2f(v1);
            // append to the page: [Hkv][K|V][64][hd]
            uint16_t* pg = pool + (size_t)p.btab[b * p.pps + pos / PAGE] * p.page_elems +
                           (size_t)g * 2 * PAGE * hd + (size_t)(pos % PAGE) * hd;
            pg[e] = k0;
            pg[e + half] = k1;
            pg[(size_t)PAGE * hd + e] = v0;
            pg[(size_t)PAGE * hd + e + half] = v1;
        }
    }
    cbar();
    float qreg[8][DPL];
#pragma unroll
    for (int qr = 0; qr < 8; ++qr)
#pragma unroll
        for (int e = 0; e < DPL; ++e) qreg[qr][e] = qr < Q ? qs[qr * hd + lane * DPL + e] : 0.f;
    GqaState<DPL> st;
#pragma unroll
    for (int qr = 0; qr < 8; ++qr) {
        st.m[qr] = -INFINITY;
        st.l[qr] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) st.o[qr][e] = 0.f;
    }
    for (int u = it.u_lo; u < it.u_hi; ++u) {
        if (u < it.nch) {
            const uint8_t* tile = c.dead ? nullptr : cons_wait(p, c.smem, c.ms, c.cr);
            if (tile) {
                const int nvalid = min(GQA_CH, pos0 - u * GQA_CH);
                gqa_rows<DPL, false>(p, st, qreg, Q, tile, tile + (size_t)GQA_CH * hd * 2, warp * 8, nvalid, 0,
                                     sc + warp * 64);
            }
            cons_release(c.ms, c.cr);
        } else if (warp == 0) {
            gqa_rows<DPL, true>(p, st, qreg, Q, tk, tv, 0, T, T, sc);
        }
    }
    // merge the 8 warps' states
    const int W = 2 + hd;
    for (int qr = 0; qr < Q; ++qr) {
        float* w = ws + ((size_t)warp * Q + qr) * W;
        if (lane == 0) {
            w[0] = st.m[qr];
            w[1] = st.l[qr];
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) w[2 + lane * DPL + e] = st.o[qr][e];
    }
    cbar();
    const size_t rbase = (((size_t)b * p.Hkv + g) * p.s_max + it.s) * Q;
    for (int i = tid; i < Q * W; i += NCT) {
        const int qr = i / W, e = i - qr * W;
        float mx = -INFINITY;
        for (int w = 0; w < NCW; ++w) mx = fmaxf(mx, ws[((size_t)w * Q + qr) * W]);
        float v = 0.f;
        if (e == 0) {
            v = mx;
        } else if (mx != -INFINITY) {
            for (int w = 0; w < NCW; ++w) {
                const float mw = ws[((size_t)w * Q + qr) * W];
                if (mw != -INFINITY) v += ws[((size_t)w * Q + qr) * W + e] * expf(mw - mx);
            }
        }
        if (e < 2)
            p.part_ml[(rbase + qr) * 2 + e] = v;
        else
            p.part[(rbase + qr) * hd + (e - 2)] = v;
    }
    cbar();
}

// ======================================================= MLA attention ====
// item (sequence b, token t, split s): 16 heads x (latent 512 + rope 64)
// against 32-position chunks of the latent cache. Scores and P.V run on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate); the queries and
// probabilities are split into bf16 hi + lo parts so the products keep ~16
// mantissa bits (the cache values are exact bf16 already).
struct MlaSmem {
    uint16_t* qhi;   // [16][MLA_QS]
    uint16_t* qlo;
    float* spart;    // [KS][16][NR]
    uint16_t* phi;   // [16][40]
    uint16_t* plo;
    float* mst;      // [16] running max
    float* lst;      // [16] running sum
    float* cst;      // [16] correction of this chunk
    uint8_t* tk;     // the step's new positions: 16 rows in 9 swizzled boxes of 2 KB
};
__device__ __forceinline__ MlaSmem mla_smem(float* stage) {
    MlaSmem s;
    uint8_t* b = reinterpret_cast<uint8_t*>(stage);
    s.qhi = reinterpret_cast<uint16_t*>(b);
    s.qlo = reinterpret_cast<uint16_t*>(b + 16 * MLA_QS * 2);
    s.spart = reinterpret_cast<float*>(b + 2 * 16 * MLA_QS * 2);                 // 37376
    s.phi = reinterpret_cast<uint16_t*>(b + 37376 + 4096);                        // 41472
    s.plo = reinterpret_cast<uint16_t*>(b + 41472 + 16 * 40 * 2);                 // 42752
    s.mst = reinterpret_cast<float*>(b + 42752 + 16 * 40 * 2);                    // 44032
    s.lst = s.mst + 16;
    s.cst = s.lst + 16;
    s.tk = b + 44288;                                                             // .. 62720
    return s;
}

__device__ __forceinline__ uint32_t lds32(const uint16_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// kb: the chunk's 9 swizzled boxes, bb bytes apart (a ring slot: boxes of
// MLA_CH rows; the step's new positions: 16 rows); rows from nvalid on are
// not positions of the sequence
template <int NR>
__device__ __forceinline__ void mla_chunk(const MlaSmem& S, const uint8_t* kb, int bb, int nvalid,
                                          float (&acc)[8][4]) {
    const int tid = ctid(), lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
    // ---- scores S[16][NR] = Q . KV^T ----
    // warp = (column block nt of 8 rows, K slice ks); the K slice's k-steps
    // fully unrolled over four accumulators (hi / lo parts x even / odd
    // steps: four MMA chains instead of one); the query fragments by
    // ldmatrix from the padded rows (lane l addresses row l & 15, columns
    // + (l >> 4) * 8)
    constexpr int NT = NR / 8, KS = 8 / NT, STEPS = 36 / KS;
    const int nt = warp % NT, ks = warp / NT;
    float sa[4][4] = {};
    const int n = nt * 8 + g;
    // this lane's chunk row: its pieces are swizzled by bits 7..9 of the row's
    // address, the same in every box (boxes are multiples of 1024 bytes apart)
    const uint8_t* const rowp = kb + n * 128 + 4 * t4;
    const unsigned sw = (su32(kb + n * 128) >> 7) & 7u;
    const uint16_t* const qh = S.qhi + (lane & 15) * MLA_QS + (lane >> 4) * 8;
    const uint16_t* const ql = S.qlo + (lane & 15) * MLA_QS + (lane >> 4) * 8;
    const auto step = [&](int i, float (&shi)[4], float (&slo)[4]) {
        const int k0 = (ks * STEPS + i) * 16;
        uint32_t ah[4], al[4];
        ldsm_x4(ah, qh + k0);
        ldsm_x4(al, ql + k0);
        // (k0 is a multiple of 16: elements k0 + 2 t4 and k0 + 8 + 2 t4 are in
        // the neighbouring 16-byte pieces j0 and j0 + 1 of the row)
        const uint8_t* const bp = rowp + (k0 >> 6) * bb;
        const unsigned j0 = ((unsigned)k0 >> 3) & 7u;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bp + ((j0 ^ sw) << 4));
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bp + (((j0 + 1u) ^ sw) << 4));
        mma_bf16(shi, ah, b0, b1);
        mma_bf16(slo, al, b0, b1);
    };
#pragma unroll 3
    for (int i = 0; i + 1 < STEPS; i += 2) {
        step(i, sa[0], sa[1]);
        step(i + 1, sa[2], sa[3]);
    }
    if (STEPS & 1) step(STEPS - 1, sa[0], sa[1]);
    float sacc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) sacc[q] = (sa[0][q] + sa[1][q]) + (sa[2][q] + sa[3][q]);
    {
        float* sp = S.spart + (size_t)ks * 16 * NR;
        sp[g * NR + nt * 8 + 2 * t4] = sacc[0];
        sp[g * NR + nt * 8 + 2 * t4 + 1] = sacc[1];
        sp[(g + 8) * NR + nt * 8 + 2 * t4] = sacc[2];
        sp[(g + 8) * NR + nt * 8 + 2 * t4 + 1] = sacc[3];
    }
    cbar();
    // ---- online softmax: warp w owns heads 2w, 2w+1; 16 lanes per head ----
    {
        const int h = 2 * warp + (lane >> 4), l16 = lane & 15;
        float s0 = -INFINITY, s1 = -INFINITY;
        if (l16 < nvalid) {
            s0 = 0.f;
            for (int q = 0; q < KS; ++q) s0 += S.spart[((size_t)q * 16 + h) * NR + l16];
        }
        if (NR == 32 && l16 + 16 < nvalid) {
            s1 = 0.f;
            for (int q = 0; q < KS; ++q) s1 += S.spart[((size_t)q * 16 + h) * NR + l16 + 16];
        }
        float mc = fmaxf(s0, s1);
#pragma unroll
        for (int o = 8; o; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
        const float mold = S.mst[h];
        const float mn = fmaxf(mold, mc);
        float corr = 1.f, p0 = 0.f, p1 = 0.f;
        if (mn != -INFINITY) {
            corr = mold == -INFINITY ? 0.f : __expf(mold - mn);
            p0 = s0 == -INFINITY ? 0.f : __expf(s0 - mn);
            p1 = s1 == -INFINITY ? 0.f : __expf(s1 - mn);
        }
        float ps = p0 + p1;
#pragma unroll
        for (int o = 8; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        __syncwarp();
        if (l16 == 0) {
            S.mst[h] = mn;
            S.lst[h] = S.lst[h] * corr + ps;
            S.cst[h] = corr;
        }
        // rows past the sequence's end came with the chunk's half page (their
        // probabilities are 0): zero their latent values so that P.V stays finite
        if (nvalid < NR) {
            const int nb = (NR - nvalid) * 8;  // 16-byte pieces per box
            for (int i = tid; i < 8 * nb; i += NCT) {
                const int bx = i / nb, rem = i - bx * nb;
                *reinterpret_cast<uint4*>(const_cast<uint8_t*>(kb) + bx * bb + (nvalid + (rem >> 3)) * 128 +
                                          (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        const uint16_t h0 = f2bf(p0), h1 = f2bf(p1);
        S.phi[h * 40 + l16] = h0;
        S.plo[h * 40 + l16] = f2bf(p0 - bf2f(h0));
        if (NR == 32) {
            S.phi[h * 40 + l16 + 16] = h1;
            S.plo[h * 40 + l16 + 16] = f2bf(p1 - bf2f(h1));
        }
    }
    cbar();
    // ---- O[16][512] = O * corr + P . V ; warp w owns dims [64w, 64w+64) ----
    {
        const float c0 = S.cst[g], c1 = S.cst[g + 8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc[j][0] *= c0;
            acc[j][1] *= c0;
            acc[j][2] *= c1;
            acc[j][3] *= c1;
        }
        // rows kp + (lane & 15): bits 7..9 of their addresses do not depend on
        // kp (a multiple of 16 rows, 2048 bytes)
        const unsigned swv = (su32(kb + (lane & 15) * 128) >> 7) & 7u;
#pragma unroll
        for (int kp = 0; kp < NR; kp += 16) {
            // probabilities [16 heads][positions kp..kp+15] by ldmatrix (rows of
            // 80 bytes: the 8 rows of a matrix hit distinct banks)
            uint32_t ah[4], al[4];
            ldsm_x4(ah, S.phi + (lane & 15) * 40 + kp + (lane >> 4) * 8);
            ldsm_x4(al, S.plo + (lane & 15) * 40 + kp + (lane >> 4) * 8);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t r[4];  // columns warp * 64 + np * 16 (+ 8): box `warp`, pieces 2 np, 2 np + 1
                ldsm_x4_t(r, kb + warp * bb + (kp + (lane & 15)) * 128 +
                                 (((unsigned)(2 * np + (lane >> 4)) ^ swv) << 4));
                mma_bf16(acc[2 * np], ah, r[0], r[1]);
                mma_bf16(acc[2 * np], al, r[0], r[1]);
                mma_bf16(acc[2 * np + 1], ah, r[2], r[3]);
                mma_bf16(acc[2 * np + 1], al, r[2], r[3]);
            }
        }
    }
}

__device__ __forceinline__ void cons_attn_mla(Ctx& c, int l, const AttnItem& it) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const int tid = ctid(), lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
    const int b = it.b, t = it.g, m = b * p.T + t, pos = p.pos[b] + t;
    const bool tail = it.u_hi == it.nch + 1;
    MlaSmem S = mla_smem(c.stage());
    const long long ta = p.trace_items ? gtimer() : 0;
    cbar();
    c.sk_src = nullptr;
    // queries: [absorbed latent query (512) | roped rope query (64)] * scale, split hi/lo
    const int qh = p.nope + p.rd;
    const float sc = p.attn_scale;
    {
        // 2048 float4 of absorbed queries: all loads in flight, then split
        // into bf16 hi/lo and store 4 values per 8-byte store
        const float* qsrc = Ld.qlat + (size_t)m * MLA_H * MLA_KL;
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcg(reinterpret_cast<const float4*>(qsrc) + tid + k * NCT);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + k * NCT;  // float4 index: head i/128, element (i%128)*4
            const int h = i >> 7, e = (i & 127) * 4;
            const float f0 = v[k].x * sc, f1 = v[k].y * sc, f2 = v[k].z * sc, f3 = v[k].w * sc;
            const uint16_t h0 = f2bf(f0), h1 = f2bf(f1), h2 = f2bf(f2), h3 = f2bf(f3);
            const uint16_t l0 = f2bf(f0 - bf2f(h0)), l1 = f2bf(f1 - bf2f(h1)), l2 = f2bf(f2 - bf2f(h2)),
                           l3 = f2bf(f3 - bf2f(h3));
            *reinterpret_cast<uint2*>(S.qhi + h * MLA_QS + e) =
                make_uint2((uint32_t)h0 | ((uint32_t)h1 << 16), (uint32_t)h2 | ((uint32_t)h3 << 16));
            *reinterpret_cast<uint2*>(S.qlo + h * MLA_QS + e) =
                make_uint2((uint32_t)l0 | ((uint32_t)l1 << 16), (uint32_t)l2 | ((uint32_t)l3 << 16));
        }
    }
    for (int i = tid; i < MLA_H * (MLA_RD / 2); i += NCT) {
        const int h = i / (MLA_RD / 2), ri = i - h * (MLA_RD / 2), hr = MLA_RD / 2;
        const float* qr = Ld.q + (size_t)m * MLA_H * qh + h * qh + p.nope;
        const float2 cs = p.rope[(size_t)pos * p.rope_half + ri];
        const float x0 = __ldcg(qr + ri), x1 = __ldcg(qr + ri + hr);
        const float f0 = (x0 * cs.x - x1 * cs.y) * sc, f1 = (x1 * cs.x + x0 * cs.y) * sc;
        const uint16_t h0 = f2bf(f0), h1 = f2bf(f1);
        S.qhi[h * MLA_QS + MLA_KL + ri] = h0;
        S.qlo[h * MLA_QS + MLA_KL + ri] = f2bf(f0 - bf2f(h0));
        S.qhi[h * MLA_QS + MLA_KL + ri + hr] = h1;
        S.qlo[h * MLA_QS + MLA_KL + ri + hr] = f2bf(f1 - bf2f(h1));
    }
    if (tid < 16) {
        S.mst[tid] = -INFINITY;
        S.lst[tid] = 0.f;
    }
    if (tail) {
        // the new positions 0..T-1 of this step (token t sees 0..t), 16 bytes
        // at a time into the layout of a ring chunk with 16-row boxes
        for (int i = tid; i < 16 * (MLA_D / 8); i += NCT) {
            const int r = i / (MLA_D / 8), k = (i - r * (MLA_D / 8)) * 8;
            const uint4 v = r <= t ? *reinterpret_cast<const uint4*>(p.newlat + (size_t)(b * p.T + r) * MLA_D + k)
                                   : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(const_cast<uint8_t*>(mla_piece(S.tk, 16 * 128, r, k))) = v;
        }
    }
    cbar();
    const long long tb = p.trace_items ? gtimer() : 0;
    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    for (int u = it.u_lo; u < it.u_hi; ++u) {
        // one code path for cached chunks (from the ring) and the new positions (tail rows in smem)
        const bool ring_chunk = u < it.nch;
        const uint8_t* tile = nullptr;
        if (ring_chunk && !c.dead) tile = cons_wait(p, c.smem, c.ms, c.cr);
        if (ring_chunk && !tile) {
            cbar();
            cbar();
        } else if (ring_chunk) {
            mla_chunk<MLA_CH>(S, tile, MLA_BOX, min(MLA_CH, p.pos[b] - u * MLA_CH), acc);
        } else {
            mla_chunk<16>(S, S.tk, 16 * 128, t + 1, acc);  // boxes of 16 rows
        }
        if (ring_chunk) cons_release(c.ms, c.cr);
    }
    const long long tc = p.trace_items ? gtimer() : 0;
    // partial: unnormalised O rows and (max, sum) per head
    const size_t base = ((size_t)m * p.s_max + it.s) * MLA_H;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int dim = warp * 64 + j * 8 + 2 * t4;
        *reinterpret_cast<float2*>(p.part + (base + g) * MLA_KL + dim) = make_float2(acc[j][0], acc[j][1]);
        *reinterpret_cast<float2*>(p.part + (base + g + 8) * MLA_KL + dim) = make_float2(acc[j][2], acc[j][3]);
    }
    cbar();
    if (tid < 16) *reinterpret_cast<float2*>(p.part_ml + (base + tid) * 2) = make_float2(S.mst[tid], S.lst[tid]);
    cbar();
    // trace: staging ns in `n`, then chunk loop [t_wait = after staging, t_ready = chunks done]
    if (p.trace_items) trace_rec(c, 0x80000000u | ((unsigned)C_ATTN << 16) | (unsigned)l, (unsigned)(tb - ta), tb, tc);
}

// producer: bulk-load one MLA chunk (32 positions) into padded smem rows;
// rows past the valid positions are filled from a zero buffer
__device__ __noinline__ void prod_mla_chunk(Ctx& c, int l, int b, int u) {
    const Params& p = c.p;
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        // 9 bulk tensor copies: the latent's 8 column blocks and the rope of
        // the chunk's 32 rows (half a page); rows past the sequence's end
        // come along and are zeroed by the consumers
        uint8_t* dst = prod_begin(p, c.smem, c.ms, c.pr, MLA_TILE_BYTES);
        if (dst) {
            const int page = p.btab[b * p.pps + (u * MLA_CH) / PAGE], r0 = (u * MLA_CH) % PAGE;
            const uint8_t* tm = static_cast<const uint8_t*>(p.kv_tmaps);
            unsigned long long* bar = &c.ms.full[c.pr.slot];
#pragma unroll 1
            for (int j = 0; j < 8; ++j) tma_load_4d(dst + j * MLA_BOX, tm, 64 * j, r0, page, l, bar);
            tma_load_4d(dst + 8 * MLA_BOX, tm + 128, 0, r0, page, l, bar);
        } else {
            ok = 0;
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
        c.dead = true;
        return;
    }
    c.bump_issued();
    prod_next(c.pr);
}

__device__ __noinline__ void prod_gqa_chunk(Ctx& c, int l, int b, int g, int u) {
    const Params& p = c.p;
    const int hd = p.hd;
    const int nvalid = min(GQA_CH, p.pos[b] - u * GQA_CH);
    const unsigned bytes = 2u * nvalid * hd * 2u;
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        uint8_t* dst = prod_begin(p, c.smem, c.ms, c.pr, bytes);
        if (dst) {
            const uint16_t* pg = page_ptr(p, (p.kv_pool + (size_t)l * p.kv_layer_elems), b, u) + (size_t)g * 2 * PAGE * hd;
            bulk_g2s(dst, pg, nvalid * hd * 2u, &c.ms.full[c.pr.slot]);
            bulk_g2s(dst + (size_t)GQA_CH * hd * 2, pg + (size_t)PAGE * hd, nvalid * hd * 2u, &c.ms.full[c.pr.slot]);
        } else {
            ok = 0;
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
        c.dead = true;
        return;
    }
    c.bump_issued();
    prod_next(c.pr);
}

__device__ __noinline__ void attn_cons(Ctx& c, int l, int lo, int hi) {
    const Params& p = c.p;
    const long long t0 = gtimer();
    cwait(c, 0x600u | (unsigned)(l << 16));
    const long long t1 = gtimer();
    for (int i = lo; i < hi; ++i) {
        const AttnItem it = attn_item(p, i);
        if (p.attn == 0) {
            if (p.hd == 128)
                cons_attn_gqa<4>(c, l, it);
            else
                cons_attn_gqa<2>(c, l, it);
        } else {
            cons_attn_mla(c, l, it);
        }
    }
    csignal(c, l, C_ATTN, (unsigned)(hi - lo));
    trace_rec(c, ((unsigned)C_ATTN << 16) | (unsigned)l, (unsigned)(hi - lo), t0, t1);
}

// ======================================================== combine ====
// GQA: item (token, q head) -> o[m][h*hd ...]
// MLA: item (token, head, 128-dim chunk) -> olat[m][h*512 ...]
__device__ int comb_items(const Params& p) { return p.attn == 0 ? p.M * p.Hq : p.M * MLA_H * 4; }

__device__ __forceinline__ void cons_comb(Ctx& c, int l, int i) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const int tid = ctid(), lane = tid & 31, warp = tid >> 5;
    size_t r0, rstride;
    int S, D, d0, OL;
    float* out;
    if (p.attn == 0) {
        const int Gq = p.Hq / p.Hkv, Q = p.T * Gq;
        const int m = i / p.Hq, h = i - m * p.Hq, b = m / p.T, t = m - b * p.T;
        const int g = h / Gq, qr = t * Gq + (h - g * Gq);
        const int units = nch_of(p, b, GQA_CH) + 1, tg = gqa_target(p);
        S = units < tg ? units : tg;
        r0 = (((size_t)b * p.Hkv + g) * p.s_max) * Q + qr;
        rstride = Q;
        D = p.hd;
        d0 = 0;
        OL = p.hd;
        out = Ld.o + (size_t)m * p.Hq * p.hd + h * p.hd;
    } else {
        const int m = i / (MLA_H * 4), r = i - m * MLA_H * 4, h = r >> 2, dc = r & 3;
        const int b = m / p.T;
        const int units = nch_of(p, b, MLA_CH) + 1, tg = mla_target(p);
        S = units < tg ? units : tg;
        r0 = (size_t)m * p.s_max * MLA_H + h;
        rstride = MLA_H;
        D = 128;
        d0 = dc * 128;
        OL = MLA_KL;
        out = Ld.olat + (size_t)m * MLA_H * MLA_KL + h * MLA_KL + d0;
    }
    // split weights: w_s = exp(m_s - max) / sum_s exp(m_s - max) * l_s
    float mv = -INFINITY, lv = 0.f;
    if (tid < S) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (r0 + tid * rstride) * 2));
        mv = ml.x;
        lv = ml.y;
    }
    const float mx = cblock_max(c, mv);
    const float w = (tid < S && mv != -INFINITY) ? expf(mv - mx) : 0.f;
    const float L = cblock_sum(c, w * lv);
    if (tid < S) c.ms.cw[tid] = w / L;
    cbar();
    // weighted sum of the O partials: warps take splits, lanes take 4 dims;
    // a thread's split loads (up to CSPW) are all issued before the first
    // is used, so the sum costs one L2 round trip instead of one per few
    // splits (the partials were just written by other CTAs)
    constexpr int CSPW = 20;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane * 4 < D) {
        for (int sb = warp; sb < S; sb += NCW * CSPW) {
            float4 v[CSPW];
#pragma unroll
            for (int k = 0; k < CSPW; ++k) {
                const int s2 = sb + NCW * k;
                v[k] = s2 < S ? __ldcg(reinterpret_cast<const float4*>(p.part + (r0 + s2 * rstride) * OL + d0 + lane * 4))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < CSPW; ++k) {
                const int s2 = sb + NCW * k;
                const float cw = s2 < S ? c.ms.cw[s2] : 0.f;
                acc.x = fmaf(cw, v[k].x, acc.x);
                acc.y = fmaf(cw, v[k].y, acc.y);
                acc.z = fmaf(cw, v[k].z, acc.z);
                acc.w = fmaf(cw, v[k].w, acc.w);
            }
        }
        *reinterpret_cast<float4*>(c.red() + warp * 128 + lane * 4) = acc;
    }
    cbar();
    const bool uv = p.attn == 1 && p.ufuse;
    float* xl = c.stage();  // fused value up-projection: this item's 128 latent values
    for (int e = tid; e < D; e += NCT) {
        float v = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NCW; ++w2) v += c.red()[w2 * 128 + e];
        if (uv)
            xl[e] = v;
        else
            out[e] = v;
    }
    cbar();
    if (uv) {
        // o[m][h][v] += sum_j olat[m][h][d0 + j] W_uv[h][v][d0 + j] over this
        // item's 128 latent dimensions j: the slab W_uv[h] (quarter d0 / 128)
        // is stored j-major [128 j][vd v]; thread: values v = 2 vp, 2 vp + 1
        // against j in [32 jq, 32 jq + 32), added into o with a reduction
        c.sk_src = nullptr;  // the staging area no longer holds a GEMV input
        const uint8_t* slab = c.dead ? nullptr : cons_wait(p, c.smem, c.ms, c.cr);
        const int vp = tid & 63, jq = tid >> 6, m = i / (MLA_H * 4), h = (i >> 2) & (MLA_H - 1);
        if (slab && 2 * vp < p.vd) {
            const uint32_t* W = reinterpret_cast<const uint32_t*>(slab) + vp;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
            for (int j = 32 * jq; j < 32 * jq + 32; ++j) {
                const uint32_t w = W[(size_t)j * (p.vd / 2)];
                a0 = fmaf(xl[j], bf_lo(w), a0);
                a1 = fmaf(xl[j], bf_hi(w), a1);
            }
            float* o = Ld.o + (size_t)m * MLA_H * p.vd + h * p.vd + 2 * vp;
            asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" ::"l"(o), "f"(a0), "f"(a1) : "memory");
        }
        cons_release(c.ms, c.cr);  // every warp's ring state advances alike
        cbar();                    // xl is free for the next item
    }
}

// producer side of the combine with the value up-projection folded in: the
// W_uv slab of each item (head, latent quarter)
__device__ __noinline__ void comb_prod(Ctx& c, int lo, int hi) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const unsigned bytes = 128u * (unsigned)p.vd * 2u;
    for (int i = lo; i < hi && !c.dead; ++i) {
        const int h = (i >> 2) & (MLA_H - 1), q = i & 3;
        int ok = 1;
        if ((threadIdx.x & 31) == 0) {
            uint8_t* dst = prod_begin(p, c.smem, c.ms, c.pr, bytes);
            if (dst)
                bulk_g2s(dst, Ld.uvq + (size_t)(h * 4 + q) * 128 * p.vd, bytes, &c.ms.full[c.pr.slot]);
            else
                ok = 0;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            c.dead = true;
            return;
        }
        c.bump_issued();
        prod_next(c.pr);
    }
}

__device__ __noinline__ void comb_cons(Ctx& c, int l, int lo, int hi) {
    const long long t0 = gtimer();
    cwait(c, 0x700u | (unsigned)(l << 16));
    const long long t1 = gtimer();
    for (int i = lo; i < hi; ++i) cons_comb(c, l, i);
    csignal(c, l, C_COMB, (unsigned)(hi - lo));
    trace_rec(c, ((unsigned)C_COMB << 16) | (unsigned)l, (unsigned)(hi - lo), t0, t1);
}

// ========================================================= MLA append ====
// item = token: latent = RMSNorm(kv_a latent part) * gain, k_rope = RoPE(kv_a
// rope part); both rounded to bf16, written to the page and to newlat.
__device__ __noinline__ void append_cons(Ctx& c, int l, int lo, int hi) {
    const Params& p = c.p;
    const long long t0 = gtimer();
    cwait(c, 0x800u | (unsigned)(l << 16));
    const long long t1 = gtimer();
    const Layer& Ld = c.layer();
    const int tid = ctid(), lane = tid & 31, warp = tid >> 5;
    for (int m = lo; m < hi; ++m) {
        const int b = m / p.T, t = m - b * p.T, pos = p.pos[b] + t;
        const float* a = Ld.a + (size_t)m * Ld.a_stride + p.ql;
        float ss = 0.f;
        for (int e = tid; e < MLA_KL; e += NCT) {
            const float v = __ldcg(a + e);
            ss = fmaf(v, v, ss);
        }
        ss = cblock_sum(c, ss);
        if (tid == 0) c.ms.rms[0] = 1.0f / sqrtf(ss / (float)MLA_KL + p.eps);
        cbar();
        uint16_t* pg = const_cast<uint16_t*>(page_ptr(p, p.kv_pool + (size_t)l * p.kv_layer_elems, b, pos / PAGE));
        const int pr = pos % PAGE;
        uint16_t* nl = p.newlat + (size_t)m * MLA_D;
        for (int e = tid; e < MLA_D; e += NCT) {
            uint16_t v;
            if (e < MLA_KL) {
                v = f2bf(__ldcg(a + e) * c.ms.rms[0] * bf2f(Ld.kv_norm[e]));
                pg[(size_t)pr * MLA_KL + e] = v;
            } else {
                const int r = e - MLA_KL, hr = MLA_RD / 2, ri = r < hr ? r : r - hr;
                const float2 cs = p.rope[(size_t)pos * p.rope_half + ri];
                const float x0 = __ldcg(a + MLA_KL + ri), x1 = __ldcg(a + MLA_KL + ri + hr);
                v = f2bf(r < hr ? (x0 * cs.x - x1 * cs.y) : (x1 * cs.x + x0 * cs.y));
                pg[(size_t)PAGE * MLA_KL + (size_t)pr * MLA_RD + r] = v;
            }
            nl[e] = v;
        }
    }
    csignal(c, l, C_APP, (unsigned)(hi - lo));
    trace_rec(c, ((unsigned)C_APP << 16) | (unsigned)l, (unsigned)(hi - lo), t0, t1);
}

// ===================================================== residual carry ====
// (only when the output projection is split over K: x_{l+1} += x_l)
__device__ __noinline__ void carry_cons(Ctx& c, int l, int lo, int hi) {
    const Params& p = c.p;
    const int chunk = 2048;
    cwait(c, 0x900u | (unsigned)(l << 16));
    const Layer& Ld = c.layer();
    const int total = p.M * p.d;
    for (int i = lo * chunk + ctid(); i < min(hi * chunk, total); i += NCT) {
        const int m = i / p.d, e = i - m * p.d;
        atomicAdd(Ld.xn + (size_t)m * p.d + e, __ldcg(Ld.x + (size_t)m * p.d + e));
    }
    csignal(c, l, C_CARRY, (unsigned)(hi - lo));
}

// ===================================================== head / verify ====
__device__ __noinline__ void argmax_cons(Ctx& c, int lo, int hi) {
    const Params& p = c.p;
    cwait(c, 0xa00u);
    const int tid = ctid(), lane = tid & 31, warp = tid >> 5;
    float* bv = c.red();
    int* bi = reinterpret_cast<int*>(c.red() + NCW);
    for (int m = lo; m < hi; ++m) {
        const float* lg = p.logits + (size_t)m * p.V;
        float v = -INFINITY;
        int id = 0x7fffffff;
        for (int e = tid; e < p.V; e += NCT) {
            const float x = __ldcg(lg + e);
            if (x > v || (x == v && e < id)) {
                v = x;
                id = e;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int oi = __shfl_xor_sync(0xffffffffu, id, o);
            if (ov > v || (ov == v && oi < id)) {
                v = ov;
                id = oi;
            }
        }
        cbar();
        if (lane == 0) {
            bv[warp] = v;
            bi[warp] = id;
        }
        cbar();
        if (tid == 0) {
            for (int w = 1; w < NCW; ++w)
                if (bv[w] > v || (bv[w] == v && bi[w] < id)) {
                    v = bv[w];
                    id = bi[w];
                }
            p.amax[m] = id;
        }
    }
    csignal(c, p.L, C_AMAX, (unsigned)(hi - lo));
}

// ====================================================== init (consumers) ====
// debug mode: 16 bytes at the end of every ring slot (no copy reaches
// them: the largest, an MLA chunk, ends 1 KB earlier) and after the staging
// area hold a pattern written at entry and compared when the CTA leaves
__device__ __noinline__ void debug_canaries(const Params& p, uint8_t* smem, bool check) {
    const uint4 pat = make_uint4(0x6d6b4341u, 0x4e415259u, blockIdx.x, 0x5a5a5a5au);
    for (int s2 = 0; s2 <= NSLOT; ++s2) {
        uint4* w = reinterpret_cast<uint4*>(smem + (s2 < NSLOT ? SMEM_RING + (s2 + 1) * SLOT_BYTES - 16 : SMEM_CANARY));
        if (!check) {
            *w = pat;
        } else {
            const uint4 v = *w;
            if (v.x != pat.x || v.y != pat.y || v.z != pat.z || v.w != pat.w) raise_status(p, ST_DEBUG, 0x9100u + s2);
        }
    }
}

__device__ __noinline__ bool init_phase(Ctx& c) {
    const Params& p = c.p;
    const int tid = ctid();
    if (p.debug && tid == 0) debug_canaries(p, c.smem, false);
    // every CTA checks the step's inputs itself (all reach the same verdict)
    if (tid == 0) {
        int bad = 0;
        for (int m = 0; m < p.M; ++m)
            if (p.tokens[m] < 0 || p.tokens[m] >= p.V) bad = 1;
        for (int b = 0; b < p.B; ++b)
            if (p.pos[b] < 0 || p.pos[b] + p.T > p.kv_cap || p.pos[b] + p.T > p.rope_npos) bad = 1;
        c.ms.abort = bad;
        if (bad && blockIdx.x == 0) raise_status(p, ST_INVALID, 0x10u);
    }
    cbar();
    if (c.ms.abort) {
        c.dead = true;
        return false;
    }
    if (p.stall && blockIdx.x == 0) {
        // failure-detection test: a wait whose counter nothing signals runs
        // into the time limit, records MK_ERR_TIMEOUT and makes every CTA leave
        if (tid == 0 && !wait_ge(p, ctr_of(p, p.L, C_GU0), 1u, 0xe00u)) c.ms.abort = 1;
        cbar();
        if (c.ms.abort) {
            c.dead = true;
            return false;
        }
    }
    // one launch per stage: only the set-up launch initialises the step
    if (p.staged == 1) return !c.dead;
    const size_t gtid = (size_t)blockIdx.x * NCT + tid, gstride = (size_t)p.G * NCT;
    // counters of the other parity are used by the next step: clear them now
    // (one launch per stage uses no counters and leaves them as they are)
    if (!p.staged) {
        unsigned* other = p.ctr + (size_t)(p.parity ^ 1) * (p.L + 1) * NCTR;
        for (size_t i = gtid; i < (size_t)(p.L + 1) * NCTR; i += gstride) other[i] = 0u;
    }
    for (int z = 0; z < p.nz; ++z)
        for (size_t i = gtid; i < (size_t)p.zn[z]; i += gstride) p.zptr[z][i] = 0.f;
    float* x0 = p.layers[0].x;
    for (size_t i = gtid; i < (size_t)p.M * p.d; i += gstride) {
        const int m = (int)(i / p.d), e = (int)(i - (size_t)m * p.d);
        x0[i] = bf2f(p.embed[(size_t)p.tokens[m] * p.d + e]);
    }
    csignal(c, p.L, C_INIT, 1u);
    trace_rec(c, ((unsigned)C_INIT << 16) | (unsigned)p.L, 1u, c.t_start, c.t_start);
    return !c.dead;
}

__device__ bool prod_check(const Params& p) {
    for (int b = 0; b < p.B; ++b)
        if (p.pos[b] < 0 || p.pos[b] + p.T > p.kv_cap || p.pos[b] + p.T > p.rope_npos) return false;
    for (int m = 0; m < p.M; ++m)
        if (p.tokens[m] < 0 || p.tokens[m] >= p.V) return false;
    return true;
}

// producer, at the start of an MLA layer: start this CTA's attention chunks
// (latent rows and rope rows of the cached prefix) towards L2, so that the
// ring fills them at L2 latency when the attention stage comes. The item
// rotation offset of the attention stage follows from the stages before it.
__device__ __noinline__ void prefetch_attn_mla(Ctx& c, int l) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const long long ahead = (long long)gemv_items(Ld.g[G_A]) + gemv_items(Ld.g[G_QB]) + p.M +
                            (p.qfuse ? 0 : gemv_items(Ld.g[G_QLAT]));
    int lo, hi;
    my_range(p, attn_items(p), (int)((c.off + ahead) % p.G), lo, hi);
    const int lane = threadIdx.x & 31;
    const uint16_t* pool = p.kv_pool + (size_t)l * p.kv_layer_elems;
    for (int i = lo; i < hi; ++i) {
        const AttnItem it = attn_item(p, i);
        const int u1 = min(it.u_hi, it.nch);
        for (int u = it.u_lo + lane; u < u1; u += 32) {
            const int nvalid = min(MLA_CH, p.pos[it.b] - u * MLA_CH);
            const uint16_t* pg = page_ptr(p, pool, it.b, (u * MLA_CH) / PAGE);
            const int r0 = (u * MLA_CH) % PAGE;
            l2_prefetch(pg + (size_t)r0 * MLA_KL, (unsigned)nvalid * MLA_KL * 2u);
            l2_prefetch(pg + (size_t)PAGE * MLA_KL + (size_t)r0 * MLA_RD, (unsigned)nvalid * MLA_RD * 2u);
        }
    }
}

// producer, at the start of layer l: the next layer's descriptors and norm
// gains (or the head's final norm gain) towards L2, kept there
__device__ __noinline__ void prefetch_next_small(Ctx& c, int l) {
    const Params& p = c.p;
    const int lane = threadIdx.x & 31;
    if (l + 1 < p.L) {
        const Layer* nx = p.layers + l + 1;
        if (lane == 0) l2_prefetch_keep(nx, (unsigned)sizeof(Layer));
        const uint16_t* gp = nullptr;
        int n = 0;
        if (lane == 1) {
            gp = nx->g[G_A].gain;
            n = nx->g[G_A].K;
        } else if (lane == 2 && nx->g[G_QB].in_kind == IN_RMS) {
            gp = nx->g[G_QB].gain;
            n = nx->g[G_QB].K;
        } else if (lane == 3 && p.attn == 1) {
            gp = nx->kv_norm;
            n = MLA_KL;
        } else if (lane == 4) {
            gp = nx->ffn.gain;
            n = p.d;
        }
        if (gp && n > 0) l2_prefetch_keep(gp, (unsigned)n * 2u);
    } else if (lane == 0 && p.lm.gain) {
        l2_prefetch_keep(p.lm.gain, (unsigned)p.lm.K * 2u);
    }
    // router folded into the output projection: layer l's router weights
    // towards L2 (64 KB per CTA), read at the end of the output projection
    if (p.rfuse && lane == 5) {
        const Gemv& gr = c.layer().g[G_ROUTER];
        const size_t bytes = (size_t)gr.N * gr.K * 2, o = (size_t)blockIdx.x * 65536;
        if (o < bytes) l2_prefetch(reinterpret_cast<const uint8_t*>(gr.W) + o, (unsigned)min((size_t)65536, bytes - o));
    }
}

// copy layer l's descriptors into this side's shared-memory slot (the
// leading barrier ends every use of the previous layer's copy)
template <bool PROD>
__device__ __forceinline__ void load_layer(Ctx& c, int l) {
    constexpr int N16 = (int)sizeof(Layer) / 16;
    static_assert(sizeof(Layer) % 16 == 0, "Layer is copied in 16-byte pieces");
    const uint4* src = reinterpret_cast<const uint4*>(c.p.layers + l);
    uint4* dst = reinterpret_cast<uint4*>(c.smem + (PROD ? SMEM_PLAYER : SMEM_LAYER));
    if constexpr (PROD) {
        __syncwarp();
        for (int i = threadIdx.x & 31; i < N16; i += 32) dst[i] = __ldg(src + i);
        __syncwarp();
    } else {
        cbar();
        for (int i = ctid(); i < N16; i += NCT) dst[i] = __ldg(src + i);
        cbar();
    }
}

// ======================================================= producer leaves ====
__device__ __noinline__ void prod_plain(Ctx& c, const Gemv& g, int lo, int hi) {
    prod_gemv(c, g, -1, lo, hi, c.p.M);
}

// attention chunks of items [lo, hi) into the ring
__device__ __noinline__ void prod_attn(Ctx& c, int l, int lo, int hi) {
    const Params& p = c.p;
    for (int i = lo; i < hi && !c.dead; ++i) {
        const AttnItem it = attn_item(p, i);
        for (int u = it.u_lo; u < min(it.u_hi, it.nch) && !c.dead; ++u) {
            if (p.attn == 0)
                prod_gqa_chunk(c, l, it.b, it.g, u);
            else
                prod_mla_chunk(c, l, it.b, u);
        }
    }
}

// ========================================================= FFN units ====
// A segment is units [u0, u1) of one expert (kind 0: a routed expert, kind 1:
// the shared expert). Consumers: gate/up rows of the segment (one GEMV over
// rows [2F u0, 2F u1) of the expert's unit-major gate/up matrix, into a
// CTA-private buffer), hidden = silu(gate) * up, then the segment's down
// columns against the hidden values, added into the residual with the
// expert's routing weight. The producer streams the same tiles.

// gate/up outputs hs [M][2F n] then hidden h [M][n][F] (n units): the upper
// half of the reduction area (the split-K GEMV uses the lower half) when
// they fit, else this CTA's slice of a global buffer
__device__ __forceinline__ float* unit_buf(Ctx& c, int floats) {
    if (floats <= RED_FLOATS / 2) return c.red() + RED_FLOATS / 2;
    return c.p.ubuf + (size_t)blockIdx.x * c.p.ubuf_stride;
}

__device__ __forceinline__ void unit_gemv(const Params& p, const Layer& Ld, Gemv& ug, int kind, int expert, int u0,
                                          int u1, float* hs) {
    const FfnKind& K = Ld.ffn.k[kind];
    ug.W = K.gu + (expert >= 0 ? (size_t)expert * K.gu_es : 0);
    ug.w_estride = 0;
    ug.N = 2 * K.Fi;
    ug.K = p.d;
    ug.Kc = Ld.ffn.Kc;
    ug.R = K.R;
    ug.n_kc = Ld.ffn.n_kc;
    ug.n_rb = 2 * K.Fi / K.R;
    ug.in_kind = IN_RMS;
    ug.src = Ld.x;
    ug.src_stride = p.d;
    ug.src_sstride = 0;
    ug.gain = Ld.ffn.gain;
    ug.grp_rows = 0;
    ug.grp_stride = 0;
    ug.sw_off = 0;
    // one K panel: every value is written once; otherwise the panels add up
    ug.out_kind = Ld.ffn.n_kc == 1 ? OUT_STORE : OUT_ACC;
    ug.dst = hs - (size_t)2 * K.F * u0;  // rows [2F u0, 2F u1) land at hs[0 ..)
    ug.dst_stride = 2 * K.F * (u1 - u0);
    ug.dst_sstride = 0;
    ug.dst2 = nullptr;
}

// add v (this lane's row of 4 consecutive rows held by lanes 4i .. 4i+3 of
// the warp) into dst + row with one vector reduction per 4 rows: the
// residual rows receive every unit's down output, and 4-wide reductions
// cut the operations the L2 performs on those few lines by 4
__device__ __forceinline__ void red4_rows(float* dst, int row, bool ok, float v) {
    const float v1 = __shfl_down_sync(0xffffffffu, v, 1);
    const float v2 = __shfl_down_sync(0xffffffffu, v, 2);
    const float v3 = __shfl_down_sync(0xffffffffu, v, 3);
    if (ok && (threadIdx.x & 3) == 0)
        asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + row), "f"(v), "f"(v1),
                     "f"(v2), "f"(v3)
                     : "memory");
}

// one thread's rows of a down tile (nr rows x F, nr a multiple of 8), one
// token, hidden values of the unit in registers; a warp takes 32 consecutive
// rows at a time
template <int F8>
__device__ __forceinline__ void down_rows1(const uint8_t* tile, int nr, const float* hu, float w, float* xo) {
    float4 ha[F8], hb[F8];
#pragma unroll
    for (int q = 0; q < F8; ++q) {
        ha[q] = *reinterpret_cast<const float4*>(hu + 8 * q);
        hb[q] = *reinterpret_cast<const float4*>(hu + 8 * q + 4);
    }
    const uint4* T4 = reinterpret_cast<const uint4*>(tile);
    const int lane = threadIdx.x & 31;
    for (int rb = (ctid() >> 5) * 32; rb < nr; rb += NCT) {
        const int r = rb + lane;
        float a = 0.f, b = 0.f;
        if (r < nr) {
#pragma unroll
            for (int q = 0; q < F8; ++q) fma8v2(a, b, T4[(size_t)r * F8 + q], ha[q], hb[q]);
        }
        red4_rows(xo, r, r < nr, w * (a + b));
    }
}

// one thread's rows of a down tile (nr rows x F, nr a multiple of 8),
// several tokens: the row's weights in registers, token i's hidden values at
// hu + i hstride, its output row gt[i] of xo (stride d), scaled by its
// routing weight
// down columns of one unit for two or more tokens on the tensor cores:
// out[token][row] = sum_f W[row][f] h[token][f] with mma.sync m16n8k16 --
// the tokens are A's 16 rows (their hidden values split into bf16 hi + lo,
// two MMAs, as for the activations of the gate/up tiles), 8 rows of the
// tile are B's 8 columns and K is the unit's F (F / 16 k-steps). A lane's
// results are two adjacent rows of one token: one 8-byte reduction into
// that token's residual row, scaled by its routing weight. Warp w takes the
// groups of 8 rows w, w + 8, ...; the tile's rows are F * 2 bytes apart in
// the ring slot (the B loads of 8 rows x 4 lanes meet two-way bank conflicts
// at F = 48).
template <int F>
__device__ __forceinline__ void down_mma(const uint8_t* tile, int nr, const float* hu, int hstride, int M,
                                         const Misc& ms, float* xo, int d) {
    constexpr int KS = F / 16;
    const int lane = threadIdx.x & 31, warp = ctid() >> 5, g = lane >> 2, t4 = lane & 3;
    for (int mb = 0; mb < M; mb += 16) {
        const int t0 = mb + g, t1 = t0 + 8;
        const bool ok0 = t0 < M, ok1 = t1 < M;
        uint32_t ah[KS][4], al[KS][4];
#pragma unroll
        for (int s2 = 0; s2 < KS; ++s2) {
            const float2 z = make_float2(0.f, 0.f);
            const float* h0 = hu + (size_t)(ok0 ? t0 : 0) * hstride + 16 * s2 + 2 * t4;
            const float* h1 = hu + (size_t)(ok1 ? t1 : 0) * hstride + 16 * s2 + 2 * t4;
            const float2 u0 = ok0 ? *reinterpret_cast<const float2*>(h0) : z;
            const float2 v0 = ok0 ? *reinterpret_cast<const float2*>(h0 + 8) : z;
            const float2 u1 = ok1 ? *reinterpret_cast<const float2*>(h1) : z;
            const float2 v1 = ok1 ? *reinterpret_cast<const float2*>(h1 + 8) : z;
            ah[s2][0] = bf2_pack(u0.x, u0.y);
            ah[s2][1] = bf2_pack(u1.x, u1.y);
            ah[s2][2] = bf2_pack(v0.x, v0.y);
            ah[s2][3] = bf2_pack(v1.x, v1.y);
            al[s2][0] = bf2_pack(u0.x - bf_lo(ah[s2][0]), u0.y - bf_hi(ah[s2][0]));
            al[s2][1] = bf2_pack(u1.x - bf_lo(ah[s2][1]), u1.y - bf_hi(ah[s2][1]));
            al[s2][2] = bf2_pack(v0.x - bf_lo(ah[s2][2]), v0.y - bf_hi(ah[s2][2]));
            al[s2][3] = bf2_pack(v1.x - bf_lo(ah[s2][3]), v1.y - bf_hi(ah[s2][3]));
        }
        const float w0 = ok0 ? ms.uw[t0] : 0.f, w1 = ok1 ? ms.uw[t1] : 0.f;
        float* const x0 = xo + (size_t)(ok0 ? ms.gt[t0] : 0) * d;
        float* const x1 = xo + (size_t)(ok1 ? ms.gt[t1] : 0) * d;
        // nr is a multiple of 8 (d and the tile height are): every group of
        // 8 rows is whole
        for (int n0 = warp * 8; n0 < nr; n0 += NCW * 8) {
            const uint8_t* br = tile + (size_t)(n0 + g) * (F * 2) + 4 * t4;
            float c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s2 = 0; s2 < KS; ++s2) {
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(br + 32 * s2);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(br + 32 * s2 + 16);
                mma_bf16(c4, ah[s2], b0, b1);
                mma_bf16(c4, al[s2], b0, b1);
            }
            const int row = n0 + 2 * t4;
            if (w0 != 0.f)
                asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" ::"l"(x0 + row), "f"(w0 * c4[0]),
                             "f"(w0 * c4[1])
                             : "memory");
            if (w1 != 0.f)
                asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" ::"l"(x1 + row), "f"(w1 * c4[2]),
                             "f"(w1 * c4[3])
                             : "memory");
        }
    }
}

// ---- MXFP8 expert weights ----
// Two E4M3 codes become two fp16 values with one conversion instruction
// (cvt.rn.f16x2.e4m3x2; every E4M3 value, subnormals included, is an fp16
// number, so the conversion is exact), then fp32. A block's partial sum times
// 2^(E - 127) is the sum of (code value x 2^(E - 127)) x input.
__device__ __forceinline__ float2 f8_pair(uint32_t w16) {
    uint32_t h;
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "r"(w16));
    float lo, hi;
    asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b; }" : "=f"(lo), "=f"(hi) : "r"(h));
    return make_float2(lo, hi);
}
// 2^(E - 127) for an E8M0 scale byte E (E = 0: 2^-127, a float subnormal;
// 0xFF, NaN in the format, is not supported and reads as infinity)
__device__ __forceinline__ float f8_scale(uint32_t E) { return E ? __uint_as_float(E << 23) : __uint_as_float(0x400000u); }

// sum of 16 codes (one 16-byte chunk) times 16 inputs
__device__ __forceinline__ float f8_dot16(const uint4 u, const float4 (&x)[4]) {
    float a = 0.f, b = 0.f;
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 p0 = f8_pair(w[q] & 0xffffu), p1 = f8_pair(w[q] >> 16);
        a = fmaf(p0.x, x[q].x, a);
        b = fmaf(p0.y, x[q].y, b);
        a = fmaf(p1.x, x[q].z, a);
        b = fmaf(p1.y, x[q].w, b);
    }
    return a + b;
}

// gate/up tiles [j_lo, j_hi) of one unit segment: a tile is R = 64 / NQ
// rows of the K = 512 NQ codes each (then their scales); lane chunk q of a
// row holds codes 16 (lane + 32 q) .. + 15, all inside one 32-code block;
// warp w takes rows RB w .. RB w + RB - 1 (RB = R / 8) and one transposed
// reduction gives the RB sums. The unit's tokens (ms.gm, their inputs
// staged) take the tile one after the other, each input loaded into
// registers for its pass (one token: once for the segment). Row r of tile j
// for token i lands at hs[i rows + (j - j_lo) R + r], rows = (j_hi - j_lo) R.
template <int NQ>
__device__ __forceinline__ void gu_f8(Ctx& c, int j_lo, int j_hi, float* hs) {
    constexpr int RB = 8 / NQ, KC = 512 * NQ, R = 8 * RB;
    const Params& p = c.p;
    Misc& ms = c.ms;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ntok = ms.gm, rows = (j_hi - j_lo) * R;
    uint8_t* const ring = c.smem + SMEM_RING;
    float4 x[NQ][4];
    const auto load_x = [&](int tk) {
        const float* xt = c.stage() + (size_t)staging_row(ms, tk) * stage_stride(KC);
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) x[q][i] = *reinterpret_cast<const float4*>(xt + 16 * (lane + 32 * q) + 4 * i);
    };
    load_x(0);
    CRing cr = c.cr;
    bool dead = c.dead, timed_out = false;
    for (int j = j_lo; j < j_hi; ++j) {
        const uint8_t* tile = nullptr;
        if (!dead) {
            if (spin_wait(p, &ms.full[cr.slot], cr.phase))
                tile = ring + cr.slot * SLOT_BYTES;
            else
                dead = timed_out = true;
        }
        if (tile) {
            const uint8_t* sc = tile + R * KC;
            for (int tk = 0; tk < ntok; ++tk) {
                if (ntok > 1) load_x(tk);
                float v[RB];
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    const int r = warp * RB + b;
                    const uint4* row = reinterpret_cast<const uint4*>(tile + (size_t)r * KC) + lane;
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < NQ; ++q)
                        acc = fmaf(f8_dot16(row[32 * q], x[q]), f8_scale(sc[r * (KC / 32) + ((lane + 32 * q) >> 1)]),
                                   acc);
                    v[b] = acc;
                }
                const int b = rx_reduce<RB>(v);
                if ((lane & (32 / RB - 1)) == 0) hs[(size_t)tk * rows + (j - j_lo) * R + warp * RB + b] = v[0];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.empty[cr.slot]);
        if (++cr.slot == NSLOT) {
            cr.slot = 0;
            cr.phase ^= 1u;
        }
    }
    if (timed_out) {
        ms.abort = 1;
        raise_status(p, ST_TIMEOUT, 0x230u);
    }
    c.set_ring(cr);
    if (dead) c.dead = true;
}

// one thread's rows of an MXFP8 down tile (nr rows x F codes, then nr x F/32
// scales; FQ = F / 16 chunks per row), one token, the unit's F hidden values
// in registers; a warp takes 32 consecutive rows at a time
template <int FQ>
__device__ __forceinline__ void down_f8(const uint8_t* tile, int nr, const float* hu, float w, float* xo) {
    constexpr int F = 16 * FQ;
    float4 hx[FQ][4];
#pragma unroll
    for (int q = 0; q < FQ; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i) hx[q][i] = *reinterpret_cast<const float4*>(hu + 16 * q + 4 * i);
    const uint8_t* sc = tile + (size_t)nr * F;
    const int lane = threadIdx.x & 31;
    for (int rb = (ctid() >> 5) * 32; rb < nr; rb += NCT) {
        const int r = rb + lane;
        float a = 0.f;
        if (r < nr) {
            const uint4* row = reinterpret_cast<const uint4*>(tile + (size_t)r * F);
#pragma unroll
            for (int q = 0; q < FQ; ++q) a = fmaf(f8_dot16(row[q], hx[q]), f8_scale(sc[r * (F / 32) + q / 2]), a);
        }
        red4_rows(xo, r, r < nr, w * a);
    }
}

// MXFP8 gate/up tiles [j_lo, j_hi) of a unit segment (one K panel): the
// inputs are staged once (the routed CTAs may have staged them already),
// then the tiles
__device__ __noinline__ void unit_gu_f8(Ctx& c, int j_lo, int j_hi, float* hs) {
    restage(c, c.ms.ug, c.ms.ug.src, 0, 0, 0, c.ms.gather ? c.ms.gm : c.p.M);
    const int Kc = c.layer().ffn.Kc;
    if (Kc == 2048) gu_f8<4>(c, j_lo, j_hi, hs);
    else if (Kc == 1024) gu_f8<2>(c, j_lo, j_hi, hs);
    else gu_f8<1>(c, j_lo, j_hi, hs);
}

// one MXFP8 down tile (units 64 wide), once per token of the unit (the
// CTA's token map in shared memory): token i's hidden values at hu + i n F
// (n units of F in the segment: half the segment's gate/up rows), its
// residual row gt[i] (xo is token 0's, rows d apart), its routing weight
__device__ __noinline__ void unit_down_f8(const uint8_t* tile, int nr, const float* hu, float* xo, int d) {
    extern __shared__ __align__(1024) uint8_t smem_base[];
    const Misc& ms = *reinterpret_cast<const Misc*>(smem_base + SMEM_MISC);
    const int M = ms.gm, hstride = ms.ug.dst_stride / 2, g0 = ms.gt[0];
    for (int i = 0; i < M; ++i) {
        const float w = ms.uw[i];
        if (w != 0.f) down_f8<4>(tile, nr, hu + (size_t)i * hstride, w, xo + (ptrdiff_t)((int)ms.gt[i] - g0) * d);
    }
}

__device__ __noinline__ void unit_seg_cons(Ctx& c, int l, int kind, int expert, int u0, int u1, int m_lo, int m_hi) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const FfnKind& K = Ld.ffn.k[kind];
    const int F = K.F, n = u1 - u0, rows = 2 * F * n, d = p.d, tid = ctid();
    const long long tue = p.trace_items ? gtimer() : 0;
    cbar();  // the previous segment's down rows may still read its hidden values here
    const long long tu0 = p.trace_items ? gtimer() : 0;
    if (p.trace_items && tid == 0) trace_rec(c, 0x80000000u | (((unsigned)C_DOWN + 5) << 16) | (unsigned)l, 0u, tue, tu0);
    // the tokens of this expert: a routed expert takes only the tokens routed
    // to it when its input is one K panel -- read from the staging area when
    // every token's input is staged there (the routed CTAs stage it before
    // routing), else its own tokens are gathered into the staging area --
    // and otherwise all tokens, weight 0 or not; the shared expert takes
    // tokens [m_lo, m_hi), gathered when not every token's input is staged.
    // A routed expert with more tokens than the staging area holds runs once
    // per group: entries [m_lo, m_hi) of its list of tokens.
    if (tid < 32) {
        const bool one_panel = p.M > 1 && Ld.ffn.n_kc == 1;
        const bool all_staged = one_panel && stage_fits(p.M, Ld.ffn.Kc);
        const bool compact = expert >= 0 && one_panel;
        const int lane = tid;
        float w[2];
        bool sel[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int m = lane + 32 * q;
            const bool in = expert < 0 ? m >= m_lo && m < m_hi : m < p.M;
            w[q] = in ? (expert < 0 ? 1.0f : route_weight(c.ms, m, expert, p.topk)) : 0.f;
            // (the producer streams this unit's tiles for the same number of
            // tokens: the routing count, tokens of weight 0 included)
            sel[q] = in && (!compact || routed_to(c.ms, m, expert, p.topk));
        }
        unsigned b0 = __ballot_sync(0xffffffffu, sel[0]), b1 = __ballot_sync(0xffffffffu, sel[1]);
        const unsigned lt = (1u << lane) - 1u;
        if (compact) {  // this group's entries of the expert's token list
            const int q0 = __popc(b0 & lt), q1 = __popc(b0) + __popc(b1 & lt);
            sel[0] = sel[0] && q0 >= m_lo && q0 < m_hi;
            sel[1] = sel[1] && q1 >= m_lo && q1 < m_hi;
            b0 = __ballot_sync(0xffffffffu, sel[0]);
            b1 = __ballot_sync(0xffffffffu, sel[1]);
        }
        const int pos[2] = {__popc(b0 & lt), __popc(b0) + __popc(b1 & lt)};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (sel[q]) {
                c.ms.gt[pos[q]] = (uint8_t)(lane + 32 * q);
                c.ms.uw[pos[q]] = w[q];
            }
        }
        __syncwarp();
        if (lane == 0) {
            c.ms.gm = __popc(b0) + __popc(b1);
            if (p.debug)  // every entry of the token map is a token of the step
                for (int i = 0; i < c.ms.gm; ++i)
                    if (c.ms.gt[i] >= p.M) {
                        raise_status(p, ST_DEBUG, 0x9300u);
                        c.ms.abort = 1;
                    }
            // a key per token list: routed expert and group, or shared group
            c.ms.gather = one_panel && !all_staged && (expert >= 0 || m_hi - m_lo < p.M)
                              ? (expert >= 0 ? 1 + expert + 256 * m_lo : (1 << 24) + m_lo)
                              : 0;
        }
    }
    cbar();
    const int M = c.ms.gm;
    float* hs = unit_buf(c, 3 * F * n * M);
    float* h = hs + (size_t)rows * M;
    // two or more tokens on the tensor cores: the warps' K slices add into
    // the zeroed buffer (OUT_ADD) instead of meeting at two barriers per tile
    if (Ld.ffn.n_kc > 1 || M >= 2)
        for (int i = tid; i < rows * M; i += NCT) hs[i] = 0.f;
    if (tid == 0) {
        unit_gemv(p, Ld, c.ms.ug, kind, expert, u0, u1, hs);
        if (M >= 2 && mma_gemv(M, c.ms.ug)) c.ms.ug.out_kind = OUT_ADD;
    }
    cbar();
    const long long tz = p.trace_items ? gtimer() : 0;
    const long long cz = clock64();
    const int n_rb = 2 * K.Fi / K.R, rpu = 2 * F / K.R;
    if (p.f8) {
        unit_gu_f8(c, u0 * rpu, u1 * rpu, hs);
    } else {
        for (int kc = 0; kc < Ld.ffn.n_kc; ++kc)
            cons_gemv(c, c.ms.ug, 0, -1, kc * n_rb + u0 * rpu, kc * n_rb + u1 * rpu);
    }
    const long long tg = p.trace_items ? gtimer() : 0;
    const long long cg = clock64();
    // clock cycles: entry of the GEMV, its run start, its run end, return
    if (p.trace_items == 1 && tid == 0)
        trace_rec(c, 0x80000000u | (((unsigned)C_DOWN + 3) << 16) | (unsigned)l, (unsigned)(c.ms.tdbg[0] - cz),
                  c.ms.tdbg[1] - cz, cg - c.ms.tdbg[2]);
    cbar();
    const long long tu1 = p.trace_items ? gtimer() : 0;
    if (p.trace_items && tid == 0) trace_rec(c, 0x80000000u | (((unsigned)C_DOWN + 2) << 16) | (unsigned)l,
                                             (unsigned)(tz - tu0), tg, tu1);
    for (int i = tid; i < F * n * M; i += NCT) {
        const int m = i / (F * n), rem = i - m * F * n, uu = rem / F, f = rem - uu * F;
        const float* g = hs + (size_t)m * rows + uu * 2 * F;
        // (from L2 when the buffer is in global memory: the atomic additions
        // of OUT_ADD bypass this SM's L1)
        const float gv = __isShared(g) ? g[f] : __ldcg(g + f), uv = __isShared(g) ? g[F + f] : __ldcg(g + F + f);
        h[i] = silu(gv) * uv;
    }
    cbar();
    // down columns of each unit: tiles of Rd rows x F from the ring
    Misc& ms = c.ms;
    uint8_t* const ring = c.smem + SMEM_RING;
    CRing cr = c.cr;
    bool dead = c.dead, timed_out = false;
    // tiles in a rotated order per CTA: the CTAs' atomic additions into the
    // residual then go to different rows at any moment instead of all to the
    // same few L2 slices (the producer streams the same order)
    const int nt = (d + K.Rd - 1) / K.Rd, rot = (int)(blockIdx.x % (unsigned)nt);
    for (int uu = 0; uu < n; ++uu) {
        for (int t0 = 0; t0 < nt; ++t0) {
            const int t = t0 + rot < nt ? t0 + rot : t0 + rot - nt;
            const int r0 = t * K.Rd, nr = min(K.Rd, d - r0);
            const uint8_t* tile = nullptr;
            if (!dead) {
                if (spin_wait(p, &ms.full[cr.slot], cr.phase))
                    tile = ring + cr.slot * SLOT_BYTES;
                else
                    dead = timed_out = true;
            }
            if (tile) {
                if (M == 1 || p.f8) {
                    const float* hu = h + uu * F;
                    float* xo = Ld.xn + (size_t)ms.gt[0] * d + r0;
                    const float w = ms.uw[0];
                    if (p.f8) {
                        unit_down_f8(tile, nr, hu, xo, d);
                    } else if (w != 0.f) {
                        if (F == 64) down_rows1<8>(tile, nr, hu, w, xo);
                        else if (F == 48) down_rows1<6>(tile, nr, hu, w, xo);
                        else if (F == 32) down_rows1<4>(tile, nr, hu, w, xo);
                        else down_rows1<2>(tile, nr, hu, w, xo);
                    }
                } else {
                    float* xo = Ld.xn + r0;
                    const float* hu = h + uu * F;
                    if (F == 64) down_mma<64>(tile, nr, hu, n * F, M, ms, xo, d);
                    else if (F == 48) down_mma<48>(tile, nr, hu, n * F, M, ms, xo, d);
                    else if (F == 32) down_mma<32>(tile, nr, hu, n * F, M, ms, xo, d);
                    else down_mma<16>(tile, nr, hu, n * F, M, ms, xo, d);
                }
            }
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(&ms.empty[cr.slot]);
            if (++cr.slot == NSLOT) {
                cr.slot = 0;
                cr.phase ^= 1u;
            }
        }
    }
    // unit trace: segment start, gate/up + hidden done, down done; the first
    // field packs the token count, the unit count and the expert id
    if (p.trace_items && tid == 0)
        trace_rec(c, 0x80000000u | (((unsigned)C_DOWN + 1) << 16) | (unsigned)l,
                  ((unsigned)M << 16) | ((unsigned)(u1 - u0) << 8) | ((unsigned)expert & 0xffu), tu0, tu1);
    if (timed_out) {
        ms.abort = 1;
        raise_status(p, ST_TIMEOUT, 0x220u);
    }
    c.set_ring(cr);
    if (dead) c.dead = true;
}

// producer, MXFP8 experts: the segment's gate/up tiles, then each unit's
// down tiles in the consumers' rotated order; whole tiles, one bulk copy each
// (codes and scales are contiguous). L2 prefetch: once the first ring-full of
// copies is requested (a prefetch issued before them would queue ahead of
// them), the rest of the first units (about UNIT_PF_BYTES); then the next
// unit's tiles a unit ahead.
__device__ __noinline__ void unit_seg_prod_f8(Ctx& c, const FfnKind& K, int expert, int u0, int u1) {
    const Params& p = c.p;
    const int lane = threadIdx.x & 31;
    const uint8_t* gu = K.qgu + (expert >= 0 ? (size_t)expert * K.qgu_es : 0);
    const uint8_t* dn = K.qdn + (expert >= 0 ? (size_t)expert * K.qdn_es : 0);
    const int rpu = 2 * K.F / K.R, nt = p.d / K.Rd;
    const size_t ugu = (size_t)rpu * K.qtb_gu, udn = (size_t)nt * K.qtb_dn;  // bytes per unit
    const int npf = min(u1 - u0, max(1, UNIT_PF_BYTES / (int)(ugu + udn)));
    const unsigned piece = 65536;
    Misc& ms = c.ms;
    uint8_t* ring = c.smem + SMEM_RING;
    PRing pr = c.pr;
    int issued = c.issued;
    const unsigned long long pol = l2_evict_first();
    const int rot = (int)(blockIdx.x % (unsigned)nt);
    // tiles of the segment: gate/up j in [0, n_gu), then down
    const int n_gu = (u1 - u0) * rpu, n_all = n_gu + (u1 - u0) * nt, first = min(NSLOT, n_gu);
    for (int i = 0; i < n_all && !c.dead; ++i) {
        if (i == first) {
            // (gate/up tiles from `first` on; the down tiles of the first units)
            const size_t g0 = (size_t)u0 * ugu + (size_t)first * K.qtb_gu, g1 = (size_t)(u0 + npf) * ugu;
            for (size_t o = g0 + (size_t)lane * piece; o < g1; o += 32 * (size_t)piece)
                l2_prefetch(gu + o, (unsigned)min((size_t)piece, g1 - o));
            for (size_t o = (size_t)lane * piece, n = (size_t)npf * udn; o < n; o += 32 * (size_t)piece)
                l2_prefetch(dn + (size_t)u0 * udn + o, (unsigned)min((size_t)piece, n - o));
        }
        const uint8_t* src;
        unsigned bytes;
        if (i < n_gu) {
            src = gu + (size_t)(u0 * rpu + i) * K.qtb_gu;
            bytes = (unsigned)K.qtb_gu;
            // the gate/up tiles of units beyond the first npf, a unit ahead
            if (i % rpu == 0 && i / rpu + 1 < u1 - u0 && i / rpu + 1 >= npf)
                for (size_t o = (size_t)lane * piece; o < ugu; o += 32 * (size_t)piece)
                    l2_prefetch(gu + (size_t)(u0 + i / rpu + 1) * ugu + o, (unsigned)min((size_t)piece, ugu - o));
        } else {
            const int k = i - n_gu, uu = k / nt, t0 = k - uu * nt;
            const int t = t0 + rot < nt ? t0 + rot : t0 + rot - nt;
            src = dn + ((size_t)(u0 + uu) * nt + t) * K.qtb_dn;
            bytes = (unsigned)K.qtb_dn;
            if (t0 == 0 && uu + 1 < u1 - u0 && uu + 1 >= npf)
                for (size_t o = (size_t)lane * piece; o < udn; o += 32 * (size_t)piece)
                    l2_prefetch(dn + (size_t)(u0 + uu + 1) * udn + o, (unsigned)min((size_t)piece, udn - o));
        }
        if (p.debug && bytes > (unsigned)(SLOT_BYTES - 16)) {
            if (lane == 0) raise_status(p, ST_DEBUG, 0x9230u);
            c.dead = true;
            break;
        }
        int ok = 1;
        if (lane == 0) {
            if (spin_wait(p, &ms.empty[pr.slot], pr.phase ^ 1u)) {
                mbar_expect_tx(&ms.full[pr.slot], bytes);
                bulk_g2s_pol(ring + pr.slot * SLOT_BYTES, src, bytes, &ms.full[pr.slot], pol);
            } else {
                ok = 0;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0) raise_status(p, ST_TIMEOUT, 0x130u);
            c.dead = true;
            break;
        }
        ++issued;
        prod_next(pr);
    }
    c.set_pring(pr, issued);
}

// producer: the segment's tiles into the ring (and, first, towards L2)
__device__ __noinline__ void unit_seg_prod(Ctx& c, int kind, int expert, int u0, int u1, int ntok) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const FfnKind& K = Ld.ffn.k[kind];
    if (p.f8) {
        unit_seg_prod_f8(c, K, expert, u0, u1);
        return;
    }
    const int F = K.F, d = p.d, lane = threadIdx.x & 31, Kc = Ld.ffn.Kc;
    const uint16_t* gu = K.gu + (expert >= 0 ? (size_t)expert * K.gu_es : 0);
    const uint16_t* dn = K.dn + (expert >= 0 ? (size_t)expert * K.dn_es : 0);
    if (lane == 0) unit_gemv(p, Ld, c.ms.pug, kind, expert, u0, u1, nullptr);
    __syncwarp();
    const int n_rb = 2 * K.Fi / K.R, rpu = 2 * F / K.R;
    // the first ring-full of gate/up tiles is requested before the L2
    // prefetch of the rest of the segment, which would queue ahead of it
    const int first = min(NSLOT, (u1 - u0) * rpu);
    prod_gemv(c, c.ms.pug, -1, u0 * rpu, u0 * rpu + first, ntok);
    // then the L2 prefetch of the segment's first units (per K panel their
    // gate/up rows are contiguous, and so are their down blocks; pieces of at
    // most 64 KB, one lane each). Only about UNIT_PF_BYTES per CTA up front:
    // every CTA's whole segment at once would not fit in L2. The gate/up
    // copies that follow keep their own prefetch window; the down loop
    // prefetches one unit ahead.
    const size_t piece = 32768;  // elements
    const int unit_elems = 3 * F * d;
    const int npf = min(u1 - u0, max(1, UNIT_PF_BYTES / (2 * unit_elems)));
    {
        for (int kc = 0; kc < Ld.ffn.n_kc; ++kc) {
            const uint16_t* b = gu + (size_t)kc * 2 * K.Fi * Kc + (size_t)u0 * 2 * F * Kc;
            const size_t n = (size_t)npf * 2 * F * Kc;
            for (size_t o = (size_t)lane * piece; o < n; o += 32 * piece)
                l2_prefetch(b + o, (unsigned)(min(piece, n - o) * 2));
        }
        const uint16_t* b = dn + (size_t)u0 * d * F;
        const size_t n = (size_t)npf * d * F;
        for (size_t o = (size_t)lane * piece; o < n; o += 32 * piece) l2_prefetch(b + o, (unsigned)(min(piece, n - o) * 2));
    }
    for (int kc = 0; kc < Ld.ffn.n_kc && !c.dead; ++kc)
        prod_gemv(c, c.ms.pug, -1, kc * n_rb + u0 * rpu + (kc == 0 ? first : 0), kc * n_rb + u1 * rpu, ntok);
    Misc& ms = c.ms;
    uint8_t* ring = c.smem + SMEM_RING;
    PRing pr = c.pr;
    int issued = c.issued;
    const unsigned long long pol = l2_evict_first();
    const int nt = (d + K.Rd - 1) / K.Rd, rot = (int)(blockIdx.x % (unsigned)nt);  // the consumers' tile order
    for (int u = u0; u < u1 && !c.dead; ++u) {
        if (u + 1 < u1 && u + 1 >= u0 + npf) {
            const uint16_t* b = dn + (size_t)(u + 1) * d * F;
            const size_t n = (size_t)d * F;
            for (size_t o = (size_t)lane * piece; o < n; o += 32 * piece)
                l2_prefetch(b + o, (unsigned)(min(piece, n - o) * 2));
        }
        for (int t0 = 0; t0 < nt; ++t0) {
            const int t = t0 + rot < nt ? t0 + rot : t0 + rot - nt;
            const int r0 = t * K.Rd, nr = min(K.Rd, d - r0);
            const unsigned bytes = (unsigned)nr * F * 2u;
            if (p.debug && bytes > (unsigned)(SLOT_BYTES - 16)) {
                if (lane == 0) raise_status(p, ST_DEBUG, 0x9220u);
                c.dead = true;
                break;
            }
            int ok = 1;
            if (lane == 0) {
                if (spin_wait(p, &ms.empty[pr.slot], pr.phase ^ 1u)) {
                    mbar_expect_tx(&ms.full[pr.slot], bytes);
                    bulk_g2s_pol(ring + pr.slot * SLOT_BYTES, dn + ((size_t)u * d + r0) * F, bytes, &ms.full[pr.slot], pol);
                } else {
                    ok = 0;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) raise_status(p, ST_TIMEOUT, 0x120u);
                c.dead = true;
                break;
            }
            ++issued;
            prod_next(pr);
        }
    }
    c.set_pring(pr, issued);
}

// the FFN of layer l: the shared expert's units on CTAs [0, gs), the router
// result and the routed experts' units (slot-major) on the others
template <bool PROD>
__device__ __noinline__ void ffn_stage(Ctx& c, int l) {
    const Params& p = c.p;
    const Layer& Ld = c.layer();
    const long long t0 = gtimer();
    c.cur_code = ((unsigned)C_DOWN << 16) | (unsigned)l;
    int done = 0;
    // the shared expert's units run once per group of tokens (work items
    // unit x group): groups of 4 when every token's input is staged in one K
    // panel (more CTAs, and the register GEMV path); groups as large as the
    // staging area holds when not (each group's tokens gathered there)
    const bool stage_all = p.M > 1 && Ld.ffn.n_kc == 1 && stage_fits(p.M, Ld.ffn.Kc);
    const int tgs = shared_group(p.M, Ld.ffn.n_kc, Ld.ffn.Kc);
    const int ntg = (p.M + tgs - 1) / tgs;
    if ((int)blockIdx.x < p.gs) {
        if (p.has_sh) {
            const int nu = Ld.ffn.k[1].nu;
            int lo, hi;
            my_range_sub(nu * ntg, 0, p.gs, lo, hi);
            if (lo < hi) {
                if constexpr (!PROD) {
                    const bool pre = ntg > 1 && stage_all;
                    if (pre && threadIdx.x == 0) unit_gemv(p, Ld, c.ms.ug, 1, -1, 0, 1, c.red() + RED_FLOATS / 2);
                    set_deps(c, deps1(l, C_O, (unsigned)gemv_items(Ld.g[G_O])));
                    cwait(c, 0x1100u | (unsigned)(l << 16));
                    if (pre) restage(c, c.ms.ug, Ld.x, 0, 0, 0, p.M);
                }
                for (int i = lo; i < hi && !(PROD && c.dead);) {
                    const int tg = i / nu, iend = min(hi, (tg + 1) * nu);
                    const int m0 = tg * tgs, m1 = min(p.M, m0 + tgs);
                    if constexpr (PROD)
                        unit_seg_prod(c, 1, -1, i - tg * nu, iend - tg * nu, m1 - m0);
                    else
                        unit_seg_cons(c, l, 1, -1, i - tg * nu, iend - tg * nu, m0, m1);
                    i = iend;
                }
                done += hi - lo;
            }
        }
        if (p.E > 0 && !route<PROD>(c, l) && PROD) {
            c.dead = true;
            return;
        }
    } else {
        if constexpr (!PROD) {
            // stage the normalised input of the expert GEMVs while the router
            // is still running (it depends only on the residual and the FFN
            // norm gain, not on the routing)
            if (threadIdx.x == 0) unit_gemv(p, Ld, c.ms.ug, 0, 0, 0, 1, c.red() + RED_FLOATS / 2);
            set_deps(c, deps1(l, C_O, (unsigned)gemv_items(Ld.g[G_O])));
            cwait(c, 0x1200u | (unsigned)(l << 16));
            if (stage_fits(p.M, Ld.ffn.Kc)) restage(c, c.ms.ug, Ld.x, 0, 0, 0, p.M);
        }
        const long long tr0 = p.trace_items ? gtimer() : 0;
        if (!route<PROD>(c, l) && PROD) {
            c.dead = true;
            return;
        }
        if (!PROD && p.trace_items && threadIdx.x == 0)
            trace_rec(c, 0x80000000u | (((unsigned)C_DOWN + 4) << 16) | (unsigned)l, 0u, tr0, gtimer());
        const FfnKind& K = Ld.ffn.k[0];
        const int nslots = PROD ? c.ms.p_nslots : c.ms.n_slots;
        const uint8_t* slot_e = PROD ? c.ms.p_slot_e : c.ms.slot_e;
        int lo, hi;
        // (the router CTAs take routed units too once their router tile is done)
        routed_range(PROD ? c.ms.p_used : c.ms.used, slot_e, nslots, K.nu, (int)blockIdx.x - p.gs, p.G - p.gs, lo,
                     hi);
        // a routed expert's units take its own tokens (one K panel), in groups
        // of as many as the staging area holds when not all tokens fit it
        // (g0: the group's first entry of the expert's token list)
        for (int i = lo, g0 = 0; i < hi && !(PROD && c.dead);) {
            const int s2 = i / K.nu, iend = min(hi, (s2 + 1) * K.nu), e = slot_e[s2];
            const bool one_panel = p.M > 1 && Ld.ffn.n_kc == 1;
            const int cnt = one_panel ? (int)(PROD ? c.ms.p_used[e] : c.ms.used[e]) : p.M;
            const int cap = one_panel && !stage_fits(p.M, Ld.ffn.Kc) ? STAGE_FLOATS / stage_stride(Ld.ffn.Kc) : MAX_M;
            const int g1 = min(cnt, g0 + cap);
            if constexpr (PROD)
                unit_seg_prod(c, 0, e, i - s2 * K.nu, iend - s2 * K.nu, one_panel ? g1 - g0 : p.M);
            else
                unit_seg_cons(c, l, 0, e, i - s2 * K.nu, iend - s2 * K.nu, g0, g1);
            if (g1 < cnt) {
                g0 = g1;
            } else {
                g0 = 0;
                i = iend;
            }
        }
        done = hi - lo;
    }
    const int nslots = PROD ? c.ms.p_nslots : c.ms.n_slots;
    c.set_count(c.n_down, (p.has_sh ? Ld.ffn.k[1].nu * ntg : 0) + (p.E > 0 ? nslots * Ld.ffn.k[0].nu : 0));
    if constexpr (!PROD) {
        csignal(c, l, C_DOWN, (unsigned)done);
        // back to all tokens in order for the stages that follow (their
        // readers pass a barrier first)
        if (threadIdx.x < MAX_M) c.ms.gt[threadIdx.x] = (uint8_t)threadIdx.x;
        if (threadIdx.x == 0) {
            c.ms.gm = p.M;
            c.ms.gather = 0;
        }
        trace_rec(c, ((unsigned)C_DOWN << 16) | (unsigned)l, (unsigned)done, t0, t0);
    }
}

// verify acceptance (consumers of CTA 0): 1 + the number of leading draft
// tokens that equal the argmax of the logits at the position before them
__device__ __noinline__ void accept_cons(Ctx& c) {
    const Params& p = c.p;
    set_deps(c, deps1(p.L, C_AMAX, (unsigned)p.M));
    cwait(c, 0xb00u);
    const int b = ctid();
    if (b < p.B && !c.dead) {
        int a = 0;
        while (a < p.T - 1 && __ldcg(p.amax + b * p.T + a) == p.tokens[b * p.T + a + 1]) ++a;
        p.accept[b] = a + 1;
    }
}

// ============================================================ program ====
// The decode step is a fixed sequence of stages: per layer
//   MLA: A QB APP QLAT ATTN COMB UV O, GQA: A ATTN COMB O,
//   then ROUTER CARRY FFN (expert units: shared on CTAs [0, gs), routed on the rest)
// (stages the model does not have are skipped), then LM ARGMAX ACCEPT.
// exec_stage() runs one stage and advances the position, which lives in
// shared memory like the rest of the program state: the stage bodies are
// large functions, and anything a caller kept in registers across a call
// into them would be spilled to local memory.
enum StageId {
    S_A = 0, S_QB, S_APP, S_QLAT, S_ATTN, S_COMB, S_UV, S_O, S_ROUTER, S_CARRY, S_FFN,
    S_NLAYER, S_LM = S_NLAYER, S_AMAX, S_ACCEPT, S_END
};

// position of (layer, stage) in the program: layer stages l * S_NLAYER + st,
// then the head's stages from L * S_NLAYER on
__host__ __device__ __forceinline__ int prog_index(const Params& p, int l, int st) {
    return l * S_NLAYER + (l < p.L ? st : st - S_LM);
}

template <bool PROD>
__device__ __noinline__ bool exec_stage(Ctx& c) {
    const Params& p = c.p;
    if constexpr (PROD) {
        if (c.dead) return false;
    }
    const int l = c.pl, st = c.pst;
    if (st == S_END || (p.staged && prog_index(p, l, st) >= p.st_hi)) {
        // the consumers' last stage ended at a barrier: every slot they read
        // was filled and released
        if (!PROD && p.debug && threadIdx.x == 0) debug_canaries(p, c.smem, true);
        return false;
    }
    {
        int nl = l, nst = st + 1;
        if (l < p.L && nst == S_NLAYER) {
            nl = l + 1;
            nst = nl == p.L ? S_LM : 0;
        }
        c.set_pos(nl, nst);
    }
    const bool mla = p.attn == 1;
    // GEMV-type stages set these and fall through to the common tail
    const Gemv* g = nullptr;
    Deps deps;
    deps.n = 0;
    int sig = 0, ls = l;
    int c0 = 0, gc = 0;  // gc > 0: the stage's items go to CTAs [c0, c0 + gc) only
    if (l < p.L) {
        const Layer& Ld = c.layer();
        switch (st) {
            case S_A: {
                load_layer<PROD>(c, l);
                if constexpr (PROD) {
                    if (mla) prefetch_attn_mla(c, l);
                    prefetch_next_small(c, l);
                }
                if (l == 0) {
                    deps = deps1(p.L, C_INIT, (unsigned)p.G);
                } else {
                    deps.n = 3;
                    deps.d[0] = {l - 1, C_DOWN, (unsigned)c.n_down};
                    deps.d[1] = {l - 1, C_SHDOWN, (unsigned)c.n_shdown};
                    deps.d[2] = {l - 1, C_CARRY, (unsigned)c.n_carry};
                }
                c.set_count(c.n_down, 0);
                c.set_count(c.n_shdown, 0);
                c.set_count(c.n_carry, 0);
                g = &c.layer().g[G_A];
                sig = C_A;
                break;
            }
            case S_QB:
                if (!mla) return true;
                if (p.qfuse) {
                    const int n = gemv_items(Ld.g[G_QB]);
                    int lo, hi;
                    my_range(p, n, c.off, lo, hi);
                    c.advance(n);
                    if (lo >= hi) return true;
                    if constexpr (PROD) {
                        qb_fused_prod(c, lo, hi);
                    } else {
                        set_deps(c, deps1(l, C_A, (unsigned)gemv_items(Ld.g[G_A])));
                        qb_fused_cons(c, l, lo, hi);
                    }
                    return true;
                }
                g = &Ld.g[G_QB];
                deps = deps1(l, C_A, (unsigned)gemv_items(Ld.g[G_A]));
                sig = C_QB;
                break;
            case S_APP: {
                if (!mla) return true;
                int lo, hi;
                my_range(p, p.M, c.off, lo, hi);
                c.advance(p.M);
                if (!PROD && lo < hi) {
                    set_deps(c, deps1(l, C_A, (unsigned)gemv_items(Ld.g[G_A])));
                    append_cons(c, l, lo, hi);
                }
                return true;
            }
            case S_QLAT:
                if (!mla || p.qfuse) return true;
                g = &Ld.g[G_QLAT];
                deps = deps1(l, C_QB, (unsigned)gemv_items(Ld.g[G_QB]));
                sig = C_QLAT;
                break;
            case S_ATTN: {
                const int n = attn_items(p);
                int lo, hi;
                my_range(p, n, c.off, lo, hi);
                c.advance(n);
                if (lo >= hi) return true;
                if constexpr (PROD) {
                    prod_attn(c, l, lo, hi);
                } else {
                    Deps da;
                    if (mla) {
                        da.n = 2;
                        da.d[0] = p.qfuse ? Dep{l, C_QB, (unsigned)gemv_items(Ld.g[G_QB])}
                                          : Dep{l, C_QLAT, (unsigned)gemv_items(Ld.g[G_QLAT])};
                        da.d[1] = {l, C_APP, (unsigned)p.M};
                    } else {
                        da = deps1(l, C_A, (unsigned)gemv_items(Ld.g[G_A]));
                    }
                    set_deps(c, da);
                    attn_cons(c, l, lo, hi);
                }
                return true;
            }
            case S_COMB: {
                const int n = comb_items(p);
                int lo, hi;
                my_range(p, n, c.off, lo, hi);
                c.advance(n);
                if (lo < hi) {
                    if constexpr (PROD) {
                        if (mla && p.ufuse) comb_prod(c, lo, hi);
                    } else {
                        set_deps(c, deps1(l, C_ATTN, (unsigned)attn_items(p)));
                        comb_cons(c, l, lo, hi);
                    }
                }
                return true;
            }
            case S_UV:
                if (!mla || p.ufuse) return true;
                g = &Ld.g[G_UV];
                deps = deps1(l, C_COMB, (unsigned)comb_items(p));
                sig = C_UV;
                break;
            case S_O:
                g = &Ld.g[G_O];
                deps = mla && !p.ufuse ? deps1(l, C_UV, (unsigned)gemv_items(Ld.g[G_UV]))
                                       : deps1(l, C_COMB, (unsigned)comb_items(p));
                sig = C_O;
                break;
            // the router runs on its own CTAs [G - gr, G): the routed units
            // wait for it, the shared units do not
            case S_ROUTER:
                if (p.E == 0 || p.rfuse) return true;
                g = &Ld.g[G_ROUTER];
                deps = deps1(l, C_O, (unsigned)gemv_items(Ld.g[G_O]));
                sig = C_ROUTER;
                c0 = p.G - p.gr;
                gc = p.gr;
                break;
            case S_CARRY: {
                if (!p.carry) return true;
                const int chunk = 2048;
                const int n = (p.M * p.d + chunk - 1) / chunk;
                c.set_count(c.n_carry, n);
                int lo, hi;
                my_range(p, n, c.off, lo, hi);
                c.advance(n);
                if (!PROD && lo < hi) {
                    set_deps(c, deps1(l, C_O, (unsigned)gemv_items(Ld.g[G_O])));
                    carry_cons(c, l, lo, hi);
                }
                return true;
            }
            case S_FFN:
                ffn_stage<PROD>(c, l);
                return true;
            default:
                return true;
        }
    } else {
        switch (st) {
            case S_LM:
                g = &p.lm;
                deps.n = 3;
                deps.d[0] = {p.L - 1, C_DOWN, (unsigned)c.n_down};
                deps.d[1] = {p.L - 1, C_SHDOWN, (unsigned)c.n_shdown};
                deps.d[2] = {p.L - 1, C_CARRY, (unsigned)c.n_carry};
                sig = C_LM;
                ls = p.L;
                break;
            case S_AMAX: {
                if (!p.accept) return true;
                int lo, hi;
                my_range(p, p.M, c.off, lo, hi);
                c.advance(p.M);
                if (!PROD && lo < hi) {
                    set_deps(c, deps1(p.L, C_LM, (unsigned)gemv_items(p.lm)));
                    argmax_cons(c, lo, hi);
                }
                return true;
            }
            case S_ACCEPT:
                if (!PROD && p.accept && blockIdx.x == 0) accept_cons(c);
                return true;
            default:
                return true;
        }
    }
    // plain GEMV stage (rank among the np CTAs that have items: for the
    // norm sums of split-panel inputs)
    const int n = gemv_items(*g);
    int lo, hi, rank, np;
    if (gc > 0) {
        my_range_sub(n, c0, gc, lo, hi);
        np = min(n, gc);
        rank = n >= gc ? (int)blockIdx.x - c0 : lo;
    } else {
        int v = (int)blockIdx.x + c.off;
        if (v >= p.G) v -= p.G;
        my_range(p, n, c.off, lo, hi);
        c.advance(n);
        np = min(n, p.G);
        rank = n >= p.G ? v : lo;
    }
    if (lo >= hi) return true;
    if constexpr (PROD) {
        if (!c.dead) prod_plain(c, *g, lo, hi);
    } else {
        set_deps(c, deps);
        c.st_rank = rank;
        c.st_np = np;
        cons_mm(c, ls, *g, sig, lo, hi);
    }
    return true;
}

// producer epilogue after an abort: wait (bounded) for the bulk copies it
// issued so none lands in shared memory after the CTA has exited
__device__ void prod_drain(Ctx& c) {
    if ((threadIdx.x & 31) != 0) return;
    // slots filled but possibly not yet consumed are the last NSLOT ones
    PRing r = c.pr;
    const int n = c.issued < NSLOT ? c.issued : NSLOT;
    for (int i = 0; i < n; ++i) {
        if (r.slot == 0) {
            r.slot = NSLOT - 1;
            r.phase ^= 1u;
        } else {
            --r.slot;
        }
        // the fill of this slot completed phase `r.phase`; wait for it
        const long long t0 = gtimer();
        while (!mbar_test(&c.ms.full[r.slot], r.phase)) {
            if (gtimer() - t0 > c.p.timeout_ns) break;
        }
    }
}


__global__ void __launch_bounds__(NTHREADS, 1) megakernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];  // 1024: the swizzled MLA boxes of the ring
    Misc& ms = *reinterpret_cast<Misc*>(smem + SMEM_MISC);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&ms.full[i], 1);
            mbar_init(&ms.empty[i], NCW);
        }
        // a step that failed earlier leaves the abort flag set until the host
        // resets it (mk_step_status): refuse to run on stale state
        ms.abort = ld_relaxed(&p.status[1]) ? 1 : 0;
        ms.n_slots = ms.p_nslots = 0;
        for (int i = 0; i < MAX_M; ++i) ms.gt[i] = (uint8_t)i;
        ms.gm = p.M;
        ms.gather = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {
        static_assert(sizeof(Params) % 4 == 0, "Params is copied in 4-byte words");
        const uint32_t* ps = reinterpret_cast<const uint32_t*>(&p);
        uint32_t* pd = reinterpret_cast<uint32_t*>(smem + SMEM_PARAMS);
        for (int i = threadIdx.x; i < (int)(sizeof(Params) / 4); i += blockDim.x) pd[i] = ps[i];
    }
    __syncthreads();
    if (ms.abort) return;
    // each warp's schedule state lives in shared memory (its lanes hold the
    // same values): local memory would miss the small L1 left beside the
    // 220 KB of shared memory this kernel uses
    Ctx* cx = reinterpret_cast<Ctx*>(smem + SMEM_CTX) + (threadIdx.x >> 5);
    if ((threadIdx.x & 31) == 0) new (cx) Ctx(*reinterpret_cast<const Params*>(smem + SMEM_PARAMS), smem);
    __syncwarp();
    Ctx& c = *cx;
    if (p.staged) {
        // one launch per stage: the previous launch's results must be visible
        // before this one reads anything it wrote (programmatic dependent
        // launch lets this launch's set-up above overlap the previous one's
        // tail); then start at the window's first stage with that layer's
        // descriptors in place
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (p.staged == 1) {
            int l = p.st_lo / S_NLAYER, st = p.st_lo - l * S_NLAYER;
            if (l >= p.L) {
                l = p.L;
                st = p.st_lo - p.L * S_NLAYER + S_LM;
            }
            c.set_pos(l, st);
            if (l < p.L && st != S_A) {
                if (threadIdx.x >= NCT)
                    load_layer<true>(c, l);
                else
                    load_layer<false>(c, l);
            }
        }
    }
    if (threadIdx.x >= NCT) {
        if (prod_check(c.p)) {
            if (p.staged != 2)
                while (exec_stage<true>(c)) {
                }
        } else {
            c.dead = true;
        }
        if (c.dead) prod_drain(c);
    } else {
        if (init_phase(c) && p.staged != 2)
            while (exec_stage<false>(c)) {
            }
    }
}

}  // namespace mk
