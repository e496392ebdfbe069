// moe_decode.cuh -- the persistent decode kernel: whole MoE layers (or a
// stack of them) for small decode batches in one cooperative launch with
// two device-wide barriers per layer.
//
// Why this shape.  At decode sizes a layer is a chain of short dependent
// steps -- router -> top-k -> experts -> combine -> next router -- and the
// time goes into the hand-offs, not the arithmetic.  The kernel therefore
//  * computes the router logits of layer l+1 inside layer l's combine: every
//    CTA owns a slice of hidden rows, forms x_{l+1} for those rows and adds
//    its partial dot products with the next router's columns into a
//    fixed-point (int64, 2^-32) accumulator -- integer sums are exact, so the
//    logits do not depend on the order in which CTAs arrive;
//  * repeats the top-k and the grouping redundantly in every CTA (a few
//    hundred bytes of logits), so no barrier separates routing from experts;
//  * streams each CTA's share of the selected experts' weights -- gate/up
//    row pairs first, then down rows -- through a shared-memory ring filled by
//    one producer warp with bulk asynchronous copies (TMA engine, mbarrier
//    completion), so the down weights are already on chip when the barrier
//    after the gate/up pass releases.
// ("MoE Performance Optimization Analysis": GPU routing, no CPU read and no
// wait per layer; "TEXT Generation Optimization Report": the layer loop runs
// without a wait; "perf(cpu-moe) ... #46": each selected expert's weights are
// read once, split by (expert, row block).)
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>

#include "moe_common.cuh"
#include "moe_ptx.cuh"

namespace moe {

constexpr int kDkConsumers = 12;                   // consumer warps
constexpr int kDkThreads = 32 * (kDkConsumers + 1);  // + one producer warp
constexpr int kDkMaxB = 4;
constexpr int kDkMaxR = 32;
constexpr int kDkMaxStages = 32;
constexpr uint32_t kDkWaitLimit = 1u << 22;
constexpr unsigned long long kDkSpinLimit = 1ull << 22;
// Counted fixed-point words (see dk_router_partials): a CTA's value v adds
// q + kFixBias + kFixCount to a word, q = round(v * scale) with |q| <
// kFixBias = 2^49.  The low 57 bits hold the sum of up to 127 such terms
// (each below 2^50) without overflow, bits 57..63 count them; a word whose
// count reaches the number of contributing CTAs holds the exact sum of
// every q, whatever order the terms arrived in.
constexpr unsigned long long kFixCount = 1ull << 57;
constexpr long long kFixBias = 1ll << 49;
constexpr float kFixScale = 268435456.0f;  // 2^28 for logits: |v| < 2^21, steps of 2^-28
constexpr float kFixScaleSq = 65536.0f;    // 2^16 for sums of x^2: |v| < 2^33
constexpr int kDkSmemMax = 227 * 1024;
constexpr int kDkGChunks = 8;  // direct mode: gate/up rows land on this many barriers (in issue order)

struct DkParams {
    int B, H, I, E, k, L;
    int x_bf16;
    unsigned flags;
    const void* x_in;       // layer input (stack: the fp32 residual stream)
    const float* residual;  // added to the layer output (stack: x itself)
    float* y;               // layer output (stack: x, updated in place)
    LayerWeights layer[MOE_MAX_LAYERS];
    int32_t* ids_out;  // [L, B, k] or nullptr
    float* w_out;      // [B, k] (single layer) or nullptr
    // the grouped route list of the layer, as moe_group_by_expert lays it
    // out (written by CTA 0; a stack leaves its last layer's)
    int32_t *g_offsets, *g_route_idx, *g_unique, *g_num_unique;
    float* h;          // [2][R, I] exchange buffer, by layer parity
    unsigned long long* xt;   // [2][B][H] tagged x: (layer << 32) | bits of x_layer[t][h], layers >= 1, by parity
    unsigned long long* acc;  // [2][kDkShadows][B][E] fixed-point logits
    float* alog;              // [B][E] next layer's logits predicted from this layer's input
    int prefetch_k;           // experts per token to prefetch into L2 for the next layer (0: off)
    unsigned* bar;            // [0] arrival counter, [1] abort word
    unsigned bar_extra;       // arrivals a barrier waits for beyond the grid (0; > 0 only to test the timeout)
    int32_t* status;
    int S, stage_bytes, maxrows;
    int W;  // consumer warps that take chunks: stage s always goes to warp s % W (S % W == 0)
    unsigned long long* trace;  // optional phase timestamps (see dk_trace), or nullptr
    int trace_words;
    int off_misc, off_x, off_xq, off_h, off_o, off_wr, off_ring;
    int off_gq;  // pre-norm stacks: [2][H] fp32, layer m's norm weights in buffer m & 1
    // pre-norm stacks: layer l's input is RMSNorm_l(x_l) = x_l * rn * norm_l
    // with rn = 1/sqrt(mean(x_l^2) + eps); the residual is x_l itself
    int has_norm;
    float eps;
};

struct __align__(16) DkMisc {
    int abort_flag;
    int sync_ok;
    int U;
    int ids[kDkMaxR];
    float selv[kDkMaxR];  // selected logits, rank order
    float w[kDkMaxR];
    int pos[kDkMaxR];   // position of route r in the grouped list
    int rat[kDkMaxR];   // route at position p
    int seg_e[kDkMaxR];
    int seg_p[kDkMaxR + 1];
    int last_pos[kDkMaxStages];  // latest ring position armed in each stage (-1: none)
    int mid_epoch;               // layers whose mid-layer barrier has completed (for the producer warp)
    float rn[kDkMaxB];           // pre-norm stacks: 1/sqrt(mean(x^2) + eps) of each token's layer input
    int ga_tab[kDkMaxR + 1];     // this CTA's gate/up pair range [ga_tab[U], gb_tab[U]) for U segments
    int gb_tab[kDkMaxR + 1];
};

// --------------------------------------------------------- work partition
// Hidden rows owned by CTA c in the down/combine/router step: groups of 8
// rows (16-byte aligned bf16 slices), split as evenly as possible.
__device__ __forceinline__ void dk_rows(int c, int G, int H, int& h0, int& h1) {
    const long long ng = H >> 3;
    h0 = 8 * (int)((long long)c * ng / G);
    h1 = 8 * (int)((long long)(c + 1) * ng / G);
}

struct DkWork {
    int ga, gb;  // gate/up pairs [ga, gb)
    int h0, h1, nr, nd_per_u, ng, n;
};

// Rows, down-chunk size and down chunks per expert are fixed per launch
// (template `base`); only the gate/up range depends on the routing, through
// the number of segments U, so it is tabulated for every U at the start.
// The U*I gate/up row pairs (numbered segment-major) are split into equal
// counts: CTA c takes [floor(c*U*I/G), floor((c+1)*U*I/G)).  (The down rows
// are split evenly too, in 8-row groups.  Equal pair counts beat an equal
// split of each CTA's total bytes, gate/up plus down: the gate/up pass ends
// at a device-wide barrier, so its slowest CTA sets the pace, while the
// down rows land during that pass anyway.)
__device__ __forceinline__ void dk_work_range(int U, int I, int& ga, int& gb) {
    const long long G = gridDim.x, c = blockIdx.x, P = (long long)U * I;
    ga = (int)(c * P / G);
    gb = (int)((c + 1) * P / G);
}

__device__ __forceinline__ DkWork dk_work(const DkWork& base, int U, const DkMisc* m) {
    DkWork w = base;
    w.ga = m->ga_tab[U];
    w.gb = m->gb_tab[U];
    w.ng = w.gb - w.ga;
    w.n = w.ng + U * w.nd_per_u;
    return w;
}

// ------------------------------------------------------------- barriers
// Device-wide barrier among the threads of named barrier `bar_id`
// (`nthreads` of them) in every CTA: after the CTA-wide barrier the leader
// thread adds 1 to a shared arrival counter with a release reduction (no
// value returned) and polls it with acquire loads until it reaches epoch * G.
// (An atomic that returns the old value, relaxed polling and an acquire
// fence measured 3 % slower on the 30-layer stack; a flag per CTA polled by
// every CTA, a master-released flag array and a two-level counter tree were
// slower still.)  The release is cumulative: it orders every access of the
// CTA that precedes the CTA-wide barrier, whichever thread made it.
// p.bar[0] = counter, p.bar[1] = abort word.  Bounded: after kDkSpinLimit
// polls the CTA sets MOE_DEV_TIMEOUT and the abort word and reports failure.
constexpr int kDkLeader = 32;  // first consumer thread
constexpr int kDkShadows = 2;  // copies of the logit accumulator (CTA c adds into copy c mod 2)

// The logit accumulators of layer l: [kDkShadows][B][E] counted fixed-point
// words, three sets in rotation (set l mod 3 is read by layer l, set l+1 is
// filled during layer l, set l+2 -- read by layer l-1 -- is cleared during
// layer l, between that layer's mid barrier and the next one).
__device__ __forceinline__ unsigned long long* dk_acc(const DkParams& p, int l) {
    return p.acc + (size_t)(l % 3) * kDkShadows * p.B * p.E;
}

// Pre-norm stacks: the counted fixed-point sums of x^2 of layer l's input,
// [kDkShadows][B], three sets behind the logit accumulators.
__device__ __forceinline__ unsigned long long* dk_nacc(const DkParams& p, int l) {
    return p.acc + (size_t)3 * kDkShadows * p.B * p.E + (size_t)(l % 3) * kDkShadows * p.B;
}

// CTAs that add into shadow copy sh (those with blockIdx.x mod kDkShadows == sh).
__device__ __forceinline__ unsigned dk_shadow_ctas(int sh) {
    return (gridDim.x - (unsigned)sh + kDkShadows - 1) / kDkShadows;
}


__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void ld_relaxed_gpu_u64x2(const unsigned long long* p, unsigned long long& a,
                                                     unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ bool dk_grid_sync(const DkParams& p, unsigned& epoch, DkMisc* m, int bar_id,
                                             int nthreads) {
    named_sync(bar_id, nthreads);
    if (threadIdx.x == kDkLeader) {
        epoch += 1;
        const unsigned target = epoch * (gridDim.x + p.bar_extra);
        int ok = 1;
        red_release_gpu_add(p.bar, 1u);
        unsigned long long spins = 0;
        while (ld_acquire_gpu(p.bar) < target) {
            ++spins;
            if ((spins & 63ull) == 0 && ld_relaxed_gpu(p.bar + 1) != 0u) {
                ok = 0;
                break;
            }
            if (spins > kDkSpinLimit) {
                set_status(p.status, MOE_DEV_TIMEOUT);
                atomicExch(p.bar + 1, 1u);
                ok = 0;
                break;
            }
        }
        m->sync_ok = ok;
        if (!ok) m->abort_flag = 1;
    }
    __syncwarp();
    named_sync(bar_id, nthreads);
    return m->sync_ok != 0;
}

// mbarrier wait that also gives up when the CTA has aborted; bounded by
// kDkWaitLimit tries.
__device__ __forceinline__ bool dk_wait(uint64_t* bar, uint32_t parity, DkMisc* m, const DkParams& p) {
    for (uint32_t i = 0; i < kDkWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 31u && *(volatile int*)&m->abort_flag) return false;
    }
    set_status(p.status, MOE_DEV_TIMEOUT);
    atomicExch(p.bar + 1, 1u);
    *(volatile int*)&m->abort_flag = 1;
    return false;
}

// Phase timestamps for profiling: word pair (globaltimer ns, SM clock) of
// event `ev` (0..23) of layer `l` (-1 = the initial router step) of this CTA.
// The kernel is compiled twice: without any of this code (the default) and
// with it (only while a trace buffer is set), so that the untraced kernel's
// instruction footprint stays small.
template <bool kTrace>
__device__ __forceinline__ void dk_trace(const DkParams& p, int l, int ev) {
    if (!kTrace || p.trace == nullptr) return;
    const long long idx = (((long long)(l + 1) * gridDim.x + blockIdx.x) * 24 + ev) * 2;
    if (idx + 1 >= p.trace_words) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.trace[idx] = t;
    p.trace[idx + 1] = (unsigned long long)clock64();
}

// ----------------------------------------------------------- small steps
// One CTA's contribution of v at `scale` into the counted word w.
// |v * scale| must stay below 2^49: a larger value is clamped
// (MOE_DEV_RANGE), a non-finite one counts as 0 (MOE_DEV_NONFINITE).
__device__ __forceinline__ void fix_add(unsigned long long* w, float v, float scale, int32_t* status) {
    const float lim = 562949953421312.0f;  // 2^49
    float z = v * scale;
    if (!(fabsf(z) < lim)) {
        const bool fin = isfinite(z);
        set_status(status, fin ? MOE_DEV_RANGE : MOE_DEV_NONFINITE);
        z = fin ? copysignf(0.5f * lim, z) : 0.f;
    }
    red_add_u64(w, (unsigned long long)(__float2ll_rn(z) + kFixBias) + kFixCount);
}

// The sum of the n contributions of a complete counted word (exact).
__device__ __forceinline__ long long fix_sum(unsigned long long w, unsigned n) {
    return (long long)(w & (kFixCount - 1ull)) - (long long)n * kFixBias;
}

// The kDkShadows copies of one counted word (copy sh at w + sh * stride),
// waited for (bounded) together: each round loads the copies not yet
// complete at once, so that the wait ends one round trip after the last of
// them completes.  sum: their exact integer sum; false when aborting.
__device__ __forceinline__ bool dk_poll_sum(const unsigned long long* w, size_t stride, long long& sum,
                                            const DkParams& p, DkMisc* m) {
    unsigned long long v[kDkShadows];
    unsigned pending = (1u << kDkShadows) - 1u;
    for (unsigned long long it = 0;; ++it) {
#pragma unroll
        for (int sh = 0; sh < kDkShadows; ++sh)
            if ((pending >> sh) & 1u) v[sh] = ld_relaxed_gpu_u64(w + (size_t)sh * stride);
#pragma unroll
        for (int sh = 0; sh < kDkShadows; ++sh)
            if ((unsigned)(v[sh] >> 57) >= dk_shadow_ctas(sh)) pending &= ~(1u << sh);
        if (pending == 0u) break;
        if ((it & 63ull) == 63ull && (ld_relaxed_gpu(p.bar + 1) != 0u || *(volatile int*)&m->abort_flag)) return false;
        if (it > kDkSpinLimit) {
            set_status(p.status, MOE_DEV_TIMEOUT);
            atomicExch(p.bar + 1, 1u);
            return false;
        }
    }
    sum = 0;
#pragma unroll
    for (int sh = 0; sh < kDkShadows; ++sh) sum += fix_sum(v[sh], dk_shadow_ctas(sh));
    return true;
}

// Top-k of one token (one warp; lane l holds experts l, l+32, ...; E <= 256).
// Each logit becomes an order-preserving unsigned key; every round takes the
// largest key over the warp with one warp-wide max reduction and, among the
// lanes holding it, the lowest expert id with one min reduction -- "logit
// descending, ties to the lower id" -- and the owning lane marks it taken.
// The routing weights follow: the fp32 softmax over all E logits followed by
// renormalisation over the selection equals the softmax over the selected
// logits alone (the full denominator cancels), w_j = e^(l_j - l_0) / sum.
// (order_key / key_value: moe_common.cuh)

// Top-k of token t by one warp from values in registers: lane L holds the
// logit of expert L + 32 s in v[s] (s < 8; entries for e >= E are ignored)
// as order-preserving keys; k rounds of a max reduction (and a min reduction
// over the ids holding it: ties to the lower id), then the weights.
__device__ __forceinline__ void dk_topk_vals(const float (&v)[8], int E, int k, int t, DkMisc* m, int32_t* status) {
    const int lane = threadIdx.x & 31;
    unsigned key[8];
    bool bad = false;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int e = lane + 32 * s;
        if (e < E && !isfinite(v[s])) bad = true;
        key[s] = e < E ? order_key(v[s]) : 0u;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_DEV_NONFINITE);
    unsigned taken = 0;
    int my_id = 0;
    float my_l = 0.f, l0 = 0.f;
    for (int j = 0; j < k; ++j) {
        unsigned kb = 0u;
        int ib = 0x7fffffff;
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if (!((taken >> s) & 1u) && key[s] > kb) {
                kb = key[s];
                ib = lane + 32 * s;
            }
        const unsigned km = __reduce_max_sync(0xffffffffu, kb);
        const int win = (int)__reduce_min_sync(0xffffffffu, kb == km ? (unsigned)ib : 0x7fffffffu);
        if ((win & 31) == lane && win < E) taken |= 1u << (win >> 5);
        const float lv = key_value(km);
        if (j == 0) l0 = lv;
        if (lane == j) {
            my_id = win < E ? win : 0;
            my_l = lv;
        }
    }
    const float ex = lane < k ? expf(my_l - l0) : 0.f;
    float den = ex;
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    if (lane < k) {
        m->ids[t * k + lane] = my_id;
        m->selv[t * k + lane] = my_l;
        m->w[t * k + lane] = ex / den;
    }
    __syncwarp();
}

// The same from token t's logits in shared memory (lg[e], e < E).
// Not inlined: the kernel runs it once on stale values before the real pass
// of each layer, and only one shared copy of the code gets warmed that way.
__device__ __noinline__ void dk_topk_smem(const float* lg, int E, int k, int t, DkMisc* m, int32_t* status) {
    const int lane = threadIdx.x & 31;
    float v[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int e = lane + 32 * s;
        v[s] = e < E ? lg[e] : 0.f;
    }
    dk_topk_vals(v, E, k, t, m, status);
}

// Router partial sums of this CTA's hidden rows [h0, h0+nrows) for every
__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

struct Tagged4 {
    unsigned long long a, b, c, d;
};

__device__ __forceinline__ void dk_ld_tagged4(const unsigned long long* w, Tagged4& t) {
    ld_relaxed_gpu_u64x2(w, t.a, t.b);
    ld_relaxed_gpu_u64x2(w + 2, t.c, t.d);
}

__device__ __forceinline__ bool dk_tags_are(const Tagged4& t, unsigned tag) {
    return (unsigned)(t.a >> 32) == tag && (unsigned)(t.b >> 32) == tag && (unsigned)(t.c >> 32) == tag &&
           (unsigned)(t.d >> 32) == tag;
}

// Four consecutive tagged elements of x (two 16-byte loads, already issued
// into t), waited for until each carries tag `tag` (bounded like dk_poll_sum);
// false when aborting.
__device__ __forceinline__ bool dk_load_tagged4(const unsigned long long* w, unsigned tag, Tagged4& t, float4& out,
                                                const DkParams& p, DkMisc* m) {
    for (unsigned long long it = 0;; ++it) {
        if (dk_tags_are(t, tag)) break;
        if ((it & 63ull) == 63ull && (ld_relaxed_gpu(p.bar + 1) != 0u || *(volatile int*)&m->abort_flag)) return false;
        if (it > kDkSpinLimit) {
            set_status(p.status, MOE_DEV_TIMEOUT);
            atomicExch(p.bar + 1, 1u);
            return false;
        }
        dk_ld_tagged4(w, t);
    }
    out = make_float4(__uint_as_float((unsigned)t.a), __uint_as_float((unsigned)t.b), __uint_as_float((unsigned)t.c),
                      __uint_as_float((unsigned)t.d));
    return true;
}

// (token, expert): one thread per pair, rows in 8-wide vectors from shared
// memory, the result added to shadow copy (CTA mod kDkShadows) of the
// fixed-point accumulator as a counted contribution.  Every CTA adds to
// every word of its copy (a CTA without rows adds zero), so a word is
// complete -- and its reader needs no barrier -- once its count reaches the
// number of CTAs of that copy.  The words carry only themselves: the rows of
// x travel with their own tags (DkParams::xt), and the buffers a CTA reads
// after the mid barrier (h, the predicted logits) alternate by layer, so no
// fence orders anything before the reductions.
//
// Pre-norm stacks (g = the layer's norm weights): the logits of RMSNorm(x)
// are rn * sum_h W[e,h] g[h] x[h] with rn = 1/sqrt(mean(x^2) + eps), one
// scalar per token, so the partial sums take g in and leave rn out, and the
// partial sums of x^2 go into a second fixed-point accumulator (nacc[t]);
// rn is applied where the logits are read.  The router stays fused into the
// residual add that forms x (the norm + residual fusion).
__device__ __forceinline__ void dk_router_partials(const uint16_t* wrs, int maxrows, const float* xs, int H,
                                                   int h0, int nrows, int B, int E,
                                                   unsigned long long* acc, int t0, int nth,
                                                   int32_t* status, const float* g = nullptr,
                                                   unsigned long long* nacc = nullptr) {
    unsigned long long* sh = acc + (size_t)(blockIdx.x % kDkShadows) * B * E;
    for (int v = t0; v < B * E; v += nth) {
        const int t = v / E, e = v - t * E;
        const uint16_t* wrow = wrs + e * maxrows;
        const float* xr = xs + (size_t)t * H + h0;
        float2 a = make_float2(0.f, 0.f);
        for (int r = 0; r < nrows; r += 8) {
            const uint4 wv = *reinterpret_cast<const uint4*>(wrow + r);
            float4 xa = *reinterpret_cast<const float4*>(xr + r);
            float4 xb = *reinterpret_cast<const float4*>(xr + r + 4);
            if (g) {
                const float4 ga = *reinterpret_cast<const float4*>(g + h0 + r);
                const float4 gb = *reinterpret_cast<const float4*>(g + h0 + r + 4);
                xa = make_float4(xa.x * ga.x, xa.y * ga.y, xa.z * ga.z, xa.w * ga.w);
                xb = make_float4(xb.x * gb.x, xb.y * gb.y, xb.z * gb.z, xb.w * gb.w);
            }
            a = ffma2(bf16x2_to_f2(wv.x), make_float2(xa.x, xa.y), a);
            a = ffma2(bf16x2_to_f2(wv.y), make_float2(xa.z, xa.w), a);
            a = ffma2(bf16x2_to_f2(wv.z), make_float2(xb.x, xb.y), a);
            a = ffma2(bf16x2_to_f2(wv.w), make_float2(xb.z, xb.w), a);
        }
        fix_add(sh + v, a.x + a.y, kFixScale, status);
    }
    if (nacc) {  // sum of squares of this CTA's rows, one thread per token
        for (int t = t0; t < B; t += nth) {
            const float* xr = xs + (size_t)t * H + h0;
            float ss = 0.f;
            for (int r = 0; r < nrows; ++r) ss = fmaf(xr[r], xr[r], ss);
            fix_add(nacc + (size_t)(blockIdx.x % kDkShadows) * B + t, ss, kFixScaleSq, status);
        }
    }
}

// Stable grouping of R <= 32 routes by expert in one warp: the position of
// route r is (#routes with a smaller expert) + (#earlier routes with the
// same expert) -- the counting sort's result, computed directly.  Not
// inlined, like dk_topk_smem.
__device__ __noinline__ void dk_group(DkMisc* m, int R, int E, bool no_dedup) {
    const int lane = threadIdx.x & 31;
    int e = 0x7fffffff;
    if (lane < R) {  // only non-finite logits can leave an entry out of range
        e = m->ids[lane];
        if (e < 0 || e >= E) {
            e = 0;
            m->ids[lane] = 0;
        }
    }
    __syncwarp();
    int pos = 0;
    for (int r = 0; r < R; ++r) {
        const int er = __shfl_sync(0xffffffffu, e, r);
        pos += (er < e) || (er == e && r < lane);
    }
    if (no_dedup) pos = lane;
    if (lane < R) {
        m->pos[lane] = pos;
        m->rat[pos] = lane;
    }
    __syncwarp();
    // segment starts in grouped order
    const int ep = lane < R ? m->ids[m->rat[lane]] : 0x7fffffff;
    const int eprev = __shfl_up_sync(0xffffffffu, ep, 1);
    const bool start = lane < R && (lane == 0 || no_dedup || ep != eprev);
    const unsigned ballot = __ballot_sync(0xffffffffu, start);
    if (start) {
        const int u = __popc(ballot & ((1u << lane) - 1u));
        m->seg_e[u] = ep;
        m->seg_p[u] = lane;
    }
    if (lane == 0) {
        const int U = __popc(ballot);
        m->U = U;
        m->seg_p[U] = R;
    }
    __syncwarp();
}

// The CTA's grouping in the layout of moe_group_by_expert (one warp):
// offsets[e] = routes whose expert id is below e, route_idx = the routes in
// grouped order, unique = the segments' experts, num_unique = U.
__device__ __forceinline__ void dk_store_grouping(const DkParams& p, const DkMisc* m, int R, int E) {
    const int lane = threadIdx.x & 31;
    const int U = m->U;
    for (int e = lane; e <= E; e += 32) {
        int off = 0;
        for (int u = 0; u < U; ++u)
            if (m->seg_e[u] < e) off += m->seg_p[u + 1] - m->seg_p[u];
        p.g_offsets[e] = off;
    }
    if (lane < R) p.g_route_idx[lane] = m->rat[lane];
    if (lane < U) p.g_unique[lane] = m->seg_e[lane];
    if (lane == 0) *p.g_num_unique = U;
}

// Sum of N values held by every lane over the 32 lanes of a warp; the N
// butterflies are interleaved so the latency is that of one.
template <int N>
__device__ __forceinline__ void warp_sum_n(float (&v)[N]) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], off);
}

// x rows are also kept lane-blocked in shared memory (xq, token stride
// lb_stride(H); see lb_index): conflict-free 16-byte loads for the warps
// that walk column groups lane by lane.
__host__ __device__ __forceinline__ int dk_hq(int H) { return lb_stride(H); }
__device__ __forceinline__ int dk_xq_index(int c) { return lb_index(c); }

// Four x values at flat index f = t*H + c (c a multiple of 4) into both
// copies: xs keeps x (the residual), xq the layer input -- x itself, or for
// a pre-norm stack RMSNorm(x) = (x * rn[t]) * g (g != nullptr: the norm
// weights in shared memory).
__device__ __forceinline__ void dk_store_x(float* xs, float* xq, int H, int f, float4 v, const float* g = nullptr,
                                           const DkMisc* m = nullptr) {
    *reinterpret_cast<float4*>(xs + f) = v;
    const int t = f / H, c = f - t * H;
    if (g) {
        const float r = m->rn[t];
        const float4 gv = *reinterpret_cast<const float4*>(g + c);
        v = make_float4((v.x * r) * gv.x, (v.y * r) * gv.y, (v.z * r) * gv.z, (v.w * r) * gv.w);
    }
    *reinterpret_cast<float4*>(xq + (size_t)t * dk_hq(H) + dk_xq_index(c)) = v;
}

// One gate/up row pair in shared memory (gate row at grow, up row at urow,
// H bf16 each) against NQ tokens' x rows (lane-blocked copy xq).  Four
// 16-byte vectors per lane are loaded before they are used.  Result: g[q],
// u[q] summed over the warp.
template <int NQ>
__device__ __forceinline__ void dk_gate_pair(const unsigned char* grow, const unsigned char* urow, const float* xq,
                                             const int (&tok)[4], int H, float (&gu)[2 * NQ]) {
    const int lane = threadIdx.x & 31;
    float2 ag[NQ], au[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) ag[q] = au[q] = make_float2(0.f, 0.f);
    const int nv = H >> 3, hq = dk_hq(H);
    auto step = [&](const uint4& gw, const uint4& uw, int v) {
        const float2 g0 = bf16x2_to_f2(gw.x), g1 = bf16x2_to_f2(gw.y);
        const float2 g2 = bf16x2_to_f2(gw.z), g3 = bf16x2_to_f2(gw.w);
        const float2 u0 = bf16x2_to_f2(uw.x), u1 = bf16x2_to_f2(uw.y);
        const float2 u2 = bf16x2_to_f2(uw.z), u3 = bf16x2_to_f2(uw.w);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const float* xp = xq + (size_t)tok[q] * hq + ((v >> 5) << 8) + ((v & 31) << 2);
            const float4 xa = *reinterpret_cast<const float4*>(xp);
            const float4 xb = *reinterpret_cast<const float4*>(xp + 128);
            ag[q] = ffma2(g0, make_float2(xa.x, xa.y), ag[q]);
            au[q] = ffma2(u0, make_float2(xa.x, xa.y), au[q]);
            ag[q] = ffma2(g1, make_float2(xa.z, xa.w), ag[q]);
            au[q] = ffma2(u1, make_float2(xa.z, xa.w), au[q]);
            ag[q] = ffma2(g2, make_float2(xb.x, xb.y), ag[q]);
            au[q] = ffma2(u2, make_float2(xb.x, xb.y), au[q]);
            ag[q] = ffma2(g3, make_float2(xb.z, xb.w), ag[q]);
            au[q] = ffma2(u3, make_float2(xb.z, xb.w), au[q]);
        }
    };
    int v = lane;
    for (; v + 96 < nv; v += 128) {
        uint4 gw[4], uw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            gw[j] = *reinterpret_cast<const uint4*>(grow + 16 * (v + 32 * j));
            uw[j] = *reinterpret_cast<const uint4*>(urow + 16 * (v + 32 * j));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) step(gw[j], uw[j], v + 32 * j);
    }
    for (; v < nv; v += 32)
        step(*reinterpret_cast<const uint4*>(grow + 16 * v), *reinterpret_cast<const uint4*>(urow + 16 * v), v);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        gu[2 * q] = ag[q].x + ag[q].y;
        gu[2 * q + 1] = au[q].x + au[q].y;
    }
    warp_sum_n<2 * NQ>(gu);
}

// Down rows [0, nrc) of a ring stage (each I bf16) against NQ routes' h rows
// in shared memory (hrow = h of the first route, consecutive routes I apart),
// four rows at a time with independent accumulators; results to
// os[q * ld + orow0 + r].
template <int NQ>
__device__ __forceinline__ void dk_down_rows(const unsigned char* st, int nrc, int I, const float* hrow,
                                             float* os, int ld, int orow0) {
    const int lane = threadIdx.x & 31;
    const int nv = I >> 3;
    for (int rb = 0; rb < nrc; rb += 4) {
        const int n4 = min(4, nrc - rb);
        float2 acc[4][NQ];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q) acc[j][q] = make_float2(0.f, 0.f);
        for (int v = lane; v < nv; v += 32) {
            uint4 wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                wv[j] = j < n4 ? *reinterpret_cast<const uint4*>(st + (size_t)(rb + j) * 2 * I + 16 * v)
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4* hp = reinterpret_cast<const float4*>(hrow + (size_t)q * I + 8 * v);
                const float4 ha = hp[0], hb = hp[1];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[j][q] = ffma2(bf16x2_to_f2(wv[j].x), make_float2(ha.x, ha.y), acc[j][q]);
                    acc[j][q] = ffma2(bf16x2_to_f2(wv[j].y), make_float2(ha.z, ha.w), acc[j][q]);
                    acc[j][q] = ffma2(bf16x2_to_f2(wv[j].z), make_float2(hb.x, hb.y), acc[j][q]);
                    acc[j][q] = ffma2(bf16x2_to_f2(wv[j].w), make_float2(hb.z, hb.w), acc[j][q]);
                }
            }
        }
        float red[4 * NQ];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q) red[j * NQ + q] = acc[j][q].x + acc[j][q].y;
        warp_sum_n<4 * NQ>(red);
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < n4)
#pragma unroll
                    for (int q = 0; q < NQ; ++q) os[(size_t)q * ld + orow0 + rb + j] = red[j * NQ + q];
        }
    }
}

// ---------------------------------------------------- block-scaled FP8
// (f8x2_to_f2: moe_common.cuh)

// The FP8 form of dk_gate_pair: rows of H E4M3 codes (gate row at grow, up
// row at urow) with their block scales along the row (gsr, usr: the scale
// rows of the 128-row blocks the two rows lie in).  Lane L takes the 8-code
// groups v = L + 32j (one 8-byte load each, a warp reads 256 contiguous
// bytes); a group lies in one 128-column block, so its 8 products are summed
// first and scaled once: sum_v s_v * sum_8 decode(q) x.
template <int NQ>
__device__ __forceinline__ void dk_gate_pair_f8(const unsigned char* grow, const unsigned char* urow,
                                                const float* gsr, const float* usr, const float* xq,
                                                const int (&tok)[4], int H, float (&gu)[2 * NQ]) {
    const int lane = threadIdx.x & 31;
    float ag[NQ], au[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) ag[q] = au[q] = 0.f;
    const int nv = H >> 3, hq = dk_hq(H);
    for (int v = lane; v < nv; v += 32) {
        const uint2 gw = *reinterpret_cast<const uint2*>(grow + 8 * v);
        const uint2 uw = *reinterpret_cast<const uint2*>(urow + 8 * v);
        const float sg = __ldg(gsr + (v >> 4)), su = __ldg(usr + (v >> 4));
        const float2 g0 = f8x2_to_f2(gw.x), g1 = f8x2_to_f2(gw.x >> 16);
        const float2 g2 = f8x2_to_f2(gw.y), g3 = f8x2_to_f2(gw.y >> 16);
        const float2 u0 = f8x2_to_f2(uw.x), u1 = f8x2_to_f2(uw.x >> 16);
        const float2 u2 = f8x2_to_f2(uw.y), u3 = f8x2_to_f2(uw.y >> 16);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const float* xp = xq + (size_t)tok[q] * hq + ((v >> 5) << 8) + ((v & 31) << 2);
            const float4 xa = *reinterpret_cast<const float4*>(xp);
            const float4 xb = *reinterpret_cast<const float4*>(xp + 128);
            float2 pg = ffma2(g0, make_float2(xa.x, xa.y), make_float2(0.f, 0.f));
            float2 pu = ffma2(u0, make_float2(xa.x, xa.y), make_float2(0.f, 0.f));
            pg = ffma2(g1, make_float2(xa.z, xa.w), pg);
            pu = ffma2(u1, make_float2(xa.z, xa.w), pu);
            pg = ffma2(g2, make_float2(xb.x, xb.y), pg);
            pu = ffma2(u2, make_float2(xb.x, xb.y), pu);
            pg = ffma2(g3, make_float2(xb.z, xb.w), pg);
            pu = ffma2(u3, make_float2(xb.z, xb.w), pu);
            ag[q] = fmaf(sg, pg.x + pg.y, ag[q]);
            au[q] = fmaf(su, pu.x + pu.y, au[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        gu[2 * q] = ag[q];
        gu[2 * q + 1] = au[q];
    }
    warp_sum_n<2 * NQ>(gu);
}

// The FP8 form of dk_down_rows: rows of I codes, four at a time; row r's
// scales are row (row_abs0 + r) / 128 of the expert's block scales dsr.
template <int NQ>
__device__ __forceinline__ void dk_down_rows_f8(const unsigned char* st, int nrc, int I, const float* dsr,
                                                int dsr_ld, int row_abs0, const float* hrow, float* os, int ld,
                                                int orow0) {
    const int lane = threadIdx.x & 31;
    const int nv = I >> 3;
    for (int rb = 0; rb < nrc; rb += 4) {
        const int n4 = min(4, nrc - rb);
        const float* sr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) sr[j] = dsr + (size_t)((row_abs0 + rb + min(j, n4 - 1)) >> 7) * dsr_ld;
        float acc[4][NQ];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q) acc[j][q] = 0.f;
        for (int v = lane; v < nv; v += 32) {
            float s[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) s[j] = __ldg(sr[j] + (v >> 4));
            uint2 wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                wv[j] = j < n4 ? *reinterpret_cast<const uint2*>(st + (size_t)(rb + j) * I + 8 * v) : make_uint2(0u, 0u);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4* hp = reinterpret_cast<const float4*>(hrow + (size_t)q * I + 8 * v);
                const float4 ha = hp[0], hb = hp[1];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float2 a = ffma2(f8x2_to_f2(wv[j].x), make_float2(ha.x, ha.y), make_float2(0.f, 0.f));
                    a = ffma2(f8x2_to_f2(wv[j].x >> 16), make_float2(ha.z, ha.w), a);
                    a = ffma2(f8x2_to_f2(wv[j].y), make_float2(hb.x, hb.y), a);
                    a = ffma2(f8x2_to_f2(wv[j].y >> 16), make_float2(hb.z, hb.w), a);
                    acc[j][q] = fmaf(s[j], a.x + a.y, acc[j][q]);
                }
            }
        }
        float red[4 * NQ];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q) red[j * NQ + q] = acc[j][q];
        warp_sum_n<4 * NQ>(red);
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < n4)
#pragma unroll
                    for (int q = 0; q < NQ; ++q) os[(size_t)q * ld + orow0 + rb + j] = red[j * NQ + q];
        }
    }
}

// ---------------------------------------------------------------- NVFP4
// (f4x2_to_f2, f8_to_f: moe_common.cuh)

// The NVFP4 form of dk_gate_pair: rows of H E2M1 codes two to a byte (gate
// row at grow, up row at urow), the rows' E4M3 block scales (gbs, ubs: one
// byte per 16 elements) and the matrix scale gsc.  Lane L takes the 8-code
// groups v = L + 32j (one 4-byte load each, a warp reads 128 contiguous
// bytes); a group lies in one 16-element block, so its 8 products are summed
// first and scaled once.
template <int NQ>
__device__ __forceinline__ void dk_gate_pair_f4(const unsigned char* grow, const unsigned char* urow,
                                                const unsigned char* gbs, const unsigned char* ubs, float gsc,
                                                const float* xq, const int (&tok)[4], int H, float (&gu)[2 * NQ]) {
    const int lane = threadIdx.x & 31;
    float ag[NQ], au[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) ag[q] = au[q] = 0.f;
    const int nv = H >> 3, hq = dk_hq(H);
    for (int v = lane; v < nv; v += 32) {
        const unsigned gw = *reinterpret_cast<const unsigned*>(grow + 4 * v);
        const unsigned uw = *reinterpret_cast<const unsigned*>(urow + 4 * v);
        const float sg = f8_to_f(__ldg(gbs + (v >> 1))) * gsc, su = f8_to_f(__ldg(ubs + (v >> 1))) * gsc;
        const float2 g0 = f4x2_to_f2(gw), g1 = f4x2_to_f2(gw >> 8), g2 = f4x2_to_f2(gw >> 16), g3 = f4x2_to_f2(gw >> 24);
        const float2 u0 = f4x2_to_f2(uw), u1 = f4x2_to_f2(uw >> 8), u2 = f4x2_to_f2(uw >> 16), u3 = f4x2_to_f2(uw >> 24);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const float* xp = xq + (size_t)tok[q] * hq + ((v >> 5) << 8) + ((v & 31) << 2);
            const float4 xa = *reinterpret_cast<const float4*>(xp);
            const float4 xb = *reinterpret_cast<const float4*>(xp + 128);
            float2 pg = ffma2(g0, make_float2(xa.x, xa.y), make_float2(0.f, 0.f));
            float2 pu = ffma2(u0, make_float2(xa.x, xa.y), make_float2(0.f, 0.f));
            pg = ffma2(g1, make_float2(xa.z, xa.w), pg);
            pu = ffma2(u1, make_float2(xa.z, xa.w), pu);
            pg = ffma2(g2, make_float2(xb.x, xb.y), pg);
            pu = ffma2(u2, make_float2(xb.x, xb.y), pu);
            pg = ffma2(g3, make_float2(xb.z, xb.w), pg);
            pu = ffma2(u3, make_float2(xb.z, xb.w), pu);
            ag[q] = fmaf(sg, pg.x + pg.y, ag[q]);
            au[q] = fmaf(su, pu.x + pu.y, au[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        gu[2 * q] = ag[q];
        gu[2 * q + 1] = au[q];
    }
    warp_sum_n<2 * NQ>(gu);
}

// The NVFP4 form of dk_down_rows: rows of I codes two to a byte, four rows at
// a time; row r's block scales at dbs + r * I/16 (dbs: the scales of the
// first row), matrix scale dgs.
template <int NQ>
__device__ __forceinline__ void dk_down_rows_f4(const unsigned char* st, int nrc, int I, const unsigned char* dbs,
                                                float dgs, const float* hrow, float* os, int ld, int orow0) {
    const int lane = threadIdx.x & 31;
    const int nv = I >> 3, rb_bytes = I >> 1, sb = I >> 4;
    for (int rb = 0; rb < nrc; rb += 4) {
        const int n4 = min(4, nrc - rb);
        float acc[4][NQ];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q) acc[j][q] = 0.f;
        for (int v = lane; v < nv; v += 32) {
            float s[4];
            unsigned wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = rb + min(j, n4 - 1);
                s[j] = f8_to_f(__ldg(dbs + (size_t)r * sb + (v >> 1))) * dgs;
                wv[j] = j < n4 ? *reinterpret_cast<const unsigned*>(st + (size_t)(rb + j) * rb_bytes + 4 * v) : 0u;
            }
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4* hp = reinterpret_cast<const float4*>(hrow + (size_t)q * I + 8 * v);
                const float4 ha = hp[0], hb = hp[1];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float2 a = ffma2(f4x2_to_f2(wv[j]), make_float2(ha.x, ha.y), make_float2(0.f, 0.f));
                    a = ffma2(f4x2_to_f2(wv[j] >> 8), make_float2(ha.z, ha.w), a);
                    a = ffma2(f4x2_to_f2(wv[j] >> 16), make_float2(hb.x, hb.y), a);
                    a = ffma2(f4x2_to_f2(wv[j] >> 24), make_float2(hb.z, hb.w), a);
                    acc[j][q] = fmaf(s[j], a.x + a.y, acc[j][q]);
                }
            }
        }
        float red[4 * NQ];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q) red[j * NQ + q] = acc[j][q];
        warp_sum_n<4 * NQ>(red);
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < n4)
#pragma unroll
                    for (int q = 0; q < NQ; ++q) os[(size_t)q * ld + orow0 + rb + j] = red[j * NQ + q];
        }
    }
}

// Gate/up pair q of the layer (segment u, row i) from shared-memory rows:
// h[p, i] = SiLU(g) * u for every route p of the segment.  kF8: the rows
// hold E4M3 codes and gsr/usr are the scale rows of gate row i and up row
// I + i.
template <int kNQ, bool kF8 = false, bool kF4 = false>
__device__ __forceinline__ void dk_pair_compute(const DkMisc* m, const unsigned char* grow, const unsigned char* urow,
                                                const float* xq, int H, int I, int k, int u, int i, float* h,
                                                const float* gsr = nullptr, const float* usr = nullptr,
                                                const unsigned char* gbs = nullptr, const unsigned char* ubs = nullptr,
                                                float gsc = 1.f) {
    const int lane = threadIdx.x & 31;
    const int p0 = m->seg_p[u], p1 = m->seg_p[u + 1];
    int tok[kDkMaxB];
#pragma unroll
    for (int qq = 0; qq < kDkMaxB; ++qq) tok[qq] = p0 + qq < p1 ? m->rat[p0 + qq] / k : 0;
    const int nq = kNQ == 1 ? 1 : p1 - p0;
    float gu[2 * kDkMaxB];
    if constexpr (kF4) {
        switch (kNQ == 1 ? 1 : nq) {
            case 1: { float r[2]; dk_gate_pair_f4<1>(grow, urow, gbs, ubs, gsc, xq, tok, H, r); gu[0] = r[0]; gu[1] = r[1]; } break;
            case 2: { float r[4]; dk_gate_pair_f4<2>(grow, urow, gbs, ubs, gsc, xq, tok, H, r);
#pragma unroll
                      for (int j = 0; j < 4; ++j) gu[j] = r[j]; } break;
            case 3: { float r[6]; dk_gate_pair_f4<3>(grow, urow, gbs, ubs, gsc, xq, tok, H, r);
#pragma unroll
                      for (int j = 0; j < 6; ++j) gu[j] = r[j]; } break;
            default: dk_gate_pair_f4<4>(grow, urow, gbs, ubs, gsc, xq, tok, H, gu); break;
        }
    } else if constexpr (kF8) {
        switch (kNQ == 1 ? 1 : nq) {
            case 1: { float r[2]; dk_gate_pair_f8<1>(grow, urow, gsr, usr, xq, tok, H, r); gu[0] = r[0]; gu[1] = r[1]; } break;
            case 2: { float r[4]; dk_gate_pair_f8<2>(grow, urow, gsr, usr, xq, tok, H, r);
#pragma unroll
                      for (int j = 0; j < 4; ++j) gu[j] = r[j]; } break;
            case 3: { float r[6]; dk_gate_pair_f8<3>(grow, urow, gsr, usr, xq, tok, H, r);
#pragma unroll
                      for (int j = 0; j < 6; ++j) gu[j] = r[j]; } break;
            default: dk_gate_pair_f8<4>(grow, urow, gsr, usr, xq, tok, H, gu); break;
        }
    } else {
        switch (kNQ == 1 ? 1 : nq) {
            case 1: { float r[2]; dk_gate_pair<1>(grow, urow, xq, tok, H, r); gu[0] = r[0]; gu[1] = r[1]; } break;
            case 2: { float r[4]; dk_gate_pair<2>(grow, urow, xq, tok, H, r);
#pragma unroll
                      for (int j = 0; j < 4; ++j) gu[j] = r[j]; } break;
            case 3: { float r[6]; dk_gate_pair<3>(grow, urow, xq, tok, H, r);
#pragma unroll
                      for (int j = 0; j < 6; ++j) gu[j] = r[j]; } break;
            default: dk_gate_pair<4>(grow, urow, xq, tok, H, gu); break;
        }
    }
    if (lane < nq) {
        float g = gu[0], uu = gu[1];
#pragma unroll
        for (int qq = 1; qq < kDkMaxB; ++qq)
            if (lane == qq) {
                g = gu[2 * qq];
                uu = gu[2 * qq + 1];
            }
        h[(size_t)(p0 + lane) * I + i] = silu_mul(g, uu);
    }
}

// Down rows [r0, r1) of segment u from shared memory (row r at base + (r -
// r0) * row bytes) into os (j-th route of the segment at row p0 + j).  kF8:
// E4M3 codes with the expert's block scales dsc ([ceil(H/128)][dsc_ld]).
template <int kNQ, bool kF8 = false, bool kF4 = false>
__device__ __forceinline__ void dk_down_compute(const DkMisc* m, const unsigned char* base, int r0, int r1, int I,
                                                const float* hs, float* os, int maxrows, int h0, int u,
                                                const float* dsc = nullptr, int dsc_ld = 0,
                                                const unsigned char* dbs = nullptr, float dgs = 1.f) {
    const int p0 = m->seg_p[u], p1 = m->seg_p[u + 1];
    const float* hrow = hs + (size_t)p0 * I;
    float* orow = os + (size_t)p0 * maxrows;
    if constexpr (kF4) {  // dbs: the expert's block scales; row r0's row of them first
        const unsigned char* sr = dbs + (size_t)r0 * (I >> 4);
        switch (kNQ == 1 ? 1 : p1 - p0) {
            case 1: dk_down_rows_f4<1>(base, r1 - r0, I, sr, dgs, hrow, orow, maxrows, r0 - h0); break;
            case 2: dk_down_rows_f4<2>(base, r1 - r0, I, sr, dgs, hrow, orow, maxrows, r0 - h0); break;
            case 3: dk_down_rows_f4<3>(base, r1 - r0, I, sr, dgs, hrow, orow, maxrows, r0 - h0); break;
            default: dk_down_rows_f4<4>(base, r1 - r0, I, sr, dgs, hrow, orow, maxrows, r0 - h0); break;
        }
        return;
    }
    if constexpr (kF8) {
        switch (kNQ == 1 ? 1 : p1 - p0) {
            case 1: dk_down_rows_f8<1>(base, r1 - r0, I, dsc, dsc_ld, r0, hrow, orow, maxrows, r0 - h0); break;
            case 2: dk_down_rows_f8<2>(base, r1 - r0, I, dsc, dsc_ld, r0, hrow, orow, maxrows, r0 - h0); break;
            case 3: dk_down_rows_f8<3>(base, r1 - r0, I, dsc, dsc_ld, r0, hrow, orow, maxrows, r0 - h0); break;
            default: dk_down_rows_f8<4>(base, r1 - r0, I, dsc, dsc_ld, r0, hrow, orow, maxrows, r0 - h0); break;
        }
        return;
    }
    switch (kNQ == 1 ? 1 : p1 - p0) {
        case 1: dk_down_rows<1>(base, r1 - r0, I, hrow, orow, maxrows, r0 - h0); break;
        case 2: dk_down_rows<2>(base, r1 - r0, I, hrow, orow, maxrows, r0 - h0); break;
        case 3: dk_down_rows<3>(base, r1 - r0, I, hrow, orow, maxrows, r0 - h0); break;
        default: dk_down_rows<4>(base, r1 - r0, I, hrow, orow, maxrows, r0 - h0); break;
    }
}

// ------------------------------------------------- next-layer L2 prefetch
// While layer l runs, the next layer's router can already be applied to
// layer l's input x_l (its true input is x_l + y_l).  The top experts of
// those predicted logits usually contain the next layer's choice, so their
// gate/up weights are prefetched into L2 during the rest of layer l and the
// next layer's bulk copies mostly hit L2.  Only a prefetch: the real routing is
// computed exactly as before and any miss is served from HBM.
//
// Predicted logits of this CTA's experts (e = blockIdx.x, + G, ...) for
// token 0 (one warp).
__device__ __forceinline__ void dk_predict_logits(const LayerWeights& wn, const float* xq, int H, int E, float* alog) {
    // (alog: this layer's half of the [2][E] buffer -- layers alternate, so a
    // CTA still reading layer l's predictions is never overwritten by layer l+1)
    const int lane = threadIdx.x & 31;
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
        const uint16_t* wrow = wn.w_router + (size_t)e * H;
        float2 a = make_float2(0.f, 0.f);
        for (int v = lane; v < (H >> 3); v += 32) {
            const uint4 wv = ld_weight_v4(wrow + 8 * v);
            const float* xp = xq + ((v >> 5) << 8) + ((v & 31) << 2);
            const float4 xa = *reinterpret_cast<const float4*>(xp);
            const float4 xb = *reinterpret_cast<const float4*>(xp + 128);
            a = ffma2(bf16x2_to_f2(wv.x), make_float2(xa.x, xa.y), a);
            a = ffma2(bf16x2_to_f2(wv.y), make_float2(xa.z, xa.w), a);
            a = ffma2(bf16x2_to_f2(wv.z), make_float2(xb.x, xb.y), a);
            a = ffma2(bf16x2_to_f2(wv.w), make_float2(xb.z, xb.w), a);
        }
        const float v = warp_sum(a.x + a.y);
        if (lane == 0) alog[e] = v + (wn.bias ? wn.bias[e] : 0.f);
    }
}

// One warp: the top-kp experts of the predicted logits (all CTAs' values,
// read after the mid-layer barrier); lane j < kp returns the j-th best
// (-1 elsewhere).
__device__ __forceinline__ int dk_predict_top(const float* alog, int E, int kp) {
    const int lane = threadIdx.x & 31;
    unsigned key[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int e = lane + 32 * s;
        key[s] = e < E ? order_key(__ldcg(alog + e)) : 0u;
    }
    unsigned taken = 0;
    int my_e = -1;
    for (int j = 0; j < kp; ++j) {
        unsigned kb = 0u;
        int ib = 0x7fffffff;
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if (!((taken >> s) & 1u) && key[s] > kb) {
                kb = key[s];
                ib = lane + 32 * s;
            }
        const unsigned km = __reduce_max_sync(0xffffffffu, kb);
        const int win = (int)__reduce_min_sync(0xffffffffu, kb == km ? (unsigned)ib : 0x7fffffffu);
        if ((win & 31) == lane && win < E) taken |= 1u << (win >> 5);
        if (lane == j) my_e = win < E ? win : -1;
    }
    return my_e;
}

// This CTA's 1/G share of each predicted expert's gate_up block prefetched
// into L2: lane j < kp takes expert j (my_e) and issues one bulk prefetch of
// its piece (pieces of equal 16-byte-aligned size, the last CTA taking the
// remainder).  Only gate_up: its rows are the ones the next layer waits for
// right after routing; the down rows are fetched during the gate/up pass,
// off the critical path, and prefetching them too only adds traffic that
// competes with this layer's own L2 round trips (2 % slower, measured).
__device__ __forceinline__ void dk_prefetch_l2(const LayerWeights& wn, int my_e, int H, int I, int kp, int w2 = 4) {
    const int lane = threadIdx.x & 31;
    if (lane < kp && my_e >= 0) {
        // (w2: bytes of two weights -- 4 bf16, 2 E4M3, 1 E2M1)
        const unsigned G = gridDim.x, c = blockIdx.x;
        const unsigned gsz = (unsigned)w2 * (unsigned)I * (unsigned)H;
        const unsigned gp = (gsz / G) & ~15u;
        const unsigned g0 = c * gp;
        const unsigned gn = c + 1 == G ? gsz - g0 : gp;
        const char* ge = reinterpret_cast<const char*>(wn.gate_up) + (size_t)my_e * gsz;
        if (gn > 0) bulk_prefetch_l2(ge + g0, gn);
    }
}

// Gate/up rows [ga, gb) of the pair list (segment u = q / I, row i = q - u*I,
// expert seg_e[u]) by bulk copies onto `bar` (armed by the caller with
// (gb - ga) * 4H bytes): per run of one segment, the gate rows to
// dg + (q - ga)*2H and the up rows to du + (q - ga)*2H.
__device__ __forceinline__ void dk_gate_runs(const uint16_t* gate_up, const int* seg_e, int ga, int gb, int H, int I,
                                             unsigned char* dg, unsigned char* du, uint64_t* bar, int w2 = 4) {
    const size_t row = ((size_t)w2 * H) >> 1;  // bytes of one row (w2: bytes of two weights)
    for (int q = ga; q < gb;) {
        const int u = q / I, i = q - u * I;
        const int qe = min(gb, (u + 1) * I);
        const uint32_t bytes = (uint32_t)((qe - q) * row);
        const unsigned char* G = reinterpret_cast<const unsigned char*>(gate_up) + (size_t)seg_e[u] * 2 * I * row;
        bulk_g2s(dg + (size_t)(q - ga) * row, G + (size_t)i * row, bytes, bar);
        bulk_g2s(du + (size_t)(q - ga) * row, G + (size_t)(I + i) * row, bytes, bar);
        q = qe;
    }
}

// ------------------------------------------------------------ the kernel
// kNQ = 1: a single token (every segment has one route), so only the
// one-token variants of the gate/up and down loops are compiled in; 4: any
// batch up to kDkMaxB.  kDirect: every layer takes direct mode (the host
// has checked that a CTA's largest possible share fits), so the ring code
// is compiled out.  Each variant that is not needed is left out of the
// instruction stream: the kernel runs every phase of a layer once per
// layer, so its speed depends on how much code it streams through the
// instruction caches.
template <bool kTrace, int kNQ, bool kDirect, bool kF8 = false, bool kF4 = false>
__global__ void __launch_bounds__(kDkThreads, 1) decode_kernel(const DkParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kDkMaxStages;
    uint64_t* dbar = empty + kDkMaxStages;  // direct mode: [0] unused, [1] down rows landed
    uint64_t* gch = dbar + 2;               // direct mode: [kDkGChunks] a chunk of gate/up pairs landed
    DkMisc* m = reinterpret_cast<DkMisc*>(smem + p.off_misc);
    float* xs = reinterpret_cast<float*>(smem + p.off_x);   // [B][H]
    float* xq = reinterpret_cast<float*>(smem + p.off_xq);  // [B][dk_hq(H)] lane-blocked copy of xs
    float* hs = reinterpret_cast<float*>(smem + p.off_h);   // [R][I]
    float* os = reinterpret_cast<float*>(smem + p.off_o);   // [R][maxrows]
    uint16_t* wrs = reinterpret_cast<uint16_t*>(smem + p.off_wr);  // [E][maxrows]
    unsigned char* ring = smem + p.off_ring;
    float* gq = reinterpret_cast<float*>(smem + p.off_gq);  // [2][H] (pre-norm stacks only)
    float* lg = reinterpret_cast<float*>(smem + p.off_misc + sizeof(DkMisc));  // [B][Ep] logits
    const int Ep = (p.E + 7) & ~7;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = kNQ == 1 ? 1 : p.B;  // a compile-time constant for one token
    const int H = p.H, I = p.I, E = p.E, k = p.k, R = B * k;
    // bytes of a gate/up row and of a down row (bf16, or one-byte E4M3 codes)
    // bytes of two weights: bf16, E4M3 or E2M1 (two codes a byte)
    constexpr int kW2 = kF4 ? 1 : (kF8 ? 2 : 4);
    const int rowg = (kW2 * H) >> 1, rowd = (kW2 * I) >> 1;
    // block-scale row lengths of gate_up [2I, H] and down [H, I] (FP8 only)
    const int sg_ld = (H + 127) >> 7, sd_ld = (I + 127) >> 7;
    const int sg_e = ((2 * I + 127) >> 7) * sg_ld, sd_e = ((H + 127) >> 7) * sd_ld;
    const bool no_dedup = (p.flags & MOE_F_NO_DEDUP) != 0;
    int h0, h1;
    dk_rows(blockIdx.x, gridDim.x, H, h0, h1);
    const int nrows = h1 - h0;
    DkWork wbase;
    wbase.h0 = h0;
    wbase.h1 = h1;
    wbase.nr = max(1, p.stage_bytes / rowd);
    if (wbase.nr >= 4) wbase.nr &= ~3;  // whole 4-row groups in the down compute
    wbase.nd_per_u = nrows > 0 ? (nrows + wbase.nr - 1) / wbase.nr : 0;
    wbase.ga = wbase.gb = wbase.ng = wbase.n = 0;

    if (tid == 0) {
        for (int s = 0; s < p.S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&dbar[0], 1);
        mbar_init(&dbar[1], 1);
        for (int c = 0; c < kDkGChunks; ++c) mbar_init(&gch[c], 1);
        m->abort_flag = 0;
        m->mid_epoch = 0;
        for (int q = 0; q < kDkMaxStages; ++q) m->last_pos[q] = -1;
        fence_mbar_init();
    }
    if (tid >= 32 && tid <= 32 + kDkMaxR) {  // gate/up pair range for U = 0 .. kDkMaxR segments
        const int U = tid - 32;
        dk_work_range(U, I, m->ga_tab[U], m->gb_tab[U]);
    }
    __syncthreads();

    unsigned epoch = 0;        // barrier count (leader thread only)
    // Ring cursor: chunks through the ring so far, as (stage, phase parity) of
    // the next chunk -- advanced incrementally, no division per chunk.
    int ring_pos = 0;
    int rs = 0;
    uint32_t rph = 0;
    // Direct mode (a CTA's whole layer share fits in the ring area): phases
    // armed so far on the two direct-mode barriers (same in every thread)
    int dg_count = 0, dd_count = 0;


    if (tid == kDkLeader) dk_trace<kTrace>(p, -1, 0);
    // ---- router of layer 0: partial dot products over this CTA's rows
    {
        const LayerWeights& w0 = p.layer[0];
        for (int v = tid; v < E * (nrows >> 3); v += blockDim.x) {
            const int e = v / (nrows >> 3), c8 = (v - e * (nrows >> 3)) << 3;
            cp_async16(wrs + e * p.maxrows + c8, w0.w_router + (size_t)e * H + h0 + c8);
        }
        if (p.has_norm)
            for (int v = tid; v < (H >> 2); v += blockDim.x) cp_async16(gq + 4 * v, w0.norm + 4 * v);
        cp_async_commit();
        for (int v = tid; v < B * nrows; v += blockDim.x) {
            const int t = v / nrows, r = v - t * nrows;
            const size_t off = (size_t)t * H + h0 + r;
            xs[t * H + h0 + r] = p.x_bf16 ? __uint_as_float((uint32_t)static_cast<const uint16_t*>(p.x_in)[off] << 16)
                                          : ld_act_f(static_cast<const float*>(p.x_in) + off);
        }
        cp_async_wait_all();
        __syncthreads();
        dk_router_partials(wrs, p.maxrows, xs, H, h0, nrows, B, E, dk_acc(p, 0), tid, blockDim.x, p.status,
                           p.has_norm ? gq : nullptr, p.has_norm ? dk_nacc(p, 0) : nullptr);
    }
    if (tid == kDkLeader) dk_trace<kTrace>(p, -1, 1);
    // (no barrier: each layer waits on its own logit words)

    for (int l = 0; l < p.L && !*(volatile int*)&m->abort_flag; ++l) {
        const LayerWeights& lw = p.layer[l];
        const bool has_next = l + 1 < p.L;
        const unsigned long long* acc_now = dk_acc(p, l);
        unsigned long long* acc_next = dk_acc(p, l + 1);
        float* hb = p.h + (size_t)(l & 1) * R * I;  // this layer's h exchange buffer
        // ---- A0: the consumers wait for the logit words of this layer
        // (complete once every CTA has added its rows of x_l) and sum their
        // shadow copies into lg; the router warps (token t: warp t) take the
        // top-k while the consumers stage x and the next router slice; the
        // producer warp then groups, hands the routing over (named barrier 4:
        // it arrives, the consumers wait) and goes on to issue the copies at once
        if (tid == kDkLeader) dk_trace<kTrace>(p, l, 0);
        if (warp == 0) {
            // A dry run of the routing steps on stale values (no status
            // bits, results overwritten below) while the consumers poll: it
            // brings their code (one non-inlined copy, shared with the real
            // pass) back into this SM's instruction caches, from which the
            // rest of the layer evicted it, so the real pass that gates the
            // layer's weight copies waits less on instruction fetches.
            dk_topk_smem(lg, E, k, 0, m, nullptr);
            dk_group(m, R, E, no_dedup);
        }
        bool polled = true;
        if (warp >= 1) {
            // consumers: every (token, expert) logit from the shadow
            // accumulators (an integer sum: exact in any order) into lg
            const int ct = tid - 32, nct = 32 * kDkConsumers;
            const unsigned long long* nacc_now = p.has_norm ? dk_nacc(p, l) : nullptr;
            for (int v = ct; v < B * Ep && polled; v += nct) {
                const int t = v / Ep, e = v - t * Ep;
                float val = -INFINITY;
                float rn = 1.f;
                if (nacc_now) {  // pre-norm: 1/sqrt(mean(x^2) + eps) of token t's input
                    long long ss = 0;
                    polled = polled && dk_poll_sum(nacc_now + t, (size_t)B, ss, p, m);
                    rn = 1.0f / sqrtf(__ll2float_rn(ss) * (1.0f / kFixScaleSq) / (float)H + p.eps);
                    if (e == 0) m->rn[t] = rn;
                }
                if (e < E) {
                    long long sum = 0;  // the shadow copies' integer sums, exact, then one rounding
                    polled = polled && dk_poll_sum(acc_now + (size_t)t * E + e, (size_t)B * E, sum, p, m);
                    val = rn * (__ll2float_rn(sum) * (1.0f / kFixScale));
                    if (lw.bias) val += __ldg(lw.bias + e);
                }
                lg[v] = val;
            }
        }
        if (__syncthreads_or(!polled)) {
            if (tid == 0) *(volatile int*)&m->abort_flag = 1;
            break;
        }
        if (tid == kDkLeader) dk_trace<kTrace>(p, l, 14);
        if (warp < B) {
            dk_topk_smem(lg + warp * Ep, E, k, warp, m, p.status);
            if (tid == 0) dk_trace<kTrace>(p, l, 7);
            if (B > 1) {  // warp 0 groups every token's selection
                if (warp == 0)
                    named_sync(3, 32 * B);
                else
                    named_arrive(3, 32 * B);
            }
        }
        if (warp == 0) {
            dk_group(m, R, E, no_dedup);
            if (blockIdx.x == 0) {
                if (p.ids_out && lane < R) p.ids_out[(size_t)l * R + lane] = m->ids[lane];
                if (p.w_out && lane < R) p.w_out[lane] = m->w[lane];
                if (p.g_offsets && !no_dedup) dk_store_grouping(p, m, R, E);
            }
            if (tid == 0) dk_trace<kTrace>(p, l, 9);
            named_arrive(4, kDkThreads);
        } else {
            const int ct = tid - 32, nct = 32 * kDkConsumers;
            if (l > 0) {
                // x_l from the tagged copy: every element carries the layer it
                // belongs to, so an element not yet visible is waited for on
                // its own (bounded), with no fence or barrier
                const int nv4 = (B * H) >> 2;
                const float* gn = p.has_norm ? gq + (size_t)(l & 1) * H : nullptr;
                const unsigned long long* xt = p.xt + (size_t)(l & 1) * B * H;
                for (int v0 = ct; v0 < nv4; v0 += 2 * nct) {
                    // both groups' loads in flight before either is checked
                    const int v1 = v0 + nct;
                    Tagged4 t0, t1;
                    dk_ld_tagged4(xt + 4 * (size_t)v0, t0);
                    if (v1 < nv4) dk_ld_tagged4(xt + 4 * (size_t)v1, t1);
                    float4 a;
                    bool ok = dk_load_tagged4(xt + 4 * (size_t)v0, (unsigned)l, t0, a, p, m);
                    if (ok) dk_store_x(xs, xq, H, 4 * v0, a, gn, m);
                    if (ok && v1 < nv4) {
                        ok = dk_load_tagged4(xt + 4 * (size_t)v1, (unsigned)l, t1, a, p, m);
                        if (ok) dk_store_x(xs, xq, H, 4 * v1, a, gn, m);
                    }
                    if (!ok) {
                        *(volatile int*)&m->abort_flag = 1;
                        break;
                    }
                }
            } else if (!p.x_bf16) {
                // both loads of a thread in flight before either store
                const float* xsrc = static_cast<const float*>(p.x_in);
                const int nv4 = (B * H) >> 2;
                const float* gn = p.has_norm ? gq + (size_t)(l & 1) * H : nullptr;
                for (int v0 = ct; v0 < nv4; v0 += 2 * nct) {
                    const int v1 = v0 + nct;
                    const float4 a = ld_act_f4(xsrc + 4 * (size_t)v0);
                    const float4 b = v1 < nv4 ? ld_act_f4(xsrc + 4 * (size_t)v1) : make_float4(0.f, 0.f, 0.f, 0.f);
                    dk_store_x(xs, xq, H, 4 * v0, a, gn, m);
                    if (v1 < nv4) dk_store_x(xs, xq, H, 4 * v1, b, gn, m);
                }
            } else {
                const uint16_t* xb = static_cast<const uint16_t*>(p.x_in);
                for (int v = ct; v < (B * H) >> 2; v += nct) {
                    const uint2 w = *reinterpret_cast<const uint2*>(xb + 4 * (size_t)v);
                    const float2 lo = bf16x2_to_f2(w.x), hi = bf16x2_to_f2(w.y);
                    dk_store_x(xs, xq, H, 4 * v, make_float4(lo.x, lo.y, hi.x, hi.y),
                               p.has_norm ? gq + (size_t)(l & 1) * H : nullptr, m);
                }
            }
            if (has_next) {
                const LayerWeights& wn = p.layer[l + 1];
                for (int v = ct; v < E * (nrows >> 3); v += nct) {
                    const int e = v / (nrows >> 3), c8 = (v - e * (nrows >> 3)) << 3;
                    cp_async16(wrs + e * p.maxrows + c8, wn.w_router + (size_t)e * H + h0 + c8);
                }
                // the next layer's norm weights into the buffer that layer l-1 used
                if (p.has_norm) {
                    float* gd = gq + (size_t)((l + 1) & 1) * H;
                    for (int v = ct; v < (H >> 2); v += nct) cp_async16(gd + 4 * v, wn.norm + 4 * v);
                }
                cp_async_commit();
            }
            if (tid == kDkLeader) dk_trace<kTrace>(p, l, 8);
            named_sync(4, kDkThreads);
        }
        const int U = m->U;
        const DkWork wk = dk_work(wbase, U, m);
        if (tid == kDkLeader) dk_trace<kTrace>(p, l, 1);
        // Direct mode: when this CTA's gate/up rows and down rows of the layer
        // fit in the ring area together, they are fetched by a handful of
        // large bulk copies (rows of one expert are contiguous) onto two
        // barriers instead of chunk by chunk through the ring.
        const uint32_t d_gate_bytes = (uint32_t)wk.ng * 2u * (uint32_t)rowg;
        const uint32_t d_down_bytes = (uint32_t)U * (uint32_t)nrows * (uint32_t)rowd;
        // (kDirect: the host has checked that every CTA's share fits for any routing)
        const bool direct = kDirect || (size_t)d_gate_bytes + d_down_bytes <= (size_t)p.S * p.stage_bytes &&
                            d_gate_bytes < (1u << 20) && d_down_bytes < (1u << 20);
        const bool d_gate = direct && wk.ng > 0, d_down = direct && d_down_bytes > 0;
        unsigned char* d_g = ring;                                       // [ng][rowg] gate rows
        unsigned char* d_u = ring + (size_t)wk.ng * rowg;                // [ng][rowg] up rows
        unsigned char* d_d = ring + (size_t)wk.ng * 2 * rowg;            // [U][nrows][rowd] down rows

        if (warp == 0 && direct) {
            // ================= producer, direct mode
            if (lane == 0 && d_gate) {
                // the CTA's pairs in up to kDkGChunks chunks, each on its own
                // barrier, so that the consumers start on the first chunk while
                // the others are still on their way (every chunk barrier
                // completes one phase per layer: unused ones with no bytes)
                const int csz = max(4, (wk.ng + kDkGChunks - 1) / kDkGChunks);
                for (int ch = 0; ch < kDkGChunks; ++ch) {
                    const int ca = min(wk.ng, ch * csz), cb = min(wk.ng, ca + csz);
                    mbar_arrive_expect_tx(&gch[ch], (uint32_t)(cb - ca) * 2u * (uint32_t)rowg);
                    if (cb > ca)
                        dk_gate_runs(lw.gate_up, m->seg_e, wk.ga + ca, wk.ga + cb, H, I, d_g + (size_t)ca * rowg,
                                     d_u + (size_t)ca * rowg, &gch[ch], kW2);
                }
            }
            __syncwarp();
            if (lane == 1 && d_down) {
                // the gate/up rows first: the down rows are needed only after
                // the mid-layer barrier, so they do not share the bandwidth
                if (d_gate) {
                    const int csz = max(4, (wk.ng + kDkGChunks - 1) / kDkGChunks);
                    dk_wait(&gch[(wk.ng - 1) / csz], (uint32_t)(dg_count & 1), m, p);
                }
                mbar_arrive_expect_tx(&dbar[1], d_down_bytes);
                for (int u = 0; u < U; ++u)
                    bulk_g2s(d_d + (size_t)u * nrows * rowd,
                             reinterpret_cast<const unsigned char*>(lw.down) + ((size_t)m->seg_e[u] * H + h0) * rowd,
                             (uint32_t)nrows * (uint32_t)rowd, &dbar[1]);
            }
            __syncwarp();
        } else if (warp == 0) {
            // ================= producer: lane s owns ring stage s (S <= 32) and
            // issues that stage's chunks of the layer in order, so the lanes
            // overlap the cost of issuing bulk copies while each stage is still
            // armed strictly in sequence (a stage is re-armed only after its
            // previous chunk was released, and the wait parity never aliases).
            // Every stage is free at the start of a layer (all of the last
            // layer's chunks were consumed before its final barrier), so only a
            // chunk that reuses a stage within this layer waits for the release.
            if (lane == 0) dk_trace<kTrace>(p, l, 15);
            const int s = lane;
            const int c_first = lane < p.S ? ((s - rs) % p.S + p.S) % p.S : wk.n;
            for (int c = c_first; c < wk.n; c += p.S) {
                const int n = ring_pos + c;
                const uint32_t ph = rph ^ (uint32_t)(((rs + c) / p.S) & 1);
                if (c >= p.S && !dk_wait(&empty[s], ph ^ 1u, m, p)) break;
                unsigned char* dst = ring + (size_t)s * p.stage_bytes;
                if (c < wk.ng) {
                    const int pq = wk.ga + c;
                    const int u = pq / I, i = pq - u * I;
                    const unsigned char* G =
                        reinterpret_cast<const unsigned char*>(lw.gate_up) + (size_t)m->seg_e[u] * 2 * I * rowg;
                    mbar_arrive_expect_tx(&full[s], 2u * (uint32_t)rowg);
                    bulk_g2s(dst, G + (size_t)i * rowg, (uint32_t)rowg, &full[s]);
                    bulk_g2s(dst + rowg, G + (size_t)(I + i) * rowg, (uint32_t)rowg, &full[s]);
                } else {
                    const int mm = c - wk.ng;
                    const int u = mm / wk.nd_per_u, sub = mm - u * wk.nd_per_u;
                    const int r0 = wk.h0 + sub * wk.nr;
                    const int r1 = min(wk.h1, r0 + wk.nr);
                    const unsigned char* D = reinterpret_cast<const unsigned char*>(lw.down) + (size_t)m->seg_e[u] * H * rowd;
                    const uint32_t bytes = (uint32_t)(r1 - r0) * (uint32_t)rowd;
                    mbar_arrive_expect_tx(&full[s], bytes);
                    bulk_g2s(dst, D + (size_t)r0 * rowd, bytes, &full[s]);
                }
                m->last_pos[s] = n;
            }
            __syncwarp();
            if (lane == 0 && p.trace) {  // profiling only: when did the first, the last gate/up and the last chunk land?
                dk_trace<kTrace>(p, l, 18);
                for (int c = 0; c < wk.n; ++c) {
                    const int n = ring_pos + c;
                    mbar_wait(&full[n % p.S], (uint32_t)((n / p.S) & 1), kDkWaitLimit);
                    if (c == 0) dk_trace<kTrace>(p, l, 19);
                    if (c == wk.ng - 1) dk_trace<kTrace>(p, l, 16);
                    if (c == wk.n - 1) dk_trace<kTrace>(p, l, 17);
                }
            }
        }
        if (warp == 0 && p.prefetch_k > 0 && has_next) {
            // ================= producer warp, once the mid-layer barrier is
            // through: the next layer's predicted experts prefetched into L2
            bool seen = false;
            for (uint32_t it = 0; it < kDkWaitLimit; ++it) {
                uint32_t v;
                asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(&m->mid_epoch)) : "memory");
                if ((int)v >= l + 1) {
                    seen = true;
                    break;
                }
                if (*(volatile int*)&m->abort_flag) break;
                __nanosleep(64);
            }
            if (__all_sync(0xffffffffu, seen)) {
                const int my_e = dk_predict_top(p.alog + (size_t)(l & 1) * E, E, p.prefetch_k);
                dk_prefetch_l2(p.layer[l + 1], my_e, H, I, p.prefetch_k, kW2);
            }
        }
        if (warp != 0) {
            // ================= consumers: gate/up pairs
            // Chunk c sits in stage (ring_pos + c) % S and is consumed by warp
            // (ring_pos + c) % W; since S % W == 0, every use of a stage goes to
            // the same warp, in order, so a warp never waits on a stage phase
            // whose predecessor it has not consumed itself (mbarrier parity
            // waits would alias otherwise).
            const int cw = warp - 1;
            const bool consumes = cw < p.W;
            int s, q0, c0;
            uint32_t ph;
            c0 = ((cw - rs % p.W) % p.W + p.W) % p.W;
            q0 = (rs + c0) / p.S;
            s = rs + c0 - q0 * p.S;
            ph = rph ^ (uint32_t)(q0 & 1);
            const bool predicting = p.prefetch_k > 0 && has_next && cw == kDkConsumers - 1;
            if (predicting) dk_predict_logits(p.layer[l + 1], xq, H, E, p.alog + (size_t)(l & 1) * E);
            if (d_gate) {
                const int csz = max(4, (wk.ng + kDkGChunks - 1) / kDkGChunks);
                int landed = -1;
                for (int c = cw; c < wk.ng; c += kDkConsumers) {
                    if (c / csz != landed) {
                        if (!dk_wait(&gch[c / csz], (uint32_t)(dg_count & 1), m, p)) break;
                        landed = c / csz;
                        if (tid == kDkLeader) dk_trace<kTrace>(p, l, 12);
                    }
                    const int q = wk.ga + c;
                    const int u = q / I, i = q - u * I;
                    const float* gsr = kF8 ? lw.gate_up_scale + (size_t)m->seg_e[u] * sg_e + (size_t)(i >> 7) * sg_ld : nullptr;
                    const float* usr = kF8 ? lw.gate_up_scale + (size_t)m->seg_e[u] * sg_e + (size_t)((I + i) >> 7) * sg_ld : nullptr;
                    const unsigned char* gbs = kF4 ? lw.gate_up_bs + ((size_t)m->seg_e[u] * 2 * I + i) * (H >> 4) : nullptr;
                    dk_pair_compute<kNQ, kF8, kF4>(m, d_g + (size_t)c * rowg, d_u + (size_t)c * rowg, xq, H, I, k, u, i,
                                                   hb, gsr, usr, gbs, kF4 ? gbs + (size_t)I * (H >> 4) : nullptr,
                                                   kF4 ? __ldg(lw.gate_up_gs + m->seg_e[u]) : 1.f);
                }
            }
            for (int c = c0; !direct && consumes && c < wk.ng; c += p.W) {
                if (*(volatile int*)&m->abort_flag) break;
                if (!dk_wait(&full[s], ph, m, p)) break;
                if (tid == kDkLeader && c == c0) dk_trace<kTrace>(p, l, 12);
                const int q = wk.ga + c;
                const int u = q / I, i = q - u * I;
                const unsigned char* st = ring + (size_t)s * p.stage_bytes;
                const float* gsr = kF8 ? lw.gate_up_scale + (size_t)m->seg_e[u] * sg_e + (size_t)(i >> 7) * sg_ld : nullptr;
                const float* usr = kF8 ? lw.gate_up_scale + (size_t)m->seg_e[u] * sg_e + (size_t)((I + i) >> 7) * sg_ld : nullptr;
                const unsigned char* gbs = kF4 ? lw.gate_up_bs + ((size_t)m->seg_e[u] * 2 * I + i) * (H >> 4) : nullptr;
                dk_pair_compute<kNQ, kF8, kF4>(m, st, st + rowg, xq, H, I, k, u, i, hb, gsr, usr, gbs,
                                               kF4 ? gbs + (size_t)I * (H >> 4) : nullptr,
                                               kF4 ? __ldg(lw.gate_up_gs + m->seg_e[u]) : 1.f);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                s += p.W;
                if (s >= p.S) {
                    s -= p.S;
                    ph ^= 1u;
                }
            }
            // ---- all gate/up pairs of every CTA done
            if (tid == kDkLeader) dk_trace<kTrace>(p, l, 2);
            const bool ok = dk_grid_sync(p, epoch, m, 1, 32 * kDkConsumers);
            // ---- B: down rows of every selected expert for this CTA's rows
            if (ok) {
            for (int v = tid - 32; v < (R * I) >> 2; v += 32 * kDkConsumers)
                reinterpret_cast<float4*>(hs)[v] = ld_act_f4(hb + 4 * (size_t)v);
            if (blockIdx.x == 0) {  // clear the accumulator set that layer l-1 read (layer l+1 fills it)
                unsigned long long* a2 = dk_acc(p, l + 2);
                for (int v = tid - 32; v < kDkShadows * B * E; v += 32 * kDkConsumers) a2[v] = 0ull;
                if (p.has_norm)
                    for (int v = tid - 32; v < kDkShadows * B; v += 32 * kDkConsumers) dk_nacc(p, l + 2)[v] = 0ull;
            }
            named_sync(1, 32 * kDkConsumers);
            if (tid == kDkLeader) dk_trace<kTrace>(p, l, 3);
            if (tid == kDkLeader) {  // tell the producer warp that every CTA's predicted logits are visible
                asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(&m->mid_epoch)), "r"(l + 1)
                             : "memory");
            }
            if (d_down) {
                const int ng4 = (nrows + 3) >> 2;
                bool landed = false;
                for (int j = cw; j < U * ng4; j += kDkConsumers) {
                    if (!landed) {
                        if (!dk_wait(&dbar[1], (uint32_t)(dd_count & 1), m, p)) break;
                        landed = true;
                    }
                    const int u = j / ng4, rg = j - u * ng4;
                    const int r0 = h0 + 4 * rg, r1 = min(h1, r0 + 4);
                    dk_down_compute<kNQ, kF8, kF4>(m, d_d + ((size_t)u * nrows + 4 * rg) * rowd, r0, r1, I, hs, os,
                                                   p.maxrows, h0, u,
                                                   kF8 ? lw.down_scale + (size_t)m->seg_e[u] * sd_e : nullptr, sd_ld,
                                                   kF4 ? lw.down_bs + (size_t)m->seg_e[u] * H * (I >> 4) : nullptr,
                                                   kF4 ? __ldg(lw.down_gs + m->seg_e[u]) : 1.f);
                }
            }
            c0 = wk.ng + ((cw - (rs + wk.ng) % p.W) % p.W + p.W) % p.W;
            q0 = (rs + c0) / p.S;
            s = rs + c0 - q0 * p.S;
            ph = rph ^ (uint32_t)(q0 & 1);
            for (int c = c0; !direct && consumes && c < wk.n; c += p.W) {
                if (*(volatile int*)&m->abort_flag) break;
                if (!dk_wait(&full[s], ph, m, p)) break;

                const int mm = c - wk.ng;
                const int u = mm / wk.nd_per_u, sub = mm - u * wk.nd_per_u;
                const int r0 = wk.h0 + sub * wk.nr;
                const int r1 = min(wk.h1, r0 + wk.nr);
                const unsigned char* st = ring + (size_t)s * p.stage_bytes;
                dk_down_compute<kNQ, kF8, kF4>(m, st, r0, r1, I, hs, os, p.maxrows, h0, u,
                                               kF8 ? lw.down_scale + (size_t)m->seg_e[u] * sd_e : nullptr, sd_ld,
                                               kF4 ? lw.down_bs + (size_t)m->seg_e[u] * H * (I >> 4) : nullptr,
                                               kF4 ? __ldg(lw.down_gs + m->seg_e[u]) : 1.f);
                __syncwarp();
                if (c == c0 && cw == 0 && lane == 0) dk_trace<kTrace>(p, l, 13);
                if (lane == 0) mbar_arrive(&empty[s]);
                s += p.W;
                if (s >= p.S) {
                    s -= p.S;
                    ph ^= 1u;
                }
            }
            named_sync(1, 32 * kDkConsumers);
            if (tid == kDkLeader) dk_trace<kTrace>(p, l, 4);
            // ---- combine (+ residual) for this CTA's rows, j ascending.  When the
            // residual is the layer input itself (a stack) it is already in xs.
            const bool res_in_xs = p.residual != nullptr && p.residual == p.x_in && !p.x_bf16;
            for (int v = tid - 32; v < B * nrows; v += 32 * kDkConsumers) {
                const int t = v / nrows, r = v - t * nrows;
                float a = 0.f;
                for (int j = 0; j < k; ++j)
                    a = fmaf(m->w[t * k + j], os[m->pos[t * k + j] * p.maxrows + r], a);
                const size_t gi = (size_t)t * H + h0 + r;
                if (res_in_xs)
                    a = xs[t * H + h0 + r] + a;
                else if (p.residual)
                    a = ld_act_f(p.residual + gi) + a;
                if (has_next)  // x_{l+1} for every CTA, tagged with its layer (buffers alternate by layer)
                    st_relaxed_gpu_u64(p.xt + (size_t)((l + 1) & 1) * B * H + gi,
                                       ((unsigned long long)(l + 1) << 32) | __float_as_uint(a));
                else
                    p.y[gi] = a;
                xs[t * H + h0 + r] = a;  // x_{l+1} rows for the next router
            }
            if (tid == kDkLeader) dk_trace<kTrace>(p, l, 10);
            if (has_next) cp_async_wait_all();
            named_sync(1, 32 * kDkConsumers);
            if (tid == kDkLeader) dk_trace<kTrace>(p, l, 11);
            // ---- router of layer l+1: partial dot products over this CTA's rows
            if (has_next)
                dk_router_partials(wrs, p.maxrows, xs, H, h0, nrows, B, E, acc_next, tid - 32,
                                   32 * kDkConsumers, p.status, p.has_norm ? gq + (size_t)((l + 1) & 1) * H : nullptr,
                                   p.has_norm ? dk_nacc(p, l + 1) : nullptr);
            }  // ok
            if (has_next) cp_async_wait_all();
        }
        if (!direct) {
            ring_pos += wk.n;
            const int t = rs + wk.n, q = t / p.S;
            rs = t - q * p.S;
            rph ^= (uint32_t)(q & 1);
        }
        dg_count += d_gate ? 1 : 0;
        dd_count += d_down ? 1 : 0;
        if (tid == kDkLeader) dk_trace<kTrace>(p, l, 5);
        // no device-wide barrier here: the next layer waits on its logit words
        __syncthreads();
        if (tid == kDkLeader) dk_trace<kTrace>(p, l, 6);
    }
    // leave only after this CTA's own copies in flight have landed: the latest
    // phase armed in each stage is the only one that can still be in flight
    // (they have all landed already unless a wait gave up)
    __syncthreads();
    if (warp == 0) {
        for (int st = lane; st < p.S; st += 32) {
            const int n = m->last_pos[st];
            if (n >= 0) mbar_wait(&full[st], (uint32_t)((n / p.S) & 1), kDkWaitLimit);
        }
        if (lane < kDkGChunks && dg_count > 0) mbar_wait(&gch[lane], (uint32_t)((dg_count - 1) & 1), kDkWaitLimit);
        if (lane == 1 && dd_count > 0) mbar_wait(&dbar[1], (uint32_t)((dd_count - 1) & 1), kDkWaitLimit);
    }
    __syncthreads();
}

}  // namespace moe
