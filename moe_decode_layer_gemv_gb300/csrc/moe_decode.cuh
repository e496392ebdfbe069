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

#include "moe_common.cuh"
#include "moe_ptx.cuh"

namespace moe {

constexpr int kDkConsumers = 8;                    // consumer warps
constexpr int kDkThreads = 32 * (kDkConsumers + 1);  // + one producer warp
constexpr int kDkMaxB = 4;
constexpr int kDkMaxR = 32;
constexpr int kDkMaxStages = 32;
constexpr uint32_t kDkWaitLimit = 1u << 22;
constexpr unsigned long long kDkSpinLimit = 1ull << 22;
constexpr float kFixScale = 4294967296.0f;  // 2^32
constexpr int kDkSmemMax = 227 * 1024;

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
    float* h;          // [R, I] exchange buffer
    unsigned long long* acc;  // [2][B][E] fixed-point logits
    unsigned* bar;            // [0] arrival counter, [1] abort word
    int32_t* status;
    int S, stage_bytes, maxrows;
    int off_misc, off_x, off_h, off_o, off_wr, off_ring;
};

struct DkMisc {
    int abort_flag;
    int sync_ok;
    int U;
    int ids[kDkMaxR];
    float w[kDkMaxR];
    int pos[kDkMaxR];   // position of route r in the grouped list
    int rat[kDkMaxR];   // route at position p
    int seg_e[kDkMaxR];
    int seg_p[kDkMaxR + 1];
};

// --------------------------------------------------------- work partition
// Hidden rows owned by CTA c in the down/combine/router step: groups of 8
// rows (16-byte aligned bf16 slices), split as evenly as possible.
__device__ __forceinline__ void dk_rows(int c, int G, int H, int& h0, int& h1) {
    const long long ng = H >> 3;
    h0 = 8 * (int)((long long)c * ng / G);
    h1 = 8 * (int)((long long)(c + 1) * ng / G);
}

// First gate/up row pair of CTA c (pairs are numbered segment-major).  The
// split balances each CTA's total bytes (its gate/up pairs plus its down rows
// of every selected expert).  Ranges [start(c), max(start(c), start(c+1)))
// cover every pair even where start() is not monotonic (tiny H).
__device__ __forceinline__ long long dk_gate_start(int c, int G, int U, int H, int I) {
    const long long P = (long long)U * I;
    if (c <= 0) return 0;
    if (c >= G) return P;
    const long long h0 = 8LL * ((long long)c * (H >> 3) / G);
    const long long target = (long long)c * U * I * 6LL * H / G;
    long long v = (target - h0 * U * 2LL * I) / (4LL * H);
    return v < 0 ? 0 : (v > P ? P : v);
}

struct DkWork {
    long long ga, gb;  // gate/up pairs [ga, gb)
    int h0, h1, nr, nd_per_u, ng, n;
};

__device__ __forceinline__ DkWork dk_work(const DkParams& p, int U) {
    DkWork w;
    const int G = gridDim.x, c = blockIdx.x;
    w.ga = dk_gate_start(c, G, U, p.H, p.I);
    const long long nb = dk_gate_start(c + 1, G, U, p.H, p.I);
    w.gb = nb > w.ga ? nb : w.ga;
    dk_rows(c, G, p.H, w.h0, w.h1);
    int nr = p.stage_bytes / (2 * p.I);
    if (nr < 1) nr = 1;
    w.nr = nr;
    w.nd_per_u = w.h1 > w.h0 ? (w.h1 - w.h0 + nr - 1) / nr : 0;
    w.ng = (int)(w.gb - w.ga);
    w.n = w.ng + U * w.nd_per_u;
    return w;
}

// ------------------------------------------------------------- barriers
// Device-wide barrier among the threads of named barrier `bar_id`
// (`nthreads` of them) in every CTA; thread kDkLeader does the arrive/wait.
constexpr int kDkLeader = 32;  // first consumer thread

__device__ __forceinline__ bool dk_grid_sync(const DkParams& p, unsigned& epoch, DkMisc* m, int bar_id,
                                             int nthreads) {
    named_sync(bar_id, nthreads);
    if (threadIdx.x == kDkLeader) {
        epoch += 1;
        const unsigned target = epoch * gridDim.x;
        __threadfence();
        red_release_gpu_add(p.bar, 1u);
        int ok = 1;
        unsigned long long spins = 0;
        while (ld_acquire_gpu(p.bar) < target) {
            ++spins;
            if ((spins & 127ull) == 0 && ld_acquire_gpu(p.bar + 1) != 0u) {
                ok = 0;
                break;
            }
            if (spins > kDkSpinLimit) {
                set_status(p.status, MOE_DEV_TIMEOUT);
                atomicExch(p.bar + 1, 1u);
                ok = 0;
                break;
            }
            if (spins > 256) __nanosleep(32);
        }
        __threadfence();
        m->sync_ok = ok;
        if (!ok) m->abort_flag = 1;
    }
    named_sync(bar_id, nthreads);
    return m->sync_ok != 0;
}

// mbarrier wait that also gives up when the CTA has aborted
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

// ----------------------------------------------------------- small steps
__device__ __forceinline__ float fix_to_float(unsigned long long v) {
    return (float)((double)(long long)v * (1.0 / 4294967296.0));
}

__device__ __forceinline__ unsigned long long float_to_fix(float v) {
    return (unsigned long long)__float2ll_rn(v * kFixScale);
}

// top-k of one token's logits held in shared memory (one warp); same rule
// as the stand-alone top-k phase: ties to the lower id, fp32 softmax,
// renormalised over the selected experts.
__device__ void dk_topk_token(const float* lg, int E, int k, int t, DkMisc* m, int32_t* status) {
    const int lane = threadIdx.x & 31;
    float v[8];
    bool bad = false;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int e = lane + 32 * s;
        v[s] = e < E ? lg[e] : -INFINITY;
        if (e < E && !isfinite(v[s])) bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_DEV_NONFINITE);
    unsigned taken = 0;
    float selv[MOE_MAX_TOPK];
    int seli[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        selv[j] = -INFINITY;
        seli[j] = 0;
        if (j < k) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int e = lane + 32 * s;
                if (e < E && !((taken >> s) & 1u) && (v[s] > bv || (v[s] == bv && e < bi))) {
                    bv = v[s];
                    bi = e;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (bi == 0x7fffffff) bi = 0;
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            selv[j] = bv;
            seli[j] = bi;
        }
    }
    const float mx = selv[0];
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (lane + 32 * q < E) s += expf(v[q] - mx);
    s = warp_sum(s);
    if (lane == 0) {
        float pr[MOE_MAX_TOPK];
        float ssel = 0.f;
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK; ++j) {
            pr[j] = 0.f;
            if (j < k) {
                pr[j] = expf(selv[j] - mx) / s;
                ssel += pr[j];
            }
        }
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK; ++j)
            if (j < k) {
                m->ids[t * k + j] = seli[j];
                m->w[t * k + j] = pr[j] / ssel;
            }
    }
}

// Stable grouping of R <= 32 routes by expert in one warp: the position of
// route r is (#routes with a smaller expert) + (#earlier routes with the
// same expert) -- the counting sort's result, computed directly.
__device__ void dk_group(DkMisc* m, int R, bool no_dedup) {
    const int lane = threadIdx.x & 31;
    const int e = lane < R ? m->ids[lane] : 0x7fffffff;
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

// ------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kDkThreads, 1) decode_kernel(const DkParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kDkMaxStages;
    DkMisc* m = reinterpret_cast<DkMisc*>(smem + p.off_misc);
    float* xs = reinterpret_cast<float*>(smem + p.off_x);   // [B][H]
    float* hs = reinterpret_cast<float*>(smem + p.off_h);   // [R][I]
    float* os = reinterpret_cast<float*>(smem + p.off_o);   // [R][maxrows]
    uint16_t* wrs = reinterpret_cast<uint16_t*>(smem + p.off_wr);  // [E][maxrows]
    unsigned char* ring = smem + p.off_ring;
    float* lg = reinterpret_cast<float*>(smem + p.off_misc + sizeof(DkMisc));  // [B][E]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B, H = p.H, I = p.I, E = p.E, k = p.k, R = B * k;
    const bool no_dedup = (p.flags & MOE_F_NO_DEDUP) != 0;
    int h0, h1;
    dk_rows(blockIdx.x, gridDim.x, H, h0, h1);
    const int nrows = h1 - h0;

    if (tid == 0) {
        for (int s = 0; s < p.S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        m->abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    unsigned epoch = 0;        // barrier count (leader thread only)
    long long ring_pos = 0;    // chunks through the ring so far (all threads agree)
    long long issued = 0;      // producer: chunks issued

    // ---- router of layer 0: partial dot products over this CTA's rows
    {
        const LayerWeights& w0 = p.layer[0];
        for (int v = tid; v < E * (nrows >> 3); v += blockDim.x) {
            const int e = v / (nrows >> 3), c8 = (v - e * (nrows >> 3)) << 3;
            cp_async16(wrs + e * p.maxrows + c8, w0.w_router + (size_t)e * H + h0 + c8);
        }
        cp_async_commit();
        for (int v = tid; v < B * nrows; v += blockDim.x) {
            const int t = v / nrows, r = v - t * nrows;
            const size_t off = (size_t)t * H + h0 + r;
            xs[t * H + h0 + r] = p.x_bf16 ? __uint_as_float((uint32_t)static_cast<const uint16_t*>(p.x_in)[off] << 16)
                                          : ld_act_f(static_cast<const float*>(p.x_in) + off);
        }
        cp_async_wait_all();
        __syncthreads();
        if (nrows > 0) {
            for (int q = warp; q < B * E; q += blockDim.x >> 5) {
                const int t = q / E, e = q - t * E;
                float part = 0.f;
                for (int r = lane; r < nrows; r += 32)
                    part = fmaf(__uint_as_float((uint32_t)wrs[e * p.maxrows + r] << 16), xs[t * H + h0 + r], part);
                part = warp_sum(part);
                if (lane == 0) red_add_u64(p.acc + (size_t)t * E + e, float_to_fix(part));
            }
        }
    }
    dk_grid_sync(p, epoch, m, 0, kDkThreads);

    for (int l = 0; l < p.L && !*(volatile int*)&m->abort_flag; ++l) {
        const LayerWeights& lw = p.layer[l];
        const bool has_next = l + 1 < p.L;
        unsigned long long* acc_now = p.acc + (size_t)(l & 1) * B * E;
        unsigned long long* acc_next = p.acc + (size_t)((l + 1) & 1) * B * E;
        // ---- A0: logits, x, next router slice
        for (int v = tid; v < B * E; v += blockDim.x) {
            const int e = v % E;
            float val = fix_to_float(__ldcg(acc_now + v));
            if (lw.bias) val += lw.bias[e];
            lg[v] = val;
        }
        if (l > 0 || !p.x_bf16) {
            const float* xsrc = (l > 0) ? p.y : static_cast<const float*>(p.x_in);
            for (int v = tid; v < (B * H) >> 2; v += blockDim.x)
                reinterpret_cast<float4*>(xs)[v] = ld_act_f4(xsrc + 4 * (size_t)v);
        } else {
            const uint16_t* xb = static_cast<const uint16_t*>(p.x_in);
            for (int v = tid; v < B * H; v += blockDim.x) xs[v] = __uint_as_float((uint32_t)xb[v] << 16);
        }
        if (has_next && tid >= 32) {
            const LayerWeights& wn = p.layer[l + 1];
            for (int v = tid - 32; v < E * (nrows >> 3); v += 32 * kDkConsumers) {
                const int e = v / (nrows >> 3), c8 = (v - e * (nrows >> 3)) << 3;
                cp_async16(wrs + e * p.maxrows + c8, wn.w_router + (size_t)e * H + h0 + c8);
            }
            cp_async_commit();
        }
        __syncthreads();
        if (warp < B) dk_topk_token(lg + warp * E, E, k, warp, m, p.status);
        __syncthreads();
        if (warp == 0) dk_group(m, R, no_dedup);
        __syncthreads();
        if (blockIdx.x == 0) {
            if (p.ids_out && tid < R) p.ids_out[(size_t)l * R + tid] = m->ids[tid];
            if (p.w_out && tid < R) p.w_out[tid] = m->w[tid];
        }
        const int U = m->U;
        const DkWork wk = dk_work(p, U);

        if (warp == 0) {
            // ================= producer: one lane issues every chunk in order
            if (lane == 0) {
                for (int c = 0; c < wk.n; ++c) {
                    const long long n = ring_pos + c;
                    const int s = (int)(n % p.S);
                    const uint32_t ph = (uint32_t)((n / p.S) & 1);
                    if (!dk_wait(&empty[s], ph ^ 1u, m, p)) break;
                    unsigned char* dst = ring + (size_t)s * p.stage_bytes;
                    if (c < wk.ng) {
                        const long long q = wk.ga + c;
                        const int u = (int)(q / I), i = (int)(q - (long long)u * I);
                        const uint16_t* G = lw.gate_up + (size_t)m->seg_e[u] * 2 * I * H;
                        mbar_arrive_expect_tx(&full[s], 4u * H);
                        bulk_g2s(dst, G + (size_t)i * H, 2u * H, &full[s]);
                        bulk_g2s(dst + 2 * H, G + (size_t)(I + i) * H, 2u * H, &full[s]);
                    } else {
                        const int mm = c - wk.ng;
                        const int u = mm / wk.nd_per_u, sub = mm - u * wk.nd_per_u;
                        const int r0 = wk.h0 + sub * wk.nr;
                        const int r1 = min(wk.h1, r0 + wk.nr);
                        const uint16_t* D = lw.down + (size_t)m->seg_e[u] * H * I;
                        const uint32_t bytes = 2u * (r1 - r0) * I;
                        mbar_arrive_expect_tx(&full[s], bytes);
                        bulk_g2s(dst, D + (size_t)r0 * I, bytes, &full[s]);
                    }
                    issued = n + 1;
                }
            }
        } else {
            // ================= consumers: gate/up pairs
            const int cw = warp - 1;
            for (int c = cw; c < wk.ng; c += kDkConsumers) {
                if (*(volatile int*)&m->abort_flag) break;
                const long long n = ring_pos + c;
                const int s = (int)(n % p.S);
                if (!dk_wait(&full[s], (uint32_t)((n / p.S) & 1), m, p)) break;
                const long long q = wk.ga + c;
                const int u = (int)(q / I), i = (int)(q - (long long)u * I);
                const unsigned char* st = ring + (size_t)s * p.stage_bytes;
                const int p0 = m->seg_p[u], p1 = m->seg_p[u + 1];
                int tok[kDkMaxB];
#pragma unroll
                for (int qq = 0; qq < kDkMaxB; ++qq) tok[qq] = p0 + qq < p1 ? m->rat[p0 + qq] / k : 0;
                float2 ag[kDkMaxB], au[kDkMaxB];
#pragma unroll
                for (int qq = 0; qq < kDkMaxB; ++qq) ag[qq] = au[qq] = make_float2(0.f, 0.f);
                const int nq = p1 - p0;
                for (int v = lane; v < (H >> 3); v += 32) {
                    const uint4 gw = *reinterpret_cast<const uint4*>(st + 16 * v);
                    const uint4 uw = *reinterpret_cast<const uint4*>(st + 2 * H + 16 * v);
                    const float2 g0 = bf16x2_to_f2(gw.x), g1 = bf16x2_to_f2(gw.y);
                    const float2 g2 = bf16x2_to_f2(gw.z), g3 = bf16x2_to_f2(gw.w);
                    const float2 u0 = bf16x2_to_f2(uw.x), u1 = bf16x2_to_f2(uw.y);
                    const float2 u2 = bf16x2_to_f2(uw.z), u3 = bf16x2_to_f2(uw.w);
#pragma unroll
                    for (int qq = 0; qq < kDkMaxB; ++qq) {
                        if (qq < nq) {
                            const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)tok[qq] * H + 8 * v);
                            const float4 xa = xp[0], xb = xp[1];
                            ag[qq] = ffma2(g0, make_float2(xa.x, xa.y), ag[qq]);
                            au[qq] = ffma2(u0, make_float2(xa.x, xa.y), au[qq]);
                            ag[qq] = ffma2(g1, make_float2(xa.z, xa.w), ag[qq]);
                            au[qq] = ffma2(u1, make_float2(xa.z, xa.w), au[qq]);
                            ag[qq] = ffma2(g2, make_float2(xb.x, xb.y), ag[qq]);
                            au[qq] = ffma2(u2, make_float2(xb.x, xb.y), au[qq]);
                            ag[qq] = ffma2(g3, make_float2(xb.z, xb.w), ag[qq]);
                            au[qq] = ffma2(u3, make_float2(xb.z, xb.w), au[qq]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
                for (int qq = 0; qq < kDkMaxB; ++qq) {
                    if (qq < nq) {
                        const float g = warp_sum(ag[qq].x + ag[qq].y);
                        const float uu = warp_sum(au[qq].x + au[qq].y);
                        if (lane == 0) p.h[(size_t)(p0 + qq) * I + i] = silu_mul(g, uu);
                    }
                }
            }
            // ---- all gate/up pairs of every CTA done
            const bool ok = dk_grid_sync(p, epoch, m, 1, 32 * kDkConsumers);
            // ---- B: down rows of every selected expert for this CTA's rows
            if (ok) {
            for (int v = tid - 32; v < (R * I) >> 2; v += 32 * kDkConsumers)
                reinterpret_cast<float4*>(hs)[v] = ld_act_f4(p.h + 4 * (size_t)v);
            named_sync(1, 32 * kDkConsumers);
            for (int c = wk.ng + cw; c < wk.n; c += kDkConsumers) {
                if (*(volatile int*)&m->abort_flag) break;
                const long long n = ring_pos + c;
                const int s = (int)(n % p.S);
                if (!dk_wait(&full[s], (uint32_t)((n / p.S) & 1), m, p)) break;
                const int mm = c - wk.ng;
                const int u = mm / wk.nd_per_u, sub = mm - u * wk.nd_per_u;
                const int r0 = wk.h0 + sub * wk.nr;
                const int r1 = min(wk.h1, r0 + wk.nr);
                const unsigned char* st = ring + (size_t)s * p.stage_bytes;
                const int p0 = m->seg_p[u], p1 = m->seg_p[u + 1];
                for (int r = r0; r < r1; ++r) {
                    const unsigned char* row = st + (size_t)(r - r0) * 2 * I;
                    float2 acc[kDkMaxB];
#pragma unroll
                    for (int qq = 0; qq < kDkMaxB; ++qq) acc[qq] = make_float2(0.f, 0.f);
                    for (int v = lane; v < (I >> 3); v += 32) {
                        const uint4 dw = *reinterpret_cast<const uint4*>(row + 16 * v);
                        const float2 d0 = bf16x2_to_f2(dw.x), d1 = bf16x2_to_f2(dw.y);
                        const float2 d2 = bf16x2_to_f2(dw.z), d3 = bf16x2_to_f2(dw.w);
#pragma unroll
                        for (int qq = 0; qq < kDkMaxB; ++qq) {
                            if (p0 + qq < p1) {
                                const float4* hp = reinterpret_cast<const float4*>(hs + (size_t)(p0 + qq) * I + 8 * v);
                                const float4 ha = hp[0], hb = hp[1];
                                acc[qq] = ffma2(d0, make_float2(ha.x, ha.y), acc[qq]);
                                acc[qq] = ffma2(d1, make_float2(ha.z, ha.w), acc[qq]);
                                acc[qq] = ffma2(d2, make_float2(hb.x, hb.y), acc[qq]);
                                acc[qq] = ffma2(d3, make_float2(hb.z, hb.w), acc[qq]);
                            }
                        }
                    }
#pragma unroll
                    for (int qq = 0; qq < kDkMaxB; ++qq) {
                        if (p0 + qq < p1) {
                            const float o = warp_sum(acc[qq].x + acc[qq].y);
                            if (lane == 0) os[(p0 + qq) * p.maxrows + (r - h0)] = o;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            named_sync(1, 32 * kDkConsumers);
            // ---- combine (+ residual) for this CTA's rows, j ascending
            for (int v = tid - 32; v < B * nrows; v += 32 * kDkConsumers) {
                const int t = v / nrows, r = v - t * nrows;
                float a = 0.f;
                for (int j = 0; j < k; ++j)
                    a = fmaf(m->w[t * k + j], os[m->pos[t * k + j] * p.maxrows + r], a);
                const size_t gi = (size_t)t * H + h0 + r;
                if (p.residual) a = ld_act_f(p.residual + gi) + a;
                p.y[gi] = a;
                xs[t * H + h0 + r] = a;  // x_{l+1} rows for the next router
            }
            if (blockIdx.x == 0) {  // acc_now was read by every CTA before the last barrier
                for (int v = tid - 32; v < B * E; v += 32 * kDkConsumers) acc_now[v] = 0ull;
            }
            if (has_next) cp_async_wait_all();
            named_sync(1, 32 * kDkConsumers);
            // ---- router of layer l+1: partial dot products over this CTA's rows
            if (has_next && nrows > 0) {
                const float* bx = xs;
                for (int q = cw; q < B * E; q += kDkConsumers) {
                    const int t = q / E, e = q - t * E;
                    float part = 0.f;
                    for (int r = lane; r < nrows; r += 32)
                        part = fmaf(__uint_as_float((uint32_t)wrs[e * p.maxrows + r] << 16), bx[t * H + h0 + r], part);
                    part = warp_sum(part);
                    if (lane == 0) red_add_u64(acc_next + (size_t)t * E + e, float_to_fix(part));
                }
            }
            }  // ok
            if (has_next) cp_async_wait_all();
        }
        ring_pos += wk.n;
        __syncthreads();
        // every thread reads the same flag: nobody writes it between the two
        // barriers around this read
        const bool aborted = *(volatile int*)&m->abort_flag != 0;
        if (has_next && !aborted) dk_grid_sync(p, epoch, m, 0, kDkThreads);
        __syncthreads();
    }
    // leave only after this CTA's own copies in flight have landed (they all
    // have, unless a wait gave up)
    __syncthreads();
    if (warp == 0 && lane == 0) {
        const long long first = issued > p.S ? issued - p.S : 0;
        for (long long n = first; n < issued; ++n)
            mbar_wait(&full[(int)(n % p.S)], (uint32_t)((n / p.S) & 1), kDkWaitLimit);
    }
    __syncthreads();
}

}  // namespace moe
