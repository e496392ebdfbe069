// moe_phases.cuh -- the steps of one MoE layer as device functions over work
// items.  Each phase is written as "process item i" so that it runs either
// as its own kernel (one CTA per item) or inside the persistent fused kernel
// (items strided over a grid of one CTA per SM, device-wide barriers between
// phases).  All phases use kThreads = 256 threads per CTA.
#pragma once

#include "moe_common.cuh"
#include "moe_ptx.cuh"

namespace moe {

// =================================================================== router
// logits[t,e] = sum_h x[t,h] * W_r[e,h] (+ bias[e]).  ("MoE Performance
// Optimization Analysis", Batch Router Design: [B,H] -> [B,E] on the GPU.)
// Item = (8 experts, 8 tokens); one warp per expert row, x staged in shared
// memory in chunks of kRouterHC columns and reused by all 8 warps.
constexpr int kRouterTB = 8;
constexpr int kRouterHC = 1024;
constexpr size_t kRouterSmem = sizeof(float) * kRouterTB * kRouterHC;  // 32 KB

// Work items of the router: blocks of kRouterTB tokens x (kWarps * EPW)
// experts; a warp takes EPW experts (EPW > 1 for larger batches: the staged
// x of a column block is then read once for EPW experts).
__host__ __device__ __forceinline__ int router_items(const Ctx& c, int epw = 1) {
    return ceil_div(c.E, kWarps * epw) * ceil_div(c.B, kRouterTB);
}

// Stage x[tok[q]][hc, hc+hn) (q < nq) into dst[q*ld + ...] as fp32; rows
// nq..nfill-1 are zero-filled.  tok == nullptr means tok[q] = t0 + q.
__device__ __forceinline__ void stage_x(const Ctx& c, const int* tok, int t0, int nq, int nfill,
                                        int hc, int hn, float* dst, int ld) {
    const int vpr = hn >> 3;  // 8-element vectors per row
    for (int v = threadIdx.x; v < nfill * vpr; v += blockDim.x) {
        const int q = v / vpr, i = (v - q * vpr) << 3;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (q < nq) {
            const int t = tok ? tok[q] : t0 + q;
            const size_t off = (size_t)t * c.H + hc + i;
            if (c.x_bf16) {
                const uint4 u = ld_act_u4(static_cast<const uint16_t*>(c.x) + off);
                const float2 f0 = bf16x2_to_f2(u.x), f1 = bf16x2_to_f2(u.y);
                const float2 f2 = bf16x2_to_f2(u.z), f3 = bf16x2_to_f2(u.w);
                a = make_float4(f0.x, f0.y, f1.x, f1.y);
                b = make_float4(f2.x, f2.y, f3.x, f3.y);
            } else {
                const float* xp = static_cast<const float*>(c.x) + off;
                a = ld_act_f4(xp);
                b = ld_act_f4(xp + 4);
            }
        }
        float4* d = reinterpret_cast<float4*>(dst + (size_t)q * ld + i);
        d[0] = a;
        d[1] = b;
    }
}

template <int EPW = 1>
__device__ void router_item(const Ctx& c, int item, float* smem) {
    const int neb = ceil_div(c.E, kWarps * EPW);
    const int eb = item % neb, tb = item / neb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = (eb * kWarps + warp) * EPW;  // this warp's experts e0 .. e0 + EPW - 1
    const int t0 = tb * kRouterTB;
    const int nt = min(kRouterTB, c.B - t0);
    float2 acc[EPW][kRouterTB];
#pragma unroll
    for (int j = 0; j < EPW; ++j)
#pragma unroll
        for (int q = 0; q < kRouterTB; ++q) acc[j][q] = make_float2(0.f, 0.f);
    // this lane's weight vectors of a chunk (kRouterHC / 256 per expert), all
    // requested together: the first chunk's before x is staged, each next
    // chunk's as soon as the current one is computed, so that the weights'
    // memory round trip overlaps the staging of x instead of following it
    constexpr int kNV = kRouterHC / 256;
    uint4 wv[EPW][kNV];
    auto load_w = [&](int hc) {
        const int hn = min(kRouterHC, c.H - hc);
#pragma unroll
        for (int s = 0; s < kNV; ++s)
#pragma unroll
            for (int j = 0; j < EPW; ++j) {
                const int i = lane * 8 + 256 * s;
                wv[j][s] = (e0 + j < c.E && i < hn) ? ld_weight_v4(c.w.w_router + (size_t)(e0 + j) * c.H + hc + i)
                                                     : make_uint4(0u, 0u, 0u, 0u);
            }
    };
    if (e0 < c.E) load_w(0);
    for (int hc = 0; hc < c.H; hc += kRouterHC) {
        const int hn = min(kRouterHC, c.H - hc);
        __syncthreads();
        stage_x(c, nullptr, t0, nt, kRouterTB, hc, hn, smem, kRouterHC);
        __syncthreads();
        if (e0 < c.E) {
#pragma unroll
            for (int s = 0; s < kNV; ++s) {
                const int i = lane * 8 + 256 * s;
                if (i >= hn) break;
                float2 w[EPW][4];
#pragma unroll
                for (int j = 0; j < EPW; ++j) {
                    w[j][0] = bf16x2_to_f2(wv[j][s].x);
                    w[j][1] = bf16x2_to_f2(wv[j][s].y);
                    w[j][2] = bf16x2_to_f2(wv[j][s].z);
                    w[j][3] = bf16x2_to_f2(wv[j][s].w);
                }
#pragma unroll
                for (int q = 0; q < kRouterTB; ++q) {
                    const float4* xp = reinterpret_cast<const float4*>(smem + q * kRouterHC + i);
                    const float4 xa = xp[0], xb = xp[1];
#pragma unroll
                    for (int j = 0; j < EPW; ++j) {
                        acc[j][q] = ffma2(w[j][0], make_float2(xa.x, xa.y), acc[j][q]);
                        acc[j][q] = ffma2(w[j][1], make_float2(xa.z, xa.w), acc[j][q]);
                        acc[j][q] = ffma2(w[j][2], make_float2(xb.x, xb.y), acc[j][q]);
                        acc[j][q] = ffma2(w[j][3], make_float2(xb.z, xb.w), acc[j][q]);
                    }
                }
            }
            if (hc + kRouterHC < c.H) load_w(hc + kRouterHC);
        }
    }
#pragma unroll
    for (int j = 0; j < EPW; ++j) {
        const int e = e0 + j;
        if (e < c.E) {
            const float b = c.w.bias ? c.w.bias[e] : 0.f;
#pragma unroll
            for (int q = 0; q < kRouterTB; ++q) {
                const float v = warp_sum(acc[j][q].x + acc[j][q].y);
                if (lane == q && q < nt) c.logits[(size_t)(t0 + q) * c.E + e] = v + b;
            }
        }
    }
}

// ==================================================================== top-k
// p = softmax(logits[t,:]) in fp32; the k largest logits, descending, ties to
// the lower expert id; w_j = p_j / sum of the selected p.  ("MoE Performance
// Optimization Analysis", GPU Router Design: selection on the GPU.)
// One warp per token; lane l holds experts l, l+32, ... (E <= 256).
__host__ __device__ __forceinline__ int topk_items(const Ctx& c) { return ceil_div(c.B, kWarps); }

// Token t by the calling warp.
__device__ void topk_token(const Ctx& c, int t, int32_t* ids_out, float* w_out) {
    const int lane = threadIdx.x & 31;
    const float* l = c.logits + (size_t)t * c.E;
    float v[8];
    bool bad = false;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int e = lane + 32 * s;
        v[s] = e < c.E ? ld_act_f(l + e) : -INFINITY;
        if (e < c.E && !isfinite(v[s])) bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(c.status, MOE_DEV_NONFINITE);
    // each round: the largest logit by a warp max over order-preserving keys,
    // then the lowest expert id holding it by a warp min -- "logit
    // descending, ties to the lower id" (zeros made +0 first, so that -0 and
    // +0 tie as they compare equal; NaN logits, key 0, are never chosen)
    unsigned key[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const float z = v[s] + 0.0f;
        key[s] = (lane + 32 * s < c.E && !isnan(z)) ? order_key(z) : 0u;
    }
    unsigned taken = 0;
    float selv[MOE_MAX_TOPK];
    int seli[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        selv[j] = -INFINITY;
        seli[j] = 0;
        if (j < c.k) {
            unsigned kb = 0u;
            int ib = 0x7fffffff;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (!((taken >> s) & 1u) && key[s] > kb) {
                    kb = key[s];
                    ib = lane + 32 * s;
                }
            const unsigned km = __reduce_max_sync(0xffffffffu, kb);
            int bi = (int)__reduce_min_sync(0xffffffffu, (km != 0u && kb == km) ? (unsigned)ib : 0x7fffffffu);
            const float bv = km != 0u ? key_value(km) : -INFINITY;
            if (bi == 0x7fffffff) bi = 0;  // only with non-finite logits (flagged above)
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            selv[j] = bv;
            seli[j] = bi;
        }
    }
    const float m = selv[0];
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (lane + 32 * q < c.E) s += expf(v[q] - m);
    s = warp_sum(s);
    if (lane == 0) {
        float p[MOE_MAX_TOPK];
        float ssel = 0.f;
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK; ++j) {
            p[j] = 0.f;
            if (j < c.k) {
                p[j] = expf(selv[j] - m) / s;
                ssel += p[j];
            }
        }
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK; ++j) {
            if (j < c.k) {
                ids_out[(size_t)t * c.k + j] = seli[j];
                w_out[(size_t)t * c.k + j] = p[j] / ssel;
            }
        }
    }
}

__device__ void topk_item(const Ctx& c, int item, int32_t* ids_out, float* w_out) {
    const int t = item * kWarps + (threadIdx.x >> 5);
    if (t < c.B) topk_token(c, t, ids_out, w_out);
}

// ================================================================= grouping
// Stable counting sort of the flat routes r = t*k + j by expert id, in one
// CTA.  ("perf(cpu-moe): dedup experts across the batch in pass 1 - #46",
// commit message: group the routes by expert, counting sort over the ids.)
// A token selects an expert at most once, so the rank of route (t, j) inside
// expert e's group is the number of earlier tokens that chose e: a popcount
// over a per-expert token bitmap.  Deterministic, no atomics-ordered scatter.
__host__ __device__ __forceinline__ size_t group_smem_bytes(int B, int E) {
    const int W = (B + 31) / 32;
    return sizeof(uint32_t) * ((size_t)E * (W > 0 ? W : 1) + 2 * (size_t)E + 2);
}

__device__ void group_cta(const int32_t* ids, int B, int k, int E, int32_t* offsets,
                          int32_t* route_idx, int32_t* unique, int32_t* num_unique,
                          int32_t* status, uint32_t* smem) {
    const int W = (B + 31) / 32 > 0 ? (B + 31) / 32 : 1;
    uint32_t* bm = smem;                                  // [E][W]
    int* cnt = reinterpret_cast<int*>(bm + (size_t)E * W);  // [E]
    int* off = cnt + E;                                   // [E + 1]
    const int R = B * k;
    const int tid = threadIdx.x, nth = blockDim.x;
    for (int i = tid; i < E * W; i += nth) bm[i] = 0u;
    __syncthreads();
    for (int r = tid; r < R; r += nth) {
        const int e = ld_act_i(ids + r);
        const int t = r / k;
        if (e < 0 || e >= E) {
            set_status(status, MOE_DEV_BAD_EXPERT_ID);
            continue;
        }
        const uint32_t bit = 1u << (t & 31);
        const uint32_t old = atomicOr(&bm[e * W + (t >> 5)], bit);
        if (old & bit) set_status(status, MOE_DEV_DUP_EXPERT);
    }
    __syncthreads();
    for (int e = tid; e < E; e += nth) {
        int s = 0;
        for (int w = 0; w < W; ++w) s += __popc(bm[e * W + w]);
        cnt[e] = s;
    }
    __syncthreads();
    if (tid < 32) {  // warp 0: exclusive scans of the counts and of the nonzero flags
        const int lane = tid;
        int loc[8], locu[8], sum = 0, sumu = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            const int v = e < E ? cnt[e] : 0;
            loc[i] = sum;
            locu[i] = sumu;
            sum += v;
            sumu += v > 0 ? 1 : 0;
        }
        int inc = sum, incu = sumu;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, inc, d);
            const int b = __shfl_up_sync(0xffffffffu, incu, d);
            if (lane >= d) {
                inc += a;
                incu += b;
            }
        }
        const int ex = inc - sum, exu = incu - sumu;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            if (e < E) {
                off[e] = ex + loc[i];
                offsets[e] = ex + loc[i];
                if (cnt[e] > 0) unique[exu + locu[i]] = e;
            }
        }
        if (lane == 31) {
            off[E] = inc;
            offsets[E] = inc;
            *num_unique = incu;
        }
    }
    __syncthreads();
    for (int r = tid; r < R; r += nth) {
        const int e = ld_act_i(ids + r);
        if (e < 0 || e >= E) continue;
        const int t = r / k, w = t >> 5;
        int rank = __popc(bm[e * W + w] & ((1u << (t & 31)) - 1u));
        for (int ww = 0; ww < w; ++ww) rank += __popc(bm[e * W + ww]);
        route_idx[off[e] + rank] = r;
    }
}

// ================================================================ classify
// Split the segments into the CUDA-core list and the tensor-core list (one
// warp, order kept): a segment with at least tc_threshold routes goes to the
// tensor cores.  Writes c.seg_list / c.seg_count.
__device__ void classify_warp(const Ctx& c) {
    const int lane = threadIdx.x & 31;
    const int nseg = no_dedup(c) ? c.B * c.k : ld_act_i(c.num_unique);
    const int maxseg = max_segments(c);
    int ng = 0, nt = 0, nmax = 0;
    for (int base = 0; base < nseg; base += 32) {
        const int s = base + lane;
        bool valid = false, tc = false;
        if (s < nseg) {
            Seg sg;
            valid = get_seg(c, s, sg);
            tc = valid && c.tc_threshold > 0 && sg.p1 - sg.p0 >= c.tc_threshold;
            if (tc) nmax = max(nmax, sg.p1 - sg.p0);
        }
        const unsigned bt = __ballot_sync(0xffffffffu, tc);
        const unsigned bg = __ballot_sync(0xffffffffu, valid && !tc);
        const unsigned below = (1u << lane) - 1u;
        if (tc) c.seg_list[maxseg + nt + __popc(bt & below)] = s;
        if (valid && !tc) c.seg_list[ng + __popc(bg & below)] = s;
        nt += __popc(bt);
        ng += __popc(bg);
    }
    nmax = __reduce_max_sync(0xffffffffu, nmax);
    if (lane == 0) {
        c.seg_count[0] = ng;
        c.seg_count[1] = nt;
        c.seg_count[2] = nmax;  // routes of the largest tensor-core segment
    }
}

// ============================================================ gate_up + SiLU
// For each segment (expert e, its routes) and each gate/up row pair i:
//   h[p, i] = SiLU(G_e[i,:] . x_t) * (U_e[i,:] . x_t)   for every route p of e.
// ("perf(cpu-moe) ... #46": pass 1 reads gate_up [2I, H]; split by (unique
// expert, row block) with the expert's routes as the inner loop, so each
// weight row is read from memory once.)  Item = (segment, 8 row pairs); one
// warp per row pair streams both rows with 16-byte loads; the routes' x rows
// are staged in shared memory and the weights are reused from registers
// across up to nt_max tokens per pass.
constexpr int kGateUnroll = 4;

__host__ __device__ __forceinline__ int gateup_items(const Ctx& c) {
    return max_segments(c) * ceil_div(c.I, kWarps);
}


template <int NT>
__device__ __forceinline__ void gateup_rowpair(const uint16_t* grow, const uint16_t* urow, int H,
                                               const float* xs, int nq, float* hdst, int I) {
    const int lane = threadIdx.x & 31;
    float2 ag[NT], au[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) ag[q] = au[q] = make_float2(0.f, 0.f);
    for (int base = 0; base < H; base += 256 * kGateUnroll) {
        uint4 gv[kGateUnroll], uv[kGateUnroll];
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const int idx = base + u * 256 + lane * 8;
            if (idx < H) {
                gv[u] = ld_weight_v4(grow + idx);
                uv[u] = ld_weight_v4(urow + idx);
            } else {
                gv[u] = uv[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const int idx = base + u * 256 + lane * 8;
            if (idx < H) {
                const float2 g0 = bf16x2_to_f2(gv[u].x), g1 = bf16x2_to_f2(gv[u].y);
                const float2 g2 = bf16x2_to_f2(gv[u].z), g3 = bf16x2_to_f2(gv[u].w);
                const float2 u0 = bf16x2_to_f2(uv[u].x), u1 = bf16x2_to_f2(uv[u].y);
                const float2 u2 = bf16x2_to_f2(uv[u].z), u3 = bf16x2_to_f2(uv[u].w);
#pragma unroll
                for (int q = 0; q < NT; ++q) {
                    const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)q * H + idx);
                    const float4 xa = xp[0], xb = xp[1];
                    const float2 x0 = make_float2(xa.x, xa.y), x1 = make_float2(xa.z, xa.w);
                    const float2 x2 = make_float2(xb.x, xb.y), x3 = make_float2(xb.z, xb.w);
                    ag[q] = ffma2(g0, x0, ag[q]);
                    au[q] = ffma2(u0, x0, au[q]);
                    ag[q] = ffma2(g1, x1, ag[q]);
                    au[q] = ffma2(u1, x1, au[q]);
                    ag[q] = ffma2(g2, x2, ag[q]);
                    au[q] = ffma2(u2, x2, au[q]);
                    ag[q] = ffma2(g3, x3, ag[q]);
                    au[q] = ffma2(u3, x3, au[q]);
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        const float g = warp_sum(ag[q].x + ag[q].y);
        const float u = warp_sum(au[q].x + au[q].y);
        if (lane == q && q < nq) hdst[(size_t)q * I] = silu_mul(g, u);
    }
}

// The block-scaled FP8 form of gateup_rowpair: rows of H one-byte E4M3
// codes (H % 16 == 0) and their scales along the row (gsr for gate row i, usr
// for up row I + i: one fp32 per 128 columns).  A lane's 16 consecutive codes
// lie in one 128-column block, so their products are summed first and
// scaled once.
template <int NT>
__device__ __forceinline__ void gateup_rowpair_f8(const unsigned char* grow, const unsigned char* urow,
                                                  const float* gsr, const float* usr, int H, const float* xs,
                                                  int nq, float* hdst, int I) {
    const int lane = threadIdx.x & 31;
    float ag[NT], au[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) ag[q] = au[q] = 0.f;
    for (int base = 0; base < H; base += 512 * kGateUnroll) {  // as many bytes in flight as the bf16 loop
        uint4 gv[kGateUnroll], uv[kGateUnroll];
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const int idx = base + u * 512 + lane * 16;
            gv[u] = idx < H ? ld_weight_v4(grow + idx) : make_uint4(0u, 0u, 0u, 0u);
            uv[u] = idx < H ? ld_weight_v4(urow + idx) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const int idx = base + u * 512 + lane * 16;
            if (idx < H) {
                const float sg = __ldg(gsr + (idx >> 7)), su = __ldg(usr + (idx >> 7));
                const unsigned gw[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
                const unsigned uw[4] = {uv[u].x, uv[u].y, uv[u].z, uv[u].w};
#pragma unroll
                for (int q = 0; q < NT; ++q) {
                    const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)q * H + idx);
                    float2 pg = make_float2(0.f, 0.f), pu = make_float2(0.f, 0.f);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {  // codes 4v .. 4v+3 against x[idx + 4v ..]
                        const float4 xv = xp[v];
                        pg = ffma2(f8x2_to_f2(gw[v]), make_float2(xv.x, xv.y), pg);
                        pg = ffma2(f8x2_to_f2(gw[v] >> 16), make_float2(xv.z, xv.w), pg);
                        pu = ffma2(f8x2_to_f2(uw[v]), make_float2(xv.x, xv.y), pu);
                        pu = ffma2(f8x2_to_f2(uw[v] >> 16), make_float2(xv.z, xv.w), pu);
                    }
                    ag[q] = fmaf(sg, pg.x + pg.y, ag[q]);
                    au[q] = fmaf(su, pu.x + pu.y, au[q]);
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        const float g = warp_sum(ag[q]);
        const float u = warp_sum(au[q]);
        if (lane == q && q < nq) hdst[(size_t)q * I] = silu_mul(g, u);
    }
}

// The NVFP4 form of gateup_rowpair: rows of H E2M1 codes two to a byte (H %
// 32 == 0), the rows' E4M3 scales of 16-element blocks (gbs, ubs) and the
// matrix scale gs.  A lane takes 16 codes (8 bytes), one scale block: their
// products are summed first and scaled once.
template <int NT>
__device__ __forceinline__ void gateup_rowpair_f4(const unsigned char* grow, const unsigned char* urow,
                                                  const unsigned char* gbs, const unsigned char* ubs, float gs, int H,
                                                  const float* xs, int nq, float* hdst, int I) {
    const int lane = threadIdx.x & 31;
    float ag[NT], au[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) ag[q] = au[q] = 0.f;
    for (int base = 0; base < H; base += 512 * kGateUnroll) {
        uint2 gv[kGateUnroll], uv[kGateUnroll];
        unsigned gb[kGateUnroll], ub[kGateUnroll];
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const int idx = base + u * 512 + lane * 16;
            const bool in = idx < H;
            gv[u] = in ? __ldg(reinterpret_cast<const uint2*>(grow + (idx >> 1))) : make_uint2(0u, 0u);
            uv[u] = in ? __ldg(reinterpret_cast<const uint2*>(urow + (idx >> 1))) : make_uint2(0u, 0u);
            gb[u] = in ? __ldg(gbs + (idx >> 4)) : 0u;
            ub[u] = in ? __ldg(ubs + (idx >> 4)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const int idx = base + u * 512 + lane * 16;
            if (idx < H) {
                const float sg = f8_to_f(gb[u]) * gs, su = f8_to_f(ub[u]) * gs;
                const unsigned gw[2] = {gv[u].x, gv[u].y};
                const unsigned uw[2] = {uv[u].x, uv[u].y};
#pragma unroll
                for (int q = 0; q < NT; ++q) {
                    const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)q * H + idx);
                    float2 pg = make_float2(0.f, 0.f), pu = make_float2(0.f, 0.f);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {  // codes 4v .. 4v+3 (two bytes) against x[idx + 4v ..]
                        const float4 xv = xp[v];
                        const unsigned gbyte = gw[v >> 1] >> (16 * (v & 1)), ubyte = uw[v >> 1] >> (16 * (v & 1));
                        pg = ffma2(f4x2_to_f2(gbyte), make_float2(xv.x, xv.y), pg);
                        pg = ffma2(f4x2_to_f2(gbyte >> 8), make_float2(xv.z, xv.w), pg);
                        pu = ffma2(f4x2_to_f2(ubyte), make_float2(xv.x, xv.y), pu);
                        pu = ffma2(f4x2_to_f2(ubyte >> 8), make_float2(xv.z, xv.w), pu);
                    }
                    ag[q] = fmaf(sg, pg.x + pg.y, ag[q]);
                    au[q] = fmaf(su, pu.x + pu.y, au[q]);
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        const float g = warp_sum(ag[q]);
        const float u = warp_sum(au[q]);
        if (lane == q && q < nq) hdst[(size_t)q * I] = silu_mul(g, u);
    }
}

// xs: nt_max * H floats of shared memory; tok: nt_max ints of shared memory.
// Block-scaled FP8 weights when c.w.gate_up_scale is set (gate_up then holds
// E4M3 codes, one byte each), NVFP4 ones when c.w.gate_up_bs is set (E2M1
// codes two to a byte).
__device__ void gateup_item(const Ctx& c, int item, float* xs, int* tok) {
    const int nib = ceil_div(c.I, kWarps);
    const int sl = item / nib, ib = item - sl * nib;
    const int s = c.seg_list ? ld_act_i(c.seg_list + sl) : sl;
    Seg sg;
    if (!get_seg(c, s, sg)) return;  // uniform over the CTA
    if (c.tc_threshold > 0 && sg.p1 - sg.p0 >= c.tc_threshold) return;  // tensor-core path
    const int warp = threadIdx.x >> 5;
    const int i = ib * kWarps + warp;
    const uint16_t* G = c.w.gate_up + (size_t)sg.e * 2 * c.I * c.H;
    for (int g0 = sg.p0; g0 < sg.p1; g0 += c.nt_max) {
        const int nq = min(c.nt_max, sg.p1 - g0);
        __syncthreads();
        if (threadIdx.x < nq) tok[threadIdx.x] = route_at(c, g0 + threadIdx.x) / c.k;
        __syncthreads();
        const int nfill = nq <= 1 ? 1 : nq <= 2 ? 2 : nq <= 4 ? 4 : 8;
        stage_x(c, tok, 0, nq, nfill, 0, c.H, xs, c.H);
        __syncthreads();
        if (i < c.I && c.w.gate_up_bs) {
            const size_t rb = (size_t)c.H >> 1, sb = (size_t)c.H >> 4;  // bytes of a row of codes, of scales
            const unsigned char* G4 = reinterpret_cast<const unsigned char*>(c.w.gate_up) + (size_t)sg.e * 2 * c.I * rb;
            const unsigned char* S4 = c.w.gate_up_bs + (size_t)sg.e * 2 * c.I * sb;
            const float gs = __ldg(c.w.gate_up_gs + sg.e);
            const unsigned char* grow = G4 + (size_t)i * rb;
            const unsigned char* urow = G4 + (size_t)(c.I + i) * rb;
            const unsigned char* gbs = S4 + (size_t)i * sb;
            const unsigned char* ubs = S4 + (size_t)(c.I + i) * sb;
            float* hdst = c.h + (size_t)g0 * c.I + i;
            switch (nfill) {
                case 1: gateup_rowpair_f4<1>(grow, urow, gbs, ubs, gs, c.H, xs, nq, hdst, c.I); break;
                case 2: gateup_rowpair_f4<2>(grow, urow, gbs, ubs, gs, c.H, xs, nq, hdst, c.I); break;
                case 4: gateup_rowpair_f4<4>(grow, urow, gbs, ubs, gs, c.H, xs, nq, hdst, c.I); break;
                default: gateup_rowpair_f4<8>(grow, urow, gbs, ubs, gs, c.H, xs, nq, hdst, c.I); break;
            }
        } else if (i < c.I && c.w.gate_up_scale) {
            const unsigned char* G8 = reinterpret_cast<const unsigned char*>(c.w.gate_up) + (size_t)sg.e * 2 * c.I * c.H;
            const int sld = (c.H + 127) >> 7, se = ((2 * c.I + 127) >> 7) * sld;
            const float* gsr = c.w.gate_up_scale + (size_t)sg.e * se + (size_t)(i >> 7) * sld;
            const float* usr = c.w.gate_up_scale + (size_t)sg.e * se + (size_t)((c.I + i) >> 7) * sld;
            const unsigned char* grow = G8 + (size_t)i * c.H;
            const unsigned char* urow = G8 + (size_t)(c.I + i) * c.H;
            float* hdst = c.h + (size_t)g0 * c.I + i;
            switch (nfill) {
                case 1: gateup_rowpair_f8<1>(grow, urow, gsr, usr, c.H, xs, nq, hdst, c.I); break;
                case 2: gateup_rowpair_f8<2>(grow, urow, gsr, usr, c.H, xs, nq, hdst, c.I); break;
                case 4: gateup_rowpair_f8<4>(grow, urow, gsr, usr, c.H, xs, nq, hdst, c.I); break;
                default: gateup_rowpair_f8<8>(grow, urow, gsr, usr, c.H, xs, nq, hdst, c.I); break;
            }
        } else if (i < c.I) {
            const uint16_t* grow = G + (size_t)i * c.H;
            const uint16_t* urow = G + (size_t)(c.I + i) * c.H;
            float* hdst = c.h + (size_t)g0 * c.I + i;
            switch (nfill) {
                case 1: gateup_rowpair<1>(grow, urow, c.H, xs, nq, hdst, c.I); break;
                case 2: gateup_rowpair<2>(grow, urow, c.H, xs, nq, hdst, c.I); break;
                case 4: gateup_rowpair<4>(grow, urow, c.H, xs, nq, hdst, c.I); break;
                default: gateup_rowpair<8>(grow, urow, c.H, xs, nq, hdst, c.I); break;
            }
        }
    }
}

// ===================================================================== down
// o[r, j] = D_e[j,:] . h[p,:] for every route p (flat index r) of the segment.
// ("perf(cpu-moe) ... #46": pass 2 reads down [H, I].)  Item = (segment,
// 32 rows of D_e); one warp streams 4 rows; the segment's h rows are staged
// in shared memory.
constexpr int kDownRowsPerWarp = 4;
constexpr int kDownRows = kWarps * kDownRowsPerWarp;
constexpr int kDownUnroll = 2;

__host__ __device__ __forceinline__ int down_items(const Ctx& c) {
    return max_segments(c) * ceil_div(c.H, kDownRows);
}

template <int NT>
__device__ __forceinline__ void down_rows(const uint16_t* D, int row0, int H, int I, const float* hs,
                                          const int* rts, int nq, float* o) {
    const int lane = threadIdx.x & 31;
    float2 acc[kDownRowsPerWarp][NT];
#pragma unroll
    for (int rr = 0; rr < kDownRowsPerWarp; ++rr)
#pragma unroll
        for (int q = 0; q < NT; ++q) acc[rr][q] = make_float2(0.f, 0.f);
    for (int base = 0; base < I; base += 256 * kDownUnroll) {
        uint4 wv[kDownRowsPerWarp][kDownUnroll];
#pragma unroll
        for (int rr = 0; rr < kDownRowsPerWarp; ++rr)
#pragma unroll
            for (int u = 0; u < kDownUnroll; ++u) {
                const int idx = base + u * 256 + lane * 8;
                const int row = row0 + rr;
                wv[rr][u] = (idx < I && row < H) ? ld_weight_v4(D + (size_t)row * I + idx)
                                                 : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
        for (int u = 0; u < kDownUnroll; ++u) {
            const int idx = base + u * 256 + lane * 8;
            if (idx < I) {
#pragma unroll
                for (int q = 0; q < NT; ++q) {
                    const float4* hp = reinterpret_cast<const float4*>(hs + (size_t)q * I + idx);
                    const float4 ha = hp[0], hb = hp[1];
                    const float2 h0 = make_float2(ha.x, ha.y), h1 = make_float2(ha.z, ha.w);
                    const float2 h2 = make_float2(hb.x, hb.y), h3 = make_float2(hb.z, hb.w);
#pragma unroll
                    for (int rr = 0; rr < kDownRowsPerWarp; ++rr) {
                        acc[rr][q] = ffma2(bf16x2_to_f2(wv[rr][u].x), h0, acc[rr][q]);
                        acc[rr][q] = ffma2(bf16x2_to_f2(wv[rr][u].y), h1, acc[rr][q]);
                        acc[rr][q] = ffma2(bf16x2_to_f2(wv[rr][u].z), h2, acc[rr][q]);
                        acc[rr][q] = ffma2(bf16x2_to_f2(wv[rr][u].w), h3, acc[rr][q]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kDownRowsPerWarp; ++rr)
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            const float v = warp_sum(acc[rr][q].x + acc[rr][q].y);
            const int row = row0 + rr;
            if (lane == ((rr * NT + q) & 31) && q < nq && row < H) o[(size_t)rts[q] * H + row] = v;
        }
}

// The block-scaled FP8 form of down_rows: rows of I E4M3 codes (I % 16 ==
// 0), the expert's scales dsc [ceil(H/128)][dsc_ld]; a lane's 16 codes lie
// in one 128-column block and are scaled once.
template <int NT>
__device__ __forceinline__ void down_rows_f8(const unsigned char* D, const float* dsc, int dsc_ld, int row0, int H,
                                             int I, const float* hs, const int* rts, int nq, float* o) {
    const int lane = threadIdx.x & 31;
    float acc[kDownRowsPerWarp][NT];
#pragma unroll
    for (int rr = 0; rr < kDownRowsPerWarp; ++rr)
#pragma unroll
        for (int q = 0; q < NT; ++q) acc[rr][q] = 0.f;
    for (int base0 = 0; base0 < I; base0 += 512 * kDownUnroll) {  // as many bytes in flight as the bf16 loop
        uint4 wvu[kDownUnroll][kDownRowsPerWarp];
        float scu[kDownUnroll][kDownRowsPerWarp];
#pragma unroll
        for (int u = 0; u < kDownUnroll; ++u)
#pragma unroll
            for (int rr = 0; rr < kDownRowsPerWarp; ++rr) {
                const int row = row0 + rr, idx = base0 + u * 512 + lane * 16;
                const bool in = row < H && idx < I;
                wvu[u][rr] = in ? ld_weight_v4(D + (size_t)row * I + idx) : make_uint4(0u, 0u, 0u, 0u);
                scu[u][rr] = in ? __ldg(dsc + (size_t)(row >> 7) * dsc_ld + (idx >> 7)) : 0.f;
            }
#pragma unroll
        for (int u = 0; u < kDownUnroll; ++u) {
        const int idx = base0 + u * 512 + lane * 16;
        if (idx >= I) continue;
        const uint4* wv = wvu[u];
        const float* sc = scu[u];
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            const float4* hp = reinterpret_cast<const float4*>(hs + (size_t)q * I + idx);
            const float4 h0 = hp[0], h1 = hp[1], h2 = hp[2], h3 = hp[3];
#pragma unroll
            for (int rr = 0; rr < kDownRowsPerWarp; ++rr) {
                float2 a = ffma2(f8x2_to_f2(wv[rr].x), make_float2(h0.x, h0.y), make_float2(0.f, 0.f));
                a = ffma2(f8x2_to_f2(wv[rr].x >> 16), make_float2(h0.z, h0.w), a);
                a = ffma2(f8x2_to_f2(wv[rr].y), make_float2(h1.x, h1.y), a);
                a = ffma2(f8x2_to_f2(wv[rr].y >> 16), make_float2(h1.z, h1.w), a);
                a = ffma2(f8x2_to_f2(wv[rr].z), make_float2(h2.x, h2.y), a);
                a = ffma2(f8x2_to_f2(wv[rr].z >> 16), make_float2(h2.z, h2.w), a);
                a = ffma2(f8x2_to_f2(wv[rr].w), make_float2(h3.x, h3.y), a);
                a = ffma2(f8x2_to_f2(wv[rr].w >> 16), make_float2(h3.z, h3.w), a);
                acc[rr][q] = fmaf(sc[rr], a.x + a.y, acc[rr][q]);
            }
        }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kDownRowsPerWarp; ++rr)
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            const float v = warp_sum(acc[rr][q]);
            const int row = row0 + rr;
            if (lane == ((rr * NT + q) & 31) && q < nq && row < H) o[(size_t)rts[q] * H + row] = v;
        }
}

// The NVFP4 form of down_rows: rows of I E2M1 codes two to a byte (I % 32 ==
// 0), row r's E4M3 block scales at dbs + r * I/16, matrix scale gs.
template <int NT>
__device__ __forceinline__ void down_rows_f4(const unsigned char* D, const unsigned char* dbs, float gs, int row0,
                                             int H, int I, const float* hs, const int* rts, int nq, float* o) {
    const int lane = threadIdx.x & 31;
    const size_t rb = (size_t)I >> 1, sb = (size_t)I >> 4;
    float acc[kDownRowsPerWarp][NT];
#pragma unroll
    for (int rr = 0; rr < kDownRowsPerWarp; ++rr)
#pragma unroll
        for (int q = 0; q < NT; ++q) acc[rr][q] = 0.f;
    for (int base0 = 0; base0 < I; base0 += 512 * kDownUnroll) {
        uint2 wvu[kDownUnroll][kDownRowsPerWarp];
        float scu[kDownUnroll][kDownRowsPerWarp];
#pragma unroll
        for (int u = 0; u < kDownUnroll; ++u)
#pragma unroll
            for (int rr = 0; rr < kDownRowsPerWarp; ++rr) {
                const int row = row0 + rr, idx = base0 + u * 512 + lane * 16;
                const bool in = row < H && idx < I;
                wvu[u][rr] = in ? __ldg(reinterpret_cast<const uint2*>(D + (size_t)row * rb + (idx >> 1)))
                                : make_uint2(0u, 0u);
                scu[u][rr] = in ? f8_to_f(__ldg(dbs + (size_t)row * sb + (idx >> 4))) * gs : 0.f;
            }
#pragma unroll
        for (int u = 0; u < kDownUnroll; ++u) {
            const int idx = base0 + u * 512 + lane * 16;
            if (idx >= I) continue;
#pragma unroll
            for (int q = 0; q < NT; ++q) {
                const float4* hp = reinterpret_cast<const float4*>(hs + (size_t)q * I + idx);
                const float4 h0 = hp[0], h1 = hp[1], h2 = hp[2], h3 = hp[3];
                const float4 hv[4] = {h0, h1, h2, h3};
#pragma unroll
                for (int rr = 0; rr < kDownRowsPerWarp; ++rr) {
                    const unsigned w[2] = {wvu[u][rr].x, wvu[u][rr].y};
                    float2 a = make_float2(0.f, 0.f);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const unsigned byte2 = w[v >> 1] >> (16 * (v & 1));
                        a = ffma2(f4x2_to_f2(byte2), make_float2(hv[v].x, hv[v].y), a);
                        a = ffma2(f4x2_to_f2(byte2 >> 8), make_float2(hv[v].z, hv[v].w), a);
                    }
                    acc[rr][q] = fmaf(scu[u][rr], a.x + a.y, acc[rr][q]);
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kDownRowsPerWarp; ++rr)
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            const float v = warp_sum(acc[rr][q]);
            const int row = row0 + rr;
            if (lane == ((rr * NT + q) & 31) && q < nq && row < H) o[(size_t)rts[q] * H + row] = v;
        }
}

// hs: nt_max * I floats of shared memory; rts: nt_max ints of shared memory.
// Block-scaled FP8 weights when c.w.down_scale is set, NVFP4 ones when
// c.w.down_bs is.
__device__ void down_item(const Ctx& c, int item, float* hs, int* rts) {
    const int nrb = ceil_div(c.H, kDownRows);
    const int sl = item / nrb, rb = item - sl * nrb;
    const int s = c.seg_list ? ld_act_i(c.seg_list + sl) : sl;
    Seg sg;
    if (!get_seg(c, s, sg)) return;
    if (c.tc_threshold > 0 && sg.p1 - sg.p0 >= c.tc_threshold) return;  // tensor-core path
    const int warp = threadIdx.x >> 5;
    const int row0 = rb * kDownRows + warp * kDownRowsPerWarp;
    const uint16_t* D = c.w.down + (size_t)sg.e * c.H * c.I;
    for (int g0 = sg.p0; g0 < sg.p1; g0 += c.nt_max) {
        const int nq = min(c.nt_max, sg.p1 - g0);
        const int nfill = nq <= 1 ? 1 : nq <= 2 ? 2 : nq <= 4 ? 4 : 8;
        __syncthreads();
        if (threadIdx.x < nq) rts[threadIdx.x] = route_at(c, g0 + threadIdx.x);
        const int vpr = c.I >> 2;
        for (int v = threadIdx.x; v < nfill * vpr; v += blockDim.x) {
            const int q = v / vpr, i = (v - q * vpr) << 2;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (q < nq) val = ld_act_f4(c.h + (size_t)(g0 + q) * c.I + i);
            *reinterpret_cast<float4*>(hs + (size_t)q * c.I + i) = val;
        }
        __syncthreads();
        if (row0 < c.H && c.w.down_bs) {
            const unsigned char* D4 = reinterpret_cast<const unsigned char*>(c.w.down) + (size_t)sg.e * c.H * (c.I >> 1);
            const unsigned char* S4 = c.w.down_bs + (size_t)sg.e * c.H * (c.I >> 4);
            const float gs = __ldg(c.w.down_gs + sg.e);
            switch (nfill) {
                case 1: down_rows_f4<1>(D4, S4, gs, row0, c.H, c.I, hs, rts, nq, c.o); break;
                case 2: down_rows_f4<2>(D4, S4, gs, row0, c.H, c.I, hs, rts, nq, c.o); break;
                case 4: down_rows_f4<4>(D4, S4, gs, row0, c.H, c.I, hs, rts, nq, c.o); break;
                default: down_rows_f4<8>(D4, S4, gs, row0, c.H, c.I, hs, rts, nq, c.o); break;
            }
        } else if (row0 < c.H && c.w.down_scale) {
            const unsigned char* D8 = reinterpret_cast<const unsigned char*>(c.w.down) + (size_t)sg.e * c.H * c.I;
            const int sld = (c.I + 127) >> 7;
            const float* dsc = c.w.down_scale + (size_t)sg.e * ((c.H + 127) >> 7) * sld;
            switch (nfill) {
                case 1: down_rows_f8<1>(D8, dsc, sld, row0, c.H, c.I, hs, rts, nq, c.o); break;
                case 2: down_rows_f8<2>(D8, dsc, sld, row0, c.H, c.I, hs, rts, nq, c.o); break;
                case 4: down_rows_f8<4>(D8, dsc, sld, row0, c.H, c.I, hs, rts, nq, c.o); break;
                default: down_rows_f8<8>(D8, dsc, sld, row0, c.H, c.I, hs, rts, nq, c.o); break;
            }
        } else if (row0 < c.H) {
            switch (nfill) {
                case 1: down_rows<1>(D, row0, c.H, c.I, hs, rts, nq, c.o); break;
                case 2: down_rows<2>(D, row0, c.H, c.I, hs, rts, nq, c.o); break;
                case 4: down_rows<4>(D, row0, c.H, c.I, hs, rts, nq, c.o); break;
                default: down_rows<8>(D, row0, c.H, c.I, hs, rts, nq, c.o); break;
            }
        }
    }
}

// ================================================================== combine
// y[t, :] = sum_j w[t,j] * o[t*k + j, :]  (j ascending)  (+ residual[t, :]).
// ("MoE Performance Optimization Analysis", GPU Router Design: combination
// on the GPU.)  Item = 256 consecutive float4 of y, one per thread, so that
// even a small batch spreads over many SMs and each thread's k loads are in
// flight together.
constexpr int kCombineVecs = kThreads;

__host__ __device__ __forceinline__ int combine_items(const Ctx& c) {
    return ceil_div(c.B * (c.H >> 2), kCombineVecs);
}

__device__ void combine_item(const Ctx& c, int item) {
    const int nv = c.B * (c.H >> 2);
    const int hv = c.H >> 2;
    for (int v = item * kCombineVecs + threadIdx.x; v < min(nv, (item + 1) * kCombineVecs);
         v += blockDim.x) {
        const int t = v / hv, col = (v - t * hv) << 2;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < c.k; ++j) {
            const int r = t * c.k + j;
            const float wj = ld_act_f(c.rw + r);
            const float4 ov = ld_act_f4(c.o + (size_t)r * c.H + col);
            acc.x = fmaf(wj, ov.x, acc.x);
            acc.y = fmaf(wj, ov.y, acc.y);
            acc.z = fmaf(wj, ov.z, acc.z);
            acc.w = fmaf(wj, ov.w, acc.w);
        }
        if (c.residual) {
            const float4 rv = ld_act_f4(c.residual + (size_t)t * c.H + col);
            acc.x = rv.x + acc.x;
            acc.y = rv.y + acc.y;
            acc.z = rv.z + acc.z;
            acc.w = rv.w + acc.w;
        }
        *reinterpret_cast<float4*>(c.y + (size_t)t * c.H + col) = acc;
    }
}

// ================================================================ RMSNorm
// a[t,:] = (x[t,:] * rn) * g, rn = 1/sqrt(mean(x[t,:]^2) + eps), fp32; one
// CTA per token.  ("TEXT Generation Optimization Report", Fused Operations:
// norm + residual add -- the norm of a pre-norm layer's input; the residual
// add happens in the layer's combine.)
__global__ void __launch_bounds__(kThreads) rmsnorm_kernel(const float* x, const float* g, int H, float eps,
                                                           float* a) {
    __shared__ float part[kWarps];
    grid_dep_wait();
    const int t = blockIdx.x;
    const float* xr = x + (size_t)t * H;
    float ss = 0.f;
    for (int h = threadIdx.x; h < H; h += blockDim.x) ss = fmaf(xr[h], xr[h], ss);
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += part[w];
    const float rn = 1.0f / sqrtf(tot / (float)H + eps);
    for (int h = threadIdx.x; h < H; h += blockDim.x) a[(size_t)t * H + h] = (xr[h] * rn) * g[h];
}

}  // namespace moe
