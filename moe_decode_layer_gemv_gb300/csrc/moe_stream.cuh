// moe_stream.cuh -- the grouped GEMV passes for experts with few routes
// (fewer than MOE_TC_MIN_ROUTES) as persistent streaming kernels, one per
// pass: gate/up + SiLU (x -> h) and down (h -> o).
//
// ("perf(cpu-moe): dedupe expert weight reads", passes 1 and 2 over the
// unique experts: every weight byte of a selected expert is read once and
// applied to all of that expert's routes.)  The work is a list of items,
// item = (segment, block of weight rows), numbered segment-major over the
// CUDA-core segment list that classify_kernel builds on the device; CTA c
// takes the contiguous range [c*N/G, (c+1)*N/G).  One producer warp streams
// each item's rows into a ring of shared-memory stages with bulk copies
// (lane s owns stage s and arms it strictly in sequence); consumer warp
// (j mod W) computes item j of the CTA from its stage (S is a multiple of W,
// so a stage is always consumed by the same warp, in order).  The
// activation rows of the current segment (x of its tokens, or h of its
// routes) are staged in shared memory when the segment changes.  HBM bound:
// the producer keeps S stages of weight rows in flight while the consumers
// compute, instead of one round trip per item.
#pragma once

#include "moe_common.cuh"
#include "moe_ptx.cuh"

namespace moe {

constexpr int kSgConsumers = 8;
constexpr int kSgThreads = 32 * (1 + kSgConsumers);
constexpr int kSgMaxStages = 32;
constexpr int kSgMaxTok = MOE_TC_MIN_ROUTES - 1;  // routes of a CUDA-core segment
constexpr uint32_t kSgWaitLimit = 1u << 22;
constexpr int kSgStageTarget = 16 * 1024;  // bytes of weight rows per item

struct SgParams {
    Ctx c;
    int gate;         // 1: gate/up + SiLU (x -> h); 0: down (h -> o)
    int rpi;          // rows per item: gate/up pairs (gate) or down rows (down)
    int ips;          // items per segment: ceil(I / rpi) or ceil(H / rpi)
    int dim;          // activation length: H (gate) or I (down)
    int S, W;         // ring stages, consuming warps (S % W == 0)
    int stage_bytes;  // bytes of one stage
    int off_act, off_ring;
};

// shared-memory header of the streaming kernels
struct __align__(16) SgMisc {
    uint64_t full[kSgMaxStages];
    uint64_t empty[kSgMaxStages];
    int abort_flag;
    int nq;                // routes of the staged segment (0: none or invalid)
    int p0;                // its first position in the grouped route list
    int rts[kSgMaxTok];    // flat route index of each of its routes
};

// bounded wait on a ring barrier; on a timeout the CTA records it and stops
__device__ __forceinline__ bool sg_wait(uint64_t* bar, uint32_t parity, SgMisc* m, int32_t* status) {
    for (uint32_t i = 0; i < kSgWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 31u && *(volatile int*)&m->abort_flag) return false;
    }
    set_status(status, MOE_DEV_TIMEOUT);
    *(volatile int*)&m->abort_flag = 1;
    return false;
}

// Four weight rows in shared memory (r0..r3, n of them valid, each n_cols
// bf16) against NQ activation rows in the lane-blocked layout (act + q*ld):
// d[j*NQ + q] = row j . act row q, summed over the warp.  The activation
// vector of a column group is loaded once for all four rows.
template <int NQ>
__device__ __forceinline__ void sg_rows4(const unsigned char* r0, const unsigned char* r1, const unsigned char* r2,
                                         const unsigned char* r3, int n, const float* act, int ld, int n_cols,
                                         float (&d)[4 * NQ]) {
    const int lane = threadIdx.x & 31;
    float2 acc[4][NQ];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < NQ; ++q) acc[j][q] = make_float2(0.f, 0.f);
    const unsigned char* rows[4] = {r0, r1, r2, r3};
    const int nv = n_cols >> 3;
#pragma unroll 2
    for (int v = lane; v < nv; v += 32) {
        uint4 wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            wv[j] = j < n ? *reinterpret_cast<const uint4*>(rows[j] + 16 * v) : make_uint4(0u, 0u, 0u, 0u);
        const int g = lb_group(v);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const float4 xa = *reinterpret_cast<const float4*>(act + (size_t)q * ld + g);
            const float4 xb = *reinterpret_cast<const float4*>(act + (size_t)q * ld + g + 128);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[j][q] = ffma2(bf16x2_to_f2(wv[j].x), make_float2(xa.x, xa.y), acc[j][q]);
                acc[j][q] = ffma2(bf16x2_to_f2(wv[j].y), make_float2(xa.z, xa.w), acc[j][q]);
                acc[j][q] = ffma2(bf16x2_to_f2(wv[j].z), make_float2(xb.x, xb.y), acc[j][q]);
                acc[j][q] = ffma2(bf16x2_to_f2(wv[j].w), make_float2(xb.z, xb.w), acc[j][q]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < NQ; ++q) d[j * NQ + q] = acc[j][q].x + acc[j][q].y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int j = 0; j < 4 * NQ; ++j) d[j] += __shfl_xor_sync(0xffffffffu, d[j], off);
}

// lane L < 4*NQ picks d[L]
template <int NQ>
__device__ __forceinline__ float sg_pick(const float (&d)[4 * NQ]) {
    const int lane = threadIdx.x & 31;
    float v = d[0];
#pragma unroll
    for (int x = 1; x < 4 * NQ; ++x)
        if (lane == x) v = d[x];
    return v;
}

// Gate/up item: pairs [i0, i0 + np) of the staged segment (gate rows at st,
// up rows at st + np*2H), two pairs per pass, routes q0 .. q0 + NQ - 1 of
// the segment; h[(p0 + q)*I + i] = SiLU(g)*u.
template <int NQ>
__device__ __forceinline__ void sg_gate_item(const SgParams& P, const SgMisc* m, const unsigned char* st, int np, int i0,
                                             const float* act, int ld, int q0) {
    const int lane = threadIdx.x & 31;
    const int H = P.c.H, I = P.c.I;
    const unsigned char* up = st + (size_t)np * 2 * H;
    for (int pi = 0; pi < np; pi += 2) {
        const int n2 = min(2, np - pi);
        float d[4 * NQ];
        // rows: gate pi, up pi, gate pi+1, up pi+1
        sg_rows4<NQ>(st + (size_t)pi * 2 * H, up + (size_t)pi * 2 * H, st + (size_t)(pi + 1) * 2 * H,
                     up + (size_t)(pi + 1) * 2 * H, 2 * n2, act + (size_t)q0 * ld, ld, H, d);
        // lane q (< NQ) and lane 2NQ + q hold gate sums of pairs pi and pi+1; the
        // up sums sit NQ lanes above them
        const float v = sg_pick<NQ>(d);
        const float u = __shfl_down_sync(0xffffffffu, v, NQ);
        const int j = lane / NQ, q = lane - j * NQ;
        if (lane < 4 * NQ && (j & 1) == 0 && (j >> 1) < n2)
            P.c.h[(size_t)(m->p0 + q0 + q) * I + i0 + pi + (j >> 1)] = silu_mul(v, u);
    }
}

// Down item: rows [r0, r0 + nr) of the segment's expert, four per pass;
// o[route*H + row].
template <int NQ>
__device__ __forceinline__ void sg_down_item(const SgParams& P, const SgMisc* m, const unsigned char* st, int nr, int r0,
                                             const float* act, int ld, int q0) {
    const int lane = threadIdx.x & 31;
    const int H = P.c.H, I = P.c.I;
    for (int rb = 0; rb < nr; rb += 4) {
        const int n4 = min(4, nr - rb);
        const unsigned char* rw = st + (size_t)rb * 2 * I;
        float d[4 * NQ];
        sg_rows4<NQ>(rw, rw + 2 * I, rw + 4 * I, rw + 6 * I, n4, act + (size_t)q0 * ld, ld, I, d);
        const float v = sg_pick<NQ>(d);
        const int j = lane / NQ, q = lane - j * NQ;
        if (lane < 4 * NQ && j < n4) P.c.o[(size_t)m->rts[q0 + q] * H + r0 + rb + j] = v;
    }
}

__global__ void __launch_bounds__(kSgThreads, 1) stream_gemv_kernel(const SgParams P) {
    extern __shared__ __align__(128) unsigned char smem[];
    SgMisc* m = reinterpret_cast<SgMisc*>(smem);
    float* act = reinterpret_cast<float*>(smem + P.off_act);  // [kSgMaxTok][lb_stride(dim)] lane-blocked
    unsigned char* ring = smem + P.off_ring;
    const Ctx& c = P.c;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    grid_dep_wait();
    const int nseg = ld_act_i(c.seg_count);  // CUDA-core segments
    const long long N = (long long)nseg * P.ips;
    const int ja = (int)(N * cta / G), jb = (int)(N * (cta + 1) / G);
    const int nloc = jb - ja;
    if (tid == 0) {
        for (int s = 0; s < P.S; ++s) {
            mbar_init(&m->full[s], 1);
            mbar_init(&m->empty[s], 1);
        }
        m->abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (nloc <= 0) return;
    const int S = P.S, W = P.W;

    if (warp == 0) {
        // ================= producer: lane s issues the items of stage s in order
        // (MOE_F_HOT_L2: these experts have few routes this step; their
        // weights are streamed with evict_first so that they do not push the
        // tensor-core experts' weights out of L2)
        const bool cold = (c.flags & MOE_F_HOT_L2) != 0;
        const uint64_t pol = cold ? l2_policy_evict_first() : 0ull;
        const int s = lane;
        int cur = -1;
        Seg sg;
        bool ok = false;
        for (int jj = s; s < S && jj < nloc; jj += S) {
            const int j = ja + jj, si = j / P.ips, b = j - si * P.ips;
            if (si != cur) {
                cur = si;
                ok = get_seg(c, ld_act_i(c.seg_list + si), sg);
            }
            if (jj >= S && !sg_wait(&m->empty[s], (uint32_t)((jj / S - 1) & 1), m, c.status)) break;
            unsigned char* dst = ring + (size_t)s * P.stage_bytes;
            if (!ok) {
                mbar_arrive(&m->full[s]);  // nothing to fetch: the phase completes at once
            } else if (P.gate) {
                const int i0 = b * P.rpi, np = min(P.rpi, c.I - i0);
                const uint16_t* Gm = c.w.gate_up + (size_t)sg.e * 2 * c.I * c.H;
                const uint32_t bytes = (uint32_t)np * 2u * c.H;
                mbar_arrive_expect_tx(&m->full[s], 2u * bytes);
                if (cold) {
                    bulk_g2s_hint(dst, Gm + (size_t)i0 * c.H, bytes, &m->full[s], pol);
                    bulk_g2s_hint(dst + bytes, Gm + (size_t)(c.I + i0) * c.H, bytes, &m->full[s], pol);
                } else {
                    bulk_g2s(dst, Gm + (size_t)i0 * c.H, bytes, &m->full[s]);
                    bulk_g2s(dst + bytes, Gm + (size_t)(c.I + i0) * c.H, bytes, &m->full[s]);
                }
            } else {
                const int r0 = b * P.rpi, nr = min(P.rpi, c.H - r0);
                const uint32_t bytes = (uint32_t)nr * 2u * c.I;
                mbar_arrive_expect_tx(&m->full[s], bytes);
                const uint16_t* src = c.w.down + (size_t)sg.e * c.H * c.I + (size_t)r0 * c.I;
                if (cold)
                    bulk_g2s_hint(dst, src, bytes, &m->full[s], pol);
                else
                    bulk_g2s(dst, src, bytes, &m->full[s]);
            }
        }
        // before leaving: the last phase armed in this lane's stage has landed
        // (it has, unless a wait gave up)
        if (s < S && s < nloc) {
            const int last = s + ((nloc - 1 - s) / S) * S;
            mbar_wait(&m->full[s], (uint32_t)((last / S) & 1), kSgWaitLimit);
        }
        return;
    }

    // ================= consumers
    const int cw = warp - 1, ct = tid - 32, nct = 32 * kSgConsumers;
    const int sa = ja / P.ips, sb = (jb - 1) / P.ips;
    for (int si = sa; si <= sb; ++si) {
        const int j0 = max(ja, si * P.ips), j1 = min(jb, (si + 1) * P.ips);
        // ---- the segment's activation rows (every consumer warp is done
        // with the previous segment's rows after the first barrier)
        named_sync(1, nct);
        if (ct == 0) {
            Seg sg;
            int nq = 0;
            if (get_seg(c, ld_act_i(c.seg_list + si), sg)) {
                nq = sg.p1 - sg.p0;
                if (nq > kSgMaxTok) nq = 0;  // never: those segments take the tensor-core path
            }
            m->nq = nq;
            m->p0 = sg.p0;
        }
        named_sync(1, nct);
        const int nq = m->nq, p0 = m->p0;
        if (ct < nq) m->rts[ct] = route_at(c, p0 + ct);
        named_sync(1, nct);
        const int dim = P.dim, vpr = dim >> 2, ld = lb_stride(dim);
        for (int v = ct; v < nq * vpr; v += nct) {
            const int q = v / vpr, i = (v - q * vpr) << 2;
            float4 a;
            if (P.gate) {
                const size_t off = (size_t)(m->rts[q] / c.k) * c.H + i;
                if (c.x_bf16) {
                    const uint2 u = __ldcg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(c.x) + off));
                    const float2 lo = bf16x2_to_f2(u.x), hi = bf16x2_to_f2(u.y);
                    a = make_float4(lo.x, lo.y, hi.x, hi.y);
                } else {
                    a = ld_act_f4(static_cast<const float*>(c.x) + off);
                }
            } else {
                a = ld_act_f4(c.h + (size_t)(p0 + q) * c.I + i);
            }
            *reinterpret_cast<float4*>(act + (size_t)q * ld + lb_index(i)) = a;
        }
        named_sync(1, nct);
        // ---- this warp's items of the segment: local index jj = j - ja with
        // jj mod W == cw, stage jj mod S
        if (cw >= W) continue;
        int j = j0 + (((cw - (j0 - ja)) % W) + W) % W;
        for (; j < j1; j += W) {
            const int jj = j - ja, s = jj % S;
            if (!sg_wait(&m->full[s], (uint32_t)((jj / S) & 1), m, c.status)) break;
            const unsigned char* st = ring + (size_t)s * P.stage_bytes;
            const int b = j - si * P.ips;
            for (int q0 = 0; q0 < nq; q0 += 4) {
                const int n = min(4, nq - q0);
                if (P.gate) {
                    const int i0 = b * P.rpi, np = min(P.rpi, c.I - i0);
                    switch (n) {
                        case 1: sg_gate_item<1>(P, m, st, np, i0, act, ld, q0); break;
                        case 2: sg_gate_item<2>(P, m, st, np, i0, act, ld, q0); break;
                        case 3: sg_gate_item<3>(P, m, st, np, i0, act, ld, q0); break;
                        default: sg_gate_item<4>(P, m, st, np, i0, act, ld, q0); break;
                    }
                } else {
                    const int r0 = b * P.rpi, nr = min(P.rpi, c.H - r0);
                    switch (n) {
                        case 1: sg_down_item<1>(P, m, st, nr, r0, act, ld, q0); break;
                        case 2: sg_down_item<2>(P, m, st, nr, r0, act, ld, q0); break;
                        case 3: sg_down_item<3>(P, m, st, nr, r0, act, ld, q0); break;
                        default: sg_down_item<4>(P, m, st, nr, r0, act, ld, q0); break;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&m->empty[s]);
        }
    }
}

}  // namespace moe
