// moe_tc.cuh -- grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory) for experts that enough tokens
// chose that the projection is a dense contraction.
//
// Swap-AB: the weight rows are the MMA's M side (128 rows per tile), the
// expert's tokens its N side (up to 128), K runs over H (gate/up) or I
// (down) in 64-element steps.  Weight tiles and activation tiles are moved
// by the TMA engine with the 128-byte swizzle into a 4-stage shared-memory
// ring; one thread issues the MMAs; the accumulator tile lives in tensor
// memory and four warps read it back for the epilogue.
//
// Precision: the MMA takes bf16 operands.  Weights are bf16 already; fp32
// activations are split into hi = bf16(a) and lo = bf16(a - hi) and the MMA
// accumulates W*hi + W*lo in fp32, so the product keeps ~16 mantissa bits of
// the activation (bf16 activations use the hi part only).
//
// Gate/up tile: A rows 0..63 are gate rows i0..i0+63 and rows 64..127 the up
// rows I+i0..; the epilogue forms h = SiLU(g) * u for those 64 i and writes
// h split into bf16 hi/lo, the down GEMM's activation operand.
// Down tile: A rows are 128 rows of D_e; the epilogue writes o[r, row] for
// every route r of the segment (combined later, j ascending).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_ptx.cuh"

namespace moe {

constexpr int kTcThreads = 128;
constexpr int kTcBK = 64;        // K elements per stage (one 128-byte swizzle row)
constexpr int kTcMaxN = 128;     // tokens per tile
constexpr int kTcBoxN = 32;      // rows per activation TMA box
constexpr int kTcStages = 4;
constexpr int kTcATile = 128 * 128;      // 128 rows x 128 B
constexpr int kTcBTile = kTcMaxN * 128;  // per activation operand
constexpr int kTcStageBytes = kTcATile + 2 * kTcBTile;
constexpr int kTcEpiLd = kTcMaxN + 1;    // fp32 row stride of the epilogue tile
constexpr int kTcSmem = 1024 + kTcStages * kTcStageBytes + 256;
constexpr uint32_t kTcWaitLimit = 1u << 24;
constexpr uint32_t kTcTmemCols = 128;

struct TcParams {
    CUtensorMap ta;      // weights [rows, K] bf16, box {64, 64 (gate) or 128 (down)}
    CUtensorMap tb_hi;   // activations (hi) [R, K] bf16, box {64, 32}
    CUtensorMap tb_lo;   // activations (lo)
    Ctx c;               // problem view: sizes, grouping, scratch
    int gate;            // 1: gate/up GEMM, 0: down GEMM
    int with_lo;
    int threshold;       // this path takes segments with at least this many routes
    uint16_t* h_hi;      // [R, I] written by the gate/up GEMM
    uint16_t* h_lo;
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// the same with an L2 cache policy (createpolicy)
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (start address and strides in 16-byte units).
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address, bits [0,14)
    d |= (uint64_t)1 << 16;                     // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset, bits [32,46)
    d |= (uint64_t)1 << 46;                     // descriptor version, bits [46,48)
    d |= (uint64_t)2 << 61;                     // layout: 128-byte swizzle, bits [61,64)
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 at bits [17,23), M >> 4 at bits [24,29).
__host__ __device__ __forceinline__ uint32_t umma_idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ uint16_t f2bf_bits(float f) {
    const __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<const uint16_t*>(&b);
}

__device__ __forceinline__ float bf_bits2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Bounded wait on a CTA-local mbarrier phase (false after kTcWaitLimit tries).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kTcWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ------------------------------------------------------------ activations
// Split the activation rows of every route position p into bf16 hi and lo:
// x_hi[p] = bf16(x[t]), x_lo[p] = bf16(x[t] - x_hi[p]), t = route_at(p) / k.
__global__ void __launch_bounds__(kThreads) tc_split_x_kernel(Ctx c, uint16_t* x_hi, uint16_t* x_lo) {
    const int p = blockIdx.x;
    if (p >= c.B * c.k) return;
    const int t = route_at(c, p) / c.k;
    for (int h = threadIdx.x; h < c.H; h += blockDim.x) {
        float v;
        if (c.x_bf16) v = bf_bits2f(static_cast<const uint16_t*>(c.x)[(size_t)t * c.H + h]);
        else v = ld_act_f(static_cast<const float*>(c.x) + (size_t)t * c.H + h);
        const uint16_t hi = f2bf_bits(v);
        x_hi[(size_t)p * c.H + h] = hi;
        x_lo[(size_t)p * c.H + h] = f2bf_bits(v - bf_bits2f(hi));
    }
}

// ------------------------------------------------------------ the GEMM
// Persistent: one CTA per SM walks the items of the tensor-core segment
// list; an item is (segment, M tile of 64 gate/up row pairs or 128 down rows,
// 128-token chunk).  The ring position and the accumulator phase carry over
// from item to item; TMEM and the barriers are set up once.
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTcStages * kTcStageBytes);
    uint64_t* empty = full + kTcStages;
    uint64_t* accum = empty + kTcStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
    int* ok_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const Ctx& c = p.c;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = p.gate ? c.H : c.I;
    const int nk = K / kTcBK;
    const int mtiles = p.gate ? c.I / 64 : c.H / 128;
    const int nchunk = (c.B + kTcMaxN - 1) / kTcMaxN;
    const int maxseg = max_segments(c);
    const int n_items = ld_act_i(c.seg_count + 1) * mtiles * nchunk;
    if ((int)blockIdx.x >= n_items) return;  // uniform: nothing for this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        *ok_flag = 1;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTcTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    float* epi = reinterpret_cast<float*>(smem);  // [128][kTcEpiLd]: stage memory, idle during the epilogue

    int g = 0;     // k-steps through the ring so far (same in every thread)
    int done = 0;  // items finished (accumulator phases)
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        // the token chunk varies slowest: items of later chunks (which exist
        // only for segments with more than 128 routes) come after every
        // first chunk, so no CTA draws only empty items
        const int per_chunk = n_items / nchunk;
        const int nc = item / per_chunk;
        const int rem = item - nc * per_chunk;
        const int sl = rem / mtiles, mt = rem - sl * mtiles;
        Seg sg;
        if (!get_seg(c, ld_act_i(c.seg_list + maxseg + sl), sg)) continue;  // uniform
        const int q0 = sg.p0 + nc * kTcMaxN;
        if (q0 >= sg.p1) continue;
        const int n = min(kTcMaxN, sg.p1 - q0);
        const int n_pad = (n + kTcBoxN - 1) / kTcBoxN * kTcBoxN;

        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer
            // MOE_F_HOT_L2: the tensor-core experts are the step's most chosen
            // ones (>= threshold routes); their weights are loaded with
            // evict_last so that they stay in L2 for the next steps
            const bool hot = (c.flags & MOE_F_HOT_L2) != 0;
            const uint64_t pol = hot ? l2_policy_evict_last() : 0ull;
            const uint32_t bytes = kTcATile + (uint32_t)n_pad * 128u * (p.with_lo ? 2u : 1u);
            int arow0, arow1 = 0;
            if (p.gate) {
                arow0 = sg.e * 2 * c.I + mt * 64;
                arow1 = arow0 + c.I;
            } else {
                arow0 = sg.e * c.H + mt * 128;
            }
            for (int kc = 0; kc < nk; ++kc) {
                const int gk = g + kc;
                const int s = gk % kTcStages;
                const uint32_t ph = (uint32_t)((gk / kTcStages) & 1);
                if (gk >= kTcStages && !tc_wait(&empty[s], ph ^ 1u)) {
                    *(volatile int*)ok_flag = 0;
                    break;
                }
                unsigned char* st = smem + (size_t)s * kTcStageBytes;
                mbar_arrive_expect_tx(&full[s], bytes);
                if (hot) {  // the expert's weights stay in L2 for the next steps
                    tma_load_2d_hint(st, &p.ta, kc * kTcBK, arow0, &full[s], pol);
                    if (p.gate) tma_load_2d_hint(st + 8192, &p.ta, kc * kTcBK, arow1, &full[s], pol);
                } else if (p.gate) {
                    tma_load_2d(st, &p.ta, kc * kTcBK, arow0, &full[s]);
                    tma_load_2d(st + 8192, &p.ta, kc * kTcBK, arow1, &full[s]);
                } else {
                    tma_load_2d(st, &p.ta, kc * kTcBK, arow0, &full[s]);
                }
                for (int r = 0; r < n_pad; r += kTcBoxN) {
                    tma_load_2d(st + kTcATile + r * 128, &p.tb_hi, kc * kTcBK, q0 + r, &full[s]);
                    if (p.with_lo)
                        tma_load_2d(st + kTcATile + kTcBTile + r * 128, &p.tb_lo, kc * kTcBK, q0 + r, &full[s]);
                }
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------- MMA issuer (one thread)
            const uint32_t idesc = umma_idesc_bf16(128, n_pad);
            for (int kc = 0; kc < nk; ++kc) {
                const int gk = g + kc;
                const int s = gk % kTcStages;
                const uint32_t ph = (uint32_t)((gk / kTcStages) & 1);
                if (!tc_wait(&full[s], ph)) {
                    *(volatile int*)ok_flag = 0;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + (size_t)s * kTcStageBytes);
                const uint32_t bh_addr = a_addr + kTcATile;
                const uint32_t bl_addr = bh_addr + kTcBTile;
#pragma unroll
                for (int kk = 0; kk < kTcBK / 16; ++kk) {
                    const uint64_t ad = umma_sdesc(a_addr + kk * 32);
                    umma_bf16(tmem, ad, umma_sdesc(bh_addr + kk * 32), idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                    if (p.with_lo) umma_bf16(tmem, ad, umma_sdesc(bl_addr + kk * 32), idesc, 1u);
                }
                umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
            }
            umma_commit(accum);  // every MMA issued so far is complete when this arrives
        }
        __syncwarp();

        // ---------------- epilogue (all four warps)
        if (!tc_wait(accum, (uint32_t)(done & 1))) *(volatile int*)ok_flag = 0;
        tc_fence_after();
        __syncthreads();
        const bool good = *(volatile int*)ok_flag != 0;  // the same in every thread
        if (good) {
            const uint32_t row_addr = tmem + ((uint32_t)(warp * 32) << 16);
            for (int col = 0; col < n_pad; col += 16) {
                float v[16];
                tmem_ld16(row_addr + col, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) epi[threadIdx.x * kTcEpiLd + col + j] = v[j];
            }
        }
        tc_fence_before();
        __syncthreads();
        if (good) {
            if (p.gate) {
                const int i0 = mt * 64;
                for (int v = threadIdx.x; v < 64 * n; v += kTcThreads) {
                    const int i = v & 63, j = v >> 6;
                    const float hv = silu_mul(epi[i * kTcEpiLd + j], epi[(64 + i) * kTcEpiLd + j]);
                    const uint16_t hi = f2bf_bits(hv);
                    const size_t at = (size_t)(q0 + j) * c.I + i0 + i;
                    p.h_hi[at] = hi;
                    p.h_lo[at] = f2bf_bits(hv - bf_bits2f(hi));
                }
            } else {
                const int r0 = mt * 128;
                for (int v = threadIdx.x; v < 128 * n; v += kTcThreads) {
                    const int row = v & 127, j = v >> 7;
                    const int r = route_at(c, q0 + j);
                    c.o[(size_t)r * c.H + r0 + row] = epi[row * kTcEpiLd + j];
                }
            }
        }
        // the next item's loads and MMAs reuse the stages and TMEM only after
        // every thread is done with this item's epilogue
        __syncthreads();
        g += nk;
        ++done;
        if (!good) {
            if (threadIdx.x == 0) set_status(c.status, MOE_DEV_TIMEOUT);
            break;
        }
    }
    // leave with no copy in flight: the latest phase of every stage has landed
    if (warp == 0 && lane == 0)
        for (int s = 0; s < kTcStages; ++s) {
            const int last = g - 1 - ((g - 1 - s) % kTcStages + kTcStages) % kTcStages;  // last k-step in stage s
            if (last >= 0) tc_wait(&full[s], (uint32_t)((last / kTcStages) & 1));
        }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTcTmemCols);
    }
}

}  // namespace moe
