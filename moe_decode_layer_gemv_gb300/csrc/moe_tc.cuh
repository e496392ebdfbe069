// moe_tc.cuh -- grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory) for experts that enough tokens
// chose that the projection is a dense contraction.
//
// Swap-AB: the weight rows are the MMA's M side (128 rows per tile), the
// expert's tokens its N side (up to 128), K runs over H (gate/up) or I
// (down) in 64-element steps.  Weight tiles and activation tiles are moved
// by the TMA engine with the 128-byte swizzle into a shared-memory ring
// whose depth follows the launch's largest token count (stages hold one
// weight tile and that many activation rows, so small N buys more weight
// bytes in flight); one warp issues the copies, one thread the MMAs into one
// of two tensor-memory accumulators, and four warps read the other one back
// for the epilogue, so copies, MMAs and the epilogue of consecutive tiles
// overlap.
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

constexpr int kTcThreads = 192;  // warps 0-3 epilogue, warp 4 TMA producer, warp 5 MMA issuer
constexpr int kTcBK = 64;        // K elements per stage (one 128-byte swizzle row)
constexpr int kTcMaxN = 128;     // tokens per tile
constexpr int kTcBoxN = 32;      // rows per activation TMA box
constexpr int kTcMaxStages = 16;
constexpr int kTcATile = 128 * 128;      // 128 rows x 128 B
constexpr int kTcEpiCols = 32;           // accumulator columns per epilogue pass
constexpr int kTcEpiLd = kTcEpiCols + 1; // fp32 row stride of the epilogue tile
constexpr int kTcEpiBytes = 17 * 1024;   // >= 128 * kTcEpiLd * 4, a multiple of 1024
constexpr int kTcSegCache = 256;         // tensor-core segments whose (e, p0, p1) are kept in shared memory
constexpr int kTcSegBytes = kTcSegCache * 16;
constexpr int kTcSmem = 227 * 1024;
constexpr uint32_t kTcWaitLimit = 1u << 24;
constexpr uint32_t kTcTmemCols = 256;    // two accumulators of 128 columns
static_assert(128 * kTcEpiLd * 4 <= kTcEpiBytes, "epilogue tile");

// Selects one of the two compiled copies of the GEMM's item loop.
template <bool B>
struct TcVar {
    static constexpr bool value = B;
};

// Barriers and flags at the start of the kernel's shared memory.
struct TcBars {
    uint64_t full[kTcMaxStages];   // a stage's tiles landed (TMA transaction count)
    uint64_t empty[kTcMaxStages];  // a stage's MMAs are done with it (tcgen05.commit)
    uint64_t acc_full[2];          // an accumulator's MMAs are complete
    uint64_t acc_empty[2];         // the epilogue has read an accumulator (4 warps arrive)
    uint64_t mma_done;             // every MMA issued has completed (teardown)
    uint32_t tmem_slot;
    int abort;                     // a bounded wait ran out: every role stops
};
static_assert(sizeof(TcBars) <= 512, "barrier block: the second half holds the route indices of an item");

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

// The same, also giving up once another role has raised the abort flag.
__device__ __forceinline__ bool tc_wait_ab(uint64_t* bar, uint32_t parity, TcBars* b) {
    for (uint32_t i = 0; i < kTcWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && *(volatile int*)&b->abort) return false;
    }
    *(volatile int*)&b->abort = 1;
    return false;
}

// ------------------------------------------------------------ activations
// Split the activation rows of every route position p into bf16 hi and lo:
// x_hi[p] = bf16(x[t]), x_lo[p] = bf16(x[t] - x_hi[p]), t = route_at(p) / k.
__global__ void __launch_bounds__(kThreads) tc_split_x_kernel(Ctx c, uint16_t* x_hi, uint16_t* x_lo) {
    grid_dep_wait();
    const int p = blockIdx.x;
    if (p >= c.B * c.k) return;
    const int t = route_at(c, p) / c.k;
    for (int h = 4 * threadIdx.x; h < c.H; h += 4 * blockDim.x) {  // four elements a thread (H % 8 == 0)
        float v[4];
        if (c.x_bf16) {
            const uint2 u = __ldcg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(c.x) + (size_t)t * c.H + h));
            v[0] = __uint_as_float(u.x << 16);
            v[1] = __uint_as_float(u.x & 0xffff0000u);
            v[2] = __uint_as_float(u.y << 16);
            v[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            const float4 f = ld_act_f4(static_cast<const float*>(c.x) + (size_t)t * c.H + h);
            v[0] = f.x;
            v[1] = f.y;
            v[2] = f.z;
            v[3] = f.w;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hi[j] = f2bf_bits(v[j]);
            lo[j] = f2bf_bits(v[j] - bf_bits2f((uint16_t)hi[j]));
        }
        *reinterpret_cast<uint2*>(x_hi + (size_t)p * c.H + h) = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
        *reinterpret_cast<uint2*>(x_lo + (size_t)p * c.H + h) = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
    }
}

// ------------------------------------------------------------ the GEMM
// Persistent: one CTA per SM walks the items of the tensor-core segment
// list; an item is (segment, M tile of 64 gate/up row pairs or 128 down rows,
// 128-token chunk).  Three roles run through the same item sequence:
//   warp 4 (one lane)  TMA producer: k-steps into the ring, waits only for a
//                      stage to be released, so it runs ahead across items;
//   warp 5 (one lane)  MMA issuer: item d accumulates into tensor-memory
//                      buffer d mod 2 once the epilogue has read that
//                      buffer's previous item;
//   warps 0-3          epilogue: accumulator lanes 32w..32w+31, 32 columns
//                      per pass through shared memory to coalesced stores.
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    TcBars* b = reinterpret_cast<TcBars*>(base);
    int* rr = reinterpret_cast<int*>(base + 512);         // [kTcMaxN] flat routes of the item's tokens (down)
    float* epi = reinterpret_cast<float*>(base + 1024);  // [128][kTcEpiLd]
    int4* segtab = reinterpret_cast<int4*>(base + 1024 + kTcEpiBytes);  // [kTcSegCache] (e, p0, p1, valid)
    unsigned char* ring = base + 1024 + kTcEpiBytes + kTcSegBytes;

    const Ctx& c = p.c;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dep_wait();
    const int K = p.gate ? c.H : c.I;
    const int nk = K / kTcBK;
    const int mtiles = p.gate ? c.I / 64 : c.H / 128;
    const int nchunk = (c.B + kTcMaxN - 1) / kTcMaxN;
    const int maxseg = max_segments(c);
    const int n_items = ld_act_i(c.seg_count + 1) * mtiles * nchunk;
    if ((int)blockIdx.x >= n_items) return;  // uniform: nothing for this CTA

    // Ring geometry from the launch's largest tensor-core token count.  A
    // stage holds ksub consecutive 64-wide k-steps (weight tile, then the
    // activation tiles): tensor-copy streams run far below the copy bandwidth
    // when each stage (one mbarrier phase) carries only 16 KB, and near it
    // from about 32 KB up, so small token counts take two k-steps a stage.
    const int nmax = min(kTcMaxN, max(1, ld_act_i(c.seg_count + 2)));
    const uint32_t bbytes = (uint32_t)((nmax + kTcBoxN - 1) / kTcBoxN * kTcBoxN) * 128u;  // one activation operand
    const uint32_t nb = p.with_lo ? 2u : 1u;
    const uint32_t ring_bytes = (uint32_t)kTcSmem - 1023u - (uint32_t)(ring - base);
    auto stage_of = [&](int ks) { return ((uint32_t)ks * (kTcATile + nb * bbytes) + 1023u) & ~1023u; };
    int ksub = 1;
    while (ksub < 4 && stage_of(ksub) < 32768u && ring_bytes / stage_of(2 * ksub) >= 3u) ksub *= 2;
    const uint32_t stage_bytes = stage_of(ksub);
    const int S = min(kTcMaxStages, (int)(ring_bytes / stage_bytes));
    // In a launch of unequal items (below), an item with fewer tokens than the
    // launch's largest packs more k-steps into a stage, up to stage_bytes: a
    // copy stream passes about one stage per round trip whatever it carries,
    // so a cheap item then takes fewer ring phases.  Every role derives the
    // same value from the item's n.
    auto ksub_of = [&](int n_pad) {
        const uint32_t per = kTcATile + nb * (uint32_t)n_pad * 128u;
        int ks = ksub;
        while (ks < 4 && (uint32_t)(2 * ks) * per <= stage_bytes) ks *= 2;
        return ks;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcMaxStages; ++s) {
            mbar_init(&b->full[s], 1);
            mbar_init(&b->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&b->acc_full[a], 1);
            mbar_init(&b->acc_empty[a], 4);
        }
        mbar_init(&b->mma_done, 1);
        b->abort = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(&b->tmem_slot, kTcTmemCols);
    // the segments' descriptors once, so that decoding an item costs no
    // dependent global loads in the producer's issue stream
    const int nts = ld_act_i(c.seg_count + 1);
    const bool cached = nts <= kTcSegCache;
    if (cached)
        for (int i = threadIdx.x; i < nts; i += blockDim.x) {
            Seg sg;
            const bool v = get_seg(c, ld_act_i(c.seg_list + maxseg + i), sg);
            segtab[i] = make_int4(sg.e, sg.p0, sg.p1, v ? 1 : 0);
        }
    // Items of unequal cost (a launch whose largest segment has more than 32
    // tokens) and few items a CTA: the segments are ordered by token count,
    // largest first (stable), and the items are dealt in a snake, so that the
    // CTAs drawing the costliest items in the first round draw the cheapest
    // (or none) in the second.  The order decides only which CTA computes an
    // item, never a value.
    const int G = (int)gridDim.x;
    const bool snake = cached && nmax > kTcBoxN && n_items <= 4 * G && nts <= kTcThreads;
    if (snake) {
        __syncthreads();
        const int i = threadIdx.x;
        int4 mine = make_int4(0, 0, 0, 0);
        int rank = 0;
        if (i < nts) {
            mine = segtab[i];
            const int ni = mine.w ? mine.z - mine.y : 0;
            for (int j = 0; j < nts; ++j) {
                const int4 o = segtab[j];
                const int nj = o.w ? o.z - o.y : 0;
                rank += (nj > ni || (nj == ni && j < i)) ? 1 : 0;
            }
        }
        __syncthreads();
        if (i < nts) segtab[rank] = mine;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b->tmem_slot;

    uint32_t g = 0;         // stages through the ring so far (same in every role)
    uint32_t g_armed = 0;   // stages whose copies the producer armed (producer lane only)
    int d = 0;              // items processed (same in every role)
    // The item loop is compiled twice.  Launches of equal items take the
    // static strided order and the launch's stage layout; launches of unequal
    // items (the snake) also give each item its own stage layout.  One copy
    // serving both measured slower on the launches of equal items.
    auto item_loop = [&](auto var) {
        constexpr bool kVar = decltype(var)::value;
        // slot = round * G + blockIdx.x; a snake's odd rounds run backwards, so
        // its last round may hold items for CTAs whose slot is past n_items
        const int slot_end = n_items + (kVar ? (int)blockIdx.x : 0);
        for (int slot = blockIdx.x; slot < slot_end; slot += G) {
            int item = slot;
            if (kVar && ((slot / G) & 1)) item = (slot / G + 1) * G - 1 - (int)blockIdx.x;
            if (kVar && item >= n_items) continue;  // uniform
            // the token chunk varies slowest: items of later chunks (which exist
            // only for segments with more than 128 routes) come after every
            // first chunk, so no CTA draws only empty items
            const int per_chunk = n_items / nchunk;
            const int nc = item / per_chunk;
            const int rem = item - nc * per_chunk;
            const int sl = rem / mtiles, mt = rem - sl * mtiles;
            Seg sg;
            if (cached) {
                const int4 t = segtab[sl];
                if (!t.w) continue;  // uniform
                sg.e = t.x;
                sg.p0 = t.y;
                sg.p1 = t.z;
            } else if (!get_seg(c, ld_act_i(c.seg_list + maxseg + sl), sg)) {
                continue;  // uniform
            }
            const int q0 = sg.p0 + nc * kTcMaxN;
            if (q0 >= sg.p1) continue;
            const int n = min(kTcMaxN, sg.p1 - q0);
            const int n_pad = (n + kTcBoxN - 1) / kTcBoxN * kTcBoxN;
            const int buf = d & 1, use = d >> 1;
            // stage layout of this item: ks weight tiles, then ks activation
            // tiles (hi), then ks (lo)
            const int ks = kVar ? ksub_of(n_pad) : ksub;
            const int nst = (nk + ks - 1) / ks;  // stages of this item
            const uint32_t bb = kVar ? (uint32_t)n_pad * 128u : bbytes;  // one activation operand
            const uint32_t b_off = (uint32_t)ks * kTcATile;

            if (warp == 4) {
                if (lane == 0) {
                    // ---------------- TMA producer
                    // MOE_F_HOT_L2: the experts with at least MOE_TC_MIN_ROUTES
                    // routes are the step's most chosen ones; their weights are
                    // loaded with evict_last so that they stay in L2 for the next
                    // steps, those of the others with evict_first
                    const bool hot = (c.flags & MOE_F_HOT_L2) != 0;
                    const uint64_t pol = !hot                                   ? 0ull
                                         : sg.p1 - sg.p0 >= MOE_TC_MIN_ROUTES ? l2_policy_evict_last()
                                                                               : l2_policy_evict_first();
                    const uint32_t bytes = kTcATile + (uint32_t)n_pad * 128u * (p.with_lo ? 2u : 1u);
                    int arow0, arow1 = 0;
                    if (p.gate) {
                        arow0 = sg.e * 2 * c.I + mt * 64;
                        arow1 = arow0 + c.I;
                    } else {
                        arow0 = sg.e * c.H + mt * 128;
                    }
                    for (int j = 0; j < nst; ++j) {
                        const uint32_t gs = g + (uint32_t)j;
                        const int s = (int)(gs % (uint32_t)S);
                        const uint32_t ph = (gs / (uint32_t)S) & 1u;
                        if (gs >= (uint32_t)S && !tc_wait_ab(&b->empty[s], ph ^ 1u, b)) break;
                        unsigned char* st = ring + (size_t)s * stage_bytes;
                        const int k0 = j * ks, ke = min(ks, nk - k0);  // k-steps k0 .. k0+ke-1
                        mbar_arrive_expect_tx(&b->full[s], (uint32_t)ke * bytes);
                        g_armed = gs + 1u;
                        for (int u = 0; u < ke; ++u) {
                            const int kx = (k0 + u) * kTcBK;
                            unsigned char* sa = st + (size_t)u * kTcATile;
                            unsigned char* sb = st + b_off + (size_t)u * bb;
                            if (hot) {
                                tma_load_2d_hint(sa, &p.ta, kx, arow0, &b->full[s], pol);
                                if (p.gate) tma_load_2d_hint(sa + 8192, &p.ta, kx, arow1, &b->full[s], pol);
                            } else {
                                tma_load_2d(sa, &p.ta, kx, arow0, &b->full[s]);
                                if (p.gate) tma_load_2d(sa + 8192, &p.ta, kx, arow1, &b->full[s]);
                            }
                            for (int r = 0; r < n_pad; r += kTcBoxN) {
                                tma_load_2d(sb + r * 128, &p.tb_hi, kx, q0 + r, &b->full[s]);
                                if (p.with_lo)
                                    tma_load_2d(sb + (size_t)ks * bb + r * 128, &p.tb_lo, kx, q0 + r, &b->full[s]);
                            }
                        }
                    }
                }
                __syncwarp();
            } else if (warp == 5) {
                if (lane == 0) {
                    // ---------------- MMA issuer (one thread)
                    bool ok = use == 0 || tc_wait_ab(&b->acc_empty[buf], (uint32_t)((use - 1) & 1), b);
                    tc_fence_after();
                    const uint32_t tacc = tmem + (uint32_t)(buf * 128);
                    const uint32_t idesc = umma_idesc_bf16(128, n_pad);
                    for (int j = 0; ok && j < nst; ++j) {
                        const uint32_t gs = g + (uint32_t)j;
                        const int s = (int)(gs % (uint32_t)S);
                        const uint32_t ph = (gs / (uint32_t)S) & 1u;
                        if (!tc_wait_ab(&b->full[s], ph, b)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const int ke = min(ks, nk - j * ks);
                        const uint32_t st_addr = smem_u32(ring + (size_t)s * stage_bytes);
                        for (int u = 0; u < ke; ++u) {
                            const uint32_t a_addr = st_addr + (uint32_t)u * kTcATile;
                            const uint32_t bh_addr = st_addr + b_off + (uint32_t)u * bb;
                            const uint32_t bl_addr = bh_addr + (uint32_t)ks * bb;
    #pragma unroll
                            for (int kk = 0; kk < kTcBK / 16; ++kk) {
                                const uint64_t ad = umma_sdesc(a_addr + kk * 32);
                                umma_bf16(tacc, ad, umma_sdesc(bh_addr + kk * 32), idesc, (j > 0 || u > 0 || kk > 0) ? 1u : 0u);
                                if (p.with_lo) umma_bf16(tacc, ad, umma_sdesc(bl_addr + kk * 32), idesc, 1u);
                            }
                        }
                        umma_commit(&b->empty[s]);  // the stage is free once these MMAs have read it
                    }
                    if (ok) umma_commit(&b->acc_full[buf]);  // arrives when every MMA of the item is complete
                }
                __syncwarp();
            } else {
                // ---------------- epilogue (warps 0-3: accumulator lanes 32w..32w+31)
                // (one decision for all 128 threads: they meet at named barriers)
                // the down pass writes o by flat route: the item's route indices
                // once into shared memory (ordered before their use by the first
                // barrier below), not a dependent global load per column
                if (!p.gate && (int)threadIdx.x < n) rr[threadIdx.x] = route_at(c, q0 + (int)threadIdx.x);
                const bool ok = !named_sync_or(1, 128, !tc_wait_ab(&b->acc_full[buf], (uint32_t)(use & 1), b));
                tc_fence_after();
                const uint32_t row_addr = tmem + (uint32_t)(buf * 128) + ((uint32_t)(warp * 32) << 16);
                for (int col0 = 0; ok && col0 < n_pad; col0 += kTcEpiCols) {
                    float v[kTcEpiCols];
                    tmem_ld16(row_addr + col0, *reinterpret_cast<float(*)[16]>(v));
                    tmem_ld16(row_addr + col0 + 16, *reinterpret_cast<float(*)[16]>(v + 16));
                    if (col0 + kTcEpiCols >= n_pad) {  // the accumulator is read: the MMA warp may reuse it
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&b->acc_empty[buf]);
                    }
    #pragma unroll
                    for (int j = 0; j < kTcEpiCols; ++j) epi[threadIdx.x * kTcEpiLd + j] = v[j];
                    named_sync(1, 128);
                    const int ncol = min(kTcEpiCols, n - col0);
                    if (p.gate) {
                        const int i0 = mt * 64;
                        for (int t = threadIdx.x; t < 64 * ncol; t += 128) {
                            const int i = t & 63, jj = t >> 6;
                            const float hv = silu_mul(epi[i * kTcEpiLd + jj], epi[(64 + i) * kTcEpiLd + jj]);
                            const uint16_t hi = f2bf_bits(hv);
                            const size_t at = (size_t)(q0 + col0 + jj) * c.I + i0 + i;
                            p.h_hi[at] = hi;
                            p.h_lo[at] = f2bf_bits(hv - bf_bits2f(hi));
                        }
                    } else {
                        const int r0 = mt * 128;
                        for (int t = threadIdx.x; t < 128 * ncol; t += 128) {
                            const int row = t & 127, jj = t >> 7;
                            c.o[(size_t)rr[col0 + jj] * c.H + r0 + row] = epi[row * kTcEpiLd + jj];
                        }
                    }
                    named_sync(1, 128);
                }
            }
            g += (uint32_t)nst;
            ++d;
            // stop on abort, with one decision per barrier group (the epilogue
            // warps meet at named barriers, a warp's lanes at __syncwarp)
            const bool stop = *(volatile int*)&b->abort != 0;
            if (warp < 4 ? named_sync_or(1, 128, stop) : __any_sync(0xffffffffu, stop)) break;
        }
    };
    if (snake)
        item_loop(TcVar<true>{});
    else
        item_loop(TcVar<false>{});
    // teardown: no MMA and no copy may still be in flight when the tensor
    // memory is freed and the CTA exits
    if (warp == 5 && lane == 0) {
        umma_commit(&b->mma_done);
        tc_wait(&b->mma_done, 0u);
    }
    if (warp == 4 && lane == 0)
        for (int s = 0; s < S && (uint32_t)s < g_armed; ++s) {
            // the latest armed use of stage s: its copies have landed once its phase completed
            const uint32_t last = g_armed - 1u - ((g_armed - 1u - (uint32_t)s) % (uint32_t)S);
            tc_wait(&b->full[s], (last / (uint32_t)S) & 1u);
        }
    __syncthreads();
    if (*(volatile int*)&b->abort && threadIdx.x == 0) set_status(c.status, MOE_DEV_TIMEOUT);
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTcTmemCols);
    }
}

}  // namespace moe
