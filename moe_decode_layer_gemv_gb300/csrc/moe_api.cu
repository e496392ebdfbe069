// moe_api.cu -- the C ABI of libmoe.so (declared in include/moe.h): argument
// checks, workspace layout and kernel launches.  Kernels: the persistent
// decode kernel for batches of up to 4 tokens (moe_decode.cuh, whole layers
// or stacks in one launch); for larger batches the phase kernels of
// moe_phases.cuh (router, top-k, grouping, combine), the streaming grouped
// GEMV passes (moe_stream.cuh) and the tensor-core GEMMs (moe_tc.cuh), or
// all phases in one persistent fused kernel when no expert needs the tensor
// cores.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "moe.h"
#include "moe_common.cuh"
#include "moe_phases.cuh"
#include "moe_decode.cuh"
#include "moe_tc.cuh"
#include "moe_stream.cuh"

namespace moe {

// ------------------------------------------------------------ grid barrier
// Device-wide barrier for the persistent kernel.  A monotonically increasing
// arrival counter (zeroed by the host before the launch): barrier number n
// completes when the counter reaches n * gridDim.x.  Every wait is bounded;
// a CTA that gives up sets MOE_DEV_TIMEOUT and the abort word, and every
// CTA then leaves the kernel at its next barrier.
constexpr unsigned long long kSpinLimit = 1ull << 22;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ bool grid_sync(unsigned* bar, unsigned& epoch, int32_t* status, unsigned extra) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        epoch += 1;
        const unsigned target = epoch * (gridDim.x + extra);
        __threadfence();
        red_release_add_u32(bar, 1u);
        int ok = 1;
        unsigned long long spins = 0;
        while (ld_acquire_u32(bar) < target) {
            ++spins;
            if ((spins & 255ull) == 0 && ld_acquire_u32(bar + 1) != 0u) {
                ok = 0;
                break;
            }
            if (spins > kSpinLimit) {
                set_status(status, MOE_DEV_TIMEOUT);
                atomicExch(bar + 1, 1u);
                ok = 0;
                break;
            }
            if (spins > 32) __nanosleep(64);
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// ----------------------------------------------------------------- kernels
struct StackArgs {
    LayerWeights layer[MOE_MAX_LAYERS];
    int L;
    int32_t* ids_out;  // [L, B, k] or nullptr
    unsigned bar_extra;  // arrivals a barrier waits for beyond the grid (0; > 0 only to test the timeout)
};

template <int EPW>
__global__ void __launch_bounds__(kThreads) router_kernel(Ctx c) {
    extern __shared__ __align__(128) unsigned char smem[];
    grid_dep_wait();
    router_item<EPW>(c, blockIdx.x, reinterpret_cast<float*>(smem));
}

__global__ void __launch_bounds__(kThreads) topk_kernel(Ctx c) {
    grid_dep_wait();
    topk_item(c, blockIdx.x, c.ids, c.rw);
}

__global__ void __launch_bounds__(kThreads) group_kernel(const int32_t* ids, int B, int k, int E,
                                                         int32_t* offsets, int32_t* route_idx,
                                                         int32_t* unique, int32_t* num_unique,
                                                         int32_t* status) {
    extern __shared__ __align__(128) unsigned char smem[];
    grid_dep_wait();
    group_cta(ids, B, k, E, offsets, route_idx, unique, num_unique, status,
              reinterpret_cast<uint32_t*>(smem));
}

__device__ __forceinline__ void split_smem(const Ctx& c, unsigned char* smem, float*& act, int*& idx) {
    const int dim = c.H > c.I ? c.H : c.I;
    act = reinterpret_cast<float*>(smem);
    idx = reinterpret_cast<int*>(smem + sizeof(float) * (size_t)c.nt_max * dim);
}

__global__ void __launch_bounds__(kThreads) gateup_kernel(Ctx c) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* xs;
    int* tok;
    split_smem(c, smem, xs, tok);
    grid_dep_wait();
    const int n = c.seg_list ? ld_act_i(c.seg_count) * ceil_div(c.I, kWarps) : gateup_items(c);
    for (int it = blockIdx.x; it < n; it += gridDim.x) gateup_item(c, it, xs, tok);
}

__global__ void __launch_bounds__(kThreads) down_kernel(Ctx c) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* hs;
    int* rts;
    split_smem(c, smem, hs, rts);
    grid_dep_wait();
    const int n = c.seg_list ? ld_act_i(c.seg_count) * ceil_div(c.H, kDownRows) : down_items(c);
    for (int it = blockIdx.x; it < n; it += gridDim.x) down_item(c, it, hs, rts);
}

__global__ void classify_kernel(Ctx c) {
    grid_dep_wait();
    classify_warp(c);
}

// The steps between the router and the expert passes of a layer in one CTA:
// the top-k of every token (one warp per token), the grouping and the split
// of the segments into the CUDA-core and tensor-core lists (c.seg_list set).
// Two launches fewer, and their dependency waits, for batches up to
// kRouteTailMaxB tokens (measured: 5-9 % off the B = 8 and 16 layers); beyond
// that the one CTA's top-k, a token per warp in turn, costs more than the
// launches it saves (+10 % at B = 128).
constexpr int kRouteTailThreads = 1024;
constexpr int kRouteTailMaxB = 32;
__global__ void __launch_bounds__(kRouteTailThreads) route_tail_kernel(Ctx c) {
    extern __shared__ __align__(128) unsigned char smem[];
    grid_dep_wait();
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int t = warp; t < c.B; t += nw) topk_token(c, t, c.ids, c.rw);
    __syncthreads();
    group_cta(c.ids, c.B, c.k, c.E, c.offsets, c.route_idx, c.unique, c.num_unique, c.status,
              reinterpret_cast<uint32_t*>(smem));
    __syncthreads();
    if (warp == 0) classify_warp(c);
}

// Grouping and classification in one CTA, for batches beyond kRouteTailMaxB
// (whose top-k runs on many CTAs): one launch fewer.
__global__ void __launch_bounds__(kRouteTailThreads) group_classify_kernel(Ctx c) {
    extern __shared__ __align__(128) unsigned char smem[];
    grid_dep_wait();
    group_cta(c.ids, c.B, c.k, c.E, c.offsets, c.route_idx, c.unique, c.num_unique, c.status,
              reinterpret_cast<uint32_t*>(smem));
    __syncthreads();
    if (threadIdx.x < 32) classify_warp(c);
}

__global__ void __launch_bounds__(kThreads) combine_kernel(Ctx c) {
    grid_dep_wait();
    combine_item(c, blockIdx.x);
}

// All phases of L layers in one launch.  For L > 1 (a stack) x, residual and
// y all point at the fp32 residual stream, updated in place by the combine.
__global__ void __launch_bounds__(kThreads) fused_kernel(Ctx c, StackArgs sa, unsigned* bar) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* act;
    int* idx;
    split_smem(c, smem, act, idx);
    unsigned epoch = 0;
    int32_t* ids_base = c.ids;
    for (int l = 0; l < sa.L; ++l) {
        c.w = sa.layer[l];
        c.ids = sa.ids_out ? sa.ids_out + (size_t)l * c.B * c.k : ids_base;
        for (int it = blockIdx.x; it < router_items(c); it += gridDim.x)
            router_item(c, it, reinterpret_cast<float*>(smem));
        if (!grid_sync(bar, epoch, c.status, sa.bar_extra)) return;
        for (int it = blockIdx.x; it < topk_items(c); it += gridDim.x) topk_item(c, it, c.ids, c.rw);
        if (!grid_sync(bar, epoch, c.status, sa.bar_extra)) return;
        if (blockIdx.x == 0)
            group_cta(c.ids, c.B, c.k, c.E, c.offsets, c.route_idx, c.unique, c.num_unique, c.status,
                      reinterpret_cast<uint32_t*>(smem));
        if (!grid_sync(bar, epoch, c.status, sa.bar_extra)) return;
        for (int it = blockIdx.x; it < gateup_items(c); it += gridDim.x) gateup_item(c, it, act, idx);
        if (!grid_sync(bar, epoch, c.status, sa.bar_extra)) return;
        for (int it = blockIdx.x; it < down_items(c); it += gridDim.x) down_item(c, it, act, idx);
        if (!grid_sync(bar, epoch, c.status, sa.bar_extra)) return;
        for (int it = blockIdx.x; it < combine_items(c); it += gridDim.x) combine_item(c, it);
        if (l + 1 < sa.L && !grid_sync(bar, epoch, c.status, sa.bar_extra)) return;
    }
}

// -------------------------------------------------------------- host side
static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr unsigned kAllFlags =
    MOE_F_NO_DEDUP | MOE_F_UNFUSED | MOE_F_FORCE_TC | MOE_F_NO_TC | MOE_F_NO_PREFETCH | MOE_F_HOT_L2 | MOE_F_SPLIT_TC;

struct WsLayout {
    size_t logits, ids, rw, offsets, route_idx, unique, num_unique, status, bar, acc, xt, acc_end, h, o;
    size_t x_hi, x_lo, h_hi, h_lo, seg_list, seg_count, alog, xn, total;
};

static WsLayout ws_layout(int B, int H, int I, int E, int k) {
    WsLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + (bytes > 0 ? bytes : 1), 256);
        return at;
    };
    const size_t R = (size_t)B * k;
    L.logits = take(sizeof(float) * (size_t)B * E);
    L.ids = take(sizeof(int32_t) * R);
    L.rw = take(sizeof(float) * R);
    L.offsets = take(sizeof(int32_t) * (E + 1));
    L.route_idx = take(sizeof(int32_t) * R);
    L.unique = take(sizeof(int32_t) * E);
    L.num_unique = take(sizeof(int32_t));
    L.status = take(sizeof(int32_t));
    L.bar = take(sizeof(unsigned) * 1056);  // abort/counter words + one barrier flag per CTA (<= 1024)
    // decode kernel: three sets of counted logit words [2][B][E] and of sums
    // of squares [2][B], and the tagged copy of x [B][H] u64 after them,
    // right after bar: one memset clears all
    const size_t acc_bytes = sizeof(unsigned long long) * 3 * 2 * (size_t)B * (E + 1);
    L.acc = take(acc_bytes);
    L.xt = take(sizeof(unsigned long long) * 2 * (size_t)B * H);
    L.acc_end = L.xt + sizeof(unsigned long long) * 2 * (size_t)B * H;
    L.h = take(sizeof(float) * 2 * R * I);  // two by layer parity (decode kernel)
    L.o = take(sizeof(float) * R * H);
    L.x_hi = take(sizeof(uint16_t) * R * H);  // tensor-core activation operands (bf16 hi/lo)
    L.x_lo = take(sizeof(uint16_t) * R * H);
    L.h_hi = take(sizeof(uint16_t) * R * I);
    L.h_lo = take(sizeof(uint16_t) * R * I);
    L.seg_list = take(sizeof(int32_t) * 2 * (R > (size_t)E ? R : (size_t)E));
    L.seg_count = take(sizeof(int32_t) * 4);  // CUDA-core and tensor-core segments, largest tensor-core segment
    L.alog = take(sizeof(float) * 2 * (size_t)B * E);  // [2][E]: predicted logits, by layer parity
    L.xn = take(sizeof(float) * (size_t)B * H);  // pre-norm stacks: the normalised layer input
    L.total = off;
    return L;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_dims(int B, int H, int I, int E, int k, bool need_I) {
    if (B < 0 || B > MOE_MAX_B) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > MOE_MAX_E) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > E || k > MOE_MAX_TOPK) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_DIM || (H & 7)) return MOE_ERR_INVALID_ARG;
    if (need_I && (I < 8 || I > MOE_MAX_DIM || (I & 7))) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

#define MOE_REQ(p) \
    do {           \
        if (!(p) || !aligned16(p)) return MOE_ERR_INVALID_ARG; \
    } while (0)
#define MOE_OPT(p) \
    do {           \
        if ((p) && !aligned16(p)) return MOE_ERR_INVALID_ARG; \
    } while (0)

static int nt_max_for(int H, int I) {
    const int dim = H > I ? H : I;
    int nt = 8;
    while (nt > 1 && (size_t)nt * dim * sizeof(float) > 64 * 1024) nt >>= 1;
    return nt;
}

static size_t act_smem(int H, int I) {
    const int dim = H > I ? H : I;
    return sizeof(float) * (size_t)nt_max_for(H, I) * dim + 64;
}

static size_t fused_smem(int B, int H, int I, int E) {
    size_t s = act_smem(H, I);
    if (kRouterSmem > s) s = kRouterSmem;
    const size_t g = group_smem_bytes(B, E);
    if (g > s) s = g;
    return align_up(s, 16);
}

static int to_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    return MOE_ERR_CUDA;
}

// Kernels this library has launched in the process (every launch site goes
// through launch_ex or launch_pdl), for measurement: moe_launch_count().
static std::atomic<unsigned long long> g_launches{0};

template <typename K, typename... Args>
static int launch_ex(const cudaLaunchConfig_t& cfg, K kernel, Args... args) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return to_status(cudaLaunchKernelEx(&cfg, kernel, args...));
}

// A launch that may start while the kernel ahead of it on the stream is
// finishing (programmatic stream serialization): the kernel's setup overlaps
// the previous kernel's tail; its first read of earlier results waits in
// grid_dep_wait().  Used for the chain of phase kernels of one layer.
template <typename K, typename... Args>
static int launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_ex(cfg, kernel, args...);
}

// dynamic shared memory above 48 KB needs an opt-in per kernel and device
template <typename K>
static int allow_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return MOE_OK;
    return to_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
}

static int tc_threshold_for(unsigned flags, int H, int I);

static Ctx make_ctx(const void* x, int x_dtype, const float* residual, float* y, int B, int H, int I,
                    int E, int k, unsigned flags, char* ws, const WsLayout& L, int32_t* status) {
    Ctx c;
    memset(&c, 0, sizeof c);
    c.x = x;
    c.x_bf16 = x_dtype == MOE_DT_BF16;
    c.residual = residual;
    c.y = y;
    c.B = B;
    c.H = H;
    c.I = I;
    c.E = E;
    c.k = k;
    c.flags = flags;
    c.nt_max = nt_max_for(H, I);
    if (ws) {
        c.logits = reinterpret_cast<float*>(ws + L.logits);
        c.ids = reinterpret_cast<int32_t*>(ws + L.ids);
        c.rw = reinterpret_cast<float*>(ws + L.rw);
        c.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
        c.route_idx = reinterpret_cast<int32_t*>(ws + L.route_idx);
        c.unique = reinterpret_cast<int32_t*>(ws + L.unique);
        c.num_unique = reinterpret_cast<int32_t*>(ws + L.num_unique);
        c.h = reinterpret_cast<float*>(ws + L.h);
        c.o = reinterpret_cast<float*>(ws + L.o);
        c.status = status ? status : reinterpret_cast<int32_t*>(ws + L.status);
        c.tc_threshold = tc_threshold_for(flags, H, I);
    } else {
        c.status = status;
        c.tc_threshold = 0;  // the tensor-core path needs workspace for its operands
    }
    return c;
}

// The router with one expert per warp for small batches (more CTAs, each
// weight row read by fewer of them), four per warp from 64 tokens on (the
// staged x read once for four experts: a quarter of the shared-memory traffic).
static int launch_router(const Ctx& c, cudaStream_t st) {
    int rc;
    if (c.B >= 64) {
        if ((rc = allow_smem(router_kernel<4>, kRouterSmem))) return rc;
        return launch_pdl(router_kernel<4>, router_items(c, 4), kThreads, kRouterSmem, st, c);
    }
    if ((rc = allow_smem(router_kernel<1>, kRouterSmem))) return rc;
    return launch_pdl(router_kernel<1>, router_items(c), kThreads, kRouterSmem, st, c);
}

static int launch_route(const Ctx& c, cudaStream_t st) {
    const int rc = launch_router(c, st);
    if (rc) return rc;
    return launch_pdl(topk_kernel, topk_items(c), kThreads, 0, st, c);
}

static int launch_group(const int32_t* ids, int B, int k, int E, int32_t* offsets, int32_t* route_idx,
                        int32_t* unique, int32_t* num_unique, int32_t* status, cudaStream_t st) {
    const size_t smem = group_smem_bytes(B, E);
    int rc = allow_smem(group_kernel, smem);
    if (rc) return rc;
    return launch_pdl(group_kernel, 1, kThreads, smem, st, ids, B, k, E, offsets, route_idx, unique, num_unique,
                      status);
}


static int sm_count();

// ------------------------------------------------------- tensor-core path
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (a function-local static
// is initialised exactly once even when several host threads call first).
static EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(f);
        return nullptr;
    }();
    return fn;
}

// 2-D bf16 tensor [rows, inner] (row-major), 128-byte swizzled boxes of
// {64, box_rows}; rows beyond the tensor read as zeros.
static bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool tc_shape_ok(int H, int I) { return H >= 128 && (H % 128) == 0 && I >= 64 && (I % 64) == 0; }

// Every chosen expert runs on the tensor cores, even one with a single
// route: one GEMM launch per projection streams all the step's experts
// through a deep TMA ring and keeps the whole GPU busy, where the split
// between a tensor-core launch for the popular experts and a CUDA-core
// streaming launch for the rest (MOE_F_SPLIT_TC) runs two launches that each
// fill only part of it, and the GEMV's consumers are bound by their fp32 FMAs.
static int tc_threshold_for(unsigned flags, int H, int I) {
    if ((flags & MOE_F_NO_TC) || !tc_shape_ok(H, I)) return 0;
    if ((flags & MOE_F_SPLIT_TC) && !(flags & MOE_F_FORCE_TC)) return MOE_TC_MIN_ROUTES;
    return 1;
}

static int launch_tc(const Ctx& c, char* ws, const WsLayout& L, cudaStream_t st) {
    int rc = allow_smem(tc_gemm_kernel, kTcSmem);
    if (rc) return rc;
    const int R = c.B * c.k;
    uint16_t* x_hi = reinterpret_cast<uint16_t*>(ws + L.x_hi);
    uint16_t* x_lo = reinterpret_cast<uint16_t*>(ws + L.x_lo);
    TcParams tp;
    memset(&tp, 0, sizeof tp);
    tp.c = c;
    tp.threshold = c.tc_threshold;
    tp.h_hi = reinterpret_cast<uint16_t*>(ws + L.h_hi);
    tp.h_lo = reinterpret_cast<uint16_t*>(ws + L.h_lo);
    tp.with_lo = c.x_bf16 ? 0 : 1;
    if ((rc = launch_pdl(tc_split_x_kernel, R, kThreads, 0, st, c, x_hi, x_lo))) return rc;
    const int nseg = max_segments(c);
    const int nchunk = (c.B + kTcMaxN - 1) / kTcMaxN;
    // gate/up: A = gate_up viewed as [E*2I, H], 64-row boxes
    if (!encode_bf16_2d(&tp.ta, c.w.gate_up, c.H, (uint64_t)c.E * 2 * c.I, 64) ||
        !encode_bf16_2d(&tp.tb_hi, x_hi, c.H, R, kTcBoxN) || !encode_bf16_2d(&tp.tb_lo, x_lo, c.H, R, kTcBoxN))
        return MOE_ERR_UNSUPPORTED;
    tp.gate = 1;
    const int grid = sm_count() > 0 ? sm_count() : 1;
    (void)nseg;
    (void)nchunk;
    return launch_pdl(tc_gemm_kernel, grid, kTcThreads, kTcSmem, st, tp);
}

static int launch_tc_down(const Ctx& c, char* ws, const WsLayout& L, cudaStream_t st) {
    const int R = c.B * c.k;
    TcParams tp;
    memset(&tp, 0, sizeof tp);
    tp.c = c;
    tp.threshold = c.tc_threshold;
    tp.with_lo = 1;  // h is fp32: always split
    const uint16_t* h_hi = reinterpret_cast<const uint16_t*>(ws + L.h_hi);
    const uint16_t* h_lo = reinterpret_cast<const uint16_t*>(ws + L.h_lo);
    if (!encode_bf16_2d(&tp.ta, c.w.down, c.I, (uint64_t)c.E * c.H, 128) ||
        !encode_bf16_2d(&tp.tb_hi, h_hi, c.I, R, kTcBoxN) || !encode_bf16_2d(&tp.tb_lo, h_lo, c.I, R, kTcBoxN))
        return MOE_ERR_UNSUPPORTED;
    tp.gate = 0;
    return launch_pdl(tc_gemm_kernel, sm_count() > 0 ? sm_count() : 1, kTcThreads, kTcSmem, st, tp);
}

// Geometry of a streaming grouped-GEMV pass; false when it does not apply
// (segments may exceed kSgMaxTok routes, or the rows do not fit).
static bool stream_plan(const Ctx& c, int gate, SgParams& P, size_t& smem) {
    if (c.tc_threshold < 2 || c.tc_threshold > MOE_TC_MIN_ROUTES || c.seg_list == nullptr) return false;
    memset(&P, 0, sizeof P);
    P.c = c;
    P.gate = gate;
    if (gate) {
        P.rpi = kSgStageTarget / (4 * c.H);
        if (P.rpi < 1) P.rpi = 1;
        P.ips = ceil_div(c.I, P.rpi);
        P.dim = c.H;
        P.stage_bytes = (int)align_up((size_t)P.rpi * 4 * c.H, 128);
    } else {
        P.rpi = kSgStageTarget / (2 * c.I);
        if (P.rpi < 1) P.rpi = 1;
        if (P.rpi > 4) P.rpi &= ~3;  // whole 4-row groups
        P.ips = ceil_div(c.H, P.rpi);
        P.dim = c.I;
        P.stage_bytes = (int)align_up((size_t)P.rpi * 2 * c.I, 128);
    }
    const size_t off_act = align_up(sizeof(SgMisc), 128);
    const size_t off_ring = align_up(off_act + sizeof(float) * kSgMaxTok * (size_t)lb_stride(P.dim), 128);
    const size_t limit = 227 * 1024;
    if (off_ring + 2 * (size_t)P.stage_bytes > limit) return false;
    size_t S = (limit - off_ring) / P.stage_bytes;
    if (S > (size_t)kSgMaxStages) S = kSgMaxStages;
    const size_t W = S < (size_t)kSgConsumers ? S : (size_t)kSgConsumers;
    S = W * (S / W);
    P.S = (int)S;
    P.W = (int)W;
    P.off_act = (int)off_act;
    P.off_ring = (int)off_ring;
    smem = off_ring + S * P.stage_bytes;
    return true;
}

static int launch_stream(const SgParams& P, size_t smem, cudaStream_t st) {
    int rc = allow_smem(stream_gemv_kernel, smem);
    if (rc) return rc;
    const int sms = sm_count();
    return launch_pdl(stream_gemv_kernel, sms > 0 ? sms : 1, kSgThreads, smem, st, P);
}

// Resident CTAs of a kernel on the whole GPU (at least 1).
template <typename K>
static int resident_grid(K kernel, int threads, size_t smem) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int sms = sm_count();
    return (sms > 0 ? sms : 1) * per_sm;
}

// The expert pass.  With a workspace the segments are first split on the
// device into a CUDA-core list and a tensor-core list, and every kernel
// walks only its own list with a resident grid; without one (the fixed-
// scratch entry point) the GEMV kernels take every segment.
static int launch_experts(const Ctx& c0, cudaStream_t st, char* ws = nullptr, const WsLayout* L = nullptr,
                          bool classified = false) {
    Ctx c = c0;
    const size_t smem = act_smem(c.H, c.I);
    int rc = allow_smem(gateup_kernel, smem);
    if (rc) return rc;
    if ((rc = allow_smem(down_kernel, smem))) return rc;
    int g_items = gateup_items(c), d_items = down_items(c);
    if (ws) {
        c.seg_list = reinterpret_cast<int32_t*>(ws + L->seg_list);
        c.seg_count = reinterpret_cast<int32_t*>(ws + L->seg_count);
        if (!classified && (rc = launch_pdl(classify_kernel, 1, 32, 0, st, c))) return rc;
        const int rg = resident_grid(gateup_kernel, kThreads, smem);
        const int rd = resident_grid(down_kernel, kThreads, smem);
        g_items = g_items < rg ? g_items : rg;
        d_items = d_items < rd ? d_items : rd;
    }
    const bool tc = c.tc_threshold > 0 && ws != nullptr;
    const bool all_tc = tc && c.tc_threshold == 1;  // the CUDA-core list is empty
    SgParams sg_gate, sg_down;
    size_t sg_gate_smem = 0, sg_down_smem = 0;
    const bool streamed = ws != nullptr && stream_plan(c, 1, sg_gate, sg_gate_smem) &&
                          stream_plan(c, 0, sg_down, sg_down_smem);
    if (tc && (rc = launch_tc(c, ws, *L, st))) return rc;
    if (!all_tc) {
        rc = streamed ? launch_stream(sg_gate, sg_gate_smem, st)
                      : launch_pdl(gateup_kernel, g_items, kThreads, smem, st, c);
        if (rc) return rc;
    }
    if (tc && (rc = launch_tc_down(c, ws, *L, st))) return rc;
    if (!all_tc) {
        rc = streamed ? launch_stream(sg_down, sg_down_smem, st)
                      : launch_pdl(down_kernel, d_items, kThreads, smem, st, c);
        if (rc) return rc;
    }
    return launch_pdl(combine_kernel, combine_items(c), kThreads, 0, st, c);
}

static int launch_unfused_layer(const Ctx& c, cudaStream_t st, char* ws, const WsLayout& L) {
    int rc;
    if (ws) {
        // router; then top-k + grouping + classification in one CTA, or for
        // larger batches the top-k on its own and grouping + classification
        Ctx cc = c;
        cc.seg_list = reinterpret_cast<int32_t*>(ws + L.seg_list);
        cc.seg_count = reinterpret_cast<int32_t*>(ws + L.seg_count);
        const size_t smem = group_smem_bytes(c.B, c.E);
        if (c.B <= kRouteTailMaxB) {
            if ((rc = launch_router(c, st))) return rc;
            if ((rc = allow_smem(route_tail_kernel, smem))) return rc;
            if ((rc = launch_pdl(route_tail_kernel, 1, kRouteTailThreads, smem, st, cc))) return rc;
        } else {
            if ((rc = launch_route(c, st))) return rc;
            if ((rc = allow_smem(group_classify_kernel, smem))) return rc;
            if ((rc = launch_pdl(group_classify_kernel, 1, kRouteTailThreads, smem, st, cc))) return rc;
        }
        return launch_experts(c, st, ws, &L, true);
    }
    rc = launch_route(c, st);
    if (rc) return rc;
    rc = launch_group(c.ids, c.B, c.k, c.E, c.offsets, c.route_idx, c.unique, c.num_unique, c.status, st);
    if (rc) return rc;
    return launch_experts(c, st, ws, &L);
}

static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

static int launch_fused(const Ctx& c, const StackArgs& sa, unsigned* bar, cudaStream_t st) {
    const size_t smem = fused_smem(c.B, c.H, c.I, c.E);
    int rc = allow_smem(fused_kernel, smem);
    if (rc) return rc;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_kernel, kThreads, smem) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int sms = sm_count();
    if (per_sm < 1 || sms < 1) return MOE_ERR_UNSUPPORTED;
    if (per_sm > 2) per_sm = 2;
    if ((rc = to_status(cudaMemsetAsync(bar, 0, 2 * sizeof(unsigned), st)))) return rc;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(sms * per_sm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_ex(cfg, fused_kernel, c, sa, bar);
}


// ------------------------------------------------------ decode kernel plan
// The decode kernel keeps x [B,H], h [R,I], the combine outputs and the next
// router's column slice in shared memory and gives the rest to the weight
// ring; it applies when B <= 4, B*k <= 32 and the ring gets >= 4 stages.
static bool decode_plan(int B, int H, int I, int E, int k, int sms, DkParams& p, size_t& smem, bool norm = false,
                        int w2 = 4) {
    const int R = B * k;
    if (B < 1 || B > kDkMaxB || R > kDkMaxR || sms < 1 || sms > 1024) return false;
    const int ng = H >> 3;
    const int maxrows = 8 * ((ng + sms - 1) / sms);
    size_t off = 1024;  // ring barriers (2 x kDkMaxStages) and the direct-mode barriers
    p.off_misc = (int)off;
    off = align_up(off + sizeof(DkMisc) + sizeof(float) * (size_t)B * ((E + 7) & ~7), 128);
    p.off_x = (int)off;
    off = align_up(off + sizeof(float) * (size_t)B * H, 128);
    p.off_xq = (int)off;
    off = align_up(off + sizeof(float) * (size_t)B * dk_hq(H), 128);
    p.off_h = (int)off;
    off = align_up(off + sizeof(float) * (size_t)R * I, 128);
    p.off_o = (int)off;
    off = align_up(off + sizeof(float) * (size_t)R * maxrows, 128);
    p.off_wr = (int)off;
    off = align_up(off + sizeof(uint16_t) * (size_t)E * maxrows, 128);
    p.off_gq = (int)off;  // pre-norm stacks: two layers' norm weights
    if (norm) off = align_up(off + 2 * sizeof(float) * (size_t)H, 128);
    p.off_ring = (int)off;
    // a stage holds one gate/up row pair or a block of down rows (w2 bytes per
    // two weights: 4 bf16, 2 E4M3, 1 E2M1)
    const size_t stage = align_up((size_t)(2 * H > I ? (size_t)w2 * H : ((size_t)w2 * I) >> 1), 128);
    if (off >= (size_t)kDkSmemMax) return false;
    size_t S = ((size_t)kDkSmemMax - off) / stage;
    if (S > (size_t)kDkMaxStages) S = kDkMaxStages;
    if (S < 4) return false;
    // stage s is always consumed by warp s % W, so S must be a multiple of W
    const size_t W = S < (size_t)kDkConsumers ? S : (size_t)kDkConsumers;
    S = W * (S / W);
    p.W = (int)W;
    p.S = (int)S;
    p.stage_bytes = (int)stage;
    p.maxrows = maxrows;
    smem = off + S * stage;
    return true;
}

// Expert weight formats of the decode kernel.
enum DkFormat { kDkBf16 = 0, kDkFp8Block = 1, kDkNvfp4 = 2 };

static int launch_decode(DkParams& p, size_t smem, int sms, char* ws, const WsLayout& L, cudaStream_t st,
                         int fmt = kDkBf16) {
    // direct mode for every layer: a CTA's largest share -- ceil(U*I/G) gate/up
    // pairs and maxrows down rows of U experts, U <= R -- fits in the ring area
    const size_t w2 = fmt == kDkNvfp4 ? 1 : (fmt == kDkFp8Block ? 2 : 4);  // bytes of two weights
    const size_t Ru = (size_t)p.B * p.k;
    const size_t g_max = ((Ru * p.I + sms - 1) / sms) * w2 * (size_t)p.H;
    const size_t d_max = (Ru * p.maxrows * w2 * (size_t)p.I) >> 1;
    const bool all_direct = g_max + d_max <= (size_t)p.S * p.stage_bytes && g_max < (1u << 20) && d_max < (1u << 20);
    void (*kernel)(DkParams);
    if (fmt == kDkNvfp4) {  // NVFP4 experts (no traced variant)
        if (p.B == 1 && all_direct)
            kernel = decode_kernel<false, 1, true, false, true>;
        else if (p.B == 1)
            kernel = decode_kernel<false, 1, false, false, true>;
        else
            kernel = decode_kernel<false, 4, false, false, true>;
    } else if (fmt == kDkFp8Block) {  // block-scaled FP8 experts (no traced variant)
        if (p.B == 1 && all_direct)
            kernel = decode_kernel<false, 1, true, true>;
        else if (p.B == 1)
            kernel = decode_kernel<false, 1, false, true>;
        else
            kernel = decode_kernel<false, 4, false, true>;
    } else if (p.B == 1 && all_direct)
        kernel = p.trace ? decode_kernel<true, 1, true> : decode_kernel<false, 1, true>;
    else if (p.B == 1)
        kernel = p.trace ? decode_kernel<true, 1, false> : decode_kernel<false, 1, false>;
    else
        kernel = p.trace ? decode_kernel<true, 4, false> : decode_kernel<false, 4, false>;
    int rc = allow_smem(kernel, smem);
    if (rc) return rc;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kDkThreads, smem) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (per_sm < 1) return MOE_ERR_UNSUPPORTED;
    p.h = reinterpret_cast<float*>(ws + L.h);
    p.xt = reinterpret_cast<unsigned long long*>(ws + L.xt);
    p.alog = reinterpret_cast<float*>(ws + L.alog);
    // next-layer L2 prefetch: single-token decode, the top k experts of the
    // predicted logits while that stays within 64 MB of weights (a stack
    // only: L > 1).  (Measured on the 30-layer stack: top k beats top k+1,
    // whose extra expert costs more HBM time than its hits save.)
    p.prefetch_k = 0;
    if (p.B == 1 && p.L > 1 && !(p.flags & MOE_F_NO_PREFETCH)) {
        const unsigned long long per_e = (3ull * w2 * p.I * p.H) >> 1;
        const int kp = p.k;
        if (per_e * kp <= (64ull << 20) && kp <= 32) p.prefetch_k = kp;
    }
    p.acc = reinterpret_cast<unsigned long long*>(ws + L.acc);
    p.bar = reinterpret_cast<unsigned*>(ws + L.bar);
    p.g_offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    p.g_route_idx = reinterpret_cast<int32_t*>(ws + L.route_idx);
    p.g_unique = reinterpret_cast<int32_t*>(ws + L.unique);
    p.g_num_unique = reinterpret_cast<int32_t*>(ws + L.num_unique);
    // the count field of a logit word holds at most 127 contributions
    static_assert(kDkShadows == 2, "workspace accumulator sets are sized for two shadow copies");
    if (sms > 127 * kDkShadows) return MOE_ERR_UNSUPPORTED;
    if ((rc = to_status(cudaMemsetAsync(ws + L.bar, 0, L.acc_end - L.bar, st)))) return rc;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(kDkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_ex(cfg, kernel, p);
}

static unsigned long long* g_trace = nullptr;
static int g_trace_words = 0;
static unsigned g_bar_extra = 0;  // moe_inject_barrier_stall

static void decode_common(DkParams& p, int B, int H, int I, int E, int k, int L, unsigned flags,
                          int32_t* status) {
    p.trace = g_trace;
    p.trace_words = g_trace_words;
    p.B = B;
    p.H = H;
    p.I = I;
    p.E = E;
    p.k = k;
    p.L = L;
    p.flags = flags;
    p.status = status;
    p.bar_extra = g_bar_extra;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_workspace_bytes(int B, int H, int I, int E, int top_k, size_t* bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    const int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    *bytes = ws_layout(B, H, I, E, top_k).total;
    return MOE_OK;
}

int moe_route(const void* x, int x_dtype, const uint16_t* w_router, const float* logit_bias, int B,
              int H, int E, int top_k, int32_t* expert_ids, float* route_w, float* logits_out,
              void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
    int rc = check_dims(B, H, 8, E, top_k, false);
    if (rc) return rc;
    if (x_dtype != MOE_DT_F32 && x_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
    if (B == 0) return MOE_OK;  // nothing to do; empty tensors may carry null pointers
    MOE_REQ(x);
    MOE_REQ(w_router);
    MOE_REQ(expert_ids);
    MOE_REQ(route_w);
    MOE_OPT(logit_bias);
    MOE_OPT(logits_out);
    MOE_OPT(workspace);
    MOE_OPT(dev_status);
    const WsLayout L = ws_layout(B, H, 8, E, top_k);
    if (!logits_out && (!workspace || workspace_bytes < L.logits + sizeof(float) * (size_t)B * E))
        return MOE_ERR_WORKSPACE;
    Ctx c = make_ctx(x, x_dtype, nullptr, nullptr, B, H, 8, E, top_k, 0, nullptr, L, dev_status);
    c.w.w_router = w_router;
    c.w.bias = logit_bias;
    c.logits = logits_out ? logits_out : reinterpret_cast<float*>(static_cast<char*>(workspace) + L.logits);
    c.ids = expert_ids;
    c.rw = route_w;
    return launch_route(c, static_cast<cudaStream_t>(stream));
}

int moe_group_by_expert(const int32_t* expert_ids, int B, int top_k, int E, int32_t* offsets,
                        int32_t* route_idx, int32_t* unique_experts, int32_t* num_unique,
                        int32_t* dev_status, void* stream) {
    int rc = check_dims(B, 8, 8, E, top_k, false);
    if (rc) return rc;
    if (B == 0) return MOE_OK;
    MOE_REQ(expert_ids);
    MOE_REQ(offsets);
    MOE_REQ(route_idx);
    MOE_REQ(unique_experts);
    MOE_REQ(num_unique);
    MOE_OPT(dev_status);
    return launch_group(expert_ids, B, top_k, E, offsets, route_idx, unique_experts, num_unique, dev_status,
                        static_cast<cudaStream_t>(stream));
}

int moe_expert_forward(const void* x, int x_dtype, const uint16_t* gate_up, const uint16_t* down,
                       const int32_t* expert_ids, const float* route_w, const int32_t* offsets,
                       const int32_t* route_idx, const int32_t* unique_experts,
                       const int32_t* num_unique, int B, int H, int I, int E, int top_k,
                       const float* residual, float* y, uint32_t flags, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, void* stream) {
    int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (x_dtype != MOE_DT_F32 && x_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
    if (flags & ~kAllFlags) return MOE_ERR_INVALID_ARG;
    if (B == 0) return MOE_OK;
    MOE_REQ(x);
    MOE_REQ(gate_up);
    MOE_REQ(down);
    MOE_REQ(expert_ids);
    MOE_REQ(route_w);
    MOE_REQ(offsets);
    MOE_REQ(route_idx);
    MOE_REQ(unique_experts);
    MOE_REQ(num_unique);
    MOE_REQ(y);
    MOE_OPT(residual);
    MOE_REQ(workspace);
    MOE_OPT(dev_status);
    const WsLayout L = ws_layout(B, H, I, E, top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    Ctx c = make_ctx(x, x_dtype, residual, y, B, H, I, E, top_k, flags, static_cast<char*>(workspace), L,
                     dev_status);
    c.ids = const_cast<int32_t*>(expert_ids);
    c.rw = const_cast<float*>(route_w);
    c.offsets = const_cast<int32_t*>(offsets);
    c.route_idx = const_cast<int32_t*>(route_idx);
    c.unique = const_cast<int32_t*>(unique_experts);
    c.num_unique = const_cast<int32_t*>(num_unique);
    c.w.gate_up = gate_up;
    c.w.down = down;
    return launch_experts(c, static_cast<cudaStream_t>(stream), static_cast<char*>(workspace), &L);
}

int moe_layer_forward(const void* x, int x_dtype, const uint16_t* w_router, const float* logit_bias,
                      const uint16_t* gate_up, const uint16_t* down, int B, int H, int I, int E,
                      int top_k, const float* residual, float* y, int32_t* expert_ids_out,
                      float* route_w_out, uint32_t flags, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream) {
    int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (x_dtype != MOE_DT_F32 && x_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
    if (flags & ~kAllFlags) return MOE_ERR_INVALID_ARG;
    if (B == 0) return MOE_OK;
    MOE_REQ(x);
    MOE_REQ(w_router);
    MOE_REQ(gate_up);
    MOE_REQ(down);
    MOE_REQ(y);
    MOE_OPT(logit_bias);
    MOE_OPT(residual);
    MOE_OPT(expert_ids_out);
    MOE_OPT(route_w_out);
    MOE_REQ(workspace);
    MOE_OPT(dev_status);
    const WsLayout L = ws_layout(B, H, I, E, top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    Ctx c = make_ctx(x, x_dtype, residual, y, B, H, I, E, top_k, flags, ws, L, dev_status);
    c.w.w_router = w_router;
    c.w.bias = logit_bias;
    c.w.gate_up = gate_up;
    c.w.down = down;
    if (expert_ids_out) c.ids = expert_ids_out;
    if (route_w_out) c.rw = route_w_out;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (flags & MOE_F_UNFUSED) return launch_unfused_layer(c, st, ws, L);
    {
        DkParams dp;
        memset(&dp, 0, sizeof dp);
        size_t dsm = 0;
        const int sms = sm_count();
        if (decode_plan(B, H, I, E, top_k, sms, dp, dsm)) {
            decode_common(dp, B, H, I, E, top_k, 1, flags, c.status);
            dp.x_bf16 = x_dtype == MOE_DT_BF16;
            dp.x_in = x;
            dp.residual = residual;
            dp.y = y;
            dp.layer[0] = c.w;
            dp.ids_out = c.ids;
            dp.w_out = c.rw;
            return launch_decode(dp, dsm, sms, ws, L, st);
        }
    }
    if (c.tc_threshold > 0) return launch_unfused_layer(c, st, ws, L);  // grouped GEMMs need their own grids
    StackArgs sa;
    memset(&sa, 0, sizeof sa);
    sa.L = 1;
    sa.bar_extra = g_bar_extra;
    sa.layer[0] = c.w;
    sa.ids_out = nullptr;
    return launch_fused(c, sa, reinterpret_cast<unsigned*>(ws + L.bar), st);
}

int moe_stack_forward(int Lc, const uint16_t* const* w_router, const float* const* logit_bias,
                      const uint16_t* const* gate_up, const uint16_t* const* down, int B, int H,
                      int I, int E, int top_k, float* x_inout, int32_t* expert_ids_out,
                      uint32_t flags, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream) {
    int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (Lc < 1 || Lc > MOE_MAX_LAYERS) return MOE_ERR_INVALID_ARG;
    if (flags & ~kAllFlags) return MOE_ERR_INVALID_ARG;
    if (B == 0) return MOE_OK;
    if (!w_router || !gate_up || !down) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < Lc; ++l) {
        MOE_REQ(w_router[l]);
        MOE_REQ(gate_up[l]);
        MOE_REQ(down[l]);
        if (logit_bias) MOE_OPT(logit_bias[l]);
    }
    MOE_REQ(x_inout);
    MOE_OPT(expert_ids_out);
    MOE_REQ(workspace);
    MOE_OPT(dev_status);
    const WsLayout L = ws_layout(B, H, I, E, top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    Ctx c = make_ctx(x_inout, MOE_DT_F32, x_inout, x_inout, B, H, I, E, top_k, flags, ws, L, dev_status);
    StackArgs sa;
    memset(&sa, 0, sizeof sa);
    sa.L = Lc;
    sa.bar_extra = g_bar_extra;
    sa.ids_out = expert_ids_out;
    for (int l = 0; l < Lc; ++l) {
        sa.layer[l].w_router = w_router[l];
        sa.layer[l].bias = logit_bias ? logit_bias[l] : nullptr;
        sa.layer[l].gate_up = gate_up[l];
        sa.layer[l].down = down[l];
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (flags & MOE_F_UNFUSED) {
        int32_t* ids_ws = c.ids;
        for (int l = 0; l < Lc; ++l) {
            c.w = sa.layer[l];
            c.ids = expert_ids_out ? expert_ids_out + (size_t)l * B * top_k : ids_ws;
            if ((rc = launch_unfused_layer(c, st, ws, L))) return rc;
        }
        return MOE_OK;
    }
    {
        DkParams dp;
        memset(&dp, 0, sizeof dp);
        size_t dsm = 0;
        const int sms = sm_count();
        if (decode_plan(B, H, I, E, top_k, sms, dp, dsm)) {
            decode_common(dp, B, H, I, E, top_k, Lc, flags, c.status);
            dp.x_bf16 = 0;
            dp.x_in = x_inout;
            dp.residual = x_inout;
            dp.y = x_inout;
            for (int l = 0; l < Lc; ++l) dp.layer[l] = sa.layer[l];
            dp.ids_out = expert_ids_out;
            dp.w_out = nullptr;
            return launch_decode(dp, dsm, sms, ws, L, st);
        }
    }
    if (c.tc_threshold > 0) {  // grouped GEMMs need their own grids: one sequence per layer
        int32_t* ids_ws = c.ids;
        for (int l = 0; l < Lc; ++l) {
            c.w = sa.layer[l];
            c.ids = expert_ids_out ? expert_ids_out + (size_t)l * B * top_k : ids_ws;
            if ((rc = launch_unfused_layer(c, st, ws, L))) return rc;
        }
        return MOE_OK;
    }
    return launch_fused(c, sa, reinterpret_cast<unsigned*>(ws + L.bar), st);
}

int moe_stack_forward_norm(int Lc, const uint16_t* const* w_router, const float* const* logit_bias,
                           const uint16_t* const* gate_up, const uint16_t* const* down, const float* const* norm_w,
                           float eps, int B, int H, int I, int E, int top_k, float* x_inout,
                           int32_t* expert_ids_out, uint32_t flags, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream) {
    int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (Lc < 1 || Lc > MOE_MAX_LAYERS) return MOE_ERR_INVALID_ARG;
    if (flags & ~kAllFlags) return MOE_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || eps > 1.f) return MOE_ERR_INVALID_ARG;  // rejects NaN too
    if (B == 0) return MOE_OK;
    if (!w_router || !gate_up || !down || !norm_w) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < Lc; ++l) {
        MOE_REQ(w_router[l]);
        MOE_REQ(gate_up[l]);
        MOE_REQ(down[l]);
        MOE_REQ(norm_w[l]);
        if (logit_bias) MOE_OPT(logit_bias[l]);
    }
    MOE_REQ(x_inout);
    MOE_OPT(expert_ids_out);
    MOE_REQ(workspace);
    MOE_OPT(dev_status);
    const WsLayout L = ws_layout(B, H, I, E, top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    LayerWeights lws[MOE_MAX_LAYERS];
    memset(lws, 0, sizeof lws);  // bf16 experts: no FP8 or NVFP4 scales
    for (int l = 0; l < Lc; ++l) {
        lws[l].w_router = w_router[l];
        lws[l].bias = logit_bias ? logit_bias[l] : nullptr;
        lws[l].gate_up = gate_up[l];
        lws[l].down = down[l];
        lws[l].norm = norm_w[l];
    }
    if (!(flags & MOE_F_UNFUSED)) {
        // small batches: the norm fused into the decode kernel's router and
        // residual add (one launch for the whole stack)
        DkParams dp;
        memset(&dp, 0, sizeof dp);
        size_t dsm = 0;
        const int sms = sm_count();
        if (decode_plan(B, H, I, E, top_k, sms, dp, dsm, true)) {
            decode_common(dp, B, H, I, E, top_k, Lc, flags, dev_status ? dev_status
                                                                       : reinterpret_cast<int32_t*>(ws + L.status));
            dp.x_bf16 = 0;
            dp.x_in = x_inout;
            dp.residual = x_inout;
            dp.y = x_inout;
            for (int l = 0; l < Lc; ++l) dp.layer[l] = lws[l];
            dp.ids_out = expert_ids_out;
            dp.w_out = nullptr;
            dp.has_norm = 1;
            dp.eps = eps;
            return launch_decode(dp, dsm, sms, ws, L, st);
        }
    }
    // otherwise layer by layer: the norm into the workspace, then the layer on
    // it with the raw input as the residual (y aliases the residual)
    float* xn = reinterpret_cast<float*>(ws + L.xn);
    Ctx c = make_ctx(xn, MOE_DT_F32, x_inout, x_inout, B, H, I, E, top_k, flags, ws, L, dev_status);
    int32_t* ids_ws = c.ids;
    for (int l = 0; l < Lc; ++l) {
        if ((rc = launch_pdl(rmsnorm_kernel, B, kThreads, 0, st, (const float*)x_inout, norm_w[l], H, eps, xn))) return rc;
        c.w = lws[l];
        c.ids = expert_ids_out ? expert_ids_out + (size_t)l * B * top_k : ids_ws;
        if ((flags & MOE_F_UNFUSED) || c.tc_threshold > 0) {
            if ((rc = launch_unfused_layer(c, st, ws, L))) return rc;
        } else {
            StackArgs sa;
            memset(&sa, 0, sizeof sa);
            sa.L = 1;
            sa.bar_extra = g_bar_extra;
            sa.layer[0] = c.w;
            sa.ids_out = c.ids;
            if ((rc = launch_fused(c, sa, reinterpret_cast<unsigned*>(ws + L.bar), st))) return rc;
        }
    }
    return MOE_OK;
}

int moe_stack_forward_fp8(int Lc, const uint16_t* const* w_router, const float* const* logit_bias,
                          const uint8_t* const* gate_up_q, const float* const* gate_up_scale,
                          const uint8_t* const* down_q, const float* const* down_scale, int B, int H, int I, int E,
                          int top_k, float* x_inout, int32_t* expert_ids_out, uint32_t flags, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, void* stream) {
    int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (Lc < 1 || Lc > MOE_MAX_LAYERS) return MOE_ERR_INVALID_ARG;
    if ((H & 15) || (I & 15)) return MOE_ERR_INVALID_ARG;  // rows of codes in whole 16-byte pieces
    if (flags & ~(MOE_F_NO_DEDUP | MOE_F_NO_PREFETCH | MOE_F_UNFUSED)) return MOE_ERR_INVALID_ARG;
    if (B == 0) return MOE_OK;
    if (!w_router || !gate_up_q || !gate_up_scale || !down_q || !down_scale) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < Lc; ++l) {
        MOE_REQ(w_router[l]);
        MOE_REQ(gate_up_q[l]);
        MOE_REQ(down_q[l]);
        if (!gate_up_scale[l] || !down_scale[l]) return MOE_ERR_INVALID_ARG;
        if (logit_bias) MOE_OPT(logit_bias[l]);
    }
    MOE_REQ(x_inout);
    MOE_OPT(expert_ids_out);
    MOE_REQ(workspace);
    MOE_OPT(dev_status);
    const WsLayout L = ws_layout(B, H, I, E, top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    DkParams dp;
    memset(&dp, 0, sizeof dp);
    size_t dsm = 0;
    const int sms = sm_count();
    if ((flags & MOE_F_UNFUSED) || !decode_plan(B, H, I, E, top_k, sms, dp, dsm, false, 2)) {
        // Batches beyond the decode kernel: the CUDA-core phase kernels, whose
        // gate/up and down items read the E4M3 codes with their block scales
        // (the tensor-core GEMMs take bf16 weights only), layer by layer --
        // 16-20 % faster than the whole stack in one cooperative launch here.
        Ctx c = make_ctx(x_inout, MOE_DT_F32, x_inout, x_inout, B, H, I, E, top_k, flags | MOE_F_NO_TC, ws, L,
                         dev_status);
        StackArgs sa;
        memset(&sa, 0, sizeof sa);
        sa.L = Lc;
        sa.bar_extra = g_bar_extra;
        sa.ids_out = expert_ids_out;
        for (int l = 0; l < Lc; ++l) {
            sa.layer[l].w_router = w_router[l];
            sa.layer[l].bias = logit_bias ? logit_bias[l] : nullptr;
            sa.layer[l].gate_up = reinterpret_cast<const uint16_t*>(gate_up_q[l]);
            sa.layer[l].down = reinterpret_cast<const uint16_t*>(down_q[l]);
            sa.layer[l].gate_up_scale = gate_up_scale[l];
            sa.layer[l].down_scale = down_scale[l];
        }
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        int32_t* ids_ws = c.ids;
        for (int l = 0; l < Lc; ++l) {
            c.w = sa.layer[l];
            c.ids = expert_ids_out ? expert_ids_out + (size_t)l * B * top_k : ids_ws;
            if ((rc = launch_unfused_layer(c, st, ws, L))) return rc;
        }
        return MOE_OK;
    }
    decode_common(dp, B, H, I, E, top_k, Lc, flags,
                  dev_status ? dev_status : reinterpret_cast<int32_t*>(ws + L.status));
    dp.trace = nullptr;
    dp.trace_words = 0;
    dp.x_bf16 = 0;
    dp.x_in = x_inout;
    dp.residual = x_inout;
    dp.y = x_inout;
    for (int l = 0; l < Lc; ++l) {
        dp.layer[l].w_router = w_router[l];
        dp.layer[l].bias = logit_bias ? logit_bias[l] : nullptr;
        dp.layer[l].gate_up = reinterpret_cast<const uint16_t*>(gate_up_q[l]);
        dp.layer[l].down = reinterpret_cast<const uint16_t*>(down_q[l]);
        dp.layer[l].gate_up_scale = gate_up_scale[l];
        dp.layer[l].down_scale = down_scale[l];
    }
    dp.ids_out = expert_ids_out;
    dp.w_out = nullptr;
    return launch_decode(dp, dsm, sms, ws, L, static_cast<cudaStream_t>(stream), kDkFp8Block);
}

int moe_stack_forward_nvfp4(int Lc, const uint16_t* const* w_router, const float* const* logit_bias,
                            const uint8_t* const* gate_up_q, const uint8_t* const* gate_up_bs,
                            const float* const* gate_up_gs, const uint8_t* const* down_q,
                            const uint8_t* const* down_bs, const float* const* down_gs, int B, int H, int I, int E,
                            int top_k, float* x_inout, int32_t* expert_ids_out, uint32_t flags, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream) {
    int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (Lc < 1 || Lc > MOE_MAX_LAYERS) return MOE_ERR_INVALID_ARG;
    if ((H & 31) || (I & 31)) return MOE_ERR_INVALID_ARG;  // rows of codes in whole 16-byte pieces
    if (flags & ~(MOE_F_NO_DEDUP | MOE_F_NO_PREFETCH | MOE_F_UNFUSED)) return MOE_ERR_INVALID_ARG;
    if (B == 0) return MOE_OK;
    if (!w_router || !gate_up_q || !gate_up_bs || !gate_up_gs || !down_q || !down_bs || !down_gs)
        return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < Lc; ++l) {
        MOE_REQ(w_router[l]);
        MOE_REQ(gate_up_q[l]);
        MOE_REQ(down_q[l]);
        if (!gate_up_bs[l] || !down_bs[l] || !gate_up_gs[l] || !down_gs[l]) return MOE_ERR_INVALID_ARG;
        if (logit_bias) MOE_OPT(logit_bias[l]);
    }
    MOE_REQ(x_inout);
    MOE_OPT(expert_ids_out);
    MOE_REQ(workspace);
    MOE_OPT(dev_status);
    const WsLayout L = ws_layout(B, H, I, E, top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    DkParams dp;
    memset(&dp, 0, sizeof dp);
    size_t dsm = 0;
    const int sms = sm_count();
    if ((flags & MOE_F_UNFUSED) || !decode_plan(B, H, I, E, top_k, sms, dp, dsm, false, 1)) {
        // beyond the decode kernel: the CUDA-core phase kernels layer by
        // layer, their items reading the E2M1 codes with both scales
        Ctx c = make_ctx(x_inout, MOE_DT_F32, x_inout, x_inout, B, H, I, E, top_k, flags | MOE_F_NO_TC, ws, L,
                         dev_status);
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        int32_t* ids_ws = c.ids;
        for (int l = 0; l < Lc; ++l) {
            memset(&c.w, 0, sizeof c.w);
            c.w.w_router = w_router[l];
            c.w.bias = logit_bias ? logit_bias[l] : nullptr;
            c.w.gate_up = reinterpret_cast<const uint16_t*>(gate_up_q[l]);
            c.w.down = reinterpret_cast<const uint16_t*>(down_q[l]);
            c.w.gate_up_bs = gate_up_bs[l];
            c.w.down_bs = down_bs[l];
            c.w.gate_up_gs = gate_up_gs[l];
            c.w.down_gs = down_gs[l];
            c.ids = expert_ids_out ? expert_ids_out + (size_t)l * B * top_k : ids_ws;
            if ((rc = launch_unfused_layer(c, st, ws, L))) return rc;
        }
        return MOE_OK;
    }
    decode_common(dp, B, H, I, E, top_k, Lc, flags,
                  dev_status ? dev_status : reinterpret_cast<int32_t*>(ws + L.status));
    dp.trace = nullptr;
    dp.trace_words = 0;
    dp.x_bf16 = 0;
    dp.x_in = x_inout;
    dp.residual = x_inout;
    dp.y = x_inout;
    for (int l = 0; l < Lc; ++l) {
        dp.layer[l].w_router = w_router[l];
        dp.layer[l].bias = logit_bias ? logit_bias[l] : nullptr;
        dp.layer[l].gate_up = reinterpret_cast<const uint16_t*>(gate_up_q[l]);
        dp.layer[l].down = reinterpret_cast<const uint16_t*>(down_q[l]);
        dp.layer[l].gate_up_bs = gate_up_bs[l];
        dp.layer[l].down_bs = down_bs[l];
        dp.layer[l].gate_up_gs = gate_up_gs[l];
        dp.layer[l].down_gs = down_gs[l];
    }
    dp.ids_out = expert_ids_out;
    dp.w_out = nullptr;
    return launch_decode(dp, dsm, sms, ws, L, static_cast<cudaStream_t>(stream), kDkNvfp4);
}

int moe_workspace_grouping(void* workspace, size_t workspace_bytes, int B, int H, int I, int E, int top_k,
                           int32_t** offsets, int32_t** route_idx, int32_t** unique_experts,
                           int32_t** num_unique) {
    const int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (!workspace || !offsets || !route_idx || !unique_experts || !num_unique) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(B, H, I, E, top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    *offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    *route_idx = reinterpret_cast<int32_t*>(ws + L.route_idx);
    *unique_experts = reinterpret_cast<int32_t*>(ws + L.unique);
    *num_unique = reinterpret_cast<int32_t*>(ws + L.num_unique);
    return MOE_OK;
}

unsigned long long moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_forward_path(int B, int H, int I, int E, int top_k, int L, uint32_t flags, int* path, int* grid) {
    int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (!path || L < 1 || L > MOE_MAX_LAYERS || (flags & ~kAllFlags)) return MOE_ERR_INVALID_ARG;
    int g = 0;
    if (B == 0) {
        *path = 0;
    } else if (flags & MOE_F_UNFUSED) {
        *path = MOE_PATH_PHASES;
    } else {
        DkParams dp;
        size_t dsm = 0;
        const int sms = sm_count();
        if (decode_plan(B, H, I, E, top_k, sms, dp, dsm)) {
            *path = MOE_PATH_DECODE;
            g = sms;
        } else if (tc_threshold_for(flags, H, I) > 0) {
            *path = MOE_PATH_PHASES;
        } else {
            *path = MOE_PATH_FUSED;
        }
    }
    if (grid) *grid = g;
    return MOE_OK;
}

int moe_inject_barrier_stall(int extra_arrivals) {
    if (extra_arrivals < 0 || extra_arrivals > 1024) return MOE_ERR_INVALID_ARG;
    g_bar_extra = (unsigned)extra_arrivals;
    return MOE_OK;
}

int moe_set_trace_buffer(unsigned long long* trace, int words) {
    if ((trace == nullptr) != (words == 0) || words < 0) return MOE_ERR_INVALID_ARG;
    g_trace = trace;
    g_trace_words = words;
    return MOE_OK;
}

const char* moe_status_string(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument (shape, limit, null or misaligned pointer)";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration on this device";
        case MOE_ERR_CUDA: return "CUDA launch or runtime error";
        case MOE_ERR_WORKSPACE: return "workspace missing or smaller than moe_workspace_bytes()";
        case MOE_DEV_TIMEOUT: return "device: a grid barrier timed out";
        case MOE_DEV_BAD_EXPERT_ID: return "device: expert id outside [0, E)";
        case MOE_DEV_DUP_EXPERT: return "device: a token lists the same expert twice";
        case MOE_DEV_NONFINITE: return "device: non-finite router logit";
        case MOE_DEV_BAD_ROUTE: return "device: route index outside [0, B*top_k)";
        case MOE_DEV_RANGE: return "device: router partial sum beyond the fixed-point range (+-2^21)";
        default: return "unknown status";
    }
}

}  // extern "C"

// ----------------------------------------------------------------------------
// moe_expert_forward_noalloc: moe_expert_forward with its scratch (the
// intermediate h [R, I] and the per-route outputs o [R, H], fp32) in a fixed
// device array owned by the library, for callers that cannot allocate device
// memory: code running inside a CUDA graph that is being captured or
// replayed, an allocator hook that must not re-enter the allocator, or an
// embedding runtime whose memory budget is fixed up front.
//
// The array below is a file-scope __device__ array of MOE_NOALLOC_SCRATCH_BYTES
// (16 MiB); every GPU that loads the library holds it until the process exits.
// In host code its name is only a host-side stand-in, so the entry point looks
// up its device address with cudaGetSymbolAddress once per device (on the
// first call made with that device current) and hands that address to the
// kernels.
namespace moe {

__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static void* g_noalloc_ptr[kMaxDevices];
static std::mutex g_noalloc_mu;

static int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

}  // namespace moe

extern "C" int moe_expert_forward_noalloc(const void* x, int x_dtype, const uint16_t* gate_up,
                                          const uint16_t* down, const int32_t* expert_ids,
                                          const float* route_w, const int32_t* offsets,
                                          const int32_t* route_idx, const int32_t* unique_experts,
                                          const int32_t* num_unique, int B, int H, int I, int E,
                                          int top_k, const float* residual, float* y, uint32_t flags,
                                          int32_t* dev_status, void* stream) {
    using namespace moe;
    int rc = check_dims(B, H, I, E, top_k, true);
    if (rc) return rc;
    if (x_dtype != MOE_DT_F32 && x_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
    if (flags & ~kAllFlags) return MOE_ERR_INVALID_ARG;
    if (flags & MOE_F_FORCE_TC) return MOE_ERR_UNSUPPORTED;  // no operand buffers for the tensor cores here
    const size_t R = (size_t)B * top_k;
    const size_t h_bytes = align_up(sizeof(float) * R * I, 256);
    if (h_bytes + sizeof(float) * R * H > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
    if (B == 0) return MOE_OK;
    MOE_REQ(x);
    MOE_REQ(gate_up);
    MOE_REQ(down);
    MOE_REQ(expert_ids);
    MOE_REQ(route_w);
    MOE_REQ(offsets);
    MOE_REQ(route_idx);
    MOE_REQ(unique_experts);
    MOE_REQ(num_unique);
    MOE_REQ(y);
    MOE_OPT(residual);
    MOE_OPT(dev_status);
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch))) return rc;
    Ctx c = make_ctx(x, x_dtype, residual, y, B, H, I, E, top_k, flags, nullptr, WsLayout(), dev_status);
    c.ids = const_cast<int32_t*>(expert_ids);
    c.rw = const_cast<float*>(route_w);
    c.offsets = const_cast<int32_t*>(offsets);
    c.route_idx = const_cast<int32_t*>(route_idx);
    c.unique = const_cast<int32_t*>(unique_experts);
    c.num_unique = const_cast<int32_t*>(num_unique);
    c.w.gate_up = gate_up;
    c.w.down = down;
    // every element of h and o is written before it is read, so the array's
    // contents from an earlier call never need clearing
    c.h = static_cast<float*>(scratch);
    c.o = reinterpret_cast<float*>(static_cast<char*>(scratch) + h_bytes);
    return launch_experts(c, static_cast<cudaStream_t>(stream));
}
