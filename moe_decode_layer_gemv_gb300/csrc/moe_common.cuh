// moe_common.cuh -- shared device helpers of the MoE decode library (sm_103a).
//
// Loads: weights are read once per step and never reused by the same SM, so
// they go through the non-coherent path without L1 allocation and with a
// 256-byte L2 prefetch; activations written earlier in the same launch (x of
// a stacked layer, h, logits, ids) are read with ld.global.cg so that no SM
// can see a stale L1 line after a device-wide barrier.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "moe.h"

namespace moe {

constexpr int kThreads = 256;  // threads per CTA in every streaming phase
constexpr int kWarps = kThreads / 32;

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ld_weight_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float4 ld_act_f4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ uint4 ld_act_u4(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ float ld_act_f(const float* p) { return __ldcg(p); }
__device__ __forceinline__ int ld_act_i(const int32_t* p) { return __ldcg(p); }

// two bf16 packed in a 32-bit word -> (low element, high element) as fp32 (exact)
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// An order-preserving unsigned key of a float (a < b as floats, neither NaN
// and not both zeros, iff key(a) < key(b)) and its inverse.
__device__ __forceinline__ unsigned order_key(float f) {
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Two E4M3 codes (low byte first) as fp32: the hardware conversion to f16 is
// exact for every E4M3 value, and so is the widening to f32.
__device__ __forceinline__ float2 f8x2_to_f2(unsigned v) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3);
    __half2 h;
    memcpy(&h, &hr, sizeof h);
    return __half22float2(h);
}

// Two E2M1 codes (one byte, low nibble first) as fp32, and one E4M3 code as
// fp32: the hardware conversions to f16 are exact for every code, and so is
// the widening to f32.
__device__ __forceinline__ float2 f4x2_to_f2(unsigned v) {
    const __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(v & 0xffu), __NV_E2M1);
    __half2 h;
    memcpy(&h, &hr, sizeof h);
    return __half22float2(h);
}

__device__ __forceinline__ float f8_to_f(unsigned v) {
    const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)(v & 0xffu), __NV_E4M3);
    __half h;
    memcpy(&h, &hr, sizeof h);
    return __half2float(h);
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// SiLU(g) * u with SiLU(z) = z / (1 + e^-z), fp32
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Lane-blocked layout of an fp32 activation row in shared memory: the 8
// values of column group g = 32*b + L (columns 8g..8g+7) sit at 256*b + 4*L
// (first four) and 256*b + 128 + 4*L (last four).  A warp that walks the
// groups g = 32*b + lane then loads 512 contiguous bytes with each 16-byte
// load -- one shared-memory wavefront per 128 bytes, where the natural
// layout (a 32-byte lane stride) needs two.  Rows are lb_stride(n) floats
// apart.
__host__ __device__ __forceinline__ int lb_stride(int n) { return (n + 255) & ~255; }

__device__ __forceinline__ int lb_index(int c) {  // column c (a multiple of 4) -> its float4
    const int g = c >> 3;
    return ((g >> 5) << 8) + ((c >> 2) & 1) * 128 + ((g & 31) << 2);
}

// first float of column group v (8 columns) in a lane-blocked row; the other
// four are 128 floats further
__device__ __forceinline__ int lb_group(int v) { return ((v >> 5) << 8) + ((v & 31) << 2); }

__device__ __forceinline__ void set_status(int32_t* status, int bits) {
    if (status) atomicOr(status, bits);
}

// ------------------------------------------------------------ problem view
struct LayerWeights {
    const uint16_t* w_router;  // [E, H]
    const float* bias;         // [E] or nullptr
    const uint16_t* gate_up;   // [E, 2I, H]
    const uint16_t* down;      // [E, H, I]
    const float* norm;         // [H] RMSNorm weights of the layer input (pre-norm stacks), or nullptr
    // block-scaled FP8 experts (gate_up / down then hold E4M3 codes, one byte
    // each): fp32 scales per 128 x 128 block, [E][ceil(2I/128)][ceil(H/128)]
    // and [E][ceil(H/128)][ceil(I/128)]; nullptr for bf16 experts
    const float* gate_up_scale;
    const float* down_scale;
    // NVFP4 experts: E4M3 scales of 16-element row blocks ([E][rows][cols/16]
    // bytes) and one fp32 scale per expert matrix ([E])
    const unsigned char* gate_up_bs;
    const unsigned char* down_bs;
    const float* gate_up_gs;
    const float* down_gs;
};

// Everything one layer step needs.  Built on the host, passed by value.
struct Ctx {
    const void* x;        // [B, H] fp32 or bf16
    int x_bf16;
    const float* residual;  // [B, H] or nullptr
    float* y;               // [B, H]
    LayerWeights w;
    int B, H, I, E, k;
    unsigned flags;
    int nt_max;  // tokens staged per pass in the grouped GEMV phases (1, 2, 4 or 8)
    int tc_threshold;  // segments with at least this many routes go to the tensor-core kernels (0: none)
    // Work lists built on the device by classify_kernel (nullptr: iterate over
    // every segment directly): seg_list[0 .. seg_count[0]) are the segments
    // for the CUDA-core GEMV, seg_list[max_segments .. + seg_count[1]) those
    // for the tensor-core GEMMs; seg_count[2] = routes of the largest
    // tensor-core segment.
    int32_t* seg_list;
    int32_t* seg_count;
    // routing (device)
    float* logits;       // [B, E]
    int32_t* ids;        // [B, k]
    float* rw;           // [B, k]
    int32_t* offsets;    // [E + 1]
    int32_t* route_idx;  // [R]
    int32_t* unique;     // [E]
    int32_t* num_unique; // [1]
    // scratch (device)
    float* h;  // [R, I]  per position in the grouped route list
    float* o;  // [R, H]  per flat route r = t*k + j
    int32_t* status;
};

// A segment is a run of routes that share one expert: one unique expert in
// the grouped list, or (MOE_F_NO_DEDUP) a single route.
struct Seg {
    int e, p0, p1;
};

__host__ __device__ __forceinline__ bool no_dedup(const Ctx& c) { return (c.flags & MOE_F_NO_DEDUP) != 0; }

__host__ __device__ __forceinline__ int max_segments(const Ctx& c) {
    const int R = c.B * c.k;
    return no_dedup(c) ? R : (R < c.E ? R : c.E);
}

__device__ __forceinline__ bool get_seg(const Ctx& c, int s, Seg& sg) {
    if (no_dedup(c)) {
        if (s >= c.B * c.k) return false;
        sg.e = ld_act_i(c.ids + s);
        sg.p0 = s;
        sg.p1 = s + 1;
    } else {
        // a caller-supplied count is trusted only up to the segment capacity
        const int nu = ld_act_i(c.num_unique);
        if (s >= nu || s >= max_segments(c)) return false;
        sg.e = ld_act_i(c.unique + s);
        sg.p0 = ld_act_i(c.offsets + sg.e);
        sg.p1 = ld_act_i(c.offsets + sg.e + 1);
    }
    // a grouping handed in by the caller is trusted only within bounds
    return sg.e >= 0 && sg.e < c.E && sg.p0 >= 0 && sg.p1 > sg.p0 && sg.p1 <= c.B * c.k;
}

// flat route index r stored at position p of the (grouped) route list.  A
// caller-supplied entry outside [0, B*k) would index x and the per-route
// outputs out of bounds: it is flagged (MOE_DEV_BAD_ROUTE) and replaced by
// route 0, so every access stays inside the buffers (the result is then
// not valid, as the status word says).
__device__ __forceinline__ int route_at(const Ctx& c, int p) {
    if (no_dedup(c)) return p;
    const int r = ld_act_i(c.route_idx + p);
    if (r < 0 || r >= c.B * c.k) {
        set_status(c.status, MOE_DEV_BAD_ROUTE);
        return 0;
    }
    return r;
}

}  // namespace moe
