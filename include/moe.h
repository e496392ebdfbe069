/*
 * moe.h -- C ABI of libmoe.so, a GB300 (sm_103a) Mixture-of-Experts decode
 * layer: router GEMV, fp32 softmax + top-k, stable grouping of the routes by
 * expert, grouped gate_up projection with SiLU(gate)*up, grouped down
 * projection and the routing-weighted combine -- all on the device, with no
 * host read-back of router scores and no synchronisation inside a layer or
 * between layers.
 *
 * Common conventions
 *  - Every tensor argument is a DEVICE pointer unless stated otherwise.
 *    The caller owns all memory; no entry point allocates or frees device
 *    memory.  Scratch space is the caller's `workspace`, sized by
 *    moe_workspace_bytes().
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every entry point only enqueues work on it and returns; none
 *    synchronises the stream or copies device -> host, so every call can be
 *    captured in a CUDA graph.
 *  - Layouts are row-major and contiguous:
 *      x        [B, H]       fp32 or bf16 (x_dtype)
 *      w_router [E, H]       bf16
 *      gate_up  [E, 2I, H]   bf16; rows [0, I) of an expert are the gate
 *                            projection, rows [I, 2I) the up projection
 *      down     [E, H, I]    bf16
 *      y        [B, H]       fp32
 *    bf16 is passed as raw 16-bit patterns (uint16_t).
 *  - Requirements: 1 <= E <= MOE_MAX_E, 1 <= top_k <= min(E, MOE_MAX_TOPK),
 *    0 <= B <= MOE_MAX_B, H and I multiples of 8 in [8, MOE_MAX_DIM], every
 *    pointer 16-byte aligned.  Violations return MOE_ERR_INVALID_ARG before
 *    anything is enqueued.
 *  - Return value: MOE_OK, or a negative moe_status.  Launch failures
 *    return MOE_ERR_CUDA.  Faults found on the device (a bad expert id, a
 *    barrier that timed out, a non-finite logit) are OR-ed as MOE_DEV_* bits
 *    into *dev_status (a device int32 the caller zeroes and reads after its
 *    own synchronisation); dev_status may be NULL to ignore them.
 *
 * The operation is the MoE layer of the pages "MoE Performance Optimization
 * Analysis" (Root Cause / GPU Router Design: router, selection and the
 * combination on the GPU with no CPU read) and "perf(cpu-moe): dedup experts
 * across the batch in pass 1 - #46" (commit message: routes grouped by
 * expert with a counting sort; pass 1 = gate_up [2I, H], pass 2 = down
 * [H, I]).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* host return codes */
typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,
    MOE_ERR_UNSUPPORTED = -2,
    MOE_ERR_CUDA = -3,
    MOE_ERR_WORKSPACE = -4
} moe_status;

/* device status bits (written asynchronously into *dev_status) */
#define MOE_DEV_TIMEOUT 1        /* a grid barrier gave up waiting           */
#define MOE_DEV_BAD_EXPERT_ID 2  /* an expert id outside [0, E)              */
#define MOE_DEV_DUP_EXPERT 4     /* one token lists the same expert twice    */
#define MOE_DEV_NONFINITE 8      /* a router logit was NaN or infinite       */
#define MOE_DEV_BAD_ROUTE 16     /* a route_idx entry outside [0, B*top_k)    */
#define MOE_DEV_RANGE 32         /* a router partial sum of the persistent     */
                                 /* decode kernel beyond +-2^21 (clamped: that */
                                 /* token's routing is not exact)              */

/* activation dtypes */
typedef enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 } moe_dtype;

/* limits */
#define MOE_MAX_E 256
#define MOE_MAX_TOPK 8
#define MOE_MAX_B 1024
#define MOE_MAX_DIM 16384
#define MOE_MAX_LAYERS 64

/* flags for moe_expert_forward / moe_layer_forward / moe_stack_forward */
#define MOE_F_NO_DEDUP 1u   /* evaluate every route on its own (each route re-reads
                               its expert's weights): the A/B baseline of the
                               dedup page; results are identical */
#define MOE_F_UNFUSED 2u    /* layer/stack: run the phases as separate kernels
                               instead of a persistent kernel */
#define MOE_F_FORCE_TC 4u   /* every expert with any route uses the tensor-core
                               GEMMs, even with MOE_F_SPLIT_TC (the default where
                               H % 128 == 0 and I % 64 == 0 and a workspace is given) */
#define MOE_F_NO_TC 8u      /* never use the tensor-core GEMMs */
#define MOE_F_NO_PREFETCH 16u /* stack: no speculative L2 prefetch of the gate/up
                               weights of the next layer's predicted experts (results
                               are unchanged; the prefetch only moves bytes earlier) */
#define MOE_F_HOT_L2 32u    /* layer/stack, batches beyond the decode kernel: keep
                               the step's most chosen experts in L2 for the next
                               steps -- the experts with at least MOE_TC_MIN_ROUTES
                               routes load their weights with an evict_last L2
                               policy, the others stream with evict_first ("MoE
                               Performance Optimization Analysis", Option 3:
                               expert caching; results are unchanged) */
#define MOE_F_SPLIT_TC 64u  /* layer/stack, batches beyond the decode kernel: only
                               the experts with at least MOE_TC_MIN_ROUTES routes
                               use the tensor-core GEMMs, the others the CUDA-core
                               streaming GEMV (two launches per projection; by
                               default every chosen expert takes the tensor cores,
                               one launch per projection) */
#define MOE_TC_MIN_ROUTES 8 /* the split of MOE_F_SPLIT_TC and MOE_F_HOT_L2 */

/*
 * moe_workspace_bytes -- size of the scratch buffer the forward entry points
 * need for a problem of this shape.  Host-only; *bytes receives the size.
 * Returns MOE_ERR_INVALID_ARG for unsupported shapes.
 */
int moe_workspace_bytes(int B, int H, int I, int E, int top_k, size_t* bytes);

/*
 * moe_route -- router GEMV + fp32 softmax + top-k + renormalisation.
 * ("MoE Performance Optimization Analysis", GPU Router Design: router
 * kernel = compute + selection; Batch Router Design: [B, H] -> [B, E].)
 *   logits[t,e] = sum_h x[t,h] * w_router[e,h] + (logit_bias ? logit_bias[e] : 0)
 *   p = softmax(logits[t,:]) in fp32
 *   expert_ids[t, 0..k) = the k largest logits, descending, ties to the lower id
 *   route_w[t,j] = p[id_j] / sum_j' p[id_j']
 * In:  x [B,H] (x_dtype), w_router [E,H] bf16, logit_bias [E] fp32 or NULL.
 * Out: expert_ids [B,k] int32, route_w [B,k] fp32, logits_out [B,E] fp32
 *      (may be NULL; then the workspace holds the logits and must be given).
 */
int moe_route(const void* x, int x_dtype, const uint16_t* w_router, const float* logit_bias,
              int B, int H, int E, int top_k, int32_t* expert_ids, float* route_w,
              float* logits_out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
              void* stream);

/*
 * moe_group_by_expert -- stable counting sort of the R = B*top_k routes
 * r = t*top_k + j by expert id ("perf(cpu-moe): dedup experts across the
 * batch in pass 1 - #46", commit message: group the routes by expert with a
 * counting sort over the ids, so each expert's weights are read once).
 * In:  expert_ids [B, top_k] int32; the ids of one token must be distinct.
 * Out: offsets [E+1]        exclusive prefix sum of the per-expert counts
 *      route_idx [R]        routes grouped by expert, increasing r in a group
 *      unique_experts [E]   experts with a nonzero count, ascending (first
 *                           *num_unique entries valid)
 *      num_unique [1]       U
 * Bad ids set MOE_DEV_BAD_EXPERT_ID / MOE_DEV_DUP_EXPERT and are skipped
 * (the outputs are then not a valid grouping).
 */
int moe_group_by_expert(const int32_t* expert_ids, int B, int top_k, int E, int32_t* offsets,
                        int32_t* route_idx, int32_t* unique_experts, int32_t* num_unique,
                        int32_t* dev_status, void* stream);

/*
 * moe_expert_forward -- the grouped experts and the combine for a given
 * routing ("perf(cpu-moe) ... #46": pass 1 = gate_up, pass 2 = down;
 * "MoE Performance Optimization Analysis": combination on the GPU).
 *   h_r = SiLU(gate_e x_t) * (up_e x_t),  o_r = down_e h_r   for each route
 *   y[t] = sum_j route_w[t,j] * o_(t,j)  (+ residual[t])
 * Each expert's weights are streamed once per call however many routes
 * chose it (unless MOE_F_NO_DEDUP).
 * In:  x [B,H], gate_up [E,2I,H], down [E,H,I], expert_ids/route_w [B,k],
 *      the grouping from moe_group_by_expert (offsets, route_idx,
 *      unique_experts, num_unique), residual [B,H] fp32 or NULL.
 * Out: y [B,H] fp32.  y may alias residual (in-place residual add).
 * A grouping handed in is used only within bounds: a unique-expert count
 * above min(B*top_k, E), expert ids outside [0, E) and offsets outside
 * [0, B*top_k] drop the segment; a route_idx entry outside [0, B*top_k) sets
 * MOE_DEV_BAD_ROUTE (route 0 is used in its place).  y is then not valid.
 */
int moe_expert_forward(const void* x, int x_dtype, const uint16_t* gate_up, const uint16_t* down,
                       const int32_t* expert_ids, const float* route_w, const int32_t* offsets,
                       const int32_t* route_idx, const int32_t* unique_experts,
                       const int32_t* num_unique, int B, int H, int I, int E, int top_k,
                       const float* residual, float* y, uint32_t flags, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * moe_expert_forward_noalloc -- moe_expert_forward for callers that cannot
 * allocate device memory (code inside a CUDA graph being captured or
 * replayed, an allocator hook that must not re-enter the allocator, a
 * runtime with a fixed memory budget).  The pages have no counterpart: this
 * is an interface convenience, not part of the method.
 * Same arguments and results as moe_expert_forward, minus the workspace,
 * except that every expert runs on the CUDA-core GEMV kernels (the tensor-
 * core path needs operand buffers of its own): MOE_F_FORCE_TC returns
 * MOE_ERR_UNSUPPORTED.  The scratch (h [R,I] and o [R,H], fp32) lives in
 * one static device array of MOE_NOALLOC_SCRATCH_BYTES inside the library,
 * held on every GPU that loads the library until the process exits.  Problems needing more than
 * that (4*R*(I+H) bytes plus alignment, R = B*top_k) return
 * MOE_ERR_WORKSPACE before anything is enqueued.  Nothing is allocated or
 * freed.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one array, so calls
 * that may overlap on the GPU (different streams, or concurrent graph
 * replays) race on it: serialise them.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (16u << 20)
int moe_expert_forward_noalloc(const void* x, int x_dtype, const uint16_t* gate_up,
                               const uint16_t* down, const int32_t* expert_ids,
                               const float* route_w, const int32_t* offsets,
                               const int32_t* route_idx, const int32_t* unique_experts,
                               const int32_t* num_unique, int B, int H, int I, int E, int top_k,
                               const float* residual, float* y, uint32_t flags,
                               int32_t* dev_status, void* stream);

/*
 * moe_layer_forward -- the whole layer: moe_route, moe_group_by_expert and
 * moe_expert_forward in one enqueue.  Unless MOE_F_UNFUSED, batches of up to
 * 4 tokens and 32 routes run in one persistent cooperative kernel (one CTA
 * per SM, device-wide barriers with a bounded wait); larger batches run the
 * phases as separate kernels (streaming GEMV for experts with few routes,
 * tensor-core GEMMs for the others), or, when no expert goes to the tensor
 * cores, all phases in one persistent fused kernel.
 * Out: y [B,H] fp32 (may alias residual); expert_ids_out / route_w_out
 *      [B,k] (may be NULL).
 */
int moe_layer_forward(const void* x, int x_dtype, const uint16_t* w_router,
                      const float* logit_bias, const uint16_t* gate_up, const uint16_t* down,
                      int B, int H, int I, int E, int top_k, const float* residual, float* y,
                      int32_t* expert_ids_out, float* route_w_out, uint32_t flags,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      void* stream);

/*
 * moe_stack_forward -- L MoE layers with the residual add between them,
 *   x <- x + layer_l(x),  l = 0..L-1,
 * entirely on the device ("TEXT Generation Optimization Report", optimized
 * forward flow: the layer loop runs with no wait; "MoE Performance
 * Optimization Analysis": GPU routing removes the per-layer router wait).
 * w_router, logit_bias, gate_up and down are HOST arrays of L device
 * pointers (logit_bias itself, or any of its entries, may be NULL).
 * x_inout [B,H] fp32 is updated in place.  expert_ids_out [L,B,k] or NULL.
 */
int moe_stack_forward(int L, const uint16_t* const* w_router, const float* const* logit_bias,
                      const uint16_t* const* gate_up, const uint16_t* const* down, int B, int H,
                      int I, int E, int top_k, float* x_inout, int32_t* expert_ids_out,
                      uint32_t flags, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream);

/*
 * moe_stack_forward_norm -- a pre-norm stack: L MoE layers, each applied to
 * the RMSNorm of its input, with the residual add between them,
 *   x <- x + layer_l(RMSNorm_l(x)),
 *   RMSNorm_l(x)[t,h] = (x[t,h] / sqrt(mean_h x[t,h]^2 + eps)) * norm_w[l][h],
 * entirely on the device ("TEXT Generation Optimization Report", Fused
 * Operations: fused_rms_norm_residual, norm + residual add; the RMSNorm
 * formula is the standard one, the page gives none).  For batches the
 * persistent decode kernel takes (up to 4 tokens, 32 routes) the norm is
 * fused into the router and the residual add: the next layer's logits are
 * formed from the CTAs' partial sums over g * x and x^2, so it costs no
 * extra pass or barrier.  Larger batches run a norm kernel per layer.
 * norm_w is a HOST array of L device pointers to [H] fp32 weights; eps in
 * [0, 1].  The other arguments are those of moe_stack_forward.
 */
int moe_stack_forward_norm(int L, const uint16_t* const* w_router, const float* const* logit_bias,
                           const uint16_t* const* gate_up, const uint16_t* const* down, const float* const* norm_w,
                           float eps, int B, int H, int I, int E, int top_k, float* x_inout,
                           int32_t* expert_ids_out, uint32_t flags, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream);

/*
 * moe_stack_forward_fp8 -- moe_stack_forward with block-scaled FP8 expert
 * weights ("fp8_block", one of the expert formats of "perf(cpu-moe): dedup
 * experts across the batch in pass 1 - #46", commit message; the encoding is
 * not on the pages: the OCP FP8 E4M3 format is taken).  Expert e's gate_up
 * [2I, H] and down [H, I] are E4M3 codes (one byte each, row-major), and
 *   w[r, c] = decode(q[r, c]) * scale[r / 128][c / 128]   (an fp32 product)
 * with the fp32 block scales gate_up_scale [E][ceil(2I/128)][ceil(H/128)] and
 * down_scale [E][ceil(H/128)][ceil(I/128)].  The router stays bf16.  The
 * experts stream half the bytes of bf16 weights; every sum stays fp32.
 * gate_up_q, gate_up_scale, down_q and down_scale are HOST arrays of L
 * device pointers.  Requires H and I multiples of 16.  Batches the persistent
 * decode kernel takes (up to 4 tokens and 32 routes) run in it; larger ones,
 * and any batch with MOE_F_UNFUSED, run layer by layer on the CUDA-core phase
 * kernels (the tensor-core GEMMs take bf16 weights only).  flags:
 * MOE_F_NO_DEDUP, MOE_F_NO_PREFETCH, MOE_F_UNFUSED.  The other arguments are
 * those of moe_stack_forward.
 */
int moe_stack_forward_fp8(int L, const uint16_t* const* w_router, const float* const* logit_bias,
                          const uint8_t* const* gate_up_q, const float* const* gate_up_scale,
                          const uint8_t* const* down_q, const float* const* down_scale, int B, int H, int I, int E,
                          int top_k, float* x_inout, int32_t* expert_ids_out, uint32_t flags, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * moe_stack_forward_nvfp4 -- moe_stack_forward with NVFP4 expert weights
 * ("nvfp4", another of the expert formats the dedup page's commit message
 * names; the encoding is not on the pages: the published NVFP4 layout is
 * taken).  Expert e's gate_up [2I, H] and down [H, I] hold E2M1 codes (sign,
 * 2 exponent bits biased by 1, 1 mantissa bit) two to a byte, element 2i of a
 * row in the low nibble of byte i; each 16 consecutive elements of a row
 * share one E4M3 scale, and each matrix one fp32 scale:
 *   w[r, c] = e2m1(q[r, c]) * e4m3(bs[r][c / 16]) * gs
 * gate_up_q [E][2I][H/2] and down_q [E][H][I/2] bytes, gate_up_bs
 * [E][2I][H/16] and down_bs [E][H][I/16] bytes, gate_up_gs and down_gs [E]
 * fp32.  The router stays bf16; the experts stream a quarter of the bytes of
 * bf16 weights (plus one scale byte per 16 weights); every sum stays fp32.
 * The six weight arguments are HOST arrays of L device pointers.  Requires H
 * and I multiples of 32.  Batches the persistent decode kernel takes (up to 4
 * tokens and 32 routes) run in it; larger ones, and any batch with
 * MOE_F_UNFUSED, run layer by layer on the CUDA-core phase kernels.  flags:
 * MOE_F_NO_DEDUP, MOE_F_NO_PREFETCH, MOE_F_UNFUSED.  The other arguments are
 * those of moe_stack_forward.
 */
int moe_stack_forward_nvfp4(int L, const uint16_t* const* w_router, const float* const* logit_bias,
                            const uint8_t* const* gate_up_q, const uint8_t* const* gate_up_bs,
                            const float* const* gate_up_gs, const uint8_t* const* down_q,
                            const uint8_t* const* down_bs, const float* const* down_gs, int B, int H, int I, int E,
                            int top_k, float* x_inout, int32_t* expert_ids_out, uint32_t flags, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * moe_workspace_grouping -- where a workspace holds the grouped route list
 * of the last layer a forward call computed in it (moe_layer_forward, and
 * the last layer of moe_stack_forward), in the layout of
 * moe_group_by_expert: offsets [E+1], route_idx [B*top_k], unique_experts
 * [E] (first *num_unique valid), num_unique [1].  Host-only pointer
 * arithmetic: the four outputs receive DEVICE addresses inside `workspace`
 * (same shape arguments as the forward call), valid after that call has
 * completed on its stream (unspecified with MOE_F_NO_DEDUP).  Exposes the
 * grouping the layer itself used, so that it can be checked against
 * moe_group_by_expert's definition ("perf(cpu-moe): dedup experts across
 * the batch in pass 1 - #46", commit message: the counting sort).
 */
int moe_workspace_grouping(void* workspace, size_t workspace_bytes, int B, int H, int I, int E, int top_k,
                           int32_t** offsets, int32_t** route_idx, int32_t** unique_experts,
                           int32_t** num_unique);

/*
 * moe_set_trace_buffer -- profiling aid.  While set, every launch of the
 * persistent decode kernel records, per CTA, per layer and per phase
 * boundary, a pair of 64-bit words (globaltimer ns, SM clock) into the device
 * buffer `trace` of `words` words: word index ((l+1)*G + cta)*48 + ev*2 for
 * layer l (-1 = the initial router step), G = grid size, event ev:
 * 0 layer start, 1 routing done, 2 gate/up done, 3 after the mid-layer
 * barrier, 4 down done, 5 layer work done, 6 after the end-of-layer barrier,
 * 7 top-k done (router warp), 8 x staged (consumers), 9 grouping done
 * (router warp), 10 combine done,
 * 11 next router slice ready, 12 first gate/up chunk landed (leader warp),
 * 13 first down chunk landed (leader warp), 16 last gate/up chunk landed,
 * 17 last chunk landed, 18 producer issued every chunk, 19 first chunk
 * landed (16..19 observed by the otherwise idle producer warp).
 * Entries that do not fit are dropped.  trace == NULL with words == 0 turns
 * it off (the default).  Host-only setting, not thread-safe.
 */
int moe_set_trace_buffer(unsigned long long* trace, int words);

/*
 * moe_inject_barrier_stall -- fault injection for the failure path.  While
 * extra_arrivals > 0, every device-wide barrier of the persistent kernels
 * (moe_layer_forward / moe_stack_forward without MOE_F_UNFUSED) waits for
 * that many arrivals beyond the grid, which never come: the first barrier's
 * bounded wait runs out (about a second), the CTA sets MOE_DEV_TIMEOUT in
 * dev_status and the abort word, every CTA leaves the kernel after its own
 * copies in flight have landed, and the launch completes with the context
 * still usable.  0 (the default) turns it off.  Returns MOE_ERR_INVALID_ARG
 * outside [0, 1024].  Host-only setting, not thread-safe.
 */
int moe_inject_barrier_stall(int extra_arrivals);

/*
 * moe_launch_count -- how many CUDA kernels the library has launched in this
 * process so far (all devices, all entry points; a relaxed atomic counter).
 * For measurement: the difference around a timed region is the number of
 * the library's kernel launches in it.  Host-only; never fails.
 */
unsigned long long moe_launch_count(void);

/*
 * moe_forward_path -- which kernels moe_layer_forward (L = 1) or
 * moe_stack_forward (L layers) runs for this shape and these flags on the
 * current device (host-only; the same decision the forward call makes):
 *   MOE_PATH_DECODE   one cooperative launch of the persistent decode kernel
 *                     (batches of up to 4 tokens and 32 routes)
 *   MOE_PATH_FUSED    one cooperative launch of the general fused kernel
 *   MOE_PATH_PHASES   the phases as separate kernels (per layer)
 *   0                 nothing (B == 0)
 * *grid (may be NULL) receives the persistent kernel's grid (0 for
 * MOE_PATH_PHASES).
 */
#define MOE_PATH_DECODE 2
#define MOE_PATH_FUSED 3
#define MOE_PATH_PHASES 4
int moe_forward_path(int B, int H, int I, int E, int top_k, int L, uint32_t flags, int* path, int* grid);

/* moe_status_string -- static text for a moe_status code or MOE_DEV_* bit. */
const char* moe_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
