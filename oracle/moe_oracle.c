/*
 * moe_oracle.c -- plain, slow CPU oracle for the MoE decode layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA library: it is written from the pages alone.
 *
 * What it computes (one MoE layer forward for a decode batch):
 *   logits[t,e] = sum_h x[t,h] * Wr[e,h]  (+ bias[e])
 *       -- the router GEMV, "MoE Performance Optimization Analysis",
 *          Technical Details / Batch Router Design ([batch, hidden] ->
 *          [batch, numExperts]).
 *   p = softmax(logits[t,:]) in fp32; the k experts with the largest logits,
 *       ties to the lower expert id; w_j = p_j / sum of the selected p
 *       -- "GPU Router Design" (router kernel: compute + selection).  The
 *          softmax placement, tie rule and renormalisation are not on the
 *          pages; this is the plainest reading, stated for the workloads.
 *   group the routes r = t*k + j by expert with a stable counting sort
 *       -- "perf(cpu-moe): dedup experts across the batch in pass 1 - #46",
 *          commit message (group the routes by expert, counting sort).
 *   for each route: g = G_e x, u = U_e x, h = SiLU(g) * u, o = D_e h
 *       -- same page: pass 1 reads gate_up shaped [2I, H], pass 2 reads
 *          down shaped [H, I].  Rows [0, I) of gate_up are the gate rows
 *          and rows [I, 2I) the up rows (reading of "gate_up").
 *   y[t] = sum_j w_j * o_(t,j), summed in j order; a stack adds x + y
 *       -- "GPU Router Design" (combination on the GPU) and the optimized
 *          forward flow of "TEXT Generation Optimization Report" (layer
 *          loop with a residual add).
 *
 * Precision: every sum is an fp32 sum in index order (the workloads fix fp32
 * accumulation and an fp32 softmax); bf16 inputs are widened exactly.  Build
 * with -ffp-contract=off so that a*b+c is never fused and the results are the
 * same on every host.
 *
 * Parity pins: see tests/test_oracle_pins.py (numpy fp64 brute force over all
 * experts, closed forms, invariants, the dedup table printed on the #46 page).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_BAD_ARG (-1)
#define OR_BAD_ID (-2)

static float bf16_to_f32(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* One FP8 E4M3 code as fp32 (the OCP 8-bit floating point format, "E4M3":
 * sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 holds the
 * subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no infinities).  The
 * format is not on the pages, which name "fp8_block" expert weights only. */
static float fp8e4m3_to_f32(uint8_t b) {
    const int sgn = b >> 7, e = (b >> 3) & 15, m = b & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexpf((float)m / 8.0f, -6);
    else
        v = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return sgn ? -v : v;
}

/* Block-scaled FP8 weights ("fp8_block"): a [R, C] matrix of E4M3 codes with
 * one fp32 scale per 128 x 128 block (row-major over the blocks, ceil(C/128)
 * per block row):  w[r,c] = decode(q[r,c]) * scale[r/128][c/128], an fp32
 * product. */
int oracle_dequant_fp8_block(const uint8_t* q, const float* scale, int R, int C, float* out) {
    if (R <= 0 || C <= 0 || !q || !scale || !out) return OR_BAD_ARG;
    const int nbc = (C + 127) / 128;
    for (int r = 0; r < R; ++r)
        for (int c = 0; c < C; ++c)
            out[(size_t)r * C + c] = fp8e4m3_to_f32(q[(size_t)r * C + c]) * scale[(size_t)(r / 128) * nbc + c / 128];
    return OR_OK;
}

/* NVFP4 element: E2M1 (sign, 2 exponent bits biased by 1, 1 mantissa bit):
 * 0, 0.5 (the one subnormal), 1, 1.5, 2, 3, 4, 6 and their negatives. */
static float fp4e2m1_to_f32(uint8_t c) {
    const int sgn = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    const float v = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
    return sgn ? -v : v;
}

/* NVFP4 weights: a [R, C] matrix of E2M1 codes packed two to a byte (element
 * 2i of a row in the low nibble of byte i), one E4M3 scale per 16
 * consecutive elements of a row ([R][C/16] bytes) and one fp32 scale for the
 * whole matrix:  w[r,c] = (e2m1(q[r,c]) * e4m3(bs[r][c/16])) * gs, fp32. */
int oracle_dequant_nvfp4(const uint8_t* q, const uint8_t* bs, float gs, int R, int C, float* out) {
    if (R <= 0 || C <= 0 || (C % 16) != 0 || !q || !bs || !out) return OR_BAD_ARG;
    for (int r = 0; r < R; ++r)
        for (int c = 0; c < C; ++c) {
            const uint8_t byte = q[(size_t)r * (C / 2) + c / 2];
            const uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            out[(size_t)r * C + c] = (fp4e2m1_to_f32(code) * fp8e4m3_to_f32(bs[(size_t)r * (C / 16) + c / 16])) * gs;
        }
    return OR_OK;
}

/* x_dtype: 0 = fp32, 1 = bf16 (raw 16-bit patterns). */
static float load_x(const void* x, int x_dtype, size_t idx) {
    if (x_dtype == 1) return bf16_to_f32(((const uint16_t*)x)[idx]);
    return ((const float*)x)[idx];
}

/* Router GEMV: logits[t,e] = sum_h x[t,h]*Wr[e,h], h ascending, + bias[e].
 * The (token, expert) pairs are independent sums, so they are spread over
 * threads; each sum still runs in h order. */
int oracle_router(const void* x, int x_dtype, const uint16_t* wr, const float* bias,
                  int B, int H, int E, float* logits) {
    if (B < 0 || H <= 0 || E <= 0 || !x || !wr || !logits) return OR_BAD_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int t = 0; t < B; ++t) {
        for (int e = 0; e < E; ++e) {
            float acc = 0.0f;
            for (int h = 0; h < H; ++h)
                acc += load_x(x, x_dtype, (size_t)t * H + h) * bf16_to_f32(wr[(size_t)e * H + h]);
            if (bias) acc += bias[e];
            logits[(size_t)t * E + e] = acc;
        }
    }
    return OR_OK;
}

/* fp32 softmax over all E logits, top-k by logit (ties -> lower id), then
 * the selected probabilities renormalised to sum 1.  ids[t,j] are in
 * selection order (descending logit).  k rounds of "take the best not yet
 * taken", written as plainly as possible. */
int oracle_topk(const float* logits, int B, int E, int k, int32_t* ids, float* w) {
    if (B < 0 || E <= 0 || k <= 0 || k > E || !logits || !ids || !w) return OR_BAD_ARG;
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    float* p = (float*)malloc(sizeof(float) * (size_t)E);
    if (!taken || !p) { free(taken); free(p); return OR_BAD_ARG; }
    for (int t = 0; t < B; ++t) {
        const float* l = logits + (size_t)t * E;
        float m = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
        float s = 0.0f;
        for (int e = 0; e < E; ++e) { p[e] = expf(l[e] - m); s += p[e]; }
        for (int e = 0; e < E; ++e) p[e] = p[e] / s;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                /* strictly greater: an equal logit never replaces a lower id */
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        float ssel = 0.0f;
        for (int j = 0; j < k; ++j) ssel += p[ids[(size_t)t * k + j]];
        for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = p[ids[(size_t)t * k + j]] / ssel;
    }
    free(taken);
    free(p);
    return OR_OK;
}

/* Stable counting sort of the R = B*k flat routes r = t*k + j by expert id.
 *   offsets[E+1]: exclusive prefix sum of the per-expert counts;
 *   route_idx[R]: route indices, grouped by expert, increasing r inside a group;
 *   unique[]:     experts with a nonzero count, ascending; *num_unique = U. */
int oracle_group(const int32_t* ids, int B, int k, int E, int32_t* offsets,
                 int32_t* route_idx, int32_t* unique, int32_t* num_unique) {
    if (B < 0 || k <= 0 || E <= 0 || !ids || !offsets || !route_idx || !unique || !num_unique)
        return OR_BAD_ARG;
    const int R = B * k;
    for (int r = 0; r < R; ++r)
        if (ids[r] < 0 || ids[r] >= E) return OR_BAD_ID;
    int32_t* counts = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    int32_t* next = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!counts || !next) { free(counts); free(next); return OR_BAD_ARG; }
    for (int r = 0; r < R; ++r) counts[ids[r]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int e = 0; e < E; ++e) next[e] = offsets[e];
    for (int r = 0; r < R; ++r) route_idx[next[ids[r]]++] = r;
    int u = 0;
    for (int e = 0; e < E; ++e) if (counts[e] > 0) unique[u++] = e;
    *num_unique = u;
    free(counts);
    free(next);
    return OR_OK;
}

/* An expert weight as fp32: wtype 0 = bf16 bit patterns (widened exactly),
 * 1 = fp32 (e.g. dequantised block-scaled FP8 weights). */
static float load_w(const void* w, int wtype, size_t idx) {
    if (wtype == 1) return ((const float*)w)[idx];
    return bf16_to_f32(((const uint16_t*)w)[idx]);
}

/* Pass 1 of one expert on one token, gate/up rows [i0, i1):
 * h[i] = SiLU(G_i . x) * (U_i . x), each dot product in h order.
 * gate_up_e: [2I, H] bf16 (rows [0,I) gate, [I,2I) up). */
static void expert_gate_rows(const void* x, int x_dtype, size_t x_off, const void* gate_up_e, int wtype,
                             int H, int I, int i0, int i1, float* hbuf) {
    for (int i = i0; i < i1; ++i) {
        float g = 0.0f, u = 0.0f;
        const size_t grow = (size_t)i * H;
        const size_t urow = (size_t)(I + i) * H;
        for (int h = 0; h < H; ++h) {
            float xv = load_x(x, x_dtype, x_off + h);
            g += load_w(gate_up_e, wtype, grow + h) * xv;
            u += load_w(gate_up_e, wtype, urow + h) * xv;
        }
        float silu = g / (1.0f + expf(-g));
        hbuf[i] = silu * u;
    }
}

/* Pass 2 of one expert on one token, down rows [r0, r1): o[r] = D_r . h,
 * each dot product in i order.  down_e: [H, I] bf16. */
static void expert_down_rows(const void* down_e, int wtype, int I, int r0, int r1, const float* hbuf,
                             float* o) {
    for (int r = r0; r < r1; ++r) {
        float acc = 0.0f;
        const size_t drow = (size_t)r * I;
        for (int i = 0; i < I; ++i) acc += load_w(down_e, wtype, drow + i) * hbuf[i];
        o[r] = acc;
    }
}

/* One expert on one token: h = SiLU(G x) * (U x), o = D h. */
static void expert_one(const void* x, int x_dtype, size_t x_off, const void* gate_up_e, const void* down_e,
                       int wtype, int H, int I, float* hbuf, float* o) {
    expert_gate_rows(x, x_dtype, x_off, gate_up_e, wtype, H, I, 0, I, hbuf);
    expert_down_rows(down_e, wtype, I, 0, H, hbuf, o);
}

/* rows per work item of the dedup passes */
#define ORACLE_ROW_BLOCK 64

/* Expert pass for given routing.  gate_up_ptrs[e] / down_ptrs[e] point at
 * expert e's weights (host memory); experts that no route selects may be
 * NULL.  o_routes: [R, H] output per flat route r (may be NULL, then a local
 * buffer is used).  h_routes: [R, I] (may be NULL).
 *   mode 0 = per route: walk t, then j, evaluating each route on its own.
 *   mode 1 = dedup: walk the grouped list expert by expert (the #46 loop
 *            order); every route's arithmetic is the same as in mode 0, so
 *            the two modes are bit-identical.
 * y[t] = sum_j w[t,j] * o[t*k+j], j ascending, then + residual[t] if given. */
int oracle_experts_w(const void* x, int x_dtype, const void* const* gate_up_ptrs,
                     const void* const* down_ptrs, int wtype, const int32_t* ids, const float* w,
                     int B, int H, int I, int E, int k, int mode, const float* residual,
                     float* y, float* h_routes, float* o_routes) {
    if (B < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || !x || !gate_up_ptrs || !down_ptrs ||
        !ids || !w || !y)
        return OR_BAD_ARG;
    const int R = B * k;
    for (int r = 0; r < R; ++r) {
        if (ids[r] < 0 || ids[r] >= E) return OR_BAD_ID;
        if (!gate_up_ptrs[ids[r]] || !down_ptrs[ids[r]]) return OR_BAD_ARG;
    }
    float* o = o_routes ? o_routes : (float*)malloc(sizeof(float) * (size_t)R * H + 1);
    float* hb = h_routes ? h_routes : (float*)malloc(sizeof(float) * (size_t)R * I + 1);
    if (!o || !hb) return OR_BAD_ARG;
    if (mode == 0) {
        for (int t = 0; t < B; ++t)
            for (int j = 0; j < k; ++j) {
                int r = t * k + j, e = ids[r];
                expert_one(x, x_dtype, (size_t)t * H, gate_up_ptrs[e], down_ptrs[e], wtype, H, I,
                           hb + (size_t)r * I, o + (size_t)r * H);
            }
    } else {
        int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
        int32_t* ridx = (int32_t*)malloc(sizeof(int32_t) * (size_t)R + 4);
        int32_t* uniq = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
        int32_t nu = 0;
        oracle_group(ids, B, k, E, offsets, ridx, uniq, &nu);
        /* The #46 loop order, split by (unique expert, row block): pass 1
         * over the gate/up rows, then pass 2 over the down rows.  Every h[r,i]
         * and o[r,c] is one dot product written to its own place, computed
         * exactly as in expert_one, so neither the split nor the order the
         * items run in changes a bit of the result. */
        const int nib = (I + ORACLE_ROW_BLOCK - 1) / ORACLE_ROW_BLOCK;
        const int nrb = (H + ORACLE_ROW_BLOCK - 1) / ORACLE_ROW_BLOCK;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
        for (int u = 0; u < nu; ++u) {
            for (int ib = 0; ib < nib; ++ib) {
                int e = uniq[u];
                int i0 = ib * ORACLE_ROW_BLOCK;
                int i1 = i0 + ORACLE_ROW_BLOCK < I ? i0 + ORACLE_ROW_BLOCK : I;
                for (int q = offsets[e]; q < offsets[e + 1]; ++q) {
                    int r = ridx[q], t = r / k;
                    expert_gate_rows(x, x_dtype, (size_t)t * H, gate_up_ptrs[e], wtype, H, I, i0, i1,
                                     hb + (size_t)r * I);
                }
            }
        }
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
        for (int u = 0; u < nu; ++u) {
            for (int rb = 0; rb < nrb; ++rb) {
                int e = uniq[u];
                int r0 = rb * ORACLE_ROW_BLOCK;
                int r1 = r0 + ORACLE_ROW_BLOCK < H ? r0 + ORACLE_ROW_BLOCK : H;
                for (int q = offsets[e]; q < offsets[e + 1]; ++q) {
                    int r = ridx[q];
                    expert_down_rows(down_ptrs[e], wtype, I, r0, r1, hb + (size_t)r * I,
                                     o + (size_t)r * H);
                }
            }
        }
        free(offsets);
        free(ridx);
        free(uniq);
    }
    for (int t = 0; t < B; ++t)
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) acc += w[(size_t)t * k + j] * o[((size_t)t * k + j) * H + c];
            if (residual) acc = residual[(size_t)t * H + c] + acc;
            y[(size_t)t * H + c] = acc;
        }
    if (!o_routes) free(o);
    if (!h_routes) free(hb);
    return OR_OK;
}

/* The expert pass with bf16 expert weights. */
int oracle_experts(const void* x, int x_dtype, const uint16_t* const* gate_up_ptrs,
                   const uint16_t* const* down_ptrs, const int32_t* ids, const float* w,
                   int B, int H, int I, int E, int k, int mode, const float* residual,
                   float* y, float* h_routes, float* o_routes) {
    return oracle_experts_w(x, x_dtype, (const void* const*)gate_up_ptrs, (const void* const*)down_ptrs, 0, ids,
                            w, B, H, I, E, k, mode, residual, y, h_routes, o_routes);
}

/* RMSNorm of every token's row, the norm half of the fused "norm + residual
 * add" operation ("TEXT Generation Optimization Report", Fused Operations:
 * fused_rms_norm_residual; the formula is not on the pages: the standard
 * RMSNorm is taken):
 *   ms = (sum_h x[t,h]^2) / H        fp32, h ascending
 *   a[t,h] = (x[t,h] * (1 / sqrtf(ms + eps))) * g[h]
 * In a stack the residual add is x_{l+1} = x_l + layer_l(a_l) (see
 * oracle_stack_norm). */
int oracle_rmsnorm(const float* x, const float* g, int B, int H, float eps, float* a) {
    if (B < 0 || H <= 0 || !x || !g || !a) return OR_BAD_ARG;
    for (int t = 0; t < B; ++t) {
        const float* xr = x + (size_t)t * H;
        float ss = 0.0f;
        for (int h = 0; h < H; ++h) ss += xr[h] * xr[h];
        const float ms = ss / (float)H;
        const float r = 1.0f / sqrtf(ms + eps);
        for (int h = 0; h < H; ++h) a[(size_t)t * H + h] = (xr[h] * r) * g[h];
    }
    return OR_OK;
}

/* Whole layer: router -> top-k -> experts -> combine.  ids/w/logits are
 * outputs ([B,k], [B,k], [B,E]); gate_up_ptrs/down_ptrs as above. */
int oracle_layer(const void* x, int x_dtype, const uint16_t* wr, const float* bias,
                 const uint16_t* const* gate_up_ptrs, const uint16_t* const* down_ptrs,
                 int B, int H, int I, int E, int k, int mode, const float* residual,
                 float* y, int32_t* ids, float* w, float* logits) {
    int rc = oracle_router(x, x_dtype, wr, bias, B, H, E, logits);
    if (rc) return rc;
    rc = oracle_topk(logits, B, E, k, ids, w);
    if (rc) return rc;
    return oracle_experts(x, x_dtype, gate_up_ptrs, down_ptrs, ids, w, B, H, I, E, k, mode,
                          residual, y, NULL, NULL);
}

/* Pre-norm stack: x <- x + layer_l(rmsnorm_l(x)) for l = 0..L-1; norm_w[l]
 * [H] fp32 holds layer l's norm weights, the other arguments are those of
 * oracle_stack. */
int oracle_stack_norm(int L, const uint16_t* const* wr, const float* const* bias,
                      const uint16_t* const* gate_up_ptrs, const uint16_t* const* down_ptrs,
                      const float* const* norm_w, float eps, int B, int H, int I, int E, int k,
                      int mode, float* x, int32_t* ids_out) {
    if (L <= 0 || B < 0 || !x || !norm_w) return OR_BAD_ARG;
    float* a = (float*)malloc(sizeof(float) * (size_t)B * H + 1);
    float* y = (float*)malloc(sizeof(float) * (size_t)B * H + 1);
    float* lg = (float*)malloc(sizeof(float) * (size_t)B * E + 1);
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)B * k + 4);
    float* w = (float*)malloc(sizeof(float) * (size_t)B * k + 4);
    int rc = OR_OK;
    if (!a || !y || !lg || !ids || !w) rc = OR_BAD_ARG;
    for (int l = 0; l < L && rc == OR_OK; ++l) {
        rc = oracle_rmsnorm(x, norm_w[l], B, H, eps, a);
        if (rc) break;
        rc = oracle_layer(a, 0, wr[l], bias ? bias[l] : NULL, gate_up_ptrs + (size_t)l * E,
                          down_ptrs + (size_t)l * E, B, H, I, E, k, mode, x, y, ids, w, lg);
        if (rc) break;
        memcpy(x, y, sizeof(float) * (size_t)B * H);
        if (ids_out) memcpy(ids_out + (size_t)l * B * k, ids, sizeof(int32_t) * (size_t)B * k);
    }
    free(a);
    free(y);
    free(lg);
    free(ids);
    free(w);
    return rc;
}

/* Stack of L layers with the residual: x <- x + layer_l(x), x fp32 [B,H]
 * updated in place.  wr[l], bias[l] (bias may be NULL or hold NULLs),
 * gate_up_ptrs[l*E + e], down_ptrs[l*E + e].  ids_out: [L,B,k] or NULL. */
int oracle_stack(int L, const uint16_t* const* wr, const float* const* bias,
                 const uint16_t* const* gate_up_ptrs, const uint16_t* const* down_ptrs,
                 int B, int H, int I, int E, int k, int mode, float* x, int32_t* ids_out) {
    if (L <= 0 || B < 0 || !x) return OR_BAD_ARG;
    float* y = (float*)malloc(sizeof(float) * (size_t)B * H + 1);
    float* lg = (float*)malloc(sizeof(float) * (size_t)B * E + 1);
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)B * k + 4);
    float* w = (float*)malloc(sizeof(float) * (size_t)B * k + 4);
    int rc = OR_OK;
    if (!y || !lg || !ids || !w) rc = OR_BAD_ARG;
    for (int l = 0; l < L && rc == OR_OK; ++l) {
        rc = oracle_layer(x, 0, wr[l], bias ? bias[l] : NULL, gate_up_ptrs + (size_t)l * E,
                          down_ptrs + (size_t)l * E, B, H, I, E, k, mode, x, y, ids, w, lg);
        if (rc) break;
        memcpy(x, y, sizeof(float) * (size_t)B * H);
        if (ids_out) memcpy(ids_out + (size_t)l * B * k, ids, sizeof(int32_t) * (size_t)B * k);
    }
    free(y);
    free(lg);
    free(ids);
    free(w);
    return rc;
}
