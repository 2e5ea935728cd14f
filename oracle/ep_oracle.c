/*
 * CPU oracle for MoE dispatch / combine (DeepEP-style expert-parallel exchange).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library and its Python binding) never calls it and shares no code,
 * header, table or constant with it.
 *
 * Every function is the plain definition of what the method computes, written
 * as slow, sequential loops in the order the definition states.  Sources:
 *   [API]  "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南" (cyqw.cn),
 *          section 核心API示例: low_latency_dispatch(hidden_states, topk_idx,
 *          num_max_dispatch_tokens_per_rank, num_experts) and
 *          low_latency_combine(hidden_states, topk_idx, topk_weights, handle,
 *          num_experts); section 技术解析: layout information computed once and
 *          reused; section 性能调优: fixed-size receive buffers.
 *   [LL]   same page, section 核心优势: FP8 dispatch and BF16 combine in the
 *          low-latency setting (128 tokens, hidden 7168, top-8).
 *   [ANN]  DeepTech announcement of DeepEP (010bt.com), feature list: native
 *          FP8 dispatch, high-throughput (normal) and low-latency kernels.
 * Where the pages are silent the reading used is stated beside the code
 * (expert e is owned by rank e / (E/R); rows of one expert are ordered by
 * (source token, k); e4m3 is OCP E4M3FN; scale = max(amax, 1e-4) / 448 per
 * 128 channels; combine is an fp32 fused multiply-add chain in ascending k).
 *
 * Number formats are written from their definitions:
 *   bfloat16   = the upper 16 bits of an IEEE-754 binary32 (1 sign, 8 exponent,
 *                7 fraction bits); rounding from binary32 is to nearest, ties to
 *                even, overflow to infinity.
 *   E4M3FN     = OCP 8-bit floating point, 1 sign, 4 exponent (bias 7),
 *                3 mantissa bits, subnormals at exponent field 0, no
 *                infinities, S.1111.111 is NaN, largest finite 448.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC (no fast-math), so every
 * float operation below is one IEEE binary32 operation rounded to nearest.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_LAYOUT_PADDED 0
#define ORC_LAYOUT_PACKED 1

/* ------------------------------------------------------------------ */
/* bfloat16                                                            */
/* ------------------------------------------------------------------ */

float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* Magnitude of the bfloat16 whose bit pattern (sign cleared) is m; the
 * pattern 0x7F80 just past the largest finite value stands for 2^128 so that
 * the overflow threshold falls out of the nearest-value comparison. */
static double bf16_mag(uint32_t m)
{
    if (m >= 0x7F80u)
        return ldexp(1.0, 128);
    return (double)orc_bf16_to_f32((uint16_t)m);
}

/* Round a binary32 to the nearest bfloat16, ties to the even pattern. */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u = f32_bits(x);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) /* NaN: keep a quiet NaN of the same sign */
        return (uint16_t)((sign >> 16) | 0x7FC0u);
    if (mag == 0x7F800000u) /* infinity */
        return (uint16_t)((sign >> 16) | 0x7F80u);
    uint32_t lo = mag >> 16;     /* bfloat16 at or below |x| */
    uint32_t hi = lo + 1;        /* next bfloat16 above */
    double ax = fabs((double)x);
    double vlo = bf16_mag(lo);
    double vhi = bf16_mag(hi);
    uint32_t pick;
    if (ax == vlo)
        pick = lo;
    else {
        double twice = 2.0 * ax, mid2 = vlo + vhi; /* both exact in double */
        if (twice < mid2)
            pick = lo;
        else if (twice > mid2)
            pick = hi;
        else
            pick = (lo & 1u) ? hi : lo;
    }
    return (uint16_t)((sign >> 16) | pick);
}

/* ------------------------------------------------------------------ */
/* OCP E4M3FN                                                          */
/* ------------------------------------------------------------------ */

float orc_e4m3_to_f32(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return s ? -NAN : NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);            /* subnormal: 0.mmm x 2^-6 */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);   /* normal: 1.mmm x 2^(e-7) */
    return (float)(s ? -v : v);
}

/* Round a binary32 to E4M3FN: nearest, ties to even code, and (satfinite)
 * anything whose magnitude is 448 or more, infinities included, becomes
 * +-448.  NaN becomes the NaN pattern of the same sign. */
uint8_t orc_f32_to_e4m3(float x)
{
    uint8_t sign = (f32_bits(x) >> 31) ? 0x80 : 0x00;
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    double ax = fabs((double)x);
    if (ax >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* values of the non-negative finite codes, decoded once */
    static double val[0x7F];
    static int ready = 0;
    if (!ready) {
        for (int i = 0; i <= 0x7E; i++)
            val[i] = orc_e4m3_to_f32((uint8_t)i);
        ready = 1;
    }
    /* largest non-negative code c (0..0x7E) whose value is <= |x| */
    int c = 0;
    while (c + 1 <= 0x7E && val[c + 1] <= ax)
        c++;
    double vlo = val[c];
    if (ax == vlo)
        return (uint8_t)(sign | c);
    double vhi = val[c + 1];
    double twice = 2.0 * ax, mid2 = vlo + vhi;
    int pick;
    if (twice < mid2)
        pick = c;
    else if (twice > mid2)
        pick = c + 1;
    else
        pick = (c & 1) ? c + 1 : c;
    return (uint8_t)(sign | pick);
}

/* ------------------------------------------------------------------ */
/* Dispatch layout  [API] section 技术解析 (layout computed once, reused) */
/* ------------------------------------------------------------------ */

/*
 * topk_idx is [R, T, K] int64 (T = tokens per rank, global token g = r*T + t).
 * Entry -1 means "no expert"; anything else outside [0, E) is invalid, is
 * counted in errors[0] and otherwise treated like -1.  In the padded layout an
 * expert's buffer has R*Tmax rows; with repeated experts in one token's row it
 * can be offered more entries than that: those past the end get no row
 * (slot -1) and are counted in errors[1].
 *
 * Outputs (all written in full):
 *   cnt_er[e*R + r]       entries of source rank r routed to expert e
 *   off_er[e*R + r]       sum over r' < r of cnt_er[e*R + r']
 *   tokens_per_expert[e]  rows expert e receives: sum over r of
 *                         cnt_er[e*R + r], capped at R*Tmax when padded
 *   base[e]               first receive row of expert e: e*R*Tmax (padded,
 *                         fixed-size per-expert buffers) or the exclusive
 *                         prefix of tokens_per_expert (packed)
 *   tokens_per_rank[d]    tokens with at least one entry owned by rank d
 *   in_rank[g*R + d]      1 if token g has an entry owned by rank d, else 0
 *   slot[g*K + k]         receive row of entry (g, k), or -1
 *   src_info[row]         g*K + k for every row that receives an entry;
 *                         rows that receive nothing are left untouched
 * Rows of expert e are its entries in ascending (g, k) order, i.e. a stable
 * counting sort of the flattened entries by expert id.
 */
void orc_layout(int R, int T, int Tmax, int K, int E, int layout,
                const int64_t *topk_idx,
                int32_t *cnt_er, int32_t *off_er, int32_t *tokens_per_expert,
                int64_t *base, int32_t *tokens_per_rank, uint8_t *in_rank,
                int32_t *slot, int32_t *src_info, int64_t rows, int64_t *errors)
{
    int64_t N = (int64_t)R * T, bad = 0, overflow = 0;
    int64_t cap = (int64_t)R * Tmax; /* rows per expert buffer when padded */
    int L = E / R; /* experts per rank; expert e lives on rank e / L */

    for (int64_t i = 0; i < (int64_t)E * R; i++)
        cnt_er[i] = 0;
    for (int64_t g = 0; g < N; g++) {
        int r = (int)(g / T);
        for (int k = 0; k < K; k++) {
            int64_t e = topk_idx[g * K + k];
            if (e == -1)
                continue;
            if (e < -1 || e >= E) {
                bad++;
                continue;
            }
            cnt_er[e * R + r]++;
        }
    }
    for (int e = 0; e < E; e++) {
        int32_t run = 0;
        for (int r = 0; r < R; r++) {
            off_er[e * R + r] = run;
            run += cnt_er[e * R + r];
        }
        tokens_per_expert[e] = run;
    }
    int64_t acc = 0;
    for (int e = 0; e < E; e++) {
        if (layout == ORC_LAYOUT_PADDED)
            base[e] = (int64_t)e * R * Tmax;
        else {
            base[e] = acc;
            acc += tokens_per_expert[e];
        }
    }

    /* stable counting sort: walk entries in (g, k) order */
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t g = 0; g < N; g++) {
        for (int k = 0; k < K; k++) {
            int64_t e = topk_idx[g * K + k];
            if (e < 0 || e >= E) {
                slot[g * K + k] = -1;
                continue;
            }
            int64_t pos = fill[e];
            fill[e]++;
            if (layout == ORC_LAYOUT_PADDED && pos >= cap) {
                slot[g * K + k] = -1;
                overflow++;
                continue;
            }
            int64_t row = base[e] + pos;
            slot[g * K + k] = (int32_t)row;
            if (row < rows)
                src_info[row] = (int32_t)(g * K + k);
        }
    }
    free(fill);
    if (layout == ORC_LAYOUT_PADDED)
        for (int e = 0; e < E; e++)
            if (tokens_per_expert[e] > cap)
                tokens_per_expert[e] = (int32_t)cap;

    /* token -> rank membership, deduplicated per token */
    for (int d = 0; d < R; d++)
        tokens_per_rank[d] = 0;
    for (int64_t g = 0; g < N; g++) {
        for (int d = 0; d < R; d++) {
            uint8_t hit = 0;
            for (int k = 0; k < K; k++) {
                int64_t e = topk_idx[g * K + k];
                if (e >= 0 && e < E && e / L == d)
                    hit = 1;
            }
            in_rank[g * R + d] = hit;
            tokens_per_rank[d] += hit;
        }
    }
    errors[0] = bad;
    errors[1] = overflow;
}

/* ------------------------------------------------------------------ */
/* Rank-deduplicated layout  [ANN] normal kernels: tokens forwarded per   */
/* destination rank rather than per expert                               */
/* ------------------------------------------------------------------ */

/*
 * Each token is sent once to every rank that owns at least one of its
 * experts.  The entry (g, k) that carries token g to rank d is the first k of
 * the token whose expert lives on d; every other entry gets rank_slot -1.
 * Rows of rank d start at rbase[d] (d * R * Tmax padded, i.e. room for every
 * token; exclusive prefix of tokens_per_rank packed) and hold its tokens in
 * ascending g.  For each written row: src_info = g * K + k of the carrying
 * entry; recv_topk_idx[row * K + k'] = local expert id (e - d * L) of the
 * token's k'-th expert if it lives on d, else -1; recv_topk_w the matching
 * weight (w == NULL: 1), else 0.  Ids outside [0, E) are ignored.
 */
void orc_rank_layout(int R, int T, int Tmax, int K, int E, int layout,
                     const int64_t *topk_idx, const float *w,
                     int32_t *rank_slot, int32_t *tokens_per_rank, int64_t *rbase,
                     int32_t *src_info, int32_t *recv_topk_idx, float *recv_topk_w,
                     int64_t rows)
{
    int64_t N = (int64_t)R * T;
    int L = E / R;
    for (int d = 0; d < R; d++)
        tokens_per_rank[d] = 0;
    for (int64_t g = 0; g < N; g++)
        for (int k = 0; k < K; k++) {
            int64_t e = topk_idx[g * K + k];
            if (e < 0 || e >= E)
                continue;
            int first = 1;
            for (int k2 = 0; k2 < k; k2++) {
                int64_t e2 = topk_idx[g * K + k2];
                if (e2 >= 0 && e2 < E && e2 / L == e / L)
                    first = 0;
            }
            if (first)
                tokens_per_rank[e / L]++;
        }
    int64_t acc = 0;
    for (int d = 0; d < R; d++) {
        rbase[d] = layout == ORC_LAYOUT_PADDED ? (int64_t)d * R * Tmax : acc;
        acc += tokens_per_rank[d];
    }
    int32_t *fill = (int32_t *)calloc(R > 0 ? (size_t)R : 1u, sizeof(int32_t));
    for (int64_t g = 0; g < N; g++) {
        for (int k = 0; k < K; k++) {
            int64_t e = topk_idx[g * K + k];
            rank_slot[g * K + k] = -1;
            if (e < 0 || e >= E)
                continue;
            int d = (int)(e / L), first = 1;
            for (int k2 = 0; k2 < k; k2++) {
                int64_t e2 = topk_idx[g * K + k2];
                if (e2 >= 0 && e2 < E && e2 / L == d)
                    first = 0;
            }
            if (!first)
                continue;
            int64_t row = rbase[d] + fill[d];
            fill[d]++;
            rank_slot[g * K + k] = (int32_t)row;
            if (row >= rows)
                continue;
            src_info[row] = (int32_t)(g * K + k);
            for (int k2 = 0; k2 < K; k2++) {
                int64_t e2 = topk_idx[g * K + k2];
                int on_d = e2 >= 0 && e2 < E && e2 / L == d;
                recv_topk_idx[row * K + k2] = on_d ? (int32_t)(e2 - (int64_t)d * L) : -1;
                recv_topk_w[row * K + k2] = on_d ? (w ? w[g * K + k2] : 1.0f) : 0.0f;
            }
        }
    }
    free(fill);
}

/* ------------------------------------------------------------------ */
/* Per-(source rank, destination rank) runs of the rank-deduplicated      */
/* transport  [API] section 技术解析 (hook-based overlap that occupies no   */
/* SM; CPU and GPU cooperating on the layout); [ANN] normal kernels:      */
/* tokens forwarded per destination domain                               */
/* ------------------------------------------------------------------ */

/*
 * A source rank r sends its tokens carried to rank d as one contiguous run.
 * Send buffer order: source rank r ascending, then destination d ascending,
 * then token t ascending (the token's carrying entry is its first k whose
 * expert lives on d, as in orc_rank_layout).  In the receive layout of
 * orc_rank_layout the rows of rank d hold its tokens in ascending g = r*T + t,
 * so the tokens rank d gets from source r are one contiguous run there too.
 *   run_cnt[r*R + d]   tokens of source rank r carried to rank d
 *   send_off[r*R + d]  first send row of the run: sum of run_cnt over the
 *                      (r', d') before (r, d) in r-major order
 *   recv_off[r*R + d]  first receive row of the run: rbase[d] plus the sum of
 *                      run_cnt[r'*R + d] over r' < r
 *   send_slot[g*K + k] send row of the carrying entry (g, k), else -1
 * Copying run_cnt rows from send_off to recv_off for every (r, d) puts every
 * token's row where orc_rank_layout's rank_slot says.  Ids outside [0, E)
 * carry nothing.  Returns the number of send rows (the sum of run_cnt).
 */
int64_t orc_rank_runs(int R, int T, int K, int E, const int64_t *topk_idx, const int64_t *rbase,
                      int32_t *send_slot, int32_t *run_cnt, int64_t *send_off, int64_t *recv_off)
{
    int64_t N = (int64_t)R * T;
    int L = E / R;
    for (int64_t i = 0; i < N * K; i++)
        send_slot[i] = -1;
    for (int i = 0; i < R * R; i++)
        run_cnt[i] = 0;
    /* carrying entry of token g for rank d: its first k with an expert on d */
    for (int64_t g = 0; g < N; g++) {
        int src = (int)(g / T); /* source rank of token g */
        for (int k = 0; k < K; k++) {
            int64_t e = topk_idx[g * K + k];
            if (e < 0 || e >= E)
                continue;
            int d = (int)(e / L), first = 1;
            for (int k2 = 0; k2 < k; k2++) {
                int64_t e2 = topk_idx[g * K + k2];
                if (e2 >= 0 && e2 < E && e2 / L == d)
                    first = 0;
            }
            if (first)
                run_cnt[src * R + d]++;
        }
    }
    int64_t acc = 0;
    for (int r = 0; r < R; r++)
        for (int d = 0; d < R; d++) {
            send_off[r * R + d] = acc;
            acc += run_cnt[r * R + d];
        }
    for (int d = 0; d < R; d++) {
        int64_t run = rbase[d];
        for (int r = 0; r < R; r++) {
            recv_off[r * R + d] = run;
            run += run_cnt[r * R + d];
        }
    }
    /* send rows: r, then d, then t ascending */
    for (int r = 0; r < R; r++)
        for (int d = 0; d < R; d++) {
            int64_t row = send_off[r * R + d];
            for (int t = 0; t < T; t++) {
                int64_t g = (int64_t)r * T + t;
                for (int k = 0; k < K; k++) {
                    int64_t e = topk_idx[g * K + k];
                    if (e >= 0 && e < E && (int)(e / L) == d) {
                        send_slot[g * K + k] = (int32_t)row;
                        row++;
                        break; /* later k on d are not carrying entries */
                    }
                }
            }
        }
    return acc;
}

/* ------------------------------------------------------------------ */
/* FP8 cast  [ANN] native FP8 dispatch; [LL] FP8 dispatch               */
/* ------------------------------------------------------------------ */

/* One 128-channel block: amax over the block, scale = max(amax, 1e-4) / 448
 * and q = e4m3(x * (448 / max(amax, 1e-4))), each an IEEE binary32 operation. */
void orc_quant_block(const uint16_t *x, uint8_t *q, float *scale)
{
    float amax = 0.0f;
    for (int i = 0; i < 128; i++) {
        float a = fabsf(orc_bf16_to_f32(x[i]));
        if (a > amax)
            amax = a;
    }
    float amax_c = amax < 1e-4f ? 1e-4f : amax;
    float s = amax_c / 448.0f;
    float inv = 448.0f / amax_c;
    for (int i = 0; i < 128; i++) {
        float v = orc_bf16_to_f32(x[i]) * inv;
        q[i] = orc_f32_to_e4m3(v);
    }
    *scale = s;
}

/* One token row of H channels (H % 128 == 0): H/128 blocks, scales in
 * channel order. */
void orc_quant_token(const uint16_t *x, int H, uint8_t *q, float *scales)
{
    for (int b = 0; b < H / 128; b++)
        orc_quant_block(x + (int64_t)b * 128, q + (int64_t)b * 128, scales + b);
}

/* ------------------------------------------------------------------ */
/* Dispatch  [API] low_latency_dispatch                                */
/* ------------------------------------------------------------------ */

/* x is [N, H] bf16; every entry with slot >= 0 copies (BF16) or quantises
 * (FP8) its token row into receive row slot.  recv is [rows, H] uint16 (BF16)
 * or uint8 (FP8); scales is [rows, H/128] fp32, row-major (FP8 only). */
void orc_dispatch(int64_t N, int K, int H, int use_fp8, const uint16_t *x,
                  const int32_t *slot, void *recv, float *scales)
{
    for (int64_t g = 0; g < N; g++) {
        const uint16_t *xg = x + g * H;
        for (int k = 0; k < K; k++) {
            int64_t s = slot[g * K + k];
            if (s < 0)
                continue;
            if (use_fp8)
                orc_quant_token(xg, H, (uint8_t *)recv + s * H, scales + s * (H / 128));
            else
                memcpy((uint16_t *)recv + s * H, xg, (size_t)H * sizeof(uint16_t));
        }
    }
}

/* ------------------------------------------------------------------ */
/* Identity expert for FP8 rows: the BF16 value each code stands for   */
/* ------------------------------------------------------------------ */

/* For every entry with slot >= 0: y[slot, c] = bf16( e4m3(q[slot, c]) * scale[slot, c / 128] )
 * (one IEEE binary32 multiply, one round to nearest-even bf16). */
void orc_dequant_rows(int64_t N, int K, int H, const uint8_t *q, const float *scales,
                      const int32_t *slot, uint16_t *y)
{
    for (int64_t i = 0; i < N * K; i++) {
        int64_t s = slot[i];
        if (s < 0)
            continue;
        for (int c = 0; c < H; c++) {
            float v = orc_e4m3_to_f32(q[s * H + c]) * scales[s * (H / 128) + c / 128];
            y[s * H + c] = orc_f32_to_bf16(v);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Combine  [API] low_latency_combine; [LL] BF16 combine               */
/* ------------------------------------------------------------------ */

/* out[g, c] = bf16( fma chain over k = 0..K-1 in ascending order of
 * w[g, k] * y[slot[g, k], c] starting from +0.0f ), entries with slot < 0
 * skipped; w == NULL means every weight is 1. */
void orc_combine(int64_t N, int K, int H, const uint16_t *y, const int32_t *slot,
                 const float *w, uint16_t *out)
{
    for (int64_t g = 0; g < N; g++) {
        for (int c = 0; c < H; c++) {
            float acc = 0.0f;
            for (int k = 0; k < K; k++) {
                int64_t s = slot[g * K + k];
                if (s < 0)
                    continue;
                float wk = w ? w[g * K + k] : 1.0f;
                acc = fmaf(wk, orc_bf16_to_f32(y[s * H + c]), acc);
            }
            out[g * H + c] = orc_f32_to_bf16(acc);
        }
    }
}

/* Array helpers for the Python side. */
void orc_f32_to_bf16_n(const float *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        y[i] = orc_f32_to_bf16(x[i]);
}

void orc_bf16_to_f32_n(const uint16_t *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        y[i] = orc_bf16_to_f32(x[i]);
}

void orc_f32_to_e4m3_n(const float *x, uint8_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        y[i] = orc_f32_to_e4m3(x[i]);
}

void orc_e4m3_to_f32_n(const uint8_t *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        y[i] = orc_e4m3_to_f32(x[i]);
}
