/*
 * moe_oracle.c -- CPU oracle for the MoE expert-parallel dispatch/combine path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline/reference leg load this file's library.  The
 * CUDA library never calls it, and the two share no code, headers or tables.
 *
 * Plain, single-threaded C99, compiled with -ffp-contract=off so that every
 * float operation is one IEEE-754 single-precision operation rounded to nearest.
 * Each function states the passage it follows.  Pins (what each function is
 * checked against, independently of itself) live in tests/test_oracle_*.py:
 *
 *   oracle_layout          numpy bincount / cumsum / stable argsort, O(N^2) brute force
 *   oracle_dispatch        row equality against the stable argsort permutation
 *   oracle_e4m3_encode     torch float8_e4m3fn cast of saturated inputs, all codes
 *   oracle_dispatch_quant  encoder pin + per-block invariants (amax -> +-448, dequant
 *                          error bound, zero block); the scale recipe itself is a
 *                          reading: the pages only name W8A8 (parity unpinned against
 *                          the pages for the recipe, pinned for the arithmetic)
 *   oracle_combine         float64 closed form within the fp32 error bound, one-hot
 *                          weights, identity-expert round trip
 *   oracle_f32_to_bf16     torch bfloat16 cast
 *   oracle_combine_backward  torch autograd of a float64 forward combine; torch's
 *                          bf16 rounding of fp32 products; numpy einsum for dw
 *   oracle_dispatch_backward oracle_combine with unit weights (special case),
 *                          float64 closed form within the fp32 bound
 *   oracle_layout_coalesced  set-based brute force in numpy; invariants (row count
 *                          = sum of distinct ranks per token, token order per rank,
 *                          expand consistent with the plain slot map)
 *   oracle_dispatch_coalesced rows equal the owning token's row
 *   oracle_combine_coalesced_pre/post  one rank (R = 1) reduces to the plain
 *                          combine; one slot per rank to bf16(w*y) summed in
 *                          fp32; integer payloads give the exact sum; within
 *                          a derived bound of the binary64 sum
 *   oracle_ep_dispatch     numpy stable argsort of all ranks' ids (the receive
 *                          buffers, concatenated, are the single-GPU order of
 *                          the concatenated tokens); per-source bincounts;
 *                          a Python brute-force sort of (expert, source, t, j)
 *   oracle_ep_combine      float64 closed form within the fp32 bound; the
 *                          identity-expert round trip returns x
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG 1
#define ORACLE_ERR_BAD_INDEX 2

/* ------------------------------------------------------------------------- */
/* bf16 <-> f32                                                               */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32 word: widening is exact. */
static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round binary32 to bf16, nearest with ties to even; NaN stays a quiet NaN. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    /* round up when the dropped half is above one half, or exactly one half
       and the kept part is odd */
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------------- */
/* Layout: count -> exclusive scan -> stable slot map                         */
/* UBEP, section 2.3 / Figure 2 (dispatch phases: per-expert token counts,    */
/* then offsets and contiguous per-expert reordering) and section 4 (receive  */
/* region pre-partitioned by source and expert); StrataCL, Appendix D (first  */
/* level: destination expert, per-expert counts, prefix-sum offsets and       */
/* token-local offsets).  Order inside an expert: source token, then k slot.  */
/* ------------------------------------------------------------------------- */
int oracle_layout(int T, int k, int E, int R, const int32_t *topk_idx,
                  int32_t *expert_counts, int32_t *expert_offsets,
                  int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of)
{
    if (T < 0 || k < 1 || E < 1 || R < 1 || E % R != 0)
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    const int El = E / R;

    /* 1. count: how many (token, slot) pairs chose each expert */
    for (int e = 0; e < E; ++e)
        expert_counts[e] = 0;
    for (int64_t i = 0; i < N; ++i) {
        int e = topk_idx[i];
        if (e < 0 || e >= E)
            return ORACLE_ERR_BAD_INDEX;
        expert_counts[e] += 1;
    }

    /* 2. exclusive prefix sum over experts; experts of rank r are the
          contiguous block r*El .. r*El+El-1, so rank offsets are a subsample */
    expert_offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        expert_offsets[e + 1] = expert_offsets[e] + expert_counts[e];
    for (int r = 0; r <= R; ++r)
        rank_offsets[r] = expert_offsets[r * El];

    /* 3. walk (token, slot) pairs in lexicographic order; each expert hands
          out its slots in that order */
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!cursor)
        return ORACLE_ERR_INVALID_ARG;
    for (int e = 0; e < E; ++e)
        cursor[e] = expert_offsets[e];
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t i = (int64_t)t * k + j;
            int e = topk_idx[i];
            int32_t s = cursor[e]++;
            slot_of[i] = s;
            src_of[s] = (int32_t)i;
        }
    }
    free(cursor);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Dispatch (bf16): every token row goes, unchanged, to each of its k slots.  */
/* UBEP section 2.3 (Phase 2: a token may be sent to several experts);        */
/* RailWave section 3.2 (payload packed without padding).                     */
/* ------------------------------------------------------------------------- */
int oracle_dispatch(int T, int H, int k, const uint16_t *x, const int32_t *slot_of,
                    uint16_t *recv)
{
    if (T < 0 || H < 1 || k < 1)
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t s = slot_of[(int64_t)t * k + j];
            if (s < 0 || s >= N)
                return ORACLE_ERR_BAD_INDEX;
            memcpy(recv + (int64_t)s * H, x + (int64_t)t * H, sizeof(uint16_t) * (size_t)H);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 encoding, written from the OCP 8-bit floating point definition:   */
/* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no infinities;   */
/* S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448;    */
/* subnormals (exponent field 0) are m * 2^-9.  Rounding: nearest, ties to    */
/* even; "satfinite": magnitudes beyond 448 (and infinities) clamp to 448.    */
/* ------------------------------------------------------------------------- */
uint8_t oracle_e4m3_encode(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint8_t sign = (uint8_t)((u >> 31) << 7);
    if (isnan(f))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)f);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2); /* a = m * 2^e2 with m in [0.5, 1) */
    int e = e2 - 1;      /* a = (1 + frac) * 2^e               */
    uint32_t code;
    if (e < -6) {
        /* subnormal: count steps of 2^-9, rounded half to even */
        double steps = ldexp(a, 9);          /* exact: power-of-two scale */
        double r = nearbyint(steps);         /* default mode: ties to even */
        code = (uint32_t)r;                  /* r == 8 is the smallest normal, code 0x08 */
    } else {
        double frac8 = (ldexp(a, -e) - 1.0) * 8.0; /* exact: 24-bit significand */
        double r = nearbyint(frac8);
        int ee = e;
        if (r == 8.0) {
            r = 0.0;
            ee += 1;
        }
        code = ((uint32_t)(ee + 7) << 3) | (uint32_t)r;
        if (code > 0x7Eu)
            code = 0x7Eu;
    }
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------- */
/* Dispatch with fused FP8 quantisation (UBEP Table 3: DeepSeek-R1/V3.2 run    */
/* W8A8; the pages give no more than that).  Reading used here: 1 x 128 blocks */
/* along H per token row; amax = max |x|; scale = amax / 448; the codes are    */
/* e4m3_satfinite(x * (448 / amax)), both quotients rounded to nearest once.  */
/* A block with amax == 0, or whose 448 / amax overflows binary32, stores      */
/* scale 1 and signed zero codes.  Scales are float32 row-major [N, H/128].    */
/* The same codes and scale go to every one of the token's k slots.           */
/* ------------------------------------------------------------------------- */
int oracle_dispatch_quant(int T, int H, int k, const uint16_t *x, const int32_t *slot_of,
                          uint8_t *recv_q, float *recv_scales)
{
    if (T < 0 || H < 128 || H % 128 != 0 || k < 1)
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    const int B = H / 128;
    uint8_t *qrow = (uint8_t *)malloc((size_t)H);
    float *srow = (float *)malloc(sizeof(float) * (size_t)B);
    if (!qrow || !srow) {
        free(qrow);
        free(srow);
        return ORACLE_ERR_INVALID_ARG;
    }
    for (int t = 0; t < T; ++t) {
        const uint16_t *xr = x + (int64_t)t * H;
        for (int b = 0; b < B; ++b) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(bf16_to_f32(xr[b * 128 + i]));
                if (v > amax)
                    amax = v;
            }
            float inv = 0.0f;
            int zero_block = (amax == 0.0f);
            if (!zero_block) {
                inv = 448.0f / amax;
                if (isinf(inv))
                    zero_block = 1;
            }
            if (zero_block) {
                srow[b] = 1.0f;
                for (int i = 0; i < 128; ++i)
                    qrow[b * 128 + i] = (uint8_t)((xr[b * 128 + i] >> 15) << 7);
            } else {
                srow[b] = amax / 448.0f;
                for (int i = 0; i < 128; ++i) {
                    float v = bf16_to_f32(xr[b * 128 + i]);
                    float p = v * inv;
                    qrow[b * 128 + i] = oracle_e4m3_encode(p);
                }
            }
        }
        for (int j = 0; j < k; ++j) {
            int32_t s = slot_of[(int64_t)t * k + j];
            if (s < 0 || s >= N) {
                free(qrow);
                free(srow);
                return ORACLE_ERR_BAD_INDEX;
            }
            memcpy(recv_q + (int64_t)s * H, qrow, (size_t)H);
            memcpy(recv_scales + (int64_t)s * B, srow, sizeof(float) * (size_t)B);
        }
    }
    free(qrow);
    free(srow);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Combine: out[t,:] = sum_j w[t,j] * y[slot_of[t,j], :]                       */
/* HyperParallel-MoE section 2.2 (outputs weighted by routing scores and       */
/* combined; Combine accumulates the top-k contributions) and section 4.1     */
/* (contributions accumulated according to routing scores); RailWave section  */
/* 3 (combine uses the saved dispatch metadata to return rows to their token  */
/* positions).  Precision: fp32 accumulation, one fused multiply-add per slot, */
/* slots in order j = 0..k-1, starting from +0; output rounded once.           */
/* out_dtype: 0 = bf16 bits (uint16), 1 = float32.                            */
/* ------------------------------------------------------------------------- */
int oracle_combine(int T, int H, int k, const uint16_t *y, const int32_t *slot_of,
                   const float *topk_w, void *out, int out_dtype)
{
    if (T < 0 || H < 1 || k < 1 || (out_dtype != 0 && out_dtype != 1))
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t s = slot_of[(int64_t)t * k + j];
            if (s < 0 || s >= N)
                return ORACLE_ERR_BAD_INDEX;
        }
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int64_t i = (int64_t)t * k + j;
                float v = bf16_to_f32(y[(int64_t)slot_of[i] * H + h]);
                acc = fmaf(topk_w[i], v, acc);
            }
            if (out_dtype == 0)
                ((uint16_t *)out)[(int64_t)t * H + h] = oracle_f32_to_bf16(acc);
            else
                ((float *)out)[(int64_t)t * H + h] = acc;
        }
    }
    return ORACLE_OK;
}

/* The same weighted sum in binary64 (products of a binary32 weight and a bf16
   value are exact in binary64).  Used as the closed-form pin of oracle_combine. */
int oracle_combine_f64(int T, int H, int k, const uint16_t *y, const int32_t *slot_of,
                       const float *topk_w, double *out, double *abs_sum)
{
    if (T < 0 || H < 1 || k < 1)
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) {
            double acc = 0.0, mag = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t i = (int64_t)t * k + j;
                int32_t s = slot_of[i];
                if (s < 0 || s >= N)
                    return ORACLE_ERR_BAD_INDEX;
                double p = (double)topk_w[i] * (double)bf16_to_f32(y[(int64_t)s * H + h]);
                acc += p;
                mag += fabs(p);
            }
            out[(int64_t)t * H + h] = acc;
            if (abs_sum)
                abs_sum[(int64_t)t * H + h] = mag;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Backward pass.  HyperParallel-MoE section 2.2 / Figure 2(b): the backward   */
/* Dispatch is the gradient of the forward Combine, and the backward Combine   */
/* returns the input-activation gradient (the gradient of the forward          */
/* Dispatch).  With out[t] = sum_j w[t,j] * y[slot_of[t,j]]:                   */
/*   dy[slot_of[t,j]] = w[t,j] * dout[t]  (one fp32 multiply, rounded to bf16) */
/*   dw[t,j]          = <y[slot_of[t,j]], dout[t]>  (returned in binary64:     */
/*                      bf16 x bf16 products are exact, so this is the exact   */
/*                      value up to binary64 rounding; abs_sum bounds the fp32 */
/*                      summation error of an implementation)                  */
/* and with recv[slot_of[t,j]] = x[t]:                                         */
/*   dx[t] = sum_j drecv[slot_of[t,j]]  (fp32, slots in order, from +0)        */
/* ------------------------------------------------------------------------- */
int oracle_combine_backward(int T, int H, int k, const uint16_t *dout, const uint16_t *y,
                            const int32_t *slot_of, const float *topk_w, uint16_t *dy,
                            double *dw, double *dw_abs_sum)
{
    if (T < 0 || H < 1 || k < 1)
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    for (int t = 0; t < T; ++t) {
        const uint16_t *d = dout + (int64_t)t * H;
        for (int j = 0; j < k; ++j) {
            int64_t i = (int64_t)t * k + j;
            int32_t s = slot_of[i];
            if (s < 0 || s >= N)
                return ORACLE_ERR_BAD_INDEX;
            const float w = topk_w[i];
            double acc = 0.0, mag = 0.0;
            for (int h = 0; h < H; ++h) {
                const float dv = bf16_to_f32(d[h]);
                const float prod = w * dv;
                dy[(int64_t)s * H + h] = oracle_f32_to_bf16(prod);
                if (y) {
                    const double p = (double)bf16_to_f32(y[(int64_t)s * H + h]) * (double)dv;
                    acc += p;
                    mag += fabs(p);
                }
            }
            if (dw)
                dw[i] = acc;
            if (dw_abs_sum)
                dw_abs_sum[i] = mag;
        }
    }
    return ORACLE_OK;
}

int oracle_dispatch_backward(int T, int H, int k, const uint16_t *drecv, const int32_t *slot_of,
                             void *dx, int out_dtype)
{
    if (T < 0 || H < 1 || k < 1 || (out_dtype != 0 && out_dtype != 1))
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t s = slot_of[(int64_t)t * k + j];
            if (s < 0 || s >= N)
                return ORACLE_ERR_BAD_INDEX;
        }
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j)
                acc = acc + bf16_to_f32(drecv[(int64_t)slot_of[(int64_t)t * k + j] * H + h]);
            if (out_dtype == 0)
                ((uint16_t *)dx)[(int64_t)t * H + h] = oracle_f32_to_bf16(acc);
            else
                ((float *)dx)[(int64_t)t * H + h] = acc;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Rank-coalesced layout and dispatch.  UBEP section 2.3: a token may go to   */
/* several experts; RailWave section 3.1 (existing token coalescing): a token */
/* needs to cross to a rank once, however many of its experts live there.     */
/* Pair (t, j) "owns" (t, rank(e_tj)) when no earlier slot j' < j of token t  */
/* chose an expert on the same rank.  Owners get one coalesced row each:      */
/* rank-segmented, in token order inside a rank, no padding.                  */
/*   crow[t,j]      coalesced row of (t, rank(e_tj)) (owners and the rest)    */
/*   src_pair_c[c]  owner pair t*k+j of coalesced row c, for c < Nc           */
/*   expand[s]      coalesced row holding the input of slot s of the plain    */
/*                  layout: expand[slot_of[t,j]] = crow[t,j]                  */
/* and the coalesced dispatch writes recv_c[c] = x[src_pair_c[c] / k].        */
/* ------------------------------------------------------------------------- */
int oracle_layout_coalesced(int T, int k, int E, int R, const int32_t *topk_idx,
                            const int32_t *slot_of, int32_t *rank_counts_c,
                            int32_t *rank_offsets_c, int32_t *crow, int32_t *src_pair_c,
                            int32_t *expand)
{
    if (T < 0 || k < 1 || E < 1 || R < 1 || E % R != 0)
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    const int El = E / R;
    for (int64_t i = 0; i < N; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E)
            return ORACLE_ERR_BAD_INDEX;
    for (int r = 0; r < R; ++r)
        rank_counts_c[r] = 0;
    /* 1. owners and their count per rank */
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int r = topk_idx[(int64_t)t * k + j] / El;
            int owner = 1;
            for (int jj = 0; jj < j; ++jj)
                if (topk_idx[(int64_t)t * k + jj] / El == r)
                    owner = 0;
            if (owner)
                rank_counts_c[r] += 1;
        }
    }
    /* 2. exclusive scan over ranks */
    rank_offsets_c[0] = 0;
    for (int r = 0; r < R; ++r)
        rank_offsets_c[r + 1] = rank_offsets_c[r] + rank_counts_c[r];
    /* 3. owners take rows in token order; the other slots share their owner's */
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    if (!cursor)
        return ORACLE_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r)
        cursor[r] = rank_offsets_c[r];
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int64_t i = (int64_t)t * k + j;
            const int r = topk_idx[i] / El;
            int owner_j = j;
            for (int jj = j - 1; jj >= 0; --jj)
                if (topk_idx[(int64_t)t * k + jj] / El == r)
                    owner_j = jj;
            if (owner_j == j) {
                const int32_t c = cursor[r]++;
                crow[i] = c;
                src_pair_c[c] = (int32_t)i;
            } else {
                crow[i] = crow[(int64_t)t * k + owner_j];
            }
        }
    }
    free(cursor);
    for (int64_t i = 0; i < N; ++i) {
        const int32_t s = slot_of[i];
        if (s < 0 || s >= N)
            return ORACLE_ERR_BAD_INDEX;
        expand[s] = crow[i];
    }
    return ORACLE_OK;
}

int oracle_dispatch_coalesced(int T, int H, int k, const uint16_t *x, const int32_t *crow,
                              uint16_t *recv_c)
{
    if (T < 0 || H < 1 || k < 1)
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int32_t c = crow[(int64_t)t * k + j];
            if (c < 0 || c >= N)
                return ORACLE_ERR_BAD_INDEX;
            memcpy(recv_c + (int64_t)c * H, x + (int64_t)t * H, sizeof(uint16_t) * (size_t)H);
        }
    }
    return ORACLE_OK;
}

/* Rank-coalesced combine: the return path of the coalesced dispatch.  One    */
/* row per (token, destination rank) comes back, so each rank first reduces  */
/* the token's slots it holds into that row (RailWave section 3.1, token      */
/* coalescing; section 3: combine reuses the dispatch metadata).  Reading:    */
/* the returned row is bf16, like the dispatched payload.                     */
/*   pre:  partial[c] = bf16( fmaf-sum over j with crow[t,j] == c, in         */
/*         increasing j, of w[t,j] * y[slot_of[t,j]] ), from +0               */
/*   post: out[t] = sum over the token's distinct rows c, in order of their   */
/*         first slot, of float(partial[c]); fp32 adds from +0, one rounding  */
/*         to the output type                                                 */
/* ------------------------------------------------------------------------- */
int oracle_combine_coalesced_pre(int T, int H, int k, const uint16_t *y, const int32_t *slot_of,
                                 const float *topk_w, const int32_t *crow, int n_rows,
                                 uint16_t *partial)
{
    if (T < 0 || H < 1 || k < 1 || n_rows < 0)
        return ORACLE_ERR_INVALID_ARG;
    const int64_t N = (int64_t)T * k;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int64_t i = (int64_t)t * k + j;
            const int32_t c = crow[i];
            if (c < 0 || c >= n_rows)
                return ORACLE_ERR_BAD_INDEX;
            int first = 1;
            for (int jj = 0; jj < j; ++jj)
                if (crow[(int64_t)t * k + jj] == c)
                    first = 0;
            if (!first)
                continue;
            for (int h = 0; h < H; ++h) {
                float acc = 0.0f;
                for (int jj = j; jj < k; ++jj) {
                    const int64_t ii = (int64_t)t * k + jj;
                    if (crow[ii] != c)
                        continue;
                    if (slot_of[ii] < 0 || slot_of[ii] >= N)
                        return ORACLE_ERR_BAD_INDEX;
                    acc = fmaf(topk_w[ii], bf16_to_f32(y[(int64_t)slot_of[ii] * H + h]), acc);
                }
                partial[(int64_t)c * H + h] = oracle_f32_to_bf16(acc);
            }
        }
    }
    return ORACLE_OK;
}

int oracle_combine_coalesced_post(int T, int H, int k, const uint16_t *partial,
                                  const int32_t *crow, int n_rows, void *out, int out_dtype)
{
    if (T < 0 || H < 1 || k < 1 || n_rows < 0 || (out_dtype != 0 && out_dtype != 1))
        return ORACLE_ERR_INVALID_ARG;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int32_t c = crow[(int64_t)t * k + j];
            if (c < 0 || c >= n_rows)
                return ORACLE_ERR_BAD_INDEX;
        }
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                const int32_t c = crow[(int64_t)t * k + j];
                int first = 1;
                for (int jj = 0; jj < j; ++jj)
                    if (crow[(int64_t)t * k + jj] == c)
                        first = 0;
                if (first)
                    acc = acc + bf16_to_f32(partial[(int64_t)c * H + h]);
            }
            if (out_dtype == 0)
                ((uint16_t *)out)[(int64_t)t * H + h] = oracle_f32_to_bf16(acc);
            else
                ((float *)out)[(int64_t)t * H + h] = acc;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Expert parallelism across W real ranks                                     */
/*                                                                            */
/* UBEP, section 2.3 and Figure 2: before dispatch each rank allocates a      */
/* receive region partitioned by source rank and expert; senders place every  */
/* token in the region of each expert it chose; the receiver learns the       */
/* per-expert counts of every source and, in Phase 5, computes offsets from   */
/* them and reorders the tokens contiguously per expert.  UBEP section 4:     */
/* the receive address space is partitioned in advance.  StrataCL Appendix D: */
/* per-expert counts and token-local offsets are the metadata that combine    */
/* reuses to return rows.                                                     */
/*                                                                            */
/* Rank s holds the tokens [tok_off[s], tok_off[s+1]) of the concatenated     */
/* arrays (topk_idx, x, topk_w are all ranks' rows, rank by rank).  Expert e  */
/* lives on rank e / El, El = E / W.  Reading taken where the pages leave the */
/* order open: the receiver's buffer holds, for each local expert el in       */
/* order, the rows of source 0, then source 1, ..., each source's rows in its */
/* own (token, slot) order.                                                   */
/*   recv_counts [W][W][El]  recv_counts[(d*W + s)*El + el]: rows receiver d  */
/*                           gets from source s for its local expert el       */
/*   recv_base   [W+1]       first row of receiver d in recv; [W] = all rows  */
/*   src_pair    [rows]      global pair t*k + j that each received row holds */
/*   recv        [rows, H]   the received rows (bf16 bits)                    */
/* ------------------------------------------------------------------------- */
int oracle_ep_dispatch(int W, const int64_t *tok_off, int k, int E, int H,
                       const int32_t *topk_idx, const uint16_t *x, int32_t *recv_counts,
                       int64_t *recv_base, int64_t *src_pair, uint16_t *recv)
{
    if (W < 1 || k < 1 || E < 1 || E % W != 0 || H < 1 || tok_off[0] != 0)
        return ORACLE_ERR_INVALID_ARG;
    for (int s = 0; s < W; ++s)
        if (tok_off[s + 1] < tok_off[s])
            return ORACLE_ERR_INVALID_ARG;
    const int El = E / W;
    const int64_t T = tok_off[W];
    for (int64_t i = 0; i < T * k; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E)
            return ORACLE_ERR_BAD_INDEX;
    int64_t row = 0;
    for (int d = 0; d < W; ++d) {
        recv_base[d] = row;
        for (int el = 0; el < El; ++el) {
            const int e = d * El + el;
            for (int s = 0; s < W; ++s) {
                int32_t cnt = 0;
                for (int64_t t = tok_off[s]; t < tok_off[s + 1]; ++t)
                    for (int j = 0; j < k; ++j)
                        if (topk_idx[t * k + j] == e) {
                            src_pair[row] = t * k + j;
                            memcpy(recv + row * H, x + t * H, sizeof(uint16_t) * (size_t)H);
                            ++row;
                            ++cnt;
                        }
                recv_counts[((int64_t)d * W + s) * El + el] = cnt;
            }
        }
    }
    recv_base[W] = row;
    return ORACLE_OK;
}

/* The return path (combine across ranks): y holds the experts' outputs in the */
/* receive buffers' order (the layout oracle_ep_dispatch gives recv).  Every   */
/* token's output is the router-weighted sum of its k rows wherever they were  */
/* received, with the precision of oracle_combine: fp32, one fused multiply-   */
/* add per slot in slot order from +0, one rounding (HyperParallel-MoE         */
/* sections 2.2 and 4.1).  out_dtype: 0 = bf16 bits, 1 = float32.              */
int oracle_ep_combine(int W, const int64_t *tok_off, int k, int E, int H,
                      const int32_t *topk_idx, const float *topk_w, const uint16_t *y,
                      void *out, int out_dtype)
{
    if (W < 1 || k < 1 || E < 1 || E % W != 0 || H < 1 || tok_off[0] != 0 ||
        (out_dtype != 0 && out_dtype != 1))
        return ORACLE_ERR_INVALID_ARG;
    const int El = E / W;
    const int64_t T = tok_off[W];
    for (int64_t i = 0; i < T * k; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E)
            return ORACLE_ERR_BAD_INDEX;
    /* row of each pair: the same walk as the dispatch */
    int64_t *row_of = (int64_t *)malloc(sizeof(int64_t) * (size_t)(T * k > 0 ? T * k : 1));
    if (row_of == NULL)
        return ORACLE_ERR_INVALID_ARG;
    int64_t row = 0;
    for (int d = 0; d < W; ++d)
        for (int el = 0; el < El; ++el)
            for (int s = 0; s < W; ++s)
                for (int64_t t = tok_off[s]; t < tok_off[s + 1]; ++t)
                    for (int j = 0; j < k; ++j)
                        if (topk_idx[t * k + j] == d * El + el)
                            row_of[t * k + j] = row++;
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                const int64_t i = t * k + j;
                acc = fmaf(topk_w[i], bf16_to_f32(y[row_of[i] * H + h]), acc);
            }
            if (out_dtype == 0)
                ((uint16_t *)out)[t * H + h] = oracle_f32_to_bf16(acc);
            else
                ((float *)out)[t * H + h] = acc;
        }
    free(row_of);
    return ORACLE_OK;
}

/* Array forms of the two encoders, for exhaustive sweeps in the tests. */
void oracle_e4m3_encode_array(const float *f, uint8_t *q, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        q[i] = oracle_e4m3_encode(f[i]);
}

void oracle_f32_to_bf16_array(const float *f, uint16_t *b, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        b[i] = oracle_f32_to_bf16(f[i]);
}

int oracle_abi_version(void) { return 1; }
