/*
 * moe_oracle.c -- plain, slow CPU oracle for the FP4-expert MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, import or
 * call this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Sources (cited by page title / address and section):
 *   [P1]  "DeepSeek-V4揭秘：细粒度专家并行隐藏通信时延，FP4量化与TileLang协同优化百万Token上下文"
 *         (itsolotime.com/archives/32374)
 *         S1.1  four-stage MoE layer: dispatch, linear-1, linear-2, combine
 *         S1.4  6hd FLOPs per token-expert pair (gate, up, down), FP8 dispatch,
 *               BF16 combine
 *         S3.1  batch invariance, no split-K;  S3.2  no atomic-order sums
 *         S4    FP4 (MXFP4, OCP MX) expert weights with 1x32 sub-block
 *               scales, FP4->FP8 dequantisation said to be lossless
 *   [P2]  "DeepSeek V4架构学习笔记" (67808.cn/a/484462.html), DeepSeekMoE
 *         paragraph: gate activation Sqrt(Softplus(.)) replaces Sigmoid.
 *   [P4]  "DeepSeek-V4 的暗线之二" (blog.xieydd.top/deepseek-v4-control-part2),
 *         S3 determinism / batch invariance, S4 FP4 QAT.
 *
 * Where the pages leave a step open, the reading taken is written beside it
 * and marked [R].  Floating point is double unless a step is defined in fp32
 * (the gate logits' fixed fp32 order, the fp32 weight sum, the fp32 combine
 * chain) -- those are written with explicit float operations and fmaf.
 * Build with -ffp-contract=off so the compiler fuses nothing on its own.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Codecs                                                                   */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern -> float (exact widening). */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* float -> bf16 bit pattern, round to nearest even.  NaN -> canonical quiet NaN. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* FP8 E4M3 (OCP "FN" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; no infinities; 0x7f / 0xff are NaN; largest finite 448. */
double orc_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* subnormal: m * 2^-9 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even encode into E4M3, saturating finite values to +-448.
 * The sign of zero results is kept. */
uint8_t orc_e4m3_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (isnan(v))
        return 0x7f;
    if (a >= 448.0)
        return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range, quantum 2^-9; a result of 8 is the smallest normal
         * 2^-6 whose code is also 8 */
        double m = nearbyint(a * 512.0);
        return sign | (uint8_t)m;
    }
    int ex;
    frexp(a, &ex);                             /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;                            /* a in [2^E, 2^(E+1)) */
    double mq = nearbyint(ldexp(a, 3 - E));    /* in [8, 16] */
    if (mq == 16.0) {
        E += 1;
        mq = 8.0;
    }
    if (E + 7 > 15)
        return sign | 0x7e;
    unsigned code = ((unsigned)(E + 7) << 3) | (unsigned)(mq - 8.0);
    if (code > 0x7e)
        code = 0x7e;
    return sign | (uint8_t)code;
}

/* FP4 E2M1: 1 sign bit (bit 3), 2 exponent bits (bias 1), 1 mantissa bit.
 * Magnitudes for codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_decode(uint8_t code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Round-to-nearest-even encode into E2M1, saturating to +-6.  Sign kept. */
uint8_t orc_e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    if (a >= 6.0)
        return sign | 0x7;
    if (a < 1.0) {
        /* subnormal range, quantum 0.5; a result of 2 is 1.0 = code 2 */
        return sign | (uint8_t)nearbyint(2.0 * a);
    }
    int ex;
    frexp(a, &ex);
    int E = ex - 1;                            /* 0, 1 or 2 */
    double mq = nearbyint(ldexp(a, 1 - E));    /* in [2, 4] */
    if (mq == 4.0) {
        E += 1;
        mq = 2.0;
    }
    if (E > 2)
        return sign | 0x7;
    return sign | (uint8_t)(((E + 1) << 1) | (int)(mq - 2.0));
}

/* Power-of-two scale exponent for FP8 E4M3 blocks [R]: the smallest integer e
 * with amax <= 448 * 2^e, clamped to [-127, 127]; e = 0 for amax = 0.  The
 * comparison is done on exact exponent/mantissa arithmetic (no log2). */
int orc_e4m3_scale_exp(double amax)
{
    if (!(amax > 0.0))
        return 0;
    int ex;
    double f = frexp(amax, &ex);               /* amax = f * 2^ex */
    /* amax = m * 2^E with m = 2f in [1, 2), E = ex - 1; 448 = 1.75 * 2^8 */
    int e = (ex - 1) - 8 + ((2.0 * f > 1.75) ? 1 : 0);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* MXFP4 shared exponent for one 32-element block ([P1] S4 cites the OCP MX
 * format): X = floor(log2(amax)) - 2, where 2 is the largest exponent of
 * E2M1; X = -127 for an all-zero block; clamped to [-127, 127]. */
int orc_mx_scale_exp(double amax)
{
    if (!(amax > 0.0))
        return -127;
    int ex;
    frexp(amax, &ex);
    int X = (ex - 1) - 2;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X;
}

/* ------------------------------------------------------------------------ */
/* Quantisation of activations and weights                                  */
/* ------------------------------------------------------------------------ */

/* x (bf16 bits) [T][d] -> xq (E4M3 codes) [T][d] and xs (UE8M0, e + 127)
 * [T][d/128]: one power-of-two scale per token per 128 channels ([P1] S1.4
 * "FP8 dispatch"; per-128 granularity [R]).  d % 128 == 0. */
void orc_quant_act(const uint16_t *x, int T, int d, uint8_t *xq, uint8_t *xs)
{
    int G = d / 128;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        for (int g = 0; g < G; g++) {
            double amax = 0.0;
            for (int c = 0; c < 128; c++) {
                double v = fabs((double)orc_bf16_to_f32(x[(size_t)t * d + g * 128 + c]));
                if (v > amax) amax = v;
            }
            int e = orc_e4m3_scale_exp(amax);
            xs[(size_t)t * G + g] = (uint8_t)(e + 127);
            for (int c = 0; c < 128; c++) {
                double v = (double)orc_bf16_to_f32(x[(size_t)t * d + g * 128 + c]);
                xq[(size_t)t * d + g * 128 + c] = orc_e4m3_encode(ldexp(v, -e));
            }
        }
    }
}

/* w fp32 [E][N][K] -> w_fp4 [E][N][K/2] (two E2M1 codes per byte, low nibble
 * holds the even K index [R]) and w_scale [E][N][K/32] (UE8M0 byte X + 127),
 * following the MXFP4 rule ([P1] S4; [P4] S4).  K % 32 == 0. */
void orc_pack_fp4(const float *w, int E, int N, int K, uint8_t *w_fp4, uint8_t *w_scale)
{
    long rows = (long)E * N;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; r++) {
        const float *src = w + r * (long)K;
        for (int b = 0; b < K / 32; b++) {
            double amax = 0.0;
            for (int c = 0; c < 32; c++) {
                double v = fabs((double)src[b * 32 + c]);
                if (v > amax) amax = v;
            }
            int X = orc_mx_scale_exp(amax);
            w_scale[r * (K / 32) + b] = (uint8_t)(X + 127);
            for (int c = 0; c < 32; c += 2) {
                uint8_t lo = orc_e2m1_encode(ldexp((double)src[b * 32 + c], -X));
                uint8_t hi = orc_e2m1_encode(ldexp((double)src[b * 32 + c + 1], -X));
                w_fp4[r * (K / 2) + (b * 32 + c) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* FP8 weights for the backward pass ("DeepSeek-V4揭秘…" section 4, FP4 QAT:
 * the FP4 weights are dequantised to FP8 for compute, losslessly while the
 * 1x32 sub-block scales of each 128x128 FP8 block stay within a ratio; the
 * backward uses these FP8 weights, and 128x128 blocks transpose without
 * re-quantisation).
 * For each 128x128 block of W[e] ([N][K]): S = the largest sub-block
 * exponent X in the block, the block exponent B = S - 6 clamped to >= -127
 * [R]; each element becomes E4M3_RNE(code_value * 2^(X - B)), exact whenever
 * X - B >= -8.  Output transposed: w8t [E][K][N] E4M3 codes, s8t
 * [E][K/128][N/128] UE8M0 bytes B + 127.  Input in the row-major layout of
 * orc_pack_fp4.  N % 128 == 0, K % 128 == 0. */
void orc_fp4_to_fp8t(const uint8_t *w_fp4, const uint8_t *w_scale, int E, int N, int K, uint8_t *w8t,
                     uint8_t *s8t)
{
    const int NB = N / 128, KB = K / 128;
#pragma omp parallel for schedule(static)
    for (long blk = 0; blk < (long)E * NB * KB; blk++) {
        const int e = (int)(blk / ((long)NB * KB));
        const int bn = (int)((blk / KB) % NB);
        const int bk = (int)(blk % KB);
        int S = -127;
        for (int n = bn * 128; n < bn * 128 + 128; n++)
            for (int j = bk * 4; j < bk * 4 + 4; j++) {
                int X = (int)w_scale[((long)e * N + n) * (K / 32) + j] - 127;
                if (X > S) S = X;
            }
        int B = S - 6;
        if (B < -127) B = -127;
        s8t[((long)e * KB + bk) * NB + bn] = (uint8_t)(B + 127);
        for (int n = bn * 128; n < bn * 128 + 128; n++)
            for (int k = bk * 128; k < bk * 128 + 128; k++) {
                const long row = (long)e * N + n;
                const uint8_t byte = w_fp4[row * (K / 2) + k / 2];
                const uint8_t code = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
                const int X = (int)w_scale[row * (K / 32) + k / 32] - 127;
                w8t[((long)e * K + k) * N + n] = orc_e4m3_encode(ldexp(orc_e2m1_decode(code), X - B));
            }
    }
}

/* ------------------------------------------------------------------------ */
/* Gate                                                                     */
/* ------------------------------------------------------------------------ */

/* Gate logits in a fixed fp32 order [R] (needed so that routing is exactly
 * reproducible): for each (t, e), 32 partial sums run over the channels
 * i = l, l+32, l+64, ... with fmaf; they are then added as a fixed binary
 * tree (offsets 16, 8, 4, 2, 1: partial[l] = partial[l] + partial[l+off]).
 * The optional per-expert bias is added last, in fp32.
 * x bf16 [T][d], gate_w fp32 [d][E], bias fp32 [E] or NULL, z fp32 [T][E]. */
void orc_gate_logits(const uint16_t *x, const float *gate_w, const float *bias,
                     int T, int d, int E, float *z)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        for (int e = 0; e < E; e++) {
            float part[32];
            for (int l = 0; l < 32; l++) {
                float acc = 0.0f;
                for (int i = l; i < d; i += 32)
                    acc = fmaf(orc_bf16_to_f32(x[(size_t)t * d + i]), gate_w[(size_t)i * E + e], acc);
                part[l] = acc;
            }
            for (int off = 16; off >= 1; off /= 2)
                for (int l = 0; l < off; l++)
                    part[l] = part[l] + part[l + off];
            float zz = part[0];
            if (bias)
                zz = zz + bias[e];
            z[(size_t)t * E + e] = zz;
        }
    }
}

/* sqrt(softplus(z)) ([P2], DeepSeekMoE: the affinity activation), evaluated in
 * double with softplus(z) = max(z, 0) + log1p(exp(-|z|)) and rounded to fp32. */
float orc_gate_score(float z)
{
    double zd = (double)z;
    double sp = (zd > 0.0 ? zd : 0.0) + log1p(exp(-fabs(zd)));
    return (float)sqrt(sp);
}

/* Top-k selection and renormalisation for every token.
 * Selection [R]: the k largest logits z under the total order (z descending,
 * then expert index ascending); sqrt(softplus(.)) is strictly increasing, so
 * this is the top-k of the scores.  Slot j is the j-th selected expert.
 * Weights: s_j = score(z_j), w_j = s_j / S with S the fp32 sum of s_j in slot
 * order (renormalisation to sum 1 as the workload states); S == 0 gives
 * w_j = 1/k [R].  No routed scaling factor [R].
 * Logits must be finite.  Returns 0, or -1 if a token had no selectable
 * expert (a non-finite logit). */
int orc_topk(const float *z, int T, int E, int k, int32_t *idx, float *w)
{
    int bad = 0;
    if (k < 1 || k > 64 || k > E || E > 1024)
        return -3;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int t = 0; t < T; t++) {
        const float *zt = z + (size_t)t * E;
        unsigned char taken[1024];
        float s[64];
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e])
                    continue;
                if (best < 0 || zt[e] > zt[best])
                    best = e;
            }
            if (best < 0 || !isfinite(zt[best])) {
                bad = 1;
                best = (best < 0) ? 0 : best;
            }
            taken[best] = 1;
            idx[(size_t)t * k + j] = best;
            s[j] = orc_gate_score(zt[best]);
        }
        float S = 0.0f;
        for (int j = 0; j < k; j++)
            S = S + s[j];
        for (int j = 0; j < k; j++)
            w[(size_t)t * k + j] = (S == 0.0f) ? 1.0f / (float)k : s[j] / S;
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Dispatch plan                                                            */
/* ------------------------------------------------------------------------ */

/* Expert-contiguous layout of the P = T*k token-expert pairs ([P1] S1.1
 * dispatch stage; S3.2 fixed token order).  Pair p = t*k + j.  sorted_pair
 * lists the pairs grouped by ascending expert and, within an expert, in
 * ascending p (a stable counting sort); expert_offsets[e] is where expert e's
 * group starts (expert_offsets[E] = P); pair_pos is the inverse permutation.
 * Returns -1 if an expert index is out of range. */
int orc_dispatch_plan(const int32_t *idx, int T, int E, int k,
                      int32_t *expert_offsets, int32_t *sorted_pair, int32_t *pair_pos)
{
    long P = (long)T * k;
    long *cnt = (long *)calloc((size_t)E + 1, sizeof(long));
    if (!cnt)
        return -2;
    for (long p = 0; p < P; p++) {
        if (idx[p] < 0 || idx[p] >= E) {
            free(cnt);
            return -1;
        }
        cnt[idx[p]]++;
    }
    long run = 0;
    for (int e = 0; e < E; e++) {
        expert_offsets[e] = (int32_t)run;
        run += cnt[e];
        cnt[e] = expert_offsets[e];            /* becomes the next free slot */
    }
    expert_offsets[E] = (int32_t)run;
    for (long p = 0; p < P; p++) {
        long pos = cnt[idx[p]]++;
        sorted_pair[pos] = (int32_t)p;
        pair_pos[p] = (int32_t)pos;
    }
    free(cnt);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Expert FFN and combine                                                   */
/* ------------------------------------------------------------------------ */

static double dq_fp4(const uint8_t *w_fp4, const uint8_t *w_scale, long row, int K, int i)
{
    uint8_t byte = w_fp4[row * (K / 2) + i / 2];
    uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xf);
    int X = (int)w_scale[row * (K / 32) + i / 32] - 127;
    return ldexp(orc_e2m1_decode(code), X);
}

/* One token-expert pair: the SwiGLU expert FFN of [P1] S1.4 (gate, up and
 * down projections) on FP8 activations and FP4 weights.
 *   a_i   = E4M3(xq[i]) * 2^(xs[i/128]-127)               (dequantised input)
 *   g_n   = fp32( sum_i a_i * W13[n][i] )                  n <  inter (gate rows) [R]
 *   u_n   = fp32( sum_i a_i * W13[inter+n][i] )            (up rows)              [R]
 *   h_n   = fp32( silu(g_n) * u_n ),  silu(g) = g / (1 + exp(-g))
 *   hq,hs = E4M3 codes of h with one power-of-two scale per 128 channels  [R]
 *   y_m   = bf16( fp32( sum_n E4M3(hq[n]) 2^(hs-127) * W2[m][n] ) )
 * Weight elements are dequantised exactly (E2M1 code * 2^(scale-127)); every
 * product is exact in double and the sums run in double in index order.
 * xq/xs: one token's row; y: d bf16 values.  Scratch a (max(d, inter)
 * doubles), h, hq, hs sized by the caller. */
void orc_expert_pair(const uint8_t *xq, const uint8_t *xs, int e,
                     const uint8_t *w13_fp4, const uint8_t *w13_scale,
                     const uint8_t *w2_fp4, const uint8_t *w2_scale,
                     int d, int inter, double *a, float *h, uint8_t *hq, uint8_t *hs, uint16_t *y)
{
    long row13 = (long)e * 2 * inter;
    for (int i = 0; i < d; i++)
        a[i] = ldexp(orc_e4m3_decode(xq[i]), (int)xs[i / 128] - 127);
    for (int n = 0; n < inter; n++) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; i++) {
            g += a[i] * dq_fp4(w13_fp4, w13_scale, row13 + n, d, i);
            u += a[i] * dq_fp4(w13_fp4, w13_scale, row13 + inter + n, d, i);
        }
        float gf = (float)g, uf = (float)u;
        double gd = (double)gf;
        h[n] = (float)(gd / (1.0 + exp(-gd)) * (double)uf);
    }
    for (int gblk = 0; gblk < inter / 128; gblk++) {
        double amax = 0.0;
        for (int c = 0; c < 128; c++) {
            double v = fabs((double)h[gblk * 128 + c]);
            if (v > amax) amax = v;
        }
        int ex = orc_e4m3_scale_exp(amax);
        hs[gblk] = (uint8_t)(ex + 127);
        for (int c = 0; c < 128; c++)
            hq[gblk * 128 + c] = orc_e4m3_encode(ldexp((double)h[gblk * 128 + c], -ex));
    }
    long row2 = (long)e * d;
    for (int n = 0; n < inter; n++)
        a[n] = ldexp(orc_e4m3_decode(hq[n]), (int)hs[n / 128] - 127);
    for (int m = 0; m < d; m++) {
        double acc = 0.0;
        for (int n = 0; n < inter; n++)
            acc += a[n] * dq_fp4(w2_fp4, w2_scale, row2 + m, inter, n);
        y[m] = orc_f32_to_bf16((float)acc);
    }
}

/* Whole layer forward for a list of tokens (every token is independent, so a
 * subset gives exactly the rows of the full output).
 * Stages ([P1] S1.1): gate + top-k, FP8 quantisation of the token, per-pair
 * expert FFN, and the combine: out[t] = bf16( fp32 chain over slots j of
 * fmaf(w_j, y_j, acc) ) with acc starting at 0 ([P1] S1.4 "BF16 combine";
 * fixed slot order, [P1] S3.2).
 * tokens: n_tok token indices into x (NULL = all T tokens in order).
 * out: [n_tok][d] bf16.  topk_idx/topk_w (optional): [n_tok][k].
 * Returns 0, or a negative code on bad arguments / non-finite logits. */
int orc_moe_forward(const uint16_t *x, const float *gate_w, const float *gate_bias,
                    const uint8_t *w13_fp4, const uint8_t *w13_scale,
                    const uint8_t *w2_fp4, const uint8_t *w2_scale,
                    int T, int d, int inter, int E, int k,
                    const int32_t *tokens, int n_tok,
                    uint16_t *out, int32_t *topk_idx, float *topk_w)
{
    if (d % 128 || inter % 128 || k < 1 || k > 64 || k > E || E > 1024 || T < 0)
        return -3;
    if (!tokens)
        n_tok = T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int q = 0; q < n_tok; q++) {
        int t = tokens ? tokens[q] : q;
        float *z = (float *)malloc(sizeof(float) * (size_t)E);
        int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
        float *w = (float *)malloc(sizeof(float) * (size_t)k);
        uint8_t *xq = (uint8_t *)malloc((size_t)d);
        uint8_t *xs = (uint8_t *)malloc((size_t)d / 128);
        float *h = (float *)malloc(sizeof(float) * (size_t)inter);
        uint8_t *hq = (uint8_t *)malloc((size_t)inter);
        uint8_t *hs = (uint8_t *)malloc((size_t)inter / 128);
        uint16_t *y = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)k * d);
        double *a = (double *)malloc(sizeof(double) * (size_t)(d > inter ? d : inter));
        if (!z || !idx || !w || !xq || !xs || !h || !hq || !hs || !y || !a) {
            bad |= 2;
        } else if (t < 0 || t >= T) {
            bad |= 4;
        } else {
            const uint16_t *xt = x + (size_t)t * d;
            orc_gate_logits(xt, gate_w, gate_bias, 1, d, E, z);
            if (orc_topk(z, 1, E, k, idx, w) != 0)
                bad |= 1;
            orc_quant_act(xt, 1, d, xq, xs);
            for (int j = 0; j < k; j++)
                orc_expert_pair(xq, xs, idx[j], w13_fp4, w13_scale, w2_fp4, w2_scale,
                                d, inter, a, h, hq, hs, y + (size_t)j * d);
            for (int m = 0; m < d; m++) {
                float acc = 0.0f;
                for (int j = 0; j < k; j++)
                    acc = fmaf(w[j], orc_bf16_to_f32(y[(size_t)j * d + m]), acc);
                out[(size_t)q * d + m] = orc_f32_to_bf16(acc);
            }
            if (topk_idx)
                memcpy(topk_idx + (size_t)q * k, idx, sizeof(int32_t) * (size_t)k);
            if (topk_w)
                memcpy(topk_w + (size_t)q * k, w, sizeof(float) * (size_t)k);
        }
        free(z); free(idx); free(w); free(xq); free(xs); free(h); free(hq); free(hs); free(y); free(a);
    }
    if (bad & 6)
        return -2;
    return bad ? -1 : 0;
}

/* Number of OpenMP threads the oracle's parallel loops use (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int orc_num_threads(void) { return omp_get_max_threads(); }
#else
int orc_num_threads(void) { return 1; }
#endif
