/*
 * ep_oracle.c -- plain, slow, obviously correct CPU oracle for the MoE
 * expert-parallel token layout -> dispatch -> combine path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Every function follows the definition on the pages, in the pages' order:
 *   - "Normal Mode API" (sgl-kernel-npu DeepEP, NORMAL_API.md):
 *       dispatch parameters num_tokens_per_rank / is_token_in_rank /
 *       num_tokens_per_expert / topk_idx (-1 = no expert) / expert_alignment,
 *       return values recv_x formats and num_recv_tokens_per_expert_list
 *       ("aligned"), and combine ("multiply by weights and sum").
 *   - "aclnnMoeDistributeDispatchV2" (CANN), Formula section: quantMode 0
 *       (no quant), quantMode 1 (static, int8, with scales of shape (1,),
 *       (H,) or (E,H)), quantMode 2 (per-token dynamic, int8 or FP8
 *       destination), quantMode 3 (per-group dynamic, FP8), quantMode 4 (MX,
 *       sharedExp = floor(log2(max)) - emax), optional smooth scales
 *       (xFp32 = CastToFp32(X) x scales) for quantModes 1-3, xActiveMask, and
 *       the constraint that localExpertNum = moeExpertNum / epWorldSize.
 *   - "max.nn.comm.ep.EPBatchManager" (Modular MAX): ep_dispatch outputs
 *       (expert_start_indices, expert_ids, expert_usage_stats) and ep_combine
 *       (weighted sum of routed outputs plus fused shared-expert outputs).
 *
 * Readings of points the pages leave open (each is listed in the design
 * notes): one receive row per valid (token, k); rows grouped by destination
 * rank, then local expert, then (source rank, token, k) ascending; padding
 * rows at the end of each expert segment, all bytes zero; int8 inverse scale
 * = fl(1/s); MX amax over each 32-element block of |x|; e8m0 byte = se + 127
 * (the decode scale 2^se); fp8/fp4 casts round to nearest even and saturate
 * to the largest finite value, keeping the sign of zero; e2m1 element 2i in
 * the low nibble of byte i; per-group quantisation uses groups of 128
 * elements; static int8 saturates to [-128, 127].
 *
 * Compile without FMA contraction or fast-math:
 *   gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 *
 * Floating point inputs are assumed finite.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Quant modes, numbered as in the C-ABI header's enum (the values are part of
 * the interface contract, not shared code). */
enum { Q_NONE = 0, Q_INT8_STATIC = 1, Q_INT8 = 2, Q_E4M3 = 4, Q_E5M2 = 5, Q_E2M1 = 6,
       Q_FP8T_E4M3 = 7, Q_FP8T_E5M2 = 8, Q_FP8G_E4M3 = 9, Q_FP8G_E5M2 = 10 };

/* Kinds of the optional input scales of quantModes 1-3 (CANN: a scalar (1,), a
 * smooth weight shared by all experts (H,), or one row per expert (E, H)). */
enum { S_NONE = 0, S_SCALAR = 1, S_CHANNEL = 2, S_EXPERT = 3 };

/* Elements per group of the per-group dynamic quantisation (quantMode 3);
 * the page's per-group buffer rule aligns H to 128. */
#define GROUP 128

void oracle_expert_rows(int64_t nrows, const int64_t* rows, const int32_t* row_expert,
                        int H, int q, const uint8_t* data, const uint8_t* scales,
                        int mark_mod, uint16_t* y);

/* Status values returned by oracle_layout. */
enum { O_OK = 0, O_CAPACITY = 3, O_BAD_EXPERT = 4 };

/* ------------------------------------------------------------------------ */
/* Number formats, written from their bit-level definitions.                */
/* ------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bfloat16 is the upper half of an IEEE binary32. */
float oracle_bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/* Round a binary32 to the nearest bfloat16, ties to the even code.  The two
 * candidates are the value truncated toward zero and the next code up in
 * magnitude; the one past the largest finite value is infinity, which the
 * comparison treats as 2^128 (the IEEE overflow rule). */
uint16_t oracle_bf16_from_f32(float f) {
    uint32_t u = bits_from_f32(f);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t mag = u & 0x7fffffffu;
    uint16_t lo = (uint16_t)(mag >> 16);            /* truncated code */
    uint16_t hi = (uint16_t)(lo + 1);               /* next code up   */
    if (lo == 0x7f80u) return (uint16_t)(sign | lo); /* infinity in, infinity out */
    double a = (double)f32_from_bits(mag);
    double vlo = (double)f32_from_bits((uint32_t)lo << 16);
    double vhi = (hi == 0x7f80u) ? ldexp(1.0, 128) : (double)f32_from_bits((uint32_t)hi << 16);
    double dlo = a - vlo, dhi = vhi - a;
    uint16_t pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = (lo & 1u) ? hi : lo;
    return (uint16_t)(sign | pick);
}

/* The three small float formats of the MX encodings (OCP MX v1.0):
 *   e4m3 (float8_e4m3fn): 4 exponent bits, bias 7, 3 mantissa bits, no
 *        infinities, S.1111.111 is NaN, largest finite 448 = 1.75 * 2^8;
 *   e5m2 (float8_e5m2):   5 exponent bits, bias 15, 2 mantissa bits, IEEE
 *        style infinities/NaN in exponent 31, largest finite 57344 = 1.75*2^15;
 *   e2m1 (float4_e2m1fn): 2 exponent bits, bias 1, 1 mantissa bit, no
 *        infinities or NaN, largest finite 6 = 1.5 * 2^2.
 * emax is the unbiased exponent of the largest finite value: 8, 15, 2. */
typedef struct { int ebits, mbits, bias, maxcode, emax; } mini_fmt;

static mini_fmt fmt_of(int q) {
    mini_fmt m;
    if (q == Q_E4M3) { m.ebits = 4; m.mbits = 3; m.bias = 7;  m.maxcode = 0x7e; m.emax = 8; }
    else if (q == Q_E5M2) { m.ebits = 5; m.mbits = 2; m.bias = 15; m.maxcode = 0x7b; m.emax = 15; }
    else { m.ebits = 2; m.mbits = 1; m.bias = 1; m.maxcode = 0x7; m.emax = 2; }
    return m;
}

/* Magnitude of a non-negative finite code: subnormal when the exponent field
 * is zero (M * 2^(1-bias-mbits)), normal otherwise ((1 + M/2^mbits) * 2^(E-bias)). */
static double mini_value(mini_fmt m, int code) {
    int ef = code >> m.mbits;
    int mf = code & ((1 << m.mbits) - 1);
    if (ef == 0) return ldexp((double)mf, 1 - m.bias - m.mbits);
    return ldexp(1.0 + (double)mf / (double)(1 << m.mbits), ef - m.bias);
}

/* Value of any code of the format (sign bit above the magnitude bits). */
double oracle_mini_decode(int q, int code) {
    mini_fmt m = fmt_of(q);
    int sbit = 1 << (m.ebits + m.mbits);
    double v = mini_value(m, code & (sbit - 1));
    return (code & sbit) ? -v : v;
}

/* Encode a finite value: round to the nearest representable magnitude, ties
 * to the even code (codes are monotone in magnitude, so the code's lowest bit
 * is the mantissa's lowest bit), saturating at the largest finite value.  The
 * sign bit is kept, so a negative value that rounds to zero gives -0. */
int oracle_mini_encode(int q, float v) {
    mini_fmt m = fmt_of(q);
    int sbit = 1 << (m.ebits + m.mbits);
    int neg = signbit(v) ? 1 : 0;
    double a = fabs((double)v);
    /* largest code c with value(c) <= a, by bisection over [0, maxcode] */
    int lo = 0, hi = m.maxcode;
    if (a >= mini_value(m, m.maxcode)) {
        lo = m.maxcode;
    } else {
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (mini_value(m, mid) <= a) lo = mid; else hi = mid;
        }
    }
    int c = lo;
    if (c < m.maxcode) {
        double dlo = a - mini_value(m, c);
        double dhi = mini_value(m, c + 1) - a;
        if (dhi < dlo || (dhi == dlo && (c & 1))) c = c + 1;
    }
    return neg ? (c | sbit) : c;
}

/* Round to nearest integer, ties to even, written out: floor, then compare
 * the fraction with one half.  Exact for |v| < 2^23. */
static float round_half_even(float v) {
    float f = floorf(v);
    float d = v - f;
    if (d > 0.5f) return f + 1.0f;
    if (d < 0.5f) return f;
    return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
}

/* ------------------------------------------------------------------------ */
/* quantMode 2: per-token dynamic int8 (CANN formula, Case 3).              */
/*   xFp32 = CastToFp32(X)   (smooth scales are null here: factor 1)         */
/*   dynamicScales = dstTypeMax / Max(Abs(xFp32)),  dstTypeMax = 127         */
/*   quantOut = CastToInt8(xFp32 * dynamicScales)  (round half even)         */
/*   sent scale = 1.0 / dynamicScales                                        */
/* An all-zero row has dynamicScales = +inf; its codes are 0 and its sent    */
/* scale is 1/inf = 0.  Non-finite input follows IEEE arithmetic: the        */
/* maximum skips NaN elements (a running greater-than maximum), an infinite  */
/* element gives dynamicScales 0, a row of subnormals overflows 127/amax to  */
/* +inf (codes +-127 from +-inf products), and a NaN product converts to 0.  */
/* ------------------------------------------------------------------------ */
/* The scaled input of quantModes 1-3: xFp32 = CastToFp32(X) x scales, one
 * factor per element (smooth == NULL: no scales, factor 1, no multiply). */
static float scaled_x(const uint16_t* x, const float* smooth, int h) {
    float v = oracle_bf16_to_f32(x[h]);
    return smooth ? v * smooth[h] : v;
}

/* Per-token int8 with optional smooth scales (the row multiplied by them
 * first). */
void oracle_quant_int8_row_scaled(int H, const uint16_t* x, const float* smooth, int8_t* q, float* inv) {
    float amax = 0.0f;
    for (int h = 0; h < H; ++h) {
        float a = fabsf(scaled_x(x, smooth, h));
        if (a > amax) amax = a;
    }
    float s = 127.0f / amax;
    for (int h = 0; h < H; ++h) {
        float r = 0.0f;
        if (amax > 0.0f) {
            r = round_half_even(scaled_x(x, smooth, h) * s);
            if (r != r) r = 0.0f;   /* NaN product (0 x inf, inf x 0, a NaN input): code 0 */
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
        }
        q[h] = (int8_t)(int)r;
    }
    *inv = 1.0f / s;
}

void oracle_quant_int8_row(int H, const uint16_t* x, int8_t* q, float* inv) {
    oracle_quant_int8_row_scaled(H, x, NULL, q, inv);
}

/* ------------------------------------------------------------------------ */
/* quantMode 4: MX block quantisation (CANN formula, Case 5), one shared     */
/* exponent per 32 consecutive elements of the row.                         */
/*   sharedExp = Floor(log2(max|x| over the block)) - emax, clamped to       */
/*               [-127, 127]; a block whose max is zero or subnormal takes   */
/*               -127 (the smallest e8m0 exponent)                           */
/*   dynamicScales = 2^sharedExp                                             */
/*   quantOut = Cast(X / dynamicScales)                                      */
/*   scale byte (e8m0) = sharedExp + 127                                     */
/* floor(log2(a)) of a normal binary32 a is its unbiased exponent field.     */
/* e2m1 codes are packed two per byte, element 2i in the low nibble.         */
/* ------------------------------------------------------------------------ */
void oracle_quant_mx_row(int H, int q, const uint16_t* x, uint8_t* codes, uint8_t* scales) {
    mini_fmt m = fmt_of(q);
    if (q == Q_E2M1) memset(codes, 0, (size_t)H / 2);
    for (int b = 0; b < H / 32; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(oracle_bf16_to_f32(x[b * 32 + i]));
            if (a > amax) amax = a;
        }
        int expfield = (int)((bits_from_f32(amax) >> 23) & 0xffu);
        int se;
        if (expfield == 0) {
            se = -127;
        } else {
            se = (expfield - 127) - m.emax;
            if (se < -127) se = -127;
            if (se > 127) se = 127;
        }
        scales[b] = (uint8_t)(se + 127);
        float dyn = ldexpf(1.0f, se);
        for (int i = 0; i < 32; ++i) {
            int h = b * 32 + i;
            float v = oracle_bf16_to_f32(x[h]) / dyn;
            int c = oracle_mini_encode(q, v);
            if (q == Q_E2M1) codes[h / 2] |= (uint8_t)(c << (4 * (h & 1)));
            else codes[h] = (uint8_t)c;
        }
    }
}

/* CANN Formula, Case 3 with an FP8 destination (quantMode 2, FLOAT8_E4M3FN or
 * FLOAT8_E5M2): dynamicScales = dstTypeMax / Max(Abs(xFp32)) over the row,
 * quantOut = Cast(xFp32 * dynamicScales) (round to nearest even, saturate),
 * sent scale 1.0 / dynamicScales.  dstTypeMax: 448 (e4m3), 57344 (e5m2).  An
 * all-zero row gives codes 0 and scale 0. */
void oracle_quant_fp8_token_row(int H, int fp8, const uint16_t* x, const float* smooth,
                                uint8_t* codes, float* inv) {
    const float dmax = (fp8 == Q_E4M3) ? 448.0f : 57344.0f;
    float amax = 0.0f;
    for (int h = 0; h < H; ++h) {
        float a = fabsf(scaled_x(x, smooth, h));
        if (a > amax) amax = a;
    }
    float s = dmax / amax;
    for (int h = 0; h < H; ++h)
        codes[h] = (amax > 0.0f) ? (uint8_t)oracle_mini_encode(fp8, scaled_x(x, smooth, h) * s) : 0;
    *inv = 1.0f / s;
}

/* CANN Formula, Case 4 (quantMode 3, per-group dynamic; FP8 destinations):
 * the per-token rule applied to every group of 128 consecutive elements;
 * one float32 scale (1.0 / dynamicScales) per group. */
void oracle_quant_fp8_group_row(int H, int fp8, const uint16_t* x, const float* smooth,
                                uint8_t* codes, float* inv) {
    for (int g = 0; g < H / GROUP; ++g)
        oracle_quant_fp8_token_row(GROUP, fp8, x + g * GROUP, smooth ? smooth + g * GROUP : NULL,
                                   codes + g * GROUP, inv + g);
}

/* CANN Formula, Case 2 (quantMode 1, static, INT8 destination):
 * quantOut = Cast(xFp32, int8), round to nearest even, saturated to the int8
 * range [-128, 127]; no scale is sent (the receiver knows the static scales). */
void oracle_quant_int8_static_row(int H, const uint16_t* x, const float* smooth, int8_t* q) {
    for (int h = 0; h < H; ++h) {
        float r = round_half_even(scaled_x(x, smooth, h));
        if (r != r) r = 0.0f;   /* NaN input or product: code 0 */
        if (r > 127.0f) r = 127.0f;
        if (r < -128.0f) r = -128.0f;
        q[h] = (int8_t)(int)r;
    }
}

/* Encode one row with an optional smooth-scale row (quantModes 1-3 only). */
void oracle_encode_row_scaled(int q, int H, const uint16_t* x, const float* smooth,
                              uint8_t* data, uint8_t* scale) {
    switch (q) {
        case Q_INT8_STATIC: oracle_quant_int8_static_row(H, x, smooth, (int8_t*)data); break;
        case Q_INT8: oracle_quant_int8_row_scaled(H, x, smooth, (int8_t*)data, (float*)scale); break;
        case Q_FP8T_E4M3: oracle_quant_fp8_token_row(H, Q_E4M3, x, smooth, data, (float*)scale); break;
        case Q_FP8T_E5M2: oracle_quant_fp8_token_row(H, Q_E5M2, x, smooth, data, (float*)scale); break;
        case Q_FP8G_E4M3: oracle_quant_fp8_group_row(H, Q_E4M3, x, smooth, data, (float*)scale); break;
        case Q_FP8G_E5M2: oracle_quant_fp8_group_row(H, Q_E5M2, x, smooth, data, (float*)scale); break;
        default: break;
    }
}

/* Bytes of one receive row's data and scale parts for a quant mode. */
int64_t oracle_row_data_bytes(int q, int H) {
    if (q == Q_NONE) return 2 * (int64_t)H;
    if (q == Q_E2M1) return H / 2;
    return H;
}
int64_t oracle_row_scale_bytes(int q, int H) {
    if (q == Q_NONE || q == Q_INT8_STATIC) return 0;
    if (q == Q_INT8 || q == Q_FP8T_E4M3 || q == Q_FP8T_E5M2) return 4;
    if (q == Q_FP8G_E4M3 || q == Q_FP8G_E5M2) return 4 * (H / GROUP);
    return H / 32;
}

/* Encode one bf16 source row into the receive-row format. */
void oracle_encode_row(int q, int H, const uint16_t* x, uint8_t* data, uint8_t* scale) {
    if (q == Q_NONE) memcpy(data, x, 2 * (size_t)H);
    else if (q == Q_INT8) oracle_quant_int8_row(H, x, (int8_t*)data, (float*)scale);
    else if (q == Q_E4M3 || q == Q_E5M2 || q == Q_E2M1) oracle_quant_mx_row(H, q, x, data, scale);
    else oracle_encode_row_scaled(q, H, x, NULL, data, scale);
}

/* Encode n consecutive source rows (rows of H bf16 elements) with
 * oracle_encode_row: the per-token encoding that dispatch copies to each of
 * the token's receive rows. */
void oracle_encode_rows(int q, int H, int64_t n, const uint16_t* x, uint8_t* data, uint8_t* scales) {
    int64_t db = oracle_row_data_bytes(q, H), sb = oracle_row_scale_bytes(q, H);
    for (int64_t i = 0; i < n; ++i)
        oracle_encode_row(q, H, x + i * H, data + i * db, sb ? scales + i * sb : NULL);
}

/* ------------------------------------------------------------------------ */
/* Routing layout.                                                          */
/*                                                                          */
/* R logical ranks, T tokens per rank, E experts, L = E / R local experts   */
/* per rank, K = topk, alpha = expert_alignment.  Expert e lives on rank     */
/* e / L as local expert e % L (no shared-expert ranks).                    */
/*                                                                          */
/* Outputs (all caller-allocated):                                          */
/*   cnt[R][E]            entries source rank s sends to expert e           */
/*                        (num_tokens_per_expert of rank s)                 */
/*   itr[R][T][R]         is_token_in_rank: token (s,t) has an expert on j  */
/*   ntpr[R][R]           num_tokens_per_rank: tokens of s that go to j     */
/*   recv_cnt[E]          entries expert e receives from all sources        */
/*   aligned[E]           recv_cnt rounded up to a multiple of alpha        */
/*   expert_start[R][L+1] row offset of each local expert inside rank j     */
/*   rank_base[R+1]       first global row of rank j; rank_base[R] = rows   */
/*   src_prefix[R][E]     entries sources s' < s send to expert e           */
/*   dst_row[R][T][K]     receive row of each entry, -1 for no expert       */
/*   recv_src[recv_cap]   source token s*T+t of each row, -1 on padding     */
/*   expert_ids[R][L]     local expert id of each grouped-matmul slot       */
/*   usage[R][2]          [max aligned count, experts with count > 0]       */
/*                                                                          */
/* Returns O_OK, O_BAD_EXPERT (an id outside [-1, E), treated as -1) or      */
/* O_CAPACITY (rows > recv_cap; recv_src holds only rows below recv_cap).   */
/* ------------------------------------------------------------------------ */
int oracle_layout(int R, int T, int E, int K, int alpha, const int64_t* topk,
                  int64_t recv_cap,
                  int32_t* cnt, uint8_t* itr, int32_t* ntpr,
                  int32_t* recv_cnt, int32_t* aligned,
                  int32_t* expert_start, int64_t* rank_base,
                  int32_t* src_prefix, int32_t* dst_row, int32_t* recv_src,
                  int32_t* expert_ids, int32_t* usage) {
    int status = O_OK;
    int L = E / R;

    /* 1. counts per (source rank, expert), token-in-rank flags, tokens per rank */
    memset(cnt, 0, sizeof(int32_t) * (size_t)R * E);
    memset(itr, 0, (size_t)R * T * R);
    memset(ntpr, 0, sizeof(int32_t) * (size_t)R * R);
    for (int s = 0; s < R; ++s) {
        for (int t = 0; t < T; ++t) {
            int64_t n = (int64_t)s * T + t;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk[n * K + k];
                if (e == -1) continue;
                if (e < -1 || e >= E) { status = O_BAD_EXPERT; continue; }
                cnt[(int64_t)s * E + e] += 1;
                itr[n * R + e / L] = 1;
            }
            for (int j = 0; j < R; ++j) ntpr[(int64_t)s * R + j] += itr[n * R + j];
        }
    }

    /* 2. received entries per expert, rounded up to the alignment */
    for (int e = 0; e < E; ++e) {
        int32_t c = 0;
        for (int s = 0; s < R; ++s) c += cnt[(int64_t)s * E + e];
        recv_cnt[e] = c;
        aligned[e] = ((c + alpha - 1) / alpha) * alpha;
    }

    /* 3. row offsets of local experts inside each rank, and of each rank */
    rank_base[0] = 0;
    for (int j = 0; j < R; ++j) {
        int32_t* es = expert_start + (int64_t)j * (L + 1);
        es[0] = 0;
        for (int l = 0; l < L; ++l) es[l + 1] = es[l] + aligned[j * L + l];
        rank_base[j + 1] = rank_base[j] + es[L];
    }

    /* 4. per-expert prefix over source ranks */
    for (int e = 0; e < E; ++e) {
        int32_t acc = 0;
        for (int s = 0; s < R; ++s) {
            src_prefix[(int64_t)s * E + e] = acc;
            acc += cnt[(int64_t)s * E + e];
        }
    }

    /* 5. receive row of every entry: rank base + expert start + source prefix
     *    + running position of this entry among source s's entries for e */
    int64_t rows = rank_base[R];
    if (rows > recv_cap) status = O_CAPACITY;
    int64_t fill = rows < recv_cap ? rows : recv_cap;
    for (int64_t r = 0; r < fill; ++r) recv_src[r] = -1;
    int32_t* pos = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int s = 0; s < R; ++s) {
        memset(pos, 0, sizeof(int32_t) * (size_t)E);
        for (int t = 0; t < T; ++t) {
            int64_t n = (int64_t)s * T + t;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk[n * K + k];
                if (e < 0 || e >= E) { dst_row[n * K + k] = -1; continue; }
                int j = (int)(e / L), l = (int)(e % L);
                int64_t d = rank_base[j] + expert_start[(int64_t)j * (L + 1) + l]
                          + src_prefix[(int64_t)s * E + e] + pos[e];
                pos[e] += 1;
                dst_row[n * K + k] = (int32_t)d;
                if (d < recv_cap) recv_src[d] = (int32_t)n;
            }
        }
    }
    free(pos);

    /* 6. grouped-matmul metadata per rank */
    for (int j = 0; j < R; ++j) {
        int32_t mx = 0, active = 0;
        for (int l = 0; l < L; ++l) {
            expert_ids[(int64_t)j * L + l] = l;
            if (aligned[j * L + l] > mx) mx = aligned[j * L + l];
            if (recv_cnt[j * L + l] > 0) active += 1;
        }
        usage[2 * j] = mx;
        usage[2 * j + 1] = active;
    }
    return status;
}

/* xActiveMask (CANN aclnnMoeDistributeDispatchV2): a false token (1-D mask,
 * [R*T]) or a false entry (2-D mask, [R*T*K]) does not take part in the
 * communication -- it is laid out exactly like an entry whose topk id is -1.
 * The page asks 1-D masks to be a prefix of true values; any pattern gives a
 * well-defined layout here. */
int oracle_layout_masked(int R, int T, int E, int K, int alpha, const int64_t* topk,
                         const uint8_t* mask, int mask_dims, int64_t recv_cap,
                         int32_t* cnt, uint8_t* itr, int32_t* ntpr,
                         int32_t* recv_cnt, int32_t* aligned,
                         int32_t* expert_start, int64_t* rank_base,
                         int32_t* src_prefix, int32_t* dst_row, int32_t* recv_src,
                         int32_t* expert_ids, int32_t* usage) {
    int64_t n_ent = (int64_t)R * T * K;
    int64_t* t2 = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_ent > 0 ? n_ent : 1));
    for (int64_t i = 0; i < n_ent; ++i) {
        int active = (mask_dims == 1) ? mask[i / K] : mask[i];
        t2[i] = active ? topk[i] : -1;
    }
    int st = oracle_layout(R, T, E, K, alpha, t2, recv_cap, cnt, itr, ntpr, recv_cnt, aligned,
                           expert_start, rank_base, src_prefix, dst_row, recv_src, expert_ids, usage);
    free(t2);
    return st;
}

/* ------------------------------------------------------------------------ */
/* Per-rank receive layout (DeepEP "Normal Mode API" dispatch returns:       */
/* recv_x has one row per received token, recv_topk_idx / recv_topk_weights */
/* give each received token's top-k as seen by the receiving rank).         */
/*                                                                          */
/* Rank j receives every source token (s,t) with is_token_in_rank[s,t,j]=1, */
/* once, in (s, t) order; ranks are back to back.  For a received row,      */
/* recv_topk_idx[k] is the local expert id e - j*L when topk[s,t,k] lives on */
/* rank j and -1 otherwise; recv_topk_weights[k] is the token's weight for  */
/* such a local expert and 0 otherwise.                                     */
/*   tok_dst[R*T][K]   rows of the token on its destination ranks, in       */
/*                     ascending rank order, -1 padded                      */
/*   recv_src_tok[rows]  source token s*T+t of each row                     */
/*   rank_tok_base[R+1]  first row of each rank; rank_tok_base[R] = rows    */
/* Entries with ids outside [0, E) take no part.  Returns the row count.    */
/* ------------------------------------------------------------------------ */
int64_t oracle_token_layout(int R, int T, int E, int K, const int64_t* topk, const float* w,
                            int64_t cap, int32_t* tok_dst, int32_t* recv_src_tok,
                            int64_t* rank_tok_base, int64_t* recv_topk_idx,
                            float* recv_topk_weights) {
    int L = E / R;
    int64_t N = (int64_t)R * T;
    for (int64_t i = 0; i < N * K; ++i) tok_dst[i] = -1;
    int32_t* nfill = (int32_t*)calloc((size_t)(N > 0 ? N : 1), sizeof(int32_t));
    int64_t row = 0;
    for (int j = 0; j < R; ++j) {
        rank_tok_base[j] = row;
        for (int64_t n = 0; n < N; ++n) {
            int hit = 0;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk[n * K + k];
                if (e >= 0 && e < E && e / L == j) hit = 1;
            }
            if (!hit) continue;
            tok_dst[n * K + nfill[n]] = (int32_t)row;
            nfill[n] += 1;
            if (row < cap) {
                recv_src_tok[row] = (int32_t)n;
                for (int k = 0; k < K; ++k) {
                    int64_t e = topk[n * K + k];
                    int local = (e >= 0 && e < E && e / L == j);
                    recv_topk_idx[row * K + k] = local ? (e - (int64_t)j * L) : -1;
                    recv_topk_weights[row * K + k] = local ? w[n * K + k] : 0.0f;
                }
            }
            row += 1;
        }
    }
    rank_tok_base[R] = row;
    free(nfill);
    return row;
}

/* Stand-in expert stage for per-rank rows: each rank applies its local
 * experts to the received row and sums them with the received weights,
 * y = bf16( sum_k recv_topk_weights[k] * 2^-(l_k mod mark_mod) * v ), k in
 * order, each step acc = acc + (w * mark) * v, where v is the dequantised row
 * (as oracle_expert_rows, no mark) and l_k the local expert id (mark_mod = 0:
 * mark 1). */
void oracle_expert_token_rows(int64_t nrows, const int64_t* rows, int H, int K, int q,
                              const uint8_t* data, const uint8_t* scales,
                              const int64_t* recv_topk_idx, const float* recv_topk_weights,
                              int mark_mod, uint16_t* y) {
    int32_t zero_expert = -1;
    uint16_t* v = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
    int64_t db = oracle_row_data_bytes(q, H), sb = oracle_row_scale_bytes(q, H);
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        int64_t one = 0;
        oracle_expert_rows(1, &one, &zero_expert, H, q, data + i * db, sb ? scales + i * sb : NULL, 0, v);
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t l = recv_topk_idx[r * K + k];
                if (l < 0) continue;
                float mark = mark_mod > 0 ? ldexpf(1.0f, -(int)(l % mark_mod)) : 1.0f;
                float coef = recv_topk_weights[r * K + k] * mark;
                acc = acc + coef * oracle_bf16_to_f32(v[h]);
            }
            y[i * H + h] = oracle_bf16_from_f32(acc);
        }
    }
    free(v);
}

/* Reduced weights of the per-rank combine (DeepEP combine returns the
 * reduced topk weights): out_w[n][k] = sum over the token's rows i of
 * rank_w[tok_dst[n][i]][k], rows in ascending rank order. */
void oracle_reduce_token_weights(int64_t N, int K, const int32_t* tok_dst, const float* rank_w,
                                 float* out_w) {
    for (int64_t n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            float acc = 0.0f;
            for (int i = 0; i < K; ++i) {
                int32_t r = tok_dst[n * K + i];
                if (r < 0) continue;
                acc = acc + rank_w[(int64_t)r * K + k];
            }
            out_w[n * K + k] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Dispatch: every valid entry (s,t,k) receives the encoded row of token     */
/* (s,t) at dst_row[s,t,k]; padding rows are all-zero bytes.                */
/* Only rows in [row_begin, row_end) are produced, into buffers whose first */
/* row is row_begin, so a large receive buffer can be built rank by rank.   */
/* ------------------------------------------------------------------------ */
void oracle_dispatch(int N, int K, int H, int q, const int32_t* dst_row,
                     const uint16_t* x, int64_t row_begin, int64_t row_end,
                     uint8_t* recv_data, uint8_t* recv_scales) {
    int64_t db = oracle_row_data_bytes(q, H), sb = oracle_row_scale_bytes(q, H);
    memset(recv_data, 0, (size_t)((row_end - row_begin) * db));
    if (sb) memset(recv_scales, 0, (size_t)((row_end - row_begin) * sb));
    uint8_t* tmp_d = (uint8_t*)malloc((size_t)db);
    uint8_t* tmp_s = (uint8_t*)malloc((size_t)(sb ? sb : 1));
    for (int64_t n = 0; n < N; ++n) {
        int encoded = 0;
        for (int k = 0; k < K; ++k) {
            int64_t d = dst_row[n * K + k];
            if (d < row_begin || d >= row_end) continue;
            if (!encoded) { oracle_encode_row(q, H, x + n * H, tmp_d, tmp_s); encoded = 1; }
            memcpy(recv_data + (d - row_begin) * db, tmp_d, (size_t)db);
            if (sb) memcpy(recv_scales + (d - row_begin) * sb, tmp_s, (size_t)sb);
        }
    }
    free(tmp_d);
    free(tmp_s);
}

/* Dispatch of rows that are already encoded (DeepEP "Normal Mode API",
 * Quantization: x passed as a (data, scale) tuple): each source row is a fixed
 * number of bytes and moves unchanged.  Every valid entry (n, k) receives
 * src row n at dst_row[n*K+k]; rows no entry reaches (padding) are zero.  Called
 * once for the data rows and once for the scale rows. */
void oracle_dispatch_bytes(int N, int K, const int32_t* dst_row, const uint8_t* src, int64_t row_bytes,
                           int64_t row_begin, int64_t row_end, uint8_t* out) {
    memset(out, 0, (size_t)((row_end - row_begin) * row_bytes));
    for (int64_t n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            int64_t d = dst_row[n * K + k];
            if (d < row_begin || d >= row_end) continue;
            memcpy(out + (d - row_begin) * row_bytes, src + n * row_bytes, (size_t)row_bytes);
        }
}

/* Dispatch with input scales (quantModes 1-3): as oracle_dispatch, but each
 * entry's row is encoded with the scale row that applies to it: the scalar
 * scale[0] for every element (S_SCALAR), the shared row scale[0..H)
 * (S_CHANNEL), or the row of the entry's expert scale[e*H .. e*H+H) (S_EXPERT,
 * e = topk[s,t,k]).  S_NONE is oracle_dispatch. */
void oracle_dispatch_scaled(int N, int K, int H, int q, const int32_t* dst_row, const int64_t* topk,
                            const uint16_t* x, const float* scales, int kind,
                            int64_t row_begin, int64_t row_end,
                            uint8_t* recv_data, uint8_t* recv_scales) {
    int64_t db = oracle_row_data_bytes(q, H), sb = oracle_row_scale_bytes(q, H);
    memset(recv_data, 0, (size_t)((row_end - row_begin) * db));
    if (sb) memset(recv_scales, 0, (size_t)((row_end - row_begin) * sb));
    float* row = (float*)malloc(sizeof(float) * (size_t)H);
    for (int64_t n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            int64_t d = dst_row[n * K + k];
            if (d < row_begin || d >= row_end) continue;
            const float* sm = NULL;
            if (kind == S_SCALAR) {
                for (int h = 0; h < H; ++h) row[h] = scales[0];
                sm = row;
            } else if (kind == S_CHANNEL) {
                sm = scales;
            } else if (kind == S_EXPERT) {
                sm = scales + topk[n * K + k] * (int64_t)H;
            }
            uint8_t* dd = recv_data + (d - row_begin) * db;
            uint8_t* ds = sb ? recv_scales + (d - row_begin) * sb : NULL;
            if (q == Q_INT8_STATIC || q == Q_INT8 || q >= Q_FP8T_E4M3) oracle_encode_row_scaled(q, H, x + n * H, sm, dd, ds);
            else oracle_encode_row(q, H, x + n * H, dd, ds);
        }
    }
    free(row);
}

/* The same receive rows, produced one by one for a list of row indices via
 * recv_src (the inverse of dst_row): used to check sampled rows of a receive
 * buffer too large to build on the host. */
void oracle_dispatch_rows(int64_t nrows, const int64_t* rows, const int32_t* recv_src,
                          int H, int q, const uint16_t* x,
                          uint8_t* out_data, uint8_t* out_scales) {
    int64_t db = oracle_row_data_bytes(q, H), sb = oracle_row_scale_bytes(q, H);
    for (int64_t i = 0; i < nrows; ++i) {
        int32_t src = recv_src[rows[i]];
        uint8_t* d = out_data + i * db;
        uint8_t* s = sb ? out_scales + i * sb : NULL;
        if (src < 0) {
            memset(d, 0, (size_t)db);
            if (s) memset(s, 0, (size_t)sb);
        } else {
            oracle_encode_row(q, H, x + (int64_t)src * H, d, s);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Stand-in expert used by the tests: the dequantised receive row, rounded  */
/* to bf16, times an exact power-of-two mark 2^-(e mod mark_mod) that       */
/* depends on the row's expert e (mark_mod = 0: no mark).                    */
/*   int8:  fl(q * inv);   MX: fl(code value * 2^sharedExp)                 */
/* ------------------------------------------------------------------------ */
void oracle_expert_rows(int64_t nrows, const int64_t* rows, const int32_t* row_expert,
                        int H, int q, const uint8_t* data, const uint8_t* scales,
                        int mark_mod, uint16_t* y) {
    int64_t db = oracle_row_data_bytes(q, H), sb = oracle_row_scale_bytes(q, H);
    for (int64_t i = 0; i < nrows; ++i) {
        const uint8_t* d = data + i * db;
        const uint8_t* s = sb ? scales + i * sb : NULL;
        int e = row_expert[rows[i]];
        float mark = (mark_mod > 0 && e >= 0) ? ldexpf(1.0f, -(e % mark_mod)) : 1.0f;
        for (int h = 0; h < H; ++h) {
            float v;
            if (q == Q_NONE) {
                uint16_t b; memcpy(&b, d + 2 * h, 2);
                v = oracle_bf16_to_f32(b);
            } else if (q == Q_INT8) {
                float inv; memcpy(&inv, s, 4);
                v = (float)(int8_t)d[h] * inv;
            } else if (q == Q_FP8T_E4M3 || q == Q_FP8T_E5M2 || q == Q_FP8G_E4M3 || q == Q_FP8G_E5M2) {
                int fp8 = (q == Q_FP8T_E4M3 || q == Q_FP8G_E4M3) ? Q_E4M3 : Q_E5M2;
                float inv;
                memcpy(&inv, s + ((q == Q_FP8G_E4M3 || q == Q_FP8G_E5M2) ? 4 * (h / GROUP) : 0), 4);
                v = (float)oracle_mini_decode(fp8, d[h]) * inv;
            } else if (q == Q_INT8_STATIC) {
                v = (float)(int8_t)d[h];
            } else {
                int code = (q == Q_E2M1) ? ((d[h / 2] >> (4 * (h & 1))) & 0xf) : d[h];
                float dyn = ldexpf(1.0f, (int)s[h / 32] - 127);
                v = (float)oracle_mini_decode(q, code) * dyn;
            }
            v = v * mark;
            y[i * H + h] = oracle_bf16_from_f32(v);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Combine (DeepEP combine: multiply by weights and sum; MAX ep_combine: the */
/* weighted sum of routed outputs, plus the fused shared-expert outputs):    */
/*   out[s,t,:] = bf16( sum_k w[s,t,k] * y[dst_row[s,t,k],:]                 */
/*                      + sum_q shared[s,q,t,:] )                            */
/* in binary32, k in order then q in order, each step acc = acc + w*y as a   */
/* separate multiply and add.  Entries with dst_row = -1 are skipped.        */
/* Tokens [tok_begin, tok_end) only; out holds those tokens' rows.           */
/* The y rows are read through row_of(): y_rows maps a receive row to its    */
/* row in the y buffer (NULL: identity).                                     */
/* ------------------------------------------------------------------------ */
void oracle_combine(int R, int T, int H, int K, int S, const int32_t* dst_row,
                    const float* w, const uint16_t* y, const int64_t* y_rows,
                    const uint16_t* shared, int64_t tok_begin, int64_t tok_end,
                    uint16_t* out) {
    (void)R;
    for (int64_t n = tok_begin; n < tok_end; ++n) {
        int64_t s = n / T, t = n % T;
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t d = dst_row[n * K + k];
                if (d < 0) continue;
                int64_t yr = y_rows ? y_rows[d] : d;
                float prod = w[n * K + k] * oracle_bf16_to_f32(y[yr * H + h]);
                acc = acc + prod;
            }
            for (int qq = 0; qq < S; ++qq)
                acc = acc + oracle_bf16_to_f32(shared[((s * S + qq) * T + t) * H + h]);
            out[(n - tok_begin) * H + h] = oracle_bf16_from_f32(acc);
        }
    }
}

/* The same sum in binary64, with the sum of the terms' magnitudes, for the
 * combine tolerance (|gpu - ref| <= 2 ulp_bf16(ref) + (2K+S+1) 2^-24 sum|terms|). */
void oracle_combine_ref64(int R, int T, int H, int K, int S, const int32_t* dst_row,
                          const float* w, const uint16_t* y, const int64_t* y_rows,
                          const uint16_t* shared, int64_t tok_begin, int64_t tok_end,
                          double* ref, double* absum) {
    (void)R;
    for (int64_t n = tok_begin; n < tok_end; ++n) {
        int64_t s = n / T, t = n % T;
        for (int h = 0; h < H; ++h) {
            double acc = 0.0, mag = 0.0;
            for (int k = 0; k < K; ++k) {
                int64_t d = dst_row[n * K + k];
                if (d < 0) continue;
                int64_t yr = y_rows ? y_rows[d] : d;
                double term = (double)w[n * K + k] * (double)oracle_bf16_to_f32(y[yr * H + h]);
                acc += term;
                mag += fabs(term);
            }
            for (int qq = 0; qq < S; ++qq) {
                double term = (double)oracle_bf16_to_f32(shared[((s * S + qq) * T + t) * H + h]);
                acc += term;
                mag += fabs(term);
            }
            ref[(n - tok_begin) * H + h] = acc;
            absum[(n - tok_begin) * H + h] = mag;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Combine fused with a residual add and RMSNorm: CANN's                    */
/* aclnnMoeDistributeCombineAddRmsNorm, which the aclnnMoeDistributeDispatchV2 */
/* page names as a combine to pair with the dispatch; its formula is not     */
/* printed there.  Reading taken (the standard AddRmsNorm applied to the     */
/* combine's output):                                                        */
/*   x    = combine(row) + residual                                          */
/*   rstd = 1 / sqrt(mean over the H elements of x^2 + eps)                  */
/*   y    = x * rstd * gamma                                                 */
/* In binary64 from binary64 combine values c[N][H] (the exact weighted sums */
/* of oracle_combine_ref64), bf16 residual[N][H] and gamma[H].               */
/* ------------------------------------------------------------------------ */
void oracle_add_rms_norm_ref64(int64_t N, int H, const double* c, const uint16_t* residual,
                               const uint16_t* gamma, double eps, double* x, double* rstd, double* y) {
    for (int64_t n = 0; n < N; ++n) {
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            double v = c[n * H + h] + (double)oracle_bf16_to_f32(residual[n * H + h]);
            x[n * H + h] = v;
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / (double)H + eps);
        rstd[n] = r;
        for (int h = 0; h < H; ++h)
            y[n * H + h] = x[n * H + h] * r * (double)oracle_bf16_to_f32(gamma[h]);
    }
}

/* The same AddRmsNorm step by step in binary32, from the combine's output
 * rounded to bf16 (the reading of CANN aclnnMoeDistributeCombineAddRmsNorm
 * taken for the fused combine, which first rounds the weighted sum to the
 * combine's bf16 output):
 *   x    = fl32(c + residual)                  c, residual: bf16 values
 *   ss   = sum over h of fl32(x_h * x_h), added left to right in binary32
 *   rstd = fl32(1 / fl32(sqrt(fl32(fl32(ss / H) + eps))))
 *   y    = bf16(fl32(fl32(x * rstd) * gamma))
 * Outputs bf16(x), rstd and y.  sqrtf is IEEE's correctly rounded square
 * root.  Any summation order is an equally valid reading of "mean"; this one
 * is the plainest. */
void oracle_add_rms_norm_f32(int64_t N, int H, const uint16_t* c, const uint16_t* residual,
                             const uint16_t* gamma, float eps, uint16_t* x_out, float* rstd, uint16_t* y) {
    float* x = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
    for (int64_t n = 0; n < N; ++n) {
        float ss = 0.0f;
        for (int h = 0; h < H; ++h) {
            float v = oracle_bf16_to_f32(c[n * H + h]) + oracle_bf16_to_f32(residual[n * H + h]);
            x[h] = v;
            x_out[n * H + h] = oracle_bf16_from_f32(v);
            float sq = v * v;
            ss = ss + sq;
        }
        float mean = ss / (float)H;
        float r = 1.0f / sqrtf(mean + eps);
        rstd[n] = r;
        for (int h = 0; h < H; ++h) {
            float t = x[h] * r;
            y[n * H + h] = oracle_bf16_from_f32(t * oracle_bf16_to_f32(gamma[h]));
        }
    }
    free(x);
}
