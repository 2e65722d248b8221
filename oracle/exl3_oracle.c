/*
 * exl3_oracle.c -- plain, slow, single-threaded CPU oracle for the EXL3
 * trellis-quantized routed-expert MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table
 * or constant with the CUDA library under trellis_quantized_moe_exl3_gb300/.
 *
 * Every function follows the written format and layer definition (format v1,
 * "gb300_v1" tile order) that the design document derives from these pages:
 *   - "GLM-5.3-Flash EXL3 (~2.1 bpw, SM70 tile order)", intro: an EXL3 tensor
 *     is packed int16 trellis words that each hold 16/K weights.
 *   - "GLM-5.3-Flash · exlr8 (K2/K3/K4)", intro: every codebook output is
 *     rounded to FP8 E4M3 (nearest-even, saturating) before the side vectors;
 *     section Loading: a 16x16 tile (k16 index), a half of 4096x128 at width
 *     K is 65,536*K bytes; section Calibration: the mcg codebook, the 128x128
 *     Hadamard matrix and the tile packing order are format primitives (the
 *     Hadamard rotation is the optional format v2 here).
 *   - "GLM-5.3 Flash EXL3 for 2x DGX Sparks", section What runs: experts are
 *     trellis + suh + svh + mcg; section Cold prefill (E3): gather, gate/up +
 *     SwiGLU, down + scatter from device-side segment tables.
 * Where the pages are silent the plainest reading is taken; each such reading
 * is marked "reading:" below.
 *
 * Arithmetic: fp64 with no intermediate rounding, except where the format
 * itself fixes a rounding (fp16 codebook value, E4M3 rule, the fp32 routing
 * softmax, the bf16 storage of activations).
 *
 * Parity status: every function here is pinned by tests/test_oracle_pins.py
 * (closed forms, exhaustive states, library converters, brute force, dense
 * reference; the Hadamard matrix against scipy's Sylvester construction and a
 * closed-form rotated layer; the E4M3 activation operand against torch's
 * float8_e4m3fn conversion).  Compatibility with real EXL3/exlr8 checkpoints is unpinned: no
 * checkpoint or test vector is available to check them against.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (contraction off so
 * that the fp32 routing arithmetic is the written sequence of roundings).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                            */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 bits -> exact double. */
double oracle_f16_to_double(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return s ? -v : v;
}

/* bfloat16 bits -> exact double. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* double -> binary16, one round-to-nearest-even step (overflow to inf). */
uint16_t oracle_double_to_f16(double v)
{
    if (isnan(v))
        return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a >= 65520.0) /* half-way above 65504 and beyond round to inf */
        return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range, quantum 2^-24; 1024 quanta is the least normal */
        double q = nearbyint(a * 16777216.0);
        return sign | (uint16_t)q;
    }
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e) */
    double ulp = ldexp(1.0, e - 1 - 10);
    double q = nearbyint(a / ulp); /* in [1024, 2048] */
    int E = e - 1 + 15;
    int M = (int)q - 1024;
    if (M == 1024) {
        E += 1;
        M = 0;
    }
    if (E >= 31)
        return sign | 0x7C00;
    return (uint16_t)(sign | (E << 10) | M);
}

/* double -> bfloat16, one round-to-nearest-even step (overflow to inf). */
uint16_t oracle_double_to_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    double maxv = ldexp(255.0, 120);             /* largest bf16, (2-2^-7)*2^127 */
    if (a >= maxv + ldexp(1.0, 119))             /* half an ulp above it */
        return sign | 0x7F80;
    if (a < ldexp(1.0, -126)) {
        double q = nearbyint(a / ldexp(1.0, -133)); /* subnormal quantum 2^-133 */
        return sign | (uint16_t)q;
    }
    int e;
    frexp(a, &e);
    double ulp = ldexp(1.0, e - 1 - 7);
    double q = nearbyint(a / ulp); /* in [128, 256] */
    int E = e - 1 + 127;
    int M = (int)q - 128;
    if (M == 128) {
        E += 1;
        M = 0;
    }
    if (E >= 255)
        return sign | 0x7F80;
    return (uint16_t)(sign | (E << 7) | M);
}

/* FP8 E4M3 ("fn": no inf, max 448) round-to-nearest-even with saturation to
 * +-448, applied to an exact value.  Page "GLM-5.3-Flash · exlr8", intro. */
double oracle_e4m3_rne_sat(double v)
{
    if (isnan(v))
        return NAN;
    double a = fabs(v), r;
    if (a >= 448.0) {
        r = 448.0;
    } else if (a < ldexp(1.0, -6)) {
        r = nearbyint(a * 512.0) / 512.0; /* subnormal quantum 2^-9 */
    } else {
        int e;
        frexp(a, &e);
        double ulp = ldexp(1.0, e - 1 - 3); /* 3 mantissa bits */
        r = nearbyint(a / ulp) * ulp;
        if (r > 448.0)
            r = 448.0;
    }
    return copysign(r, v);
}

/* ------------------------------------------------------------------------ */
/* Trellis format v1                                                         */
/* ------------------------------------------------------------------------ */

/* Bit p of a tile's bitstream.  reading: the 16*K little-endian uint16 words
 * of a tile form one bit string, least significant bit of word 0 first, and
 * the string is circular (tail-biting) so that a K-bit code costs exactly K
 * bits per weight, as the exlr8 "Widths" section requires. */
static int tile_bit(const uint16_t *words, int K, long p)
{
    long n = 256L * K;
    p %= n;
    return (words[p >> 4] >> (p & 15)) & 1;
}

/* 16-bit trellis state of weight t: the window of 16 bits starting at bit
 * t*K.  reading: bitshift trellis with a 16-bit state, each step shifting in
 * K new bits ("16/K weights per int16 word", page 1 intro). */
uint32_t oracle_tile_state(const uint16_t *words, int K, int t)
{
    uint32_t s = 0;
    for (int b = 0; b < 16; b++)
        s |= (uint32_t)tile_bit(words, K, (long)t * K + b) << b;
    return s;
}

/* "mcg" codebook: state -> fp16 bits.  reading (published computed-code
 * construction of QTIP, with a pure multiplicative generator): x = s * mult
 * mod 2^32; keep sign and low 12 bits of each 16-bit half and fix the upper
 * exponent bits (mask 0x8FFF8FFF, xor 0x3B603B60); the halves are two fp16
 * numbers a (low) and b (high); the weight is fp16(a + b). */
uint16_t oracle_codebook_f16(uint32_t s, uint32_t mult)
{
    uint32_t x = s * mult;
    uint32_t m = (x & 0x8FFF8FFFu) ^ 0x3B603B60u;
    double a = oracle_f16_to_double((uint16_t)(m & 0xFFFFu));
    double b = oracle_f16_to_double((uint16_t)(m >> 16));
    return oracle_double_to_f16(a + b); /* a + b is exact in double */
}

/* Codebook value with the optional exlr8 E4M3 rule applied (fp16 bits; every
 * E4M3 value is exact in fp16). */
uint16_t oracle_weight_f16(uint32_t s, uint32_t mult, int fp8_round)
{
    uint16_t v = oracle_codebook_f16(s, mult);
    if (fp8_round)
        v = oracle_double_to_f16(oracle_e4m3_rne_sat(oracle_f16_to_double(v)));
    return v;
}

/* Tile order "gb300_v1": position of weight t inside its 16x16 tile.
 * reading: the pages name tile orders (sm70_colmajor, sm80, strip-major) but
 * define none, so the library fixes its own.  t = 64*c + 8*r0 + 4*hf + j with
 * c, j in 0..3, r0 in 0..7, hf in 0..1:
 *   output row  = r0 + 8*(j & 1)
 *   input col   = c + 4*(j >> 1) + 8*hf                                       */
void oracle_tile_position(int t, int *out_row, int *in_col)
{
    int c = t >> 6, u = t & 63;
    int r0 = u >> 3, hf = (u >> 2) & 1, j = u & 3;
    *out_row = r0 + 8 * (j & 1);
    *in_col = c + 4 * (j >> 1) + 8 * hf;
}

/* Decode one 16x16 tile to fp16 bits in [input 16][output 16] order. */
void oracle_decode_tile(const uint16_t *words, int K, uint32_t mult, int fp8_round,
                        uint16_t *out /* [16][16], in-major */)
{
    for (int t = 0; t < 256; t++) {
        int r, q;
        oracle_tile_position(t, &r, &q);
        out[q * 16 + r] = oracle_weight_f16(oracle_tile_state(words, K, t), mult, fp8_round);
    }
}

/* Dense decode of one projection of one expert.
 * codes: [in/16][out/16][16*K] uint16; suh: [in] fp16; svh: [out] fp16.
 * out: [in][out] fp16 bits.  apply_side = 0 gives the codebook values; 1
 * gives fp16(fp32(fp32(v*suh[i]) * svh[o])), one correctly rounded step each.
 * reading (side vectors, page "What runs"): W[i][o] = suh[i] * v[i][o] *
 * svh[o], suh over inputs and svh over outputs, applied after the E4M3 rule. */
void oracle_decode_dense(const uint16_t *codes, int in, int out, int K, uint32_t mult,
                         int fp8_round, const uint16_t *suh, const uint16_t *svh,
                         int apply_side, uint16_t *dst)
{
    int nti = in / 16, nto = out / 16;
    uint16_t tile[256];
    for (int i = 0; i < nti; i++)
        for (int j = 0; j < nto; j++) {
            const uint16_t *w = codes + ((size_t)i * nto + j) * 16 * K;
            oracle_decode_tile(w, K, mult, fp8_round, tile);
            for (int q = 0; q < 16; q++)
                for (int r = 0; r < 16; r++) {
                    int ii = 16 * i + q, oo = 16 * j + r;
                    uint16_t v = tile[q * 16 + r];
                    if (apply_side) {
                        float p1 = (float)(oracle_f16_to_double(v) * oracle_f16_to_double(suh[ii]));
                        float p2 = p1 * (float)oracle_f16_to_double(svh[oo]);
                        v = oracle_double_to_f16((double)p2);
                    }
                    dst[(size_t)ii * out + oo] = v;
                }
        }
}

/* ------------------------------------------------------------------------ */
/* Routing                                                                   */
/* ------------------------------------------------------------------------ */

/* exp for the routing softmax, fixed so that CPU and GPU agree bit for bit.
 * Cody-Waite reduction x = n*ln2 + r with the two-part ln2 of the Cephes
 * library (0.693359375 and -2.12194440e-4), a degree-7 Taylor polynomial in
 * Horner form with fused multiply-adds, and an exact scaling by 2^n.  Inputs
 * below -86 (including -inf) give 0, so 2^n * p never leaves the normal
 * range.  reading: the pages do not give the router; this is the build's
 * definition of "softmax over the k selected". */
float oracle_exp_route(float x)
{
    if (!(x >= -86.0f))
        return 0.0f;
    float t = x * 1.44269504088896341f;
    float n = rintf(t);
    float r = fmaf(-n, 0.693359375f, x);
    r = fmaf(-n, -2.12194440e-4f, r);
    float p = (float)(1.0 / 5040.0);
    p = fmaf(p, r, (float)(1.0 / 720.0));
    p = fmaf(p, r, (float)(1.0 / 120.0));
    p = fmaf(p, r, (float)(1.0 / 24.0));
    p = fmaf(p, r, (float)(1.0 / 6.0));
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return ldexpf(p, (int)n);
}

/* Top-k of one token's logits and the softmax over the k selected.
 * Order: larger logit first, ties to the lower expert index, NaN counts as
 * -inf.  Weights: e_j = exp(l_j - l_max) (0 difference when l_j == l_max,
 * which also covers -inf == -inf), summed in j order in fp32, w_j = e_j / sum.
 * Page "GLM-5.3-Flash · exlr8", intro: 288 routed experts, top-8. */
void oracle_route_token(const float *logits, int E, int k, int32_t *ids, float *w)
{
    char *taken = (char *)calloc((size_t)E, 1);
    float lsel[64];
    for (int j = 0; j < k; j++) {
        int best = -1;
        float bv = 0.0f;
        for (int e = 0; e < E; e++) {
            if (taken[e])
                continue;
            float v = isnan(logits[e]) ? -INFINITY : logits[e];
            if (best < 0 || v > bv) {
                best = e;
                bv = v;
            }
        }
        taken[best] = 1;
        ids[j] = best;
        lsel[j] = bv;
    }
    free(taken);
    float lmax = lsel[0];
    float ex[64], sum = 0.0f;
    for (int j = 0; j < k; j++) {
        float d = (lsel[j] == lmax) ? 0.0f : lsel[j] - lmax;
        ex[j] = oracle_exp_route(d);
        sum = sum + ex[j];
    }
    for (int j = 0; j < k; j++)
        w[j] = ex[j] / sum;
}

/* Route all T tokens and build the segment tables.
 * seg_offsets[e] = number of pairs whose expert is < e (E+1 entries);
 * seg_pairs lists pair ids p = t*k + j grouped by expert, ascending p inside
 * each group.  Page "GLM-5.3 Flash EXL3 for 2x DGX Sparks", section Cold
 * prefill (E3): launches built from device-side segment tables. */
void oracle_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                  int32_t *seg_offsets, int32_t *seg_pairs)
{
    for (int t = 0; t < T; t++)
        oracle_route_token(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k);
    int32_t *cursor = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    for (long p = 0; p < (long)T * k; p++)
        cursor[ids[p] + 1]++;
    for (int e = 0; e < E; e++)
        cursor[e + 1] += cursor[e];
    memcpy(seg_offsets, cursor, ((size_t)E + 1) * sizeof(int32_t));
    for (long p = 0; p < (long)T * k; p++)
        seg_pairs[cursor[ids[p]]++] = (int32_t)p;
    free(cursor);
}

/* ------------------------------------------------------------------------ */
/* MoE layer                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    int num_experts, hidden, inter;
    int K[3];          /* gate, up, down */
    int fp8_round;
    uint32_t mult;
    const uint16_t *codes[3]; /* [E][in/16][out/16][16K] */
    const uint16_t *suh[3];   /* [E][in] fp16 */
    const uint16_t *svh[3];   /* [E][out] fp16 */
    const uint16_t *shared_w[3]; /* dense fp16 [in][out] or NULL */
    int hadamard;      /* 1: format v2, the 128-point rotation on both sides */
    int shared_coded;  /* 1: expert num_experts of the code arrays is a trellis-coded shared
                          expert that every token uses with weight 1 */
    const uint8_t *expert_K; /* NULL, or [experts][3] widths per expert and projection: the
                                codes of projection p are then the experts' arrays back to
                                back, each at its own width */
    int act_fp8;       /* 1: every projection's input row is quantised to E4M3 with a
                          per-row scale (the FP8 x FP8 product's activation operand) */
} oracle_layer;

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------------------ */
/* Hadamard rotation (format v2)                                             */
/* ------------------------------------------------------------------------ */

/* Entry (i, j), 0 <= i, j < 128, of the normalized 128x128 Hadamard matrix
 * of Sylvester's construction: (-1)^popcount(i & j) / sqrt(128).
 * reading: page "GLM-5.3-Flash · exlr8 (K2/K3/K4)", section Calibration,
 * names "the 128x128 Hadamard matrix" as one of the format's primitives
 * without printing it; the Sylvester matrix (the 2x2 [[1, 1], [1, -1]]
 * raised to the 7th Kronecker power) is the plain 128x128 one, and its
 * normalization makes it orthogonal and its own inverse. */
double oracle_hadamard128_entry(int i, int j)
{
    int bits = i & j, par = 0;
    while (bits) {
        par ^= bits & 1;
        bits >>= 1;
    }
    return (par ? -1.0 : 1.0) / sqrt(128.0);
}

/* Per-row E4M3 quantisation of an activation row for an FP8 x FP8 product.
 * Page "GLM-5.3-Flash · exlr8 (K2/K3/K4)", Widths: with the E4M3 codebook the
 * prefill runs on FP8 tensor cores; the pages give no activation recipe.
 * reading: the row is taken in fp32 (the precision in which a kernel makes
 * these integer decisions), s = fp32(amax / 448) with amax the row's largest
 * magnitude, q_i = E4M3_RNE_sat(fp32(a_i / s)), and the row becomes q_i * s
 * (exact in double).  An all-zero row stays zero.  out may alias a. */
void oracle_quantize_row_e4m3(const double *a, int n, double *out)
{
    float amax = 0.0f;
    for (int i = 0; i < n; i++) {
        float ai = (float)a[i];
        if (fabsf(ai) > amax)
            amax = fabsf(ai);
    }
    if (amax == 0.0f) {
        for (int i = 0; i < n; i++)
            out[i] = 0.0;
        return;
    }
    float s = amax / 448.0f;
    for (int i = 0; i < n; i++) {
        float q = (float)a[i] / s;
        out[i] = oracle_e4m3_rne_sat((double)q) * (double)s;
    }
}

/* v <- v . Hb for a row vector of n values (n a multiple of 128), where Hb is
 * block diagonal with n/128 copies of the 128x128 matrix above.  Plain
 * matrix-vector products from the entries (no fast transform). */
void oracle_hadamard_blocks(double *v, int n)
{
    double tmp[128];
    double *Hm = (double *)malloc(128 * 128 * sizeof(double));
    for (int i = 0; i < 128; i++)
        for (int j = 0; j < 128; j++)
            Hm[i * 128 + j] = oracle_hadamard128_entry(i, j);
    for (int b = 0; b < n; b += 128) {
        for (int j = 0; j < 128; j++) {
            double acc = 0.0;
            for (int i = 0; i < 128; i++)
                acc += v[b + i] * Hm[i * 128 + j];
            tmp[j] = acc;
        }
        for (int j = 0; j < 128; j++)
            v[b + j] = tmp[j];
    }
    free(Hm);
}

/* Decode projection p of expert e to doubles [in][out] (codebook values,
 * side vectors not applied). */
/* Width of projection p of expert e, and the word offset of its codes.
 * reading: pages "GLM-5.3-Flash · exlr8 (K2/K3/K4)", Loading (manifests that
 * give some experts or projections another width) and
 * "GLM-5.3-Flash-EXL3-TR3-3.5bpw" (every routed tensor K3 or K4) mix widths
 * inside a layer without giving a file layout; the plainest one stores each
 * projection's experts back to back, expert e after experts 0 .. e-1, each
 * at its own width. */
static int proj_width(const oracle_layer *L, int p, int e)
{
    return L->expert_K ? L->expert_K[(size_t)e * 3 + p] : L->K[p];
}

static size_t proj_offset(const oracle_layer *L, int p, int e)
{
    int in = (p == 2) ? L->inter : L->hidden;
    int out = (p == 2) ? L->hidden : L->inter;
    size_t tile_words = (size_t)(in / 16) * (out / 16) * 16;
    size_t off = 0;
    for (int f = 0; f < e; f++)
        off += tile_words * proj_width(L, p, f);
    return off;
}

static void decode_proj_double(const oracle_layer *L, int p, int e, double *dst)
{
    int in = (p == 2) ? L->inter : L->hidden;
    int out = (p == 2) ? L->hidden : L->inter;
    int K = proj_width(L, p, e);
    uint16_t *tmp = (uint16_t *)malloc((size_t)in * out * sizeof(uint16_t));
    oracle_decode_dense(L->codes[p] + proj_offset(L, p, e), in, out, K, L->mult, L->fp8_round,
                        NULL, NULL, 0, tmp);
    for (size_t i = 0; i < (size_t)in * out; i++)
        dst[i] = oracle_f16_to_double(tmp[i]);
    free(tmp);
}

/* One routed expert applied to one activation row (fp64), times router weight.
 * g = svh_g * ((x * suh_g) . Vg), u likewise, h = silu(g) * u,
 * r = w * svh_d * ((h * suh_d) . Vd).  Page "GLM-5.3 Flash EXL3 for 2x DGX
 * Sparks", section Cold prefill (E3): gate/up + SwiGLU, then down + scatter.
 * With the Hadamard rotation (format v2) every projection becomes
 * svh * ((((in * suh) . Hb) . V) . Hb), i.e. the effective weight matrix is
 * diag(suh) Hb V Hb diag(svh).
 * reading: the pages name the matrix but not where it acts; the input is
 * scaled by suh and then rotated, the product rotated and then scaled by svh,
 * so that with Hb = identity this is format v1. */
static void project(const oracle_layer *L, const double *in, int n_in, const uint16_t *suh,
                    const double *V, int n_out, double *out)
{
    double *a = (double *)malloc((size_t)n_in * sizeof(double));
    for (int i = 0; i < n_in; i++)
        a[i] = in[i] * oracle_f16_to_double(suh[i]);
    if (L->hadamard)
        oracle_hadamard_blocks(a, n_in);
    if (L->act_fp8)   /* the operand the tensor core multiplies: the rotated row */
        oracle_quantize_row_e4m3(a, n_in, a);
    for (int o = 0; o < n_out; o++)
        out[o] = 0.0;
    for (int i = 0; i < n_in; i++) {
        const double *vr = V + (size_t)i * n_out;
        for (int o = 0; o < n_out; o++)
            out[o] += a[i] * vr[o];
    }
    if (L->hadamard)
        oracle_hadamard_blocks(out, n_out);
    free(a);
}

static void expert_row(const oracle_layer *L, int e, const double *Vg, const double *Vu,
                       const double *Vd, const double *x, double wgt, double *r)
{
    int H = L->hidden, I = L->inter;
    const uint16_t *svh_g = L->svh[0] + (size_t)e * I, *svh_u = L->svh[1] + (size_t)e * I;
    const uint16_t *svh_d = L->svh[2] + (size_t)e * H;
    double *g = (double *)malloc((size_t)I * sizeof(double));
    double *u = (double *)malloc((size_t)I * sizeof(double));
    double *h = (double *)malloc((size_t)I * sizeof(double));
    project(L, x, H, L->suh[0] + (size_t)e * H, Vg, I, g);
    project(L, x, H, L->suh[1] + (size_t)e * H, Vu, I, u);
    for (int o = 0; o < I; o++) {
        double gg = g[o] * oracle_f16_to_double(svh_g[o]);
        double uu = u[o] * oracle_f16_to_double(svh_u[o]);
        h[o] = silu(gg) * uu;
    }
    project(L, h, I, L->suh[2] + (size_t)e * I, Vd, H, r);
    for (int o = 0; o < H; o++)
        r[o] *= wgt * oracle_f16_to_double(svh_d[o]);
    free(g);
    free(u);
    free(h);
}

/* Shared expert: unquantized fp16 SwiGLU MLP of the same shape, weight 1
 * (page "GLM-5.3-Flash · exlr8", intro: one shared expert per MoE layer;
 * page 1 Recipe: shared experts kept FP16). */
static void shared_row(const oracle_layer *L, const double *x, double *y)
{
    int H = L->hidden, I = L->inter;
    double *g = (double *)calloc((size_t)I, sizeof(double));
    double *u = (double *)calloc((size_t)I, sizeof(double));
    for (int i = 0; i < H; i++)
        for (int o = 0; o < I; o++) {
            g[o] += x[i] * oracle_f16_to_double(L->shared_w[0][(size_t)i * I + o]);
            u[o] += x[i] * oracle_f16_to_double(L->shared_w[1][(size_t)i * I + o]);
        }
    for (int o = 0; o < I; o++)
        g[o] = silu(g[o]) * u[o];
    for (int i = 0; i < I; i++)
        for (int o = 0; o < H; o++)
            y[o] += g[i] * oracle_f16_to_double(L->shared_w[2][(size_t)i * H + o]);
    free(g);
    free(u);
}

/* MoE layer forward for a subset of tokens (tokens are independent).
 * x: [T][H] bf16 or fp16 bits; logits: [T][E] fp32; tokens: n_sel token
 * indices; y: [n_sel][H] doubles, y_t = sum_{j=0..k-1} r_{t,j} (+ shared).
 * With shared_coded the shared term is the trellis-coded expert E applied
 * with weight 1 after the routed pairs (page "GLM-5.3-Flash · exlr8
 * (K2/K3/K4)", Loading: the shared expert is stored as expert 288, after the
 * routed ones, at the routed experts' width).
 * Each used expert is decoded once.  Returns 0 on success. */
int oracle_moe_forward(const oracle_layer *L, const uint16_t *x, int x_is_bf16,
                       const float *logits, int T, int k, const int32_t *tokens, int n_sel,
                       double *y)
{
    int E = L->num_experts, H = L->hidden, I = L->inter;
    (void)T;
    int32_t *ids = (int32_t *)malloc((size_t)n_sel * k * sizeof(int32_t));
    float *w = (float *)malloc((size_t)n_sel * k * sizeof(float));
    double *xr = (double *)malloc((size_t)n_sel * H * sizeof(double));
    double *r = (double *)calloc((size_t)n_sel * k * H, sizeof(double));
    if (!ids || !w || !xr || !r)
        return 1;
    for (int s = 0; s < n_sel; s++) {
        int t = tokens[s];
        oracle_route_token(logits + (size_t)t * E, E, k, ids + (size_t)s * k, w + (size_t)s * k);
        for (int i = 0; i < H; i++) {
            uint16_t b = x[(size_t)t * H + i];
            xr[(size_t)s * H + i] = x_is_bf16 ? oracle_bf16_to_double(b) : oracle_f16_to_double(b);
        }
    }
    double *Vg = (double *)malloc((size_t)H * I * sizeof(double));
    double *Vu = (double *)malloc((size_t)H * I * sizeof(double));
    double *Vd = (double *)malloc((size_t)I * H * sizeof(double));
    if (!Vg || !Vu || !Vd)
        return 1;
    for (int e = 0; e < E; e++) {
        int used = 0;
        for (long p = 0; p < (long)n_sel * k; p++)
            used |= (ids[p] == e);
        if (!used)
            continue;
        decode_proj_double(L, 0, e, Vg);
        decode_proj_double(L, 1, e, Vu);
        decode_proj_double(L, 2, e, Vd);
        for (long p = 0; p < (long)n_sel * k; p++)
            if (ids[p] == e)
                expert_row(L, e, Vg, Vu, Vd, xr + (size_t)(p / k) * H, (double)w[p],
                           r + (size_t)p * H);
    }
    double *rs = NULL;
    if (L->shared_coded) {
        rs = (double *)malloc((size_t)n_sel * H * sizeof(double));
        if (!rs)
            return 1;
        decode_proj_double(L, 0, E, Vg);
        decode_proj_double(L, 1, E, Vu);
        decode_proj_double(L, 2, E, Vd);
        for (int s = 0; s < n_sel; s++)
            expert_row(L, E, Vg, Vu, Vd, xr + (size_t)s * H, 1.0, rs + (size_t)s * H);
    }
    free(Vg);
    free(Vu);
    free(Vd);
    for (int s = 0; s < n_sel; s++) {
        double *ys = y + (size_t)s * H;
        for (int o = 0; o < H; o++)
            ys[o] = 0.0;
        for (int j = 0; j < k; j++)
            for (int o = 0; o < H; o++)
                ys[o] += r[((size_t)s * k + j) * H + o];
        if (rs)
            for (int o = 0; o < H; o++)
                ys[o] += rs[(size_t)s * H + o];
        if (L->shared_w[0])
            shared_row(L, xr + (size_t)s * H, ys);
    }
    free(rs);
    free(ids);
    free(w);
    free(xr);
    free(r);
    return 0;
}

/* One (token, expert) pair: decode the expert and compute w * expert(x) for
 * one activation row (fp64).  The unit of the CPU baseline's bounded sample. */
int oracle_expert_pair(const oracle_layer *L, const uint16_t *x_row, int x_is_bf16, int e,
                       float wgt, double *r)
{
    int H = L->hidden, I = L->inter;
    double *xr = (double *)malloc((size_t)H * sizeof(double));
    double *Vg = (double *)malloc((size_t)H * I * sizeof(double));
    double *Vu = (double *)malloc((size_t)H * I * sizeof(double));
    double *Vd = (double *)malloc((size_t)I * H * sizeof(double));
    if (!xr || !Vg || !Vu || !Vd)
        return 1;
    for (int i = 0; i < H; i++)
        xr[i] = x_is_bf16 ? oracle_bf16_to_double(x_row[i]) : oracle_f16_to_double(x_row[i]);
    decode_proj_double(L, 0, e, Vg);
    decode_proj_double(L, 1, e, Vu);
    decode_proj_double(L, 2, e, Vd);
    expert_row(L, e, Vg, Vu, Vd, xr, (double)wgt, r);
    free(xr);
    free(Vg);
    free(Vu);
    free(Vd);
    return 0;
}

/* Shared expert of one activation row (fp64), added into y. */
void oracle_shared_row(const oracle_layer *L, const uint16_t *x_row, int x_is_bf16, double *y)
{
    int H = L->hidden;
    double *xr = (double *)malloc((size_t)H * sizeof(double));
    for (int i = 0; i < H; i++)
        xr[i] = x_is_bf16 ? oracle_bf16_to_double(x_row[i]) : oracle_f16_to_double(x_row[i]);
    if (L->shared_w[0])
        shared_row(L, xr, y);
    free(xr);
}

/* Unweighted RMSNorm of one row (fp64), eps added to the mean square.
 * reading: the long-prefill workload chains layers with a residual add; the
 * pages give no norm, and without one the synthetic magnitudes overflow, so
 * each layer's input is the standard pre-norm rmsnorm(x) of the residual. */
void oracle_rmsnorm_row(const double *x, int H, double eps, double *out)
{
    double ss = 0.0;
    for (int i = 0; i < H; i++)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / H + eps);
    for (int i = 0; i < H; i++)
        out[i] = x[i] * inv;
}
