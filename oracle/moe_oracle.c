/*
 * moe_oracle.c -- plain, slow CPU oracle of one routed mixture-of-experts FFN
 * layer run over a fixed expert-slot pool.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; the two meet only through the seeded inputs.
 *
 * What the layer computes (the "plain definition"): the pool only changes
 * where the expert weights live, never the result, so the oracle evaluates
 * the dense MoE layer restricted to the routed experts:
 *
 *   - routing: top-k of the router logits, softmax over the k selected
 *     (tinyserve README, "Performance": GPT-OSS-20B with top_k=4);
 *   - grouping: per-expert histogram and a stable permutation, so each
 *     unique expert is loaded once (tinyserve README, "How it works",
 *     item 6, Batched prefill);
 *   - expert FFN: gate, up, SwiGLU, down on MXFP4 weights used in their
 *     native format (tinyserve README, "How it works", item 2: three
 *     products per expert, no intermediate BF16 weights);
 *   - combine: weighted merge of the expert outputs (llama.cpp discussion
 *     "fixed GPU expert working set with Native CPU miss execution", main
 *     post: hits and misses are merged with the routing weights);
 *   - pool: (layer, expert) -> slot map with LRU eviction, one fused event
 *     per (layer, step) (tinyserve README, "How it works", item 3 and
 *     "Configuration" cache_policy; "Expert Offloading" topic page, the
 *     replay-semantics study: fused-event contract).
 *
 * Number formats follow the OCP Microscaling Formats (MX) v1.0 specification:
 * E2M1 elements, E8M0 block-32 scales, E4M3 elements for MXFP8.  The GGUF
 * expert formats Q8_0 and Q4_K follow the published GGUF block layouts.
 *
 * Precision: the expert path is the one the method states -- bf16
 * activations times fp32-dequantised fp4, products and sums in fp32 taken in
 * ascending reduction index, SwiGLU in fp32, its output rounded to bf16.
 * The routing softmax, which the pages leave open, is taken in fp64 and
 * rounded to fp32.  Build with -ffp-contract=off so a*b+c is never fused.
 *
 * Where the pages are silent the readings are: ties in the top-k go to the
 * lower expert id; the k selected are kept in descending-logit order; the
 * permutation is stable in the assignment index a = t*k + j; MX blocks run
 * along the reduction dimension with the even element in the low nibble;
 * SwiGLU is silu(gate)*up with no clamp or bias; the routing weight is
 * applied after the down projection.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID (-1)
#define ORACLE_ERR_CAPACITY (-3)

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 (OCP MX v1.0, FP4): sign bit, 2 exponent bits with bias 1, 1 mantissa
 * bit; exponent field 0 is subnormal (value = mantissa * 0.5).               */
double oracle_e2m1_value(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int ef = (code >> 1) & 3;
    int m = code & 1;
    double mag = (ef == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, ef - 1);
    return sign ? -mag : mag;
}

/* E8M0 (OCP MX v1.0 shared scale): 2^(byte-127); byte 255 is NaN.          */
double oracle_e8m0_value(uint8_t b)
{
    if (b == 255) return NAN;
    return ldexp(1.0, (int)b - 127);
}

float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even (bf16 keeps the top 16 bits
 * of the fp32 pattern).                                                    */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (uint16_t)((u >> 16) | 0x40); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* E4M3 (OCP 8-bit FP, "fn" variant used by MXFP8): sign, 4 exponent bits
 * bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite
 * 448, smallest normal 2^-6, subnormals k*2^-9.  Encoding rounds to nearest
 * even and saturates finite overflow to +-448.                              */
double oracle_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int ef = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (ef == 15 && m == 7) return NAN;
    if (ef == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + m / 8.0, ef - 7);
    return sign ? -mag : mag;
}

uint8_t oracle_e4m3_encode(double v)
{
    if (isnan(v)) return 0x7f;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid 2^-9; n == 8 lands on the smallest normal, whose
         * bit pattern is exactly 8 as well                                  */
        double n = nearbyint(a / ldexp(1.0, -9));
        return sign | (uint8_t)n;
    }
    int ex;
    frexp(a, &ex);                 /* a = f * 2^ex, f in [0.5, 1)          */
    int e = ex - 1;                /* floor(log2 a)                        */
    double n = nearbyint(a / ldexp(1.0, e - 3)); /* in [8, 16]             */
    if (n == 16.0) { e += 1; n = 8.0; }
    /* a < 448 keeps (e, n) at or below (8, 14), never the NaN pattern      */
    return sign | (uint8_t)(((e + 7) << 3) | ((int)n - 8));
}

/* MXFP8 quantisation of one row of K bf16 values, K a multiple of 32
 * (OCP MX v1.0, section 6.3 conversion): per block of 32,
 *   shared exponent = floor(log2(amax)) - emax_elem, emax_elem = 8 for E4M3,
 *   scale byte = shared exponent + 127 clamped to [0, 254] (0 when amax = 0),
 *   element = E4M3_RNE_satfinite(x / 2^(byte-127)).                          */
void oracle_mxfp8_quant_row(const uint16_t* x_bf16, int K, uint8_t* codes, uint8_t* scales)
{
    for (int b = 0; b < K / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double v = fabs((double)oracle_bf16_to_f32(x_bf16[b * 32 + i]));
            if (v > amax) amax = v;
        }
        int sb;
        if (amax == 0.0) {
            sb = 0;
        } else {
            int ex;
            frexp(amax, &ex);
            sb = (ex - 1) - 8 + 127;
            if (sb < 0) sb = 0;
            if (sb > 254) sb = 254;
        }
        scales[b] = (uint8_t)sb;
        for (int i = 0; i < 32; ++i) {
            double v = (double)oracle_bf16_to_f32(x_bf16[b * 32 + i]);
            codes[b * 32 + i] = oracle_e4m3_encode(ldexp(v, 127 - sb));
        }
    }
}

/* E2M1 encoding (OCP MX v1.0, FP4 E2M1: bias 1, one mantissa bit, no
 * infinities or NaN, largest 6, subnormal 0.5): round to nearest, ties to
 * the even code, finite overflow saturated to +-6.  Sign kept for zero.    */
uint8_t oracle_e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    if (isnan(v)) return 0x7;
    double a = fabs(v);
    if (a >= 6.0) return sign | 0x7;
    if (a < 1.0) {
        /* subnormal grid 0.5; n == 2 lands on 1.0, whose code is 2 as well */
        double n = nearbyint(a / 0.5);
        return sign | (uint8_t)n;
    }
    int ex;
    frexp(a, &ex);                 /* a = f * 2^ex, f in [0.5, 1)          */
    int e = ex - 1;                /* floor(log2 a), 0..2                  */
    double n = nearbyint(a / ldexp(1.0, e - 1)); /* in [2, 4]              */
    if (n == 4.0) { e += 1; n = 2.0; }
    return sign | (uint8_t)(((e + 1) << 1) | ((int)n - 2));
}

/* MXFP4 quantisation of one row of K bf16 values, K a multiple of 32 (OCP
 * MX v1.0, section 6.3 conversion with emax_elem = 2 for E2M1): per block
 * of 32, scale byte = floor(log2(amax)) - 2 + 127 clamped to [0, 254] (0
 * when amax = 0), element = E2M1_RNE_satfinite(x / 2^(byte-127)); codes
 * packed two per byte, element 2i in the low nibble.                      */
void oracle_mxfp4_quant_row(const uint16_t* x_bf16, int K, uint8_t* packed, uint8_t* scales)
{
    for (int b = 0; b < K / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double v = fabs((double)oracle_bf16_to_f32(x_bf16[b * 32 + i]));
            if (v > amax) amax = v;
        }
        int sb;
        if (amax == 0.0) {
            sb = 0;
        } else {
            int ex;
            frexp(amax, &ex);
            sb = (ex - 1) - 2 + 127;
            if (sb < 0) sb = 0;
            if (sb > 254) sb = 254;
        }
        scales[b] = (uint8_t)sb;
        for (int i = 0; i < 16; ++i) {
            double v0 = (double)oracle_bf16_to_f32(x_bf16[b * 32 + 2 * i]);
            double v1 = (double)oracle_bf16_to_f32(x_bf16[b * 32 + 2 * i + 1]);
            uint8_t c0 = oracle_e2m1_encode(ldexp(v0, 127 - sb));
            uint8_t c1 = oracle_e2m1_encode(ldexp(v1, 127 - sb));
            packed[b * 16 + i] = (uint8_t)(c0 | (c1 << 4));
        }
    }
}

/* One element of a canonical MXFP4 matrix [rows][K]: codes [rows][K/2] with
 * element 2i in the low nibble, scales [rows][K/32].  Exact in fp32.        */
static float mxfp4_at(const uint8_t* codes, const uint8_t* scales, int K, int r, int c)
{
    uint8_t byte = codes[(size_t)r * (K / 2) + c / 2];
    uint8_t nib = (c & 1) ? (byte >> 4) : (byte & 15);
    double v = oracle_e2m1_value(nib) * oracle_e8m0_value(scales[(size_t)r * (K / 32) + c / 32]);
    return (float)v;
}

void oracle_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, int rows, int K, float* out)
{
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < K; ++c)
            out[(size_t)r * K + c] = mxfp4_at(codes, scales, K, r, c);
}

/* ---- GGUF block formats Q8_0 and Q4_K ------------------------------------
 * The tinyserve README ("How it works" item 2; "Supported models",
 * Formats) runs GGUF experts in their native block formats (Q4_K, Q5_K,
 * Q6_K, Q8_0).  The pages name the formats without defining them; the
 * layouts below are the published GGUF / ggml block formats, restated.
 * Blocks run along a row (the reduction dimension); a row of K elements is
 * K/32 Q8_0 blocks or K/256 Q4_K super-blocks, stored back to back.         */

/* IEEE 754 binary16: sign, 5 exponent bits with bias 15, 10 fraction bits;
 * exponent field 0 is subnormal (fraction * 2^-24), 31 is infinity / NaN.  */
double oracle_f16_value(uint16_t h)
{
    int sign = h >> 15;
    int ef = (h >> 10) & 31;
    int fr = h & 1023;
    double mag;
    if (ef == 31) mag = fr ? NAN : INFINITY;
    else if (ef == 0) mag = ldexp((double)fr, -24);
    else mag = ldexp(1024.0 + fr, ef - 25);
    return sign ? -mag : mag;
}

static double f16_le(const uint8_t* p) { return oracle_f16_value((uint16_t)(p[0] | (p[1] << 8))); }

#define Q8_0_BLOCK_BYTES 34
#define Q4_K_BLOCK_BYTES 144

/* Q8_0: per 32 elements, a little-endian binary16 scale d and 32 signed
 * bytes q; element = d * q (exact in fp32: 11 by 8 significant bits).      */
void oracle_dequant_q8_0(const uint8_t* blocks, int rows, int K, float* out)
{
    const size_t rb = (size_t)(K / 32) * Q8_0_BLOCK_BYTES;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < K / 32; ++b) {
            const uint8_t* blk = blocks + r * rb + (size_t)b * Q8_0_BLOCK_BYTES;
            double d = f16_le(blk);
            for (int i = 0; i < 32; ++i)
                out[(size_t)r * K + b * 32 + i] = (float)(d * (double)(int8_t)blk[2 + i]);
        }
}

/* The 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes
 * p of a Q4_K super-block: sub-blocks 0-3 keep theirs in the low 6 bits of
 * p[j] (scale) and p[j+4] (min); sub-blocks 4-7 keep their low 4 bits in
 * the two nibbles of p[j+4] (scale low, min high) and their top 2 bits in
 * the top 2 bits of p[j-4] (scale) and p[j] (min).                         */
static void q4_k_scale_min(const uint8_t* p, int j, int* sc, int* m)
{
    if (j < 4) {
        *sc = p[j] & 63;
        *m = p[j + 4] & 63;
    } else {
        *sc = (p[j + 4] & 15) | ((p[j - 4] >> 6) << 4);
        *m = (p[j + 4] >> 4) | ((p[j] >> 6) << 4);
    }
}

/* Q4_K: per 256 elements (8 sub-blocks of 32), 144 bytes:
 *   0-1 d, 2-3 dmin (little-endian binary16); 4-15 the packed 6-bit
 *   scales and mins; 16-143 the 4-bit values: sub-blocks 2g and 2g+1 share
 *   the 32 bytes 16+32g .. 16+32g+31, element l of sub-block 2g in the low
 *   nibble of byte l, element l of sub-block 2g+1 in its high nibble.
 * element = d*sc*q - dmin*m, rounded once to fp32.  d*sc and dmin*m are
 * exact in fp32 (11 by 6 significant bits), so one fused multiply-add
 * gives that single rounding.                                              */
void oracle_dequant_q4_k(const uint8_t* blocks, int rows, int K, float* out)
{
    const size_t rb = (size_t)(K / 256) * Q4_K_BLOCK_BYTES;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < K / 256; ++b) {
            const uint8_t* blk = blocks + r * rb + (size_t)b * Q4_K_BLOCK_BYTES;
            double d = f16_le(blk), dmin = f16_le(blk + 2);
            for (int j = 0; j < 8; ++j) {
                int sc, m;
                q4_k_scale_min(blk + 4, j, &sc, &m);
                float dl = (float)(d * sc), ml = (float)(dmin * m);
                const uint8_t* qs = blk + 16 + 32 * (j / 2);
                for (int l = 0; l < 32; ++l) {
                    int q = (j & 1) ? (qs[l] >> 4) : (qs[l] & 15);
                    out[(size_t)r * K + b * 256 + j * 32 + l] = fmaf(dl, (float)q, -ml);
                }
            }
        }
}

/* Bytes of one row of K elements in a GGUF format (0: Q8_0, 1: Q4_K), or 0
 * when K does not fit the format's block.                                  */
long oracle_gguf_row_bytes(int fmt, int K)
{
    if (K <= 0) return 0;
    if (fmt == 0) return K % 32 ? 0 : (long)(K / 32) * Q8_0_BLOCK_BYTES;
    if (fmt == 1) return K % 256 ? 0 : (long)(K / 256) * Q4_K_BLOCK_BYTES;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Routing: top-k, softmax over the selected, histogram, permutation          */
/* ------------------------------------------------------------------------ */

/* Order of candidates: larger logit first, equal logits by lower id; NaN
 * ranks below every number (NaN logits are never generated).                */
static int ranks_before(float la, int a, float lb, int b)
{
    int na = isnan(la), nb = isnan(lb);
    if (na != nb) return nb;
    if (!na && la != lb) return la > lb;
    return a < b;
}

int oracle_route(const float* logits, int T, int E, int k, int32_t* ids, float* w)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E) return ORACLE_ERR_INVALID;
    char* taken = (char*)malloc((size_t)E);
    double* ex = (double*)malloc(sizeof(double) * (size_t)k);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {       /* selection, one rank at a time */
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        /* softmax over the k selected logits, max-subtracted, in fp64     */
        double m = (double)l[ids[(size_t)t * k]];
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            ex[j] = exp((double)l[ids[(size_t)t * k + j]] - m);
            sum += ex[j];
        }
        for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = (float)(ex[j] / sum);
    }
    free(taken);
    free(ex);
    return ORACLE_OK;
}

/* counts[e] = number of assignments routed to e; offsets = exclusive prefix
 * sum (offsets[E] = T*k); perm lists assignment indices a = t*k + j grouped
 * by expert ascending, ascending a inside a group; inv[perm[p]] = p.        */
int oracle_hist_perm(const int32_t* ids, int T, int k, int E,
                     int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv)
{
    long n = (long)T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long a = 0; a < n; ++a) {
        if (ids[a] < 0 || ids[a] >= E) return ORACLE_ERR_INVALID;
        counts[ids[a]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    long p = 0;
    for (int e = 0; e < E; ++e)
        for (long a = 0; a < n; ++a)
            if (ids[a] == e) { perm[p] = (int32_t)a; inv[a] = (int32_t)p; ++p; }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Pool: one LRU event per (layer, step)                                      */
/* ------------------------------------------------------------------------ */

/* State of one layer's pool: slot_expert[S] (-1 free), expert_slot[E] (-1
 * absent), stamp[S], *clock.  The event is the unique routed set U (experts
 * with counts > 0) in ascending id.
 *  1. each resident e in U is a hit and receives a fresh stamp (++clock);
 *  2. each absent e in U, ascending, takes the lowest free slot, else evicts
 *     the resident expert with the smallest stamp, and receives a fresh stamp.
 * Everything in U was stamped during the event, so U is never evicted.  With
 * |U| > S the event cannot be served: nothing changes, ORACLE_ERR_CAPACITY.
 * load_expert/load_slot list the copies the event needs, in issue order.    */
int oracle_lru_step(int S, int E, const int32_t* counts,
                    int32_t* slot_expert, int32_t* expert_slot, int64_t* stamp, int64_t* clock,
                    int64_t* hits, int64_t* misses, int64_t* evictions,
                    int32_t* load_expert, int32_t* load_slot, int32_t* n_loads)
{
    int uniq = 0;
    for (int e = 0; e < E; ++e) uniq += counts[e] > 0;
    *n_loads = 0;
    if (uniq > S) return ORACLE_ERR_CAPACITY;
    for (int e = 0; e < E; ++e) {
        if (counts[e] > 0 && expert_slot[e] >= 0) {
            stamp[expert_slot[e]] = ++(*clock);
            *hits += 1;
        }
    }
    for (int e = 0; e < E; ++e) {
        if (counts[e] <= 0 || expert_slot[e] >= 0) continue;
        int s = -1;
        for (int i = 0; i < S; ++i)
            if (slot_expert[i] < 0) { s = i; break; }
        if (s < 0) {
            for (int i = 0; i < S; ++i)
                if (s < 0 || stamp[i] < stamp[s]) s = i;
            expert_slot[slot_expert[s]] = -1;
            *evictions += 1;
        }
        slot_expert[s] = e;
        expert_slot[e] = s;
        stamp[s] = ++(*clock);
        *misses += 1;
        load_expert[*n_loads] = e;
        load_slot[*n_loads] = s;
        *n_loads += 1;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Expert FFN                                                                 */
/* ------------------------------------------------------------------------ */

static float silu_f32(float g) { return g / (1.0f + expf(-g)); }

/* Row r of the gate/up pair for an fp32 activation vector xf[K]:
 * g = sum_c Wg[r][c]*xf[c], u likewise (fp32, ascending c),
 * h = bf16(silu(g) * u).                                                     */
static uint16_t gateup_row(const uint8_t* gc, const uint8_t* gs, const uint8_t* uc, const uint8_t* us,
                           int H, int r, const float* xf, float* g_out, float* u_out)
{
    float g = 0.0f, u = 0.0f;
    for (int c = 0; c < H; ++c) {
        g = g + mxfp4_at(gc, gs, H, r, c) * xf[c];
        u = u + mxfp4_at(uc, us, H, r, c) * xf[c];
    }
    if (g_out) *g_out = g;
    if (u_out) *u_out = u;
    float s = silu_f32(g);
    return oracle_f32_to_bf16(s * u);
}

/* y[r] = sum_c Wd[r][c]*hf[c] (fp32, ascending c).                          */
static float down_row(const uint8_t* dc, const uint8_t* ds, int I, int r, const float* hf)
{
    float y = 0.0f;
    for (int c = 0; c < I; ++c) y = y + mxfp4_at(dc, ds, I, r, c) * hf[c];
    return y;
}

/* Single-expert pieces, exposed so the tests can pin them on their own.     */
void oracle_expert_gateup(const uint8_t* gc, const uint8_t* gs, const uint8_t* uc, const uint8_t* us,
                          int H, int I, const float* xf, float* g, float* u, uint16_t* h_bf16)
{
    for (int r = 0; r < I; ++r) h_bf16[r] = gateup_row(gc, gs, uc, us, H, r, xf, g + r, u + r);
}

void oracle_expert_down(const uint8_t* dc, const uint8_t* ds, int H, int I, const float* hf, float* y)
{
    for (int r = 0; r < H; ++r) y[r] = down_row(dc, ds, I, r, hf);
}

/* ---- a minimal static parallel-for over independent items --------------- */

typedef void (*item_fn)(void* ctx, long item);
typedef struct { item_fn fn; void* ctx; long lo, hi; } span_t;

static void* run_span(void* p)
{
    span_t* s = (span_t*)p;
    for (long i = s->lo; i < s->hi; ++i) s->fn(s->ctx, i);
    return NULL;
}

/* Items are independent (each writes only its own outputs), so splitting
 * them over threads changes no arithmetic.                                  */
static void parallel_for(long n, int threads, item_fn fn, void* ctx)
{
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (threads == 1 || n < 2) {
        for (long i = 0; i < n; ++i) fn(ctx, i);
        return;
    }
    pthread_t th[256];
    span_t sp[256];
    for (int i = 0; i < threads; ++i) {
        sp[i].fn = fn;
        sp[i].ctx = ctx;
        sp[i].lo = n * i / threads;
        sp[i].hi = n * (i + 1) / threads;
        pthread_create(&th[i], NULL, run_span, &sp[i]);
    }
    for (int i = 0; i < threads; ++i) pthread_join(th[i], NULL);
}

/* ---- whole layer ------------------------------------------------------- */

typedef struct {
    int T, H, I, k, prefill;
    const int32_t* ids;
    const float* w;
    const uint8_t *gc, *gs, *uc, *us, *dc, *ds;   /* stacked [E][...]       */
    const float* xf;       /* [T][H] fp32 view of the activations used       */
    uint16_t* h;           /* [T*k][I] bf16 SwiGLU output                    */
    float* hf;             /* [T*k][I] fp32 view of the down-projection input */
    float* out;            /* [T][H]                                          */
} layer_ctx;

static void item_gateup(void* p, long item)
{
    layer_ctx* c = (layer_ctx*)p;
    long a = item / c->I;
    int r = (int)(item % c->I);
    int t = (int)(a / c->k);
    size_t e = (size_t)c->ids[a];
    size_t gsz = (size_t)c->I * (c->H / 2), ssz = (size_t)c->I * (c->H / 32);
    c->h[(size_t)a * c->I + r] = gateup_row(c->gc + e * gsz, c->gs + e * ssz, c->uc + e * gsz,
                                            c->us + e * ssz, c->H, r, c->xf + (size_t)t * c->H,
                                            NULL, NULL);
}

static void item_down_combine(void* p, long item)
{
    layer_ctx* c = (layer_ctx*)p;
    int t = (int)(item / c->H);
    int r = (int)(item % c->H);
    size_t dsz = (size_t)c->H * (c->I / 2), ssz = (size_t)c->H * (c->I / 32);
    float acc = 0.0f;
    for (int j = 0; j < c->k; ++j) {
        size_t a = (size_t)t * c->k + j;
        size_t e = (size_t)c->ids[a];
        float y = down_row(c->dc + e * dsz, c->ds + e * ssz, c->I, r, c->hf + a * c->I);
        acc = acc + c->w[a] * y;
    }
    c->out[(size_t)t * c->H + r] = acc;
}

/* The whole layer for T tokens.
 *   prefill = 0 (decode path): the expert input is the bf16 activation and
 *     the down projection reads bf16(h).
 *   prefill = 1 (prefill path): the expert input is MXFP8(x) per token and
 *     the down projection reads MXFP8(bf16(h)) per assignment; both use the
 *     block-32 rule of oracle_mxfp8_quant_row.
 *   prefill = 2 (FP4-activation variant of the prefill path): as 1, with
 *     MXFP4 in place of MXFP8 for both quantisation points, by the block-32
 *     rule of oracle_mxfp4_quant_row (E2M1 x E2M1 products, the all-FP4
 *     block-scaled MMA of the Blackwell MX formats).
 * Weights are stacked canonical arrays indexed by the ids.  Optional outputs
 * (may be NULL): h_bf16 [T*k][I]; xq/xs [T][H], [T][H/32]; hq/hs [T*k][I],
 * [T*k][I/32] (prefill only; with prefill = 2 the codes are packed two per
 * byte, so xq is [T][H/2] and hq [T*k][I/2]).                               */
int oracle_layer(int prefill, int T, int H, int I, int k,
                 const uint16_t* x_bf16, const int32_t* ids, const float* w,
                 const uint8_t* gate_codes, const uint8_t* gate_scales,
                 const uint8_t* up_codes, const uint8_t* up_scales,
                 const uint8_t* down_codes, const uint8_t* down_scales,
                 float* out, uint16_t* h_bf16,
                 uint8_t* xq, uint8_t* xs, uint8_t* hq, uint8_t* hs, int threads)
{
    if (T < 0 || H <= 0 || I <= 0 || k <= 0 || H % 32 || I % 32) return ORACLE_ERR_INVALID;
    if (prefill < 0 || prefill > 2) return ORACLE_ERR_INVALID;
    size_t A = (size_t)T * k;
    float* xf = (float*)malloc(sizeof(float) * (size_t)T * H + 1);
    float* hf = (float*)malloc(sizeof(float) * A * I + 1);
    uint16_t* h = h_bf16 ? h_bf16 : (uint16_t*)malloc(sizeof(uint16_t) * A * I + 1);
    uint8_t* q = (uint8_t*)malloc((size_t)(H > I ? H : I) + 1);
    uint8_t* s = (uint8_t*)malloc((size_t)(H > I ? H : I) / 32 + 1);

    for (int t = 0; t < T; ++t) {
        const uint16_t* xr = x_bf16 + (size_t)t * H;
        float* xo = xf + (size_t)t * H;
        if (!prefill) {
            for (int c = 0; c < H; ++c) xo[c] = oracle_bf16_to_f32(xr[c]);
        } else if (prefill == 2) {
            oracle_mxfp4_quant_row(xr, H, q, s);
            for (int c = 0; c < H; ++c) xo[c] = mxfp4_at(q, s, H, 0, c);
            if (xq) memcpy(xq + (size_t)t * (H / 2), q, (size_t)H / 2);
            if (xs) memcpy(xs + (size_t)t * (H / 32), s, (size_t)H / 32);
        } else {
            oracle_mxfp8_quant_row(xr, H, q, s);
            for (int c = 0; c < H; ++c) xo[c] = (float)(oracle_e4m3_value(q[c]) * oracle_e8m0_value(s[c / 32]));
            if (xq) memcpy(xq + (size_t)t * H, q, (size_t)H);
            if (xs) memcpy(xs + (size_t)t * (H / 32), s, (size_t)H / 32);
        }
    }

    layer_ctx c = {T, H, I, k, prefill, ids, w, gate_codes, gate_scales, up_codes, up_scales,
                   down_codes, down_scales, xf, h, hf, out};
    parallel_for((long)A * I, threads, item_gateup, &c);

    for (size_t a = 0; a < A; ++a) {
        const uint16_t* hr = h + a * I;
        float* ho = hf + a * I;
        if (!prefill) {
            for (int i = 0; i < I; ++i) ho[i] = oracle_bf16_to_f32(hr[i]);
        } else if (prefill == 2) {
            oracle_mxfp4_quant_row(hr, I, q, s);
            for (int i = 0; i < I; ++i) ho[i] = mxfp4_at(q, s, I, 0, i);
            if (hq) memcpy(hq + a * (I / 2), q, (size_t)I / 2);
            if (hs) memcpy(hs + a * (I / 32), s, (size_t)I / 32);
        } else {
            oracle_mxfp8_quant_row(hr, I, q, s);
            for (int i = 0; i < I; ++i) ho[i] = (float)(oracle_e4m3_value(q[i]) * oracle_e8m0_value(s[i / 32]));
            if (hq) memcpy(hq + a * I, q, (size_t)I);
            if (hs) memcpy(hs + a * (I / 32), s, (size_t)I / 32);
        }
    }

    parallel_for((long)T * H, threads, item_down_combine, &c);

    free(xf);
    free(hf);
    if (!h_bf16) free(h);
    free(q);
    free(s);
    return ORACLE_OK;
}

/* ---- whole decode layer on GGUF expert weights -------------------------- */

typedef struct {
    int H, I, n;           /* n assignments of the current expert            */
    const int32_t* as;     /* their assignment indices a = t*k + j           */
    int k;
    const float *wg, *wu, *wd;  /* the expert's dequantised matrices         */
    const float* xf;       /* [T][H] fp32 activations                        */
    uint16_t* h;           /* [T*k][I]                                       */
    float* hf;             /* [T*k][I]                                       */
    float* y;              /* [T*k][H]                                       */
} gguf_ctx;

static void item_gguf_gateup(void* p, long item)
{
    gguf_ctx* c = (gguf_ctx*)p;
    int a = c->as[item / c->I];
    int r = (int)(item % c->I);
    const float* x = c->xf + (size_t)(a / c->k) * c->H;
    const float* gr = c->wg + (size_t)r * c->H;
    const float* ur = c->wu + (size_t)r * c->H;
    float g = 0.0f, u = 0.0f;
    for (int i = 0; i < c->H; ++i) {
        g = g + gr[i] * x[i];
        u = u + ur[i] * x[i];
    }
    uint16_t hb = oracle_f32_to_bf16(silu_f32(g) * u);
    c->h[(size_t)a * c->I + r] = hb;
    c->hf[(size_t)a * c->I + r] = oracle_bf16_to_f32(hb);
}

static void item_gguf_down(void* p, long item)
{
    gguf_ctx* c = (gguf_ctx*)p;
    int a = c->as[item / c->H];
    int r = (int)(item % c->H);
    const float* dr = c->wd + (size_t)r * c->I;
    const float* hr = c->hf + (size_t)a * c->I;
    float y = 0.0f;
    for (int i = 0; i < c->I; ++i) y = y + dr[i] * hr[i];
    c->y[(size_t)a * c->H + r] = y;
}

/* The decode path of oracle_layer on GGUF expert weights (fmt 0: Q8_0,
 * 1: Q4_K): bf16 activations times the fp32-dequantised weights, products
 * and sums in fp32 in ascending reduction index, h = bf16(silu(g)*u), and
 * the combine in rank order.  Weights are stacked [E][rows][row bytes]:
 * gate and up I rows of H elements, down H rows of I elements.  h_bf16
 * [T*k][I] may be NULL.                                                    */
int oracle_layer_gguf(int fmt, int T, int H, int I, int k, const uint16_t* x_bf16, const int32_t* ids,
                      const float* w, const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                      int E, float* out, uint16_t* h_bf16, int threads)
{
    long rbh = oracle_gguf_row_bytes(fmt, H), rbi = oracle_gguf_row_bytes(fmt, I);
    if (T < 0 || k <= 0 || E <= 0 || !rbh || !rbi) return ORACLE_ERR_INVALID;
    size_t A = (size_t)T * k;
    for (size_t a = 0; a < A; ++a)
        if (ids[a] < 0 || ids[a] >= E) return ORACLE_ERR_INVALID;
    void (*deq)(const uint8_t*, int, int, float*) = fmt == 0 ? oracle_dequant_q8_0 : oracle_dequant_q4_k;
    float* xf = (float*)malloc(sizeof(float) * (size_t)T * H + 1);
    float* wg = (float*)malloc(sizeof(float) * (size_t)I * H);
    float* wu = (float*)malloc(sizeof(float) * (size_t)I * H);
    float* wd = (float*)malloc(sizeof(float) * (size_t)H * I);
    uint16_t* h = h_bf16 ? h_bf16 : (uint16_t*)malloc(sizeof(uint16_t) * A * I + 1);
    float* hf = (float*)malloc(sizeof(float) * A * I + 1);
    float* y = (float*)malloc(sizeof(float) * A * H + 1);
    int32_t* as = (int32_t*)malloc(sizeof(int32_t) * A + 1);
    for (size_t i = 0; i < (size_t)T * H; ++i) xf[i] = oracle_bf16_to_f32(x_bf16[i]);

    for (int e = 0; e < E; ++e) {
        int n = 0;
        for (size_t a = 0; a < A; ++a)
            if (ids[a] == e) as[n++] = (int32_t)a;
        if (!n) continue;
        const size_t eg = (size_t)I * rbh, ed = (size_t)H * rbi;
        deq(gate + e * eg, I, H, wg);
        deq(up + e * eg, I, H, wu);
        deq(down + e * ed, H, I, wd);
        gguf_ctx c = {H, I, n, as, k, wg, wu, wd, xf, h, hf, y};
        parallel_for((long)n * I, threads, item_gguf_gateup, &c);
        parallel_for((long)n * H, threads, item_gguf_down, &c);
    }

    for (int t = 0; t < T; ++t)
        for (int r = 0; r < H; ++r) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                size_t a = (size_t)t * k + j;
                acc = acc + w[a] * y[a * H + r];
            }
            out[(size_t)t * H + r] = acc;
        }

    free(xf);
    free(wg);
    free(wu);
    free(wd);
    if (!h_bf16) free(h);
    free(hf);
    free(y);
    free(as);
    return ORACLE_OK;
}

/* Weighted combine on its own: out[t][r] = sum_j w[t][j] * y[t*k+j][r], in
 * ascending j, fp32, starting from 0.                                       */
void oracle_combine(const float* y, const float* w, int T, int k, int H, float* out)
{
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < H; ++r) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j)
                acc = acc + w[(size_t)t * k + j] * y[((size_t)t * k + j) * H + r];
            out[(size_t)t * H + r] = acc;
        }
}
