/*
 * oracle.c -- plain, slow, single-threaded CPU reference for the paged decode
 * path: ReshapeAndCache, GQA paged decode attention, Quest metadata, Quest
 * block scoring and top-K selection, Quest sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker the CUDA kernels are
 * compared against. It shares no code, header, table or helper with the CUDA
 * library. Only the test suite, the smoke check and the benchmark's CPU
 * baseline may build, load or call it; the product path never does.
 *
 * Sources (web pages, by title and section):
 *   [P1] "Ascend Kernel-to-Serving Pipeline": sections "ReshapeAndCache",
 *        "GQA Paged Attention", "Quest Sparse Attention", "Sparse precision".
 *   [P2] "18 e2e inference serving" (TileLang tutorial): section 2.6 (paged KV
 *        layout and block table), section 4.1 (split-KV partial outputs and
 *        their weighted combine).
 *   Quest scoring rule (not printed on the pages; fixed by the project's
 *   statement of the method): per physical block and KV head, elementwise
 *   min/max of K; block score = sum over the GQA group of
 *   sum_d max(q_d*min_d, q_d*max_d); top-K blocks, ties to the lower index.
 *
 * Conventions:
 *   bf16 values are passed as uint16 bit patterns.
 *   Cache layout [NB][BS][Hkv][D] per layer ([P2] 2.6).
 *   block_tables [B][MBS] int32, context_lens [B] int32, slot_mapping [T] int64.
 *   Query head h uses KV head h / G, G = Hq / Hkv (contiguous groups; [P1]
 *   "GQA Paged Attention" says only that several query heads share one KV head).
 *   Attention arithmetic is fp64 (at least the fp32 the method asks for).
 *
 * The Quest block score exists twice: oracle_quest_scores_plain is the
 * method's sum written out term by term in fp64 (the definition the selected
 * sets are checked against); oracle_quest_scores_kernel_order evaluates the
 * same sum in fp32 in the CUDA kernel's fixed order, a bit-exact reproduction
 * of the kernel's arithmetic that the tests hold to a stated error bound
 * around the plain form.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared oracle.c -lm
 * (no fused multiply-add contraction: the kernel-order score is defined as a
 * sequence of individually rounded fp32 operations).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- helpers */

static double bf16_val(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE-754 totalOrder key of a bf16 bit pattern: numeric order for non-NaN
 * values, with -0 ranked below +0 (so min/max are unique bit patterns). */
static uint16_t bf16_order_key(uint16_t h)
{
    return (h & 0x8000u) ? (uint16_t)(~h & 0xFFFFu) : (uint16_t)(h | 0x8000u);
}

/* totalOrder key of an fp32 value (same idea, 32 bits). */
static uint32_t f32_order_key(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

/* totalOrder key of an fp64 value (same idea, 64 bits). */
static uint64_t f64_order_key(double f)
{
    uint64_t u;
    memcpy(&u, &f, sizeof u);
    return (u >> 63) ? ~u : (u | (1ull << 63));
}

/* ------------------------------------------------- 8-bit float (E4M3) */

/* The E4M3 variant of the OCP 8-bit floating-point format (the "fn" variant:
 * no infinities). Bit 7 is the sign, bits 6..3 the exponent field e (bias 7),
 * bits 2..0 the mantissa m:
 *   e = 0:          (-1)^s * (m / 8) * 2^-6          (zero and subnormals)
 *   e = 1 .. 15:    (-1)^s * (1 + m / 8) * 2^(e - 7)
 *   e = 15, m = 7:  NaN (0x7F and 0xFF).
 * Largest finite magnitude 448 (0x7E), smallest nonzero 2^-9 (0x01). */
double oracle_e4m3_decode(uint8_t c)
{
    const int sgn = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -mag : mag;
}

/* Nearest E4M3 value to x, ties to the even mantissa; magnitudes beyond 448
 * (infinities included) saturate to +-448; NaN gives 0x7F. The grid spacing
 * is 2^(E-3) in the binade [2^E, 2^(E+1)) for E >= -6 and 2^-9 below 2^-6,
 * so x / spacing is exact in double and is rounded to an integer. */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return sgn | 0x7E;
    int E = 0;
    if (a > 0.0) {
        (void)frexp(a, &E); /* a = f * 2^E, f in [0.5, 1): binade exponent E - 1 */
        E -= 1;
    }
    if (a == 0.0 || E < -6)
        E = -6;
    const double q = ldexp(1.0, E - 3);
    const double n = a / q;
    double r = floor(n);
    const double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) == 1.0))
        r += 1.0;
    const double v = r * q; /* <= 448: 448 is on the grid and a < 448 */
    if (v == 0.0)
        return sgn;
    if (v < ldexp(1.0, -6))
        return sgn | (uint8_t)(v / ldexp(1.0, -9));
    int ev = 0;
    (void)frexp(v, &ev);
    ev -= 1; /* v in [2^ev, 2^(ev+1)) */
    const int mant = (int)((v / ldexp(1.0, ev) - 1.0) * 8.0);
    return sgn | (uint8_t)(((ev + 7) << 3) | mant);
}

/* encode / decode whole arrays (for the tests) */
void oracle_e4m3_encode_array(const float *x, uint8_t *c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        c[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t *c, double *x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        x[i] = oracle_e4m3_decode(c[i]);
}

/* Order key of an E4M3 code: numeric order for non-NaN codes, -0 below +0
 * (the same totalOrder convention as the bf16 metadata). */
static uint8_t e4m3_order_key(uint8_t c)
{
    return (c & 0x80u) ? (uint8_t)(~c & 0x7Fu) : (uint8_t)(c | 0x80u);
}

/* Layout of an E4M3 V cache. K codes keep the bf16 layout [NB][BS][Hkv][D]
 * (one token's row of all KV heads). V codes are stored per block and KV head
 * as a [D][16] byte matrix: the 16 bytes of dim d hold the block's 16 tokens
 * in the order 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15, i.e. token o at byte
 *     pos(o) = 4 * ((o mod 8) div 2) + 2 * (o div 8) + (o mod 2).
 * (That order makes the GPU's 4-byte fragment loads hold two consecutive
 * token pairs; for the method it is only an address function.) Block size 16. */
static int64_t vt_token_pos(int64_t o)
{
    return 4 * ((o & 7) >> 1) + 2 * (o >> 3) + (o & 1);
}

static int64_t vt_index(int64_t p, int64_t o, int64_t h, int64_t d, int Hkv, int D)
{
    return ((p * Hkv + h) * D + d) * 16 + vt_token_pos(o);
}

/* code of one bf16 element quantised with a per-KV-head scale:
 * e4m3(fl32(x / scale)) */
static uint8_t quantize(uint16_t x, float scale)
{
    const float y = bf16_f32(x) / scale;
    return oracle_e4m3_encode(y);
}

/* ------------------------------------------------------ ReshapeAndCache */

/* [P1] "ReshapeAndCache": for every new token t with slot = slot_mapping[t]:
 *   block_idx = slot // block_size, block_offset = slot % block_size,
 *   and the token's K and V rows (all KV heads) go to that block and offset;
 *   slot < 0 means the token is skipped.
 * Tokens are applied in order. A slot past the pool (block_idx >= NB) is not
 * written; the return value counts such slots. */
int64_t oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                                 uint16_t *key_cache, uint16_t *value_cache,
                                 const int64_t *slot_mapping, int64_t T,
                                 int Hkv, int D, int BS, int64_t NB)
{
    const int64_t row = (int64_t)Hkv * D;
    int64_t out_of_range = 0;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        const int64_t block_idx = slot / BS;
        const int64_t block_offset = slot % BS;
        if (block_idx >= NB) {
            ++out_of_range;
            continue;
        }
        const int64_t dst = (block_idx * BS + block_offset) * row;
        for (int64_t e = 0; e < row; ++e) {
            key_cache[dst + e] = key[t * row + e];
            value_cache[dst + e] = value[t * row + e];
        }
    }
    return out_of_range;
}

/* ---------------------------------------------------- Quest metadata */

/* Incremental metadata update for the tokens of one ReshapeAndCache call.
 * Metadata is per physical block p and KV head h: kmin[p][h][d], kmax[p][h][d]
 * = elementwise min / max of K over the block's tokens.
 * For each physical block touched by a valid slot in this call:
 *   - if some token of the call lands at offset 0 of the block (the block
 *     starts fresh), the new metadata is the min/max over this call's tokens
 *     in that block only;
 *   - otherwise it is min/max of the old metadata and this call's tokens.
 * min/max follow IEEE totalOrder (so -0 < +0) and the result does not depend
 * on token order. Returns the number of out-of-pool slots ignored. */
int64_t oracle_quest_update_meta(uint16_t *kmin, uint16_t *kmax,
                                 const uint16_t *key, const int64_t *slot_mapping,
                                 int64_t T, int Hkv, int D, int BS, int64_t NB)
{
    const int64_t row = (int64_t)Hkv * D;
    int64_t out_of_range = 0;
    unsigned char *done = (unsigned char *)calloc((size_t)T, 1);
    uint16_t *lo = (uint16_t *)malloc((size_t)row * sizeof(uint16_t));
    uint16_t *hi = (uint16_t *)malloc((size_t)row * sizeof(uint16_t));
    for (int64_t t = 0; t < T; ++t) {
        const int64_t s = slot_mapping[t];
        if (s < 0 || done[t])
            continue;
        const int64_t p = s / BS;
        if (p >= NB) {
            ++out_of_range;
            done[t] = 1;
            continue;
        }
        /* every token of this call that lands in block p */
        int reset = 0;
        for (int64_t u = t; u < T; ++u) {
            const int64_t su = slot_mapping[u];
            if (su >= 0 && su / BS == p && su % BS == 0)
                reset = 1;
        }
        int have = 0;
        if (!reset) {
            memcpy(lo, kmin + p * row, (size_t)row * sizeof(uint16_t));
            memcpy(hi, kmax + p * row, (size_t)row * sizeof(uint16_t));
            have = 1;
        }
        for (int64_t u = t; u < T; ++u) {
            const int64_t su = slot_mapping[u];
            if (su < 0 || su / BS != p)
                continue;
            done[u] = 1;
            const uint16_t *k = key + u * row;
            for (int64_t e = 0; e < row; ++e) {
                if (!have) {
                    lo[e] = k[e];
                    hi[e] = k[e];
                } else {
                    if (bf16_order_key(k[e]) < bf16_order_key(lo[e]))
                        lo[e] = k[e];
                    if (bf16_order_key(k[e]) > bf16_order_key(hi[e]))
                        hi[e] = k[e];
                }
            }
            have = 1;
        }
        memcpy(kmin + p * row, lo, (size_t)row * sizeof(uint16_t));
        memcpy(kmax + p * row, hi, (size_t)row * sizeof(uint16_t));
    }
    free(done);
    free(lo);
    free(hi);
    return out_of_range;
}

/* Metadata from scratch: for each sequence b and logical block j < ceil(ctx/BS),
 * p = block_tables[b][j], min/max over the block's valid tokens
 * (positions j*BS .. min(ctx, (j+1)*BS) - 1). Returns -1 on a table entry
 * outside the pool, else 0. */
int oracle_quest_rebuild_meta(uint16_t *kmin, uint16_t *kmax,
                              const uint16_t *key_cache,
                              const int32_t *block_tables, int MBS,
                              const int32_t *context_lens, int B,
                              int Hkv, int D, int BS, int64_t NB)
{
    const int64_t row = (int64_t)Hkv * D;
    for (int b = 0; b < B; ++b) {
        const int64_t ctx = context_lens[b] > 0 ? context_lens[b] : 0;
        const int64_t nblk = (ctx + BS - 1) / BS;
        for (int64_t j = 0; j < nblk && j < MBS; ++j) {
            const int64_t p = block_tables[(int64_t)b * MBS + j];
            if (p < 0 || p >= NB)
                return -1;
            const int64_t t_end = (j + 1) * BS < ctx ? (j + 1) * BS : ctx;
            for (int64_t e = 0; e < row; ++e) {
                uint16_t lo = 0, hi = 0;
                for (int64_t t = j * BS; t < t_end; ++t) {
                    const uint16_t v = key_cache[(p * BS + (t % BS)) * row + e];
                    if (t == j * BS || bf16_order_key(v) < bf16_order_key(lo))
                        lo = v;
                    if (t == j * BS || bf16_order_key(v) > bf16_order_key(hi))
                        hi = v;
                }
                kmin[p * row + e] = lo;
                kmax[p * row + e] = hi;
            }
        }
    }
    return 0;
}

/* ------------------------------------------- fp8 KV cache: write path */

/* ReshapeAndCache into an E4M3 cache: the same slot arithmetic as
 * oracle_reshape_and_cache; element d of KV head h of the token's K row is
 * stored as e4m3(fl32(k / k_scale[h])), likewise V with v_scale[h].
 * Returns the number of out-of-pool slots skipped. */
int64_t oracle_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value,
                                     uint8_t *key_cache, uint8_t *value_cache,
                                     const int64_t *slot_mapping, int64_t T,
                                     const float *k_scale, const float *v_scale,
                                     int Hkv, int D, int BS, int64_t NB)
{
    const int64_t row = (int64_t)Hkv * D;
    int64_t out_of_range = 0;
    if (BS != 16)
        return -2;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        const int64_t block_idx = slot / BS;
        const int64_t block_offset = slot % BS;
        if (block_idx >= NB) {
            ++out_of_range;
            continue;
        }
        const int64_t dst = (block_idx * BS + block_offset) * row;
        for (int64_t e = 0; e < row; ++e) {
            const int h = (int)(e / D);
            key_cache[dst + e] = quantize(key[t * row + e], k_scale[h]);
            value_cache[vt_index(block_idx, block_offset, h, e % D, Hkv, D)] =
                quantize(value[t * row + e], v_scale[h]);
        }
    }
    return out_of_range;
}

/* Quest metadata of an E4M3 cache: per physical block and KV head, the
 * elementwise min / max of the stored K codes (numeric order, -0 < +0), with
 * the update rule of oracle_quest_update_meta (reset when a token of the call
 * lands at offset 0 of the block, else merge). The new tokens' codes are
 * e4m3(fl32(k / k_scale[h])), as in the cache. */
int64_t oracle_quest_update_meta_fp8(uint8_t *kmin, uint8_t *kmax, const uint16_t *key,
                                     const int64_t *slot_mapping, int64_t T,
                                     const float *k_scale, int Hkv, int D, int BS, int64_t NB)
{
    const int64_t row = (int64_t)Hkv * D;
    int64_t out_of_range = 0;
    unsigned char *done = (unsigned char *)calloc((size_t)T, 1);
    uint8_t *lo = (uint8_t *)malloc((size_t)row);
    uint8_t *hi = (uint8_t *)malloc((size_t)row);
    for (int64_t t = 0; t < T; ++t) {
        const int64_t s = slot_mapping[t];
        if (s < 0 || done[t])
            continue;
        const int64_t p = s / BS;
        if (p >= NB) {
            ++out_of_range;
            done[t] = 1;
            continue;
        }
        int reset = 0;
        for (int64_t u = t; u < T; ++u) {
            const int64_t su = slot_mapping[u];
            if (su >= 0 && su / BS == p && su % BS == 0)
                reset = 1;
        }
        int have = 0;
        if (!reset) {
            memcpy(lo, kmin + p * row, (size_t)row);
            memcpy(hi, kmax + p * row, (size_t)row);
            have = 1;
        }
        for (int64_t u = t; u < T; ++u) {
            const int64_t su = slot_mapping[u];
            if (su < 0 || su / BS != p)
                continue;
            done[u] = 1;
            for (int64_t e = 0; e < row; ++e) {
                const uint8_t c = quantize(key[u * row + e], k_scale[e / D]);
                if (!have) {
                    lo[e] = c;
                    hi[e] = c;
                } else {
                    if (e4m3_order_key(c) < e4m3_order_key(lo[e]))
                        lo[e] = c;
                    if (e4m3_order_key(c) > e4m3_order_key(hi[e]))
                        hi[e] = c;
                }
            }
            have = 1;
        }
        memcpy(kmin + p * row, lo, (size_t)row);
        memcpy(kmax + p * row, hi, (size_t)row);
    }
    free(done);
    free(lo);
    free(hi);
    return out_of_range;
}

/* Metadata of an E4M3 cache from scratch (as oracle_quest_rebuild_meta, on
 * the stored codes). */
int oracle_quest_rebuild_meta_fp8(uint8_t *kmin, uint8_t *kmax, const uint8_t *key_cache,
                                  const int32_t *block_tables, int MBS,
                                  const int32_t *context_lens, int B,
                                  int Hkv, int D, int BS, int64_t NB)
{
    const int64_t row = (int64_t)Hkv * D;
    for (int b = 0; b < B; ++b) {
        const int64_t ctx = context_lens[b] > 0 ? context_lens[b] : 0;
        const int64_t nblk = (ctx + BS - 1) / BS;
        for (int64_t j = 0; j < nblk && j < MBS; ++j) {
            const int64_t p = block_tables[(int64_t)b * MBS + j];
            if (p < 0 || p >= NB)
                return -1;
            const int64_t t_end = (j + 1) * BS < ctx ? (j + 1) * BS : ctx;
            for (int64_t e = 0; e < row; ++e) {
                uint8_t lo = 0, hi = 0;
                for (int64_t t = j * BS; t < t_end; ++t) {
                    const uint8_t v = key_cache[(p * BS + (t % BS)) * row + e];
                    if (t == j * BS || e4m3_order_key(v) < e4m3_order_key(lo))
                        lo = v;
                    if (t == j * BS || e4m3_order_key(v) > e4m3_order_key(hi))
                        hi = v;
                }
                kmin[p * row + e] = lo;
                kmax[p * row + e] = hi;
            }
        }
    }
    return 0;
}

/* ------------------- fp8 KV cache with per-block power-of-two scales */

/* The 8-bit cache with a scale per physical block instead of per KV head
 * (the pages name "fp8 K/V with a per-block scale" as the quantised form of
 * the cache without fixing how the scale is chosen; this is the plainest
 * reading that works for a cache filled one token at a time). Every
 * (physical block p, KV head h) has a K scale k_bscale[p*Hkv + h] and a V
 * scale v_bscale[p*Hkv + h], each a power of two, or 0 while the block holds
 * nothing. One call's write to block p, for K (V alike, without metadata):
 *   1. members: the call's tokens whose slot lands in p; the block restarts
 *      (reset) if a member lands at offset 0;
 *   2. a = the largest finite |x| over the members' elements of head h;
 *   3. e_call = the smallest integer e >= -126 with a <= 448 * 2^e;
 *   4. e_old = log2 of the stored scale, unless the block restarts or the
 *      stored scale is 0 (then there is no e_old);
 *   5. e = max(e_old, e_call); the stored scale becomes 2^e;
 *   6. if e > e_old, every stored code of (p, h) at an offset no member
 *      writes is re-encoded: c <- e4m3(decode(c) * 2^(e_old - e));
 *   7. each member's element is stored as e4m3(fl32(x / 2^e)) (the division
 *      by a power of two is exact);
 *   8. metadata (K): on a restart the min / max of the members' codes; else
 *      the stored min / max, re-encoded as in 6 when e grew, merged with the
 *      members' codes.
 * Because 2^(e_old - e) is a power of two, step 6 changes no value that
 * stays in the E4M3 normal range; only codes that fall below 2^-6 round.
 * Step 8 equals the min / max of the re-encoded codes, as rounding to
 * nearest is monotone. Returns the number of out-of-pool slots skipped, -2
 * for block_size != 16. */
static int block_fit_exponent(double a)
{
    int e = -126;
    while (a > ldexp(448.0, e))
        ++e;
    return e;
}

static void block_scale_step(float *scale_slot, int reset, double amax, int *e_old, int *e_new)
{
    const float s = *scale_slot;
    int have_old = 0, eo = 0;
    if (!reset && s > 0.0f) {
        int E = 0;
        (void)frexp((double)s, &E); /* s = 0.5 * 2^E for a power of two */
        eo = E - 1;
        have_old = 1;
    }
    const int ec = block_fit_exponent(amax);
    const int en = have_old && eo > ec ? eo : ec;
    *e_old = have_old ? eo : en; /* no rescale without an old scale */
    *e_new = en;
    *scale_slot = (float)ldexp(1.0, en);
}

static uint8_t rescale_code(uint8_t c, int shift) /* shift = e_old - e_new <= 0 */
{
    if (shift == 0)
        return c;
    return oracle_e4m3_encode((float)(oracle_e4m3_decode(c) * ldexp(1.0, shift)));
}

int64_t oracle_reshape_and_cache_fp8_block(const uint16_t *key, const uint16_t *value,
                                           uint8_t *key_cache, uint8_t *value_cache,
                                           uint8_t *kmin, uint8_t *kmax,
                                           float *k_bscale, float *v_bscale,
                                           const int64_t *slot_mapping, int64_t T,
                                           int Hkv, int D, int BS, int64_t NB)
{
    if (BS != 16)
        return -2;
    const int64_t row = (int64_t)Hkv * D;
    int64_t out_of_range = 0;
    unsigned char *done = (unsigned char *)calloc((size_t)T + 1, 1);
    int64_t *members = (int64_t *)malloc(sizeof(int64_t) * (size_t)(T + 1));
    for (int64_t t = 0; t < T; ++t) {
        const int64_t s = slot_mapping[t];
        if (s < 0 || done[t])
            continue;
        const int64_t p = s / BS;
        if (p >= NB) {
            ++out_of_range;
            done[t] = 1;
            continue;
        }
        /* step 1: members (t and the later tokens of the call in block p, in order) */
        int reset = 0;
        unsigned written = 0; /* offsets the call writes */
        int64_t nm = 0;
        for (int64_t u = t; u < T; ++u) {
            const int64_t su = slot_mapping[u];
            if (su < 0 || su / BS != p)
                continue;
            members[nm++] = u;
            done[u] = 1;
            written |= 1u << (su % BS);
            if (su % BS == 0)
                reset = 1;
        }
        for (int h = 0; h < Hkv; ++h) {
            /* step 2 */
            double ak = 0.0, av = 0.0;
            for (int64_t i = 0; i < nm; ++i) {
                const int64_t u = members[i];
                for (int d = 0; d < D; ++d) {
                    const double xk = fabs(bf16_val(key[u * row + (int64_t)h * D + d]));
                    const double xv = fabs(bf16_val(value[u * row + (int64_t)h * D + d]));
                    if (isfinite(xk) && xk > ak)
                        ak = xk;
                    if (isfinite(xv) && xv > av)
                        av = xv;
                }
            }
            /* steps 3-5 */
            int eko, ekn, evo, evn;
            block_scale_step(&k_bscale[p * Hkv + h], reset, ak, &eko, &ekn);
            block_scale_step(&v_bscale[p * Hkv + h], reset, av, &evo, &evn);
            /* step 6: the block's other offsets, and step 8's stored min / max */
            for (int o = 0; o < BS; ++o) {
                if (written & (1u << o))
                    continue;
                for (int d = 0; d < D; ++d) {
                    uint8_t *kc = &key_cache[(p * BS + o) * row + (int64_t)h * D + d];
                    *kc = rescale_code(*kc, eko - ekn);
                    uint8_t *vc = &value_cache[vt_index(p, o, h, d, Hkv, D)];
                    *vc = rescale_code(*vc, evo - evn);
                }
            }
            const float ks = (float)ldexp(1.0, ekn), vs = (float)ldexp(1.0, evn);
            int have = 0;
            if (kmin && !reset) {
                for (int d = 0; d < D; ++d) {
                    const int64_t m = (p * Hkv + h) * (int64_t)D + d;
                    kmin[m] = rescale_code(kmin[m], eko - ekn);
                    kmax[m] = rescale_code(kmax[m], eko - ekn);
                }
                have = 1;
            }
            /* step 7, and step 8's merge */
            for (int64_t i = 0; i < nm; ++i) {
                const int64_t u = members[i];
                const int64_t o = slot_mapping[u] % BS;
                for (int d = 0; d < D; ++d) {
                    const int64_t e = (int64_t)h * D + d;
                    const uint8_t c = quantize(key[u * row + e], ks);
                    key_cache[(p * BS + o) * row + e] = c;
                    value_cache[vt_index(p, o, h, d, Hkv, D)] = quantize(value[u * row + e], vs);
                    if (kmin) {
                        const int64_t m = (p * Hkv + h) * (int64_t)D + d;
                        if (!have || e4m3_order_key(c) < e4m3_order_key(kmin[m]))
                            kmin[m] = c;
                        if (!have || e4m3_order_key(c) > e4m3_order_key(kmax[m]))
                            kmax[m] = c;
                    }
                }
                have = 1;
            }
        }
    }
    free(done);
    free(members);
    return out_of_range;
}

/* ------------------------------------------------------------ attention */

/* The tokens one (sequence, KV head) attends to, in order.
 * Dense ([P1] "GQA Paged Attention"): positions 0 .. ctx-1.
 * Sparse ([P1] "Quest Sparse Attention"): for each selected logical block j
 * (in the order given, negative entries skipped), the positions
 * j*BS .. min(ctx, (j+1)*BS) - 1; blocks and tokens past ctx are skipped.
 * Writes positions into pos[] and returns their count. */
static int64_t token_list(int64_t *pos, int64_t ctx, int BS,
                          const int32_t *sel_row, int topk)
{
    int64_t n = 0;
    if (ctx < 0)
        ctx = 0;
    if (!sel_row) {
        for (int64_t t = 0; t < ctx; ++t)
            pos[n++] = t;
        return n;
    }
    for (int i = 0; i < topk; ++i) {
        const int64_t j = sel_row[i];
        if (j < 0)
            continue;
        for (int64_t t = j * BS; t < (j + 1) * BS && t < ctx; ++t)
            pos[n++] = t;
    }
    return n;
}

/* A K or V cache as the attention reads it: bf16 elements, or E4M3 codes
 * with one fp32 scale per KV head, or per (physical block, KV head) when
 * per_block is set (element value = decode(code) * scale, exact in fp64). */
typedef struct {
    const uint16_t *bf16;
    const uint8_t *e4m3;
    const float *scale;
    int vt, Hkv, D, BS; /* vt: E4M3 codes in the V layout (vt_index) */
    int per_block;      /* scale[p * Hkv + kvh] instead of scale[kvh] */
} kvsrc;

/* element idx of the [NB][BS][Hkv][D] index space */
static double kv_val(const kvsrc *c, int64_t idx, int kvh)
{
    if (c->bf16)
        return bf16_val(c->bf16[idx]);
    const int64_t p = idx / ((int64_t)c->D * c->Hkv * c->BS);
    const double sc = (double)c->scale[c->per_block ? p * c->Hkv + kvh : kvh];
    if (c->vt) {
        const int64_t d = idx % c->D, o = (idx / ((int64_t)c->D * c->Hkv)) % c->BS;
        idx = vt_index(p, o, kvh, d, c->Hkv, c->D);
    }
    return oracle_e4m3_decode(c->e4m3[idx]) * sc;
}

/* Element index of K (or V) of sequence position t for one KV head through
 * the block table ([P2] 2.6: K_cache[physical_block][block_size][kv_head]
 * [head_dim], block_table[seq][logical_block] = physical_block); -1 if the
 * table entry is outside the pool. */
static int64_t kv_index(const int32_t *bt_row, int64_t t, int kvh, int Hkv, int D, int BS,
                        int64_t NB)
{
    const int64_t p = bt_row[t / BS];
    if (p < 0 || p >= NB)
        return -1;
    return ((p * BS + t % BS) * Hkv + kvh) * (int64_t)D;
}

/* scores s_i = scale * q . K[pos_i] for every listed position (fp64). */
static int compute_scores(double *s, const uint16_t *qrow, const kvsrc *K,
                          const int32_t *bt_row, const int64_t *pos, int64_t n,
                          int kvh, int Hkv, int D, int BS, int64_t NB, double scale)
{
    for (int64_t i = 0; i < n; ++i) {
        const int64_t k = kv_index(bt_row, pos[i], kvh, Hkv, D, BS, NB);
        if (k < 0)
            return -1;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += bf16_val(qrow[d]) * kv_val(K, k + d, kvh);
        s[i] = scale * dot;
    }
    return 0;
}

/* Reference form: explicit two-pass softmax over the listed tokens,
 *   m = max_i s_i, p_i = exp(s_i - m), l = sum p_i, out = sum p_i V_i / l.
 * An empty token list gives a zero output. */
static int attend_two_pass(double *out, const uint16_t *qrow, const kvsrc *K, const kvsrc *V,
                           const int32_t *bt_row, const int64_t *pos, int64_t n,
                           int kvh, int Hkv, int D, int BS, int64_t NB,
                           double scale, double *s)
{
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (n == 0)
        return 0;
    if (compute_scores(s, qrow, K, bt_row, pos, n, kvh, Hkv, D, BS, NB, scale))
        return -1;
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
        if (s[i] > m)
            m = s[i];
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double p = exp(s[i] - m);
        l += p;
        const int64_t v = kv_index(bt_row, pos[i], kvh, Hkv, D, BS, NB);
        for (int d = 0; d < D; ++d)
            out[d] += p * kv_val(V, v + d, kvh);
    }
    for (int d = 0; d < D; ++d)
        out[d] /= l;
    return 0;
}

/* Online softmax ([P1] "GQA Paged Attention"): one pass over the tokens in
 * chunks of `chunk`, keeping a running max m, normaliser l and accumulator acc;
 * when a chunk raises the max, the old l and acc are rescaled by
 * exp(m_old - m_new). The full score vector is not needed by the method (the
 * scores buffer here is only a convenience). */
static int attend_online(double *out, const uint16_t *qrow, const kvsrc *K, const kvsrc *V,
                         const int32_t *bt_row, const int64_t *pos, int64_t n,
                         int kvh, int Hkv, int D, int BS, int64_t NB,
                         double scale, int64_t chunk, double *s, double *acc)
{
    for (int d = 0; d < D; ++d) {
        out[d] = 0.0;
        acc[d] = 0.0;
    }
    if (n == 0)
        return 0;
    if (compute_scores(s, qrow, K, bt_row, pos, n, kvh, Hkv, D, BS, NB, scale))
        return -1;
    double m = -INFINITY, l = 0.0;
    for (int64_t c0 = 0; c0 < n; c0 += chunk) {
        const int64_t c1 = c0 + chunk < n ? c0 + chunk : n;
        double m_chunk = -INFINITY;
        for (int64_t i = c0; i < c1; ++i)
            if (s[i] > m_chunk)
                m_chunk = s[i];
        const double m_new = m_chunk > m ? m_chunk : m;
        const double alpha = exp(m - m_new);  /* exp(-inf) = 0 on the first chunk */
        l *= alpha;
        for (int d = 0; d < D; ++d)
            acc[d] *= alpha;
        for (int64_t i = c0; i < c1; ++i) {
            const double p = exp(s[i] - m_new);
            l += p;
            const int64_t v = kv_index(bt_row, pos[i], kvh, Hkv, D, BS, NB);
            for (int d = 0; d < D; ++d)
                acc[d] += p * kv_val(V, v + d, kvh);
        }
        m = m_new;
    }
    for (int d = 0; d < D; ++d)
        out[d] = acc[d] / l;
    return 0;
}

/* Split-KV ([P2] 4.1): the token list is cut into num_splits ranges with the
 * proportional boundaries n*s/num_splits; each range writes its normalised
 * output O_s and its log-sum-exp lse_s = m_s + log(l_s); the combine weights
 * each O_s by l_s relative to a common max:
 *   m* = max_s lse_s, w_s = exp(lse_s - m*), out = sum_s w_s O_s / sum_s w_s.
 * (The page prints out = sum l_s O_s / sum l_s, which is this formula when all
 * ranges share one max; rebasing to m* makes it hold for any maxima.) Empty
 * ranges carry no weight. */
static int attend_split(double *out, const uint16_t *qrow, const kvsrc *K, const kvsrc *V,
                        const int32_t *bt_row, const int64_t *pos, int64_t n,
                        int kvh, int Hkv, int D, int BS, int64_t NB,
                        double scale, int num_splits, double *s, double *part)
{
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (n == 0)
        return 0;
    double *lse = (double *)malloc(sizeof(double) * (size_t)num_splits);
    for (int sp = 0; sp < num_splits; ++sp) {
        const int64_t a = n * sp / num_splits, b = n * (sp + 1) / num_splits;
        lse[sp] = -INFINITY;
        if (b <= a)
            continue;
        if (attend_two_pass(part + (int64_t)sp * D, qrow, K, V, bt_row,
                            pos + a, b - a, kvh, Hkv, D, BS, NB, scale, s)) {
            free(lse);
            return -1;
        }
        double m = -INFINITY, l = 0.0;
        for (int64_t i = 0; i < b - a; ++i)
            if (s[i] > m)
                m = s[i];
        for (int64_t i = 0; i < b - a; ++i)
            l += exp(s[i] - m);
        lse[sp] = m + log(l);
    }
    double mstar = -INFINITY;
    for (int sp = 0; sp < num_splits; ++sp)
        if (lse[sp] > mstar)
            mstar = lse[sp];
    double wsum = 0.0;
    for (int sp = 0; sp < num_splits; ++sp) {
        if (lse[sp] == -INFINITY)
            continue;
        const double w = exp(lse[sp] - mstar);
        wsum += w;
        for (int d = 0; d < D; ++d)
            out[d] += w * part[(int64_t)sp * D + d];
    }
    for (int d = 0; d < D; ++d)
        out[d] /= wsum;
    free(lse);
    return 0;
}

/* mode: 0 = two-pass, 1 = online (chunk = param), 2 = split (num_splits = param) */
static int attention_rows(double *out, const uint16_t *q, const kvsrc *K, const kvsrc *V,
                          const int32_t *block_tables, int MBS,
                          const int32_t *context_lens, const int32_t *selected, int topk,
                          int B, int Hq, int Hkv, int D, int BS, int64_t NB, double scale,
                          const int32_t *rows, int64_t nrows, int mode, int64_t param)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || BS <= 0)
        return -2;
    const int G = Hq / Hkv;
    int64_t max_tokens = (int64_t)MBS * BS;
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(max_tokens + 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_tokens + 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)D * (size_t)(mode == 2 ? param + 1 : 1));
    int rc = 0;
    const int64_t total = rows ? nrows : (int64_t)B * Hq;
    for (int64_t r = 0; r < total && rc == 0; ++r) {
        const int64_t b = rows ? rows[2 * r] : r / Hq;
        const int64_t h = rows ? rows[2 * r + 1] : r % Hq;
        const int kvh = (int)(h / G);
        int64_t ctx = context_lens[b];
        if (ctx > max_tokens)
            ctx = max_tokens;
        const int32_t *sel_row = selected ? selected + (b * Hkv + kvh) * (int64_t)topk : NULL;
        const int64_t n = token_list(pos, ctx, BS, sel_row, topk);
        const uint16_t *qrow = q + (b * Hq + h) * (int64_t)D;
        const int32_t *bt_row = block_tables + b * (int64_t)MBS;
        double *o = out + r * (int64_t)D;
        if (mode == 0)
            rc = attend_two_pass(o, qrow, K, V, bt_row, pos, n, kvh, Hkv, D, BS, NB, scale, s);
        else if (mode == 1)
            rc = attend_online(o, qrow, K, V, bt_row, pos, n, kvh, Hkv, D, BS, NB, scale, param,
                               s, acc);
        else
            rc = attend_split(o, qrow, K, V, bt_row, pos, n, kvh, Hkv, D, BS, NB, scale,
                              (int)param, s, acc);
    }
    free(pos);
    free(s);
    free(acc);
    return rc;
}

/* Dense GQA paged decode attention ([P1] "GQA Paged Attention"): one query
 * token per sequence; out [B][Hq][D] (fp64), or only the (b, h) pairs listed
 * in rows[2*nrows] (out then [nrows][D]) when rows is not NULL.
 * Returns 0, -1 on a table entry outside the pool, -2 on bad sizes. */
int oracle_paged_attention(double *out, const uint16_t *q,
                           const uint16_t *key_cache, const uint16_t *value_cache,
                           const int32_t *block_tables, int MBS,
                           const int32_t *context_lens, int B, int Hq, int Hkv,
                           int D, int BS, int64_t NB, double scale,
                           const int32_t *rows, int64_t nrows)
{
    const kvsrc K = {key_cache, NULL, NULL, 0, 0, 0, 0, 0}, V = {value_cache, NULL, NULL, 0, 0, 0, 0, 0};
    return attention_rows(out, q, &K, &V, block_tables, MBS, context_lens,
                          NULL, 0, B, Hq, Hkv, D, BS, NB, scale, rows, nrows, 0, 0);
}

/* Same attention through the online-softmax recurrence, tokens taken `chunk`
 * at a time. */
int oracle_paged_attention_online(double *out, const uint16_t *q,
                                  const uint16_t *key_cache, const uint16_t *value_cache,
                                  const int32_t *block_tables, int MBS,
                                  const int32_t *context_lens, int B, int Hq, int Hkv,
                                  int D, int BS, int64_t NB, double scale, int64_t chunk)
{
    if (chunk <= 0)
        return -2;
    const kvsrc K = {key_cache, NULL, NULL, 0, 0, 0, 0, 0}, V = {value_cache, NULL, NULL, 0, 0, 0, 0, 0};
    return attention_rows(out, q, &K, &V, block_tables, MBS, context_lens,
                          NULL, 0, B, Hq, Hkv, D, BS, NB, scale, NULL, 0, 1, chunk);
}

/* Same attention through split-KV partials and their combine. */
int oracle_paged_attention_split(double *out, const uint16_t *q,
                                 const uint16_t *key_cache, const uint16_t *value_cache,
                                 const int32_t *block_tables, int MBS,
                                 const int32_t *context_lens, int B, int Hq, int Hkv,
                                 int D, int BS, int64_t NB, double scale, int num_splits)
{
    if (num_splits <= 0)
        return -2;
    const kvsrc K = {key_cache, NULL, NULL, 0, 0, 0, 0, 0}, V = {value_cache, NULL, NULL, 0, 0, 0, 0, 0};
    return attention_rows(out, q, &K, &V, block_tables, MBS, context_lens,
                          NULL, 0, B, Hq, Hkv, D, BS, NB, scale, NULL, 0, 2, num_splits);
}

/* Quest sparse paged attention ([P1] "Quest Sparse Attention", "Sparse
 * precision"): exact attention over only the tokens of the selected logical
 * blocks, selected[B][Hkv][topk] (shared by the GQA group of each KV head,
 * negative entries are padding), tokens past ctx skipped. */
int oracle_sparse_attention(double *out, const uint16_t *q,
                            const uint16_t *key_cache, const uint16_t *value_cache,
                            const int32_t *block_tables, int MBS,
                            const int32_t *context_lens, const int32_t *selected, int topk,
                            int B, int Hq, int Hkv, int D, int BS, int64_t NB, double scale,
                            const int32_t *rows, int64_t nrows)
{
    if (topk <= 0)
        return -2;
    const kvsrc K = {key_cache, NULL, NULL, 0, 0, 0, 0, 0}, V = {value_cache, NULL, NULL, 0, 0, 0, 0, 0};
    return attention_rows(out, q, &K, &V, block_tables, MBS, context_lens,
                          selected, topk, B, Hq, Hkv, D, BS, NB, scale, rows, nrows, 0, 0);
}

/* Attention over an E4M3 cache (dense when selected is NULL, else Quest
 * sparse): the same two-pass softmax in fp64 on the dequantised elements
 * decode(code) * scale[kvh] of K and V (V codes in the V layout). */
int oracle_attention_fp8(double *out, const uint16_t *q,
                         const uint8_t *key_cache, const uint8_t *value_cache,
                         const float *k_scale, const float *v_scale,
                         const int32_t *block_tables, int MBS,
                         const int32_t *context_lens, const int32_t *selected, int topk,
                         int B, int Hq, int Hkv, int D, int BS, int64_t NB, double scale,
                         const int32_t *rows, int64_t nrows)
{
    if ((selected && topk <= 0) || BS != 16)
        return -2;
    const kvsrc K = {NULL, key_cache, k_scale, 0, Hkv, D, BS, 0};
    const kvsrc V = {NULL, value_cache, v_scale, 1, Hkv, D, BS, 0};
    return attention_rows(out, q, &K, &V, block_tables, MBS, context_lens,
                          selected, selected ? topk : 0, B, Hq, Hkv, D, BS, NB, scale, rows,
                          nrows, 0, 0);
}

/* The same attention over an E4M3 cache with per-block scales: element value
 * decode(code) * k_bscale[p * Hkv + kvh] (V alike), p the token's physical
 * block. */
int oracle_attention_fp8_block(double *out, const uint16_t *q,
                               const uint8_t *key_cache, const uint8_t *value_cache,
                               const float *k_bscale, const float *v_bscale,
                               const int32_t *block_tables, int MBS,
                               const int32_t *context_lens, const int32_t *selected, int topk,
                               int B, int Hq, int Hkv, int D, int BS, int64_t NB, double scale,
                               const int32_t *rows, int64_t nrows)
{
    if ((selected && topk <= 0) || BS != 16)
        return -2;
    const kvsrc K = {NULL, key_cache, k_bscale, 0, Hkv, D, BS, 1};
    const kvsrc V = {NULL, value_cache, v_bscale, 1, Hkv, D, BS, 1};
    return attention_rows(out, q, &K, &V, block_tables, MBS, context_lens,
                          selected, selected ? topk : 0, B, Hq, Hkv, D, BS, NB, scale, rows,
                          nrows, 0, 0);
}

/* Multi-token query rows (chunked prefill or speculative tokens mixed into a
 * decode batch): sequence b owns query rows cu_seqlens_q[b] ..
 * cu_seqlens_q[b+1]-1, the newest q_len_b = cu[b+1] - cu[b] tokens of the
 * sequence, at positions ctx_b - q_len_b .. ctx_b - 1 (context_lens includes
 * them; the causal mask is right-aligned). Row i of sequence b attends to
 * positions t < ctx_b - q_len_b + i + 1, i.e. to itself and everything
 * before it; a row whose limit is <= 0 gets a zero output. q and out are
 * [total_q][Hq][D]; the attention per row is the two-pass softmax above.
 * rows (if not NULL) lists (row, head) pairs to compute; out is then
 * [nrows][D]. Returns 0, -1 on a table entry outside the pool, -2 on bad
 * sizes or a malformed cu_seqlens_q. */
int oracle_paged_attention_multi(double *out, const uint16_t *q,
                                 const uint16_t *key_cache, const uint16_t *value_cache,
                                 const int32_t *block_tables, int MBS,
                                 const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                 int B, int total_q, int Hq, int Hkv, int D, int BS, int64_t NB,
                                 double scale, const int32_t *rows, int64_t nrows)
{
    if (B <= 0 || total_q < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || BS <= 0)
        return -2;
    if (cu_seqlens_q[0] != 0 || cu_seqlens_q[B] != total_q)
        return -2;
    for (int b = 0; b < B; ++b)
        if (cu_seqlens_q[b + 1] < cu_seqlens_q[b])
            return -2;
    const int G = Hq / Hkv;
    const kvsrc K = {key_cache, NULL, NULL, 0, 0, 0, 0, 0}, V = {value_cache, NULL, NULL, 0, 0, 0, 0, 0};
    const int64_t max_tokens = (int64_t)MBS * BS;
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(max_tokens + 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_tokens + 1));
    int rc = 0;
    const int64_t total = rows ? nrows : (int64_t)total_q * Hq;
    for (int64_t r = 0; r < total && rc == 0; ++r) {
        const int64_t row = rows ? rows[2 * r] : r / Hq;
        const int64_t h = rows ? rows[2 * r + 1] : r % Hq;
        int b = 0;
        while (cu_seqlens_q[b + 1] <= row)
            ++b;
        int64_t ctx = context_lens[b];
        if (ctx > max_tokens)
            ctx = max_tokens;
        if (ctx < 0)
            ctx = 0;
        const int64_t q_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        int64_t lim = ctx - q_len + (row - cu_seqlens_q[b]) + 1;
        if (lim < 0)
            lim = 0;
        const int64_t n = token_list(pos, lim, BS, NULL, 0);
        rc = attend_two_pass(out + r * (int64_t)D, q + (row * Hq + h) * (int64_t)D, &K, &V,
                             block_tables + (int64_t)b * MBS, pos, n, (int)(h / G), Hkv, D, BS, NB,
                             scale, s);
    }
    free(pos);
    free(s);
    return rc;
}

/* ------------------------------------------------ Quest score, plain form */

/* metadata element as fp32: bf16, or an E4M3 code (decoded exactly) */
static float meta_f32(const uint16_t *m16, const uint8_t *m8, int64_t idx)
{
    return m16 ? bf16_f32(m16[idx]) : (float)oracle_e4m3_decode(m8[idx]);
}

/* Quest block score as the method states it ([P1] "Quest Sparse Attention":
 * a cheap upper-bound score per logical block; the bound itself is fixed by
 * the statement of the method), written out term by term:
 *
 *   score(b, kvh, j) = sum_{h in group(kvh)} sum_{d < D}
 *                      max(q[b,h,d] * min[p,kvh,d], q[b,h,d] * max[p,kvh,d])
 *
 * with p = block_tables[b][j] and group(kvh) = {kvh*G, ..., kvh*G + G-1}.
 * Arithmetic is fp64: every product of two bf16 (or E4M3) values is exact in
 * fp64, and the G*D additions are done in the order written (h ascending,
 * then d ascending), each rounded once at 2^-53 relative.
 *
 * abs_sum (if not NULL) receives A = sum_h sum_d |q[b,h,d]| *
 * max(|min_d|, |max_d|): every term of the sum above is at most its share of
 * A in magnitude, so A scales the rounding error of any floating-point
 * evaluation of the score.
 *
 * Logical blocks j >= ceil(ctx/BS) and table entries outside the pool score
 * -inf (abs_sum 0). scores, abs_sum: [B][Hkv][MBS] fp64. */
static int quest_scores_plain_impl(double *scores, double *abs_sum, const uint16_t *q,
                                   const uint16_t *kmin, const uint16_t *kmax,
                                   const uint8_t *kmin8, const uint8_t *kmax8,
                                   const float *k_bscale,
                                   const int32_t *block_tables, int MBS,
                                   const int32_t *context_lens, int B, int Hq, int Hkv,
                                   int D, int BS, int64_t NB)
{
    if (Hq % Hkv != 0)
        return -2;
    const int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        const int64_t ctx = context_lens[b] > 0 ? context_lens[b] : 0;
        const int64_t nblk = (ctx + BS - 1) / BS;
        for (int kvh = 0; kvh < Hkv; ++kvh) {
            for (int64_t j = 0; j < MBS; ++j) {
                const int64_t o = ((int64_t)b * Hkv + kvh) * MBS + j;
                const int64_t p = j < nblk ? block_tables[(int64_t)b * MBS + j] : -1;
                if (p < 0 || p >= NB) {
                    scores[o] = -INFINITY;
                    if (abs_sum)
                        abs_sum[o] = 0.0;
                    continue;
                }
                const int64_t base = (p * Hkv + kvh) * (int64_t)D;
                double s = 0.0, a = 0.0;
                for (int g = 0; g < G; ++g) {
                    const int64_t h = (int64_t)kvh * G + g;
                    const uint16_t *qrow = q + ((int64_t)b * Hq + h) * D;
                    for (int d = 0; d < D; ++d) {
                        const double qv = bf16_val(qrow[d]);
                        const double lo = (double)meta_f32(kmin, kmin8, base + d);
                        const double hi = (double)meta_f32(kmax, kmax8, base + d);
                        const double x = qv * lo, y = qv * hi;
                        s += x > y ? x : y;
                        const double m = fabs(lo) > fabs(hi) ? fabs(lo) : fabs(hi);
                        a += fabs(qv) * m;
                    }
                }
                if (k_bscale) { /* per-block K scale: min, max and the score scale with it */
                    s *= (double)k_bscale[p * Hkv + kvh];
                    a *= (double)k_bscale[p * Hkv + kvh];
                }
                scores[o] = s;
                if (abs_sum)
                    abs_sum[o] = a;
            }
        }
    }
    return 0;
}

int oracle_quest_scores_plain(double *scores, double *abs_sum, const uint16_t *q,
                              const uint16_t *kmin, const uint16_t *kmax,
                              const int32_t *block_tables, int MBS,
                              const int32_t *context_lens, int B, int Hq, int Hkv,
                              int D, int BS, int64_t NB)
{
    return quest_scores_plain_impl(scores, abs_sum, q, kmin, kmax, NULL, NULL, NULL, block_tables, MBS,
                                   context_lens, B, Hq, Hkv, D, BS, NB);
}

/* The same plain score over E4M3 metadata (min_d, max_d = the decoded codes;
 * the cache's per-KV-head K scale is a positive factor of a whole row and is
 * left out, as it cannot change that row's top-K). */
int oracle_quest_scores_plain_fp8(double *scores, double *abs_sum, const uint16_t *q,
                                  const uint8_t *kmin, const uint8_t *kmax,
                                  const int32_t *block_tables, int MBS,
                                  const int32_t *context_lens, int B, int Hq, int Hkv,
                                  int D, int BS, int64_t NB)
{
    return quest_scores_plain_impl(scores, abs_sum, q, NULL, NULL, kmin, kmax, NULL, block_tables, MBS,
                                   context_lens, B, Hq, Hkv, D, BS, NB);
}

/* The plain score over E4M3 metadata of a cache with per-block scales: the
 * block's metadata stand for decode(code) * k_bscale[p * Hkv + kvh], so the
 * block's score (and abs_sum) carry that factor, which differs from block to
 * block. */
int oracle_quest_scores_plain_fp8_block(double *scores, double *abs_sum, const uint16_t *q,
                                        const uint8_t *kmin, const uint8_t *kmax,
                                        const float *k_bscale,
                                        const int32_t *block_tables, int MBS,
                                        const int32_t *context_lens, int B, int Hq, int Hkv,
                                        int D, int BS, int64_t NB)
{
    return quest_scores_plain_impl(scores, abs_sum, q, NULL, NULL, kmin, kmax, k_bscale, block_tables,
                                   MBS, context_lens, B, Hq, Hkv, D, BS, NB);
}

/* --------------------------------- Quest score, fp32 kernel-order reproduction */

/* The same block score evaluated in fp32 in the one fixed order the GPU
 * kernel uses. It serves as a bit-exact check of the kernel's arithmetic;
 * agreement with the method's definition is checked against the plain form
 * above (the selected sets must match it except where the fp32 rounding
 * error bound covers the score gap at the K-th place).
 *
 * Definition: score(b, kvh, j) = sum_{h in group(kvh)} sum_d
 *                                max(q[b,h,d]*min_d, q[b,h,d]*max_d)
 * with min/max the metadata of physical block p = block_tables[b][j].
 * Since max >= min, max(q*min, q*max) = q+ * max + q- * min with
 * q+ = max(q, 0) and q- = min(q, 0); summing over the group first:
 *     score = sum_d ( P_d * max_d + N_d * min_d ),
 *     P_d = sum_h q+[h,d],  N_d = sum_h q-[h,d].
 * fp32 evaluation order:
 *   1. P_d, N_d: start at +0, add h = 0, 1, ..., G-1 in turn;
 *   2. t_d = fl(fl(P_d * max_d) + fl(N_d * min_d));
 *   3. D is cut into 32 equal chunks of C = D/32 consecutive d; chunk sum
 *      c_l = (((t_{lC} + t_{lC+1}) + ...) + t_{lC+C-1}), left to right;
 *   4. the 32 chunk sums are combined pairwise: for off = 16, 8, 4, 2, 1:
 *      c_l <- c_l + c_{l xor off}; the score is c_0;
 *   5. (E4M3 cache with per-block scales only) fl(c_0 * k_bscale[p, kvh]).
 * Logical blocks j >= ceil(ctx/BS) are excluded (score -inf). A table entry
 * outside the pool also scores -inf.
 * scores: [B][Hkv][MBS] fp32. Requires D % 32 == 0. */
static int quest_scores_impl(float *scores, const uint16_t *q,
                             const uint16_t *kmin, const uint16_t *kmax,
                             const uint8_t *kmin8, const uint8_t *kmax8,
                             const float *k_bscale,
                             const int32_t *block_tables, int MBS,
                             const int32_t *context_lens, int B, int Hq, int Hkv,
                             int D, int BS, int64_t NB)
{
    if (Hq % Hkv != 0 || D % 32 != 0)
        return -2;
    const int G = Hq / Hkv, C = D / 32;
    float *P = (float *)malloc(sizeof(float) * (size_t)D);
    float *N = (float *)malloc(sizeof(float) * (size_t)D);
    float c[32];
    for (int b = 0; b < B; ++b) {
        const int64_t ctx = context_lens[b] > 0 ? context_lens[b] : 0;
        const int64_t nblk = (ctx + BS - 1) / BS;
        for (int kvh = 0; kvh < Hkv; ++kvh) {
            for (int d = 0; d < D; ++d) {
                float pp = 0.0f, nn = 0.0f;
                for (int g = 0; g < G; ++g) {
                    const float v = bf16_f32(q[((int64_t)b * Hq + (int64_t)kvh * G + g) * D + d]);
                    pp = pp + (v > 0.0f ? v : 0.0f);
                    nn = nn + (v < 0.0f ? v : 0.0f);
                }
                P[d] = pp;
                N[d] = nn;
            }
            float *srow = scores + ((int64_t)b * Hkv + kvh) * MBS;
            for (int64_t j = 0; j < MBS; ++j) {
                if (j >= nblk) {
                    srow[j] = -INFINITY;
                    continue;
                }
                const int64_t p = block_tables[(int64_t)b * MBS + j];
                if (p < 0 || p >= NB) {
                    srow[j] = -INFINITY;
                    continue;
                }
                const int64_t base = (p * Hkv + kvh) * (int64_t)D;
                for (int l = 0; l < 32; ++l) {
                    float acc = 0.0f;
                    for (int i = 0; i < C; ++i) {
                        const int d = l * C + i;
                        const float a = P[d] * meta_f32(kmax, kmax8, base + d);
                        const float bb = N[d] * meta_f32(kmin, kmin8, base + d);
                        const float t = a + bb;
                        acc = (i == 0) ? t : acc + t;
                    }
                    c[l] = acc;
                }
                for (int off = 16; off >= 1; off >>= 1) {
                    float nc[32];
                    for (int l = 0; l < 32; ++l)
                        nc[l] = c[l] + c[l ^ off];
                    memcpy(c, nc, sizeof c);
                }
                /* 5. per-block K scale (E4M3 cache with block scales): one
                 * fp32 product, exact for a power of two */
                srow[j] = k_bscale ? c[0] * k_bscale[p * Hkv + kvh] : c[0];
            }
        }
    }
    free(P);
    free(N);
    return 0;
}

int oracle_quest_scores_kernel_order(float *scores, const uint16_t *q,
                        const uint16_t *kmin, const uint16_t *kmax,
                        const int32_t *block_tables, int MBS,
                        const int32_t *context_lens, int B, int Hq, int Hkv,
                        int D, int BS, int64_t NB)
{
    return quest_scores_impl(scores, q, kmin, kmax, NULL, NULL, NULL, block_tables, MBS,
                             context_lens, B, Hq, Hkv, D, BS, NB);
}

/* The same score on E4M3 metadata: min_d and max_d are the decoded codes
 * (exact in fp32), every other step as above. The cache's per-KV-head scale
 * is left out: it multiplies every score of a (sequence, KV head) row by the
 * same positive factor and cannot change that row's top-K. */
int oracle_quest_scores_kernel_order_fp8(float *scores, const uint16_t *q,
                            const uint8_t *kmin, const uint8_t *kmax,
                            const int32_t *block_tables, int MBS,
                            const int32_t *context_lens, int B, int Hq, int Hkv,
                            int D, int BS, int64_t NB)
{
    return quest_scores_impl(scores, q, NULL, NULL, kmin, kmax, NULL, block_tables, MBS,
                             context_lens, B, Hq, Hkv, D, BS, NB);
}

/* The kernel-order score of a cache with per-block scales: the sum above,
 * then one fp32 product with the block's K scale (step 5). */
int oracle_quest_scores_kernel_order_fp8_block(float *scores, const uint16_t *q,
                                               const uint8_t *kmin, const uint8_t *kmax,
                                               const float *k_bscale,
                                               const int32_t *block_tables, int MBS,
                                               const int32_t *context_lens, int B, int Hq,
                                               int Hkv, int D, int BS, int64_t NB)
{
    return quest_scores_impl(scores, q, NULL, NULL, kmin, kmax, k_bscale, block_tables, MBS,
                             context_lens, B, Hq, Hkv, D, BS, NB);
}

/* ------------------------------------------------------------ Quest top-K */

typedef struct {
    uint64_t key; /* totalOrder key of the score (fp32 keys zero-extended) */
    int32_t j;
} ranked_block;

static int rank_cmp(const void *a, const void *b)
{
    const ranked_block *x = (const ranked_block *)a, *y = (const ranked_block *)b;
    if (x->key != y->key)
        return x->key > y->key ? -1 : 1; /* higher score first */
    return x->j < y->j ? -1 : (x->j > y->j); /* tie: lower block index first */
}

static int index_cmp(const void *a, const void *b)
{
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return x < y ? -1 : (x > y);
}

/* Top-K per (sequence, KV head) ([P1] "Quest Sparse Attention": pick the
 * top-K logical blocks; ties go to the lower block index). Candidates are the
 * logical blocks j < ceil(ctx/BS); they are fully sorted by (score desc,
 * j asc) with scores ranked by IEEE totalOrder; the first min(topk, nblk) are
 * returned in ascending block order and the row is padded with -1.
 * Scores are fp32 (s32) or fp64 (s64), whichever is not NULL.
 * selected: [B][Hkv][topk] int32. */
static int quest_topk_impl(int32_t *selected, const float *s32, const double *s64, int MBS,
                           const int32_t *context_lens, int B, int Hkv, int BS, int topk)
{
    if (topk <= 0)
        return -2;
    ranked_block *items = (ranked_block *)malloc(sizeof(ranked_block) * (size_t)(MBS + 1));
    for (int b = 0; b < B; ++b) {
        const int64_t ctx = context_lens[b] > 0 ? context_lens[b] : 0;
        int64_t nblk = (ctx + BS - 1) / BS;
        if (nblk > MBS)
            nblk = MBS;
        for (int kvh = 0; kvh < Hkv; ++kvh) {
            const int64_t row = ((int64_t)b * Hkv + kvh) * MBS;
            for (int64_t j = 0; j < nblk; ++j) {
                items[j].key = s32 ? (uint64_t)f32_order_key(s32[row + j]) : f64_order_key(s64[row + j]);
                items[j].j = (int32_t)j;
            }
            qsort(items, (size_t)nblk, sizeof(ranked_block), rank_cmp);
            const int64_t k = nblk < topk ? nblk : topk;
            int32_t *out = selected + ((int64_t)b * Hkv + kvh) * topk;
            for (int64_t i = 0; i < k; ++i)
                out[i] = items[i].j;
            qsort(out, (size_t)k, sizeof(int32_t), index_cmp);
            for (int64_t i = k; i < topk; ++i)
                out[i] = -1;
        }
    }
    free(items);
    return 0;
}

int oracle_quest_topk(int32_t *selected, const float *scores, int MBS,
                      const int32_t *context_lens, int B, int Hkv, int BS, int topk)
{
    return quest_topk_impl(selected, scores, NULL, MBS, context_lens, B, Hkv, BS, topk);
}

/* The same selection over fp64 scores (the plain form of the score). */
int oracle_quest_topk_f64(int32_t *selected, const double *scores, int MBS,
                          const int32_t *context_lens, int B, int Hkv, int BS, int topk)
{
    return quest_topk_impl(selected, NULL, scores, MBS, context_lens, B, Hkv, BS, topk);
}
