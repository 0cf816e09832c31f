/*
 * rar_oracle.c -- plain, slow CPU oracle for the ring all-reduce.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  It shares no code
 * with the CUDA library.  Every function says which passage of the source
 * pages it restates; rar_oracle.h lists the pages.
 *
 * Readings taken where the pages leave a step open:
 *   - hop arithmetic is in the buffer's dtype, rounded after every hop with
 *     IEEE round-to-nearest-even, subnormals kept, overflow to +-inf; int32
 *     wraps modulo 2^32;
 *   - max keeps the running value unless the receiver's own element is
 *     strictly greater (so the first value seen wins a +-0 tie);
 *   - avg is the ring-order sum times 1/p, with 1/p the fp32 value nearest
 *     to it, applied once by the chunk's owner after the last reduce-scatter
 *     step, the product rounded once to fp32 and then to a 16-bit dtype.
 */
#include "rar_oracle.h"

#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- partition */

/* "Ring All-Reduce, in depth", section "An implementation": chunk_bounds.
 * base = n div p, extra = n mod p, start_i = i * base + min(i, extra), so
 * the first `extra` chunks are one element longer. */
void orc_chunk_bounds(int64_t n, int p, int64_t *starts)
{
    int64_t base = n / p;
    int64_t extra = n % p;
    for (int i = 0; i <= p; i++) {
        int64_t bonus = (i < extra) ? i : extra;
        starts[i] = (int64_t)i * base + bonus;
    }
}

int orc_elem_size(int dtype)
{
    switch (dtype) {
    case ORC_I32: return 4;
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_F16: return 2;
    default: return 0;
    }
}

/* ------------------------------------------------- IEEE 754 conversions */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bfloat16 is the top half of a binary32: widening is exact. */
float orc_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Narrowing binary32 -> bfloat16, round to nearest, ties to even: the 16
 * dropped bits are compared against one half of the kept unit in the last
 * place.  A carry out of the significand moves into the exponent, which is
 * exactly the next representable value (and +-inf past the largest finite
 * one).  NaN stays a (quiet) NaN. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

static int bit_length(uint64_t v)
{
    int b = 0;
    while (v) { b++; v >>= 1; }
    return b;
}

/* binary16 -> binary32 is exact. */
float orc_f16_to_f32(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t e = ((uint32_t)h >> 10) & 0x1Fu;
    uint32_t m = (uint32_t)h & 0x3FFu;
    if (e == 0x1Fu)
        return bits_f32(sign | 0x7F800000u | (m << 13));
    if (e == 0) {
        /* subnormal: m * 2^-24, exact in binary32 */
        float v = (float)m;
        for (int k = 0; k < 24; k++) v *= 0.5f;
        return sign ? -v : v;
    }
    return bits_f32(sign | ((e - 15u + 127u) << 23) | (m << 13));
}

/* binary32 -> binary16, round to nearest, ties to even.  The binary32 value
 * is sig * 2^e2 with an integer sig; the binary16 quantum at that magnitude
 * is 2^q with q = max(floor(log2 |v|), -14) - 10; the result is
 * round(sig * 2^(e2 - q)) * 2^q, renormalised if rounding carried, +-inf
 * above the largest finite value, and subnormal below 2^-14. */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t exp = (u >> 23) & 0xFFu;
    uint32_t man = u & 0x7FFFFFu;
    if (exp == 0xFFu)
        return (uint16_t)(sign | (man ? 0x7E00u : 0x7C00u));
    uint64_t sig;
    int e2;
    if (exp == 0) { sig = man; e2 = -149; }
    else { sig = man | 0x800000u; e2 = (int)exp - 150; }
    if (sig == 0)
        return sign;
    int lg = bit_length(sig) - 1 + e2;      /* floor(log2 |v|) */
    int q = (lg > -14 ? lg : -14) - 10;     /* quantum exponent */
    int sh = q - e2;                        /* low bits of sig to drop */
    uint64_t M;
    if (sh <= 0) {
        M = sig << (-sh);
    } else if (sh >= 63) {
        M = 0;                              /* below half the smallest quantum */
    } else {
        uint64_t kept = sig >> sh;
        uint64_t rem = sig & ((1ull << sh) - 1ull);
        uint64_t half = 1ull << (sh - 1);
        if (rem > half || (rem == half && (kept & 1ull)))
            kept += 1ull;
        M = kept;
    }
    while (M >= 2048u) { M >>= 1; q += 1; }  /* rounding carried a binade */
    if (q > 5)
        return (uint16_t)(sign | 0x7C00u);   /* beyond 65504: infinity */
    if (M < 1024u)
        return (uint16_t)(sign | (uint16_t)M);   /* subnormal, q == -24 */
    return (uint16_t)(sign | (uint16_t)((q + 10 + 15) << 10) | (uint16_t)(M - 1024u));
}

/* ------------------------------------------------------------------ one hop */

static float load_float(int dtype, const void *p)
{
    if (dtype == ORC_F32) { float f; memcpy(&f, p, 4); return f; }
    uint16_t h; memcpy(&h, p, 2);
    return dtype == ORC_BF16 ? orc_bf16_to_f32(h) : orc_f16_to_f32(h);
}

static void store_float(int dtype, void *p, float v)
{
    if (dtype == ORC_F32) { memcpy(p, &v, 4); return; }
    uint16_t h = dtype == ORC_BF16 ? orc_f32_to_bf16(v) : orc_f32_to_f16(v);
    memcpy(p, &h, 2);
}

/* One reduce-scatter hop ("Ring All-Reduce, in depth", "The schedule": the
 * receiver adds the incoming chunk into its own copy).  For the 16-bit types
 * the sum is taken in binary32 and rounded once: binary32 has at least
 * 2 * 11 + 2 significand bits, so that double rounding equals the correctly
 * rounded 16-bit sum (Figueroa, "When is double rounding innocuous?", 1995). */
void orc_combine(int dtype, int op, const void *acc, const void *own, void *out)
{
    int es = orc_elem_size(dtype);
    if (dtype == ORC_I32) {
        uint32_t a, b, r;
        memcpy(&a, acc, 4);
        memcpy(&b, own, 4);
        if (op == ORC_MAX) {
            int32_t sa, sb;
            memcpy(&sa, acc, 4);
            memcpy(&sb, own, 4);
            r = (sb > sa) ? b : a;
        } else {
            r = a + b;   /* two's complement wrap */
        }
        memcpy(out, &r, 4);
        return;
    }
    float a = load_float(dtype, acc);
    float b = load_float(dtype, own);
    if (op == ORC_MAX) {
        /* keep the exact bits of the winner, so -0 and +0 stay apart */
        unsigned char winner[4];
        memcpy(winner, (b > a) ? own : acc, (size_t)es);
        memcpy(out, winner, (size_t)es);
        return;
    }
    store_float(dtype, out, a + b);
}

/* avg epilogue at the owner: x * (1/p), 1/p rounded to binary32. */
static void scale_by_inv_p(int dtype, void *elem, int p)
{
    float inv_p = 1.0f / (float)p;
    float v = load_float(dtype, elem);
    float r = v * inv_p;
    store_float(dtype, elem, r);
}

static int valid_kind(int dtype, int op)
{
    if (orc_elem_size(dtype) == 0) return 0;
    if (op != ORC_SUM && op != ORC_MAX && op != ORC_AVG && op != ORC_AVG_PREDIV) return 0;
    if ((op == ORC_AVG || op == ORC_AVG_PREDIV) && dtype == ORC_I32) return 0;
    return 1;
}

/* The op a hop applies: both averages add. */
static int hop_of(int op)
{
    return (op == ORC_AVG || op == ORC_AVG_PREDIV) ? ORC_SUM : op;
}

static int mod_p(int64_t v, int p)
{
    int64_t r = v % p;
    return (int)(r < 0 ? r + p : r);
}

/* ------------------------------------------------------------- simulator */

/* "Ring All-Reduce, in depth", sections "The schedule" and "An
 * implementation".  Each step first copies every rank's outgoing chunk
 * (the sends happen at once), then delivers each copy to its receiver,
 * which combines it into its own chunk (reduce-scatter) or overwrites its
 * chunk with it (all-gather).  The mirrored ring (the opposite direction of
 * "Bidirectional rings") sends to r - 1 and walks the chunk indices the
 * other way: reduce-scatter step s sends chunk (r + s), all-gather step s
 * sends chunk (r - 1 + s), and the owner of chunk c is rank c + 1. */
int orc_ring_simulate(void *const *bufs, int p, int64_t n, int dtype, int op,
                      int direction, int first_step, int n_steps,
                      int64_t *sends)
{
    if (p < 1 || n < 0 || !valid_kind(dtype, op)) return -1;
    if (direction != ORC_FORWARD && direction != ORC_MIRRORED) return -1;
    if (first_step < 0 || n_steps < 0) return -1;
    if (p == 1 || n == 0 || n_steps == 0) return 0;
    if (first_step + n_steps > 2 * (p - 1)) return -1;
    for (int r = 0; r < p; r++)
        if (!bufs[r]) return -1;

    int es = orc_elem_size(dtype);
    int64_t *starts = (int64_t *)malloc(sizeof(int64_t) * (size_t)(p + 1));
    int *msg_chunk = (int *)malloc(sizeof(int) * (size_t)p);
    if (!starts || !msg_chunk) { free(starts); free(msg_chunk); return -1; }
    orc_chunk_bounds(n, p, starts);
    int64_t maxlen = 0;
    for (int c = 0; c < p; c++)
        if (starts[c + 1] - starts[c] > maxlen) maxlen = starts[c + 1] - starts[c];
    unsigned char *msg = (unsigned char *)malloc((size_t)p * (size_t)(maxlen > 0 ? maxlen : 1) * (size_t)es);
    if (!msg) { free(starts); free(msg_chunk); return -1; }

    int hop_op = hop_of(op);
    /* pre-divide: each rank scales its own contribution before the ring */
    if (op == ORC_AVG_PREDIV && first_step == 0) {
        for (int r = 0; r < p; r++)
            for (int64_t i = 0; i < n; i++)
                scale_by_inv_p(dtype, (unsigned char *)bufs[r] + (size_t)i * (size_t)es, p);
    }
    for (int step = first_step; step < first_step + n_steps; step++) {
        int reduce = step < p - 1;
        int s = reduce ? step : step - (p - 1);
        /* every rank puts its outgoing chunk on the wire */
        for (int r = 0; r < p; r++) {
            int c;
            if (direction == ORC_FORWARD)
                c = reduce ? mod_p(r - s, p) : mod_p(r + 1 - s, p);
            else
                c = reduce ? mod_p(r + s, p) : mod_p(r - 1 + s, p);
            int64_t len = starts[c + 1] - starts[c];
            msg_chunk[r] = c;
            memcpy(msg + (size_t)r * (size_t)maxlen * (size_t)es,
                   (unsigned char *)bufs[r] + (size_t)starts[c] * (size_t)es,
                   (size_t)len * (size_t)es);
            if (sends) sends[r] += len;
        }
        /* every receiver takes its message */
        for (int r = 0; r < p; r++) {
            int dst = direction == ORC_FORWARD ? mod_p(r + 1, p) : mod_p(r - 1, p);
            int c = msg_chunk[r];
            int64_t len = starts[c + 1] - starts[c];
            unsigned char *in = msg + (size_t)r * (size_t)maxlen * (size_t)es;
            unsigned char *mine = (unsigned char *)bufs[dst] + (size_t)starts[c] * (size_t)es;
            if (reduce) {
                for (int64_t i = 0; i < len; i++) {
                    void *e = mine + (size_t)i * (size_t)es;
                    orc_combine(dtype, hop_op, in + (size_t)i * (size_t)es, e, e);
                }
            } else {
                memcpy(mine, in, (size_t)len * (size_t)es);
            }
        }
        /* after the last reduce-scatter step each rank owns one finished
         * chunk; avg scales it there, before the all-gather copies it */
        if (reduce && s == p - 2 && op == ORC_AVG) {
            for (int r = 0; r < p; r++) {
                int c = direction == ORC_FORWARD ? mod_p(r + 1, p) : mod_p(r - 1, p);
                for (int64_t i = starts[c]; i < starts[c + 1]; i++)
                    scale_by_inv_p(dtype, (unsigned char *)bufs[r] + (size_t)i * (size_t)es, p);
            }
        }
    }
    free(msg);
    free(msg_chunk);
    free(starts);
    return 0;
}

/* "Ring All-Reduce, in depth", "What real libraries add", "Bidirectional
 * rings": the first half of the buffer (chunk_bounds(n, 2)) runs the forward
 * ring, the second half the mirrored ring. */
int orc_ring_simulate_bidir(void *const *bufs, int p, int64_t n, int dtype,
                            int op, int rs_only, int64_t *sends)
{
    if (p < 1 || n < 0 || !valid_kind(dtype, op)) return -1;
    if (p == 1 || n == 0) return 0;
    int es = orc_elem_size(dtype);
    int64_t halves[3];
    orc_chunk_bounds(n, 2, halves);
    void **second = (void **)malloc(sizeof(void *) * (size_t)p);
    if (!second) return -1;
    for (int r = 0; r < p; r++)
        second[r] = (unsigned char *)bufs[r] + (size_t)halves[1] * (size_t)es;
    int steps = rs_only ? p - 1 : 2 * (p - 1);
    int rc = orc_ring_simulate(bufs, p, halves[1], dtype, op, ORC_FORWARD, 0, steps, sends);
    if (rc == 0)
        rc = orc_ring_simulate(second, p, n - halves[1], dtype, op, ORC_MIRRORED, 0, steps, sends);
    free(second);
    return rc;
}

/* ----------------------------------------------------- per-element folds */

static int chunk_of(const int64_t *starts, int p, int64_t i)
{
    for (int c = 0; c < p; c++)
        if (starts[c] <= i && i < starts[c + 1]) return c;
    return -1;
}

/* Level-by-level pairwise fold over the rank index (tree order), in place
 * over `vals` (cnt elements of size es). */
static void tree_levels(int dtype, int hop_op, unsigned char *vals, int cnt)
{
    int es = orc_elem_size(dtype);
    while (cnt > 1) {
        int half = cnt / 2;
        for (int k = 0; k < half; k++)
            orc_combine(dtype, hop_op, vals + (size_t)(2 * k) * (size_t)es,
                        vals + (size_t)(2 * k + 1) * (size_t)es,
                        vals + (size_t)k * (size_t)es);
        if (cnt & 1)
            memmove(vals + (size_t)half * (size_t)es, vals + (size_t)(cnt - 1) * (size_t)es, (size_t)es);
        cnt = half + (cnt & 1);
    }
}

/* The value the ring leaves at index i, read off the schedule: chunk c starts
 * at rank c (reduce-scatter step 0 sends chunk r from rank r), and each hop
 * adds the next receiver's own element -- x_c, then x_(c+1), ..., then
 * x_(c+p-1) for the forward ring; x_c, x_(c-1), ... for the mirrored one. */
int orc_fold_sampled(const void *vals, const int64_t *idx, int64_t m, int p,
                     int64_t n, int dtype, int op, int mode, void *out)
{
    if (p < 1 || n < 0 || m < 0 || !valid_kind(dtype, op)) return -1;
    if (mode < 0 || mode > 2) return -1;
    int es = orc_elem_size(dtype);
    const unsigned char *v = (const unsigned char *)vals;
    unsigned char *o = (unsigned char *)out;
    int64_t halves[3];
    orc_chunk_bounds(n, 2, halves);
    int64_t *fwd = (int64_t *)malloc(sizeof(int64_t) * (size_t)(p + 1));
    int64_t *mir = (int64_t *)malloc(sizeof(int64_t) * (size_t)(p + 1));
    unsigned char *tmp = (unsigned char *)malloc((size_t)p * (size_t)es);
    if (!fwd || !mir || !tmp) { free(fwd); free(mir); free(tmp); return -1; }
    if (mode == 1) {
        orc_chunk_bounds(halves[1], p, fwd);
        orc_chunk_bounds(n - halves[1], p, mir);
    } else {
        orc_chunk_bounds(n, p, fwd);
    }
    int hop_op = hop_of(op);
    int rc = 0;
    for (int64_t j = 0; j < m; j++) {
        int64_t i = idx[j];
        if (i < 0 || i >= n) { rc = -1; break; }
        unsigned char acc[4];
        /* rank r's contribution at this index (pre-divided if asked) */
        for (int r = 0; r < p; r++) {
            memcpy(tmp + (size_t)r * (size_t)es, v + ((size_t)r * (size_t)m + (size_t)j) * (size_t)es, (size_t)es);
            if (op == ORC_AVG_PREDIV)
                scale_by_inv_p(dtype, tmp + (size_t)r * (size_t)es, p);
        }
        if (mode == 2) {
            tree_levels(dtype, hop_op, tmp, p);
            memcpy(acc, tmp, (size_t)es);
        } else {
            int c, dir;
            if (mode == 1 && i >= halves[1]) {
                c = chunk_of(mir, p, i - halves[1]);
                dir = -1;
            } else {
                c = chunk_of(fwd, p, i);
                dir = +1;
            }
            memcpy(acc, tmp + (size_t)c * (size_t)es, (size_t)es);
            for (int k = 1; k < p; k++) {
                int r = mod_p((int64_t)c + (int64_t)dir * k, p);
                orc_combine(dtype, hop_op, acc, tmp + (size_t)r * (size_t)es, acc);
            }
        }
        if (op == ORC_AVG)
            scale_by_inv_p(dtype, acc, p);
        memcpy(o + (size_t)j * (size_t)es, acc, (size_t)es);
    }
    free(fwd);
    free(mir);
    free(tmp);
    return rc;
}

/* Tree order over whole buffers; every rank ends with the result. */
int orc_tree_fold(void *const *bufs, int p, int64_t n, int dtype, int op)
{
    if (p < 1 || n < 0 || !valid_kind(dtype, op)) return -1;
    int es = orc_elem_size(dtype);
    unsigned char *tmp = (unsigned char *)malloc((size_t)p * (size_t)es);
    if (!tmp) return -1;
    int hop_op = hop_of(op);
    for (int64_t i = 0; i < n; i++) {
        for (int r = 0; r < p; r++) {
            memcpy(tmp + (size_t)r * (size_t)es, (unsigned char *)bufs[r] + (size_t)i * (size_t)es, (size_t)es);
            if (op == ORC_AVG_PREDIV)
                scale_by_inv_p(dtype, tmp + (size_t)r * (size_t)es, p);
        }
        tree_levels(dtype, hop_op, tmp, p);
        if (op == ORC_AVG)
            scale_by_inv_p(dtype, tmp, p);
        for (int r = 0; r < p; r++)
            memcpy((unsigned char *)bufs[r] + (size_t)i * (size_t)es, tmp, (size_t)es);
    }
    free(tmp);
    return 0;
}

int orc_f64_sum(const void *const *bufs, int p, int64_t n, int dtype,
                double *ref, double *mag)
{
    if (p < 1 || n < 0 || dtype == ORC_I32 || orc_elem_size(dtype) == 0) return -1;
    int es = orc_elem_size(dtype);
    for (int64_t i = 0; i < n; i++) {
        double s = 0.0, a = 0.0;
        for (int r = 0; r < p; r++) {
            double x = (double)load_float(dtype, (const unsigned char *)bufs[r] + (size_t)i * (size_t)es);
            s += x;
            a += x < 0 ? -x : x;
        }
        ref[i] = s;
        mag[i] = a;
    }
    return 0;
}

/* ------------------------------------------------------- hierarchical ring */

/* "Ring All-Reduce, in depth", "Hierarchy" / "Worked example": the three
 * phases below, each a ring of the schedule above on a subset of the ranks
 * (declared in rar_oracle.h). */
int orc_hier_simulate(void *const *bufs, int p, int g, int64_t n, int dtype,
                      int op, int64_t *sends_intra, int64_t *sends_inter)
{
    if (p < 1 || g < 1 || p % g != 0 || n < 0 || !valid_kind(dtype, op)) return -1;
    for (int r = 0; r < p; r++)
        if (!bufs[r] && n > 0) return -1;
    if (n == 0 || p == 1) return 0;
    const int m = p / g;
    const int es = orc_elem_size(dtype);
    const int hop_op = hop_of(op);
    void **ptrs = (void **)malloc(sizeof(void *) * (size_t)p);
    int64_t *tmp = (int64_t *)malloc(sizeof(int64_t) * (size_t)p);
    int64_t *gb = (int64_t *)malloc(sizeof(int64_t) * (size_t)(g + 1));
    int64_t *sb = (int64_t *)malloc(sizeof(int64_t) * (size_t)(m + 1));
    if (!ptrs || !tmp || !gb || !sb) { free(ptrs); free(tmp); free(gb); free(sb); return -1; }

    if (op == ORC_AVG_PREDIV)
        for (int r = 0; r < p; r++)
            for (int64_t i = 0; i < n; i++)
                scale_by_inv_p(dtype, (unsigned char *)bufs[r] + (size_t)i * (size_t)es, p);

    /* 1. reduce-scatter inside every node */
    for (int j = 0; j < m; j++) {
        for (int l = 0; l < g; l++) { ptrs[l] = bufs[j * g + l]; tmp[l] = 0; }
        orc_ring_simulate(ptrs, g, n, dtype, hop_op, ORC_FORWARD, 0, g - 1, tmp);
        if (sends_intra) for (int l = 0; l < g; l++) sends_intra[j * g + l] += tmp[l];
    }
    /* 2. all-reduce of every shard across the nodes */
    orc_chunk_bounds(n, g, gb);
    for (int l = 0; l < g; l++) {
        const int c = (l + 1) % g;
        const int64_t s0 = gb[c], len = gb[c + 1] - gb[c];
        for (int j = 0; j < m; j++) {
            ptrs[j] = (unsigned char *)bufs[j * g + l] + (size_t)s0 * (size_t)es;
            tmp[j] = 0;
        }
        orc_ring_simulate(ptrs, m, len, dtype, hop_op, ORC_FORWARD, 0, m - 1, tmp);
        if (op == ORC_AVG) {
            /* the shard's owner scales by 1/p before the all-gather */
            orc_chunk_bounds(len, m, sb);
            for (int j = 0; j < m; j++) {
                const int own = (j + 1) % m;
                for (int64_t i = sb[own]; i < sb[own + 1]; i++)
                    scale_by_inv_p(dtype, (unsigned char *)ptrs[j] + (size_t)i * (size_t)es, p);
            }
        }
        orc_ring_simulate(ptrs, m, len, dtype, hop_op, ORC_FORWARD, m - 1, m - 1, tmp);
        if (sends_inter) for (int j = 0; j < m; j++) sends_inter[j * g + l] += tmp[j];
    }
    /* 3. all-gather inside every node */
    for (int j = 0; j < m; j++) {
        for (int l = 0; l < g; l++) { ptrs[l] = bufs[j * g + l]; tmp[l] = 0; }
        orc_ring_simulate(ptrs, g, n, dtype, hop_op, ORC_FORWARD, g - 1, g - 1, tmp);
        if (sends_intra) for (int l = 0; l < g; l++) sends_intra[j * g + l] += tmp[l];
    }
    free(ptrs);
    free(tmp);
    free(gb);
    free(sb);
    return 0;
}

int orc_hier_fold_sampled(const void *vals, const int64_t *idx, int64_t m_samples,
                          int p, int g, int64_t n, int dtype, int op, void *out)
{
    if (p < 1 || g < 1 || p % g != 0 || n < 0 || m_samples < 0 || !valid_kind(dtype, op)) return -1;
    const int m = p / g;
    const int es = orc_elem_size(dtype);
    const int hop_op = hop_of(op);
    const unsigned char *v = (const unsigned char *)vals;
    unsigned char *o = (unsigned char *)out;
    int64_t *gb = (int64_t *)malloc(sizeof(int64_t) * (size_t)(g + 1));
    int64_t *sb = (int64_t *)malloc(sizeof(int64_t) * (size_t)(m + 1));
    unsigned char *tmp = (unsigned char *)malloc((size_t)p * (size_t)es);
    if (!gb || !sb || !tmp) { free(gb); free(sb); free(tmp); return -1; }
    orc_chunk_bounds(n, g, gb);
    int rc = 0;
    for (int64_t jx = 0; jx < m_samples; jx++) {
        const int64_t i = idx[jx];
        if (i < 0 || i >= n) { rc = -1; break; }
        for (int r = 0; r < p; r++) {
            memcpy(tmp + (size_t)r * (size_t)es, v + ((size_t)r * (size_t)m_samples + (size_t)jx) * (size_t)es, (size_t)es);
            if (op == ORC_AVG_PREDIV) scale_by_inv_p(dtype, tmp + (size_t)r * (size_t)es, p);
        }
        const int c = chunk_of(gb, g, i);
        orc_chunk_bounds(gb[c + 1] - gb[c], m, sb);
        const int s = chunk_of(sb, m, i - gb[c]);
        unsigned char acc[4], part[4];
        for (int t = 0; t < m; t++) {
            const int node = (s + t) % m;
            memcpy(part, tmp + (size_t)(node * g + c) * (size_t)es, (size_t)es);
            for (int k = 1; k < g; k++)
                orc_combine(dtype, hop_op, part, tmp + (size_t)(node * g + (c + k) % g) * (size_t)es, part);
            if (t == 0) memcpy(acc, part, (size_t)es);
            else orc_combine(dtype, hop_op, acc, part, acc);
        }
        if (op == ORC_AVG) scale_by_inv_p(dtype, acc, p);
        memcpy(o + (size_t)jx * (size_t)es, acc, (size_t)es);
    }
    free(gb);
    free(sb);
    free(tmp);
    return rc;
}
