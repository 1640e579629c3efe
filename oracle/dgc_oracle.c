/*
 * dgc_oracle.c -- the oracle: a plain, slow, single-threaded CPU restatement of the
 * per-worker compressor of Deep Gradient Compression (DGC), of its sparse message format and
 * of the decode-and-sum step that aggregates the learners' messages.
 *
 * TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU-baseline
 * leg call it; the product path never does. It shares no code with the CUDA library.
 *
 * Sources, by page title and section:
 *   [DGC] "[Paper Review] Deep Gradient Compression: Reducing the Communication Bandwidth for
 *         Distributed Training" -- Abstract (99.9% of the exchange is redundant; sizes
 *         97MB -> 0.35MB, 488MB -> 0.74MB), "Proposed method" (six bullets: send the large
 *         entries and keep the rest in a local accumulator; 32-bit values with 16-bit zero-run
 *         lengths; momentum correction; local clipping; momentum factor masking; warm-up),
 *         "Research questions" RQ4 (hierarchical thresholding).
 *   [ADA] "AdaComp : Adaptive Residual Gradient Compression for Data-Parallel Distributed
 *         Training" -- abstract (residues selected locally), citation snippets (entries ranked
 *         by magnitude, e.g. the largest 1%).
 *   [SC]  the ScaleComp abstract (Scalable Sparsified Gradient Compression) on the first page,
 *         a taxoreview.com listing -- a commutative compressor that uses how alike the
 *         learners' gradients are, keeps the traffic independent of the number of learners and
 *         works with all-reduce; a low-pass filter in the local gradient accumulation.
 * The pages give bullets, not formulas. Each step below names the reading it takes where the
 * pages leave a detail open.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off (no fast-math): every float operation below is a
 * single IEEE-754 binary32 or binary64 operation rounded to nearest-even, and fmaf is the
 * single-rounding fused multiply-add.
 */
#include "dgc_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BILLION 1000000000ull
#define ORC_GOLDEN 0x9E3779B97F4A7C15ull /* SplitMix64 increment (Steele, Lea, Flood 2014) */
#define ORC_RUN_ESCAPE 0xFFFFu
#define ORC_MAGIC 0x31434744u /* bytes 'D','G','C','1' read little-endian */

static uint32_t orc_key(float x) {
    /* |x| as an integer that orders like |x| for finite x; -0 and +0 both give 0 */
    uint32_t b;
    memcpy(&b, &x, sizeof b);
    return b & 0x7FFFFFFFu;
}

/* A fraction as an integer number of parts per billion. Reading: counts are then exact
 * integer arithmetic, so 1 - 0.999 = 0.0010000000000000009 cannot turn k = 1000 into 1001. */
uint64_t orc_ppb(double fraction) { return (uint64_t)llround(fraction * 1e9); }

/* ceil(n * ppb / 1e9). [DGC] Abstract: nearly all (99.9%) of what learners exchange is found
 * redundant, so 0.1% of the entries are sent; the count is rounded up (n = 1,048,576 at 99.9%
 * sparsity sends 1049). */
uint64_t orc_count(uint64_t n, uint64_t ppb) {
    return (n * ppb + (ORC_BILLION - 1)) / ORC_BILLION; /* n < 2^32, ppb <= 1e9: no overflow */
}

/* SplitMix64 output function (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): the j-th output of a generator seeded with s is mix(s + (j+1)*g). */
uint64_t orc_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t orc_mulhi64(uint64_t a, uint64_t b) {
    return (uint64_t)(((unsigned __int128)a * (unsigned __int128)b) >> 64);
}

/* Sampled threshold, [DGC] RQ4 (hierarchical thresholding): the sample is a fixed set of
 * positions per segment, drawn with replacement from SplitMix64 seeded per segment. Reading:
 * segment s uses seed_s = mix(seed + (s+1)*g); draw j lands at floor(mix(seed_s + (j+1)*g) *
 * n_s / 2^64). The same seed gives the same positions every step. */
uint64_t orc_sample_position(uint64_t seed, uint32_t segment, uint64_t j, uint64_t n_s) {
    uint64_t seg_seed = orc_mix64(seed + ORC_GOLDEN * ((uint64_t)segment + 1));
    return orc_mulhi64(orc_mix64(seg_seed + ORC_GOLDEN * (j + 1)), n_s);
}

/* The sum of squares is kept exactly as a non-negative integer X in base-2^32 digits, least
 * significant first. Entry x = m 2^(e'-150) (m its 24-bit significand with the hidden bit,
 * e' = max(biased exponent, 1)) has x^2 = m^2 2^(2e'-300), and X collects m^2 2^(2e'-2), so
 * that the sum of squares is X 2^-298. With m^2 < 2^48, 2e'-2 <= 506 and at most 2^32 entries,
 * X < 2^586: twenty digits hold it. */
#define ORC_SQ_DIGITS 20

/* d += x 2^(32 i), carrying upward */
static void orc_digits_add(uint32_t* d, int i, uint64_t x) {
    uint64_t carry = x;
    while (carry != 0 && i < ORC_SQ_DIGITS) {
        const uint64_t t = (uint64_t)d[i] + (carry & 0xFFFFFFFFull);
        d[i] = (uint32_t)t;
        carry = (carry >> 32) + (t >> 32);
        ++i;
    }
}

static int orc_digits_bit(const uint32_t* d, int b) { return (int)((d[b / 32] >> (b % 32)) & 1u); }

/* X 2^-298 rounded to the nearest binary64, ties to the even significand. The result is never
 * below 2^-298 (unless X = 0) nor near the binary64 overflow, so the significand is kept whole
 * and ldexp only moves the exponent. */
static double orc_digits_round(const uint32_t* d) {
    int top = -1;
    for (int b = ORC_SQ_DIGITS * 32 - 1; b >= 0 && top < 0; --b)
        if (orc_digits_bit(d, b)) top = b;
    if (top < 0) return 0.0;
    int low = top - 52;  /* the last bit kept */
    if (low < 0) low = 0;
    uint64_t mant = 0;
    for (int b = top; b >= low; --b) mant = (mant << 1) | (uint64_t)orc_digits_bit(d, b);
    if (low > 0) {
        const int half = orc_digits_bit(d, low - 1);
        int rest = 0;
        for (int b = low - 2; b >= 0 && !rest; --b) rest = orc_digits_bit(d, b);
        if (half && (rest || (mant & 1u))) {
            mant += 1;
            if (mant == (1ull << 53)) {
                mant >>= 1;
                low += 1;
            }
        }
    }
    return ldexp((double)mant, low - 298);
}

/* Squared L2 norm for local gradient clipping, [DGC] Proposed method, bullet 4. Reading: the
 * pages fix no order for the sum, so S is the exact sum of the squares rounded once to the
 * nearest binary64 (ties to even) -- the one value that every order of exact arithmetic
 * reaches. A NaN entry makes S NaN; otherwise an infinite entry makes it +infinity. */
double orc_sumsq(const float* g, int64_t n) {
    uint32_t d[ORC_SQ_DIGITS];
    memset(d, 0, sizeof d);
    int has_inf = 0, has_nan = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t bits;
        memcpy(&bits, &g[i], sizeof bits);
        const uint32_t e = (bits >> 23) & 0xFFu;
        const uint32_t f = bits & 0x7FFFFFu;
        if (e == 0xFFu) {
            if (f) has_nan = 1; else has_inf = 1;
            continue;
        }
        const uint64_t m = e ? (f | 0x800000u) : f;
        const uint64_t m2 = m * m;
        const int at = 2 * (int)(e ? e : 1u) - 2;  /* the bit of X where m^2 starts */
        orc_digits_add(d, at / 32, (m2 & 0xFFFFFFFFull) << (at % 32));
        orc_digits_add(d, at / 32 + 1, (m2 >> 32) << (at % 32));
    }
    if (has_nan) return NAN;
    if (has_inf) return INFINITY;
    return orc_digits_round(d);
}

/* Local gradient clipping, [DGC] Proposed method, bullet 4. Reading: it bounds the L2 norm of
 * each segment's fresh gradient by c before momentum is applied; when sqrt(S) > c the gradient
 * is multiplied by the binary32 rounding of c / sqrt(S), otherwise it is left as it is. */
float orc_clip_scale(const float* g, int64_t n, float clip_norm, int* clipped) {
    *clipped = 0;
    if (!(clip_norm > 0.0f) || isinf(clip_norm) || n == 0) return 1.0f;
    double norm = sqrt(orc_sumsq(g, n));
    if (norm > (double)clip_norm) {
        *clipped = 1;
        return (float)((double)clip_norm / norm);
    }
    return 1.0f;
}

/* Momentum correction, [DGC] Proposed method, bullet 3, with local accumulation, bullet 1:
 * u <- m*u + g (one fused multiply-add, one rounding), then v <- v + u. */
void orc_accumulate_one(float g, float u, float v, float momentum, float scale, int clipped,
                        float* u_out, float* v_out) {
    float gp = clipped ? g * scale : g;
    float un = fmaf(momentum, u, gp);
    *u_out = un;
    *v_out = v + un;
}

/* The accumulation with [SC]'s low-pass filter. Reading: the accumulator becomes a first-order
 * (leaky) low-pass filter, v <- leak*v + u in one fused multiply-add, 0 < leak <= 1; leak = 1 is
 * DGC's plain accumulation (fmaf(1, v, u) rounds v + u once, exactly as the addition does). */
void orc_accumulate_leak(float g, float u, float v, float momentum, float scale, int clipped,
                         float leak, float* u_out, float* v_out) {
    float gp = clipped ? g * scale : g;
    float un = fmaf(momentum, u, gp);
    *u_out = un;
    *v_out = fmaf(leak, v, un);
}

typedef struct {
    uint32_t key;
    uint32_t idx;
} orc_entry;

/* selection order: larger key first; among equal keys the lower index first */
static int orc_entry_cmp(const void* a, const void* b) {
    const orc_entry* x = (const orc_entry*)a;
    const orc_entry* y = (const orc_entry*)b;
    if (x->key != y->key) return x->key > y->key ? -1 : 1;
    if (x->idx != y->idx) return x->idx < y->idx ? -1 : 1;
    return 0;
}

/* Top-k by magnitude, [ADA] citation snippets (only the gradients that matter are sent, ranked
 * by magnitude, e.g. the largest 1%): the first k entries after sorting the candidates by
 * (|v| descending, index ascending). selected[cand[i]] is set for each chosen entry. */
int orc_topk(const float* v, const uint32_t* cand, int64_t ncand, int64_t k, uint8_t* selected) {
    if (k <= 0 || ncand <= 0) return ORC_OK;
    orc_entry* e = (orc_entry*)malloc((size_t)ncand * sizeof *e);
    if (!e) return ORC_ENOMEM;
    for (int64_t i = 0; i < ncand; ++i) {
        e[i].idx = cand[i];
        e[i].key = orc_key(v[cand[i]]);
    }
    qsort(e, (size_t)ncand, sizeof *e, orc_entry_cmp);
    int64_t take = k < ncand ? k : ncand;
    for (int64_t i = 0; i < take; ++i) selected[e[i].idx] = 1;
    free(e);
    return ORC_OK;
}

/* AdaComp selection, [ADA] abstract (residues are selected locally, so the compression rate
 * follows local activity) and citation snippet (each layer's residual is cut into fixed-size
 * bins; a bin's largest |residual| is its threshold). Reading: bins are runs of bin_size
 * consecutive entries from the start of the segment (the last one may be shorter); the entries
 * whose |v| reaches the bin's largest |v| are selected, ties included; a bin whose largest |v|
 * is 0 selects nothing. */
void orc_bin_select(const float* v, int64_t n, uint32_t bin_size, uint8_t* selected) {
    for (int64_t b = 0; b < n; b += bin_size) {
        const int64_t e = (b + (int64_t)bin_size < n) ? b + (int64_t)bin_size : n;
        uint32_t mx = 0;
        for (int64_t i = b; i < e; ++i)
            if (orc_key(v[i]) > mx) mx = orc_key(v[i]);
        if (mx == 0) continue;
        for (int64_t i = b; i < e; ++i)
            if (orc_key(v[i]) == mx) selected[i] = 1;
    }
}

static int orc_u32_desc(const void* a, const void* b) {
    uint32_t x = *(const uint32_t*)a, y = *(const uint32_t*)b;
    return x > y ? -1 : (x < y ? 1 : 0);
}

/* One compressor step over a set of segments (tensors), each compressed on its own.
 *   1. k = ceil(n_s * (1 - sparsity)), [DGC] Abstract.
 *   2. local gradient clipping of the fresh gradient, [DGC] Proposed method, bullet 4.
 *   3. u <- m*u + g; v <- v + u, [DGC] Proposed method, bullets 3 and 1.
 *   4. selection S of the largest |v|:
 *      exact   -- the k largest under (|v| desc, index asc);
 *      AdaComp -- per fixed-size bin, the entries at the bin's largest |v| (orc_bin_select);
 *      sampled -- [DGC] RQ4: t = the k_s-th largest |v| among m_s = ceil(n_s * ratio) sampled
 *                 entries, k_s = ceil(m_s * (1 - sparsity)); C = {i : |v_i| >= t}; reading of
 *                 "hierarchical": when |C| > factor * k, S = the exact top-k of C, else S = C.
 *   5. send (i, v_i) for i in S in ascending i; the sent entries leave the accumulator
 *      (v_i <- 0) and, with momentum factor masking ([DGC] Proposed method, bullet 5), u_i <- 0.
 * Unsent entries keep their accumulated values: the residual of [DGC] bullet 1. */
int orc_compress(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
                 int32_t nseg, const orc_params* p, uint32_t* out_idx, float* out_val,
                 int64_t out_cap, int64_t* out_count, orc_seg_stats* stats) {
    if (!p || !seg_off || nseg < 1 || n < 0 || n > 0xFFFFFFFFll) return ORC_EINVAL;
    if (!(p->sparsity >= 0.0 && p->sparsity <= 1.0)) return ORC_EINVAL;
    if (p->mode != ORC_EXACT && p->mode != ORC_SAMPLED && p->mode != ORC_ADACOMP) return ORC_EINVAL;
    if (p->mode == ORC_ADACOMP && p->bin_size == 0) return ORC_EINVAL;
    if (!(p->leak >= 0.0f && p->leak <= 1.0f)) return ORC_EINVAL; /* 0: no filter (leak 1) */
    if (seg_off[0] != 0 || seg_off[nseg] != n) return ORC_EINVAL;
    for (int32_t s = 0; s < nseg; ++s)
        if (seg_off[s + 1] < seg_off[s]) return ORC_EINVAL;
    if (p->mode == ORC_SAMPLED && !(p->sample_ratio > 0.0 && p->sample_ratio <= 1.0))
        return ORC_EINVAL;
    if (p->mode == ORC_SAMPLED && orc_ppb(p->sample_ratio) == 0) return ORC_EINVAL;

    const uint64_t d_ppb = orc_ppb(1.0 - p->sparsity);
    const uint64_t r_ppb = orc_ppb(p->sample_ratio);
    const uint64_t q_ppb = orc_ppb(p->reselect_factor);
    const int mask_momentum = (p->flags & ORC_MASK_MOMENTUM) != 0;
    int64_t total = 0;

    for (int32_t s = 0; s < nseg; ++s) {
        const int64_t a = seg_off[s], b = seg_off[s + 1], ns = b - a;
        orc_seg_stats st;
        memset(&st, 0, sizeof st);
        st.thresh_key = 0xFFFFFFFFu;
        const uint64_t k = (p->mode == ORC_ADACOMP)
                               ? ((uint64_t)ns + p->bin_size - 1) / p->bin_size
                               : orc_count((uint64_t)ns, d_ppb);
        st.k = k;

        int clipped = 0;
        const float scale = orc_clip_scale(g + a, ns, p->clip_norm, &clipped);
        st.clip_scale = scale;
        if (p->clip_norm > 0.0f && !isinf(p->clip_norm)) st.clip_sumsq = orc_sumsq(g + a, ns);

        const float leak = p->leak == 0.0f ? 1.0f : p->leak;
        for (int64_t i = a; i < b; ++i)
            orc_accumulate_leak(g[i], u[i], v[i], p->momentum, scale, clipped, leak, &u[i], &v[i]);

        uint8_t* sel = (uint8_t*)calloc((size_t)(ns > 0 ? ns : 1), 1);
        uint32_t* cand = (uint32_t*)malloc((size_t)(ns > 0 ? ns : 1) * sizeof(uint32_t));
        if (!sel || !cand) {
            free(sel);
            free(cand);
            return ORC_ENOMEM;
        }
        const float* vs = v + a; /* segment-local view: indices below are segment-relative */

        if (p->mode == ORC_ADACOMP) {
            orc_bin_select(vs, ns, p->bin_size, sel);
        } else if (k > 0 && p->mode == ORC_EXACT) {
            for (int64_t i = 0; i < ns; ++i) cand[i] = (uint32_t)i;
            if (orc_topk(vs, cand, ns, (int64_t)k, sel) != ORC_OK) goto nomem;
        } else if (k > 0) {
            const uint64_t ms = orc_count((uint64_t)ns, r_ppb);
            const uint64_t ks = orc_count(ms, d_ppb);
            uint32_t* keys = (uint32_t*)malloc((size_t)ms * sizeof(uint32_t));
            if (!keys) goto nomem;
            for (uint64_t j = 0; j < ms; ++j)
                keys[j] = orc_key(vs[orc_sample_position(p->seed, (uint32_t)s, j, (uint64_t)ns)]);
            qsort(keys, (size_t)ms, sizeof(uint32_t), orc_u32_desc);
            const uint32_t t = keys[ks - 1];
            free(keys);
            st.sample_key = t;
            int64_t nc = 0;
            for (int64_t i = 0; i < ns; ++i)
                if (orc_key(vs[i]) >= t) cand[nc++] = (uint32_t)i;
            st.candidates = (uint64_t)nc;
            /* reading of "1.3k": |C| > factor * k, compared in parts per billion */
            if ((unsigned __int128)nc * ORC_BILLION > (unsigned __int128)q_ppb * k) {
                st.reselected = 1;
                if (orc_topk(vs, cand, nc, (int64_t)k, sel) != ORC_OK) goto nomem;
            } else {
                for (int64_t c = 0; c < nc; ++c) sel[cand[c]] = 1;
            }
        }

        for (int64_t i = 0; i < ns; ++i) {
            if (!sel[i]) continue;
            if (total >= out_cap) {
                free(sel);
                free(cand);
                return ORC_ECAPACITY;
            }
            const uint32_t key = orc_key(vs[i]);
            if (key < st.thresh_key) st.thresh_key = key;
            out_idx[total] = (uint32_t)(a + i);
            out_val[total] = vs[i];
            ++total;
            ++st.sent;
            v[a + i] = 0.0f;
            if (mask_momentum) u[a + i] = 0.0f;
        }
        if (p->mode != ORC_SAMPLED) st.candidates = st.sent;
        if (stats) stats[s] = st;
        free(sel);
        free(cand);
        continue;
    nomem:
        free(sel);
        free(cand);
        return ORC_ENOMEM;
    }
    *out_count = total;
    return ORC_OK;
}

/* ---- codec: [DGC] Proposed method, bullet 2 (each sent value takes 32 bits and each stretch
 * of zeros before it a 16-bit length). Reading of the layout (the pages fix only the widths):
 *   header, 32 bytes little-endian: magic "DGC1", u16 version 1, u16 flags 0, u64 n, u64 T,
 *   u64 nnz; then T binary32 values; then T u16 run lengths; zero bytes up to a multiple of 4.
 * Entry j skips r_j = idx_j - idx_{j-1} - 1 zeros (idx_{-1} = -1). A gap of 65535 or more is
 * written as escape tokens (run 0xFFFF, value bits 0) that each skip 65535 zeros without
 * placing a value, followed by the entry's own token with the remainder. ---- */

static void orc_put16(uint8_t* p, uint16_t x) {
    p[0] = (uint8_t)(x & 0xFF);
    p[1] = (uint8_t)(x >> 8);
}
static void orc_put32(uint8_t* p, uint32_t x) {
    for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(x >> (8 * i));
}
static void orc_put64(uint8_t* p, uint64_t x) {
    for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(x >> (8 * i));
}
static uint16_t orc_get16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t orc_get32(const uint8_t* p) {
    uint32_t x = 0;
    for (int i = 0; i < 4; ++i) x |= (uint32_t)p[i] << (8 * i);
    return x;
}
static uint64_t orc_get64(const uint8_t* p) {
    uint64_t x = 0;
    for (int i = 0; i < 8; ++i) x |= (uint64_t)p[i] << (8 * i);
    return x;
}

static uint64_t orc_tokens(const uint32_t* idx, int64_t count) {
    uint64_t T = 0;
    int64_t prev = -1;
    for (int64_t j = 0; j < count; ++j) {
        int64_t gap = (int64_t)idx[j] - prev - 1;
        T += 1 + (uint64_t)gap / ORC_RUN_ESCAPE;
        prev = idx[j];
    }
    return T;
}

static uint64_t orc_size_for(uint64_t T) { return 32 + 6 * T + ((T & 1) ? 2 : 0); }

uint64_t orc_encoded_size(const uint32_t* idx, int64_t count) {
    return orc_size_for(orc_tokens(idx, count));
}

int orc_encode(const uint32_t* idx, const float* val, int64_t count, int64_t n, uint8_t* out,
               uint64_t out_cap, uint64_t* out_bytes) {
    if (count < 0 || n < 0) return ORC_EINVAL;
    int64_t prev = -1;
    for (int64_t j = 0; j < count; ++j) {
        if ((int64_t)idx[j] <= prev || (int64_t)idx[j] >= n) return ORC_EINVAL;
        prev = idx[j];
    }
    const uint64_t T = orc_tokens(idx, count);
    const uint64_t size = orc_size_for(T);
    *out_bytes = size;
    if (size > out_cap) return ORC_ECAPACITY;
    memset(out, 0, (size_t)size);
    orc_put32(out, ORC_MAGIC);
    orc_put16(out + 4, 1);
    orc_put16(out + 6, 0);
    orc_put64(out + 8, (uint64_t)n);
    orc_put64(out + 16, T);
    orc_put64(out + 24, (uint64_t)count);
    uint8_t* vals = out + 32;
    uint8_t* runs = out + 32 + 4 * T;
    uint64_t tok = 0;
    prev = -1;
    for (int64_t j = 0; j < count; ++j) {
        uint64_t r = (uint64_t)((int64_t)idx[j] - prev - 1);
        while (r >= ORC_RUN_ESCAPE) {
            orc_put32(vals + 4 * tok, 0);
            orc_put16(runs + 2 * tok, ORC_RUN_ESCAPE);
            ++tok;
            r -= ORC_RUN_ESCAPE;
        }
        uint32_t bits;
        memcpy(&bits, &val[j], 4);
        orc_put32(vals + 4 * tok, bits);
        orc_put16(runs + 2 * tok, (uint16_t)r);
        ++tok;
        prev = idx[j];
    }
    return ORC_OK;
}

/* Decode and sum W learners' messages into one dense gradient: in synchronous distributed SGD
 * every learner's update is added up ([DGC] Abstract, Motivation). Reading: the sum
 * is taken in the fixed learner order 0..W-1, one binary32 addition per received value, onto
 * +0 (accumulate = 0) or onto the existing dense contents (accumulate = 1). A stream that is
 * malformed (magic, version, n, size, or a position past n) makes the call fail and leaves
 * dense unchanged. */
int orc_decode_accumulate(const uint8_t* const* streams, const uint64_t* stream_bytes,
                          int32_t W, float* dense, int64_t n, int accumulate) {
    if (W < 0 || n < 0) return ORC_EINVAL;
    for (int32_t w = 0; w < W; ++w) {
        const uint8_t* s = streams[w];
        const uint64_t bytes = stream_bytes[w];
        if (bytes < 32) return ORC_ECORRUPT;
        if (orc_get32(s) != ORC_MAGIC || orc_get16(s + 4) != 1) return ORC_ECORRUPT;
        if (orc_get64(s + 8) != (uint64_t)n) return ORC_ECORRUPT;
        const uint64_t T = orc_get64(s + 16);
        if (T > bytes || orc_size_for(T) != bytes) return ORC_ECORRUPT;
        const uint8_t* runs = s + 32 + 4 * T;
        int64_t pos = -1;
        for (uint64_t t = 0; t < T; ++t) {
            const uint16_t r = orc_get16(runs + 2 * t);
            pos += (r == ORC_RUN_ESCAPE) ? (int64_t)ORC_RUN_ESCAPE : (int64_t)r + 1;
            if (pos >= n) return ORC_ECORRUPT;
        }
    }
    if (!accumulate)
        for (int64_t i = 0; i < n; ++i) dense[i] = 0.0f;
    for (int32_t w = 0; w < W; ++w) {
        const uint8_t* s = streams[w];
        const uint64_t T = orc_get64(s + 16);
        const uint8_t* vals = s + 32;
        const uint8_t* runs = s + 32 + 4 * T;
        int64_t pos = -1;
        for (uint64_t t = 0; t < T; ++t) {
            const uint16_t r = orc_get16(runs + 2 * t);
            if (r == ORC_RUN_ESCAPE) {
                pos += ORC_RUN_ESCAPE;
                continue;
            }
            pos += (int64_t)r + 1;
            const uint32_t bits = orc_get32(vals + 4 * t);
            float x;
            memcpy(&x, &bits, 4);
            dense[pos] = dense[pos] + x;
        }
    }
    return ORC_OK;
}

/* Decode, sum and apply as one plain SGD step: s = the ordered sum of the W messages (exactly
 * as orc_decode_accumulate builds it from +0), then w_i <- fmaf(-lr, s_i, w_i) for every i.
 * [DGC] Abstract: the setting is distributed SGD; "Proposed method", momentum-correction
 * bullet: the velocity is accumulated locally, so what the learners send is already the
 * momentum-corrected update. Reading: the receiver therefore takes a plain SGD step
 * w <- w - lr * s with the summed message, one rounding (fmaf); the caller folds any 1/W
 * average into lr. lr must be finite with its sign bit clear (+0 allowed): then entries that no
 * message touches (s_i = +0) keep their bits, -0 included. On any error w is left unchanged. */
int orc_decode_apply(const uint8_t* const* streams, const uint64_t* stream_bytes, int32_t W,
                     float* w, int64_t n, float lr) {
    if (W < 0 || n < 0 || !isfinite(lr) || signbit(lr)) return ORC_EINVAL;
    float* s = (float*)calloc(n > 0 ? (size_t)n : 1, sizeof(float));
    if (!s) return ORC_ENOMEM;
    const int rc = orc_decode_accumulate(streams, stream_bytes, W, s, n, 0);
    if (rc == ORC_OK)
        for (int64_t i = 0; i < n; ++i) w[i] = fmaf(-lr, s[i], w[i]);
    free(s);
    return rc;
}

/* ---- integer values: [ADA] abstract (AdaComp sends the selected residues both sparse and
 * quantized); the IntSGD page, abstract (each learner multiplies its vector by a number every
 * learner knows and rounds to integers, so no float is sent). Reading of the quantizer (the pages
 * give no bit format):
 *   q_j = clamp(rint(alpha * val_j), -Q, Q), Q = 2^(b-1) - 1, b in {8, 16}; the product is one
 *         binary32 multiply, rint rounds half to even, NaN gives 0;
 *   deq(q) = (float)q / alpha (one binary32 divide); the residual keeps what the integer did
 *         not carry: v[idx_j] <- val_j - deq(q_j) (one binary32 subtract; [DGC] Proposed method,
 *         bullet 1: what is not sent stays in the local accumulator).
 * Message, version 2: header "DGC1", u16 version 2, u16 b, u64 n, u64 T, binary32 alpha, u32
 * nnz; then T two's-complement integers of b bits (escape tokens carry 0), zero bytes up to an
 * even offset, T u16 runs (no padding after them). Receivers sum the integers exactly
 * (order does not matter) and divide once: dense_i = (float)S_i / alpha. ---- */
static int32_t orc_quantize(float val, float alpha, int bits) {
    const float x = rintf(alpha * val);
    const float Q = (float)((1 << (bits - 1)) - 1);
    if (isnan(x)) return 0;
    if (x > Q) return (int32_t)Q;
    if (x < -Q) return -(int32_t)Q;
    return (int32_t)x;
}

static uint64_t orc_runs_offset(uint64_t T, int bits) {
    const uint64_t at = 32 + T * (uint64_t)(bits / 8);
    return at + (at & 1); /* runs start at an even offset */
}

/* no padding after the runs: the size then fixes T, so a receiver that knows b can lay out the
 * messages from their sizes alone (a pad to 4 bytes would make 8-bit messages of 3 and 4 tokens
 * the same size) */
static uint64_t orc_size_quant(uint64_t T, int bits) { return orc_runs_offset(T, bits) + 2 * T; }

int orc_encode_quant(const uint32_t* idx, const float* val, int64_t count, int64_t n, float alpha,
                     int bits, float* v, uint8_t* out, uint64_t out_cap, uint64_t* out_bytes) {
    if (count < 0 || n < 0 || (bits != 8 && bits != 16) || !isfinite(alpha) || !(alpha > 0.0f))
        return ORC_EINVAL;
    int64_t prev = -1;
    for (int64_t j = 0; j < count; ++j) {
        if ((int64_t)idx[j] <= prev || (int64_t)idx[j] >= n) return ORC_EINVAL;
        prev = idx[j];
    }
    const uint64_t T = orc_tokens(idx, count);
    const uint64_t size = orc_size_quant(T, bits);
    *out_bytes = size;
    if (size > out_cap) return ORC_ECAPACITY;
    memset(out, 0, (size_t)size);
    orc_put32(out, ORC_MAGIC);
    orc_put16(out + 4, 2);
    orc_put16(out + 6, (uint16_t)bits);
    orc_put64(out + 8, (uint64_t)n);
    orc_put64(out + 16, T);
    uint32_t abits;
    memcpy(&abits, &alpha, 4);
    orc_put32(out + 24, abits);
    orc_put32(out + 28, (uint32_t)count);
    const int vb = bits / 8;
    uint8_t* vals = out + 32;
    uint8_t* runs = out + orc_runs_offset(T, bits);
    uint64_t tok = 0;
    prev = -1;
    for (int64_t j = 0; j < count; ++j) {
        uint64_t r = (uint64_t)((int64_t)idx[j] - prev - 1);
        while (r >= ORC_RUN_ESCAPE) { /* value bytes stay 0 */
            orc_put16(runs + 2 * tok, ORC_RUN_ESCAPE);
            ++tok;
            r -= ORC_RUN_ESCAPE;
        }
        const int32_t q = orc_quantize(val[j], alpha, bits);
        if (vb == 1)
            vals[tok] = (uint8_t)(q & 0xFF);
        else
            orc_put16(vals + 2 * tok, (uint16_t)(q & 0xFFFF));
        orc_put16(runs + 2 * tok, (uint16_t)r);
        ++tok;
        if (v) v[idx[j]] = val[j] - (float)q / alpha;
        prev = idx[j];
    }
    return ORC_OK;
}

/* The integer sums of W version-2 messages: S (int64) and which positions a value token reached.
 * Every message must carry the caller's width and alpha (bitwise): like alpha, the width is
 * fixed for all learners, and the receiver needs it to find each message's runs. */
static int orc_sum_quant(const uint8_t* const* streams, const uint64_t* stream_bytes, int32_t W,
                         int64_t n, int qbits, float alpha, int64_t* S, uint8_t* touched) {
    uint32_t abits;
    memcpy(&abits, &alpha, 4);
    for (int32_t w = 0; w < W; ++w) {
        const uint8_t* s = streams[w];
        const uint64_t bytes = stream_bytes[w];
        if (bytes < 32) return ORC_ECORRUPT;
        const int bits = orc_get16(s + 6);
        if (orc_get32(s) != ORC_MAGIC || orc_get16(s + 4) != 2 || bits != qbits ||
            orc_get64(s + 8) != (uint64_t)n || orc_get32(s + 24) != abits)
            return ORC_ECORRUPT;
        const uint64_t T = orc_get64(s + 16);
        if (T > bytes || orc_size_quant(T, bits) != bytes) return ORC_ECORRUPT;
        const uint8_t* runs = s + orc_runs_offset(T, bits);
        int64_t pos = -1;
        for (uint64_t t = 0; t < T; ++t) {
            const uint16_t r = orc_get16(runs + 2 * t);
            pos += (r == ORC_RUN_ESCAPE) ? (int64_t)ORC_RUN_ESCAPE : (int64_t)r + 1;
            if (pos >= n) return ORC_ECORRUPT;
        }
    }
    for (int64_t i = 0; i < n; ++i) {
        S[i] = 0;
        touched[i] = 0;
    }
    for (int32_t w = 0; w < W; ++w) {
        const uint8_t* s = streams[w];
        const int bits = orc_get16(s + 6);
        const uint64_t T = orc_get64(s + 16);
        const uint8_t* runs = s + orc_runs_offset(T, bits);
        int64_t pos = -1;
        for (uint64_t t = 0; t < T; ++t) {
            const uint16_t r = orc_get16(runs + 2 * t);
            if (r == ORC_RUN_ESCAPE) {
                pos += ORC_RUN_ESCAPE;
                continue;
            }
            pos += (int64_t)r + 1;
            const int32_t q = (bits == 8) ? (int32_t)(int8_t)s[32 + t]
                                          : (int32_t)(int16_t)orc_get16(s + 32 + 2 * t);
            S[pos] += q;
            touched[pos] = 1;
        }
    }
    return ORC_OK;
}

/* Decode and sum version-2 messages: dense_i = (float)S_i / alpha at every position some message
 * reaches, added onto dense_i when accumulate is set (one binary32 addition); +0 elsewhere
 * unless accumulating. W is at most 65536, so |S_i| < 2^31. */
int orc_decode_accumulate_quant(const uint8_t* const* streams, const uint64_t* stream_bytes,
                                int32_t W, int bits, float alpha, float* dense, int64_t n,
                                int accumulate) {
    if (W < 0 || n < 0 || (bits != 8 && bits != 16) || !isfinite(alpha) || !(alpha > 0.0f))
        return ORC_EINVAL;
    if (W > 65536) return ORC_EUNSUPPORTED;
    int64_t* S = (int64_t*)malloc((n > 0 ? (size_t)n : 1) * sizeof(int64_t));
    uint8_t* touched = (uint8_t*)malloc(n > 0 ? (size_t)n : 1);
    if (!S || !touched) {
        free(S);
        free(touched);
        return ORC_ENOMEM;
    }
    const int rc = orc_sum_quant(streams, stream_bytes, W, n, bits, alpha, S, touched);
    if (rc == ORC_OK)
        for (int64_t i = 0; i < n; ++i) {
            const float x = (float)S[i] / alpha;
            if (!accumulate)
                dense[i] = x;
            else if (touched[i])
                dense[i] = dense[i] + x;
        }
    free(S);
    free(touched);
    return rc;
}

/* The SGD step of orc_decode_apply with version-2 messages: w_i <- fmaf(-lr, (float)S_i / alpha,
 * w_i); lr as there. */
int orc_decode_apply_quant(const uint8_t* const* streams, const uint64_t* stream_bytes, int32_t W,
                           int bits, float alpha, float* w, int64_t n, float lr) {
    if (!isfinite(lr) || signbit(lr)) return ORC_EINVAL;
    float* s = (float*)malloc((n > 0 ? (size_t)n : 1) * sizeof(float));
    if (!s) return ORC_ENOMEM;
    const int rc = orc_decode_accumulate_quant(streams, stream_bytes, W, bits, alpha, s, n, 0);
    if (rc == ORC_OK)
        for (int64_t i = 0; i < n; ++i) w[i] = fmaf(-lr, s[i], w[i]);
    free(s);
    return rc;
}

/* ---- [SC]'s commutative compressor. Reading: every learner sends its accumulator at one
 * shared index set S (the same positions for all), so the learners' messages are vectors of
 * the same |S| entries that add up position by position -- what an all-reduce computes -- and
 * each learner's traffic is |S| values whatever the number of learners. Which learner chooses S
 * is the caller's choice (for instance one learner in turn, with orc_compress); the others then
 * call orc_compress_shared with that S. ---- */

/* One step of a learner that sends at the given S: clipping and accumulation exactly as in
 * orc_compress (same parameters; the selection mode and sparsity are not used), then for each
 * j < count: out_val[j] = v[idx[j]], and the sent entry leaves the accumulator (v <- 0, u <- 0
 * with masking). idx must be strictly ascending and below n. */
int orc_compress_shared(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
                        int32_t nseg, const orc_params* p, const uint32_t* idx, int64_t count,
                        float* out_val) {
    if (!p || !seg_off || nseg < 1 || n < 0 || n > 0xFFFFFFFFll || count < 0) return ORC_EINVAL;
    if (!(p->leak >= 0.0f && p->leak <= 1.0f)) return ORC_EINVAL;
    if (seg_off[0] != 0 || seg_off[nseg] != n) return ORC_EINVAL;
    for (int32_t s = 0; s < nseg; ++s)
        if (seg_off[s + 1] < seg_off[s]) return ORC_EINVAL;
    int64_t prev = -1;
    for (int64_t j = 0; j < count; ++j) {
        if ((int64_t)idx[j] <= prev || (int64_t)idx[j] >= n) return ORC_EINVAL;
        prev = idx[j];
    }
    const float leak = p->leak == 0.0f ? 1.0f : p->leak;
    for (int32_t s = 0; s < nseg; ++s) {
        const int64_t a = seg_off[s], b = seg_off[s + 1];
        int clipped = 0;
        const float scale = orc_clip_scale(g + a, b - a, p->clip_norm, &clipped);
        for (int64_t i = a; i < b; ++i)
            orc_accumulate_leak(g[i], u[i], v[i], p->momentum, scale, clipped, leak, &u[i], &v[i]);
    }
    for (int64_t j = 0; j < count; ++j) {
        out_val[j] = v[idx[j]];
        v[idx[j]] = 0.0f;
        if (p->flags & ORC_MASK_MOMENTUM) u[idx[j]] = 0.0f;
    }
    return ORC_OK;
}

/* The sum of W learners' value vectors over one shared S: out[j] = the learner-ordered sum
 * from +0 of vals[w][j], one binary32 addition each (the order the decoder uses). */
int orc_sum_shared(const float* const* vals, int32_t W, int64_t count, float* out) {
    if (W < 0 || count < 0) return ORC_EINVAL;
    for (int64_t j = 0; j < count; ++j) {
        float acc = 0.0f;
        for (int32_t w = 0; w < W; ++w) acc = acc + vals[w][j];
        out[j] = acc;
    }
    return ORC_OK;
}
