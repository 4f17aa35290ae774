/*
 * Oracle for sliding-window softmax attention with attention sinks, SWA(w,s).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; both sides only see the same seeded 16-bit inputs.
 *
 * What it computes (the plain definition, fp64 throughout):
 *
 *   Window formula -- "Sliding-window beats linear attention" (paper summary
 *   page), section "Prerequisites / Sliding-window attention SWA(w, s)", the
 *   displayed equation for x_t: each position t attends to the most recent w
 *   tokens with scale 1/sqrt(d), and the softmax is normalised only over the
 *   attended tokens.
 *
 *   Sinks -- same page, same section, the notation paragraph, and section
 *   "Method steps", step two: in SWA(w,s) the window w keeps s of its places
 *   for the first tokens of the sequence, so position t attends to the first s
 *   tokens plus the most recent w-s tokens.  The blog page "Microsoft SWA paper
 *   overturns linear attention", section "What they tested", gives the worked
 *   case w=64, s=4: the first 4 tokens plus the latest 60.
 *
 *   Fixed cache -- news page "No post-training, just 4 more tokens: sliding
 *   window attention overtakes linear attention", section "Research method":
 *   once the cache holds the window it stops growing; the blog page above says
 *   the method only changes the attention mask and the KV-cache eviction rule.
 *
 * Readings taken where the pages are silent (each is restated in the design
 * notes):
 *   - indices are 0-based: A(t) = {i : 0 <= i < min(s, t+1)}
 *                                 U {i : max(0, t-(w-s)+1) <= i <= t},
 *     a set union, so a token in both parts counts once; |A(t)| = min(t+1, w);
 *   - w < 0 stands for w = infinity, i.e. full causal attention, A(t) = [0, t];
 *   - grouped-query heads: query head h reads key/value head h / (Hq/Hkv);
 *   - a cache slot for position p is p for p < s and s + (p-s) mod (w-s)
 *     otherwise (for w = infinity, slot = p); appending writes positions in
 *     increasing order, so a later position overwrites an earlier one in the
 *     same slot;
 *   - inputs are 16-bit floating-point bit patterns, bf16 or IEEE binary16
 *     (fp16, the precision of the pages' own system measurements: paper
 *     summary page, section "Method steps", step five), widened exactly to
 *     fp64; every entry point takes the element type as its last argument
 *     (ORACLE_BF16 or ORACLE_F16).
 *
 * Softmax is the usual two-pass, max-subtracted form, which equals the
 * equation above in exact arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element types of the 16-bit inputs. */
#define ORACLE_BF16 0
#define ORACLE_F16 1

typedef double (*widen_fn)(uint16_t bits);

/* Exact widening of a bf16 bit pattern to double: bf16 is the upper half of
 * an IEEE binary32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Exact widening of an IEEE binary16 bit pattern to double: 1 sign bit, a
 * 5-bit exponent with bias 15 and a 10-bit fraction.  Exponent 0 holds zero
 * and the subnormals (fraction x 2^-24); exponent 31 holds the infinities
 * (fraction 0) and NaN. */
static double f16_bits_to_double(uint16_t bits)
{
    int negative = (bits >> 15) & 1;
    int e = (bits >> 10) & 31;
    int f = bits & 1023;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) 2^(e-15) */
    return negative ? -mag : mag;
}

static widen_fn widen_for(int dtype)
{
    if (dtype == ORACLE_BF16) return bf16_bits_to_double;
    if (dtype == ORACLE_F16) return f16_bits_to_double;
    return 0;
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Membership of key position i in the attended set A(t) of query position t. */
int oracle_in_window(int64_t t, int64_t i, int64_t w, int64_t s)
{
    if (i < 0 || i > t) return 0;            /* causal: keys up to t only      */
    if (w < 0) return 1;                      /* w = infinity: full causal      */
    if (i < s) return 1;                      /* one of the first s tokens      */
    return i >= t - (w - s) + 1;              /* one of the latest w-s tokens   */
}

/*
 * Softmax attention of one query row over an explicit list of key rows.
 * q: d values; keys/vals: base pointers, row r of the list is at
 * keys + idx[r]*row_stride.  Writes out[d] and returns the log-sum-exp of the
 * scaled scores (natural log).
 */
static double attend_list(const uint16_t *q, const uint16_t *keys, const uint16_t *vals,
                          const int64_t *idx, int64_t n, int64_t row_stride, int d,
                          widen_fn widen, double *score, double *out)
{
    const double scale = 1.0 / sqrt((double)d);
    double m = -INFINITY;
    for (int64_t r = 0; r < n; ++r) {
        const uint16_t *k = keys + idx[r] * row_stride;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += widen(q[c]) * widen(k[c]);
        score[r] = dot * scale;
        if (score[r] > m) m = score[r];
    }
    double den = 0.0;
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    for (int64_t r = 0; r < n; ++r) {
        const uint16_t *v = vals + idx[r] * row_stride;
        double p = exp(score[r] - m);
        den += p;
        for (int c = 0; c < d; ++c) out[c] += p * widen(v[c]);
    }
    for (int c = 0; c < d; ++c) out[c] /= den;
    return m + log(den);
}

/* The attended positions of query position t, in increasing order. */
static int64_t window_indices(int64_t t, int64_t w, int64_t s, int64_t *idx)
{
    int64_t n = 0;
    if (w < 0) {
        for (int64_t i = 0; i <= t; ++i) idx[n++] = i;
        return n;
    }
    /* the first s tokens (those that exist by position t) */
    int64_t sink_end = s < t + 1 ? s : t + 1;
    for (int64_t i = 0; i < sink_end; ++i) idx[n++] = i;
    /* the latest w-s tokens; start at s so that a sink is not counted twice */
    int64_t lo = t - (w - s) + 1;
    if (lo < s) lo = s;
    for (int64_t i = lo; i <= t; ++i) idx[n++] = i;
    return n;
}

/*
 * One output row (b, t, h) of prefill.  q, k, v: 16-bit patterns, q [B,L,Hq,d],
 * k and v [B,L,Hkv,d].  o_row: d doubles.  Returns the row's log-sum-exp.
 * scratch_idx / scratch_score: room for L entries each.
 */
static double prefill_row(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t b, int64_t t, int64_t h, int64_t L, int64_t Hq,
                          int64_t Hkv, int d, int64_t w, int64_t s, widen_fn widen,
                          int64_t *scratch_idx, double *scratch_score, double *o_row)
{
    int64_t G = Hq / Hkv;
    int64_t kvh = h / G;
    int64_t n = window_indices(t, w, s, scratch_idx);
    const uint16_t *qrow = q + ((b * L + t) * Hq + h) * d;
    const uint16_t *kbase = k + (b * L * Hkv + kvh) * d;   /* position 0 of (b, kvh) */
    const uint16_t *vbase = v + (b * L * Hkv + kvh) * d;
    return attend_list(qrow, kbase, vbase, scratch_idx, n, Hkv * d, d, widen, scratch_score,
                       o_row);
}

/*
 * Full prefill: o [B,L,Hq,d] (double), lse [B,Hq,L] (double, may be NULL).
 * Work buffers: work_idx holds nthreads*L int64, work_score nthreads*L
 * doubles; nthreads >= 1 is the number of OpenMP threads used; dtype is
 * ORACLE_BF16 or ORACLE_F16.
 */
int oracle_swa_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       double *o, double *lse, int64_t B, int64_t L, int64_t Hq,
                       int64_t Hkv, int64_t d, int64_t w, int64_t s,
                       int64_t *work_idx, double *work_score, int nthreads, int dtype)
{
    widen_fn widen = widen_for(dtype);
    if (!widen || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    if (w >= 0 && w <= s) return -1;
    int64_t rows = B * L * Hq;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
    for (int64_t r = 0; r < rows; ++r) {
#ifdef _OPENMP
        int tid = omp_get_thread_num();
#else
        int tid = 0;
#endif
        int64_t h = r % Hq;
        int64_t t = (r / Hq) % L;
        int64_t b = r / (Hq * L);
        double ls = prefill_row(q, k, v, b, t, h, L, Hq, Hkv, (int)d, w, s, widen,
                                work_idx + (int64_t)tid * L, work_score + (int64_t)tid * L,
                                o + r * d);
        if (lse) lse[(b * Hq + h) * L + t] = ls;
    }
    return 0;
}

/*
 * Selected prefill rows.  rows: n triples (b, t, h).  o: n*d doubles,
 * lse: n doubles (may be NULL).  Work buffers as above.
 */
int oracle_swa_prefill_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int64_t *rows, int64_t n, double *o, double *lse,
                            int64_t B, int64_t L, int64_t Hq, int64_t Hkv, int64_t d,
                            int64_t w, int64_t s, int64_t *work_idx, double *work_score,
                            int nthreads, int dtype)
{
    widen_fn widen = widen_for(dtype);
    if (!widen || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    if (w >= 0 && w <= s) return -1;
    for (int64_t r = 0; r < n; ++r) {
        int64_t b = rows[3 * r], t = rows[3 * r + 1], h = rows[3 * r + 2];
        if (b < 0 || b >= B || t < 0 || t >= L || h < 0 || h >= Hq) return -1;
    }
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
    for (int64_t r = 0; r < n; ++r) {
#ifdef _OPENMP
        int tid = omp_get_thread_num();
#else
        int tid = 0;
#endif
        double ls = prefill_row(q, k, v, rows[3 * r], rows[3 * r + 1], rows[3 * r + 2], L, Hq,
                                Hkv, (int)d, w, s, widen, work_idx + (int64_t)tid * L,
                                work_score + (int64_t)tid * L, o + r * d);
        if (lse) lse[r] = ls;
    }
    return 0;
}

/*
 * Decode over the full history: the query of sequence b sits at position
 * pos[b] and attends to A(pos[b]) of k_hist/v_hist [B,P,Hkv,d] (P > pos[b]).
 * q [B,Hq,d], o [B,Hq,d] doubles.  Work buffers: nthreads * P entries each.
 */
int oracle_swa_decode(const uint16_t *q, const uint16_t *k_hist, const uint16_t *v_hist,
                      const int64_t *pos, double *o, int64_t B, int64_t P, int64_t Hq,
                      int64_t Hkv, int64_t d, int64_t w, int64_t s, int64_t *work_idx,
                      double *work_score, int nthreads, int dtype)
{
    widen_fn widen = widen_for(dtype);
    if (!widen || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    if (w >= 0 && w <= s) return -1;
    for (int64_t b = 0; b < B; ++b)
        if (pos[b] < 0 || pos[b] >= P) return -1;
    int64_t G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t r = 0; r < B * Hq; ++r) {
#ifdef _OPENMP
        int tid = omp_get_thread_num();
#else
        int tid = 0;
#endif
        int64_t b = r / Hq, h = r % Hq, kvh = h / G;
        int64_t *idx = work_idx + (int64_t)tid * P;
        int64_t n = window_indices(pos[b], w, s, idx);
        const uint16_t *kbase = k_hist + (b * P * Hkv + kvh) * d;
        const uint16_t *vbase = v_hist + (b * P * Hkv + kvh) * d;
        attend_list(q + r * d, kbase, vbase, idx, n, Hkv * d, (int)d, widen,
                    work_score + (int64_t)tid * P, o + r * d);
    }
    return 0;
}

/* Cache slot of position p: sinks keep their own slot, the rest share a ring. */
int64_t oracle_cache_slot(int64_t p, int64_t w, int64_t s)
{
    if (w < 0 || p < s) return p;
    return s + (p - s) % (w - s);
}

/*
 * Host simulation of appending positions pos0 .. pos0+n-1 to a cache.
 * cache_k, cache_v: [B,Hkv,cap,d] 16-bit patterns (copied, whatever their
 * type); k_new, v_new: [B,n,Hkv,d].
 * Positions are written one after the other, so where two positions share a
 * slot the later one is what remains.  Returns -1 if a slot falls outside cap.
 */
int oracle_cache_append(uint16_t *cache_k, uint16_t *cache_v, const uint16_t *k_new,
                        const uint16_t *v_new, int64_t B, int64_t Hkv, int64_t d, int64_t cap,
                        int64_t w, int64_t s, int64_t n, int64_t pos0)
{
    for (int64_t b = 0; b < B; ++b)
        for (int64_t j = 0; j < n; ++j) {
            int64_t slot = oracle_cache_slot(pos0 + j, w, s);
            if (slot < 0 || slot >= cap) return -1;
            for (int64_t h = 0; h < Hkv; ++h) {
                const uint16_t *ks = k_new + ((b * n + j) * Hkv + h) * d;
                const uint16_t *vs = v_new + ((b * n + j) * Hkv + h) * d;
                uint16_t *kd = cache_k + ((b * Hkv + h) * cap + slot) * d;
                uint16_t *vd = cache_v + ((b * Hkv + h) * cap + slot) * d;
                memcpy(kd, ks, (size_t)d * sizeof(uint16_t));
                memcpy(vd, vs, (size_t)d * sizeof(uint16_t));
            }
        }
    return 0;
}

/*
 * Decode over the cache contents: attention of q over the filled slots
 * [0, min(pos+1, cap_eff)) of each (b, kv head), cap_eff = w (or cap for
 * w = infinity).  Slot order is not position order; the softmax over a set
 * does not depend on the order, so this equals oracle_swa_decode on the same
 * history.  Work buffers: nthreads * cap entries each.
 */
int oracle_swa_decode_cache(const uint16_t *q, const uint16_t *cache_k, const uint16_t *cache_v,
                            const int64_t *pos, double *o, int64_t B, int64_t Hq, int64_t Hkv,
                            int64_t d, int64_t cap, int64_t w, int64_t s, int64_t *work_idx,
                            double *work_score, int nthreads, int dtype)
{
    widen_fn widen = widen_for(dtype);
    if (!widen || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    if (w >= 0 && (w <= s || w > cap)) return -1;
    int64_t G = Hq / Hkv;
    int64_t cap_eff = w < 0 ? cap : w;
    for (int64_t b = 0; b < B; ++b)
        if (pos[b] < 0 || (w < 0 && pos[b] >= cap)) return -1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t r = 0; r < B * Hq; ++r) {
#ifdef _OPENMP
        int tid = omp_get_thread_num();
#else
        int tid = 0;
#endif
        int64_t b = r / Hq, h = r % Hq, kvh = h / G;
        int64_t n = pos[b] + 1 < cap_eff ? pos[b] + 1 : cap_eff;
        int64_t *idx = work_idx + (int64_t)tid * cap;
        for (int64_t i = 0; i < n; ++i) idx[i] = i;
        const uint16_t *kbase = cache_k + (b * Hkv + kvh) * cap * d;
        const uint16_t *vbase = cache_v + (b * Hkv + kvh) * cap * d;
        attend_list(q + r * d, kbase, vbase, idx, n, d, (int)d, widen,
                    work_score + (int64_t)tid * cap, o + r * d);
    }
    return 0;
}


/*
 * Hybrid window + linear attention (LoLCATs-style; NEXT of the scope).
 *
 * Linear attention -- "Sliding-window beats linear attention" (paper summary
 * page), section "Prerequisites / Linear attention": a feature map phi
 * replaces exp(q k^T) by phi(q) phi(k)^T, and the output of query t is
 * phi(q_t) s_t / (phi(q_t) z_t) with s_t = sum_i phi(k_i)^T v_i and
 * z_t = sum_i phi(k_i)^T.  Feature map -- same page, section "Post-training
 * linearisation and LoLCATs": the Hedgehog map phi(x) = (exp(f(x)),
 * exp(-f(x))), mixed with a sliding window.
 *
 * Readings (the pages give no formula for the mixture): f(x) = x W with W a
 * d x df matrix per key/value head (synthetic: an input, no training), so
 * phi(x) has F = 2 df features; the softmax part covers the attended set
 * A(t) of SWA(w,s) and the linear part every earlier position outside it
 * (the tokens the fixed cache has evicted), with one shared normaliser:
 *
 *   y_t = ( sum_{i in A(t)} exp(c q.k_i) v_i + sum_{i <= t, i not in A(t)} phi(q).phi(k_i) v_i )
 *       / ( sum_{i in A(t)} exp(c q.k_i)     + sum_{i <= t, i not in A(t)} phi(q).phi(k_i) ).
 *
 * This is the direct sum; the library keeps the running state instead.
 */

/* phi(x) for one row x of d 16-bit values: out[0..df) = exp(f), out[df..2df) = exp(-f). */
static void hedgehog_phi(const uint16_t *x, const double *W, int d, int df, widen_fn widen,
                         double *out)
{
    for (int j = 0; j < df; ++j) {
        double f = 0.0;
        for (int c = 0; c < d; ++c) f += widen(x[c]) * W[(int64_t)c * df + j];
        out[j] = exp(f);
        out[df + j] = exp(-f);
    }
}

/*
 * Hybrid decode over the full history: q [B,Hq,d], k_hist/v_hist [B,P,Hkv,d]
 * (16-bit patterns), W [Hkv,d,df] doubles, pos [B] (< P), o [B,Hq,d]
 * doubles.  Work buffers: nthreads * (P + 2*F) doubles and nthreads * P
 * indices.
 */
int oracle_hybrid_decode(const uint16_t *q, const uint16_t *k_hist, const uint16_t *v_hist,
                         const double *W, const int64_t *pos, double *o, int64_t B, int64_t P,
                         int64_t Hq, int64_t Hkv, int64_t d, int64_t df, int64_t w, int64_t s,
                         int64_t *work_idx, double *work, int nthreads, int dtype)
{
    widen_fn widen = widen_for(dtype);
    if (!widen || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || df <= 0) return -1;
    if (w >= 0 && w <= s) return -1;
    for (int64_t b = 0; b < B; ++b)
        if (pos[b] < 0 || pos[b] >= P) return -1;
    const int64_t G = Hq / Hkv, F = 2 * df;
    const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t r = 0; r < B * Hq; ++r) {
#ifdef _OPENMP
        int tid = omp_get_thread_num();
#else
        int tid = 0;
#endif
        const int64_t b = r / Hq, h = r % Hq, kvh = h / G, t = pos[b];
        int64_t *idx = work_idx + (int64_t)tid * P;
        double *score = work + (int64_t)tid * (P + 2 * F);
        double *phq = score + P, *phk = phq + F;
        const double *Wh = W + kvh * d * df;
        const uint16_t *qrow = q + r * d;
        const int64_t n = window_indices(t, w, s, idx);
        /* softmax part over A(t), max-subtracted */
        double m = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            const uint16_t *kr = k_hist + ((b * P + idx[i]) * Hkv + kvh) * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += widen(qrow[c]) * widen(kr[c]);
            score[i] = dot * scale;
            if (score[i] > m) m = score[i];
        }
        double *out = o + r * d;
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        double den = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            const uint16_t *vr = v_hist + ((b * P + idx[i]) * Hkv + kvh) * d;
            const double p = exp(score[i] - m);
            den += p;
            for (int c = 0; c < d; ++c) out[c] += p * widen(vr[c]);
        }
        /* linear part over the earlier positions outside A(t), scaled by e^-m */
        hedgehog_phi(qrow, Wh, (int)d, (int)df, widen, phq);
        const double em = exp(-m);
        for (int64_t i = 0; i <= t; ++i) {
            if (oracle_in_window(t, i, w, s)) continue;
            const uint16_t *kr = k_hist + ((b * P + i) * Hkv + kvh) * d;
            const uint16_t *vr = v_hist + ((b * P + i) * Hkv + kvh) * d;
            hedgehog_phi(kr, Wh, (int)d, (int)df, widen, phk);
            double wt = 0.0;
            for (int64_t f = 0; f < F; ++f) wt += phq[f] * phk[f];
            den += em * wt;
            for (int c = 0; c < d; ++c) out[c] += em * wt * widen(vr[c]);
        }
        for (int c = 0; c < d; ++c) out[c] /= den;
    }
    return 0;
}

/*
 * The linear state after positions 0 .. P-1 have been appended to an SWA(w,s)
 * cache: S [B,Hkv,F,d] = sum over evicted positions i of phi(k_i)^T v_i and
 * z [B,Hkv,F] = sum of phi(k_i), evicted = s <= i <= P-1-(w-s) (nothing for
 * w = infinity).  k_hist/v_hist [B,P,Hkv,d] 16-bit patterns, W [Hkv,d,df].
 */
int oracle_hybrid_state(const uint16_t *k_hist, const uint16_t *v_hist, const double *W,
                        double *S, double *z, int64_t B, int64_t P, int64_t Hkv, int64_t d,
                        int64_t df, int64_t w, int64_t s, double *work, int nthreads, int dtype)
{
    widen_fn widen = widen_for(dtype);
    if (!widen || Hkv <= 0 || d <= 0 || df <= 0) return -1;
    if (w >= 0 && w <= s) return -1;
    const int64_t F = 2 * df;
    const int64_t last = w < 0 ? -1 : P - 1 - (w - s); /* last evicted position */
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t r = 0; r < B * Hkv; ++r) {
#ifdef _OPENMP
        int tid = omp_get_thread_num();
#else
        int tid = 0;
#endif
        const int64_t b = r / Hkv, kvh = r % Hkv;
        double *phk = work + (int64_t)tid * F;
        double *Sr = S + r * F * d, *zr = z + r * F;
        for (int64_t i = 0; i < F * d; ++i) Sr[i] = 0.0;
        for (int64_t f = 0; f < F; ++f) zr[f] = 0.0;
        for (int64_t i = s; i <= last; ++i) {
            const uint16_t *kr = k_hist + ((b * P + i) * Hkv + kvh) * d;
            const uint16_t *vr = v_hist + ((b * P + i) * Hkv + kvh) * d;
            hedgehog_phi(kr, W + kvh * d * df, (int)d, (int)df, widen, phk);
            for (int64_t f = 0; f < F; ++f) {
                zr[f] += phk[f];
                for (int c = 0; c < d; ++c) Sr[f * d + c] += phk[f] * widen(vr[c]);
            }
        }
    }
    return 0;
}
