/*
 * Paged-KV GQA/MQA attention: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file defines what the CUDA path must
 * compute, written as the plain definition, slowly and in double precision.
 * It shares no source, header, table or helper with the CUDA library, and
 * nothing in the library links it.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it.
 *
 * Sources (web pages on the subject):
 *  - vLLM issue #1880, "[Performance] Use optimized kernels for MQA/GQA",
 *    item 1 (prefill): grouped-query attention is computed as plain
 *    multi-head attention after each KV head's keys and values are expanded
 *    (broadcast) to the G = Hq / Hkv query heads that share it, i.e. the
 *    tensor [T, Hkv, D] becomes [T, Hkv, G, D] and is flattened to
 *    [T, Hq, D].  Query head h therefore reads KV head h / G.
 *  - same issue, item 2 (decode): attention over a paged KV cache, where a
 *    block table maps a sequence's logical blocks to physical cache blocks.
 *  - vLLM PR #14431, "[Kernel][V1] Further optimizations to ROCm (Triton)
 *    Backend to better handle GQA", opening post and review thread: one
 *    batch mixes sequences with a query chunk (query length > 1, chunked
 *    prefill over a cached prefix) and decode sequences (query length 1).
 *
 * Readings taken where the pages are silent (all fixed here, stated once):
 *  - cache layout: k_cache and v_cache are both [NB, Hkv, bs, D];
 *  - context_lens[b] counts every token of sequence b in the cache, including
 *    this step's query tokens, which reshape_and_cache has already written;
 *  - causal alignment is bottom-right: query token t of a chunk of qlen
 *    tokens sits at absolute position p = ctx - qlen + t and sees keys 0..p;
 *    a decode row is the case qlen = 1 (p = ctx - 1, all keys);
 *  - softmax base e over scale * q.k; no soft-cap, bias or window;
 *  - a sequence with no key gives a zero output row (and lse = -inf);
 *  - the output is the fp64 result rounded to nearest-even into the element
 *    type;
 *  - split-KV partitions cut the sequence's blocks into S ranges of
 *    ceil(nb / S) blocks; each range gives a normalised partial output and
 *    the natural-log log-sum-exp of its scaled logits; empty ranges give
 *    lse = -inf and weight 0 in the combine.
 *
 * Element types: 0 = IEEE binary16, 1 = bfloat16; buffers carry raw uint16
 * bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F16 0
#define ORC_BF16 1

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_BLOCK (-2)
#define ORC_ERR_SLOT (-3)
#define ORC_ERR_MEM (-4)

/* ---------------------------------------------------------------------- */
/* Element decoding and rounding (IEEE 754 definitions, written out).      */
/* ---------------------------------------------------------------------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double orc_f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + f, e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the top 16 bits of an IEEE binary32. */
static double orc_bf16_value(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133); /* subnormal: f * 2^-126 * 2^-7 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(128.0 + f, e - 134); /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

static double orc_value(uint16_t bits, int dtype)
{
    return dtype == ORC_F16 ? orc_f16_value(bits) : orc_bf16_value(bits);
}

/*
 * Round x to the nearest value of a binary format with p significand bits
 * (implicit bit included), minimum normal exponent emin and maximum exponent
 * emax; ties go to the even significand.  Returns the rounded value (which
 * may be +-inf on overflow).
 */
static double orc_round_format(double x, int p, int emin, int emax)
{
    if (isnan(x) || isinf(x) || x == 0.0)
        return x;
    int e2;
    frexp(fabs(x), &e2);          /* |x| = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;               /* |x| in [2^E, 2^(E+1)) */
    if (E < emin)
        E = emin;                 /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, E - (p - 1));
    double r = nearbyint(x / quantum) * quantum; /* default mode: ties-to-even */
    double maxfin = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(r) > maxfin)
        return x > 0 ? INFINITY : -INFINITY;
    return r;
}

/* Encode a value that is exactly representable in the format into bits. */
static uint16_t orc_encode(double r, int dtype)
{
    int mant_bits = dtype == ORC_F16 ? 10 : 7;
    int ebits = dtype == ORC_F16 ? 5 : 8;
    int bias = (1 << (ebits - 1)) - 1;
    int emax_field = (1 << ebits) - 1;
    uint16_t sign = signbit(r) ? (uint16_t)(1u << 15) : 0;
    if (isnan(r))
        return (uint16_t)((emax_field << mant_bits) | (1u << (mant_bits - 1)));
    if (isinf(r))
        return (uint16_t)(sign | (emax_field << mant_bits));
    double a = fabs(r);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;
    int emin = 1 - bias;
    if (E < emin) { /* subnormal: a = f * 2^(emin - mant_bits) */
        uint32_t f = (uint32_t)ldexp(a, mant_bits - emin);
        return (uint16_t)(sign | f);
    }
    uint32_t f = (uint32_t)(ldexp(a, mant_bits - E) - ldexp(1.0, mant_bits));
    return (uint16_t)(sign | ((uint32_t)(E + bias) << mant_bits) | f);
}

double orc_round_to_dtype(double x, int dtype)
{
    if (dtype == ORC_F16)
        return orc_round_format(x, 11, -14, 15);
    return orc_round_format(x, 8, -126, 127);
}

uint16_t orc_to_bits(double x, int dtype)
{
    return orc_encode(orc_round_to_dtype(x, dtype), dtype);
}

double orc_from_bits(uint16_t bits, int dtype)
{
    return orc_value(bits, dtype);
}

/* Vector forms for the tests. */
void orc_to_bits_n(const double* x, int64_t n, int dtype, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_to_bits(x[i], dtype);
}

void orc_from_bits_n(const uint16_t* b, int64_t n, int dtype, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_value(b[i], dtype);
}

/* ---------------------------------------------------------------------- */
/* reshape_and_cache: write this step's K/V rows into their cache slots.   */
/* ---------------------------------------------------------------------- */

/*
 * k, v:        [T, Hkv, D] element bits
 * k_cache/v_cache: [NB, Hkv, bs, D] element bits, updated in place
 * slot_mapping: [T]; slot = block * bs + offset; -1 skips the token.
 * Returns ORC_ERR_SLOT (and writes nothing) if any slot is out of range.
 */
int orc_reshape_and_cache(const uint16_t* k, const uint16_t* v,
                          uint16_t* k_cache, uint16_t* v_cache,
                          const int64_t* slot_mapping, int64_t T, int Hkv,
                          int D, int bs, int64_t NB)
{
    if (T < 0 || Hkv <= 0 || D <= 0 || bs <= 0 || NB < 0)
        return ORC_ERR_ARG;
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slot_mapping[t];
        if (s < -1 || s >= NB * (int64_t)bs)
            return ORC_ERR_SLOT;
    }
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        int64_t blk = s / bs, off = s % bs;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t src = ((t * Hkv) + h) * (int64_t)D + d;
                int64_t dst = (((blk * Hkv) + h) * (int64_t)bs + off) * D + d;
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
        }
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Attention over the paged cache.                                         */
/* ---------------------------------------------------------------------- */

typedef struct {
    const uint16_t* q;            /* [Tq, Hq, D] */
    const uint16_t* k_cache;      /* [NB, Hkv, bs, D] */
    const uint16_t* v_cache;
    const int32_t* block_tables;  /* [B, mbs] */
    const int32_t* cu_query_lens; /* [B+1] */
    const int32_t* context_lens;  /* [B] */
    int mbs, B, Hq, Hkv, D, bs, dtype;
    int64_t NB;
    double scale;
} orc_problem;

/* Sequence that owns query token row `tok` (cu_query_lens is non-decreasing). */
static int orc_seq_of_token(const orc_problem* P, int64_t tok)
{
    int lo = 0, hi = P->B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (P->cu_query_lens[mid] <= tok)
            lo = mid;
        else
            hi = mid - 1;
    }
    while (lo < P->B - 1 && P->cu_query_lens[lo + 1] <= tok)
        ++lo; /* skip sequences with no query tokens */
    return lo;
}

/*
 * Gather sequence b's keys and values through its block table and expand
 * them to query head h: Kh[j][d] = K[j][h / G][d] for j < n.  This is the
 * per-query-head expansion of the MQA/GQA issue, materialised one query head
 * at a time (the full [ctx, Hq, D] copy is the same numbers, repeated).
 */
static int orc_gather_expanded(const orc_problem* P, int b, int h, int n,
                               double* Kh, double* Vh)
{
    int G = P->Hq / P->Hkv;
    int kvh = h / G;
    for (int j = 0; j < n; ++j) {
        int32_t blk = P->block_tables[(int64_t)b * P->mbs + j / P->bs];
        if (blk < 0 || blk >= P->NB)
            return ORC_ERR_BLOCK;
        int64_t base = (((int64_t)blk * P->Hkv + kvh) * P->bs + j % P->bs) * P->D;
        for (int d = 0; d < P->D; ++d) {
            Kh[(int64_t)j * P->D + d] = orc_value(P->k_cache[base + d], P->dtype);
            Vh[(int64_t)j * P->D + d] = orc_value(P->v_cache[base + d], P->dtype);
        }
    }
    return ORC_OK;
}

/*
 * Softmax attention of one query vector over keys [j0, j1) of the expanded
 * head: s_j = scale * q . k_j, o = sum_j e^(s_j - m) v_j / sum_j e^(s_j - m).
 * Writes o (D values) and returns the natural-log log-sum-exp of the s_j
 * (-inf, with o = 0, when the range is empty).
 */
static double orc_softmax_attend(const double* qv, const double* Kh,
                                 const double* Vh, int j0, int j1, int D,
                                 double scale, double* s, double* o)
{
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (j1 <= j0)
        return -INFINITY;
    double m = -INFINITY;
    for (int j = j0; j < j1; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qv[d] * Kh[(int64_t)j * D + d];
        s[j - j0] = scale * dot;
        if (s[j - j0] > m)
            m = s[j - j0];
    }
    double l = 0.0;
    for (int j = j0; j < j1; ++j) {
        double w = exp(s[j - j0] - m);
        l += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * Vh[(int64_t)j * D + d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= l;
    return m + log(l);
}

static int orc_check(const orc_problem* P)
{
    if (!P->q || !P->k_cache || !P->v_cache || !P->block_tables ||
        !P->cu_query_lens || !P->context_lens)
        return ORC_ERR_ARG;
    if (P->B < 0 || P->Hq <= 0 || P->Hkv <= 0 || P->Hq % P->Hkv || P->D <= 0 ||
        P->bs <= 0 || P->mbs < 0 || (P->dtype != ORC_F16 && P->dtype != ORC_BF16))
        return ORC_ERR_ARG;
    if (P->B > 0 && P->cu_query_lens[0] != 0)
        return ORC_ERR_ARG;
    for (int b = 0; b < P->B; ++b) {
        int ql = P->cu_query_lens[b + 1] - P->cu_query_lens[b];
        int ctx = P->context_lens[b];
        /* a sequence with no cached key may still carry query rows: they
         * read nothing and are zero */
        if (ql < 0 || ctx < 0 || (ctx < ql && ctx != 0) || ctx > P->mbs * P->bs)
            return ORC_ERR_ARG;
    }
    return ORC_OK;
}

/*
 * Attention for selected query-token rows (all Hq heads of each row).
 *
 * rows:   query-token indices into q (NULL: all Tq = cu_query_lens[B] rows)
 * out64:  [n_rows, Hq, D] fp64 results
 * out_bits: [n_rows, Hq, D] results rounded into the element type, or NULL
 * num_splits: 0 or 1 = one range over all keys; S > 1 = compute the S
 *   split-KV partials of each row (part_o [n_rows, Hq, S, D] and
 *   part_lse [n_rows, Hq, S], each may be NULL) and still write the unsplit
 *   result to out64/out_bits.
 */
int orc_paged_attention(const uint16_t* q, const uint16_t* k_cache,
                        const uint16_t* v_cache, const int32_t* block_tables,
                        int mbs, const int32_t* cu_query_lens,
                        const int32_t* context_lens, double scale, int B,
                        int Hq, int Hkv, int D, int bs, int64_t NB, int dtype,
                        const int64_t* rows, int64_t n_rows, double* out64,
                        uint16_t* out_bits, int num_splits, double* part_o,
                        double* part_lse, int num_threads)
{
    orc_problem P = {q, k_cache, v_cache, block_tables, cu_query_lens,
                     context_lens, mbs, B, Hq, Hkv, D, bs, dtype, NB, scale};
    int rc = orc_check(&P);
    if (rc != ORC_OK)
        return rc;
    int64_t Tq = B > 0 ? cu_query_lens[B] : 0;
    if (!rows)
        n_rows = Tq;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t tok = rows ? rows[r] : r;
        if (tok < 0 || tok >= Tq)
            return ORC_ERR_ARG;
    }
    int S = num_splits > 1 ? num_splits : 1;

    /* One work item per (selected row, query head); each gathers and expands
     * its own head's keys and values. */
    int64_t n_items = n_rows * Hq;
    int err = ORC_OK;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
    {
        int cap = 0;
        double *Kh = NULL, *Vh = NULL, *s = NULL;
        double* qv = (double*)malloc(sizeof(double) * (size_t)D);
        double* o = (double*)malloc(sizeof(double) * (size_t)D);
        double* op = (double*)malloc(sizeof(double) * (size_t)D);
        if (!qv || !o || !op) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = ORC_ERR_MEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t it = 0; it < n_items; ++it) {
            if (err != ORC_OK)
                continue;
            int64_t r = it / Hq;
            int h = (int)(it % Hq);
            int64_t tok = rows ? rows[r] : r;
            int b = orc_seq_of_token(&P, tok);
            int qlen = cu_query_lens[b + 1] - cu_query_lens[b];
            int ctx = context_lens[b];
            int t = (int)(tok - cu_query_lens[b]);
            int p = ctx - qlen + t; /* absolute position of this query token */
            int n = p + 1;          /* keys 0..p are visible */
            if (ctx == 0) {         /* no key at all: zero row, empty splits */
                int64_t zb = (r * Hq + h) * (int64_t)D;
                for (int d = 0; d < D; ++d) {
                    out64[zb + d] = 0.0;
                    if (out_bits)
                        out_bits[zb + d] = 0;
                }
                if (S > 1 && (part_o || part_lse))
                    for (int sp = 0; sp < S; ++sp) {
                        int64_t pi = (r * Hq + h) * (int64_t)S + sp;
                        if (part_lse)
                            part_lse[pi] = -INFINITY;
                        if (part_o)
                            for (int d = 0; d < D; ++d)
                                part_o[pi * D + d] = 0.0;
                    }
                continue;
            }
            if (n > cap) {
                free(Kh); free(Vh); free(s);
                cap = n;
                Kh = (double*)malloc(sizeof(double) * (size_t)cap * D);
                Vh = (double*)malloc(sizeof(double) * (size_t)cap * D);
                s = (double*)malloc(sizeof(double) * (size_t)cap);
                if (!Kh || !Vh || !s) {
#ifdef _OPENMP
#pragma omp critical
#endif
                    err = ORC_ERR_MEM;
                    cap = 0;
                    continue;
                }
            }
            int grc = orc_gather_expanded(&P, b, h, n, Kh, Vh);
            if (grc != ORC_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
                err = grc;
                continue;
            }
            for (int d = 0; d < D; ++d)
                qv[d] = orc_value(q[(tok * Hq + h) * (int64_t)D + d], dtype);

            orc_softmax_attend(qv, Kh, Vh, 0, n, D, scale, s, o);
            int64_t ob = (r * Hq + h) * (int64_t)D;
            for (int d = 0; d < D; ++d) {
                out64[ob + d] = o[d];
                if (out_bits)
                    out_bits[ob + d] = orc_to_bits(o[d], dtype);
            }
            if (S > 1 && (part_o || part_lse)) {
                int nb = (ctx + bs - 1) / bs;
                int per = (nb + S - 1) / S; /* blocks per split */
                for (int sp = 0; sp < S; ++sp) {
                    int j0 = sp * per * bs;
                    int j1 = (sp + 1) * per * bs;
                    if (j0 > n) j0 = n;
                    if (j1 > n) j1 = n;
                    double lse = orc_softmax_attend(qv, Kh, Vh, j0, j1, D,
                                                    scale, s, op);
                    int64_t pi = (r * Hq + h) * (int64_t)S + sp;
                    if (part_lse)
                        part_lse[pi] = lse;
                    if (part_o)
                        for (int d = 0; d < D; ++d)
                            part_o[pi * D + d] = op[d];
                }
            }
        }
        free(Kh); free(Vh); free(s); free(qv); free(o); free(op);
    }
    return err;
}

/*
 * Cross-attention over a static paged cache, for selected query rows.
 *
 * vLLM PR #7448, "[Core] More-efficient cross-attention parallel QKV
 * computation", opening post: in a cross-attention layer Q comes from the
 * decoder's hidden states and K, V from the encoder output; during decode
 * only Q is new, because the encoder sequence is static.  Reading taken
 * (the page does not spell out the mask): encoder-decoder attention has no
 * causal mask, so every query row of sequence b attends to all
 * context_lens[b] cached encoder keys, whatever its position among the
 * sequence's query rows, and a sequence may carry more query rows than
 * keys.  The cache, block tables, head map (h / G), scale, empty-context
 * rule (a zero row) and output rounding are those of orc_paged_attention.
 *
 * rows, out64, out_bits: as for orc_paged_attention.
 */
int orc_cross_attention(const uint16_t* q, const uint16_t* k_cache,
                        const uint16_t* v_cache, const int32_t* block_tables,
                        int mbs, const int32_t* cu_query_lens,
                        const int32_t* context_lens, double scale, int B,
                        int Hq, int Hkv, int D, int bs, int64_t NB, int dtype,
                        const int64_t* rows, int64_t n_rows, double* out64,
                        uint16_t* out_bits, int num_threads)
{
    orc_problem P = {q, k_cache, v_cache, block_tables, cu_query_lens,
                     context_lens, mbs, B, Hq, Hkv, D, bs, dtype, NB, scale};
    if (!q || !k_cache || !v_cache || !block_tables || !cu_query_lens ||
        !context_lens || !out64)
        return ORC_ERR_ARG;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || bs <= 0 ||
        mbs < 0 || (dtype != ORC_F16 && dtype != ORC_BF16))
        return ORC_ERR_ARG;
    if (B > 0 && cu_query_lens[0] != 0)
        return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int ql = cu_query_lens[b + 1] - cu_query_lens[b];
        int ctx = context_lens[b];
        if (ql < 0 || ctx < 0 || ctx > mbs * bs) /* no ql <= ctx rule here */
            return ORC_ERR_ARG;
    }
    int64_t Tq = B > 0 ? cu_query_lens[B] : 0;
    if (!rows)
        n_rows = Tq;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t tok = rows ? rows[r] : r;
        if (tok < 0 || tok >= Tq)
            return ORC_ERR_ARG;
    }

    int64_t n_items = n_rows * Hq;
    int err = ORC_OK;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
    {
        int cap = 0;
        double *Kh = NULL, *Vh = NULL, *s = NULL;
        double* qv = (double*)malloc(sizeof(double) * (size_t)D);
        double* o = (double*)malloc(sizeof(double) * (size_t)D);
        if (!qv || !o) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = ORC_ERR_MEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t it = 0; it < n_items; ++it) {
            if (err != ORC_OK)
                continue;
            int64_t r = it / Hq;
            int h = (int)(it % Hq);
            int64_t tok = rows ? rows[r] : r;
            int b = orc_seq_of_token(&P, tok);
            int n = context_lens[b]; /* every encoder key is visible */
            int64_t ob = (r * Hq + h) * (int64_t)D;
            if (n == 0) {
                for (int d = 0; d < D; ++d) {
                    out64[ob + d] = 0.0;
                    if (out_bits)
                        out_bits[ob + d] = 0;
                }
                continue;
            }
            if (n > cap) {
                free(Kh); free(Vh); free(s);
                cap = n;
                Kh = (double*)malloc(sizeof(double) * (size_t)cap * D);
                Vh = (double*)malloc(sizeof(double) * (size_t)cap * D);
                s = (double*)malloc(sizeof(double) * (size_t)cap);
                if (!Kh || !Vh || !s) {
#ifdef _OPENMP
#pragma omp critical
#endif
                    err = ORC_ERR_MEM;
                    cap = 0;
                    continue;
                }
            }
            int grc = orc_gather_expanded(&P, b, h, n, Kh, Vh);
            if (grc != ORC_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
                err = grc;
                continue;
            }
            for (int d = 0; d < D; ++d)
                qv[d] = orc_value(q[(tok * Hq + h) * (int64_t)D + d], dtype);
            orc_softmax_attend(qv, Kh, Vh, 0, n, D, scale, s, o);
            for (int d = 0; d < D; ++d) {
                out64[ob + d] = o[d];
                if (out_bits)
                    out_bits[ob + d] = orc_to_bits(o[d], dtype);
            }
        }
        free(Kh); free(Vh); free(s); free(qv); free(o);
    }
    return err;
}

/*
 * GQA prefill over contiguous (not paged) keys and values of a varlen batch.
 *
 * vLLM issue #1880, "[Performance] Use optimized kernels for MQA/GQA",
 * item 1: for prefill the incoming keys and values [T, Hkv, D] are expanded
 * to [T, Hkv, G, D] (a broadcast of each KV head to its G query heads) and
 * handed to a multi-head attention op.  That is the definition computed
 * here, literally: the batch holds B sequences whose query rows are
 * q[cu_q[b] .. cu_q[b+1]) and whose key/value rows are
 * k, v[cu_k[b] .. cu_k[b+1]); each KV row is expanded to the Hq heads (head
 * h reads KV head h / G) and every query row attends, causally, to its own
 * sequence's keys.  Causal alignment as in orc_paged_attention
 * (bottom-right: with klen keys and qlen query rows, query row t sits at
 * position klen - qlen + t and sees keys 0..that); klen >= qlen.  With
 * cu_q == cu_k this is plain causal self-attention over each prompt.
 *
 * rows, out64, out_bits: as for orc_paged_attention (rows index q).
 */
int orc_varlen_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* cu_q, const int32_t* cu_k, double scale,
                         int B, int Hq, int Hkv, int D, int dtype,
                         const int64_t* rows, int64_t n_rows, double* out64,
                         uint16_t* out_bits, int num_threads)
{
    if (!q || !k || !v || !cu_q || !cu_k || !out64)
        return ORC_ERR_ARG;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 ||
        (dtype != ORC_F16 && dtype != ORC_BF16))
        return ORC_ERR_ARG;
    if (B > 0 && (cu_q[0] != 0 || cu_k[0] != 0))
        return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int ql = cu_q[b + 1] - cu_q[b], kl = cu_k[b + 1] - cu_k[b];
        if (ql < 0 || kl < ql)
            return ORC_ERR_ARG;
    }
    int64_t Tq = B > 0 ? cu_q[B] : 0;
    if (!rows)
        n_rows = Tq;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t tok = rows ? rows[r] : r;
        if (tok < 0 || tok >= Tq)
            return ORC_ERR_ARG;
    }
    const int G = Hq / Hkv;
    int64_t n_items = n_rows * Hq;
    int err = ORC_OK;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
    {
        int cap = 0;
        double *Kh = NULL, *Vh = NULL, *s = NULL;
        double* qv = (double*)malloc(sizeof(double) * (size_t)D);
        double* o = (double*)malloc(sizeof(double) * (size_t)D);
        if (!qv || !o) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = ORC_ERR_MEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t it = 0; it < n_items; ++it) {
            if (err != ORC_OK)
                continue;
            int64_t r = it / Hq;
            int h = (int)(it % Hq);
            int64_t tok = rows ? rows[r] : r;
            int b = 0; /* sequence owning query row tok */
            while (b < B - 1 && cu_q[b + 1] <= tok)
                ++b;
            int qlen = cu_q[b + 1] - cu_q[b], klen = cu_k[b + 1] - cu_k[b];
            int n = klen - qlen + (int)(tok - cu_q[b]) + 1; /* keys 0..position */
            if (n > cap) {
                free(Kh); free(Vh); free(s);
                cap = n;
                Kh = (double*)malloc(sizeof(double) * (size_t)cap * D);
                Vh = (double*)malloc(sizeof(double) * (size_t)cap * D);
                s = (double*)malloc(sizeof(double) * (size_t)cap);
                if (!Kh || !Vh || !s) {
#ifdef _OPENMP
#pragma omp critical
#endif
                    err = ORC_ERR_MEM;
                    cap = 0;
                    continue;
                }
            }
            /* the expansion: query head h reads KV head h / G of each row */
            for (int j = 0; j < n; ++j) {
                int64_t src = ((int64_t)(cu_k[b] + j) * Hkv + h / G) * D;
                for (int d = 0; d < D; ++d) {
                    Kh[(int64_t)j * D + d] = orc_value(k[src + d], dtype);
                    Vh[(int64_t)j * D + d] = orc_value(v[src + d], dtype);
                }
            }
            for (int d = 0; d < D; ++d)
                qv[d] = orc_value(q[(tok * Hq + h) * (int64_t)D + d], dtype);
            orc_softmax_attend(qv, Kh, Vh, 0, n, D, scale, s, o);
            int64_t ob = (r * Hq + h) * (int64_t)D;
            for (int d = 0; d < D; ++d) {
                out64[ob + d] = o[d];
                if (out_bits)
                    out_bits[ob + d] = orc_to_bits(o[d], dtype);
            }
        }
        free(Kh); free(Vh); free(s); free(qv); free(o);
    }
    return err;
}

/*
 * Log-sum-exp combine of S split partials, for n rows of D values:
 *   M = max_s lse_s,  w_s = e^(lse_s - M),  out = sum_s w_s o_s / sum_s w_s.
 * Partials with lse = -inf carry weight 0; a row whose partials are all
 * empty is zero.
 */
void orc_lse_combine(const double* part_o, const double* part_lse, int64_t n,
                     int S, int D, double* out)
{
    for (int64_t i = 0; i < n; ++i) {
        double M = -INFINITY;
        for (int s = 0; s < S; ++s)
            if (part_lse[i * S + s] > M)
                M = part_lse[i * S + s];
        for (int d = 0; d < D; ++d)
            out[i * D + d] = 0.0;
        if (M == -INFINITY)
            continue;
        double wsum = 0.0;
        for (int s = 0; s < S; ++s) {
            double lse = part_lse[i * S + s];
            if (lse == -INFINITY)
                continue;
            double w = exp(lse - M);
            wsum += w;
            for (int d = 0; d < D; ++d)
                out[i * D + d] += w * part_o[(i * S + s) * D + d];
        }
        for (int d = 0; d < D; ++d)
            out[i * D + d] /= wsum;
    }
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
