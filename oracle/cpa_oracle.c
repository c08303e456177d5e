/*
 * cpa_oracle.c -- plain, slow, fp64 CPU oracle for paged chunked-prefill
 * attention.  TEST INFRASTRUCTURE ONLY: nothing on the product path links,
 * loads or calls this file; only the tests, the smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (sources, cited by page title and section):
 *
 *  - "Prefill Processing" (AWS Neuron vLLM design doc), "Key Concepts" and
 *    "How Segmentation Works with KV Segments": each active token of a
 *    request attends to all cached_seq_len tokens of prior KV plus, causally,
 *    to the active tokens of its own chunk; the new K/V of every active token
 *    is written into the cache.
 *  - "Prefill Optimisation", section 2 "Causal equivalence and numerical
 *    tolerance": active token i of a chunk sits at absolute position
 *    num_computed_tokens + i, so chunked attention equals one-shot causal
 *    attention over the full prompt (positions j <= i).
 *  - "Prefill Processing", "Block Allocation": the block table maps logical
 *    block j / block_size of a request to a physical block of the pool.
 *  - "Prefill Optimisation", section 6: grouped-query attention keeps H_kv
 *    key/value heads for H_q query heads.
 *  - "Prefill Processing", "Kernel Interface" and "Partial KV Segment
 *    Handling": the cached KV is walked in kv_segment_size pieces, the
 *    number of pieces derived from cached_seq_len, a last partial piece
 *    masked; "Prefill Optimisation", section 2, names the online-softmax
 *    rescaling of running normalisers that combines the pieces.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - query head h uses key/value head h / (H_q / H_kv) (contiguous groups);
 *  - pool layout is [num_blocks, block_size, H_kv, head_dim], slot =
 *    block * block_size + offset, i.e. slot == row of the pool;
 *  - keys at positions >= cached_seq_len are taken from the new K/V inputs
 *    (the same values the write puts into the pool);
 *  - lse is the natural log of the softmax denominator of the scaled scores.
 *
 * Rotary position embedding (optional, cpa_oracle_rope): "Prefill
 * Optimisation", section 2, and "Chunked Prefill" note that the active
 * tokens of a chunk take their absolute positions num_computed_tokens + i,
 * which is where a rotary embedding must rotate them.  The pages fix no
 * rotary convention; the reading taken is the rotate-half form of the
 * RoFormer rotary embedding as used by Llama models: for a head vector x of
 * dimension d at position p, each pair (x_c, x_{c+d/2}), c < d/2, turns by
 * the angle p * theta^(-2c/d).
 *
 * FP8 key/value cache (optional, kv_fp8 = 1): "Prefill Optimisation",
 * section 3 (prefix caching), names a KV cache data representation (FP8
 * E4M3) with quantization scales as part of what makes cached KV reusable,
 * and says nothing more.  The reading
 * taken: the pools hold E4M3 codes (the OCP FP8 E4M3 format: 1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes the
 * subnormals m * 2^-9; S.1111.111 is NaN; no infinities; largest finite
 * value 448) with one fp32 scale per kv head for keys and one for values.
 * An element x is stored as the code nearest to y = fl32(x / scale) (the
 * quotient rounded to fp32, then rounded to nearest, ties to an even
 * mantissa), saturated to +-448 when |y| >= 448; a NaN becomes the NaN
 * code.  A code c stands for value(c) * scale.  Attention sees every key and
 * value through this representation, the active tokens' own new rows
 * included, so chunked prefill over the FP8 cache still equals one-shot
 * attention over the quantized prompt.
 *
 * Parity pins (see tests/test_oracle.py): closed forms (first token of a
 * fresh prompt returns v_0; zero queries give the mean of visible values;
 * constant values; one-hot scores), a pure-Python fsum brute force over the
 * dense prompt, chunk invariance against one-shot causal attention, segment
 * invariance, prefix-hit equivalence, and planted-mistake runs that each
 * pin must catch.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t num_reqs;
    int32_t max_blocks_per_seq;
    int32_t total_new_tokens;
    int32_t num_heads_q;
    int32_t num_heads_kv;
    int32_t head_dim;
    int32_t block_size;
    int32_t num_blocks;
    int32_t dtype;      /* 0: float32 values, 1: bfloat16 bit patterns (uint16), 2: float64 */
    int32_t mutation;   /* 0 in every real use; >0 plants a known mistake (tests only) */
    double scale;
    const int32_t *cached_seq_len;  /* [num_reqs] */
    const int32_t *num_new_tokens;  /* [num_reqs] */
    const int32_t *cu_new_tokens;   /* [num_reqs + 1] */
    const int32_t *block_table;     /* [num_reqs, max_blocks_per_seq] */
    const void *q;                  /* [T, H_q, d] */
    const void *k_new;              /* [T, H_kv, d] */
    const void *v_new;              /* [T, H_kv, d] */
    const void *k_cache;            /* [num_blocks, block_size, H_kv, d] */
    const void *v_cache;
    int32_t kv_fp8;                 /* 1: pools hold FP8 E4M3 codes (uint8), see the header */
    const float *k_scale;           /* [H_kv] key scales (kv_fp8 only) */
    const float *v_scale;           /* [H_kv] value scales (kv_fp8 only) */
} orc_problem;

/* Planted mistakes, used only by the tests that prove the pins can fail. */
enum {
    MUT_NONE = 0,
    MUT_DROP_DIAGONAL = 1,     /* token does not see itself */
    MUT_GQA_MODULO = 2,        /* query head h uses kv head h % H_kv */
    MUT_NO_POSITION_OFFSET = 3,/* active token i treated as position i */
    MUT_DROP_CACHED = 4,       /* cached prefix ignored */
    MUT_NO_BLOCK_TABLE = 5,    /* pool read as if contiguous: slot = position */
    MUT_NO_SCALE = 6,          /* scores not scaled */
    MUT_MERGE_NO_RESCALE = 7,  /* segment merge forgets to rescale l */
    MUT_WRITE_OFF_BY_ONE = 8,  /* KV write one slot too far */
    MUT_ROPE_INTERLEAVED = 9,  /* rotary pairs (2c, 2c+1) instead of (c, c + d/2) */
    MUT_ROPE_NO_OFFSET = 10,   /* rotary angle from i instead of cached_seq_len + i */
    MUT_FP8_NEW_UNQUANTIZED = 11, /* FP8 cache: the active tokens' own keys/values skip the cache format */
    MUT_FP8_HEAD0_SCALE = 12,  /* FP8 cache: every kv head uses head 0's scales */
    MUT_FP8_TRUNCATE = 13,     /* FP8 encoder truncates instead of rounding to nearest */
    MUT_SEES_NEXT_KEY = 14,    /* causal limit one too far: token also sees the key after its own */
};

/* Value of an FP8 E4M3 code (NaN for S.1111.111). */
static double e4m3_value(uint8_t code) {
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                /* subnormal: m * 2^-9 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);         /* normal: 1.mmm * 2^(e - 7) */
    return sign ? -v : v;
}

/* Code of an fp32 value: nearest representable value, ties to an even
 * mantissa; |y| >= 448 saturates to +-448 (every value in [448, 464] rounds
 * to 448, and larger ones clamp there); NaN gives the NaN code 0x7F. */
static uint8_t e4m3_encode(float y, int mutation) {
    if (isnan(y)) return 0x7F;
    const uint8_t sign = signbit(y) ? 0x80 : 0;
    const double a = fabs((double)y);
    if (a >= 448.0) return sign | 0x7E;
    int ex;
    frexp(a, &ex);           /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;          /* a in [2^E, 2^(E+1)) */
    if (E < -6) E = -6;      /* below the normal range the spacing stays 2^-9 */
    const double quantum = ldexp(1.0, E - 3);            /* 3 mantissa bits */
    const double n = (mutation == MUT_FP8_TRUNCATE) ? floor(a / quantum)
                                                    : nearbyint(a / quantum); /* exact quotient; RNE */
    const double v = n * quantum;                       /* may round up to 2^(E+1) */
    if (v == 0.0) return sign;
    frexp(v, &ex);
    E = ex - 1;
    if (E < -6) return sign | (uint8_t)(v / ldexp(1.0, -9));   /* subnormal code = m */
    const int m = (int)(v / ldexp(1.0, E) * 8.0) - 8;
    return sign | (uint8_t)((E + 7) << 3) | (uint8_t)m;
}

static float kv_scale(const orc_problem *P, int is_v, int g) {
    const float *sc = is_v ? P->v_scale : P->k_scale;
    return sc[P->mutation == MUT_FP8_HEAD0_SCALE ? 0 : g];
}

static double load_elem(const void *base, int dtype, size_t idx) {
    if (dtype == 0) return (double)((const float *)base)[idx];
    if (dtype == 2) return ((const double *)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int request_of_token(const orc_problem *P, int t) {
    /* Plain linear search: the oracle favours obviousness over speed. */
    for (int r = 0; r < P->num_reqs; ++r)
        if (t >= P->cu_new_tokens[r] && t < P->cu_new_tokens[r + 1]) return r;
    return -1;
}

/* Element c of the key (is_v = 0) or value (is_v = 1) of request r at
 * absolute position j, kv head g. */
static double kv_elem(const orc_problem *P, int is_v, int r, int j, int g, int c) {
    const int d = P->head_dim, hkv = P->num_heads_kv, bs = P->block_size;
    const int C = P->cached_seq_len[r];
    if (j < C) {
        long slot;
        if (P->mutation == MUT_NO_BLOCK_TABLE) {
            slot = j;
        } else {
            int blk = P->block_table[(size_t)r * P->max_blocks_per_seq + j / bs];
            slot = (long)blk * bs + j % bs;
        }
        size_t idx = ((size_t)slot * hkv + g) * d + c;
        if (P->kv_fp8)
            return e4m3_value(((const uint8_t *)(is_v ? P->v_cache : P->k_cache))[idx]) * kv_scale(P, is_v, g);
        return load_elem(is_v ? P->v_cache : P->k_cache, P->dtype, idx);
    }
    int t = P->cu_new_tokens[r] + (j - C);
    size_t idx = ((size_t)t * hkv + g) * d + c;
    double x = load_elem(is_v ? P->v_new : P->k_new, P->dtype, idx);
    if (P->kv_fp8 && P->mutation != MUT_FP8_NEW_UNQUANTIZED) {
        /* the active token's own row, as the cache holds it */
        const float sc = kv_scale(P, is_v, g);
        x = e4m3_value(e4m3_encode((float)x / sc, P->mutation)) * sc;
    }
    return x;
}

typedef struct {
    int r, i, t, h, g;
    int first_key;   /* first visible absolute key position */
    int last_key;    /* last visible absolute key position (inclusive) */
} row_info;

static int make_row(const orc_problem *P, int t, int h, row_info *ri) {
    int r = request_of_token(P, t);
    if (r < 0) return -1;
    const int G = P->num_heads_q / P->num_heads_kv;
    ri->r = r;
    ri->t = t;
    ri->h = h;
    ri->i = t - P->cu_new_tokens[r];
    ri->g = (P->mutation == MUT_GQA_MODULO) ? h % P->num_heads_kv : h / G;
    int C = P->cached_seq_len[r];
    int p = (P->mutation == MUT_NO_POSITION_OFFSET) ? ri->i : C + ri->i;
    ri->first_key = (P->mutation == MUT_DROP_CACHED) ? C : 0;
    ri->last_key = (P->mutation == MUT_DROP_DIAGONAL) ? p - 1 : p;
    if (P->mutation == MUT_SEES_NEXT_KEY && p + 1 < C + P->num_new_tokens[r]) ri->last_key = p + 1;
    if (ri->last_key < ri->first_key) ri->last_key = ri->first_key; /* keep >= 1 key */
    return 0;
}

static double score(const orc_problem *P, const row_info *ri, int j) {
    const int d = P->head_dim;
    double acc = 0.0;
    for (int c = 0; c < d; ++c) {
        size_t qi = ((size_t)ri->t * P->num_heads_q + ri->h) * d + c;
        acc += load_elem(P->q, P->dtype, qi) * kv_elem(P, 0, ri->r, j, ri->g, c);
    }
    double s = (P->mutation == MUT_NO_SCALE) ? 1.0 : P->scale;
    return s * acc;
}

/* Definition: softmax over every visible key at once, fp64. */
static void row_definition(const orc_problem *P, const row_info *ri, double *out, double *lse,
                           double *sbuf) {
    const int d = P->head_dim;
    int nk = ri->last_key - ri->first_key + 1;
    double m = -INFINITY;
    for (int k = 0; k < nk; ++k) {
        sbuf[k] = score(P, ri, ri->first_key + k);
        if (sbuf[k] > m) m = sbuf[k];
    }
    double sum = 0.0;
    for (int k = 0; k < nk; ++k) {
        sbuf[k] = exp(sbuf[k] - m);
        sum += sbuf[k];
    }
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int k = 0; k < nk; ++k) acc += sbuf[k] * kv_elem(P, 1, ri->r, ri->first_key + k, ri->g, c);
        out[c] = acc / sum;
    }
    *lse = m + log(sum);
}

/* The method step by step: cached keys in kv_segment_size pieces (the last
 * one partial), then the active chunk; each piece yields its own maximum m_s,
 * normaliser l_s = sum exp(s - m_s) and unnormalised output o_s; the running
 * state is combined piece by piece with the online-softmax rescaling. */
static void piece(const orc_problem *P, const row_info *ri, int k0, int k1, double *m_s, double *l_s,
                  double *o_s, double *sbuf) {
    const int d = P->head_dim;
    int nk = k1 - k0;
    double m = -INFINITY;
    for (int k = 0; k < nk; ++k) {
        sbuf[k] = score(P, ri, k0 + k);
        if (sbuf[k] > m) m = sbuf[k];
    }
    double l = 0.0;
    for (int k = 0; k < nk; ++k) {
        sbuf[k] = exp(sbuf[k] - m);
        l += sbuf[k];
    }
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int k = 0; k < nk; ++k) acc += sbuf[k] * kv_elem(P, 1, ri->r, k0 + k, ri->g, c);
        o_s[c] = acc;
    }
    *m_s = m;
    *l_s = l;
}

static void merge_into(const orc_problem *P, double *m, double *l, double *o, double m_s, double l_s,
                       const double *o_s) {
    const int d = P->head_dim;
    if (l_s == 0.0) return; /* empty piece contributes nothing */
    double mn = (*m > m_s) ? *m : m_s;
    double a = (*l == 0.0) ? 0.0 : exp(*m - mn);
    double b = exp(m_s - mn);
    if (P->mutation == MUT_MERGE_NO_RESCALE)
        *l = *l + l_s;
    else
        *l = *l * a + l_s * b;
    for (int c = 0; c < d; ++c) o[c] = o[c] * a + o_s[c] * b;
    *m = mn;
}

static void row_segmented(const orc_problem *P, const row_info *ri, int seg, double *out, double *lse,
                          double *sbuf, double *o_s) {
    const int d = P->head_dim;
    const int C = P->cached_seq_len[ri->r];
    double m = -INFINITY, l = 0.0;
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    /* cached part: ceil(C / seg) pieces; the count is derived, never given */
    int cached_end = (ri->last_key + 1 < C) ? ri->last_key + 1 : C;
    int seg_len = seg > 0 ? seg : (C > 0 ? C : 1);
    int n_pieces = (cached_end - ri->first_key + seg_len - 1) / seg_len;
    for (int s = 0; s < n_pieces; ++s) {
        int k0 = ri->first_key + s * seg_len;
        int k1 = k0 + seg_len;
        if (k1 > cached_end) k1 = cached_end; /* partial last piece */
        if (k1 <= k0) continue;
        double m_s, l_s;
        piece(P, ri, k0, k1, &m_s, &l_s, o_s, sbuf);
        merge_into(P, &m, &l, out, m_s, l_s, o_s);
    }
    /* active chunk: keys C .. position of this token (causal) */
    int a0 = (ri->first_key > C) ? ri->first_key : C;
    if (ri->last_key >= a0) {
        double m_s, l_s;
        piece(P, ri, a0, ri->last_key + 1, &m_s, &l_s, o_s, sbuf);
        merge_into(P, &m, &l, out, m_s, l_s, o_s);
    }
    for (int c = 0; c < d; ++c) out[c] /= l;
    *lse = m + log(l);
}

typedef struct {
    const orc_problem *P;
    const int32_t *rows;  /* token indices, or NULL for 0..n_rows-1 */
    int n_rows;
    int segmented;
    int kv_segment_size;
    double *out;  /* [n_rows, H_q, d] */
    double *lse;  /* [n_rows, H_q] */
    int begin, end;  /* range of (row, head) work items */
    int status;
} worker_arg;

static void *worker(void *argp) {
    worker_arg *A = (worker_arg *)argp;
    const orc_problem *P = A->P;
    const int hq = P->num_heads_q, d = P->head_dim;
    int max_keys = 1;
    for (int r = 0; r < P->num_reqs; ++r) {
        int L = P->cached_seq_len[r] + P->num_new_tokens[r];
        if (L > max_keys) max_keys = L;
    }
    double *sbuf = (double *)malloc(sizeof(double) * (size_t)max_keys);
    double *o_s = (double *)malloc(sizeof(double) * (size_t)d);
    if (!sbuf || !o_s) {
        free(sbuf);
        free(o_s);
        A->status = -2;
        return NULL;
    }
    for (int w = A->begin; w < A->end; ++w) {
        int n = w / hq, h = w % hq;
        int t = A->rows ? A->rows[n] : n;
        row_info ri;
        if (make_row(P, t, h, &ri) != 0) {
            A->status = -1;
            break;
        }
        double *o = A->out + ((size_t)n * hq + h) * d;
        double *l = A->lse + (size_t)n * hq + h;
        if (A->segmented)
            row_segmented(P, &ri, A->kv_segment_size, o, l, sbuf, o_s);
        else
            row_definition(P, &ri, o, l, sbuf);
    }
    free(sbuf);
    free(o_s);
    return NULL;
}

/* Attention for the rows listed in `rows` (token indices into the packed
 * batch; NULL means every token 0..n_rows-1), all query heads.  segmented = 0
 * evaluates the definition; segmented = 1 walks the method's pieces.
 * Returns 0, or -1 for a token outside every request, -2 on allocation
 * failure, -3 on bad arguments. */
int cpa_oracle_attention(const orc_problem *P, const int32_t *rows, int n_rows, int segmented,
                         int kv_segment_size, double *out, double *lse, int nthreads) {
    if (!P || !out || !lse || n_rows < 0 || P->num_heads_kv <= 0 ||
        P->num_heads_q % P->num_heads_kv != 0)
        return -3;
    if (nthreads < 1) nthreads = 1;
    int items = n_rows * P->num_heads_q;
    if (nthreads > items) nthreads = items > 0 ? items : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    worker_arg *args = (worker_arg *)malloc(sizeof(worker_arg) * (size_t)nthreads);
    if (!th || !args) {
        free(th);
        free(args);
        return -2;
    }
    for (int i = 0; i < nthreads; ++i) {
        worker_arg a = {P, rows, n_rows, segmented, kv_segment_size, out, lse,
                        (int)((long)items * i / nthreads), (int)((long)items * (i + 1) / nthreads), 0};
        args[i] = a;
    }
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &args[i]);
    worker(&args[0]);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
    int status = 0;
    for (int i = 0; i < nthreads; ++i)
        if (args[i].status) status = args[i].status;
    free(th);
    free(args);
    return status;
}

/* The write of new K/V into the pool: active token i of request r goes to
 * slot block_table[r][(C + i) / bs] * bs + (C + i) % bs.  A byte copy, so
 * the element type only sets the row size.  k_cache/v_cache are the
 * oracle's own copies and are updated in place.  Returns 0 or -3. */
int cpa_oracle_kv_write(const orc_problem *P, int elem_bytes, void *k_cache, void *v_cache) {
    if (!P || !k_cache || !v_cache || elem_bytes <= 0) return -3;
    const size_t row = (size_t)P->num_heads_kv * P->head_dim * elem_bytes;
    for (int r = 0; r < P->num_reqs; ++r) {
        int C = P->cached_seq_len[r];
        for (int i = 0; i < P->num_new_tokens[r]; ++i) {
            int pos = C + i;
            if (P->mutation == MUT_WRITE_OFF_BY_ONE) pos += 1;
            if (pos / P->block_size >= P->max_blocks_per_seq) return -3;
            int blk = P->block_table[(size_t)r * P->max_blocks_per_seq + pos / P->block_size];
            size_t slot = (size_t)blk * P->block_size + pos % P->block_size;
            if (blk < 0 || blk >= P->num_blocks) return -3;
            int t = P->cu_new_tokens[r] + i;
            memcpy((char *)k_cache + slot * row, (const char *)P->k_new + (size_t)t * row, row);
            memcpy((char *)v_cache + slot * row, (const char *)P->v_new + (size_t)t * row, row);
        }
    }
    return 0;
}

/* The write into FP8 pools: every element of the active tokens' K/V rows is
 * encoded with its kv head's scale (see the header) and stored as one byte
 * in the slot row.  k_cache/v_cache are the oracle's own uint8 copies.
 * Returns 0 or -3. */
int cpa_oracle_kv_write_fp8(const orc_problem *P, uint8_t *k_cache, uint8_t *v_cache) {
    if (!P || !k_cache || !v_cache || !P->k_scale || !P->v_scale) return -3;
    const int hkv = P->num_heads_kv, d = P->head_dim;
    for (int r = 0; r < P->num_reqs; ++r) {
        int C = P->cached_seq_len[r];
        for (int i = 0; i < P->num_new_tokens[r]; ++i) {
            int pos = C + i;
            if (P->mutation == MUT_WRITE_OFF_BY_ONE) pos += 1;
            if (pos / P->block_size >= P->max_blocks_per_seq) return -3;
            int blk = P->block_table[(size_t)r * P->max_blocks_per_seq + pos / P->block_size];
            if (blk < 0 || blk >= P->num_blocks) return -3;
            size_t slot = (size_t)blk * P->block_size + pos % P->block_size;
            int t = P->cu_new_tokens[r] + i;
            for (int g = 0; g < hkv; ++g)
                for (int c = 0; c < d; ++c) {
                    size_t src = ((size_t)t * hkv + g) * d + c, dst = (slot * hkv + g) * d + c;
                    k_cache[dst] = e4m3_encode((float)load_elem(P->k_new, P->dtype, src) / kv_scale(P, 0, g),
                                               P->mutation);
                    v_cache[dst] = e4m3_encode((float)load_elem(P->v_new, P->dtype, src) / kv_scale(P, 1, g),
                                               P->mutation);
                }
        }
    }
    return 0;
}

/* Element-wise E4M3 encode of fp32 values and decode of codes (for the
 * tests of the format itself). */
void cpa_oracle_e4m3_encode(const float *y, uint8_t *codes, long n, int mutation) {
    for (long i = 0; i < n; ++i) codes[i] = e4m3_encode(y[i], mutation);
}
void cpa_oracle_e4m3_decode(const uint8_t *codes, double *out, long n) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

/* Rotary position embedding of the active tokens' queries and new keys
 * (see the header).  q_out [T, H_q, d] and k_out [T, H_kv, d] receive the
 * rotated values in fp64 (either may be NULL).  Active token i of request r
 * is at absolute position cached_seq_len[r] + i.  Returns 0 or -3. */
int cpa_oracle_rope(const orc_problem *P, double theta, double *q_out, double *k_out) {
    if (!P || !(theta > 0.0) || (P->head_dim & 1)) return -3;
    const int d = P->head_dim, half = d / 2;
    for (int t = 0; t < P->total_new_tokens; ++t) {
        int r = request_of_token(P, t);
        if (r < 0) return -3;
        int i = t - P->cu_new_tokens[r];
        double p = (P->mutation == MUT_ROPE_NO_OFFSET) ? (double)i : (double)(P->cached_seq_len[r] + i);
        for (int which = 0; which < 2; ++which) {
            const int heads = which == 0 ? P->num_heads_q : P->num_heads_kv;
            const void *src = which == 0 ? P->q : P->k_new;
            double *dst = which == 0 ? q_out : k_out;
            if (!dst) continue;
            for (int h = 0; h < heads; ++h) {
                size_t base = ((size_t)t * heads + h) * d;
                for (int c = 0; c < half; ++c) {
                    /* pair members: (c, c + d/2); the planted mistake pairs (2c, 2c+1) */
                    int a = c, b = c + half;
                    if (P->mutation == MUT_ROPE_INTERLEAVED) {
                        a = 2 * c;
                        b = 2 * c + 1;
                    }
                    double angle = p * pow(theta, -2.0 * c / d);
                    double x0 = load_elem(src, P->dtype, base + a), x1 = load_elem(src, P->dtype, base + b);
                    dst[base + a] = x0 * cos(angle) - x1 * sin(angle);
                    dst[base + b] = x1 * cos(angle) + x0 * sin(angle);
                }
            }
        }
    }
    return 0;
}
