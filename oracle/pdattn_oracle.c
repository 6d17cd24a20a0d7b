/*
 * Plain CPU oracle for one decode step of grouped-query attention over a
 * paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  It shares no
 * code with the CUDA path (no headers, helpers or tables) and is deliberately
 * slow: serial loops, fp64 wherever the pages leave the precision open.
 *
 * What each function follows (page title, section):
 *   oracle_rope_tables   Llama example page, "src/rope.linnet" (`tables`):
 *                        inv_freq from theta and iota in f32, angles = s *
 *                        inv_freq, full = concat(angles, angles), cos and sin
 *                        cast to T.
 *   oracle_rope_write_kv Llama example page, "src/attention.linnet"
 *                        (`decode`): rope on q and the new k at pos, then
 *                        write_at of k and v; the paged slot comes from the
 *                        llama-3.1-8b-instruct architecture page, entry table
 *                        (`decode_paged`, `table: Tensor[Rows, Pages; i32]`)
 *                        and the `PageSize: Dim = 64` generic of
 *                        GroupedQueryAttention.
 *   oracle_prefill_paged rope + write of packed prompt tokens at their slots,
 *                        then each token's causal attention over its row
 *                        (llama-3.1-8b-instruct page, `prefill_paged`).
 *   oracle_packed        Llama example page, "src/attention.linnet"
 *                        (`packed`): sequences packed into one row, rope at
 *                        each token's own position, mask own[i, j] =
 *                        segments[i] == segments[j] && positions[j] <=
 *                        positions[i], no cache.
 *   oracle_decode(_sinks) Llama example page, "src/attention.linnet"
 *                        (`decode`): mask seen[s] = s <= pos, scale
 *                        rsqrt(f32(head dim)), grouped attention where query
 *                        head h reads kv head h / (Heads / KvHeads) ("Key
 *                        ideas", grouped-query attention); sliding window from
 *                        the gpt-oss-20b architecture page (`window: i32`);
 *                        attention sinks from the same page (SinkAttention
 *                        `param sinks`), read as one extra value-less logit
 *                        per query head in the softmax.
 *
 * Readings where the pages leave a step open:
 *   - rope(x, cos, sin) = x * cos + rotate_half(x) * sin with
 *     rotate_half(x) = concat(-x[D/2:], x[:D/2]); the halves share frequency i
 *     because the table is concat(angles, angles).  Each product is an f32
 *     product, the sum one f32 add, the result rounded once to T.  The
 *     rotation direction is a convention the pages do not print: parity for
 *     the direction alone is unpinned.
 *   - cos, sin, exp and log are the correctly rounded f32 results, computed
 *     in double and rounded to f32 (then to T for the tables).
 *   - Attention scores, softmax and the weighted sum are computed in double
 *     and the output rounded once to T.
 *   - window W > 0 attends positions in (pos - W, pos]; W <= 0 attends [0, pos].
 *
 * Element types: dtype 0 = bf16 (stored as uint16 bit patterns), 1 = f32.
 * Build with -ffp-contract=off so that no product and sum fuse.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t rows, heads, kv_heads, head_dim;
    int32_t page_size, pages_per_row, num_pages;
    int32_t dtype;      /* 0 = bf16, 1 = f32 */
    int32_t window;     /* <= 0: every cached position up to pos */
    float rope_theta;   /* <= 0: no rotation (GPT-2: learned positions upstream) */
} oracle_shape;

enum { ORACLE_OK = 0, ORACLE_EINVAL = 1, ORACLE_EBADPAGE = 4 };

/* ---- element access ---------------------------------------------------- */

static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an f32 to bf16, to nearest with ties to even. */
static uint16_t float_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN stays NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

static float load_t(const void* base, size_t i, int dtype) {
    if (dtype == 0) return bf16_bits_to_float(((const uint16_t*)base)[i]);
    return ((const float*)base)[i];
}

/* Round an f32 value to T and store it. */
static void store_t(void* base, size_t i, float v, int dtype) {
    if (dtype == 0) ((uint16_t*)base)[i] = float_to_bf16_bits(v);
    else ((float*)base)[i] = v;
}

/* Round an f32 value to T and return it as f32. */
static float round_t(float v, int dtype) {
    return dtype == 0 ? bf16_bits_to_float(float_to_bf16_bits(v)) : v;
}

static void copy_t(void* dst, size_t di, const void* src, size_t si, int dtype) {
    if (dtype == 0) ((uint16_t*)dst)[di] = ((const uint16_t*)src)[si];
    else ((float*)dst)[di] = ((const float*)src)[si];
}

/* ---- rotary tables ----------------------------------------------------- */

/* inv_freq[i] = exp(-(f32(i) * 2.0 / f32(D)) * log(theta)), all in f32. */
static float inv_freq_f32(int i, int D, float theta) {
    float two_i = (float)i * 2.0f;
    float ratio = two_i / (float)D;
    float log_theta = (float)log((double)theta);
    float arg = (-ratio) * log_theta;
    return (float)exp((double)arg);
}

/* cos and sin (f32, not yet rounded to T) of f32(s) * inv_freq[i]. */
static void angle_cos_sin(int s, int i, int D, float theta, float* c, float* sn) {
    float angle = (float)s * inv_freq_f32(i, D, theta);
    *c = (float)cos((double)angle);
    *sn = (float)sin((double)angle);
}

/* Tables [S, D] of T: column i and i + D/2 hold the same frequency. */
int oracle_rope_tables(float theta, int D, int S, int dtype, void* cos_out, void* sin_out) {
    if (D <= 0 || D % 2 != 0 || S < 0 || theta <= 0.0f || (dtype != 0 && dtype != 1))
        return ORACLE_EINVAL;
    int half = D / 2;
    for (int s = 0; s < S; ++s) {
        for (int j = 0; j < D; ++j) {
            float c, sn;
            angle_cos_sin(s, j % half, D, theta, &c, &sn);
            store_t(cos_out, (size_t)s * D + j, c, dtype);
            store_t(sin_out, (size_t)s * D + j, sn, dtype);
        }
    }
    return ORACLE_OK;
}

/* rope of one head vector x[D] (T) at position pos into y[D] (T). */
static void rope_vector(const void* x, size_t xo, void* y, size_t yo, int D, int pos,
                        float theta, int dtype) {
    int half = D / 2;
    for (int j = 0; j < D; ++j) {
        float c, sn;
        angle_cos_sin(pos, j % half, D, theta, &c, &sn);
        c = round_t(c, dtype);   /* cos(full) and sin(full) are cast to T */
        sn = round_t(sn, dtype);
        float xj = load_t(x, xo + j, dtype);
        /* rotate_half(x)[j] = -x[j + D/2] for j < D/2, x[j - D/2] otherwise */
        float rh = j < half ? -load_t(x, xo + j + half, dtype) : load_t(x, xo + j - half, dtype);
        float a = xj * c;
        float b = rh * sn;
        store_t(y, yo + j, a + b, dtype);
    }
}

static int shape_ok(const oracle_shape* p) {
    if (!p) return 0;
    if (p->rows < 0 || p->heads <= 0 || p->kv_heads <= 0 || p->heads % p->kv_heads != 0) return 0;
    if (p->head_dim <= 0 || p->head_dim % 2 != 0) return 0;
    if (p->page_size <= 0 || p->pages_per_row <= 0 || p->num_pages <= 0) return 0;
    if (p->dtype != 0 && p->dtype != 1) return 0;
    return 1;
}

/* Pool element index of (page, kv head, offset, d) in [NumPages, KvHeads, PageSize, D]. */
static size_t pool_index(const oracle_shape* p, int page, int kvh, int off, int d) {
    return (((size_t)page * p->kv_heads + kvh) * p->page_size + off) * p->head_dim + d;
}

/*
 * RoPE on q [R, Hq, D] and k_new [R, Hk, D] at positions[r]; q_out receives
 * the rotated q, and the rotated k and the unrotated v_new go into the pool
 * slot table[r, pos / PageSize], offset pos % PageSize.
 */
int oracle_rope_write_kv(const oracle_shape* p, const void* q, const void* k_new,
                         const void* v_new, const int32_t* positions, const int32_t* table,
                         void* q_out, void* k_pool, void* v_pool) {
    if (!shape_ok(p)) return ORACLE_EINVAL;
    const int D = p->head_dim, Hq = p->heads, Hk = p->kv_heads, PS = p->page_size;
    int status = ORACLE_OK;
    for (int r = 0; r < p->rows; ++r) {
        int pos = positions[r];
        if (pos < 0 || pos >= p->pages_per_row * PS) { status = ORACLE_EINVAL; continue; }
        int page = table[(size_t)r * p->pages_per_row + pos / PS];
        int off = pos % PS;
        for (int h = 0; h < Hq; ++h) {
            size_t o = ((size_t)r * Hq + h) * D;
            if (p->rope_theta > 0.0f) rope_vector(q, o, q_out, o, D, pos, p->rope_theta, p->dtype);
            else for (int d = 0; d < D; ++d) copy_t(q_out, o + d, q, o + d, p->dtype);
        }
        if (page < 0 || page >= p->num_pages) { status = ORACLE_EBADPAGE; continue; }
        for (int h = 0; h < Hk; ++h) {
            size_t o = ((size_t)r * Hk + h) * D;
            size_t slot = pool_index(p, page, h, off, 0);
            if (p->rope_theta > 0.0f) rope_vector(k_new, o, k_pool, slot, D, pos, p->rope_theta, p->dtype);
            else for (int d = 0; d < D; ++d) copy_t(k_pool, slot + d, k_new, o + d, p->dtype);
            for (int d = 0; d < D; ++d) copy_t(v_pool, slot + d, v_new, o + d, p->dtype);
        }
    }
    return status;
}

/*
 * Attention of the rotated queries q_rot [R, Hq, D] over the cached positions
 * of each row.  out [R, Hq, D] is rounded to T; out64 (may be NULL) receives
 * the unrounded double result.  sinks (may be NULL) holds one logit per
 * query head [Hq] of T (gpt-oss-20b architecture page, SinkAttention
 * `param sinks: Tensor[Heads; T]`); its reading: the sink joins the softmax
 * as one more logit that carries no value, so it only enlarges the
 * denominator.
 */
/* One row of oracle_decode_sinks; scores holds max_ctx doubles, acc D. */
static int decode_row(const oracle_shape* p, int r, const void* q_rot, const int32_t* positions,
                      const int32_t* table, const void* k_pool, const void* v_pool, const void* sinks,
                      void* out, double* out64, double* scores, double* acc) {
    const int D = p->head_dim, Hq = p->heads, Hk = p->kv_heads, PS = p->page_size;
    const int group = Hq / Hk;
    const double scale = (double)(float)(1.0 / sqrt((double)D)); /* rsqrt(f32(D)) */
    const int max_ctx = p->pages_per_row * PS;
    int pos = positions[r];
    if (pos < 0 || pos >= max_ctx) return ORACLE_EINVAL;
    int lo = 0;
    if (p->window > 0 && pos - p->window + 1 > 0) lo = pos - p->window + 1;
    for (int t = lo; t <= pos; ++t) {
        int page = table[(size_t)r * p->pages_per_row + t / PS];
        if (page < 0 || page >= p->num_pages) return ORACLE_EBADPAGE;
    }
    for (int h = 0; h < Hq; ++h) {
        int kvh = h / group;
        size_t qo = ((size_t)r * Hq + h) * D;
        double m = -INFINITY;
        const double sink = sinks ? (double)load_t(sinks, (size_t)h, p->dtype) : -INFINITY;
        for (int t = lo; t <= pos; ++t) {
            int page = table[(size_t)r * p->pages_per_row + t / PS];
            size_t ko = pool_index(p, page, kvh, t % PS, 0);
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += (double)load_t(q_rot, qo + d, p->dtype) * (double)load_t(k_pool, ko + d, p->dtype);
            scores[t - lo] = scale * dot;
            if (scores[t - lo] > m) m = scores[t - lo];
        }
        if (sink > m) m = sink;
        double l = sinks ? exp(sink - m) : 0.0;
        for (int t = lo; t <= pos; ++t) {
            scores[t - lo] = exp(scores[t - lo] - m);
            l += scores[t - lo];
        }
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        for (int t = lo; t <= pos; ++t) {
            int page = table[(size_t)r * p->pages_per_row + t / PS];
            size_t vo = pool_index(p, page, kvh, t % PS, 0);
            double w = scores[t - lo] / l;
            for (int d = 0; d < D; ++d) acc[d] += w * (double)load_t(v_pool, vo + d, p->dtype);
        }
        for (int d = 0; d < D; ++d) {
            if (out64) out64[qo + d] = acc[d];
            store_t(out, qo + d, (float)acc[d], p->dtype);
        }
    }
    return ORACLE_OK;
}

/*
 * Rows are independent; when the library is built with OpenMP they run on
 * oracle_set_threads() threads (one row at a time per thread, the same
 * arithmetic), and the status is that of the last failing row, as in order.
 */
int oracle_decode_sinks(const oracle_shape* p, const void* q_rot, const int32_t* positions,
                        const int32_t* table, const void* k_pool, const void* v_pool,
                        const void* sinks, void* out, double* out64) {
    if (!shape_ok(p)) return ORACLE_EINVAL;
    const int max_ctx = p->pages_per_row * p->page_size;
    int* row_status = (int*)calloc((size_t)(p->rows > 0 ? p->rows : 1), sizeof(int));
    if (!row_status) return ORACLE_EINVAL;
    int oom = 0;
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)max_ctx);
        double* acc = (double*)malloc(sizeof(double) * (size_t)p->head_dim);
        if (!scores || !acc) {
            oom = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int r = 0; r < p->rows; ++r)
                row_status[r] = decode_row(p, r, q_rot, positions, table, k_pool, v_pool, sinks, out, out64,
                                           scores, acc);
        }
        free(scores);
        free(acc);
    }
    int status = oom ? ORACLE_EINVAL : ORACLE_OK;
    for (int r = 0; r < p->rows; ++r)
        if (row_status[r] != ORACLE_OK) status = row_status[r];
    free(row_status);
    return status;
}

/* Threads for the row loop (no effect without OpenMP); returns the count in use. */
int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int oracle_decode(const oracle_shape* p, const void* q_rot, const int32_t* positions,
                  const int32_t* table, const void* k_pool, const void* v_pool, void* out,
                  double* out64) {
    return oracle_decode_sinks(p, q_rot, positions, table, k_pool, v_pool, NULL, out, out64);
}

/*
 * One whole step: rope + cache write, then attention of the rotated queries.
 * q_rot is caller scratch of the size of q.
 */
int oracle_step(const oracle_shape* p, const void* q, const void* k_new, const void* v_new,
                const int32_t* positions, const int32_t* table, void* k_pool, void* v_pool,
                void* q_rot, void* out, double* out64) {
    int s1 = oracle_rope_write_kv(p, q, k_new, v_new, positions, table, q_rot, k_pool, v_pool);
    int s2 = oracle_decode(p, q_rot, positions, table, k_pool, v_pool, out, out64);
    return s1 != ORACLE_OK ? s1 : s2;
}

/*
 * Prefill of packed prompt tokens over the paged cache (llama-3.1-8b-instruct
 * architecture page, `prefill_paged(x: Tensor[1, P, H; T], positions:
 * Tensor[P; i32], rows: Tensor[P; i32], slots: Tensor[P; i32], table:
 * Tensor[Rows, Pages; i32])`).  Reading: token i belongs to cache row
 * rows[i] at position positions[i]; slots[i] is its flat pool slot (page *
 * PageSize + offset), where its rotated k and its v are written.  All tokens
 * are written first; then each token attends, like `decode`, over its row's
 * cached positions [lo, pos] read through the table.  q, k_new, v_new, out:
 * [P, heads or kv_heads, D].  sinks may be NULL.
 */
int oracle_prefill_paged(const oracle_shape* p, int n_tokens, const void* q, const void* k_new,
                         const void* v_new, const int32_t* positions, const int32_t* rows,
                         const int32_t* slots, const int32_t* table, void* k_pool, void* v_pool,
                         const void* sinks, void* q_rot, void* out, double* out64) {
    if (!shape_ok(p) || n_tokens < 0) return ORACLE_EINVAL;
    const int D = p->head_dim, Hq = p->heads, Hk = p->kv_heads, PS = p->page_size;
    int status = ORACLE_OK;
    /* 1. rotate q and k at each token's position; write k and v at its slot */
    for (int i = 0; i < n_tokens; ++i) {
        int pos = positions[i];
        int slot = slots[i];
        int page = slot / PS, off = slot % PS;
        for (int h = 0; h < Hq; ++h) {
            size_t o = ((size_t)i * Hq + h) * D;
            if (p->rope_theta > 0.0f) rope_vector(q, o, q_rot, o, D, pos, p->rope_theta, p->dtype);
            else for (int d = 0; d < D; ++d) copy_t(q_rot, o + d, q, o + d, p->dtype);
        }
        if (slot < 0 || page >= p->num_pages) { status = ORACLE_EBADPAGE; continue; }
        for (int h = 0; h < Hk; ++h) {
            size_t o = ((size_t)i * Hk + h) * D;
            size_t dst = pool_index(p, page, h, off, 0);
            if (p->rope_theta > 0.0f) rope_vector(k_new, o, k_pool, dst, D, pos, p->rope_theta, p->dtype);
            else for (int d = 0; d < D; ++d) copy_t(k_pool, dst + d, k_new, o + d, p->dtype);
            for (int d = 0; d < D; ++d) copy_t(v_pool, dst + d, v_new, o + d, p->dtype);
        }
    }
    /* 2. each token attends over its row's cache through the table */
    oracle_shape one = *p;
    one.rows = 1;
    for (int i = 0; i < n_tokens; ++i) {
        int r = rows[i];
        if (r < 0 || r >= p->rows) { status = ORACLE_EINVAL; continue; }
        int st = oracle_decode_sinks(&one, (const char*)q_rot + (size_t)i * Hq * D * (p->dtype == 0 ? 2 : 4),
                                     positions + i, table + (size_t)r * p->pages_per_row, k_pool, v_pool,
                                     sinks, (char*)out + (size_t)i * Hq * D * (p->dtype == 0 ? 2 : 4),
                                     out64 ? out64 + (size_t)i * Hq * D : NULL);
        if (st != ORACLE_OK) status = st;
    }
    return status;
}

/* Exposed for pins on the rounding helper itself. */
/*
 * Packed attention (Llama example page, "src/attention.linnet", `packed`):
 * n tokens of several sequences packed into one row; token p sits at
 * positions[p] of sequence segments[p].  q [n, Hq, D] and k [n, Hk, D] are
 * rotated at each token's own position into q_rot and k_rot (caller
 * buffers of the same shapes); v [n, Hk, D] is used as given.  Token i
 * attends to every token j of the pack with segments[j] == segments[i] and
 * positions[j] <= positions[i] (the pages' mask `own`), and with a window
 * W > 0 also positions[j] > positions[i] - W (the gpt-oss-20b page's
 * windowed variants), scale rsqrt(f32(D)), optional sinks as in decode.
 * Uses heads, kv_heads, head_dim, dtype, window and rope_theta of the shape.
 * Written out directly from the definition: it shares no code with decode.
 */
int oracle_packed(const oracle_shape* p, int n, const void* q, const void* k, const void* v,
                  const int32_t* positions, const int32_t* segments, const void* sinks,
                  void* q_rot, void* k_rot, void* out, double* out64) {
    if (!p || n < 0 || p->heads <= 0 || p->kv_heads <= 0 || p->heads % p->kv_heads != 0 ||
        p->head_dim <= 0 || p->head_dim % 2 != 0 || (p->dtype != 0 && p->dtype != 1))
        return ORACLE_EINVAL;
    const int D = p->head_dim, Hq = p->heads, Hk = p->kv_heads, group = Hq / Hk;
    for (int i = 0; i < n; ++i) {
        if (positions[i] < 0) return ORACLE_EINVAL;
        for (int h = 0; h < Hq; ++h) {
            size_t o = ((size_t)i * Hq + h) * D;
            if (p->rope_theta > 0.0f) rope_vector(q, o, q_rot, o, D, positions[i], p->rope_theta, p->dtype);
            else for (int d = 0; d < D; ++d) copy_t(q_rot, o + d, q, o + d, p->dtype);
        }
        for (int h = 0; h < Hk; ++h) {
            size_t o = ((size_t)i * Hk + h) * D;
            if (p->rope_theta > 0.0f) rope_vector(k, o, k_rot, o, D, positions[i], p->rope_theta, p->dtype);
            else for (int d = 0; d < D; ++d) copy_t(k_rot, o + d, k, o + d, p->dtype);
        }
    }
    const double scale = (double)(float)(1.0 / sqrt((double)D)); /* rsqrt(f32(D)) */
    /* Tokens are independent once q and k are rotated; with OpenMP they run on
     * oracle_set_threads() threads, each with its own score and sum buffers
     * (the same arithmetic in the same order as the serial loop). */
#ifdef _OPENMP
    const int nthr = omp_get_max_threads();
#else
    const int nthr = 1;
#endif
    const size_t per = (size_t)(n > 0 ? n : 1) + (size_t)D;
    double* buf = (double*)malloc(sizeof(double) * per * (size_t)nthr);
    if (!buf) return ORACLE_EINVAL;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthr)
#endif
    for (int i = 0; i < n; ++i) {
#ifdef _OPENMP
        double* w = buf + per * (size_t)omp_get_thread_num();
#else
        double* w = buf;
#endif
        double* acc = w + (n > 0 ? n : 1);
        for (int h = 0; h < Hq; ++h) {
            const int kvh = h / group;
            const size_t qo = ((size_t)i * Hq + h) * D;
            /* scores of the keys the mask lets through, max-subtracted softmax */
            double m = sinks ? (double)load_t(sinks, (size_t)h, p->dtype) : -INFINITY;
            for (int j = 0; j < n; ++j) {
                int own = segments[j] == segments[i] && positions[j] <= positions[i];
                if (own && p->window > 0) own = positions[j] > positions[i] - p->window;
                if (!own) { w[j] = -INFINITY; continue; }
                const size_t ko = ((size_t)j * Hk + kvh) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += (double)load_t(q_rot, qo + d, p->dtype) * (double)load_t(k_rot, ko + d, p->dtype);
                w[j] = scale * dot;
                if (w[j] > m) m = w[j];
            }
            double l = sinks ? exp((double)load_t(sinks, (size_t)h, p->dtype) - m) : 0.0;
            for (int j = 0; j < n; ++j) {
                w[j] = w[j] == -INFINITY ? 0.0 : exp(w[j] - m);
                l += w[j];
            }
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int j = 0; j < n; ++j) {
                if (w[j] == 0.0) continue;
                const size_t vo = ((size_t)j * Hk + kvh) * D;
                for (int d = 0; d < D; ++d) acc[d] += (w[j] / l) * (double)load_t(v, vo + d, p->dtype);
            }
            for (int d = 0; d < D; ++d) {
                if (out64) out64[qo + d] = acc[d];
                store_t(out, qo + d, (float)acc[d], p->dtype);
            }
        }
    }
    free(buf);
    return ORACLE_OK;
}

uint16_t oracle_f32_to_bf16(float f) { return float_to_bf16_bits(f); }
