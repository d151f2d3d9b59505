/*
 * pa_oracle.c -- CPU oracle for PagedAttention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, fp64 statement of what
 * the paged decode computes.  It exists to check the CUDA library, and only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no source, header, table or helper with the CUDA path.
 *
 * What it follows (page title, section):
 *  - "LLM Serving Engine Shootout: vLLM vs TensorRT-LLM vs SGLang vs
 *    llama.cpp", 3.1 PagedAttention Mechanics: the KV cache of a sequence is
 *    split into fixed-size physical blocks; a block table maps logical block
 *    index to physical block; the logit of query i against key j is
 *    q_i . k_j / sqrt(d_head), with k_j fetched through
 *    BlockTable[floor(j / B_size)].
 *  - zhichai.net "vLLM ... TRT-LLM / SGLang / TGI / llama.cpp" (Chinese
 *    original), section 1, block-table diagram: tokens 0-15 live in physical
 *    block #7, tokens 16-31 in physical block #2; tokens keep their order
 *    inside a block.
 *  - "Serving engines" (inference.tusharamrit.in), How vLLM works: the kernel
 *    gathers K/V through a block table and a slot mapping; physical blocks may
 *    be shared between sequences (copy-on-write).
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes): offset of token j inside its block is j mod block_size; softmax and
 * the value product are standard attention, V gathered exactly like K; the
 * scale is a caller-supplied fp32 value, widened to fp64; query head h reads
 * KV head h / (Hq / Hkv); a slot is physical_block * block_size + offset, and a
 * negative slot means "no token"; a sequence with context length 0 yields a
 * zero output.  The split-context form (partitions combined by log-sum-exp) is
 * not on the pages: it is the reading that the unsplit result is the target,
 * and the partition-wise function below exists to pin that combination.
 *
 * Precision: every element is converted exactly to double; scores, softmax
 * and the weighted sum are fp64, summed in increasing token order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_FP16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_BAD_INDEX = 4, ORC_NO_MEM = 5 };

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double pa_oracle_fp16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                  /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);      /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double pa_oracle_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                 /* subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 128), e - 134);      /* (1.f) * 2^(e-127) */
    return sign ? -v : v;
}

static double to_f64(uint16_t x, int dtype)
{
    return dtype == ORC_BF16 ? pa_oracle_bf16_to_f64(x) : pa_oracle_fp16_to_f64(x);
}

/*
 * FP8 E4M3 (the "fn" variant: no infinities): 1 sign, 4 exponent (bias 7),
 * 3 fraction bits; exponent 15 with fraction 111 is NaN, so the largest
 * finite magnitude is 1.75 * 2^8 = 448; subnormals are f * 2^-9.
 * (KV-cache quantisation, FP8 = 1 byte per element: zhichai.net, section 4
 * byte table; "Serving engines", quantisation of weights and increasingly KV.)
 */
double pa_oracle_e4m3_to_f64(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);                   /* subnormal: f * 2^(1-7-3) */
    else
        v = ldexp((double)(f + 8), e - 10);         /* (1.f) * 2^(e-7) */
    return sign ? -v : v;
}

/*
 * Nearest E4M3 code to x, ties to the even code, magnitudes beyond 448
 * clamped to 448 (saturating), NaN to NaN (0x7f with x's sign).
 */
uint8_t pa_oracle_e4m3_from_f32(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return sign | 0x7f;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7e;
    /* spacing of representable values around a: 2^(E-3) in binade 2^E
       (E >= -6), 2^-9 for the subnormals below 2^-6 */
    int E;
    frexp(a, &E);           /* a = m * 2^E, m in [0.5, 1): binade exponent E-1 */
    int be = E - 1;
    double quantum = be >= -6 ? ldexp(1.0, be - 3) : ldexp(1.0, -9);
    double q = a / quantum;          /* exact: quantum is a power of two */
    double r = floor(q);
    double frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) == 1.0))
        r += 1.0;
    double v = r * quantum;          /* at most 448: a < 448 rounds to 448 at most */
    /* encode v exactly */
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6))
        return sign | (uint8_t)(v / ldexp(1.0, -9));            /* subnormal */
    int e2;
    double m = frexp(v, &e2);        /* v = m * 2^e2, m in [0.5, 1) */
    int exp_field = e2 - 1 + 7;
    int frac_field = (int)((m * 2.0 - 1.0) * 8.0);
    return sign | (uint8_t)(exp_field << 3) | (uint8_t)frac_field;
}

/* Element idx of a cache of the given storage type, times mult. */
static double kv_value(const void *cache, int64_t idx, int dtype, double mult)
{
    if (dtype == ORC_E4M3)
        return mult * pa_oracle_e4m3_to_f64(((const uint8_t *)cache)[idx]);
    return mult * to_f64(((const uint16_t *)cache)[idx], dtype);
}

/*
 * reshape_and_cache: for every new token t whose slot s = slot_mapping[t] is
 * not negative, copy the raw 16-bit words of key[t, h, :] and value[t, h, :]
 * into k_cache[s / bs, h, s % bs, :] and v_cache[...] for every KV head h.
 * key[t, h, c] is at key[t * key_stride + h * d + c].
 * Returns ORC_BAD_INDEX (and writes nothing further) on a slot >= NB * bs.
 */
int pa_oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                                int64_t key_stride, int64_t value_stride,
                                uint16_t *k_cache, uint16_t *v_cache,
                                const int64_t *slot_mapping, int T, int Hkv, int d,
                                int bs, int64_t NB)
{
    for (int t = 0; t < T; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= NB * (int64_t)bs)
            return ORC_BAD_INDEX;
        int64_t blk = s / bs, off = s % bs;
        for (int h = 0; h < Hkv; ++h) {
            int64_t dst = ((blk * Hkv + h) * bs + off) * d;
            memcpy(k_cache + dst, key + t * key_stride + (int64_t)h * d, (size_t)d * 2);
            memcpy(v_cache + dst, value + t * value_stride + (int64_t)h * d, (size_t)d * 2);
        }
    }
    return ORC_OK;
}

/*
 * reshape_and_cache into an E4M3 cache: like pa_oracle_reshape_and_cache, but
 * every element x of the new rows (fp16/bf16 `dtype`) is stored as the E4M3
 * code of (float)x / scale (an IEEE single-precision quotient), rounded to
 * nearest even with saturation at 448.
 */
int pa_oracle_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value,
                                    int64_t key_stride, int64_t value_stride, uint8_t *k_cache,
                                    uint8_t *v_cache, const int64_t *slot_mapping, int T, int Hkv,
                                    int d, int bs, int64_t NB, int dtype, float k_scale,
                                    float v_scale)
{
    for (int t = 0; t < T; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= NB * (int64_t)bs)
            return ORC_BAD_INDEX;
        int64_t blk = s / bs, off = s % bs;
        for (int h = 0; h < Hkv; ++h) {
            int64_t dst = ((blk * Hkv + h) * bs + off) * d;
            for (int c = 0; c < d; ++c) {
                volatile float kq = (float)to_f64(key[t * key_stride + (int64_t)h * d + c], dtype) / k_scale;
                volatile float vq = (float)to_f64(value[t * value_stride + (int64_t)h * d + c], dtype) / v_scale;
                k_cache[dst + c] = pa_oracle_e4m3_from_f32(kq);
                v_cache[dst + c] = pa_oracle_e4m3_from_f32(vq);
            }
        }
    }
    return ORC_OK;
}

/*
 * Gather the first ctx rows of one sequence's KV head `kvh` into a contiguous
 * fp64 array out[ctx][d]: row j comes from physical block bt_row[j / bs],
 * row j % bs of that block; each element is its exact value times `mult`
 * (the dequantisation scale of an FP8 cache, 1 otherwise).  Returns
 * ORC_BAD_INDEX if a needed table entry is outside [0, NB) or beyond the
 * table's width MB.
 */
int pa_oracle_gather(double *out, const void *cache, int dtype, double mult,
                     const int32_t *bt_row, int MB, int ctx, int Hkv, int kvh, int d, int bs,
                     int64_t NB)
{
    for (int j = 0; j < ctx; ++j) {
        int lb = j / bs;
        if (lb >= MB)
            return ORC_BAD_INDEX;
        int64_t phys = bt_row[lb];
        if (phys < 0 || phys >= NB)
            return ORC_BAD_INDEX;
        int64_t row = ((phys * Hkv + kvh) * bs + (j % bs)) * (int64_t)d;
        for (int c = 0; c < d; ++c)
            out[(int64_t)j * d + c] = kv_value(cache, row + c, dtype, mult);
    }
    return ORC_OK;
}

/*
 * Softmax attention of one query row over n contiguous keys/values:
 *   s_j = scale * sum_c q[c] K[j][c];  m = max_j s_j;  p_j = exp(s_j - m);
 *   l = sum_j p_j;  o = (sum_j p_j V[j]) / l.
 * Writes o[d] (unnormalised sum divided by l), and *m_out, *l_out.
 * n == 0 gives o = 0, m = -inf, l = 0.
 */
static void attend(double *o, double *m_out, double *l_out, const double *q, const double *K,
                   const double *V, int n, int d, double scale, double *s)
{
    for (int c = 0; c < d; ++c)
        o[c] = 0.0;
    if (n == 0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += q[c] * K[(int64_t)j * d + c];
        s[j] = scale * acc;
        if (s[j] > m)
            m = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; ++j) {
        double p = exp(s[j] - m);
        l += p;
        for (int c = 0; c < d; ++c)
            o[c] += p * V[(int64_t)j * d + c];
    }
    for (int c = 0; c < d; ++c)
        o[c] /= l;
    *m_out = m;
    *l_out = l;
}

/*
 * Decode attention for a list of (sequence, query head) pairs.
 *
 * query [B, Hq, d] (dtype fp16/bf16), k_cache/v_cache [NB, Hkv, bs, d] of
 * kv_dtype (fp16, bf16, or E4M3 whose element e stands for k_scale * e or
 * v_scale * e), block_tables [B, MB] int32 (-1 = unused), context_lens [B]
 * int32.  pairs = 2*npairs ints (seq, head); NULL means all B*Hq pairs in
 * (seq, head) order.
 *
 * partition_size == 0: out[k, :] = softmax attention over all ctx tokens.
 * partition_size  > 0: the ctx tokens are cut into partitions of
 *   partition_size; each partition p gets (m_p, l_p, o_p) from `attend`, and
 *   the results are joined by log-sum-exp: M = max_p m_p,
 *   w_p = l_p exp(m_p - M), out = sum_p w_p o_p / sum_p w_p.  If part_m,
 *   part_l, part_o are not NULL they receive the per-partition values,
 *   shaped [npairs, max_parts] and [npairs, max_parts, d]; partitions past a
 *   sequence's end get m = -inf, l = 0, o = 0.
 *
 * nthreads > 0 sets the OpenMP thread count.  Returns ORC_OK, ORC_BAD_ARG,
 * ORC_BAD_INDEX or ORC_NO_MEM.
 */
int pa_oracle_decode(double *out, double *part_m, double *part_l, double *part_o,
                     int max_parts, const uint16_t *query, const void *k_cache,
                     const void *v_cache, const int32_t *block_tables, int MB,
                     const int32_t *context_lens, int B, int Hq, int Hkv, int d, int bs,
                     int64_t NB, float scale, int dtype, int kv_dtype, double k_scale,
                     double v_scale, const int32_t *pairs, int npairs, int partition_size,
                     int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || bs <= 0 || partition_size < 0)
        return ORC_BAD_ARG;
    int n = pairs ? npairs : B * Hq;
    int group = Hq / Hkv;
    double sc = (double)scale;
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int k = 0; k < n; ++k) {
        int i = pairs ? pairs[2 * k] : k / Hq;
        int h = pairs ? pairs[2 * k + 1] : k % Hq;
        double *o = out + (int64_t)k * d;
        if (i < 0 || i >= B || h < 0 || h >= Hq) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORC_BAD_ARG;
            continue;
        }
        int ctx = context_lens[i];
        int kvh = h / group;
        double *K = malloc(sizeof(double) * ((size_t)ctx * d + 1));
        double *V = malloc(sizeof(double) * ((size_t)ctx * d + 1));
        double *q = malloc(sizeof(double) * (size_t)d);
        double *s = malloc(sizeof(double) * ((size_t)ctx + 1));
        if (!K || !V || !q || !s) {
            free(K); free(V); free(q); free(s);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORC_NO_MEM;
            continue;
        }
        const int32_t *bt_row = block_tables + (int64_t)i * MB;
        int rc = pa_oracle_gather(K, k_cache, kv_dtype, k_scale, bt_row, MB, ctx, Hkv, kvh, d,
                                  bs, NB);
        if (rc == ORC_OK)
            rc = pa_oracle_gather(V, v_cache, kv_dtype, v_scale, bt_row, MB, ctx, Hkv, kvh, d,
                                  bs, NB);
        if (rc != ORC_OK) {
            free(K); free(V); free(q); free(s);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = rc;
            continue;
        }
        const uint16_t *qrow = query + ((int64_t)i * Hq + h) * d;
        for (int c = 0; c < d; ++c)
            q[c] = to_f64(qrow[c], dtype);

        double m, l;
        if (partition_size == 0) {
            attend(o, &m, &l, q, K, V, ctx, d, sc, s);
        } else {
            int np = (ctx + partition_size - 1) / partition_size;
            double M = -INFINITY;
            double *pm = malloc(sizeof(double) * ((size_t)np + 1));
            double *pl = malloc(sizeof(double) * ((size_t)np + 1));
            double *po = malloc(sizeof(double) * ((size_t)np * d + 1));
            for (int p = 0; p < np; ++p) {
                int j0 = p * partition_size;
                int len = ctx - j0 < partition_size ? ctx - j0 : partition_size;
                attend(po + (int64_t)p * d, &pm[p], &pl[p], q, K + (int64_t)j0 * d,
                       V + (int64_t)j0 * d, len, d, sc, s);
                if (pm[p] > M)
                    M = pm[p];
            }
            double W = 0.0;
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            for (int p = 0; p < np; ++p) {
                double w = pl[p] * exp(pm[p] - M);
                W += w;
                for (int c = 0; c < d; ++c)
                    o[c] += w * po[(int64_t)p * d + c];
            }
            if (W > 0.0)
                for (int c = 0; c < d; ++c)
                    o[c] /= W;
            if (part_m) {
                for (int p = 0; p < max_parts; ++p) {
                    int have = p < np;
                    part_m[(int64_t)k * max_parts + p] = have ? pm[p] : -INFINITY;
                    part_l[(int64_t)k * max_parts + p] = have ? pl[p] : 0.0;
                    for (int c = 0; c < d; ++c)
                        part_o[((int64_t)k * max_parts + p) * d + c] = have ? po[(int64_t)p * d + c] : 0.0;
                }
            }
            free(pm); free(pl); free(po);
        }
        free(K); free(V); free(q); free(s);
    }
    return status;
}

/*
 * Prefill (chunked-prefill) attention over the paged cache ("Serving engines",
 * How vLLM works: chunked prefill slices a prompt into pieces; "LLM Serving
 * Engine Shootout", 1: prefill attends over all prompt tokens).  The chunk of
 * sequence i is query rows query_start[i] .. query_start[i+1]-1 (q_len_i
 * rows); its K/V are already in the cache, whose sequence now holds ctx_i =
 * context_lens[i] tokens.  Row t of the chunk sits at position
 * p = ctx_i - q_len_i + t and attends causally to tokens 0 .. p:
 *   out[row, h, :] = softmax_j(scale q[row, h] . K_j) V_j over j <= p.
 * query/out [total_q, Hq, d].  Rows are independent; each is the decode
 * computation on the sequence cut after position p.  The caches are read as
 * in pa_oracle_decode: kv_dtype E4M3 means codes standing for k_scale * e and
 * v_scale * e, any other kv_dtype the query's 16-bit type (scales 1).
 */
int pa_oracle_prefill(double *out, const uint16_t *query, const int32_t *query_start,
                      const void *k_cache, const void *v_cache, const int32_t *block_tables,
                      int MB, const int32_t *context_lens, int B, int Hq, int Hkv, int d, int bs,
                      int64_t NB, float scale, int dtype, int kv_dtype, double k_scale,
                      double v_scale, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || bs <= 0)
        return ORC_BAD_ARG;
    int total_q = B > 0 ? query_start[B] : 0;
    int group = Hq / Hkv;
    double sc = (double)scale;
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int k = 0; k < total_q * Hq; ++k) {
        int row = k / Hq, h = k % Hq;
        int i = 0;
        while (i < B && query_start[i + 1] <= row)
            ++i;
        int q_len = query_start[i + 1] - query_start[i];
        int ctx = context_lens[i];
        int pos = ctx - q_len + (row - query_start[i]);
        double *o = out + (int64_t)k * d;
        if (pos < 0 || pos >= ctx) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORC_BAD_ARG;
            continue;
        }
        int n = pos + 1;
        double *K = malloc(sizeof(double) * ((size_t)n * d + 1));
        double *V = malloc(sizeof(double) * ((size_t)n * d + 1));
        double *q = malloc(sizeof(double) * (size_t)d);
        double *s = malloc(sizeof(double) * ((size_t)n + 1));
        int rc = (K && V && q && s) ? ORC_OK : ORC_NO_MEM;
        const int32_t *bt_row = block_tables + (int64_t)i * MB;
        if (rc == ORC_OK)
            rc = pa_oracle_gather(K, k_cache, kv_dtype, k_scale, bt_row, MB, n, Hkv, h / group, d,
                                  bs, NB);
        if (rc == ORC_OK)
            rc = pa_oracle_gather(V, v_cache, kv_dtype, v_scale, bt_row, MB, n, Hkv, h / group, d,
                                  bs, NB);
        if (rc == ORC_OK) {
            const uint16_t *qrow = query + ((int64_t)row * Hq + h) * d;
            for (int c = 0; c < d; ++c)
                q[c] = to_f64(qrow[c], dtype);
            double m, l;
            attend(o, &m, &l, q, K, V, n, d, sc, s);
        } else {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = rc;
        }
        free(K); free(V); free(q); free(s);
    }
    return status;
}

/*
 * Join partition results by log-sum-exp, the combination step stated above,
 * for inputs that did not come from pa_oracle_decode (for example fp32
 * partials rounded from it).  m, l: [n, P]; o: [n, P, d]; nparts[k] partitions
 * of row k are valid.  out[k] = sum_p l_p e^(m_p - M) o_p / sum_p l_p e^(m_p - M).
 */
void pa_oracle_lse_combine(double *out, const double *m, const double *l, const double *o,
                           const int32_t *nparts, int n, int P, int d)
{
    for (int k = 0; k < n; ++k) {
        double M = -INFINITY, W = 0.0;
        double *ok = out + (int64_t)k * d;
        for (int c = 0; c < d; ++c)
            ok[c] = 0.0;
        for (int p = 0; p < nparts[k]; ++p)
            if (m[(int64_t)k * P + p] > M)
                M = m[(int64_t)k * P + p];
        for (int p = 0; p < nparts[k]; ++p) {
            double w = l[(int64_t)k * P + p] * exp(m[(int64_t)k * P + p] - M);
            W += w;
            for (int c = 0; c < d; ++c)
                ok[c] += w * o[((int64_t)k * P + p) * d + c];
        }
        if (W > 0.0)
            for (int c = 0; c < d; ++c)
                ok[c] /= W;
    }
}

int pa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
