/*
 * wfo.c -- fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE (see wfo.h for who may use it and for
 * the passages each function follows).  Plain loops, fp64, no blocking, no
 * online softmax, no reordering: a reader can hold it against the definition.
 *
 * Threads only split the independent (query row, head) outputs; every output
 * is computed by one thread in one fixed order, so results do not depend on
 * the thread count.
 */
#include "wfo.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---- fp8 e4m3 (paged KV quantization, ember "Deliberately out of scope":
 * "paged KV quantization (fp8/int8)") ---------------------------------------
 * OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is
 * subnormal (2^-6 * m/8); S.1111.111 is NaN; no infinities; largest 448. */
double wfo_e4m3_decode(uint8_t code) {
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to the nearest e4m3 value, ties to the even code; magnitudes above 448
 * become 448 (saturating); NaN stays NaN; the sign of zero is kept.  Written as a
 * search over the 127 finite magnitudes, plainly. */
uint8_t wfo_e4m3_encode(float y) {
    if (isnan(y)) return 0x7F;
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    const double a = fabs((double)y);
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double d = fabs(wfo_e4m3_decode((uint8_t)c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return sign | (uint8_t)best;
}

/* ---- exact widening of a stored element to double -------------------- */
static double load_elem(const void* base, int64_t idx, int dtype) {
    if (dtype == WFO_FP8) return wfo_e4m3_decode(((const uint8_t*)base)[idx]);
    if (dtype == WFO_F32) {
        float f;
        memcpy(&f, (const char*)base + idx * 4, 4);
        return (double)f;
    } else {
        uint16_t h;
        uint32_t u;
        float f;
        memcpy(&h, (const char*)base + idx * 2, 2);
        u = ((uint32_t)h) << 16; /* bfloat16 is the top half of a float32 */
        memcpy(&f, &u, 4);
        return (double)f;
    }
}

static int elem_bytes(int dtype) { return dtype == WFO_F32 ? 4 : (dtype == WFO_FP8 ? 1 : 2); }

/* ---- scatter (weft "Cache layouts": write = scatter via slot_mapping) -- */
int wfo_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                          const int64_t* slot_mapping, int64_t T,
                          int64_t N, int64_t P, int64_t H_kv, int64_t D, int dtype) {
    if ((dtype != WFO_F32 && dtype != WFO_BF16) || T < 0 || N < 1 || P < 1 || H_kv < 1 || D < 1)
        return WFO_ERR_ARG;
    const int64_t row_bytes = H_kv * D * elem_bytes(dtype);
    /* validate everything before writing anything */
    for (int64_t t = 0; t < T; ++t)
        if (slot_mapping[t] >= N * P) return WFO_ERR_SLOT;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue; /* padding token: nothing to write */
        const int64_t block = slot / P;
        const int64_t offset = slot % P;
        const int64_t dst = (block * P + offset) * row_bytes;
        memcpy((char*)k_pool + dst, (const char*)k + t * row_bytes, (size_t)row_bytes);
        memcpy((char*)v_pool + dst, (const char*)v + t * row_bytes, (size_t)row_bytes);
    }
    return 0;
}

static int scales_ok(const float* s, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        if (!(s[i] > 0.0f) || isinf(s[i])) return 0;
    return 1;
}

/* ---- scatter into an fp8 pool: code = e4m3(float(x) * (1 / scale_h)), with the
 * reciprocal and the product rounded to float32 (the precision the device uses
 * for this decision); k, v are bfloat16 [T, H_kv, D]; scale_h is KV head h's
 * scale (one per head; a per-tensor scale is the same value for every head) --- */
int wfo_reshape_and_cache_fp8(const void* k, const void* v, void* k_pool, void* v_pool,
                              const int64_t* slot_mapping, int64_t T, int64_t N, int64_t P,
                              int64_t H_kv, int64_t D, const float* k_scales, const float* v_scales) {
    if (T < 0 || N < 1 || P < 1 || H_kv < 1 || D < 1 || !scales_ok(k_scales, H_kv) || !scales_ok(v_scales, H_kv))
        return WFO_ERR_ARG;
    for (int64_t t = 0; t < T; ++t)
        if (slot_mapping[t] >= N * P) return WFO_ERR_SLOT;
    const int64_t row = H_kv * D;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        const int64_t dst = ((slot / P) * P + slot % P) * row;
        for (int64_t i = 0; i < row; ++i) {
            const int64_t h = i / D;
            const float kinv = 1.0f / k_scales[h], vinv = 1.0f / v_scales[h];
            const float xk = (float)load_elem(k, t * row + i, WFO_BF16);
            const float xv = (float)load_elem(v, t * row + i, WFO_BF16);
            volatile float yk = xk * kinv; /* one float32 rounding, no contraction */
            volatile float yv = xv * vinv;
            ((uint8_t*)k_pool)[dst + i] = wfo_e4m3_encode(yk);
            ((uint8_t*)v_pool)[dst + i] = wfo_e4m3_encode(yv);
        }
    }
    return 0;
}

/* ---- block copy for copy-on-write (tiny-vllm-py "Prefix Sharing": a shared
 * partial tail block is copied before a request appends to it) ------------ */
int wfo_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int64_t n_pairs,
                    int64_t N, int64_t P, int64_t H_kv, int64_t D, int dtype) {
    if ((dtype != WFO_F32 && dtype != WFO_BF16 && dtype != WFO_FP8) || n_pairs < 0 || N < 1 || P < 1 ||
        H_kv < 1 || D < 1)
        return WFO_ERR_ARG;
    for (int64_t i = 0; i < 2 * n_pairs; ++i)
        if (pairs[i] < 0 || pairs[i] >= N) return WFO_ERR_BLOCK;
    if (n_pairs == 0) return 0;
    const int64_t block_bytes = P * H_kv * D * elem_bytes(dtype);
    /* every copy reads the pools as they were before the call */
    char* snap = (char*)malloc((size_t)(2 * n_pairs * block_bytes));
    if (!snap) return WFO_ERR_MEM;
    for (int64_t i = 0; i < n_pairs; ++i) {
        const int64_t src = pairs[2 * i];
        memcpy(snap + (2 * i) * block_bytes, (const char*)k_pool + src * block_bytes, (size_t)block_bytes);
        memcpy(snap + (2 * i + 1) * block_bytes, (const char*)v_pool + src * block_bytes, (size_t)block_bytes);
    }
    for (int64_t i = 0; i < n_pairs; ++i) {
        const int64_t dst = pairs[2 * i + 1];
        memcpy((char*)k_pool + dst * block_bytes, snap + (2 * i) * block_bytes, (size_t)block_bytes);
        memcpy((char*)v_pool + dst * block_bytes, snap + (2 * i + 1) * block_bytes, (size_t)block_bytes);
    }
    free(snap);
    return 0;
}

/* ---- one attention row: softmax over positions 0..len-1 of one sequence -- */
typedef struct {
    const void* q;          /* query rows [rows, H_q, D]          */
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* row_req;  /* query row -> request               */
    const int32_t* row_len;  /* query row -> number of positions   */
    int64_t rows, M, H_q, H_kv, D, N, P;
    double scale;
    int dtype;              /* of q (and of the pools unless kv_dtype says fp8) */
    int kv_dtype;
    const float* k_scales;   /* fp8 pools: per KV head, value = scale * stored value; */
    const float* v_scales;   /*   NULL: stored values are the values                */
    double* out;
    int64_t next;            /* shared work counter (atomic)       */
    int status;
} job_t;

/* out_row[d] = sum_p w_p V_p[d] / sum_p w_p with w_p = exp(s_p - max_p s_p),
 * s_p = scale * sum_d q[d] K_p[d]; K_p, V_p read at block_table[p / P],
 * offset p % P, KV head h. */
static int attend_row(const job_t* J, int64_t row, int64_t g, double* s, double* acc) {
    const int64_t b = J->row_req[row];
    const int64_t len = J->row_len[row];
    const int64_t G = J->H_q / J->H_kv;
    const int64_t h = g / G;
    const int64_t qbase = (row * J->H_q + g) * J->D;
    const int32_t* table = J->block_tables + b * J->M;
    const double ks = J->k_scales ? (double)J->k_scales[h] : 1.0;
    const double vs = J->v_scales ? (double)J->v_scales[h] : 1.0;
    double m = -INFINITY;
    for (int64_t p = 0; p < len; ++p) {
        const int64_t block = table[p / J->P];
        const int64_t offset = p % J->P;
        if (block < 0 || block >= J->N) return WFO_ERR_BLOCK;
        const int64_t kbase = ((block * J->P + offset) * J->H_kv + h) * J->D;
        double dot = 0.0;
        for (int64_t d = 0; d < J->D; ++d)
            dot += load_elem(J->q, qbase + d, J->dtype) * (ks * load_elem(J->k_pool, kbase + d, J->kv_dtype));
        s[p] = J->scale * dot;
        if (s[p] > m) m = s[p];
    }
    double den = 0.0;
    for (int64_t d = 0; d < J->D; ++d) acc[d] = 0.0;
    for (int64_t p = 0; p < len; ++p) {
        const double w = exp(s[p] - m);
        const int64_t block = table[p / J->P];
        const int64_t offset = p % J->P;
        const int64_t vbase = ((block * J->P + offset) * J->H_kv + h) * J->D;
        den += w;
        for (int64_t d = 0; d < J->D; ++d)
            acc[d] += w * (vs * load_elem(J->v_pool, vbase + d, J->kv_dtype));
    }
    double* o = J->out + (row * J->H_q + g) * J->D;
    for (int64_t d = 0; d < J->D; ++d) o[d] = acc[d] / den;
    return 0;
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    int64_t maxlen = 1;
    for (int64_t r = 0; r < J->rows; ++r)
        if (J->row_len[r] > maxlen) maxlen = J->row_len[r];
    double* s = (double*)malloc(sizeof(double) * (size_t)maxlen);
    double* acc = (double*)malloc(sizeof(double) * (size_t)J->D);
    if (!s || !acc) {
        __atomic_store_n(&J->status, WFO_ERR_MEM, __ATOMIC_RELAXED);
        free(s);
        free(acc);
        return NULL;
    }
    const int64_t total = J->rows * J->H_q;
    for (;;) {
        const int64_t item = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (item >= total) break;
        const int rc = attend_row(J, item / J->H_q, item % J->H_q, s, acc);
        if (rc) __atomic_store_n(&J->status, rc, __ATOMIC_RELAXED);
    }
    free(s);
    free(acc);
    return NULL;
}

static int run_job(job_t* J, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    J->next = 0;
    J->status = 0;
    if (nthreads == 1) {
        worker(J);
        return J->status;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return WFO_ERR_MEM;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, J) != 0) break;
        ++started;
    }
    if (started == 0) worker(J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return J->status;
}

static int check_common(const int32_t* block_tables, int64_t M, int64_t B, int64_t H_q,
                        int64_t H_kv, int64_t D, int64_t N, int64_t P, int dtype) {
    if ((dtype != WFO_F32 && dtype != WFO_BF16) || B < 0 || M < 1 || H_q < 1 || H_kv < 1 ||
        D < 1 || N < 1 || P < 1 || H_q % H_kv != 0)
        return WFO_ERR_ARG;
    (void)block_tables;
    return 0;
}

/* ---- decode (one query per sequence; attends to all its positions) ---- */
static int decode_impl(double* out, const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* block_tables, int64_t M, const int32_t* seq_lens,
                       int64_t B, int64_t H_q, int64_t H_kv, int64_t D, int64_t N, int64_t P,
                       double scale, int q_dtype, int kv_dtype, const float* k_scales,
                       const float* v_scales, int nthreads) {
    int rc = check_common(block_tables, M, B, H_q, H_kv, D, N, P, q_dtype);
    if (rc) return rc;
    for (int64_t b = 0; b < B; ++b)
        if (seq_lens[b] < 1 || seq_lens[b] > M * P) return WFO_ERR_LEN;
    int32_t* row_req = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
    int32_t* row_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
    if (!row_req || !row_len) {
        free(row_req);
        free(row_len);
        return WFO_ERR_MEM;
    }
    for (int64_t b = 0; b < B; ++b) {
        row_req[b] = (int32_t)b;
        row_len[b] = seq_lens[b];
    }
    job_t J = {q, k_pool, v_pool, block_tables, seq_lens, row_req, row_len,
               B, M, H_q, H_kv, D, N, P, scale, q_dtype, kv_dtype, k_scales, v_scales, out, 0, 0};
    rc = run_job(&J, nthreads);
    free(row_req);
    free(row_len);
    return rc;
}

int wfo_paged_decode(double* out, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* block_tables, int64_t M, const int32_t* seq_lens,
                     int64_t B, int64_t H_q, int64_t H_kv, int64_t D, int64_t N, int64_t P,
                     double scale, int dtype, int nthreads) {
    return decode_impl(out, q, k_pool, v_pool, block_tables, M, seq_lens, B, H_q, H_kv, D, N, P, scale,
                       dtype, dtype, NULL, NULL, nthreads);
}

int wfo_paged_decode_fp8(double* out, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, int64_t M, const int32_t* seq_lens,
                         int64_t B, int64_t H_q, int64_t H_kv, int64_t D, int64_t N, int64_t P,
                         double scale, const float* k_scales, const float* v_scales, int nthreads) {
    if (H_kv < 1 || !scales_ok(k_scales, H_kv) || !scales_ok(v_scales, H_kv)) return WFO_ERR_ARG;
    return decode_impl(out, q, k_pool, v_pool, block_tables, M, seq_lens, B, H_q, H_kv, D, N, P, scale,
                       WFO_BF16, WFO_FP8, k_scales, v_scales, nthreads);
}

/* ---- prefill (causal varlen over the cached prefix plus the new rows) --- */
int wfo_paged_prefill(double* out, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, int64_t M, const int32_t* seq_lens,
                      const int32_t* cu_q_lens, int64_t B, int64_t H_q, int64_t H_kv,
                      int64_t D, int64_t N, int64_t P, double scale, int dtype, int nthreads) {
    int rc = check_common(block_tables, M, B, H_q, H_kv, D, N, P, dtype);
    if (rc) return rc;
    if (cu_q_lens[0] != 0) return WFO_ERR_ARG;
    for (int64_t b = 0; b < B; ++b) {
        const int64_t n = (int64_t)cu_q_lens[b + 1] - cu_q_lens[b];
        if (n < 0) return WFO_ERR_ARG;
        if (seq_lens[b] < n || seq_lens[b] > M * P || (n > 0 && seq_lens[b] < 1)) return WFO_ERR_LEN;
    }
    const int64_t rows = cu_q_lens[B];
    int32_t* row_req = (int32_t*)malloc(sizeof(int32_t) * (size_t)(rows > 0 ? rows : 1));
    int32_t* row_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)(rows > 0 ? rows : 1));
    if (!row_req || !row_len) {
        free(row_req);
        free(row_len);
        return WFO_ERR_MEM;
    }
    for (int64_t b = 0; b < B; ++b) {
        const int64_t n = (int64_t)cu_q_lens[b + 1] - cu_q_lens[b];
        const int64_t c = seq_lens[b] - n; /* cached prefix length */
        for (int64_t i = 0; i < n; ++i) {
            row_req[cu_q_lens[b] + i] = (int32_t)b;
            row_len[cu_q_lens[b] + i] = (int32_t)(c + i + 1); /* positions 0 .. c+i */
        }
    }
    job_t J = {q, k_pool, v_pool, block_tables, seq_lens, row_req, row_len,
               rows, M, H_q, H_kv, D, N, P, scale, dtype, dtype, NULL, NULL, out, 0, 0};
    rc = run_job(&J, nthreads);
    free(row_req);
    free(row_len);
    return rc;
}
