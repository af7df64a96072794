/*
 * wfo.h -- fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Definitions followed (page titles and sections):
 *   - weft, "Cache layouts": per-layer paged view [N, P, H_kv, D]; writes are a
 *     scatter through slot_mapping, reads a gather through block_table.
 *   - ember, "The core idea, in one picture": position p of a sequence lives in
 *     block block_table[p // P] at offset p % P.
 *   - tiny-vllm-py, "KV Cache / Mental Model" and "Mistakes I made": decode
 *     attends to every cached position including the new token (not causal);
 *     prefill is causal.
 *   - weft, "Shapes and symbols": H_q / H_kv query heads share one KV head.
 * Attention is exact softmax(q K^T * scale) V, evaluated as written in fp64.
 *
 * Storage types: 0 = float32, 1 = bfloat16 (raw 16-bit patterns).  Values are
 * widened exactly to double before any arithmetic.  Results are double.
 * All functions return 0 on success and a negative code on a bad argument
 * (they never read or write out of bounds on a bad table or slot).
 */
#ifndef WFO_H
#define WFO_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WFO_F32 0
#define WFO_BF16 1
#define WFO_FP8 2   /* e4m3 pool codes (queries and new rows stay bfloat16) */

#define WFO_ERR_ARG   (-1)   /* shape / dtype argument invalid            */
#define WFO_ERR_SLOT  (-2)   /* slot >= N*P                               */
#define WFO_ERR_BLOCK (-3)   /* block id outside [0, N)                   */
#define WFO_ERR_LEN   (-4)   /* seq_len < 1, > M*P, or q_len > seq_len    */
#define WFO_ERR_MEM   (-5)   /* host allocation failed                    */

/* Scatter: for every t with slot_mapping[t] >= 0, copy the [H_kv, D] rows of
 * k[t] and v[t] into block slot/P, offset slot%P of k_pool / v_pool (a byte
 * copy; no conversion).  Negative slots are skipped. */
int wfo_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                          const int64_t* slot_mapping, int64_t T,
                          int64_t N, int64_t P, int64_t H_kv, int64_t D, int dtype);

/* fp8 e4m3 (OCP): the exact value of a code, and float -> code rounding to
 * nearest (ties to the even code), saturating at +-448, NaN kept. */
double wfo_e4m3_decode(uint8_t code);
uint8_t wfo_e4m3_encode(float y);

/* Scatter into fp8 pools: k, v are bfloat16 [T, H_kv, D]; an element of KV head h
 * is stored as e4m3(float(x) * (1.0f / scale[h])), the reciprocal and product
 * rounded to float32.  A stored code c of head h stands for scale[h] * value(c).
 * k_scales, v_scales: H_kv finite positive scales each. */
int wfo_reshape_and_cache_fp8(const void* k, const void* v, void* k_pool, void* v_pool,
                              const int64_t* slot_mapping, int64_t T, int64_t N, int64_t P,
                              int64_t H_kv, int64_t D, const float* k_scales, const float* v_scales);

/* Decode over fp8 pools (q bfloat16): K_p of head h = k_scales[h] * value(code),
 * V_p likewise. */
int wfo_paged_decode_fp8(double* out, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, int64_t M, const int32_t* seq_lens,
                         int64_t B, int64_t H_q, int64_t H_kv, int64_t D, int64_t N, int64_t P,
                         double scale, const float* k_scales, const float* v_scales, int nthreads);

/* Copy-on-write block copy: for every pair i, block pairs[2i+1] of both pools
 * becomes a byte copy of block pairs[2i] as it was before the call (a pair list
 * with a repeated destination applies its pairs in order).  Any id outside
 * [0, N) fails before anything is written. */
int wfo_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int64_t n_pairs,
                    int64_t N, int64_t P, int64_t H_kv, int64_t D, int dtype);

/* Decode: out[b, g, :] = softmax_p(scale * q[b,g,:] . K_p) V_p over positions
 * p = 0 .. seq_lens[b]-1 of KV head g / (H_q/H_kv), gathered through
 * block_tables[b, :] (row-major [B, M]).  q is [B, H_q, D] in storage dtype. */
int wfo_paged_decode(double* out, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* block_tables, int64_t M, const int32_t* seq_lens,
                     int64_t B, int64_t H_q, int64_t H_kv, int64_t D, int64_t N, int64_t P,
                     double scale, int dtype, int nthreads);

/* Prefill: request b owns query rows cu_q_lens[b] .. cu_q_lens[b+1]-1 of q
 * ([T_total, H_q, D]); with n_b = its row count and c_b = seq_lens[b] - n_b,
 * row i attends causally over positions 0 .. c_b + i. */
int wfo_paged_prefill(double* out, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, int64_t M, const int32_t* seq_lens,
                      const int32_t* cu_q_lens, int64_t B, int64_t H_q, int64_t H_kv,
                      int64_t D, int64_t N, int64_t P, double scale, int dtype, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
