/*
 * pkd_oracle.c -- plain fp64 CPU oracle for batched paged-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Loaded by the tests and by the CPU-baseline leg of
 * the benchmark through ctypes; nothing on the product path links or calls it,
 * and it shares no code with the CUDA path.
 *
 * It computes the plain definition, one (request, qo head) row at a time, in
 * double precision, parallelised over rows with OpenMP:
 *   - page-table walk: request b owns pages indices[indptr[b] .. indptr[b+1]-1],
 *     every page full but the last, which holds last_page_len[b] tokens
 *     (FlashInfer deep dive, snackonai.com, "The Code, Annotated", snippet one);
 *   - s_j = sm_scale * <q_h, k_j>, m = max_j s_j,
 *     lse = m + ln sum_j exp(s_j - m), o = sum_j exp(s_j - lse) v_j
 *     (decode attention of the quickstart single_decode_with_kv_cache, ai-tldr.dev
 *     tool card, "Getting started", step 4); qo head h reads kv head h / (Hq/Hk);
 *   - an empty request gives o = 0, lse = -inf.
 * Element decoding follows the published formats: IEEE 754 binary16, bfloat16
 * (the upper half of an IEEE binary32), and OCP FP8 E4M3 ("fn": no infinities,
 * S.1111.111 is NaN).  fp8 values are multiplied by their per-kv-head scale.
 *
 * Pool layout: element (page, slot, kv_head, d) sits at
 *   page * page_stride + slot * Hk * D + kv_head * D + d      (NHD pages).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_F32 = 3, ORC_F64 = 4 };

double orc_decode_bf16(uint16_t bits) {
  union { uint32_t u; float f; } x;
  x.u = ((uint32_t)bits) << 16;
  return (double)x.f;
}

double orc_decode_f16(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1f;
  int m = bits & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(1024 + m), e - 25);            /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

double orc_decode_e4m3(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int e = (bits >> 3) & 0xf;
  int m = bits & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);                  /* subnormal: m/8 * 2^-6 */
  else v = ldexp((double)(8 + m), e - 10);               /* (1 + m/8) * 2^(e-7) */
  return sign ? -v : v;
}

static double load_elem(const void* base, int dtype, int64_t i) {
  switch (dtype) {
    case ORC_F16: return orc_decode_f16(((const uint16_t*)base)[i]);
    case ORC_BF16: return orc_decode_bf16(((const uint16_t*)base)[i]);
    case ORC_E4M3: return orc_decode_e4m3(((const uint8_t*)base)[i]);
    case ORC_F32: return (double)((const float*)base)[i];
    default: return ((const double*)base)[i];
  }
}

/* One output row (b, h).  Returns 0, or -1 on allocation failure. */
static int decode_row(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                      int kv_dtype, int64_t page_stride, int P, int Hq, int Hk, int D,
                      const int32_t* indptr, const int32_t* indices, const int32_t* last,
                      double sm_scale, const double* k_scale, const double* v_scale, int b, int h,
                      double* o_row, double* lse_out) {
  const int g = Hq / Hk;
  const int kvh = h / g;
  const int32_t p0 = indptr[b], p1 = indptr[b + 1];
  int64_t L = 0;
  for (int32_t i = p0; i < p1; ++i) L += (i == p1 - 1) ? last[b] : P;
  for (int d = 0; d < D; ++d) o_row[d] = 0.0;
  if (L == 0) { *lse_out = -INFINITY; return 0; }
  double* qv = (double*)malloc(sizeof(double) * (size_t)D);
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  if (!qv || !s) { free(qv); free(s); return -1; }
  for (int d = 0; d < D; ++d) qv[d] = load_elem(q, q_dtype, ((int64_t)b * Hq + h) * D + d);
  const double ks = k_scale ? k_scale[kvh] : 1.0;
  const double vs = v_scale ? v_scale[kvh] : 1.0;
  /* scores, in sequence order */
  int64_t j = 0;
  for (int32_t i = p0; i < p1; ++i) {
    const int64_t page = indices[i];
    const int n = (i == p1 - 1) ? last[b] : P;
    for (int t = 0; t < n; ++t, ++j) {
      const int64_t base = page * page_stride + ((int64_t)t * Hk + kvh) * D;
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += qv[d] * (load_elem(k_cache, kv_dtype, base + d) * ks);
      s[j] = sm_scale * acc;
    }
  }
  double m = s[0];
  for (int64_t t = 1; t < L; ++t) if (s[t] > m) m = s[t];
  double sum = 0.0;
  for (int64_t t = 0; t < L; ++t) sum += exp(s[t] - m);
  const double lse = m + log(sum);
  j = 0;
  for (int32_t i = p0; i < p1; ++i) {
    const int64_t page = indices[i];
    const int n = (i == p1 - 1) ? last[b] : P;
    for (int t = 0; t < n; ++t, ++j) {
      const int64_t base = page * page_stride + ((int64_t)t * Hk + kvh) * D;
      const double w = exp(s[j] - lse);
      for (int d = 0; d < D; ++d) o_row[d] += w * (load_elem(v_cache, kv_dtype, base + d) * vs);
    }
  }
  *lse_out = lse;
  free(qv);
  free(s);
  return 0;
}

/*
 * Decode attention for the listed rows (rows[2*r] = b, rows[2*r+1] = h), or for
 * every (b, h) when rows == NULL.  o is [B, Hq, D] and lse [B, Hq] (double);
 * rows not listed are left untouched.  num_threads <= 0 keeps the OpenMP
 * default.  Returns 0 on success, -1 on a bad argument or allocation failure.
 */
int pkd_oracle_paged_decode(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                            int kv_dtype, int64_t page_stride, int page_size, int batch,
                            int num_qo_heads, int num_kv_heads, int head_dim,
                            const int32_t* kv_indptr, const int32_t* kv_page_indices,
                            const int32_t* kv_last_page_len, double sm_scale,
                            const double* k_scale, const double* v_scale, const int32_t* rows,
                            int64_t n_rows, int num_threads, double* o, double* lse) {
  if (!q || !k_cache || !v_cache || !kv_indptr || !o || !lse) return -1;
  if (num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 || head_dim <= 0) return -1;
  const int64_t total = rows ? n_rows : (int64_t)batch * num_qo_heads;
  int failed = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
  for (int64_t r = 0; r < total; ++r) {
    const int b = rows ? rows[2 * r] : (int)(r / num_qo_heads);
    const int h = rows ? rows[2 * r + 1] : (int)(r % num_qo_heads);
    double* o_row = o + ((int64_t)b * num_qo_heads + h) * head_dim;
    double* l_out = lse + (int64_t)b * num_qo_heads + h;
    if (decode_row(q, q_dtype, k_cache, v_cache, kv_dtype, page_stride, page_size, num_qo_heads,
                   num_kv_heads, head_dim, kv_indptr, kv_page_indices, kv_last_page_len, sm_scale,
                   k_scale, v_scale, b, h, o_row, l_out) != 0)
      failed |= 1;
  }
  return failed ? -1 : 0;
}

/* Threads OpenMP would use (1 without OpenMP). */
int pkd_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
