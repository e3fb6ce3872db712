/*
 * Host-side fills of the seeded synthetic inputs (see synth_gen.h).
 * Used by the CPU oracle and by tests; holds none of the layer's arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include "synth_gen.h"

/* x rows for the listed tokens: bf16(z) or bf16(outlier_scale * z) for rows
 * whose flag is set.  rows[i] is a token index; out is [n_rows, H]. */
void synth_host_x_rows(uint64_t seed, int64_t H, const int64_t* rows, int64_t n_rows,
                       const uint8_t* outlier_flag, float outlier_scale, uint16_t* out) {
  uint64_t key = synth_key(seed, SYNTH_T_X);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t t = rows[i];
    float s = (outlier_flag && outlier_flag[t]) ? outlier_scale : 1.0f;
    for (int64_t h = 0; h < H; ++h) {
      float z = synth_normal(key, (uint64_t)(t * H + h));
      out[i * H + h] = synth_bf16_bits(s == 1.0f ? z : s * z);
    }
  }
}

/* Router weight W_r [E,H] = bf16(z * inv_sqrt_h). */
void synth_host_router(uint64_t seed, int64_t E, int64_t H, float inv_sqrt_h, uint16_t* out) {
  uint64_t key = synth_key(seed, SYNTH_T_ROUTER);
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < E; ++e)
    for (int64_t h = 0; h < H; ++h)
      out[e * H + h] = synth_bf16_bits(synth_normal(key, (uint64_t)(e * H + h)) * inv_sqrt_h);
}

/* Uniform router bias b[e] = fp32(lo + (hi - lo) * u), u = u24 / 2^24, in fp64. */
void synth_host_bias_uniform(uint64_t seed, int64_t E, double lo, double hi, float* out) {
  uint64_t key = synth_key(seed, SYNTH_T_BIAS);
  for (int64_t e = 0; e < E; ++e) {
    double u = (double)synth_u24(key, (uint64_t)e) * 5.9604644775390625e-08;
    double span = hi - lo;
    double v = span * u;
    v = lo + v;
    out[e] = (float)v;
  }
}

/* Popularity rank (1..E) of each expert: experts sorted by a seeded hash. */
static uint64_t g_rank_key;
static int cmp_rank(const void* a, const void* b) {
  int64_t ea = *(const int64_t*)a, eb = *(const int64_t*)b;
  uint64_t ha = synth_h64(g_rank_key, (uint64_t)ea), hb = synth_h64(g_rank_key, (uint64_t)eb);
  if (ha != hb) return ha < hb ? -1 : 1;
  return ea < eb ? -1 : (ea > eb);
}
void synth_host_expert_rank(uint64_t seed, int64_t E, int32_t* rank_out) {
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
  for (int64_t e = 0; e < E; ++e) order[e] = e;
  g_rank_key = synth_key(seed, SYNTH_T_RANK);
  qsort(order, (size_t)E, sizeof(int64_t), cmp_rank);
  for (int64_t r = 0; r < E; ++r) rank_out[order[r]] = (int32_t)(r + 1);
  free(order);
}

/* Zipf-skewed bias: b_e = -c * s * ln(rank_e); the n_cold least popular
 * experts get cold_bias instead.  Computed in fp64, rounded to fp32 once. */
void synth_host_bias_zipf(uint64_t seed, int64_t E, double c, double s, int64_t n_cold,
                          double cold_bias, float* out) {
  int32_t* rank = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  synth_host_expert_rank(seed, E, rank);
  for (int64_t e = 0; e < E; ++e) {
    double v = (rank[e] > E - n_cold) ? cold_bias : -(c * s) * log((double)rank[e]);
    out[e] = (float)v;
  }
  free(rank);
}

/* Outlier token rows: the n_out tokens with the smallest seeded hash. */
static uint64_t g_out_key;
static int cmp_out(const void* a, const void* b) {
  int64_t ta = *(const int64_t*)a, tb = *(const int64_t*)b;
  uint64_t ha = synth_h64(g_out_key, (uint64_t)ta), hb = synth_h64(g_out_key, (uint64_t)tb);
  if (ha != hb) return ha < hb ? -1 : 1;
  return ta < tb ? -1 : (ta > tb);
}
void synth_host_outlier_flags(uint64_t seed, int64_t T, int64_t n_out, uint8_t* flags) {
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);
  for (int64_t t = 0; t < T; ++t) { order[t] = t; flags[t] = 0; }
  g_out_key = synth_key(seed, SYNTH_T_OUTLIER);
  qsort(order, (size_t)T, sizeof(int64_t), cmp_out);
  for (int64_t i = 0; i < n_out && i < T; ++i) flags[order[i]] = 1;
  free(order);
}

/* One expert's fp32 master matrix [N,K] = z * inv_sqrt_k for tensor
 * (SYNTH_T_GATE / UP / DOWN); element (e, n, kk) has index (e*N + n)*K + kk. */
void synth_host_expert_matrix(uint64_t seed, int tensor, int64_t e, int64_t N, int64_t K,
                              float inv_sqrt_k, float* out) {
  uint64_t key = synth_key(seed, (uint32_t)tensor);
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t kk = 0; kk < K; ++kk)
      out[n * K + kk] = synth_normal(key, (uint64_t)((e * N + n) * K + kk)) * inv_sqrt_k;
}

/* Raw generator outputs, for pinning the generator itself. */
void synth_host_normals(uint64_t seed, int tensor, int64_t i0, int64_t n, float* out) {
  uint64_t key = synth_key(seed, (uint32_t)tensor);
  for (int64_t i = 0; i < n; ++i) out[i] = synth_normal(key, (uint64_t)(i0 + i));
}
