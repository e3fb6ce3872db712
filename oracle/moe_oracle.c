/*
 * CPU oracle of the routed block-scaled MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow reference that the
 * CUDA library is checked against.  Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load it.  It shares no code with
 * the CUDA library and the library never calls it.
 *
 * What it computes, and where each step comes from (pages on the model
 * release of Inkling 2 Small):
 *   - "SGLang and Miles Add Day-0 Support for Inkling 2 Small", section
 *     Performance, kernel-fusion bullet: one router kernel does the sigmoid,
 *     the bias and the top-k; activation quantisation sits inside the expert
 *     GEMMs.
 *   - "Inkling-2-Small" (SGLang cookbook), section 2 Configuration Tips,
 *     MegaMoE paragraph: the fused unit is dispatch, both expert GEMMs, the
 *     capped SwiGLU and the combine; Parallelism paragraph: NVFP4 activation
 *     scales cover an expert's full input width.
 *   - "TML Inkling 2 Small at Day 0" (TokenSpeed), table "What's new": 384
 *     experts, top-8, no shared experts, capped SwiGLU; NVFP4 and MXFP8
 *     expert formats.
 *   - "inkling-2-small" (Miles docs), section 1 Model Introduction:
 *     sigmoid-routed MoE with soft-capped SwiGLU; section 5.3: W4A4 / W8A8
 *     activation quantisation.
 * The pages name these steps but give no formulas; the readings taken where
 * they are silent are written next to each function below.
 *
 * Arithmetic rules: quantiser steps are single IEEE fp32 operations in the
 * stated order (built with -ffp-contract=off, no fast-math), so codes are
 * reproducible bit for bit; every sum and product after decoding is fp64.
 *
 * Parity: every function here is pinned by tests/test_oracle_pins.py
 * (worked micro-cases, closed forms, invariants, brute force on tiny shapes).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================== */
/* O1. Number formats.  The pages give only the names NVFP4 and MXFP8       */
/* ("Inkling-2-Small" cookbook, Checkpoints paragraph; TokenSpeed table,    */
/* Checkpoint row).  Reading: the public OCP MX v1.0 / NVIDIA definitions.  */
/* ======================================================================== */

/* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(uint8_t code) {
  double m = E2M1_MAG[code & 7u];
  return (code & 8u) ? -m : m;
}

/* Nearest representable magnitude, ties to the even code; saturating.
 * The sign bit follows the input, also when the result is zero. */
uint8_t orc_e2m1_encode(float v) {
  uint8_t sign = signbit(v) ? 8u : 0u;
  double a = fabs((double)v);
  if (!(a < 6.0)) return (uint8_t)(sign | 7u); /* saturate (NaN input: unspecified) */
  int i = 0;
  while (!(E2M1_MAG[i] <= a && a < E2M1_MAG[i + 1])) ++i;
  double dlo = a - E2M1_MAG[i], dhi = E2M1_MAG[i + 1] - a;
  int q;
  if (dlo < dhi) q = i;
  else if (dhi < dlo) q = i + 1;
  else q = (i % 2 == 0) ? i : i + 1; /* tie: even code */
  return (uint8_t)(sign | (uint8_t)q);
}

/* E4M3 (the "FN" variant): bias 7, no infinities, 0x7F/0xFF are NaN,
 * largest finite 448 = 0x7E, subnormals m * 2^-9. */
double orc_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

/* Nearest finite E4M3 value (codes 0x00..0x7E are increasing in value),
 * ties to the even code, magnitudes above 448 saturate to 448.  The sign bit
 * follows the input, also when the result is zero. */
uint8_t orc_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80u : 0u;
  double a = fabs((double)v);
  if (!(a < 448.0)) return (uint8_t)(sign | 0x7Eu); /* saturate (NaN input: unspecified) */
  int lo = 0, hi = 0x7E; /* invariant: value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (orc_e4m3_value((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  double dlo = a - orc_e4m3_value((uint8_t)lo), dhi = orc_e4m3_value((uint8_t)hi) - a;
  int q;
  if (dlo < dhi) q = lo;
  else if (dhi < dlo) q = hi;
  else q = (lo % 2 == 0) ? lo : hi;
  return (uint8_t)(sign | (uint8_t)q);
}

/* E8M0: an unsigned power of two 2^(c-127); 0xFF is NaN. */
double orc_e8m0_value(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

double orc_bf16_value(uint16_t bits) {
  union { uint32_t u; float f; } c;
  c.u = (uint32_t)bits << 16;
  return (double)c.f;
}

/* Round an fp64 value to the nearest bf16 (8 significant bits), ties to
 * even.  Finite, in-range inputs only. */
uint16_t orc_bf16_from_f64(double v) {
  if (v == 0.0) return signbit(v) ? 0x8000u : 0u;
  int e = ilogb(v);
  if (e < -126) e = -126;               /* bf16 subnormal quantum 2^-133 */
  double quantum = ldexp(1.0, e - 7);
  double r = nearbyint(v / quantum) * quantum; /* default mode: ties to even */
  union { float f; uint32_t u; } c;
  c.f = (float)r;                       /* exact: r has <= 8 significant bits */
  return (uint16_t)(c.u >> 16);
}

/* ======================================================================== */
/* O4. NVFP4 quantiser.  Format named on the cookbook page (Checkpoints) and */
/* on the TokenSpeed page (Checkpoint row); the Miles page (section 5.2)    */
/* says NVFP4 carries global scales that are recomputed on re-encode;        */
/* the cookbook (Parallelism) says activation scales span the expert's full */
/* input width.  Reading: one fp32 global per row of K (activations) or per  */
/* whole matrix (weights), E4M3 scale per 16-element block along K, E2M1    */
/* codes packed two per byte, low nibble = lower k index.                   */
/* Steps, each one fp32 operation rounded to nearest:                        */
/*   G = 2688 / amax (G = 1 if amax = 0); g = 1 / G (stored, decode factor)  */
/*   sb = E4M3((amax_b / 6) * G); inv = G / sb; q = E2M1(v * inv)            */
/*   decode: v^ = e2m1(q) * sb * g                                           */
/* ======================================================================== */

static float absmax_f32(const float* v, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > m) m = a;
  }
  return m;
}

static void nvfp4_row(const float* v, int64_t K, float G, uint8_t* codes, uint8_t* sf) {
  for (int64_t b = 0; b < K / 16; ++b) {
    const float* blk = v + b * 16;
    float amax_b = absmax_f32(blk, 16);
    float t = amax_b / 6.0f;
    t = t * G;
    uint8_t sb = orc_e4m3_encode(t);
    sf[b] = sb;
    float inv = 0.0f;
    if (sb != 0) inv = G / (float)orc_e4m3_value(sb);
    for (int i = 0; i < 16; i += 2) {
      uint8_t q0 = 0, q1 = 0;
      if (sb != 0) {
        q0 = orc_e2m1_encode(blk[i] * inv);
        q1 = orc_e2m1_encode(blk[i + 1] * inv);
      }
      codes[(b * 16 + i) / 2] = (uint8_t)(q0 | (q1 << 4));
    }
  }
}

static float nvfp4_global_G(float amax) {
  if (amax == 0.0f) return 1.0f;
  return 2688.0f / amax;
}

/* v [rows, K] fp32 -> codes [rows, K/2], sf [rows, K/16], g [rows] (or g[0]
 * for the whole matrix when per_tensor != 0). */
void orc_nvfp4_quantize(const float* v, int64_t rows, int64_t K, int per_tensor, uint8_t* codes,
                        uint8_t* sf, float* g) {
  if (per_tensor) {
    float amax = 0.0f;
    for (int64_t r = 0; r < rows; ++r) {
      float m = absmax_f32(v + r * K, K);
      if (m > amax) amax = m;
    }
    float G = nvfp4_global_G(amax);
    g[0] = 1.0f / G;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) nvfp4_row(v + r * K, K, G, codes + r * (K / 2), sf + r * (K / 16));
  } else {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      float G = nvfp4_global_G(absmax_f32(v + r * K, K));
      g[r] = 1.0f / G;
      nvfp4_row(v + r * K, K, G, codes + r * (K / 2), sf + r * (K / 16));
    }
  }
}

/* Static activation globals (act_global_mode 1): row r is encoded with the
 * given decode factor g_rows[r], G = 1/g (fp32); block maxima beyond
 * 2688 g saturate.  g_out[r] = g_rows[r]. */
void orc_nvfp4_quantize_static(const float* v, int64_t rows, int64_t K, const float* g_rows, uint8_t* codes,
                               uint8_t* sf, float* g_out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    float G = 1.0f / g_rows[r];
    g_out[r] = g_rows[r];
    nvfp4_row(v + r * K, K, G, codes + r * (K / 2), sf + r * (K / 16));
  }
}

void orc_nvfp4_decode(const uint8_t* codes, const uint8_t* sf, const float* g, int64_t rows, int64_t K,
                      int per_tensor, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double gr = (double)(per_tensor ? g[0] : g[r]);
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t q = (k % 2 == 0) ? (byte & 15u) : (byte >> 4);
      out[r * K + k] = orc_e2m1_value(q) * orc_e4m3_value(sf[r * (K / 16) + k / 16]) * gr;
    }
  }
}

/* ======================================================================== */
/* O5. MXFP8 quantiser.  Format named on the cookbook page (Checkpoints) and */
/* the TokenSpeed page (Checkpoint row).  Reading: OCP MX v1.0 — one E8M0   */
/* scale per 32-element block along K, E4M3 codes.                          */
/*   mode 0 (OCP): e = floor(log2 amax_b); X = 2^(e - 8)  (8 = emax of E4M3) */
/*   mode 1 (no saturation): X = 2^ceil(log2(amax_b / 448))                 */
/*   stored = clamp(log2 X + 127, 0, 254); q = E4M3(v * 2^(127 - stored))   */
/*   all-zero block: stored 0, codes 0.                                      */
/* ======================================================================== */

static uint8_t mx_scale_code(float amax_b, int mode) {
  int e;
  if (mode == 0) {
    int ex;
    frexpf(amax_b, &ex); /* amax_b = f * 2^ex, f in [0.5, 1): floor(log2) = ex - 1 */
    e = (ex - 1) - 8;
  } else {
    float r = amax_b / 448.0f;
    int ex;
    float f = frexpf(r, &ex);
    e = (f == 0.5f) ? ex - 1 : ex; /* ceil(log2 r) */
  }
  int s = e + 127;
  if (s < 0) s = 0;
  if (s > 254) s = 254;
  return (uint8_t)s;
}

void orc_mxfp8_quantize(const float* v, int64_t rows, int64_t K, int mode, uint8_t* codes, uint8_t* sf) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < K / 32; ++b) {
      const float* blk = v + r * K + b * 32;
      float amax_b = absmax_f32(blk, 32);
      uint8_t s = 0;
      if (amax_b != 0.0f) s = mx_scale_code(amax_b, mode);
      sf[r * (K / 32) + b] = s;
      float mul = ldexpf(1.0f, 127 - (int)s); /* exact power of two */
      for (int i = 0; i < 32; ++i)
        codes[r * K + b * 32 + i] = (amax_b == 0.0f) ? 0u : orc_e4m3_encode(blk[i] * mul);
    }
  }
}

void orc_mxfp8_decode(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t K, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k)
      out[r * K + k] = orc_e4m3_value(codes[r * K + k]) * orc_e8m0_value(sf[r * (K / 32) + k / 32]);
}

/* ======================================================================== */
/* O2. Router.  SGLang blog, Performance, kernel-fusion bullet (sigmoid,    */
/* bias and top-k in that order); Miles docs section 1 (sigmoid routing,   */
/* 384 routed experts, 8 per token).  Readings: l = x . W_r (fp64 over the  */
/* inputs); s = 1 / (1 + exp(-l)); the bias is added after the sigmoid and   */
/* steers selection only: key = s + b; top-k by key descending, ties to the */
/* lower expert index; slots j = 0..k-1 in that order; weights              */
/* w_j = routed_scale * s_j / sum_i s_i  (bias_in_weights = 1 uses the keys */
/* instead of s).                                                           */
/* ======================================================================== */

void orc_router_logits(int64_t T, int64_t H, int64_t E, const uint16_t* x, const uint16_t* wr,
                       double* logits, double* absdot) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        double p = orc_bf16_value(x[t * H + h]) * orc_bf16_value(wr[e * H + h]);
        acc += p;
        aacc += fabs(p);
      }
      logits[t * E + e] = acc;
      if (absdot) absdot[t * E + e] = aacc;
    }
  }
}

/* Select and normalise from logits [T,E]. keys_out [T,E] optional. */
void orc_router_select(int64_t T, int64_t E, int64_t k, const double* logits, const float* bias,
                       int bias_in_weights, double routed_scale, int32_t* idx, double* w, double* keys_out) {
  double* key = (double*)malloc(sizeof(double) * (size_t)E);
  double* sig = (double*)malloc(sizeof(double) * (size_t)E);
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      sig[e] = 1.0 / (1.0 + exp(-logits[t * E + e]));
      key[e] = sig[e] + (double)bias[e];
      taken[e] = 0;
      if (keys_out) keys_out[t * E + e] = key[e];
    }
    double den = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || key[e] > key[best]) best = e; /* strict: ties keep the lower index */
      }
      taken[best] = 1;
      idx[t * k + j] = (int32_t)best;
      den += bias_in_weights ? key[best] : sig[best];
    }
    for (int64_t j = 0; j < k; ++j) {
      int64_t e = idx[t * k + j];
      double num = bias_in_weights ? key[e] : sig[e];
      w[t * k + j] = routed_scale * (num / den);
    }
  }
  free(key);
  free(sig);
  free(taken);
}

/* ======================================================================== */
/* O3. Dispatch (cookbook, MegaMoE paragraph: dispatch step).  Pairs (t, j) */
/* with expert e = idx[t,j] are listed grouped by expert ascending and, in  */
/* an expert, by token ascending.  counts[e], offsets = exclusive scan      */
/* (E+1 entries), perm[p] = t*k + j, pair_pos[t*k + j] = p.                 */
/* ======================================================================== */

void orc_dispatch(int64_t T, int64_t E, int64_t k, const int32_t* idx, int32_t* counts, int32_t* offsets,
                  int32_t* perm, int32_t* pair_pos) {
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t p = 0; p < T * k; ++p) counts[idx[p]] += 1;
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int64_t p = 0;
  for (int64_t e = 0; e < E; ++e)
    for (int64_t t = 0; t < T; ++t)
      for (int64_t j = 0; j < k; ++j)
        if (idx[t * k + j] == e) {
          perm[p] = (int32_t)(t * k + j);
          pair_pos[t * k + j] = (int32_t)p;
          ++p;
        }
}

/* ======================================================================== */
/* O6. Expert FFN of one expert over n pairs (cookbook MegaMoE paragraph:   */
/* the two expert GEMMs with the capped SwiGLU between them; TokenSpeed     */
/* table and Miles section 1 name the capped / soft-capped SwiGLU; Miles    */
/* 5.3: W4A4 / W8A8 activation quantisation).                               */
/*   g = W_gate a, u = W_up a          (fp64 over decoded operands)         */
/*   cap(v) = c * tanh(v / c)  (c = 0: no cap)   [reading: form and c]       */
/*   h = silu(cap g) * cap u = cap g / (1 + exp(-cap g)) * cap u             */
/*   h rounded to bf16 [reading: the unfused path's rounding point]          */
/*   h quantised along F (NVFP4 per-row global or the expert's static one,   */
/*   or MXFP8), decoded                                                      */
/*   y = W_down h^                                                           */
/* Wg, Wu: [F,H] decoded fp64; Wd: [H,F]; a: [n,H] decoded activations.      */
/* Optional outputs: h_bf16 [n,F]; h codes / scales / globals.              */
/* ======================================================================== */

void orc_expert_ffn(int fmt /*0 nvfp4, 1 mxfp8*/, int64_t H, int64_t F, double cap, int h_round_bf16,
                    int mx_mode, const double* Wg, const double* Wu, const double* Wd, int64_t n,
                    const double* a, double* y, uint16_t* h_bf16_out, uint8_t* hq_codes, uint8_t* hq_sf,
                    float* hq_g, const float* h_static_g /* NVFP4: the expert's static h global, or NULL */) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t p = 0; p < n; ++p) {
    const double* ap = a + p * H;
    float* hrow = (float*)malloc(sizeof(float) * (size_t)F);
    double* hdec = (double*)malloc(sizeof(double) * (size_t)F);
    int64_t code_bytes = (fmt == 0) ? F / 2 : F;
    int64_t sf_n = (fmt == 0) ? F / 16 : F / 32;
    uint8_t* codes = (uint8_t*)malloc((size_t)code_bytes);
    uint8_t* sf = (uint8_t*)malloc((size_t)sf_n);
    float gq = 1.0f;
    for (int64_t f = 0; f < F; ++f) {
      double gs = 0.0, us = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        gs += Wg[f * H + h] * ap[h];
        us += Wu[f * H + h] * ap[h];
      }
      double cg = (cap > 0.0) ? cap * tanh(gs / cap) : gs;
      double cu = (cap > 0.0) ? cap * tanh(us / cap) : us;
      double hv = cg / (1.0 + exp(-cg)) * cu;
      if (h_round_bf16) {
        uint16_t b = orc_bf16_from_f64(hv);
        if (h_bf16_out) h_bf16_out[p * F + f] = b;
        hrow[f] = (float)orc_bf16_value(b);
      } else {
        hrow[f] = (float)hv;
      }
    }
    if (fmt == 0 && h_static_g) {
      orc_nvfp4_quantize_static(hrow, 1, F, h_static_g, codes, sf, &gq);
      orc_nvfp4_decode(codes, sf, &gq, 1, F, 0, hdec);
    } else if (fmt == 0) {
      orc_nvfp4_quantize(hrow, 1, F, 0, codes, sf, &gq);
      orc_nvfp4_decode(codes, sf, &gq, 1, F, 0, hdec);
    } else {
      orc_mxfp8_quantize(hrow, 1, F, mx_mode, codes, sf);
      orc_mxfp8_decode(codes, sf, 1, F, hdec);
    }
    if (hq_codes) memcpy(hq_codes + p * code_bytes, codes, (size_t)code_bytes);
    if (hq_sf) memcpy(hq_sf + p * sf_n, sf, (size_t)sf_n);
    if (hq_g) hq_g[p] = gq;
    for (int64_t o = 0; o < H; ++o) {
      double acc = 0.0;
      for (int64_t f = 0; f < F; ++f) acc += Wd[o * F + f] * hdec[f];
      y[p * H + o] = acc;
    }
    free(hrow);
    free(hdec);
    free(codes);
    free(sf);
  }
}

/* ======================================================================== */
/* O7. Combine (cookbook MegaMoE paragraph: the combine step).             */
/*   out[t] = sum_j w[t,j] * y[pair_pos[t,j]]   (fp64, slot order)          */
/* ======================================================================== */

void orc_combine(int64_t T, int64_t k, int64_t H, const double* w, const int32_t* pair_pos, const double* y,
                 double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int64_t j = 0; j < k; ++j) acc += w[t * k + j] * y[(int64_t)pair_pos[t * k + j] * H + h];
      out[t * H + h] = acc;
    }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
