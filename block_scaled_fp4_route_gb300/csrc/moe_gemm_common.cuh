// Pieces shared by the decode expert GEMM (moe_gemm.cu) and the fused decode
// expert FFN (moe_ffn_decode.cu): the 64-row-tile configuration, the kernel
// arguments, the soft cap and SiLU of the gated epilogue, and the mapping of a
// tile index to (expert, weight block, row tile).
#pragma once

#include "moe_common.cuh"

namespace moe {

// internal linkage: every translation unit that includes this gets its own copy
namespace {

template <int FMT, bool GATED>
struct Cfg {
  static constexpr int NA = 2;                              // weight blocks per tile
  static constexpr int ROWS = GATED ? 128 : 256;            // output features per tile
  static constexpr int NT = kNTDecode;                      // token rows per tile
  static constexpr int ACC_BUFS = 2;                        // TMEM accumulator buffers
  static constexpr int EPI_WARPS = 4;                       // one warp per TMEM lane quadrant
  static constexpr int THREADS = (4 + EPI_WARPS) * 32;
  static constexpr int STAGES = FMT == MOE_FMT_NVFP4 ? 4 : 5;
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = NT * 128;
  static constexpr int SF_ATOMS = FMT == MOE_FMT_NVFP4 ? 4 : 1;  // 512-byte atoms per operand per stage
  static constexpr int SF_BYTES = SF_ATOMS * 512;
  static constexpr int RAW_STAGE = NA * A_BYTES + B_BYTES + (NA + 1) * SF_BYTES;
  static constexpr int STAGE_BYTES = (RAW_STAGE + 1023) / 1024 * 1024;
  static constexpr int BAR_BYTES = 256;
  static constexpr int RTB_BYTES = (kMaxE + 1) * 4;
  static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + RTB_BYTES + 1024;
  static constexpr int ELEMS_PER_STAGE = FMT == MOE_FMT_NVFP4 ? 256 : 128;  // 128 bytes of codes
  static constexpr int BLOCK = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  static constexpr int ACC_COLS = NT;            // one accumulator: 128 lanes x N columns
  static constexpr int ACC_BUF = NA * ACC_COLS;  // both weight blocks of one tile
  static constexpr int SF_COLS_OP = SF_ATOMS * 4;
  static constexpr int SF_COLS_STAGE = (NA + 1) * SF_COLS_OP;
  static constexpr int TMEM_SF = ACC_BUFS * ACC_BUF;
  static constexpr int TMEM_COLS = 512;
  static_assert(TMEM_SF + STAGES * SF_COLS_STAGE <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(16 * STAGES + 64 <= BAR_BYTES, "barrier area");
};

struct GemmArgs {
  const uint8_t* sfA0;
  const uint8_t* sfA1;
  const uint8_t* sfB;
  const float* gA0;
  const float* gA1;
  const float* gB;
  const RowTile* tiles;
  const int32_t* rt_base;
  int E;
  int NA;  // weight rows per expert (= output features; also the output row stride)
  int K;   // reduction length in elements
  float cap;
  float inv_cap;  // fp32(1 / cap), 0 when cap == 0
  __nv_bfloat16* h_out;  // NVFP4: bf16 h (quantised by a row pass: its global spans the row)
  uint8_t* hq_codes;     // MXFP8: h codes and scales written by the epilogue
  uint8_t* hq_scales;
  int mx_mode;
  void* y_out;     // y rows: fp32, or fp16 codes (y16)
  int8_t* y_exp;   // y16: exponents [P, NA/32]
  int y16;
  uint32_t* status;
  long long limit;
  int withhold_loads;
  int64_t R;      // padded activation rows (h / x rows are below R)
  int64_t P;      // pairs (canonical y rows are below P)
  int max_tiles;  // capacity of the row-tile list
};

// One MOE_Y_FP16E block held by one thread: the 32 values lo[0..15],
// hi[0..15] (fp32 bits) times sc, the same fp32 products the fp32 format
// stores; their codes go to pk (32 fp16, two per word, in feature order) and
// the block's exponent is returned.
__device__ __forceinline__ int y16_block_codes(const uint32_t (&lo)[16], const uint32_t (&hi)[16], float sc,
                                               uint32_t (&pk)[16]) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[j] = __fmul_rn(__uint_as_float(lo[j]), sc);
    v[16 + j] = __fmul_rn(__uint_as_float(hi[j]), sc);
  }
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(v[j]));
  const int e = y16_exponent(m);
  const float mul = exp2i(-e);
#pragma unroll
  for (int j = 0; j < 16; ++j) pk[j] = f16x2_encode(__fmul_rn(v[2 * j], mul), __fmul_rn(v[2 * j + 1], mul));
  return e;
}

// One MOE_Y_FP16E value per lane of a warp whose 32 lanes hold one 32-feature
// block of a row (weight-major epilogues): the block's exponent (reduced
// across the warp; every lane must call) and this lane's code.
__device__ __forceinline__ uint16_t y16_lane_code(float v, int& e) {
  const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
  e = y16_exponent(m);
  return f16_encode(__fmul_rn(v, exp2i(-e)));
}

// The tile plan's row-tile prefix rtb[0..E] must be non-decreasing and end at
// most at max_tiles.  Checked build: every thread of the CTA checks a share
// after the plan is in shared memory (this replaces the __syncthreads that
// follows the load), and a plan that fails runs no tile in any role.  Normal
// build: the barrier only.
__device__ __forceinline__ bool plan_ok_sync(const int32_t* s_rtb, int E, int max_tiles) {
#ifdef MOE_DEBUG_BOUNDS
  __syncthreads();  // every thread's share of the plan is in shared memory
  int bad = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) bad |= s_rtb[i + 1] < s_rtb[i];
  if (threadIdx.x == 0) bad |= s_rtb[0] != 0 || s_rtb[E] > max_tiles;
  return MOE_IN_BOUNDS(!__syncthreads_or(bad));
#else
  (void)s_rtb;
  (void)E;
  (void)max_tiles;
  __syncthreads();
  return true;
#endif
}

// tanh for the soft cap c * tanh(v / c), in fp32 to a few ulp: below 0.5,
// x + x^3 P(x^2) with P of degree 3, fitted to (tanh x - x) / x^3 on
// [0, 1/2] by least squares on 400 Chebyshev nodes, reweighted toward the
// smallest maximum relative error of tanh (1.5e-8 in exact arithmetic,
// under 0.75 ulp evaluated in fp32; the odd Taylor series needs terms up to
// x^15 for the same accuracy, three more fused multiply-adds per call);
// above, 1 - 2 / (e^{2|x|} + 1), which has no cancellation there, with the
// hardware base-2 exponential and reciprocal.
__device__ __forceinline__ float tanh_soft(float x) {
  const float ax = fabsf(x);
  if (ax < 0.5f) {
    const float x2 = x * x;
    float p = 0.0172414667904377f;
    p = fmaf(p, x2, -0.05304548144340515f);
    p = fmaf(p, x2, 0.13325878977775574f);
    p = fmaf(p, x2, -0.333331435918808f);
    return fmaf(x * x2, p, x);
  }
  const float e = ex2_approx(2.8853900817779268f * ax);  // e^{2|x|}; +inf for large |x|
  return copysignf(1.0f - 2.0f * rcp_approx(e + 1.0f), x);
}

// The soft cap c * tanh(v / c) (inv_c = fp32(1 / c)): with x = v inv_c below
// 0.5 it is c x + (c x) x^2 P(x^2), and c x differs from v by at most
// |v| 2^-24 (inv_c is rounded once), so it is evaluated as fma(v x^2, P, v):
// one multiply fewer than scaling tanh_soft's result.
__device__ __forceinline__ float cap_soft(float v, float c, float inv_c) {
  const float x = v * inv_c;
  if (fabsf(x) < 0.5f) {
    const float x2 = x * x;
    float p = 0.0172414667904377f;
    p = fmaf(p, x2, -0.05304548144340515f);
    p = fmaf(p, x2, 0.13325878977775574f);
    p = fmaf(p, x2, -0.333331435918808f);
    return fmaf(v * x2, p, v);
  }
  return c * tanh_soft(x);
}

// silu(g) = g / (1 + e^{-g}), with the hardware base-2 exponential and
// reciprocal (a few ulp; -0 for large negative g, g for large positive g).
__device__ __forceinline__ float silu(float g) {
  return g * rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * g));
}

// Tile t -> (expert e, weight-row block mt, row tile index rt) in the order
// expert, mt, token block.  rtb[e] is the first row tile of expert e.
__device__ __forceinline__ void map_tile(int t, int MT, const int32_t* rtb, int E, int& mt, int& rt) {
  int lo = 0, hi = E;  // rtb[lo]*MT <= t < rtb[hi]*MT
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (rtb[mid] * MT <= t) lo = mid;
    else hi = mid;
  }
  const int nrt = rtb[lo + 1] - rtb[lo];
  const int l = t - rtb[lo] * MT;
  mt = l / nrt;
  rt = rtb[lo] + l % nrt;
}

// A tile descriptor through L2 (it may be read before this grid's dependency
// wait, when this SM's L1 could still hold an older copy).
__device__ __forceinline__ RowTile load_tile(const RowTile* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  return RowTile{v.x, v.y, v.z, v.w};
}

inline GemmArgs gemm_args(const GemmLaunch& g) {
  GemmArgs a;
  a.sfA0 = g.sfA0;
  a.sfA1 = g.sfA1;
  a.sfB = g.sfB;
  a.gA0 = g.gA0;
  a.gA1 = g.gA1;
  a.gB = g.gB;
  a.tiles = g.tiles;
  a.rt_base = g.rt_base;
  a.E = g.E;
  a.NA = g.NA;
  a.K = g.K;
  a.cap = g.cfg->swiglu_cap;
  a.inv_cap = a.cap > 0.0f ? 1.0f / a.cap : 0.0f;
  a.h_out = g.h_out;
  a.hq_codes = g.hq_codes;
  a.hq_scales = g.hq_scales;
  a.mx_mode = g.cfg->mx_scale_mode;
  a.y_out = g.y_out;
  a.y_exp = g.y_exp;
  a.y16 = y16(*g.cfg) ? 1 : 0;
  a.status = g.status;
  a.limit = g.wait_limit > 0 ? g.wait_limit : 4000000000LL;  // default ~2 s of SM clock
  a.withhold_loads = g.withhold_loads;
  a.R = padded_rows(*g.cfg);
  a.P = (int64_t)g.cfg->T * g.cfg->k;
  a.max_tiles = (int)max_row_tiles(*g.cfg);
  return a;
}

}  // namespace

}  // namespace moe
