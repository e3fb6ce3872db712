// Block quantisers: NVFP4 (E2M1 codes, E4M3 scale per 16, fp32 global) and
// MXFP8 (E4M3 codes, E8M0 scale per 32).  Every arithmetic step is a single
// correctly rounded fp32 operation (__fdiv_rn / __fmul_rn), so the codes are
// reproducible bit for bit.
//
// Three uses:
//   - x:   one token row per CTA, written to each of its k expert-grouped rows
//          (the GEMM1 B operand).  The activation is quantised once per token,
//          over the full hidden width, as the NVFP4 activation scales of an
//          expert must span its whole input (cookbook, Parallelism paragraph).
//   - h:   one pair row per CTA (the GEMM2 B operand), global over F.
//   - API: moe_quantize (weights with one global per expert matrix).
#include "moe_quant_dev.cuh"

namespace moe {

namespace {

constexpr int kQThreads = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float m = 0.0f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  return m;
}

template <typename Src>
__device__ float row_absmax(const Src* row, int K, float* red) {
  float m = 0.0f;
  for (int i = threadIdx.x; i < K; i += blockDim.x) {
    float v;
    if constexpr (sizeof(Src) == 2) v = __bfloat162float(row[i]);
    else v = row[i];
    m = fmaxf(m, fabsf(v));
  }
  return block_max(m, red);
}


// Quantise one row (K elements) to up to `ndst` destination rows.
enum ScaleLayout { SL_ROWMAJOR = 0, SL_TILED = 1, SL_ACT = 2 };

__device__ __forceinline__ int64_t scale_index(int layout, int64_t r, int64_t c, int64_t C) {
  return layout == SL_TILED ? tiled_scale_offset(r, c, C) : r * C + c;
}

template <int FMT, typename Src>
__device__ void quant_row(const Src* row, int K, float G, int mx_mode, int ndst, const int64_t* dst_rows,
                          uint8_t* codes, uint8_t* scales, int layout, int64_t scale_cols) {
  constexpr int BS = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  const int nb = K / BS;
  const int64_t cbytes = FMT == MOE_FMT_NVFP4 ? K / 2 : K;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    float v[BS];
    load_block<Src>(row + (int64_t)b * BS, BS, v);
    if constexpr (FMT == MOE_FMT_NVFP4) {
      uint2 c;
      uint32_t s = nvfp4_block(v, G, &c);
      for (int d = 0; d < ndst; ++d) {
        int64_t r = dst_rows[d];
        *reinterpret_cast<uint2*>(codes + r * cbytes + (int64_t)b * 8) = c;
        scales[scale_index(layout, r, b, scale_cols)] = (uint8_t)s;
      }
    } else {
      uint4 c[2];
      uint32_t s = mxfp8_block(v, mx_mode, c);
      for (int d = 0; d < ndst; ++d) {
        int64_t r = dst_rows[d];
        uint4* o = reinterpret_cast<uint4*>(codes + r * cbytes + (int64_t)b * 32);
        o[0] = c[0];
        o[1] = c[1];
        scales[scale_index(layout, r, b, scale_cols)] = (uint8_t)s;
      }
    }
  }
}

// Activation rows (x, h): each thread keeps its blocks of the row in
// registers, so the row is read once: absolute maximum (NVFP4 global), then
// the codes.  Rows of up to kRowRounds<FMT> * kQThreads blocks: 16384
// elements in both formats (the largest H and F the API accepts).
template <int FMT>
constexpr int kRowRounds = FMT == MOE_FMT_NVFP4 ? 4 : 2;

// sg (NVFP4, static activation globals): the decode factor of each
// destination (its expert's); nullptr = dynamic, from the row maximum.
template <int FMT>
constexpr int kBlockOf = FMT == MOE_FMT_NVFP4 ? 16 : 32;

// This thread's blocks of the row into registers; returns their |max|.
template <int FMT>
__device__ __forceinline__ float quant_row_load(const __nv_bfloat16* __restrict__ row, int K,
                                                float (&v)[kRowRounds<FMT>][kBlockOf<FMT>]) {
  constexpr int BS = kBlockOf<FMT>;
  const int nb = K / BS;
  float m = 0.0f;
#pragma unroll
  for (int r = 0; r < kRowRounds<FMT>; ++r) {
    const int b = threadIdx.x + r * blockDim.x;
    if (b < nb) {
      load_block_bf16(row + (int64_t)b * BS, BS, v[r]);
#pragma unroll
      for (int i = 0; i < BS; ++i) m = fmaxf(m, fabsf(v[r][i]));
    }
  }
  return m;
}

// Codes and scales of the row loaded by quant_row_load (m: this thread's
// |max|) to the ndst destination rows.
template <int FMT>
__device__ __forceinline__ void quant_row_encode(float (&v)[kRowRounds<FMT>][kBlockOf<FMT>], float m, int K,
                                                 int mx_mode, int ndst, const int64_t* dst, const float* sg,
                                                 uint8_t* codes, uint8_t* scales, float* glob, float* red, int nt) {
  const int nb = K / kBlockOf<FMT>;
  const int64_t cbytes = FMT == MOE_FMT_NVFP4 ? K / 2 : K;
  const int64_t C = nb;
  float G = 1.0f;
  if constexpr (FMT == MOE_FMT_NVFP4) {
    if (sg) {  // static: each destination encodes with its own expert's global
      if (threadIdx.x < ndst) glob[dst[threadIdx.x]] = sg[threadIdx.x];
      for (int d = 0; d < ndst; ++d) {
        const float Gd = __fdiv_rn(1.0f, sg[d]);
        const int64_t rr = dst[d];
#pragma unroll
        for (int r = 0; r < kRowRounds<FMT>; ++r) {
          const int b = threadIdx.x + r * blockDim.x;
          if (b >= nb) continue;
          uint2 c;
          const uint32_t sc = nvfp4_block(v[r], Gd, &c);
          *reinterpret_cast<uint2*>(codes + rr * cbytes + (int64_t)b * 8) = c;
          scales[act_scale_offset(rr, b, C, nt)] = (uint8_t)sc;
        }
      }
      return;
    }
    G = nvfp4_G(block_max(m, red));
    if (threadIdx.x < ndst) glob[dst[threadIdx.x]] = __fdiv_rn(1.0f, G);
  }
#pragma unroll
  for (int r = 0; r < kRowRounds<FMT>; ++r) {
    const int b = threadIdx.x + r * blockDim.x;
    if (b >= nb) continue;
    if constexpr (FMT == MOE_FMT_NVFP4) {
      uint2 c;
      uint32_t sc = nvfp4_block(v[r], G, &c);
      for (int d = 0; d < ndst; ++d) {
        const int64_t rr = dst[d];
        *reinterpret_cast<uint2*>(codes + rr * cbytes + (int64_t)b * 8) = c;
        scales[act_scale_offset(rr, b, C, nt)] = (uint8_t)sc;
      }
    } else {
      uint4 c[2];
      uint32_t sc = mxfp8_block(v[r], mx_mode, c);
      for (int d = 0; d < ndst; ++d) {
        const int64_t rr = dst[d];
        uint4* o = reinterpret_cast<uint4*>(codes + rr * cbytes + (int64_t)b * 32);
        o[0] = c[0];
        o[1] = c[1];
        scales[act_scale_offset(rr, b, C, nt)] = (uint8_t)sc;
      }
    }
  }
}

template <int FMT>
__device__ __forceinline__ void quant_row_regs(const __nv_bfloat16* __restrict__ row, int K, int mx_mode, int ndst,
                                               const int64_t* dst, const float* sg, uint8_t* codes, uint8_t* scales,
                                               float* glob, float* red, int nt) {
  float v[kRowRounds<FMT>][kBlockOf<FMT>];
  const float m = quant_row_load<FMT>(row, K, v);
  quant_row_encode<FMT>(v, m, K, mx_mode, ndst, dst, sg, codes, scales, glob, red, nt);
}

// x: one CTA per token; written to the k expert-grouped rows of the token.
// x is the layer's input, not the previous kernel's output: its row is read
// before the dependency wait.
template <int FMT>
__global__ void __launch_bounds__(kQThreads) k_quant_x(const __nv_bfloat16* __restrict__ x, int H, int k,
                                                       int mx_mode, const int32_t* __restrict__ idx,
                                                       const int32_t* __restrict__ offsets,
                                                       const int32_t* __restrict__ pair_pos,
                                                       const int32_t* __restrict__ seg_start, uint8_t* codes,
                                                       uint8_t* scales, float* glob, const float* act_static, int nt,
                                                       int E, int64_t R) {
  __shared__ float red[32];
  __shared__ int64_t dst[kMaxK];
  __shared__ float sg[kMaxK];
  const int t = blockIdx.x;
  float v[kRowRounds<FMT>][kBlockOf<FMT>];
  const float m = quant_row_load<FMT>(x + (int64_t)t * H, H, v);
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < k) {
    const int pid = t * k + threadIdx.x;
    const int e = idx[pid];
    dst[threadIdx.x] = -1;
    if (MOE_IN_BOUNDS((unsigned)e < (unsigned)E)) {
      const int64_t d = (int64_t)seg_start[e] + (pair_pos[pid] - offsets[e]);
      if (MOE_IN_BOUNDS(d >= 0 && d < R)) dst[threadIdx.x] = d;
      if (act_static) sg[threadIdx.x] = act_static[2 * e];
    }
  }
  __syncthreads();
  int ndst = k;
#ifdef MOE_DEBUG_BOUNDS
  // drop the destinations that failed their check (their rows are not written)
  __shared__ int s_ndst;
  if (threadIdx.x == 0) {
    int n = 0;
    for (int j = 0; j < k; ++j)
      if (dst[j] >= 0) {
        dst[n] = dst[j];
        sg[n] = sg[j];
        ++n;
      }
    s_ndst = n;
  }
  __syncthreads();
  ndst = s_ndst;
#endif
  quant_row_encode<FMT>(v, m, H, mx_mode, ndst, dst, act_static ? sg : nullptr, codes, scales, glob, red, nt);
}

// h: one CTA per canonical pair position p; row = its padded row.
template <int FMT>
__global__ void __launch_bounds__(kQThreads) k_quant_h(const __nv_bfloat16* __restrict__ h, int F, int mx_mode,
                                                       const int32_t* __restrict__ idx,
                                                       const int32_t* __restrict__ offsets,
                                                       const int32_t* __restrict__ perm,
                                                       const int32_t* __restrict__ seg_start, uint8_t* codes,
                                                       uint8_t* scales, float* glob, const float* act_static, int nt,
                                                       int E, int64_t R, int P) {
  __shared__ float red[32];
  __shared__ int64_t dst[1];
  __shared__ float sg[1];
  const int p = blockIdx.x;
  // The row's place comes from the routing and the dispatch, which had
  // completed before the previous kernel's threads passed their own
  // dependency wait: looked up (through L2) before this one's.
  if (threadIdx.x == 0) {
    dst[0] = -1;
    const int pid = __ldcg(perm + p);
    if (MOE_IN_BOUNDS((unsigned)pid < (unsigned)P)) {
      const int e = __ldcg(idx + pid);
      if (MOE_IN_BOUNDS((unsigned)e < (unsigned)E)) {
        const int64_t d = (int64_t)__ldcg(seg_start + e) + (p - __ldcg(offsets + e));
        if (MOE_IN_BOUNDS(d >= 0 && d < R)) dst[0] = d;
        if (act_static) sg[0] = act_static[2 * e + 1];
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();
#ifdef MOE_DEBUG_BOUNDS
  if (dst[0] < 0) return;  // the whole CTA: its row failed a check
#endif
  quant_row_regs<FMT>(h + dst[0] * F, F, mx_mode, 1, dst, act_static ? sg : nullptr, codes, scales, glob, red, nt);
}

// rows: x tokens (is_h = 0, k destinations each) or h pair positions (is_h = 1).
template <int FMT>
__global__ void __launch_bounds__(256) k_quant_rows_warp(const __nv_bfloat16* __restrict__ src, int rows, int K, int k,
                                                         int is_h, int mx_mode, const int32_t* __restrict__ idx,
                                                         const int32_t* __restrict__ offsets,
                                                         const int32_t* __restrict__ pair_pos,
                                                         const int32_t* __restrict__ perm,
                                                         const int32_t* __restrict__ seg_start, uint8_t* codes,
                                                         uint8_t* scales, float* glob, const float* act_static,
                                                         int nt, int E, int64_t R, int P) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (r >= rows) return;  // whole warp
  int64_t dst = -1;
  float sg = 0.0f;
  const __nv_bfloat16* row;
  int ndst;
  if (is_h) {
    const int pid = perm[r];
    if (MOE_IN_BOUNDS((unsigned)pid < (unsigned)P)) {
      const int e = idx[pid];
      if (MOE_IN_BOUNDS((unsigned)e < (unsigned)E)) {
        const int64_t d = (int64_t)seg_start[e] + (r - offsets[e]);
        if (MOE_IN_BOUNDS(d >= 0 && d < R)) dst = d;
        if (act_static) sg = act_static[2 * e + 1];
      }
    }
#ifdef MOE_DEBUG_BOUNDS
    if (dst < 0) return;  // whole warp (every lane holds the same row)
#endif
    row = src + dst * K;
    ndst = 1;
  } else {
    if (lane < k) {
      const int pid = r * k + lane;
      const int e = idx[pid];
      if (MOE_IN_BOUNDS((unsigned)e < (unsigned)E)) {
        const int64_t d = (int64_t)seg_start[e] + (pair_pos[pid] - offsets[e]);
        if (MOE_IN_BOUNDS(d >= 0 && d < R)) dst = d;
        if (act_static) sg = act_static[2 * e];
      }
    }
    row = src + (int64_t)r * K;
    ndst = k;
#ifdef MOE_DEBUG_BOUNDS
    // drop the destinations that failed their check: lane d takes the d-th
    // valid one
    const unsigned ok = __ballot_sync(0xffffffffu, lane < k && dst >= 0);
    int64_t d2 = -1;
    float s2 = 0.0f;
    for (int j = 0; j < 32; ++j) {
      const int64_t dj = __shfl_sync(0xffffffffu, dst, j);
      const float sj = __shfl_sync(0xffffffffu, sg, j);
      if (((ok >> j) & 1u) && lane == __popc(ok & ((1u << j) - 1u))) {
        d2 = dj;
        s2 = sj;
      }
    }
    dst = d2;
    sg = s2;
    ndst = __popc(ok);
#endif
  }
  quant_row_warp<FMT>(row, K, mx_mode, ndst, dst, sg, act_static != nullptr, codes, scales, glob, nt);
}

constexpr int kWarpRowsFrom = 2048;  // x rows from which one warp per row is used
// h rows from which one warp per row is used: a CTA for each of a few hundred
// rows fills the SMs and holds back the down GEMM's CTAs (decode64: the layer
// 2.8 us faster with warps)
constexpr int kWarpRowsFromH = 256;

// --- general API quantiser -------------------------------------------------
__global__ void k_zero_f32(float* p, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0.0f;
}

// Per-group absolute maximum, accumulated as float bits (non-negative floats
// order like their unsigned bit patterns).
template <typename Src>
__global__ void k_group_amax(const Src* __restrict__ src, int64_t cols, int64_t group_rows, int64_t chunk,
                             float* amax) {
  __shared__ float red[32];
  const int64_t g = blockIdx.y;
  const int64_t n = group_rows * cols;
  const Src* base = src + g * n;
  int64_t lo = (int64_t)blockIdx.x * chunk, hi = lo + chunk < n ? lo + chunk : n;
  float m = 0.0f;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    float v;
    if constexpr (sizeof(Src) == 2) v = __bfloat162float(base[i]);
    else v = base[i];
    m = fmaxf(m, fabsf(v));
  }
  m = block_max(m, red);
  if (threadIdx.x == 0 && m > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(amax + g), __float_as_uint(m));
}

template <int FMT, typename Src>
__global__ void __launch_bounds__(kQThreads) k_quantize_rows(const Src* __restrict__ src, int64_t cols,
                                                             int64_t group_rows, int mx_mode, bool tiled,
                                                             uint8_t* codes, uint8_t* scales,
                                                             const float* group_amax, float* glob_rows) {
  __shared__ float red[32];
  __shared__ int64_t dst[1];
  const int64_t r = blockIdx.x;
  const Src* row = src + r * cols;
  if (threadIdx.x == 0) dst[0] = r;
  float G = 1.0f;
  if constexpr (FMT == MOE_FMT_NVFP4) {
    if (group_rows > 0) G = nvfp4_G(group_amax[r / group_rows]);
    else G = nvfp4_G(row_absmax(row, (int)cols, red));
  }
  __syncthreads();
  if constexpr (FMT == MOE_FMT_NVFP4) {
    if (group_rows == 0 && threadIdx.x == 0) glob_rows[r] = __fdiv_rn(1.0f, G);
  }
  quant_row<FMT, Src>(row, (int)cols, G, mx_mode, 1, dst, codes, scales, tiled ? SL_TILED : SL_ROWMAJOR,
                      cols / (FMT == MOE_FMT_NVFP4 ? 16 : 32));
}

// Fake quantisation: out = decode(encode(v)) in fp32, rounded once (the
// products e2m1*scale and e4m3*2^k are exact; NVFP4 multiplies by g last).
template <int FMT, typename Src>
__global__ void __launch_bounds__(kQThreads) k_fake_quant_rows(const Src* __restrict__ src, int64_t cols,
                                                               int64_t group_rows, int mx_mode,
                                                               const float* group_amax, float* glob_rows,
                                                               float* __restrict__ out) {
  __shared__ float red[32];
  constexpr int BS = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  const int64_t r = blockIdx.x;
  const Src* row = src + r * cols;
  float G = 1.0f;
  if constexpr (FMT == MOE_FMT_NVFP4) {
    if (group_rows > 0) G = nvfp4_G(group_amax[r / group_rows]);
    else G = nvfp4_G(row_absmax(row, (int)cols, red));
  }
  const float g = __fdiv_rn(1.0f, G);
  if constexpr (FMT == MOE_FMT_NVFP4) {
    if (group_rows == 0 && threadIdx.x == 0 && glob_rows) glob_rows[r] = g;
  }
  for (int64_t b = threadIdx.x; b < cols / BS; b += blockDim.x) {
    float v[BS];
    load_block<Src>(row + b * BS, BS, v);
    float* o = out + r * cols + b * BS;
    if constexpr (FMT == MOE_FMT_NVFP4) {
      uint2 c;
      const uint32_t sb = nvfp4_block(v, G, &c);
      const float sv = e4m3_value(sb);
      for (int i = 0; i < 16; ++i) {
        const uint32_t q = ((i < 8 ? c.x : c.y) >> (4 * (i & 7))) & 15u;
        o[i] = __fmul_rn(__fmul_rn(e2m1_value(q), sv), g);
      }
    } else {
      uint4 c[2];
      const uint32_t s = mxfp8_block(v, mx_mode, c);
      const float X = exp2i((int)s - 127);
      const uint32_t w[8] = {c[0].x, c[0].y, c[0].z, c[0].w, c[1].x, c[1].y, c[1].z, c[1].w};
      for (int i = 0; i < 32; ++i) o[i] = __fmul_rn(e4m3_value((w[i / 4] >> (8 * (i % 4))) & 0xFFu), X);
    }
  }
}

__global__ void k_finalize_groups(float* glob, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    glob[i] = __fdiv_rn(1.0f, nvfp4_G(glob[i]));
}

__global__ void k_pack_scales(const uint8_t* __restrict__ src, int64_t rows, int64_t cols, uint8_t* dst) {
  int64_t n = rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / cols, c = i % cols;
    dst[tiled_scale_offset(r, c, cols)] = src[i];
  }
}

int grid_1d(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  if (g > 152 * 32) g = 152 * 32;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

cudaError_t launch_quant_x(const moe_config& c, const __nv_bfloat16* x, const int32_t* idx, const int32_t* offsets,
                           const int32_t* pair_pos, const int32_t* seg_start, uint8_t* codes, uint8_t* scales,
                           float* glob, const float* act_static, cudaStream_t st, bool pdl) {
  if (c.T >= kWarpRowsFrom) {
    auto kw = c.fmt == MOE_FMT_NVFP4 ? k_quant_rows_warp<MOE_FMT_NVFP4> : k_quant_rows_warp<MOE_FMT_MXFP8>;
    return launch_k(kw, dim3((c.T + 7) / 8), dim3(256), 0, st, pdl, x, c.T, c.H, c.k, 0, c.mx_scale_mode, idx, offsets,
                    pair_pos, (const int32_t*)nullptr, seg_start, codes, scales, glob, act_static, tile_rows(c), c.E,
                    padded_rows(c), c.T * c.k);
  }
  auto kern = c.fmt == MOE_FMT_NVFP4 ? k_quant_x<MOE_FMT_NVFP4> : k_quant_x<MOE_FMT_MXFP8>;
  return launch_k(kern, dim3(c.T), dim3(kQThreads), 0, st, pdl, x, c.H, c.k, c.mx_scale_mode, idx, offsets, pair_pos,
                  seg_start, codes, scales, glob, act_static, tile_rows(c), c.E, padded_rows(c));
}

cudaError_t launch_quant_h(const moe_config& c, const __nv_bfloat16* h, const int32_t* idx, const int32_t* offsets,
                           const int32_t* perm, const int32_t* seg_start, uint8_t* codes, uint8_t* scales,
                           float* glob, const float* act_static, cudaStream_t st, bool pdl) {
  int P = c.T * c.k;
  if (P >= kWarpRowsFromH) {
    auto kw = c.fmt == MOE_FMT_NVFP4 ? k_quant_rows_warp<MOE_FMT_NVFP4> : k_quant_rows_warp<MOE_FMT_MXFP8>;
    return launch_k(kw, dim3((P + 7) / 8), dim3(256), 0, st, pdl, h, P, c.F, c.k, 1, c.mx_scale_mode, idx, offsets,
                    (const int32_t*)nullptr, perm, seg_start, codes, scales, glob, act_static, tile_rows(c), c.E,
                    padded_rows(c), P);
  }
  auto kern = c.fmt == MOE_FMT_NVFP4 ? k_quant_h<MOE_FMT_NVFP4> : k_quant_h<MOE_FMT_MXFP8>;
  return launch_k(kern, dim3(P), dim3(kQThreads), 0, st, pdl, h, c.F, c.mx_scale_mode, idx, offsets, perm, seg_start,
                  codes, scales, glob, act_static, tile_rows(c), c.E, padded_rows(c), P);
}

cudaError_t launch_quantize(moe_format fmt, int mx_mode, int src_fp32, const void* src, int64_t rows, int64_t cols,
                            int64_t group_rows, moe_scale_layout layout, uint8_t* codes, uint8_t* scales,
                            float* glob, float* /*unused*/, cudaStream_t st) {
  bool tiled = layout == MOE_SCALES_TILED;
  bool nv = fmt == MOE_FMT_NVFP4;
  if (nv && group_rows > 0) {
    int64_t ng = rows / group_rows;
    int64_t n = group_rows * cols;
    int64_t chunk = 1 << 16;
    int64_t nchunks = (n + chunk - 1) / chunk;
    k_zero_f32<<<grid_1d(ng, 256), 256, 0, st>>>(glob, ng);
    dim3 grid((unsigned)nchunks, (unsigned)ng);
    if (src_fp32) k_group_amax<float><<<grid, 256, 0, st>>>((const float*)src, cols, group_rows, chunk, glob);
    else k_group_amax<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)src, cols, group_rows, chunk, glob);
  }
  dim3 grid((unsigned)rows);
  if (nv) {
    if (src_fp32)
      k_quantize_rows<MOE_FMT_NVFP4, float><<<grid, kQThreads, 0, st>>>((const float*)src, cols, group_rows, mx_mode,
                                                                       tiled, codes, scales, glob, glob);
    else
      k_quantize_rows<MOE_FMT_NVFP4, __nv_bfloat16><<<grid, kQThreads, 0, st>>>(
          (const __nv_bfloat16*)src, cols, group_rows, mx_mode, tiled, codes, scales, glob, glob);
    if (group_rows > 0) k_finalize_groups<<<grid_1d(rows / group_rows, 256), 256, 0, st>>>(glob, rows / group_rows);
  } else {
    if (src_fp32)
      k_quantize_rows<MOE_FMT_MXFP8, float><<<grid, kQThreads, 0, st>>>((const float*)src, cols, 0, mx_mode, tiled,
                                                                       codes, scales, nullptr, nullptr);
    else
      k_quantize_rows<MOE_FMT_MXFP8, __nv_bfloat16><<<grid, kQThreads, 0, st>>>(
          (const __nv_bfloat16*)src, cols, 0, mx_mode, tiled, codes, scales, nullptr, nullptr);
  }
  return cudaGetLastError();
}

cudaError_t launch_fake_quant(moe_format fmt, int mx_mode, int src_fp32, const void* src, int64_t rows, int64_t cols,
                              int64_t group_rows, float* out, float* glob, cudaStream_t st) {
  float* group_scratch = glob;
  const bool nv = fmt == MOE_FMT_NVFP4;
  if (nv && group_rows > 0) {
    int64_t ng = rows / group_rows, n = group_rows * cols, chunk = 1 << 16;
    k_zero_f32<<<grid_1d(ng, 256), 256, 0, st>>>(group_scratch, ng);
    dim3 grid((unsigned)((n + chunk - 1) / chunk), (unsigned)ng);
    if (src_fp32) k_group_amax<float><<<grid, 256, 0, st>>>((const float*)src, cols, group_rows, chunk, group_scratch);
    else k_group_amax<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)src, cols, group_rows, chunk, group_scratch);
  }
  dim3 grid((unsigned)rows);
  if (nv) {
    if (src_fp32)
      k_fake_quant_rows<MOE_FMT_NVFP4, float><<<grid, kQThreads, 0, st>>>((const float*)src, cols, group_rows, mx_mode,
                                                                         group_scratch, glob, out);
    else
      k_fake_quant_rows<MOE_FMT_NVFP4, __nv_bfloat16><<<grid, kQThreads, 0, st>>>(
          (const __nv_bfloat16*)src, cols, group_rows, mx_mode, group_scratch, glob, out);
    if (group_rows > 0) k_finalize_groups<<<grid_1d(rows / group_rows, 256), 256, 0, st>>>(glob, rows / group_rows);
  } else {
    if (src_fp32)
      k_fake_quant_rows<MOE_FMT_MXFP8, float><<<grid, kQThreads, 0, st>>>((const float*)src, cols, 0, mx_mode, nullptr,
                                                                         nullptr, out);
    else
      k_fake_quant_rows<MOE_FMT_MXFP8, __nv_bfloat16><<<grid, kQThreads, 0, st>>>(
          (const __nv_bfloat16*)src, cols, 0, mx_mode, nullptr, nullptr, out);
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_scales(const uint8_t* src, int64_t rows, int64_t cols, uint8_t* dst, cudaStream_t st) {
  k_pack_scales<<<grid_1d(rows * cols, 256), 256, 0, st>>>(src, rows, cols, dst);
  return cudaGetLastError();
}

}  // namespace moe
