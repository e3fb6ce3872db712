// Device helpers of the block quantisers, shared by the quantiser kernels
// and the decode expert-FFN kernel (its NVFP4 h row pass): loading a block,
// encoding one NVFP4 16-block / MXFP8 32-block, and a whole row per warp.
// Every arithmetic step is a single correctly rounded fp32 operation, so the
// codes are reproducible bit for bit wherever these run.
#pragma once

#include "moe_common.cuh"

namespace moe {

// internal linkage: every translation unit that includes this gets its own copy
namespace {

__device__ __forceinline__ void load_block_bf16(const __nv_bfloat16* p, int n, float* v) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  for (int i = 0; i < n / 8; ++i) {
    uint4 u = q[i];
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
    for (int j = 0; j < 4; ++j) {
      v[i * 8 + 2 * j] = __uint_as_float(w[j] << 16);
      v[i * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}
__device__ __forceinline__ void load_block_f32(const float* p, int n, float* v) {
  const float4* q = reinterpret_cast<const float4*>(p);
  for (int i = 0; i < n / 4; ++i) {
    float4 f = q[i];
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
}

template <typename Src>
__device__ __forceinline__ void load_block(const Src* p, int n, float* v);
template <>
__device__ __forceinline__ void load_block<__nv_bfloat16>(const __nv_bfloat16* p, int n, float* v) {
  load_block_bf16(p, n, v);
}
template <>
__device__ __forceinline__ void load_block<float>(const float* p, int n, float* v) {
  load_block_f32(p, n, v);
}

// NVFP4 block of 16: returns the scale byte, writes 8 code bytes.
__device__ __forceinline__ uint32_t nvfp4_block(const float* v, float G, uint2* codes_out) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  float t = __fdiv_rn(amax, 6.0f);
  t = __fmul_rn(t, G);
  uint32_t sb = e4m3_encode(t);
  uint32_t lo = 0, hi = 0;
  if (sb != 0) {
    float inv = __fdiv_rn(G, e4m3_value(sb));
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= e2m1x2_encode(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv)) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      hi |= e2m1x2_encode(__fmul_rn(v[8 + 2 * i], inv), __fmul_rn(v[8 + 2 * i + 1], inv)) << (8 * i);
  }
  *codes_out = make_uint2(lo, hi);
  return sb;
}

// MXFP8 block of 32: returns the E8M0 byte, writes 32 code bytes.
__device__ __forceinline__ uint32_t mxfp8_block(const float* v, int mode, uint4* codes_out) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  uint32_t s = 0;
  if (amax != 0.0f) {
    s = mx_scale_code(amax, mode);
    float mul = exp2i(127 - (int)s);
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i / 2] |= e4m3x2_encode(__fmul_rn(v[2 * i], mul), __fmul_rn(v[2 * i + 1], mul)) << (16 * (i % 2));
  }
  codes_out[0] = make_uint4(w[0], w[1], w[2], w[3]);
  codes_out[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return s;
}

__device__ __forceinline__ float nvfp4_G(float amax) { return amax == 0.0f ? 1.0f : __fdiv_rn(2688.0f, amax); }

// Many short rows (prefill): one warp per row, eight rows per CTA.  Pass 1
// finds the row maximum (NVFP4, dynamic globals only), pass 2 re-reads the row
// (now in L1) block by block.  Every lane runs every iteration (lanes past the
// last block only skip their loads and stores), so the shuffles see the whole
// warp.  dst_lane: lane d < ndst holds destination row d; sg_lane (NVFP4,
// static globals) its decode factor, else 0.
template <int FMT>
__device__ __forceinline__ void quant_row_warp(const __nv_bfloat16* __restrict__ row, int K, int mx_mode, int ndst,
                                               int64_t dst_lane, float sg_lane, bool is_static, uint8_t* codes,
                                               uint8_t* scales, float* glob, int nt) {
  constexpr int BS = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  const int lane = threadIdx.x & 31;
  const int nb = K / BS;
  const int64_t cbytes = FMT == MOE_FMT_NVFP4 ? K / 2 : K;
  float G = 1.0f;
  if constexpr (FMT == MOE_FMT_NVFP4) {
    if (is_static) {
      if (lane < ndst) glob[dst_lane] = sg_lane;
    } else {
      float m = 0.0f;
      const uint4* q = reinterpret_cast<const uint4*>(row);
      for (int i = lane; i < K / 8; i += 32) {
        uint4 u = q[i];
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
      }
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      G = nvfp4_G(m);
      if (lane < ndst) glob[dst_lane] = __fdiv_rn(1.0f, G);
    }
  }
  for (int b0 = 0; b0 < nb; b0 += 32) {
    const int b = b0 + lane;
    const bool in = b < nb;
    float v[BS];
    if (in) load_block_bf16(row + (int64_t)b * BS, BS, v);
    else
#pragma unroll
      for (int i = 0; i < BS; ++i) v[i] = 0.0f;
    if constexpr (FMT == MOE_FMT_NVFP4) {
      uint2 c;
      uint32_t sc = is_static ? 0u : nvfp4_block(v, G, &c);
      for (int d = 0; d < ndst; ++d) {
        const int64_t rr = __shfl_sync(0xffffffffu, dst_lane, d);
        if (is_static) sc = nvfp4_block(v, __fdiv_rn(1.0f, __shfl_sync(0xffffffffu, sg_lane, d)), &c);
        if (in) {
          *reinterpret_cast<uint2*>(codes + rr * cbytes + (int64_t)b * 8) = c;
          scales[act_scale_offset(rr, b, nb, nt)] = (uint8_t)sc;
        }
      }
    } else {
      uint4 c[2];
      const uint32_t sc = mxfp8_block(v, mx_mode, c);
      // the scales of lanes 4j .. 4j + 3 (four consecutive blocks) are four
      // consecutive bytes of the scale layout: lane 4j stores them as one
      // word (nb is a multiple of 4, so the four are valid together)
      const uint32_t sw = sc | (__shfl_down_sync(0xffffffffu, sc, 1) << 8) |
                          (__shfl_down_sync(0xffffffffu, sc, 2) << 16) | (__shfl_down_sync(0xffffffffu, sc, 3) << 24);
      // the warp's 32 blocks are 1 KB of consecutive codes: lane L stores the
      // 16 bytes at 16 L (half L & 1 of block L >> 1) and at 512 + 16 L (of
      // block 16 + (L >> 1)), so that every store instruction writes 512
      // consecutive bytes
      const bool odd = lane & 1;
      const int s0 = lane >> 1, s1 = 16 + (lane >> 1);
      auto pick = [&](uint32_t lo, uint32_t hi, int src) {
        const uint32_t a = __shfl_sync(0xffffffffu, lo, src), bb = __shfl_sync(0xffffffffu, hi, src);
        return odd ? bb : a;
      };
      const uint4 w0 = make_uint4(pick(c[0].x, c[1].x, s0), pick(c[0].y, c[1].y, s0), pick(c[0].z, c[1].z, s0),
                                  pick(c[0].w, c[1].w, s0));
      const uint4 w1 = make_uint4(pick(c[0].x, c[1].x, s1), pick(c[0].y, c[1].y, s1), pick(c[0].z, c[1].z, s1),
                                  pick(c[0].w, c[1].w, s1));
      const bool in0 = b0 + s0 < nb, in1 = b0 + s1 < nb;
      for (int d = 0; d < ndst; ++d) {
        const int64_t rr = __shfl_sync(0xffffffffu, dst_lane, d);
        uint4* o = reinterpret_cast<uint4*>(codes + rr * cbytes + (int64_t)b0 * 32);
        if (in0) o[lane] = w0;
        if (in1) o[32 + lane] = w1;
        if (in && (lane & 3) == 0) *reinterpret_cast<uint32_t*>(scales + act_scale_offset(rr, b, nb, nt)) = sw;
      }
    }
  }
}

}  // namespace

}  // namespace moe
