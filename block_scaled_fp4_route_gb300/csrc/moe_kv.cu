// MXFP8 KV-cache quantiser (SGLang blog on Inkling 2 Small, features table:
// a block-scaled MXFP8 KV cache on Blackwell).  New K or V rows of a batch,
// bf16 [tokens, heads, head_dim], are encoded along head_dim in 32-element
// blocks (E4M3 codes, one E8M0 scale per block, the OCP MX rule of the layer's
// MXFP8 activations) and written to their cache slots.
//
// Four lanes share one 32-element block: each loads 8 bf16 (16 bytes), the
// block maximum is two xor shuffles, and each lane stores its 8 codes (8
// bytes).  A warp so covers 8 consecutive blocks (512 bytes of input) per
// instruction, and kKvUnroll such groups per loop trip, whose loads are all
// issued before the first block is encoded (64 bytes in flight per thread).
// The kernel is bound by HBM: 2 bytes in, 1 + 1/32 out per element.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kKvThreads = 256;
constexpr int kKvUnroll = 4;
constexpr int kKvBlocksPerTrip = (kKvThreads / 32) * 8 * kKvUnroll;  // 32-element blocks per CTA per trip

// I: the index type (32-bit when every block index fits, else 64-bit)
template <typename I>
__global__ void __launch_bounds__(kKvThreads, 4)
    k_kv_quant_mxfp8(const __nv_bfloat16* __restrict__ kv, I tokens, I heads, I head_dim, int64_t token_stride,
                     const int64_t* __restrict__ slot, int64_t num_slots, int mode, uint8_t* __restrict__ codes,
                     uint8_t* __restrict__ scales) {
  const I bpr = head_dim >> 5;                           // blocks per (token, head) row
  const I nblk = tokens * heads * bpr;
  const int sub = threadIdx.x & 3;                       // lane within the block's group of four
  const int grp = (threadIdx.x & 31) >> 2;               // the warp's 8 groups take 8 consecutive blocks
  const I warp_first = ((I)blockIdx.x * (kKvThreads / 32) + (I)(threadIdx.x >> 5)) * (8 * kKvUnroll);
  const I stride = (I)gridDim.x * kKvBlocksPerTrip;
  // the loop runs on the warp's first block, so every lane of a warp runs the
  // same trips and the shuffles below see the whole warp; lanes past the last
  // block only skip their memory accesses
  for (I wb = warp_first; wb < nblk; wb += stride) {
    uint4 u[kKvUnroll];
    I tok[kKvUnroll], hd[kKvUnroll], blk[kKvUnroll];
    bool live[kKvUnroll];
#pragma unroll
    for (int j = 0; j < kKvUnroll; ++j) {
      const I b = wb + (I)(8 * j + grp);
      live[j] = b < nblk;
      const I row = live[j] ? b / bpr : 0;
      blk[j] = live[j] ? b - row * bpr : 0;
      tok[j] = row / heads;
      hd[j] = row - tok[j] * heads;
      u[j] = make_uint4(0, 0, 0, 0);
      if (live[j])
        u[j] = __ldcs(reinterpret_cast<const uint4*>(kv + (int64_t)tok[j] * token_stride +
                                                     (int64_t)hd[j] * head_dim + blk[j] * 32 + sub * 8));
    }
    int64_t dst[kKvUnroll];
#pragma unroll
    for (int j = 0; j < kKvUnroll; ++j) {
      dst[j] = (int64_t)tok[j];
      if (slot != nullptr && live[j]) dst[j] = __ldg(slot + tok[j]);
    }
#pragma unroll
    for (int j = 0; j < kKvUnroll; ++j) {
      const uint32_t wv[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(wv[i] << 16);
        v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      uint32_t s = 0, lo = 0, hi = 0;
      if (amax != 0.0f) {
        s = mx_scale_code(amax, mode);
        const float mul = exp2i(127 - (int)s);
        lo = e4m3x2_encode(__fmul_rn(v[0], mul), __fmul_rn(v[1], mul)) |
             (e4m3x2_encode(__fmul_rn(v[2], mul), __fmul_rn(v[3], mul)) << 16);
        hi = e4m3x2_encode(__fmul_rn(v[4], mul), __fmul_rn(v[5], mul)) |
             (e4m3x2_encode(__fmul_rn(v[6], mul), __fmul_rn(v[7], mul)) << 16);
      }
      if (live[j] && dst[j] >= 0 && dst[j] < num_slots) {
        const int64_t drow = dst[j] * (int64_t)heads + hd[j];
        *reinterpret_cast<uint2*>(codes + drow * head_dim + blk[j] * 32 + sub * 8) = make_uint2(lo, hi);
        if (sub == 0) scales[drow * bpr + blk[j]] = (uint8_t)s;
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_quant_mxfp8(const __nv_bfloat16* kv, int64_t tokens, int heads, int head_dim,
                                  int64_t token_stride, const int64_t* slot, int64_t num_slots, int mode,
                                  uint8_t* codes, uint8_t* scales, int sms, cudaStream_t st) {
  const int64_t nblk = tokens * heads * (int64_t)(head_dim / 32);
  if (nblk == 0) return cudaSuccess;
  // one wave (4 resident CTAs per SM), the grid stride covering the rest
  const int64_t want = (nblk + kKvBlocksPerTrip - 1) / kKvBlocksPerTrip;
  const int64_t cap = (int64_t)sms * 4;
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  // 32-bit indices while the last trip's block index still fits
  if (nblk + (int64_t)grid * kKvBlocksPerTrip < ((int64_t)1 << 31)) {
    k_kv_quant_mxfp8<uint32_t><<<grid, kKvThreads, 0, st>>>(kv, (uint32_t)tokens, (uint32_t)heads,
                                                           (uint32_t)head_dim, token_stride, slot, num_slots, mode,
                                                           codes, scales);
  } else {
    k_kv_quant_mxfp8<int64_t><<<grid, kKvThreads, 0, st>>>(kv, tokens, (int64_t)heads, (int64_t)head_dim,
                                                          token_stride, slot, num_slots, mode, codes, scales);
  }
  return cudaGetLastError();
}

}  // namespace moe
