// MXFP8 KV-cache quantiser (SGLang blog on Inkling 2 Small, features table:
// a block-scaled MXFP8 KV cache on Blackwell).  New K or V rows of a batch,
// bf16 [tokens, heads, head_dim], are encoded along head_dim in 32-element
// blocks (E4M3 codes, one E8M0 scale per block, the OCP MX rule of the layer's
// MXFP8 activations) and written to their cache slots.
//
// Four lanes share one 32-element block: each loads 8 bf16 (16 bytes), the
// block maximum is two xor shuffles, and each lane stores its 8 codes (8
// bytes).  A warp so covers 8 consecutive blocks (512 bytes of input) per
// instruction; the kernel is bound by HBM (2 bytes in, 1 + 1/32 out per
// element).
#include "moe_common.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) k_kv_quant_mxfp8(const __nv_bfloat16* __restrict__ kv, int64_t tokens, int heads,
                                                        int head_dim, int64_t token_stride,
                                                        const int64_t* __restrict__ slot, int64_t num_slots, int mode,
                                                        uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int bpr = head_dim >> 5;                         // blocks per (token, head) row
  const int64_t nblk = tokens * heads * (int64_t)bpr;
  const int sub = threadIdx.x & 3;                       // lane within the block's group of four
  const int grp = (threadIdx.x & 31) >> 2;               // the warp's 8 groups take 8 consecutive blocks
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 2);
  // the loop runs on the warp's first block, so every lane of a warp runs the
  // same iterations and the shuffles below see the whole warp; lanes past the
  // last block only skip their memory accesses
  for (int64_t wb = (int64_t)blockIdx.x * (blockDim.x >> 2) + ((threadIdx.x >> 5) << 3); wb < nblk; wb += stride) {
    const int64_t b = wb + grp;
    const bool live = b < nblk;
    const int64_t row = live ? b / bpr : 0;
    const int blk = live ? (int)(b - row * bpr) : 0;
    const int64_t t = row / heads;
    const int hd = (int)(row - t * heads);
    int64_t dst_row = t;
    if (slot != nullptr && live) dst_row = slot[t];
    const bool store = live && dst_row >= 0 && dst_row < num_slots;

    uint4 u = make_uint4(0, 0, 0, 0);
    if (live) u = *reinterpret_cast<const uint4*>(kv + t * token_stride + (int64_t)hd * head_dim + blk * 32 + sub * 8);
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
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
    if (store) {
      const int64_t drow = dst_row * heads + hd;
      *reinterpret_cast<uint2*>(codes + drow * head_dim + blk * 32 + sub * 8) = make_uint2(lo, hi);
      if (sub == 0) scales[drow * bpr + blk] = (uint8_t)s;
    }
  }
}

}  // namespace

cudaError_t launch_kv_quant_mxfp8(const __nv_bfloat16* kv, int64_t tokens, int heads, int head_dim,
                                  int64_t token_stride, const int64_t* slot, int64_t num_slots, int mode,
                                  uint8_t* codes, uint8_t* scales, int sms, cudaStream_t st) {
  const int64_t nblk = tokens * heads * (int64_t)(head_dim / 32);
  if (nblk == 0) return cudaSuccess;
  // 64 blocks per CTA; at most 8 resident CTAs per SM in one wave, the grid
  // stride covering the rest
  const int64_t want = (nblk + 63) / 64;
  const int64_t cap = (int64_t)sms * 8;
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  k_kv_quant_mxfp8<<<grid, 256, 0, st>>>(kv, tokens, heads, head_dim, token_stride, slot, num_slots, mode, codes,
                                         scales);
  return cudaGetLastError();
}

}  // namespace moe
