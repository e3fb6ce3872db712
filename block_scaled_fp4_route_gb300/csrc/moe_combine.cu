// Weighted combine back to token order (cookbook page on Inkling-2-Small,
// MegaMoE paragraph: the combine closes the fused MoE unit):
//   out[t] = bf16_rne( sum_j w[t,j] * y[pair_pos[t,j]] ), fp32, slot order.
#include "moe_common.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ y, const float* __restrict__ w,
                                                 const int32_t* __restrict__ pair_pos, int H, int k,
                                                 __nv_bfloat16* __restrict__ out) {
  __shared__ int pos[kMaxK];
  __shared__ float ww[kMaxK];
  const int t = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < k) {
    pos[threadIdx.x] = pair_pos[(int64_t)t * k + threadIdx.x];
    ww[threadIdx.x] = w[(int64_t)t * k + threadIdx.x];
  }
  __syncthreads();
  const int H4 = H / 4;
  for (int c = threadIdx.x; c < H4; c += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      float4 v = reinterpret_cast<const float4*>(y + (int64_t)pos[j] * H)[c];
      float s = ww[j];
      acc.x = __fmaf_rn(s, v.x, acc.x);
      acc.y = __fmaf_rn(s, v.y, acc.y);
      acc.z = __fmaf_rn(s, v.z, acc.z);
      acc.w = __fmaf_rn(s, v.w, acc.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    reinterpret_cast<uint2*>(out + (int64_t)t * H)[c] = o;
  }
}

}  // namespace

cudaError_t launch_combine(const moe_config& c, const float* y, const float* w, const int32_t* pair_pos,
                           __nv_bfloat16* out, cudaStream_t st, bool pdl) {
  return launch_k(k_combine, dim3(c.T), dim3(256), 0, st, pdl, y, w, pair_pos, c.H, c.k, out);
}

}  // namespace moe
