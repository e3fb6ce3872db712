// Weighted combine back to token order (cookbook page on Inkling-2-Small,
// MegaMoE paragraph: the combine closes the fused MoE unit):
//   out[t] = bf16_rne( sum_j w[t,j] * y[pair_pos[t,j]] ), fp32, slot order.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kCombThreads = 128;

// grid (T, slices): the columns of a token split over `slices` CTAs (many for
// small T, one for large T); one float4 per thread per step.
__global__ void __launch_bounds__(kCombThreads) k_combine(const float* __restrict__ y, const float* __restrict__ w,
                                                          const int32_t* __restrict__ pair_pos, int H, int k,
                                                          __nv_bfloat16* __restrict__ out) {
  __shared__ int pos[kMaxK];
  __shared__ float ww[kMaxK];
  const int t = blockIdx.x;
  // the routing weights and pair positions come from kernels that had
  // completed before the previous kernel's threads passed their own
  // dependency wait: read (through L2) before this one's
  if (threadIdx.x < k) {
    pos[threadIdx.x] = __ldcg(pair_pos + (int64_t)t * k + threadIdx.x);
    ww[threadIdx.x] = __ldcg(w + (int64_t)t * k + threadIdx.x);
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  for (int c = blockIdx.y * kCombThreads + threadIdx.x; c < H / 4; c += gridDim.y * kCombThreads) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < k; j0 += 8) {  // slot order; 8 loads in flight per group (read once: evict first)
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (j0 + i < k) {
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (MOE_IN_BOUNDS((unsigned)pos[j0 + i] < (unsigned)(gridDim.x * k)))
          v[i] = __ldcs(reinterpret_cast<const float4*>(y + (int64_t)pos[j0 + i] * H) + c);
      }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (j0 + i < k) {
        const float s = ww[j0 + i];
        acc.x = __fmaf_rn(s, v[i].x, acc.x);
        acc.y = __fmaf_rn(s, v[i].y, acc.y);
        acc.z = __fmaf_rn(s, v[i].z, acc.z);
        acc.w = __fmaf_rn(s, v[i].w, acc.w);
      }
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
  const int full = (c.H / 4 + kCombThreads - 1) / kCombThreads;
  int slices = (1184 + c.T - 1) / c.T;  // about eight CTAs per SM in total
  slices = slices < 1 ? 1 : (slices > full ? full : slices);
  dim3 grid(c.T, slices);
  return launch_k(k_combine, grid, dim3(kCombThreads), 0, st, pdl, y, w, pair_pos, c.H, c.k, out);
}

}  // namespace moe
