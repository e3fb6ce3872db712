// Weighted combine back to token order (cookbook page on Inkling-2-Small,
// MegaMoE paragraph: the combine closes the fused MoE unit):
//   out[t] = bf16_rne( sum_j w[t,j] * y[pair_pos[t,j]] ), fp32, slot order.
// y rows are fp32, or (MOE_Y_FP16E) fp16 codes with an exponent per 32
// features, where each product is fma(w * 2^e, code, sum): the weight times a
// power of two is exact, so the sum is the same as over the decoded rows.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kCombThreads = 128;

// grid (T, slices): the columns of a token split over `slices` CTAs (many for
// small T, one for large T).  Per thread and step: 4 fp32 columns (one float4
// per pair) or 8 fp16 columns (one 16-byte load of codes and one exponent
// byte per pair).
template <bool Y16>
__global__ void __launch_bounds__(kCombThreads) k_combine(const void* __restrict__ yv, const int8_t* __restrict__ yexp,
                                                          const float* __restrict__ w,
                                                          const int32_t* __restrict__ pair_pos, int H, int k,
                                                          __nv_bfloat16* __restrict__ out) {
  constexpr int CPT = Y16 ? 8 : 4;  // columns per thread and step
  __shared__ int pos[kMaxK];
  __shared__ float ww[kMaxK];
  const int t = blockIdx.x;
  const unsigned P = gridDim.x * (unsigned)k;
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
  for (int c = blockIdx.y * kCombThreads + threadIdx.x; c < H / CPT; c += gridDim.y * kCombThreads) {
    float acc[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += 8) {  // slot order; 8 loads in flight per group (read once: evict first)
      uint4 v[8];
      int ev[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (j0 + i < k) {
          v[i] = make_uint4(0, 0, 0, 0);
          ev[i] = 0;
          const unsigned p = (unsigned)pos[j0 + i];
          if (MOE_IN_BOUNDS(p < P)) {
            if constexpr (Y16) {
              v[i] = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(yv) + (int64_t)p * H) + c);
              ev[i] = __ldg(yexp + (int64_t)p * (H >> 5) + (c >> 2));
            } else {
              v[i] = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(yv) + (int64_t)p * H) + c);
            }
          }
        }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (j0 + i < k) {
          const float s = Y16 ? __fmul_rn(ww[j0 + i], exp2i(ev[i])) : ww[j0 + i];
          const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if constexpr (Y16) {
              float lo, hi;
              f16x2_values(u[q], lo, hi);
              acc[2 * q] = __fmaf_rn(s, lo, acc[2 * q]);
              acc[2 * q + 1] = __fmaf_rn(s, hi, acc[2 * q + 1]);
            } else {
              acc[q] = __fmaf_rn(s, __uint_as_float(u[q]), acc[q]);
            }
          }
        }
    }
    uint32_t o[CPT / 2];
#pragma unroll
    for (int q = 0; q < CPT / 2; ++q) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      o[q] = *reinterpret_cast<const uint32_t*>(&b);
    }
    if constexpr (Y16) {
      reinterpret_cast<uint4*>(out + (int64_t)t * H)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      reinterpret_cast<uint2*>(out + (int64_t)t * H)[c] = make_uint2(o[0], o[1]);
    }
  }
}

}  // namespace

cudaError_t launch_combine(const moe_config& c, const void* y, const float* w, const int32_t* pair_pos,
                           __nv_bfloat16* out, cudaStream_t st, bool pdl) {
  const int cpt = y16(c) ? 8 : 4;
  const int full = (c.H / cpt + kCombThreads - 1) / kCombThreads;
  int slices = (1184 + c.T - 1) / c.T;  // about eight CTAs per SM in total
  slices = slices < 1 ? 1 : (slices > full ? full : slices);
  dim3 grid(c.T, slices);
  const int8_t* yexp = y_exponents(c, const_cast<void*>(y));
  if (y16(c)) return launch_k(k_combine<true>, grid, dim3(kCombThreads), 0, st, pdl, y, yexp, w, pair_pos, c.H, c.k, out);
  return launch_k(k_combine<false>, grid, dim3(kCombThreads), 0, st, pdl, y, yexp, w, pair_pos, c.H, c.k, out);
}

}  // namespace moe
