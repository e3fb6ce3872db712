/*
 * Device-side fills of the seeded synthetic inputs (see synth_gen.h), so that
 * multi-GB expert weights never cross PCIe/C2C.  Bit-identical to the host
 * fills in synth_host.c.  Holds none of the layer's arithmetic.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth_gen.h"

__global__ void synth_k_x(uint64_t key, int64_t T, int64_t H, const uint8_t* outlier_flag,
                          float outlier_scale, uint16_t* out) {
  int64_t n = T * H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t t = i / H;
    float z = synth_normal(key, (uint64_t)i);
    bool o = outlier_flag && outlier_flag[t];
    out[i] = synth_bf16_bits(o ? outlier_scale * z : z);
  }
}

__global__ void synth_k_router(uint64_t key, int64_t n, float inv_sqrt_h, uint16_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = synth_bf16_bits(synth_normal(key, (uint64_t)i) * inv_sqrt_h);
}

__global__ void synth_k_matrix(uint64_t key, int64_t first, int64_t n, float inv_sqrt_k, float* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = synth_normal(key, (uint64_t)(first + i)) * inv_sqrt_k;
}

static int grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  if (g > 152 * 64) g = 152 * 64;
  if (g < 1) g = 1;
  return (int)g;
}

extern "C" int synth_dev_x(uint64_t seed, int64_t T, int64_t H, const uint8_t* outlier_flag_dev,
                           float outlier_scale, uint16_t* out_dev, cudaStream_t st) {
  synth_k_x<<<grid_for(T * H), 256, 0, st>>>(synth_key(seed, SYNTH_T_X), T, H, outlier_flag_dev,
                                               outlier_scale, out_dev);
  return (int)cudaGetLastError();
}

extern "C" int synth_dev_router(uint64_t seed, int64_t E, int64_t H, float inv_sqrt_h,
                                uint16_t* out_dev, cudaStream_t st) {
  synth_k_router<<<grid_for(E * H), 256, 0, st>>>(synth_key(seed, SYNTH_T_ROUTER), E * H, inv_sqrt_h,
                                                    out_dev);
  return (int)cudaGetLastError();
}

/* Experts [e0, e0+ne) of one tensor, [ne, N, K] fp32. */
extern "C" int synth_dev_expert_matrices(uint64_t seed, int tensor, int64_t e0, int64_t ne, int64_t N,
                                         int64_t K, float inv_sqrt_k, float* out_dev, cudaStream_t st) {
  int64_t n = ne * N * K;
  synth_k_matrix<<<grid_for(n), 256, 0, st>>>(synth_key(seed, (uint32_t)tensor), e0 * N * K, n,
                                               inv_sqrt_k, out_dev);
  return (int)cudaGetLastError();
}
