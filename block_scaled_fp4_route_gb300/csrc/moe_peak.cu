// Block-scaled tensor-core peak of this GPU, measured (TokenSpeed page on
// Inkling 2 Small, section on serving on NVIDIA Blackwell: the expert GEMMs
// run directly on block-scaled tensor cores).  The roofline of a prefill-sized
// layer divides by this rate, so it is measured here with the same MMA forms
// the expert GEMMs issue instead of being taken from a datasheet.
//
// One CTA per SM.  The operands of one k-step of the token-major GEMM tile
// (128 token rows x 128 bytes of codes, 256 weight rows x 128 bytes, their
// block scales) sit in shared memory, filled once with hashed codes (no NaN
// codes; scales 1.0); the scales are copied into TMEM once; then one thread
// issues n back-to-back `tcgen05.mma ... block_scale` of M = 128, N = 256
// (kind::mxf4nvf4 scale_vec::4X, K = 64; or kind::mxf8f6f4 scale_vec::1X,
// K = 32) into one fp32 accumulator, walking the four K offsets of the 128-byte
// rows as the GEMM does.  No global memory is touched while they run.  The
// caller times the launch with events; each CTA also records its SM-cycle
// count, so that the rate can be stated per cycle as well.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kPeakThreads = 128;
constexpr int kPeakA = 128 * 128;            // token operand bytes
constexpr int kPeakB = 256 * 128;            // weight operand bytes
constexpr int kPeakSF = 12 * 512;            // scale atoms: up to 4 (A) + 8 (B)
// shared memory asked for: above half of an SM's, so two CTAs never share an SM
constexpr int kPeakSmem = 128 * 1024;

__device__ __forceinline__ uint32_t peak_hash(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

template <int FMT>
__global__ void __launch_bounds__(kPeakThreads, 1) k_mma_peak(long long n_mma, unsigned long long* cycles,
                                                             uint32_t* status, long long limit) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kPeakA;
  uint8_t* sSF = sB + kPeakB;
  uint64_t* done = reinterpret_cast<uint64_t*>(sSF + kPeakSF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // operands: hashed codes (E4M3: 0x7F / 0xFF are NaN, replaced by 0x7E / 0xFE;
  // every E2M1 nibble is a number); scales 1.0 (UE4M3 0x38 / UE8M0 127)
  uint32_t* w32 = reinterpret_cast<uint32_t*>(smem);
  for (int i = threadIdx.x; i < (kPeakA + kPeakB) / 4; i += kPeakThreads) {
    uint32_t v = peak_hash((uint32_t)i * 2654435761u + blockIdx.x);
    if (FMT == MOE_FMT_MXFP8) {
      uint32_t nan = ~v & 0x7F7F7F7Fu;  // a zero 7-bit field marks a NaN byte
      nan = (nan - 0x01010101u) & ~nan & 0x80808080u;
      v &= ~(nan >> 7);                 // 0x7F -> 0x7E, 0xFF -> 0xFE
    }
    w32[i] = v;
  }
  const uint32_t one = FMT == MOE_FMT_NVFP4 ? 0x38383838u : 0x7F7F7F7Fu;
  for (int i = threadIdx.x; i < kPeakSF / 4; i += kPeakThreads) reinterpret_cast<uint32_t*>(sSF)[i] = one;
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_barrier_init();
  }
  fence_proxy_async();  // the generic-proxy stores above, seen by the tensor core
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sfa_t = tmem + 256;   // after the 256-column accumulator
  const uint32_t sfb_t = sfa_t + 16;
  constexpr int ATOMS = FMT == MOE_FMT_NVFP4 ? 4 : 1;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int at = 0; at < ATOMS; ++at) {
      tc_cp_32x128b_x4(sfa_t + 4 * at, sdesc_atom(smem_u32(sSF + at * 512)));
      tc_cp_32x128b_x4(sfb_t + 8 * at, sdesc_atom(smem_u32(sSF + (4 + at) * 512)));
      tc_cp_32x128b_x4(sfb_t + 8 * at + 4, sdesc_atom(smem_u32(sSF + (8 + at) * 512)));
    }
    const uint64_t dA = sdesc_sw128(smem_u32(sA));
    const uint64_t dB = sdesc_sw128(smem_u32(sB));
    const long long c0 = clock64();
    for (long long i = 0; i < n_mma; i += 4) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t accum = (i | s) != 0;
        const uint64_t koff = (uint64_t)((s * 32) >> 4);
        if constexpr (FMT == MOE_FMT_NVFP4) {
          mma_nvfp4(tmem, dA + koff, dB + koff, idesc_nvfp4(256), sfa_t + 4 * s, sfb_t + 8 * s, accum);
        } else {
          mma_mxfp8(tmem, dA + koff, dB + koff, idesc_mxfp8(256, (uint32_t)s), sfa_t, sfb_t, accum);
        }
      }
    }
    tc_commit(done);
    bool ok = mbar_try_wait(done, 0);
    const long long t0 = clock64();
    while (!ok && clock64() - t0 < limit) ok = mbar_try_wait(done, 0);
    if (!ok) atomicOr(status, ST_TIMEOUT_MMA);
    if (cycles) cycles[blockIdx.x] = (unsigned long long)(clock64() - c0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int mma_peak_flops_per_mma(moe_format fmt) { return 2 * 128 * 256 * (fmt == MOE_FMT_NVFP4 ? 64 : 32); }

cudaError_t launch_mma_peak(moe_format fmt, int ctas, long long n_mma, unsigned long long* cycles, uint32_t* status,
                            cudaStream_t st) {
  auto kern = fmt == MOE_FMT_NVFP4 ? k_mma_peak<MOE_FMT_NVFP4> : k_mma_peak<MOE_FMT_MXFP8>;
  static PerDeviceOnce attr;
  cudaError_t e = once_per_device(attr, [] {
    cudaError_t r = cudaFuncSetAttribute(k_mma_peak<MOE_FMT_NVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPeakSmem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(k_mma_peak<MOE_FMT_MXFP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
    return r;
  });
  if (e != cudaSuccess) return e;
  static_assert(kPeakA + kPeakB + kPeakSF + 64 + 1024 <= kPeakSmem, "peak kernel shared memory");
  kern<<<ctas, kPeakThreads, kPeakSmem, st>>>(n_mma, cycles, status, 4000000000LL);
  return cudaGetLastError();
}

}  // namespace moe
