// Shared device helpers of the MoE library: PTX wrappers for mbarrier, TMA
// (cp.async.bulk[.tensor]) and the 5th-generation tensor core (tcgen05), the
// block-scale TILED layout, and bit-exact E2M1 / E4M3 / E8M0 encoders.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "moe_internal.h"

namespace moe {

// ----------------------------------------------------------------------------
// host: per-device one-time set-up (kernel attributes are per device)
// ----------------------------------------------------------------------------
struct PerDeviceOnce {
  static constexpr int kMaxDevices = 64;
  std::atomic<bool> done[kMaxDevices] = {};
  std::mutex mu;
};

// Runs `fn` (returning cudaError_t) once for the current device; later calls
// on that device return cudaSuccess without running it.  A failed `fn` is
// retried on the next call.  Thread-safe.
template <typename Fn>
inline cudaError_t once_per_device(PerDeviceOnce& o, Fn fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= PerDeviceOnce::kMaxDevices) return cudaErrorInvalidDevice;
  if (o.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lk(o.mu);
  if (o.done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess) o.done[dev].store(true, std::memory_order_release);
  return e;
}

// ----------------------------------------------------------------------------
// status word bits written by kernels whose bounded waits ran out
// ----------------------------------------------------------------------------
enum : uint32_t {
  ST_TIMEOUT_PRODUCER = 1u << 0,
  ST_TIMEOUT_MMA = 1u << 1,
  ST_TIMEOUT_EPILOGUE = 1u << 2,
  ST_TIMEOUT_DRAIN = 1u << 3,
  ST_TIMEOUT_DEPEND = 1u << 4,  // a down tile of the fused decode FFN waited too long for its h rows
};

// ----------------------------------------------------------------------------
// Bounds-checked build (-DMOE_DEBUG_BOUNDS): the indices the kernels derive
// from data (pair positions, padded activation rows, canonical pair rows,
// row-tile indices) are checked before the accesses they address.  A failed
// check skips the access and sets this translation unit's device flag, which
// moe_debug_bounds_status reads and clears; nothing traps.  Without the macro
// MOE_IN_BOUNDS(cond) is `true` and the condition is not evaluated.
// ----------------------------------------------------------------------------
#ifdef MOE_DEBUG_BOUNDS
namespace {
__device__ uint32_t g_bounds_flag;  // one per translation unit
}  // namespace
// the flag holds the largest source line of a failed check (0: none)
__device__ __forceinline__ bool bounds_check(bool ok, uint32_t line) {
  if (!ok) atomicMax(&g_bounds_flag, line);
  return ok;
}
#define MOE_IN_BOUNDS(cond) (::moe::bounds_check((cond), __LINE__))
// host: every translation unit registers a reader of its flag
using BoundsReader = cudaError_t (*)(uint32_t* value);
void register_bounds_reader(BoundsReader r);
namespace {
inline cudaError_t read_and_clear_bounds_flag(uint32_t* v) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_bounds_flag, sizeof(uint32_t));
  if (e == cudaSuccess && *v != 0u) {
    const uint32_t zero = 0u;
    e = cudaMemcpyToSymbol(g_bounds_flag, &zero, sizeof(uint32_t));
  }
  return e;
}
struct BoundsRegistrar {
  BoundsRegistrar() { register_bounds_reader(read_and_clear_bounds_flag); }
};
const BoundsRegistrar g_bounds_registrar;
}  // namespace
#else
#define MOE_IN_BOUNDS(cond) (true)
#endif

// ----------------------------------------------------------------------------
// TILED block-scale layout (see moe.h): 512-byte atoms of 128 rows x 4 scale
// columns; inside an atom row r sits at lane r%32, 4-byte word (r/32)%4.
// ----------------------------------------------------------------------------
__host__ __device__ __forceinline__ int64_t tiled_scale_offset(int64_t r, int64_t c, int64_t C) {
  return ((r >> 7) * (C >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}
// Activation (MMA B operand) scales: one 512-byte atom per row tile of nt
// (64 or 128) rows and 4 scale columns; row rr of the tile at lane rr%32,
// word rr/32.
__host__ __device__ __forceinline__ int64_t act_scale_offset(int64_t r, int64_t c, int64_t C, int nt) {
  const int64_t rr = r % nt;
  return ((r / nt) * (C >> 2) + (c >> 2)) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (c & 3);
}

// ----------------------------------------------------------------------------
// number formats (round to nearest even, saturate to the largest finite,
// the sign bit follows the input also for zero)
// ----------------------------------------------------------------------------
__device__ __forceinline__ float exp2i(int n) {  // 2^n, n in [-127, 127], exact
  return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23) : __uint_as_float(0x00400000u);
}

// E2M1 and E4M3 encoders: the hardware conversions (cvt.rn.satfinite):
// round to nearest even, saturation to the largest finite (6 / 448), the sign
// bit kept also for zero.  The pair forms put the first value in the low
// nibble / byte.
__device__ __forceinline__ uint32_t e2m1x2_encode(float lo, float hi) {
  uint32_t r;
  asm("{\n.reg .b8 t;\ncvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\ncvt.u32.u8 %0, t;\n}" : "=r"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}
__device__ __forceinline__ uint32_t e2m1_encode(float v) { return e2m1x2_encode(v, 0.0f) & 0xFu; }

__device__ __forceinline__ uint32_t e4m3x2_encode(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}
__device__ __forceinline__ uint32_t e4m3_encode(float v) { return e4m3x2_encode(v, 0.0f) & 0xFFu; }

// E2M1 code -> value {0, .5, 1, 1.5, 2, 3, 4, 6} with sign (exact).
__device__ __forceinline__ float e2m1_value(uint32_t q) {
  const uint32_t m = q & 7u;
  const float v = m < 2u ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1u)) * ((m & 1u) ? 1.5f : 1.0f);
  return (q & 8u) ? -v : v;
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  uint32_t e = (c >> 3) & 15, m = c & 7;
  float v = (e == 0) ? (float)m * 0.001953125f : __uint_as_float(((e + 120) << 23) | (m << 20));
  return (c & 0x80u) ? -v : v;
}

// floor(log2 a) for a finite a > 0, exact from the bits.
__device__ __forceinline__ int ilog2_floor(float a) {
  const uint32_t b = __float_as_uint(a);
  const int ef = (int)(b >> 23);
  const int sub = (31 - __clz(b & 0x7FFFFFu)) - 149;  // subnormal: position of the leading bit
  return ef > 0 ? ef - 127 : sub;
}

__device__ __forceinline__ int ilog2_ceil(float a) {
  const uint32_t b = __float_as_uint(a);
  const int ef = (int)(b >> 23);
  const uint32_t m = b & 0x7FFFFFu;
  const int p = 31 - __clz(m);
  const int sub = p - 149 + (m != (1u << (p & 31)));
  return ef > 0 ? ef - 127 + (m != 0u) : sub;
}

// MOE_Y_FP16E expert outputs: the exponent of a 32-feature block with
// absolute maximum amax (its largest value then lands in [2^14, 2^15) of the
// fp16 range), and the fp16 codes (round to nearest even; the pair form puts
// the first value in the low half).
__device__ __forceinline__ int y16_exponent(float amax) {
  if (amax == 0.0f) return 0;
  const int e = ilog2_floor(amax) - 14;
  return e < -110 ? -110 : e;
}
__device__ __forceinline__ uint32_t f16x2_encode(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t f16_encode(float v) {
  uint16_t r;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float f16_value(uint16_t c) {
  float r;
  asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(c));
  return r;
}
// Both fp16 values of a 32-bit word (low half first), exactly.
__device__ __forceinline__ void f16x2_values(uint32_t u, float& lo, float& hi) {
  asm("{.reg .f16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}"
      : "=f"(lo), "=f"(hi)
      : "r"(u));
}

// E8M0 scale byte of one MXFP8 block with absolute maximum amax_b > 0.
__device__ __forceinline__ uint32_t mx_scale_code(float amax_b, int mode) {
  int e = (mode == 0) ? ilog2_floor(amax_b) - 8 : ilog2_ceil(__fdiv_rn(amax_b, 448.0f));
  int s = e + 127;
  s = s < 0 ? 0 : (s > 254 ? 254 : s);
  return (uint32_t)s;
}

// ----------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with the PDL attribute may
// start while its predecessor on the stream drains; pdl_wait() blocks until
// the predecessor has completed and its writes are visible (a no-op when the
// kernel was launched without the attribute); pdl_trigger() lets the next
// kernel's launch begin.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kern` on `st`, with programmatic stream serialisation when `pdl`.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ----------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete, for at most `limit` cycles.
// Returns false (and raises *abort, ORs `code` into *status) if it ran out or
// if another role has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status, uint32_t code, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(status, code);
      return false;
    }
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2D tiled TMA load into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"((uint64_t)src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// --- tcgen05 ---------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// Copy 32 rows x 16 bytes of shared memory into TMEM lanes 0..31 (replicated
// to all four lane quadrants), 4 columns starting at `taddr`.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T with NVFP4 operands (E2M1, UE4M3 scale per
// 16 elements, K = 64 per instruction).
__device__ __forceinline__ void mma_nvfp4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
          d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
// Same for MXFP8 operands (E4M3, UE8M0 scale per 32 elements, K = 32).
__device__ __forceinline__ void mma_mxfp8(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
          d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

// Hardware approximations (PTX ex2.approx / rcp.approx, relative error of a
// few 2^-23).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 lanes x 16 consecutive 32-bit columns of TMEM into registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): K-major, 128-byte swizzle,
// rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)2 << 61;            // SWIZZLE_128B
  return d;
}
// Descriptor of a 512-byte scale atom (32 rows x 16 bytes, no swizzle) for
// tcgen05.cp.  Only one 16-byte column, so both byte offsets may be 128.
__device__ __forceinline__ uint64_t sdesc_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptors (M = 128, K-major A and B, dense).
__device__ __forceinline__ uint32_t idesc_nvfp4(uint32_t N) {
  return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (0u << 23) | ((128u >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_mxfp8(uint32_t N, uint32_t sf_id) {
  return (sf_id << 4) | (0u << 7) | (0u << 10) | ((N >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
         (sf_id << 29);
}

}  // namespace moe
