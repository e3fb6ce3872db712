// Fused router: logits GEMM, sigmoid, additive bias, top-k, normalisation
// (SGLang blog on Inkling 2 Small, Performance section, kernel-fusion bullet:
// sigmoid, bias and top-k form one router kernel; Miles docs section 1:
// sigmoid routing over 384 experts, 8 per token).
//
// Logits: fp32 on CUDA cores.  Each output sums its bf16 x bf16 products
// (exact in fp32) in chunks of 32 with plain fp32 adds, and the chunk sums are
// added with Kahan compensation (within a K split and again across splits).
// Hence |l_gpu - l| <= (gamma_31 + 3u) * sum_h |x_h w_eh| <= 40u * sum|x w|,
// u = 2^-24, which the top-k parity check uses to certify near-ties.  Decode
// batches (T <= 256) use these kernels; larger batches the tensor-core router
// with an exact re-check (moe_route_tc.cu).
#include <mutex>

#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kKC = 64;        // K elements per smem stage
constexpr int kChunk = 32;     // plain-sum chunk length
constexpr int kPad = 4;        // fp32 row padding (conflict-free float4 reads)

struct Kahan {
  float s = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float v) {
    float y = __fsub_rn(v, c);
    float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
};

// CTA tile (16*RM tokens) x (16*RN experts); 256 threads as 16 x 16.
template <int RM, int RN>
__global__ void __launch_bounds__(256) k_router_logits(const __nv_bfloat16* __restrict__ x,
                                                       const __nv_bfloat16* __restrict__ wr, float* __restrict__ part,
                                                       int T, int H, int E, int k_len, uint32_t* status) {
  constexpr int TM = 16 * RM, TE = 16 * RN;
  extern __shared__ __align__(16) float router_smem[];
  float(*As)[TM][kKC + kPad] = reinterpret_cast<float(*)[TM][kKC + kPad]>(router_smem);
  float(*Bs)[TE][kKC + kPad] = reinterpret_cast<float(*)[TE][kKC + kPad]>(router_smem + 2 * TM * (kKC + kPad));
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int e0 = blockIdx.x * TE, t0 = blockIdx.y * TM;
  const int split = blockIdx.z;
  const int kbeg = split * k_len;
  const int nst = k_len / kKC;
  pdl_wait();
  if (status && (blockIdx.x | blockIdx.y | blockIdx.z | threadIdx.x) == 0) *status = 0u;

  // register staging of one stage: rows x 8 uint4 (8 bf16 each)
  constexpr int A_VEC = TM * (kKC / 8), B_VEC = TE * (kKC / 8);
  constexpr int A_PER = (A_VEC + 255) / 256, B_PER = (B_VEC + 255) / 256;
  uint4 ra[A_PER], rb[B_PER];

  auto gload = [&](int st) {
    int kk = kbeg + st * kKC;
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
      int v = threadIdx.x + 256 * i;
      ra[i] = make_uint4(0, 0, 0, 0);
      if (v < A_VEC) {
        int r = v >> 3, q = v & 7;
        if (t0 + r < T) ra[i] = *reinterpret_cast<const uint4*>(x + (int64_t)(t0 + r) * H + kk + 8 * q);
      }
    }
#pragma unroll
    for (int i = 0; i < B_PER; ++i) {
      int v = threadIdx.x + 256 * i;
      rb[i] = make_uint4(0, 0, 0, 0);
      if (v < B_VEC) {
        int r = v >> 3, q = v & 7;
        if (e0 + r < E) rb[i] = *reinterpret_cast<const uint4*>(wr + (int64_t)(e0 + r) * H + kk + 8 * q);
      }
    }
  };
  auto unpack_store = [&](float* dst, uint4 u) {
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float4 lo = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                            __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
    float4 hi = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                            __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
    reinterpret_cast<float4*>(dst)[0] = lo;
    reinterpret_cast<float4*>(dst)[1] = hi;
  };
  auto sstore = [&](int buf) {
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
      int v = threadIdx.x + 256 * i;
      if (v < A_VEC) unpack_store(&As[buf][v >> 3][8 * (v & 7)], ra[i]);
    }
#pragma unroll
    for (int i = 0; i < B_PER; ++i) {
      int v = threadIdx.x + 256 * i;
      if (v < B_VEC) unpack_store(&Bs[buf][v >> 3][8 * (v & 7)], rb[i]);
    }
  };

  Kahan acc[RM][RN];
  gload(0);
  sstore(0);
  __syncthreads();
  for (int st = 0; st < nst; ++st) {
    const int buf = st & 1;
    if (st + 1 < nst) gload(st + 1);
#pragma unroll
    for (int ch = 0; ch < kKC / kChunk; ++ch) {
      float p[RM][RN];
#pragma unroll
      for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < RN; ++j) p[i][j] = 0.0f;
#pragma unroll
      for (int kq = 0; kq < kChunk; kq += 4) {
        float4 a[RM], b[RN];
#pragma unroll
        for (int i = 0; i < RM; ++i) a[i] = *reinterpret_cast<const float4*>(&As[buf][ty + 16 * i][ch * kChunk + kq]);
#pragma unroll
        for (int j = 0; j < RN; ++j) b[j] = *reinterpret_cast<const float4*>(&Bs[buf][tx + 16 * j][ch * kChunk + kq]);
#pragma unroll
        for (int i = 0; i < RM; ++i)
#pragma unroll
          for (int j = 0; j < RN; ++j) {
            p[i][j] = __fmaf_rn(a[i].x, b[j].x, p[i][j]);
            p[i][j] = __fmaf_rn(a[i].y, b[j].y, p[i][j]);
            p[i][j] = __fmaf_rn(a[i].z, b[j].z, p[i][j]);
            p[i][j] = __fmaf_rn(a[i].w, b[j].w, p[i][j]);
          }
      }
#pragma unroll
      for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < RN; ++j) acc[i][j].add(p[i][j]);
    }
    if (st + 1 < nst) {
      sstore(buf ^ 1);
    }
    __syncthreads();
  }
  float* out = part + (int64_t)split * T * E;
#pragma unroll
  for (int i = 0; i < RM; ++i)
#pragma unroll
    for (int j = 0; j < RN; ++j) {
      int t = t0 + ty + 16 * i, e = e0 + tx + 16 * j;
      if (t < T && e < E) out[(int64_t)t * E + e] = acc[i][j].s;
    }
  pdl_trigger();
}

constexpr int kMaxSplits = 24;

// One CTA per token, one thread per expert: sum the K-split partials (Kahan,
// fixed order; all loads of the token in flight at once), sigmoid, bias, into
// shared memory; then warp 0 runs k rounds of a warp arg-max over them (ties
// in the key go to the lower expert index) and normalises the weights over
// the winners in selection order.
// KPL: keys per lane of the selection warp (E <= 32 KPL).
template <int KPL>
__global__ void __launch_bounds__(1024) k_router_topk(const float* __restrict__ part, int nsplit,
                                                      const float* __restrict__ bias, int T, int E, int k,
                                                      int bias_in_weights, float routed_scale,
                                                      int32_t* __restrict__ idx, float* __restrict__ w) {
  extern __shared__ float topk_smem[];  // key[E], sg[E]
  float* key = topk_smem;
  float* sgm = key + E;
  const int t = blockIdx.x;
  const int e = threadIdx.x;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (e < E) {
    float v[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) v[s] = s < nsplit ? part[((int64_t)s * T + t) * E + e] : 0.0f;
    Kahan l;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
      if (s < nsplit) l.add(v[s]);
    const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l.s)));
    sgm[e] = sg;
    key[e] = __fadd_rn(sg, bias[e]);
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  // warp 0: lane l holds the keys of experts l, l + 32, ... in registers and
  // its best one; each round the warp takes the best of the lanes' bests (ties
  // in the key go to the lower expert index) and only the winner's lane drops
  // it and rescans its own keys
  float kv[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) kv[i] = lane + 32 * i < E ? key[lane + 32 * i] : -INFINITY;
  auto lane_best = [&](float& bv, int& be) {
    bv = -INFINITY;
    be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      if (32 * i >= E) break;
      if (kv[i] > bv) {  // ascending index: the first of equal keys stays
        bv = kv[i];
        be = lane + 32 * i;
      }
    }
  };
  float lb;
  int le;
  lane_best(lb, le);
  float num = 0.0f;  // lane j keeps winner j's numerator
  int win = 0;
  for (int j = 0; j < k; ++j) {
    float bv = lb;
    int be = le;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be >= E) be = 0;  // only if every remaining key is NaN; stays in bounds
    if (lane == j) {
      win = be;
      num = bias_in_weights ? key[be] : sgm[be];
    }
    if (lane == (be & 31)) {
#pragma unroll
      for (int i = 0; i < KPL; ++i)
        if (i == (be >> 5)) kv[i] = -INFINITY;
      lane_best(lb, le);
    }
  }
  float den = 0.0f;
  for (int j = 0; j < k; ++j) den = __fadd_rn(den, __shfl_sync(0xffffffffu, num, j));
  if (lane < k) {
    idx[(int64_t)t * k + lane] = win;
    w[(int64_t)t * k + lane] = __fmul_rn(routed_scale, __fdiv_rn(num, den));
  }
}

constexpr int router_smem_bytes(int rm, int rn) { return 2 * 16 * (rm + rn) * (kKC + kPad) * 4; }

}  // namespace

// Number of K splits of the logits GEMM (also sizes the partials buffer):
// enough 64x64 output tiles x splits to fill the GPU for decode batches, each
// split a whole number of 64-element stages.  Above 64 tokens 12 splits
// (measured on GB300: a 192-token layer 1172 -> 1159 us against 8; 24 gain
// nothing more); the static array of moe_route_noalloc keeps 8 there.
int router_splits(const moe_config& c, bool fixed_scratch) {
  int cap = c.T <= 64 ? kMaxSplits : (c.T <= 256 ? (fixed_scratch ? 8 : 12) : 1);
  for (int s = cap; s > 1; --s)
    if (c.H % (kKC * s) == 0) return s;
  return 1;
}

size_t router_scratch_floats(const moe_config& c, bool fixed_scratch) {
  return router_uses_tc(c) ? router_tc_scratch_floats(c) : (size_t)router_splits(c, fixed_scratch) * c.T * c.E;
}

cudaError_t launch_router(const moe_config& c, const __nv_bfloat16* x, const __nv_bfloat16* wr, const float* bias,
                          float* logits, int32_t* idx, float* w, uint32_t* status, cudaStream_t st, bool pdl,
                          bool fixed_scratch) {
  if (router_uses_tc(c)) return launch_router_tc(c, x, wr, bias, logits, idx, w, status, st, pdl);
  const int ns = router_splits(c, fixed_scratch);
  const int k_len = c.H / ns;
  static PerDeviceOnce attr;
  cudaError_t e = once_per_device(attr, [] {
    cudaError_t r = cudaFuncSetAttribute(k_router_logits<4, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         router_smem_bytes(4, 4));
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(k_router_logits<1, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               router_smem_bytes(1, 4));
    return r;
  });
  if (e != cudaSuccess) return e;
  // token tiles of 16 rows for the smallest batches (a quarter of the FMAs
  // of the 64-row tile; every logit's arithmetic is the same)
  if (c.T <= 16) {
    e = launch_k(k_router_logits<1, 4>, dim3((c.E + 63) / 64, 1, ns), dim3(256), router_smem_bytes(1, 4), st, pdl, x,
                 wr, logits, c.T, c.H, c.E, k_len, status);
  } else {
    e = launch_k(k_router_logits<4, 4>, dim3((c.E + 63) / 64, (c.T + 63) / 64, ns), dim3(256),
                 router_smem_bytes(4, 4), st, pdl, x, wr, logits, c.T, c.H, c.E, k_len, status);
  }
  if (e != cudaSuccess) return e;
  auto topk = c.E <= 128 ? k_router_topk<4> : c.E <= 256 ? k_router_topk<8> : c.E <= 512 ? k_router_topk<16>
                                                                                  : k_router_topk<32>;
  static_assert(32 * 32 >= kMaxE, "selection keys per lane");
  return launch_k(topk, dim3(c.T), dim3((c.E + 31) / 32 * 32), (size_t)2 * c.E * 4, st, true, (const float*)logits,
                  ns, bias, c.T, c.E, c.k, c.bias_in_weights, c.routed_scale, idx, w);
}

// ----------------------------------------------------------------------------
// Router without a caller-provided workspace (moe_route_noalloc).
//
// Some callers cannot allocate device memory at the point where they route
// tokens: for example code running inside a captured CUDA graph region, a
// plugin that has no access to its host framework's allocator, or a runtime
// that forbids allocation after start-up.  For them the router's scratch (a
// status word and the fp32 logits) lives in a fixed array that the CUDA module
// reserves when the library is loaded, so the call itself allocates nothing.
// ----------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchFloats = (size_t)1 << 20;  // 4 MiB: status word area + router scratch
constexpr size_t kNoAllocHeaderFloats = 64;
static __device__ __align__(256) float g_route_scratch[kNoAllocScratchFloats];

struct NoAllocDevice {
  bool ready = false;
  moe_status status = MOE_OK;
  float* scratch = nullptr;  // device address of g_route_scratch on that device
};
NoAllocDevice g_noalloc[64];
std::mutex g_noalloc_mu;

// Once per device, with that device current: look up the device address of
// the scratch array (the host-side name is only a stand-in for it).
moe_status noalloc_setup(float** scratch) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      d.status = MOE_ERR_CUDA;
    } else if (!(major == 10 && minor == 3)) {
      d.status = MOE_ERR_ARCH;
    } else {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
      if (e != cudaSuccess || p == nullptr) {
        d.status = MOE_ERR_CUDA;
      } else {
        d.scratch = static_cast<float*>(p);
        d.status = MOE_OK;
      }
    }
    d.ready = true;
  }
  *scratch = d.scratch;
  return d.status;
}

}  // namespace

}  // namespace moe

extern "C" moe_status moe_route_noalloc_poll_status(void* stream) {
  using namespace moe;
  float* scratch = nullptr;
  moe_status s = noalloc_setup(&scratch);
  if (s != MOE_OK) return s;
  // the status word is the first word of the array's header area
  return moe_poll_device_status(scratch, stream);
}

extern "C" moe_status moe_route_noalloc(const moe_config* cfg, const void* x_dev, const void* w_router_dev,
                                        const float* bias_dev, int32_t* topk_idx_dev, float* topk_w_dev,
                                        void* stream) {
  using namespace moe;
  size_t ws_bytes = 0;
  moe_status s = moe_workspace_size(cfg, &ws_bytes);  // validates the configuration
  if (s != MOE_OK) return s;
  const void* ptrs[] = {x_dev, w_router_dev, bias_dev, topk_idx_dev, topk_w_dev};
  for (const void* p : ptrs) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return MOE_ERR_MISALIGNED;
  }
  // the array holds a 256-byte status word area, then the router's scratch
  const size_t need = kNoAllocHeaderFloats + router_scratch_floats(*cfg, true);
  if (need > kNoAllocScratchFloats) return MOE_ERR_WORKSPACE_TOO_SMALL;
  float* scratch = nullptr;
  s = noalloc_setup(&scratch);
  if (s != MOE_OK) return s;
  // every logits partial the top-k kernel reads is written first by the
  // logits kernel of the same call, so nothing needs clearing
  cudaError_t e = launch_router(*cfg, (const __nv_bfloat16*)x_dev, (const __nv_bfloat16*)w_router_dev, bias_dev,
                                scratch + kNoAllocHeaderFloats, topk_idx_dev, topk_w_dev,
                                reinterpret_cast<uint32_t*>(scratch), (cudaStream_t)stream, false, true);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
