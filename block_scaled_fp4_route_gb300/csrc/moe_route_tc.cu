// Router for prefill batches: logits on the tensor cores, with an exact
// re-check of every expert that could reach the top-k.
//
// The pages' router (SGLang blog on Inkling 2 Small, Performance section,
// kernel-fusion bullet; Miles docs section 1) is sigmoid(logits) + bias, top-k,
// weights s / sum s.  For thousands of tokens the logits GEMM (2 H E flop per
// token) is a dense contraction, so it runs on tcgen05 (kind::f16, bf16 x bf16
// products exact, fp32 accumulation).  The tensor core's accumulation order
// and rounding are not specified, so its logits only nominate candidates:
//
//   A_e = sigmoid(l_tc) + b_e,  m_e = (gamma/4) ||x|| ||w_e|| + slack
//   (the sigmoid's slope is at most 1/4, Cauchy-Schwarz bounds sum|x w|)
//   L   = k-th largest of A_e - m_e
//   C   = { e : A_e + m_e >= L }   (contains the exact top-k; |C| >= k)
//
// and every candidate's logit is recomputed on CUDA cores with the error
// bound of the decode router (fp32 chunks of 32 products, Kahan across
// chunks, an exact two-sum tree across the warp: at most 34u sum|x w|).  The
// top-k and the weights come from those recomputed logits only, so the
// result is the one the exact-arithmetic router would give up to the same
// rounding bound as the CUDA-core path, whatever the tensor core's rounding
// within gamma = 2^-11 relative to ||x|| ||w_e|| (about 2^12 times the
// rounding of an fp32 accumulation over 4608 terms).
//
// Three kernels: k_router_prep (||w_e|| for every expert; clears the status
// word), k_router_tc (one 128-token x 128-expert tile per CTA, TMA -> smem ->
// tcgen05.mma -> TMEM -> fp32 logits), k_router_select (one warp per token).
#include <type_traits>

#include "moe_common.cuh"

namespace moe {

namespace {

constexpr float kTcGamma = 1.0f / 2048.0f;        // assumed |l_tc - l| / (||x|| ||w_e||) bound
// the approximate keys' own arithmetic: a sigmoid from __expf and a
// reciprocal (|error| below 2^-22 of the key: s(1-s) times the exponential's
// relative error, plus the two roundings) and the fp32 bias add
constexpr float kKeySlack = 1.0f / 262144.0f;
constexpr float kNormInflate = 1.0f + 1.0f / 1024.0f;  // fp32 sum-of-squares rounding -> upper bound

// ---------------------------------------------------------------------------
// ||w_e|| (an upper bound: the fp32 sum of H exact squares is inflated), one
// warp per expert.  Block 0 clears the status word of the call.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_router_prep(const __nv_bfloat16* __restrict__ wr, int E, int H,
                                                     float* __restrict__ wnorm, uint32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x == 0 && status) *status = 0u;
  if (e >= E) return;
  const __nv_bfloat16* row = wr + (int64_t)e * H;
  float ss = 0.0f;
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + i);
    const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = __uint_as_float(v[j] << 16), b = __uint_as_float(v[j] & 0xFFFF0000u);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) wnorm[e] = sqrtf(ss) * kNormInflate;
}

// ---------------------------------------------------------------------------
// Logits tile: 128 tokens (MMA M, TMEM lanes) x up to NE experts (MMA N,
// TMEM columns) x all of H.  Warp 0: TMA producer; warp 1: MMA issuer; warp 2:
// TMEM allocator; warps 4..7: epilogue (warp w reads lane quadrant w % 4).
// NE = 128 (six stages), or 192 for large batches (five stages): each token
// tile is then read by fewer CTAs, and 128 token tiles x 2 expert tiles fill
// the GPU in under two waves where 128 x 3 take three.
// ---------------------------------------------------------------------------
constexpr int kRtBox = 128 * 128;  // the token operand per stage: 128 rows x 64 bf16
template <int NE>
struct RtCfg {
  static constexpr int STAGES = NE == 128 ? 6 : 5;
  static constexpr int BOXW = NE * 128;                    // the expert operand per stage
  static constexpr int STAGE = kRtBox + BOXW;
  static constexpr int SMEM = STAGES * STAGE + 256 + 1024;
  static constexpr int TMEM_COLS = NE <= 128 ? 128 : 256;  // a power of two
  static_assert(SMEM <= 232448, "router tile shared memory");
};

__device__ __forceinline__ uint32_t idesc_bf16(uint32_t N) {
  // fp32 accumulator, bf16 A and B, both K-major, M = 128
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((128u >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int NE>
__global__ void __launch_bounds__(256, 1) k_router_tc(const __grid_constant__ CUtensorMap tmx,
                                                     const __grid_constant__ CUtensorMap tmw,
                                                     float* __restrict__ lt, int T, int E, int H,
                                                     uint32_t* status, long long limit) {
  using R = RtCfg<NE>;
  constexpr int kRtStages = R::STAGES;
  extern __shared__ uint8_t rt_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rt_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRtStages * R::STAGE);
  uint64_t* empty = full + kRtStages;
  uint64_t* done = empty + kRtStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * NE, t0 = blockIdx.y * 128;
  const int N = min(NE, E - e0);  // a multiple of 16
  const int KB = H / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, R::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmx);
    prefetch_tmap(&tmw);
  }
  pdl_wait();  // the previous kernel cleared the status word
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, status, ST_TIMEOUT_PRODUCER, limit)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + stage * R::STAGE;
        mbar_expect_tx(&full[stage], R::STAGE);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        tma_load_2d(sA, &tmx, &full[stage], kb * 128, t0);
        tma_load_2d(sA + kRtBox, &tmw, &full[stage], kb * 128, e0);
        if (++stage == kRtStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {  // wait (bounded) for the copies this thread put in flight
        for (int s = 0; s < kRtStages; ++s) {
          if (!((armed >> s) & 1u)) continue;
          const uint32_t par = (armed_par >> s) & 1u;
          const long long c0 = clock64();
          while (!mbar_try_wait(&full[s], par) && clock64() - c0 < limit) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t id = idesc_bf16((uint32_t)N);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag, status, ST_TIMEOUT_MMA, limit)) break;
        tc_fence_after();
        uint8_t* sA = smem + stage * R::STAGE;
        const uint64_t da = sdesc_sw128(smem_u32(sA));
        const uint64_t db = sdesc_sw128(smem_u32(sA + kRtBox));
#pragma unroll
        for (int s = 0; s < 4; ++s)  // K = 16 per instruction: 32 bytes along the swizzled row
          mma_bf16(tmem, da + (uint64_t)(2 * s), db + (uint64_t)(2 * s), id, (kb | s) != 0);
        tc_commit(&empty[stage]);
        if (++stage == kRtStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      // every tcgen05 operation of this thread completes before TMEM is read or freed
      tc_commit(done);
      const long long c0 = clock64();
      while (!mbar_try_wait(done, 0) && clock64() - c0 < limit) {
      }
    }
  } else if (warp >= 4) {
    const int q = warp & 3;
    const int t = t0 + q * 32 + lane;
    // the warp decides together: tcgen05.ld needs all lanes
    if (__all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, status, ST_TIMEOUT_EPILOGUE, limit))) {
      tc_fence_after();
      for (int c = 0; c < N; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, r);
        tmem_wait_ld();
        if (t < T) {
          float4* dst = reinterpret_cast<float4*>(lt + (int64_t)t * E + e0 + c);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, R::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Selection: one warp per token.
// ---------------------------------------------------------------------------
constexpr int kSelWarps = 4;

struct Kahan {
  float s = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float v) {
    const float y = __fsub_rn(v, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
};

// sum_h x_h w_h for NC experts at once, on CUDA cores.  The warp reads x and
// w in coalesced 512-byte slots: in slot q lane i holds the 8 elements at
// 256 q + 8 i.  A lane's chunk is its 32 elements of four consecutive slots
// (fewer in the last chunk), summed as an in-order chain of fp32 FMAs (the
// bf16 products are exact); the lane adds its chunk sums with Kahan
// compensation, and the lanes' (sum, compensation) pairs meet in an xor tree
// of exact two-sums, so every lane returns the same value.  Error at most
// (31 + 2 + 1) u sum|x w|, u = 2^-24.  The NC experts share the loads of x
// and their loads are issued together.
// The products go straight from the bf16 halves of each word into an fp32
// fused multiply-add (fma.rn.f32.bf16: the bf16 operands are exact in fp32,
// the product is exact, one rounding per add), lower element first: the
// same chain as unpacking both to fp32 and using fmaf, without the unpacking.
__device__ __forceinline__ void slot_fma(const uint4& xa, const uint4& wa, float& p) {
  const uint32_t xv[4] = {xa.x, xa.y, xa.z, xa.w};
  const uint32_t wv[4] = {wa.x, wa.y, wa.z, wa.w};
#pragma unroll
  for (int j = 0; j < 4; ++j)
    asm("{\n.reg .b16 xl, xh, wl, wh;\nmov.b32 {xl, xh}, %1;\nmov.b32 {wl, wh}, %2;\n"
        "fma.rn.f32.bf16 %0, xl, wl, %0;\nfma.rn.f32.bf16 %0, xh, wh, %0;\n}"
        : "+f"(p)
        : "r"(xv[j]), "r"(wv[j]));
}

template <int NC>
__device__ void exact_logits(const __nv_bfloat16* __restrict__ xr, const __nv_bfloat16* const (&wrow)[NC], int H,
                             int lane, float (&out)[NC]) {
  Kahan acc[NC];
  const int Q = (H + 255) / 256;  // slots; H % 128 == 0, so the last one has 16 or 32 lanes
  for (int q0 = 0; q0 < Q; q0 += 4) {
    uint4 xa[4], wa[NC][4];
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      const int off = 256 * (q0 + d) + 8 * lane;
      const bool in = q0 + d < Q && off < H;
      xa[d] = in ? *reinterpret_cast<const uint4*>(xr + off) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int n = 0; n < NC; ++n)
        wa[n][d] = in ? __ldg(reinterpret_cast<const uint4*>(wrow[n] + off)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int n = 0; n < NC; ++n) {
      float p = 0.0f;  // zero padding adds exact zeros
#pragma unroll
      for (int d = 0; d < 4; ++d) slot_fma(xa[d], wa[n][d], p);
      acc[n].add(p);
    }
  }
#pragma unroll
  for (int n = 0; n < NC; ++n) {
    float s = acc[n].s, e = -acc[n].c;  // the lane's sum is s + e
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float e2 = __shfl_xor_sync(0xffffffffu, e, o);
      const float t = __fadd_rn(s, s2);
      const float bp = __fsub_rn(t, s);
      const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(s2, bp));  // s + s2 - t exactly
      s = t;
      e = __fadd_rn(__fadd_rn(e, e2), err);
    }
    out[n] = __fadd_rn(s, e);
  }
}

__device__ __forceinline__ float router_sigmoid(float l) { return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l))); }

// Warp arg-max of (v, e): larger v, then lower e; every lane gets the winner.
__device__ __forceinline__ void warp_argmax(float& v, int& e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oe = __shfl_xor_sync(0xffffffffu, e, o);
    if (ov > v || (ov == v && oe < e)) {
      v = ov;
      e = oe;
    }
  }
}

// KPL: experts per lane (E <= 32 KPL); lane l holds experts l, l + 32, ...
template <int KPL>
__global__ void __launch_bounds__(kSelWarps * 32) k_router_select(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wr, const float* __restrict__ lt,
    const float* __restrict__ wnorm, const float* __restrict__ bias, int T, int H, int E, int k,
    int bias_in_weights, float routed_scale, int32_t* __restrict__ idx, float* __restrict__ w) {
  extern __shared__ float sel_smem[];  // per warp: ckey[E], cs[E], cid[E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + warp;
  pdl_wait();
  pdl_trigger();
  if (t >= T) return;  // whole warp
  float* ckey = sel_smem + (size_t)warp * 3 * E;
  float* cs = ckey + E;
  int* cid = reinterpret_cast<int*>(cs + E);
  const __nv_bfloat16* xr = x + (int64_t)t * H;

  // this lane's tensor-core logits, requested together (they land while
  // ||x|| is summed)
  float ltv[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) ltv[i] = lane + 32 * i < E ? lt[(int64_t)t * E + lane + 32 * i] : 0.0f;

  // ||x|| (upper bound)
  float ss = 0.0f;
#pragma unroll 6
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 u = *reinterpret_cast<const uint4*>(xr + i);
    const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm("{\n.reg .b16 l, h;\nmov.b32 {l, h}, %1;\nfma.rn.f32.bf16 %0, l, l, %0;\nfma.rn.f32.bf16 %0, h, h, %0;\n}"
          : "+f"(ss)
          : "r"(v[j]));
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float xn = sqrtf(ss) * kNormInflate;

  // approximate keys and their margins, in registers
  float lov[KPL], hiv[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    lov[i] = -INFINITY;
    hiv[i] = -INFINITY;
    if (e < E) {
      const float a = __fadd_rn(__frcp_rn(__fadd_rn(1.0f, __expf(-ltv[i]))), bias[e]);
      const float m = 0.25f * kTcGamma * xn * wnorm[e] + kKeySlack;
      lov[i] = a - m;
      hiv[i] = a + m;
    }
  }

  // L = k-th largest lower bound: each round the warp takes the best of the
  // lanes' bests (ties to the lower expert index); only the winner's lane
  // drops it and rescans its own bounds
  float lb;
  int le;
  auto lane_best = [&]() {
    lb = -INFINITY;
    le = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      if (32 * i >= E) break;
      if (lov[i] > lb) {
        lb = lov[i];
        le = lane + 32 * i;
      }
    }
  };
  lane_best();
  float L = -INFINITY;
  for (int r = 0; r < k; ++r) {
    float bv = lb;
    int be = le;
    warp_argmax(bv, be);
    L = bv;
    if (be != 0x7fffffff && (be & 31) == lane) {
#pragma unroll
      for (int i = 0; i < KPL; ++i)
        if (i == (be >> 5)) lov[i] = -INFINITY;
      lane_best();
    }
  }

  // candidates, in expert order
  int nc = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    if (32 * i >= E) break;
    const bool cand = lane + 32 * i < E && hiv[i] >= L;
    const unsigned bal = __ballot_sync(0xffffffffu, cand);
    if (cand) cid[nc + __popc(bal & ((1u << lane) - 1u))] = lane + 32 * i;
    nc += __popc(bal);
  }
  __syncwarp();

  // exact keys of the candidates: three at a time (larger groups measured
  // slower: their registers cost resident warps), the last one or two in a
  // group of their own size (no padded dot products)
  auto exact_group = [&](auto g_tag, int i0) {
    constexpr int G = decltype(g_tag)::value;
    const __nv_bfloat16* rows[G];
#pragma unroll
    for (int n = 0; n < G; ++n) rows[n] = wr + (int64_t)cid[i0 + n] * H;
    float l[G];
    exact_logits<G>(xr, rows, H, lane, l);
#pragma unroll
    for (int n = 0; n < G; ++n)
      if (lane == n) {
        const float sg = router_sigmoid(l[n]);
        cs[i0 + n] = sg;
        ckey[i0 + n] = __fadd_rn(sg, bias[cid[i0 + n]]);
      }
  };
  int i0 = 0;
  for (; i0 + 3 <= nc; i0 += 3) exact_group(std::integral_constant<int, 3>{}, i0);
  if (nc - i0 == 2) exact_group(std::integral_constant<int, 2>{}, i0);
  else if (nc - i0 == 1) exact_group(std::integral_constant<int, 1>{}, i0);
  __syncwarp();

  // top-k of the candidates by exact key, ties to the lower expert index
  // (slots are in expert order, so the lower slot is the lower expert)
  float num = 0.0f;  // lane r keeps winner r's numerator
  int win = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bs = 0x7fffffff;
    for (int i = lane; i < nc; i += 32)
      if (ckey[i] > bv) {  // ascending slots: the first of equal keys stays
        bv = ckey[i];
        bs = i;
      }
    warp_argmax(bv, bs);
    if (bs >= nc) bs = 0;  // only if every remaining key is NaN; stays in bounds
    if (lane == r) {
      win = cid[bs];
      num = bias_in_weights ? ckey[bs] : cs[bs];
    }
    __syncwarp();
    if (lane == (bs & 31)) ckey[bs] = -INFINITY;
    __syncwarp();
  }
  // weights: sum of the numerators in selection order (one lane, fixed order)
  float den = 0.0f;
  for (int r = 0; r < k; ++r) den = __fadd_rn(den, __shfl_sync(0xffffffffu, num, r));
  if (lane < k) {
    idx[(int64_t)t * k + lane] = win;
    w[(int64_t)t * k + lane] = __fmul_rn(routed_scale, __fdiv_rn(num, den));
  }
}

}  // namespace

bool router_uses_tc(const moe_config& c) { return c.T > 256 && c.E % 16 == 0 && c.H % 64 == 0; }

size_t router_tc_scratch_floats(const moe_config& c) {
  return (size_t)c.T * c.E + (((size_t)c.E + 63) / 64) * 64;  // logits [T, E], then ||w_e|| [E]
}

cudaError_t launch_router_tc(const moe_config& c, const __nv_bfloat16* x, const __nv_bfloat16* wr,
                             const float* bias, float* scratch, int32_t* idx, float* w, uint32_t* status,
                             cudaStream_t st, bool pdl) {
  static PerDeviceOnce attr;
  const size_t sel_smem = (size_t)kSelWarps * 3 * c.E * 4;
  auto select = c.E <= 128 ? k_router_select<4> : c.E <= 256 ? k_router_select<8>
                : c.E <= 512 ? k_router_select<16> : k_router_select<32>;
  static_assert(32 * 32 >= kMaxE, "selection experts per lane");
  cudaError_t ea = once_per_device(attr, [] {
    cudaError_t r = cudaFuncSetAttribute(k_router_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         RtCfg<128>::SMEM);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(k_router_tc<192>, cudaFuncAttributeMaxDynamicSharedMemorySize, RtCfg<192>::SMEM);
    for (auto kern : {k_router_select<4>, k_router_select<8>, k_router_select<16>, k_router_select<32>})
      if (r == cudaSuccess)
        r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelWarps * 3 * kMaxE * 4);
    return r;
  });
  if (ea != cudaSuccess) return ea;
  // 192-expert tiles once 128-expert tiles would take more than two waves
  int dev = 0, sms = 0;
  cudaError_t ea2 = cudaGetDevice(&dev);
  if (ea2 == cudaSuccess) ea2 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ea2 != cudaSuccess) return ea2;
  const bool wide = (int64_t)((c.T + 127) / 128) * ((c.E + 127) / 128) > 2 * (int64_t)sms;
  const int ne = wide ? 192 : 128;
  CUtensorMap tmx, tmw;
  if (!make_map(&tmx, x, c.T, (int64_t)c.H * 2, 128) || !make_map(&tmw, wr, c.E, (int64_t)c.H * 2, ne))
    return cudaErrorInvalidValue;
  float* lt = scratch;
  float* wnorm = scratch + (size_t)c.T * c.E;
  cudaError_t e = launch_k(k_router_prep, dim3((c.E + 7) / 8), dim3(256), 0, st, pdl, wr, c.E, c.H, wnorm, status);
  if (e != cudaSuccess) return e;
  if (wide)
    e = launch_k(k_router_tc<192>, dim3((c.E + 191) / 192, (c.T + 127) / 128), dim3(256), RtCfg<192>::SMEM, st, true,
                 tmx, tmw, lt, c.T, c.E, c.H, status, 4000000000LL);
  else
    e = launch_k(k_router_tc<128>, dim3((c.E + 127) / 128, (c.T + 127) / 128), dim3(256), RtCfg<128>::SMEM, st, true,
                 tmx, tmw, lt, c.T, c.E, c.H, status, 4000000000LL);
  if (e != cudaSuccess) return e;
  return launch_k(select, dim3((c.T + kSelWarps - 1) / kSelWarps), dim3(kSelWarps * 32), sel_smem, st, true,
                  x, wr, (const float*)lt, (const float*)wnorm, bias, c.T, c.H, c.E, c.k, c.bias_in_weights,
                  c.routed_scale, idx, w);
}

}  // namespace moe
