// Decode batches: the whole expert FFN (both grouped GEMMs, the capped SwiGLU
// between them and the quantisation of h) in one persistent launch.
//
// The pages fuse the layer's stages into one kernel (SGLang blog on Inkling 2
// Small, Performance, MegaMoE bullet: one fused kernel replaced the grouped
// GEMM path; cookbook, MegaMoE paragraph: dispatch, both expert GEMMs, the
// capped SwiGLU and the combine in one unit), and the TokenSpeed page says
// single-user decode is bound by kernel launches and dependency waits rather
// than math.  For a decode batch the two GEMMs stream the touched experts'
// weights once each; as separate kernels the down GEMM's weight stream starts
// only after the last gate/up tile, the h pass and a launch.  Here every CTA
// runs its gate/up tiles (the tile list of the separate GEMM1) and then its
// down tiles (that of GEMM2) in one loop, with the same 64-row-tile pipeline,
// and a down tile waits only for the h rows it multiplies:
//
//   * each gate/up tile's epilogue, once its four warps have stored their h
//     (bf16 for NVFP4, codes and scales for MXFP8), adds one to the row
//     tile's completion count (release);
//   * NVFP4: the epilogue whose addition completes a row tile (all F / 128
//     gate/up tiles of it) quantises that tile's h rows (a warp per row, the
//     row-pass arithmetic of the separate h kernel, global over the whole
//     row) and then publishes the row tile as ready;
//   * the producer of a down tile requests the tile's weight stages (as many
//     as the pipeline holds) before it waits (bounded, acquire) for its row
//     tile, and the h rows afterwards, so the down weights stream while the
//     last gate/up tiles finish.
//
// Tiles are handed out in one global order, all gate/up tiles before all down
// tiles, by a counter in global memory: a CTA's producer takes the next index
// when it is ready for a new tile and passes it to the CTA's MMA and epilogue
// warps through a small ring in shared memory.  A down tile is therefore
// taken only after every gate/up tile has been taken by a running CTA, and a
// gate/up tile waits on nothing, so every down tile's wait ends whether or not
// all CTAs are resident at once (no cooperative launch is needed, and the
// kernel starts early behind the previous one by programmatic dependent
// launch).  Taking tiles on demand also balances the gate/up tiles (K = H)
// against the shorter down tiles (K = F).  Each wait is bounded anyway and
// reports ST_TIMEOUT_DEPEND in the status word when it runs out.
//
// The counters (two int32 per row tile, then the tile counter) are zeroed by
// the kernel that builds the tile plan, earlier on the same stream.
#include "moe_gemm_common.cuh"
#include "moe_quant_dev.cuh"

namespace moe {

namespace {

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_relaxed(const int32_t* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// after a relaxed read that saw a release store: together an acquire
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_release(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// order this thread's generic-proxy accesses with its async-proxy (TMA) ones
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// named barrier 1 over the four epilogue warps (128 threads): plain, and with
// an AND of a predicate
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_all(bool p) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred a, b;\nsetp.ne.u32 a, %1, 0;\nbar.red.and.pred b, 1, 128, a;\nselp.u32 %0, 1, 0, b;\n}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}

constexpr int kSchedDepth = 4;  // tiles in flight between the producer and the epilogue

struct FfnSync {
  int32_t* done1;            // [row tiles] gate/up tiles finished
  int32_t* ready;            // [row tiles] NVFP4: h rows quantised
  int32_t* next_tile;        // the tile counter
  uint32_t* h_amax;          // [R] NVFP4: |h| maximum of each row (float bits), from the gate/up epilogues
  const float* act_static;   // NVFP4 static activation globals [E, 2] or nullptr
  uint8_t* hq_codes;         // NVFP4 row pass: h codes, block scales, globals
  uint8_t* hq_scales;
  float* hq_global;
  int withhold_arrivals;     // self-test: gate/up tiles never report, so down tiles time out
};

template <int FMT>
__global__ void __launch_bounds__(Cfg<FMT, true>::THREADS, 1)
    k_moe_ffn_decode(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmU,
                     const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ CUtensorMap tmH, const GemmArgs a1, const GemmArgs a2,
                     const FfnSync sy) {
  using C = Cfg<FMT, true>;
  using C2 = Cfg<FMT, false>;
  static_assert(C::STAGE_BYTES == C2::STAGE_BYTES && C::STAGES == C2::STAGES && C::SMEM == C2::SMEM &&
                    C::TMEM_COLS == C2::TMEM_COLS && C::THREADS == C2::THREADS,
                "gate/up and down tiles share one pipeline");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tmem_full = empty + C::STAGES;  // [2]
  uint64_t* tmem_empty = tmem_full + 2;     // [2]
  uint64_t* drain = tmem_empty + 2;
  uint64_t* sched_full = drain + 1;                  // [kSchedDepth] a tile index is in the ring
  uint64_t* sched_empty = sched_full + kSchedDepth;  // [kSchedDepth] the MMA and the epilogue have read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sched_empty + kSchedDepth);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;  // the epilogue's "this tile completed its row tile"
  volatile int* ring = last_flag + 1;        // [kSchedDepth] tile indices (-1: no more tiles)
  volatile int* ring_nv = ring + kSchedDepth;  // [kSchedDepth] their token rows (n_valid)
  static_assert(16 * C::STAGES + 8 * 5 + 16 * kSchedDepth + 4 * (3 + 2 * kSchedDepth) <= C::BAR_BYTES,
                "barrier area");
  int32_t* s_rtb = reinterpret_cast<int32_t*>(smem + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], C::EPI_WARPS);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      mbar_init(&sched_full[i], 1);
      mbar_init(&sched_empty[i], 2);  // the MMA thread and the epilogue
    }
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmG);
    prefetch_tmap(&tmU);
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmD);
    prefetch_tmap(&tmH);
  }
  // the tile plan is read before the dependency wait, as in k_moe_gemm
  for (int i = threadIdx.x; i <= a1.E; i += blockDim.x) s_rtb[i] = __ldcg(a1.rt_base + i);
  tc_fence_before();
  const bool plan_ok = plan_ok_sync(s_rtb, a1.E, a1.max_tiles);
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp != 0) pdl_wait();

  const int E = a1.E;
  const int MT1 = (a1.NA + C::ROWS - 1) / C::ROWS;    // gate/up tiles per row tile (F / 128)
  const int MT2 = (a2.NA + C2::ROWS - 1) / C2::ROWS;  // down tiles per row tile (H / 256)
  const int nrt = plan_ok ? s_rtb[E] : 0;
  const int total1 = nrt * MT1;
  const int total = total1 + nrt * MT2;
  const int KB1 = a1.K / C::ELEMS_PER_STAGE, KB2 = a2.K / C::ELEMS_PER_STAGE;
  const int64_t apr1 = (a1.K / C::BLOCK) / 4, apr2 = (a2.K / C::BLOCK) / 4;  // scale atoms per 128 rows
  uint32_t* status = a1.status;
  const long long limit = a1.limit;

  // tile t -> gate/up (g1) or down, weight block mt, row tile rti
  auto tile_of = [&](int t, bool& g1, int& mt, int& rti) {
    g1 = t < total1;
    if (g1) map_tile(t, MT1, s_rtb, E, mt, rti);
    else map_tile(t - total1, MT2, s_rtb, E, mt, rti);
  };
  // h rows of row tile rti ready for the down GEMM (acquire; relaxed: a hint)
  auto h_ready = [&](int rti) {
    return FMT == MOE_FMT_NVFP4 ? ld_acquire(sy.ready + rti) != 0 : ld_acquire(sy.done1 + rti) >= MT1;
  };
  auto h_ready_relaxed = [&](int rti) {
    return FMT == MOE_FMT_NVFP4 ? ld_relaxed(sy.ready + rti) != 0 : ld_relaxed(sy.done1 + rti) >= MT1;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      // A stage's weight part (both weight blocks and their scales) and its
      // token part (the tile's rows of x or h and their scales) complete the
      // same barrier; the token part of the first stages of a tile is held
      // back until the rows exist: for the first tile until the previous
      // kernel has finished, for a down tile until its row tile is ready.
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      bool prev_done = false;  // pdl_wait returned
      int held_stage[C::STAGES], held_kb[C::STAGES];
      // tiles are claimed one ahead: the next index is requested when a tile
      // starts, and its descriptor (and, for a down tile, a first look at its
      // row tile's flag) is read halfway through the tile, so that neither
      // the counter's round trip nor a global load sits between the last
      // stage of one tile and the first stage of the next
      // (a CTA that runs no tile, e.g. one whose plan failed its check in the
      // bounds-checked build, takes no index from the counter)
      int claimed = total > 0 ? atomicAdd(sy.next_tile, 1) : 0;
      bool c_have = false, c_g1 = false, c_ready = false;
      int c_mt = 0, c_rti = 0;
      RowTile c_rt{};
      auto fetch_claimed = [&]() {
        if (claimed < total) {
          tile_of(claimed, c_g1, c_mt, c_rti);
          c_rt = load_tile(a1.tiles + c_rti);
          // relaxed: a hint only; a tile found ready is acquired with a fence
          c_ready = !c_g1 && !sy.withhold_arrivals && h_ready_relaxed(c_rti);
        }
        c_have = true;
      };
      for (int i = 0; ok; ++i) {
        // pass the claimed tile on (the slot is free once the MMA and the
        // epilogue have read the index kSchedDepth tiles back)
        const int slot = i % kSchedDepth;
        if (!mbar_wait(&sched_empty[slot], ((i / kSchedDepth) & 1) ^ 1, abort_flag, status, ST_TIMEOUT_PRODUCER,
                       limit)) {
          ok = false;
          break;
        }
        if (!c_have) fetch_claimed();
        const int t = claimed < total ? claimed : -1;
        const bool g1 = c_g1;
        const int mt = c_mt, rti = c_rti;
        const RowTile rt = c_rt;
        ring[slot] = t;
        ring_nv[slot] = t >= 0 ? rt.n_valid : 0;
        mbar_arrive(&sched_full[slot]);
        if (t < 0) break;
        claimed = atomicAdd(sy.next_tile, 1);
        c_have = false;
        const GemmArgs& a = g1 ? a1 : a2;
        const CUtensorMap* mA0 = g1 ? &tmG : &tmD;
        const CUtensorMap* mA1 = g1 ? &tmU : &tmD;
        const CUtensorMap* mB = g1 ? &tmX : &tmH;
        const int rows = g1 ? C::ROWS : C2::ROWS;
        const int KB = g1 ? KB1 : KB2;
        const int64_t apr = g1 ? apr1 : apr2;
        const int N = (rt.n_valid + 15) & ~15;
        const int arow = rt.e * a.NA + mt * rows;
        // down: the second block of the last tile lies past the expert when
        // NA % 256 == 128; it then re-reads the first block and the epilogue
        // drops its results
        const bool second = g1 || (mt * rows + 128 < a.NA);
        const int arow1 = (g1 || !second) ? arow : arow + 128;
        const uint8_t* sfa0 = a.sfA0 + (int64_t)(arow >> 7) * apr * 512;
        const uint8_t* sfa1 = a.sfA1 + (int64_t)(arow1 >> 7) * apr * 512;
        const uint8_t* sfb = a.sfB + (int64_t)(rt.row / C::NT) * apr * 512;
        const uint32_t bytes = C::NA * C::A_BYTES + N * 128 + (C::NA + 1) * C::SF_BYTES;
        bool tok = g1 ? prev_done : c_ready;  // may the token part go out now
        if (!g1 && tok) {
          fence_acquire_gpu();  // with the relaxed read of the flag: an acquire
          fence_proxy_async_global();
        }
        int nh = 0;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, status, ST_TIMEOUT_PRODUCER, limit)) {
            ok = false;
            break;
          }
          uint8_t* sbase = smem + stage * C::STAGE_BYTES;
          uint8_t* sB = sbase + C::NA * C::A_BYTES;
          uint8_t* sSF = sB + C::B_BYTES;
          if (a1.withhold_loads) {  // bounded-wait self-test: nothing arrives
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          mbar_expect_tx(&full[stage], bytes);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          tma_load_2d(sbase, mA0, &full[stage], kb * 128, arow);
          tma_load_2d(sbase + C::A_BYTES, mA1, &full[stage], kb * 128, arow1);
          bulk_load(sSF, sfa0 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
          bulk_load(sSF + C::SF_BYTES, sfa1 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
          held_stage[nh] = stage;
          held_kb[nh] = kb;
          ++nh;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (!tok && (nh == C::STAGES || kb == KB - 1)) {
            // the pipeline is full of weight parts: now the rows must exist
            if (g1) {
              pdl_wait();
              prev_done = true;
            } else {
              const long long t0 = clock64();
              while (!(!sy.withhold_arrivals && h_ready(rti))) {
                if (*abort_flag || clock64() - t0 > limit) {
                  if (!*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(status, ST_TIMEOUT_DEPEND);
                  }
                  ok = false;
                  break;
                }
              }
              if (!ok) break;
              fence_proxy_async_global();
            }
            tok = true;
          }
          if (tok) {
            for (int i = 0; i < nh; ++i) {
              uint8_t* hB = smem + held_stage[i] * C::STAGE_BYTES + C::NA * C::A_BYTES;
              for (int r = 0; r < N / 16; ++r)
                tma_load_2d(hB + r * 2048, mB, &full[held_stage[i]], held_kb[i] * 128, rt.row + 16 * r);
              bulk_load(hB + C::B_BYTES + C::NA * C::SF_BYTES, sfb + (int64_t)held_kb[i] * C::SF_BYTES,
                        C::SF_BYTES, &full[held_stage[i]]);
            }
            nh = 0;
          }
          if (!c_have && kb == KB / 2) fetch_claimed();
        }
      }
      if (!prev_done) pdl_wait();
      if (!ok) {
        // wait (bounded) for the copies this thread put in flight
        for (int s = 0; s < C::STAGES; ++s) {
          if (!((armed >> s) & 1u)) continue;
          const uint32_t par = (armed_par >> s) & 1u;
          const long long t0 = clock64();
          while (!mbar_try_wait(&full[s], par) && clock64() - t0 < limit) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer (as in k_moe_gemm) ----------------
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int slot = it % kSchedDepth;
        if (!mbar_wait(&sched_full[slot], (it / kSchedDepth) & 1, abort_flag, status, ST_TIMEOUT_MMA, limit)) {
          ok = false;
          break;
        }
        const int t = ring[slot];
        const int nv = ring_nv[slot];
        mbar_arrive(&sched_empty[slot]);
        if (t < 0) break;
        bool g1;
        int mt, rti;
        tile_of(t, g1, mt, rti);
        const uint32_t N = (uint32_t)((nv + 15) & ~15);
        const int KB = g1 ? KB1 : KB2;
        const int buf = it % C::ACC_BUFS;
        const uint32_t use = (uint32_t)(it / C::ACC_BUFS) & 1u;
        if (!mbar_wait(&tmem_empty[buf], use ^ 1, abort_flag, status, ST_TIMEOUT_MMA, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc0 = tmem + buf * C::ACC_BUF;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, status, ST_TIMEOUT_MMA, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* sbase = smem + stage * C::STAGE_BYTES;
          uint8_t* sB = sbase + C::NA * C::A_BYTES;
          uint8_t* sSF = sB + C::B_BYTES;
          const uint32_t sf_t = tmem + C::TMEM_SF + stage * C::SF_COLS_STAGE;
#pragma unroll
          for (int op = 0; op < C::NA + 1; ++op)
#pragma unroll
            for (int at = 0; at < C::SF_ATOMS; ++at)
              tc_cp_32x128b_x4(sf_t + op * C::SF_COLS_OP + at * 4,
                               sdesc_atom(smem_u32(sSF + op * C::SF_BYTES + at * 512)));
          const uint64_t da0 = sdesc_sw128(smem_u32(sbase));
          const uint64_t da1 = sdesc_sw128(smem_u32(sbase + C::A_BYTES));
          const uint64_t db = sdesc_sw128(smem_u32(sB));
          const uint32_t sfb_t = sf_t + C::NA * C::SF_COLS_OP;
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t accum = (kb | s) != 0;
            const uint64_t koff = (uint64_t)((s * 32) >> 4);
            if constexpr (FMT == MOE_FMT_NVFP4) {
              const uint32_t id = idesc_nvfp4(N);
              mma_nvfp4(acc0, da0 + koff, db + koff, id, sf_t + 4 * s, sfb_t + 4 * s, accum);
              mma_nvfp4(acc0 + C::ACC_COLS, da1 + koff, db + koff, id, sf_t + C::SF_COLS_OP + 4 * s, sfb_t + 4 * s,
                        accum);
            } else {
              const uint32_t id = idesc_mxfp8(N, (uint32_t)s);
              mma_mxfp8(acc0, da0 + koff, db + koff, id, sf_t, sfb_t, accum);
              mma_mxfp8(acc0 + C::ACC_COLS, da1 + koff, db + koff, id, sf_t + C::SF_COLS_OP, sfb_t, accum);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tmem_full[buf]);
      }
      tc_commit(drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(drain, 0) && clock64() - t0 < limit) {
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    // Warp (4 + q) reads TMEM lane quadrant q (its 32 output features) for the
    // tile's up to 64 token columns, as in k_moe_gemm.  The four warps agree
    // on every step that needs all of them (named barrier 1), so none is left
    // waiting for another that gave up.
    const int q = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    const bool capped = a1.cap > 0.0f;
    for (int it = 0;; ++it) {
      const int slot = it % kSchedDepth;
      const bool got = __all_sync(0xffffffffu, mbar_wait(&sched_full[slot], (it / kSchedDepth) & 1, abort_flag,
                                                         status, ST_TIMEOUT_EPILOGUE, limit));
      const int t = ring[slot];
      // the four warps agree, then the slot is released once for all of them
      if (!epi_all(got)) break;
      if (threadIdx.x == 128) mbar_arrive(&sched_empty[slot]);
      if (t < 0) break;
      bool g1;
      int mt, rti;
      tile_of(t, g1, mt, rti);
      const GemmArgs& a = g1 ? a1 : a2;
      const RowTile rt = a.tiles[rti];
      const int rows = g1 ? C::ROWS : C2::ROWS;
      const int f = mt * rows + q * 32 + lane;  // feature of accumulator 0 (down: +128 for 1)
      const bool second = g1 || (mt * rows + 128 < a.NA);
      const int col_hi = min(rt.n_valid, 64);
      const int buf = it % C::ACC_BUFS;
      const uint32_t use = (uint32_t)(it / C::ACC_BUFS) & 1u;
      const bool waited = __all_sync(0xffffffffu, mbar_wait(&tmem_full[buf], use, abort_flag, status,
                                                            ST_TIMEOUT_EPILOGUE, limit));
      if (!epi_all(waited)) break;
      tc_fence_after();
      float sA0 = 1.0f, sA1 = 1.0f, gb_lo = 1.0f, gb_hi = 1.0f;
      if constexpr (FMT == MOE_FMT_NVFP4) {
        // the h globals of a down tile were published with its row tile
        // (its MMAs ran on them, so the flag is set): acquire it first
        if (!g1) (void)ld_acquire(sy.ready + rti);
        sA0 = a.gA0[rt.e];
        sA1 = a.gA1[rt.e];
        if (lane < col_hi) gb_lo = a.gB[rt.row + lane];
        if (32 + lane < col_hi) gb_hi = a.gB[rt.row + 32 + lane];
      }
      const uint32_t tacc = tq + buf * C::ACC_BUF;
      uint32_t r0[4][16], r1[4][16];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if (ch * 16 < col_hi) {
          tmem_ld16(tacc + ch * 16, r0[ch]);
          tmem_ld16(tacc + C::ACC_COLS + ch * 16, r1[ch]);
        }
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[buf]);
      if (g1) {
        // h = bf16(silu(cap g) cap u); MXFP8: its codes and block scale (the
        // warp's 32 lanes are one 32-feature block of a token row); NVFP4:
        // the bf16 h, quantised by the row pass below
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          if (ch * 16 >= col_hi) break;
          const float gbv = ch < 2 ? gb_lo : gb_hi;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = ch * 16 + j;
            const bool valid = n < col_hi;  // warp-uniform
            float gb = 1.0f;
            if constexpr (FMT == MOE_FMT_NVFP4) gb = __shfl_sync(0xffffffffu, gbv, (ch * 16 + j) & 31);
            const int64_t row = (int64_t)rt.row + n;
            float g = __uint_as_float(r0[0][j]) * (sA0 * gb);
            float u = __uint_as_float(r1[0][j]) * (sA1 * gb);
            g = capped ? cap_soft(g, a1.cap, a1.inv_cap) : g;
            u = capped ? cap_soft(u, a1.cap, a1.inv_cap) : u;
            const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * u);
            if constexpr (FMT == MOE_FMT_MXFP8) {
              const float v = __bfloat162float(hb);
              const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
              const uint32_t sc = m != 0.0f ? mx_scale_code(m, a1.mx_mode) : 0u;
              const uint32_t code = m != 0.0f ? e4m3_encode(__fmul_rn(v, exp2i(127 - (int)sc))) : 0u;
              const bool ok = valid && MOE_IN_BOUNDS(row < a1.R);
              if (ok) a1.hq_codes[row * a1.NA + f] = (uint8_t)code;
              if (ok && lane == 0) a1.hq_scales[act_scale_offset(row, f >> 5, a1.NA >> 5, C::NT)] = (uint8_t)sc;
            } else {
              const bool ok = valid && MOE_IN_BOUNDS(row < a1.R);
              if (ok) a1.h_out[row * a1.NA + f] = hb;
              // the row's |h| maximum over this warp's 32 features, for the
              // row pass (non-negative floats order like their bits)
              const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(__bfloat162float(hb))));
              if (ok && lane == 0 && !sy.act_static) atomicMax(sy.h_amax + row, m);
            }
          }
          // the next chunk moves to the front (register moves, no indexing)
#pragma unroll
          for (int i = 0; i < 3; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              r0[i][j] = r0[i + 1][j];
              r1[i][j] = r1[i + 1][j];
            }
        }
        // this tile's h is stored by all four warps: count it for its row tile
        epi_sync();
        if (threadIdx.x == 128) {
          int last = 0;
          if (!sy.withhold_arrivals) {
            __threadfence();
            fence_proxy_async_global();
            last = atomicAdd(sy.done1 + rti, 1) == MT1 - 1;
          }
          *last_flag = last;
        }
        epi_sync();
        if (FMT == MOE_FMT_NVFP4 && *last_flag) {
          // the row tile's h is complete: quantise its rows, the 128 threads
          // taking (row, 16-block) pairs, each row's global from its maximum
          // gathered above (or the expert's static global), the steps of the
          // row pass; then publish the row tile
          __threadfence();
          const bool stat = sy.act_static != nullptr;
          const float sg = stat ? sy.act_static[2 * rt.e + 1] : 0.0f;
          const int nb = a1.NA / 16;
          const int64_t cbytes = a1.NA / 2;
          for (int idx = threadIdx.x - 128; idx < rt.n_valid * nb; idx += 128) {
            const int n = idx / nb, b = idx - n * nb;
            const int64_t row = (int64_t)rt.row + n;
            if (!MOE_IN_BOUNDS(row < a1.R)) continue;
            const float G = stat ? __fdiv_rn(1.0f, sg) : nvfp4_G(__uint_as_float(__ldcg(sy.h_amax + row)));
            if (b == 0) sy.hq_global[row] = stat ? sg : __fdiv_rn(1.0f, G);
            float v[16];
            const uint4* src = reinterpret_cast<const uint4*>(a1.h_out + row * a1.NA + b * 16);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const uint4 u = __ldcg(src + i);
              const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
              }
            }
            uint2 c;
            const uint32_t sc = nvfp4_block(v, G, &c);
            *reinterpret_cast<uint2*>(sy.hq_codes + row * cbytes + (int64_t)b * 8) = c;
            sy.hq_scales[act_scale_offset(row, b, nb, C::NT)] = (uint8_t)sc;
          }
          epi_sync();
          if (threadIdx.x == 128) {
            __threadfence();
            fence_proxy_async_global();
            st_release(sy.ready + rti, 1);
          }
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          if (ch * 16 >= col_hi) continue;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = ch * 16 + j;
            const float gb = __shfl_sync(0xffffffffu, ch < 2 ? gb_lo : gb_hi, (ch * 16 + j) & 31);
            if (n >= col_hi) continue;  // warp-uniform
            const float v0 = __uint_as_float(r0[ch][j]) * (sA0 * gb);
            const float v1 = __uint_as_float(r1[ch][j]) * (sA1 * gb);
            const bool ok = MOE_IN_BOUNDS(rt.canon + n < a2.P);
            const int64_t prow = (int64_t)rt.canon + n;
            if (a2.y16) {
              // the warp's 32 lanes are one 32-feature exponent block
              int e0, e1 = 0;
              const uint16_t c0 = y16_lane_code(v0, e0);
              const uint16_t c1 = second ? y16_lane_code(v1, e1) : (uint16_t)0;
              if (ok) {
                uint16_t* yrow = reinterpret_cast<uint16_t*>(a2.y_out) + prow * a2.NA;
                int8_t* erow = a2.y_exp + prow * (a2.NA >> 5);
                yrow[f] = c0;
                if (lane == 0) erow[f >> 5] = (int8_t)e0;
                if (second) {
                  yrow[f + 128] = c1;
                  if (lane == 0) erow[(f + 128) >> 5] = (int8_t)e1;
                }
              }
            } else if (ok) {
              float* yrow = reinterpret_cast<float*>(a2.y_out) + prow * a2.NA;
              yrow[f] = v0;
              if (second) yrow[f + 128] = v1;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  pdl_trigger();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int FMT>
cudaError_t launch_ffn_decode_t(const GemmLaunch& g1, const GemmLaunch& g2, const FfnSync& sy,
                                const CUtensorMap* tmH, cudaStream_t st, bool pdl) {
  using C = Cfg<FMT, true>;
  static PerDeviceOnce attr;
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(k_moe_ffn_decode<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (e != cudaSuccess) return e;
  const GemmArgs a1 = gemm_args(g1), a2 = gemm_args(g2);
  // one CTA per SM; tiles are taken on demand, so no co-residency is assumed
  return launch_k(k_moe_ffn_decode<FMT>, dim3(g1.num_sms), dim3(C::THREADS), C::SMEM, st, pdl, *g1.tmA0, *g1.tmA1,
                  *g1.tmB, *g2.tmA0, *tmH, a1, a2, sy);
}

}  // namespace

cudaError_t launch_ffn_decode(const GemmLaunch& g1, const GemmLaunch& g2, int32_t* sync, const float* act_static,
                              uint8_t* hq_codes, uint8_t* hq_scales, float* hq_global, int withhold_arrivals,
                              cudaStream_t st, bool pdl) {
  const int64_t nt = max_row_tiles(*g1.cfg);
  const FfnSync sy{sync,     sync + nt,  sync + 2 * nt, reinterpret_cast<uint32_t*>(sync + 2 * nt + 1),
                   act_static, hq_codes, hq_scales,     hq_global,
                   withhold_arrivals};
  if (g1.cfg->fmt == MOE_FMT_NVFP4) return launch_ffn_decode_t<MOE_FMT_NVFP4>(g1, g2, sy, g2.tmB, st, pdl);
  return launch_ffn_decode_t<MOE_FMT_MXFP8>(g1, g2, sy, g2.tmB, st, pdl);
}

}  // namespace moe
