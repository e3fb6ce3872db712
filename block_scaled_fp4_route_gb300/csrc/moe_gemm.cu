// Persistent grouped expert GEMM on block-scaled tensor cores (tcgen05).
//
// TokenSpeed page on Inkling 2 Small (section on serving on NVIDIA
// Blackwell): the expert GEMMs run directly on block-scaled tensor cores.
// Cookbook page, MegaMoE paragraph: the two expert GEMMs with the capped
// SwiGLU between them.  Both formats of the checkpoint are covered: NVFP4
// (kind::mxf4nvf4, E2M1 x E2M1 with UE4M3 scales per 16) and MXFP8
// (kind::mxf8f6f4, E4M3 x E4M3 with UE8M0 scales per 32).
//
// Two tile shapes, both persistent and warp-specialised (warp 0 = TMA
// producer, warp 1 = MMA issuer, warp 2 = TMEM allocator, the rest epilogue;
// an epilogue warp w reads TMEM lane quadrant w % 4):
//
// Decode batches (64-row token tiles, k_moe_gemm), "swap-AB": two 128-row
// weight blocks fill M (two MMAs sharing the token operand) and up to 64
// token rows of one expert fill N (rounded up to 16), so a batch with one or
// two tokens per expert wastes no weight bytes; each stage carries 32 KB of
// weights; the TMEM accumulators are double-buffered (the epilogue of one
// tile runs while the next accumulates).
//   GEMM1 (gated):  A0 = 128 W_gate rows, A1 = the same 128 W_up rows,
//                   epilogue h = bf16(silu(cap g) * cap u); for MXFP8 the
//                   epilogue also quantises h (a warp holds one 32-feature
//                   block of a token row); NVFP4 h goes to a row pass (its
//                   global spans the row)
//   GEMM2:          A0, A1 = 256 consecutive W_down rows,
//                   epilogue y = acc * g_w * g_h (fp32)
//
// Prefill batches (128-row token tiles, k_moe_gemm_tm), token-major: the 128
// token rows fill M and the two weight blocks one N = 256 operand (see there).
//
// Tiles are walked expert by expert, then weight-row block, then token block,
// so CTAs running side by side share an expert's weights and activations in
// L2.
// Every mbarrier wait is bounded; a wait that runs out sets a status bit in
// global memory, every role leaves its loop, the producer waits for its own
// copies in flight, the MMA thread for its tcgen05 operations, and the CTA
// frees its TMEM.
#include "moe_gemm_common.cuh"

namespace moe {

namespace {

template <int FMT, bool GATED>
__global__ void __launch_bounds__(Cfg<FMT, GATED>::THREADS, 1)
    k_moe_gemm(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
               const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
  using C = Cfg<FMT, GATED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tmem_full = empty + C::STAGES;  // [2]
  uint64_t* tmem_empty = tmem_full + 2;     // [2]
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
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
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmA0);
    prefetch_tmap(&tmA1);
    prefetch_tmap(&tmB);
  }
  // The tile plan was written by the dispatch, which had completed before
  // the previous kernel's threads passed their own dependency wait, and this
  // grid starts only after all of them have: it is read now (through L2).
  // What the previous kernel writes is read only after pdl_wait; the
  // producer waits after it has requested its first weight stages.
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_rtb[i] = __ldcg(a.rt_base + i);
  tc_fence_before();
  const bool plan_ok = plan_ok_sync(s_rtb, a.E, a.max_tiles);
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // warp 0 stays out: a wait taken by some of its lanes would hold the
  // producer lane too (its other lanes read nothing the previous kernel wrote)
  if (warp != 0) pdl_wait();

  const int MT = (a.NA + C::ROWS - 1) / C::ROWS;
  const int total = plan_ok ? s_rtb[a.E] * MT : 0;
  const int KB = a.K / C::ELEMS_PER_STAGE;
  const int64_t atoms_per_row = (a.K / C::BLOCK) / 4;  // scale atoms per 128 weight rows or per token tile

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;  // per stage: armed at least once / parity of last arming
      bool ok = true;
      // the next tile's descriptor is fetched one tile ahead, so no global
      // load sits between the last stage of a tile and the first of the next
      int mt = 0, rti = 0;
      RowTile rt{};
      if (blockIdx.x < total) {
        map_tile(blockIdx.x, MT, s_rtb, a.E, mt, rti);
        rt = load_tile(a.tiles + rti);
      }
      // The first tile's weight blocks and their scales for the first stages
      // do not depend on the previous kernel: requested before the wait, they
      // stream while it finishes.
      const int pre = (blockIdx.x < total && !a.withhold_loads) ? min(KB, C::STAGES) : 0;
      if (pre > 0) {
        const int N = (rt.n_valid + 15) & ~15;
        const int arow = rt.e * a.NA + mt * C::ROWS;
        const bool second = GATED || (mt * C::ROWS + 128 < a.NA);
        const int arow1 = (GATED || !second) ? arow : arow + 128;
        const uint8_t* sfa0 = a.sfA0 + (int64_t)(arow >> 7) * atoms_per_row * 512;
        const uint8_t* sfa1 = a.sfA1 + (int64_t)(arow1 >> 7) * atoms_per_row * 512;
        const uint32_t bytes = C::NA * C::A_BYTES + N * 128 + (C::NA + 1) * C::SF_BYTES;
#pragma unroll 1
        for (int kb = 0; kb < pre; ++kb) {  // fresh stages, phase 0
          uint8_t* sbase = smem + kb * C::STAGE_BYTES;
          uint8_t* sSF = sbase + C::NA * C::A_BYTES + C::B_BYTES;
          mbar_expect_tx(&full[kb], bytes);
          armed |= 1u << kb;
          tma_load_2d(sbase, &tmA0, &full[kb], kb * 128, arow);
          tma_load_2d(sbase + C::A_BYTES, &tmA1, &full[kb], kb * 128, arow1);
          bulk_load(sSF, sfa0 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[kb]);
          bulk_load(sSF + C::SF_BYTES, sfa1 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[kb]);
        }
      }
      pdl_wait();
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        int mt_n = 0, rti_n = 0;
        RowTile rt_n{};
        if (t + (int)gridDim.x < total) {
          map_tile(t + gridDim.x, MT, s_rtb, a.E, mt_n, rti_n);
          rt_n = load_tile(a.tiles + rti_n);
        }
        const int N = (rt.n_valid + 15) & ~15;
        const int arow = rt.e * a.NA + mt * C::ROWS;
        // down: the second block of the last tile lies past the expert when
        // NA % 256 == 128; it then re-reads the first block (never past the
        // scale buffer) and the epilogue drops its results
        const bool second = GATED || (mt * C::ROWS + 128 < a.NA);
        const int arow1 = (GATED || !second) ? arow : arow + 128;
        const uint8_t* sfa0 = a.sfA0 + (int64_t)(arow >> 7) * atoms_per_row * 512;
        const uint8_t* sfa1 = a.sfA1 + (int64_t)(arow1 >> 7) * atoms_per_row * 512;
        const uint8_t* sfb = a.sfB + (int64_t)(rt.row / C::NT) * atoms_per_row * 512;
        const uint32_t bytes = C::NA * C::A_BYTES + N * 128 + (C::NA + 1) * C::SF_BYTES;
        const bool first = t == (int)blockIdx.x;
        for (int kb = 0; kb < KB; ++kb) {
          if (first && kb < pre) {  // weights requested before the wait: now the token rows and scales
            uint8_t* sB = smem + stage * C::STAGE_BYTES + C::NA * C::A_BYTES;
            uint8_t* sSF = sB + C::B_BYTES;
            for (int i = 0; i < N / 16; ++i) tma_load_2d(sB + i * 2048, &tmB, &full[stage], kb * 128, rt.row + 16 * i);
            bulk_load(sSF + C::NA * C::SF_BYTES, sfb + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.status, ST_TIMEOUT_PRODUCER, a.limit)) {
            ok = false;
            break;
          }
          uint8_t* sbase = smem + stage * C::STAGE_BYTES;
          uint8_t* sB = sbase + C::NA * C::A_BYTES;
          uint8_t* sSF = sB + C::B_BYTES;
          if (a.withhold_loads) {  // bounded-wait self-test: nothing arrives
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          mbar_expect_tx(&full[stage], bytes);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          tma_load_2d(sbase, &tmA0, &full[stage], kb * 128, arow);
          tma_load_2d(sbase + C::A_BYTES, &tmA1, &full[stage], kb * 128, arow1);
          // 16-row boxes, only the rows the tile holds
          for (int i = 0; i < N / 16; ++i) tma_load_2d(sB + i * 2048, &tmB, &full[stage], kb * 128, rt.row + 16 * i);
          bulk_load(sSF, sfa0 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
          bulk_load(sSF + C::SF_BYTES, sfa1 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
          bulk_load(sSF + C::NA * C::SF_BYTES, sfb + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        mt = mt_n;
        rt = rt_n;
      }
      if (!ok) {
        // wait (bounded) for the copies this thread put in flight
        for (int s = 0; s < C::STAGES; ++s) {
          if (!((armed >> s) & 1u)) continue;
          uint32_t par = (armed_par >> s) & 1u;
          long long t0 = clock64();
          while (!mbar_try_wait(&full[s], par) && clock64() - t0 < a.limit) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      int nv_next = 0;
      if (blockIdx.x < total) {
        int mt0, rti0;
        map_tile(blockIdx.x, MT, s_rtb, a.E, mt0, rti0);
        nv_next = a.tiles[rti0].n_valid;
      }
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++it) {
        const uint32_t N = (uint32_t)((nv_next + 15) & ~15);
        if (t + (int)gridDim.x < total) {  // fetched one tile ahead
          int mt_n, rti_n;
          map_tile(t + gridDim.x, MT, s_rtb, a.E, mt_n, rti_n);
          nv_next = a.tiles[rti_n].n_valid;
        }
        const int buf = it % C::ACC_BUFS;
        const uint32_t use = (uint32_t)(it / C::ACC_BUFS) & 1u;
        if (!mbar_wait(&tmem_empty[buf], use ^ 1, abort_flag, a.status, ST_TIMEOUT_MMA, a.limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc0 = tmem + buf * C::ACC_BUF;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.status, ST_TIMEOUT_MMA, a.limit)) {
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
      // every tcgen05 operation of this thread has completed before TMEM is freed
      tc_commit(drain);
      long long t0 = clock64();
      while (!mbar_try_wait(drain, 0) && clock64() - t0 < a.limit) {
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    // Warp (4 + i) reads TMEM lane quadrant i (its 32 output features) for
    // the tile's up to 64 token columns: the whole share goes to registers
    // first, the accumulator buffer is released, then the arithmetic and
    // stores run.
    const int q = warp & 3;
    constexpr int col_lo = 0;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      int mt, rti;
      map_tile(t, MT, s_rtb, a.E, mt, rti);
      const RowTile rt = a.tiles[rti];
      const int f = mt * C::ROWS + q * 32 + lane;       // feature of accumulator 0 (down: +128 for 1)
      const bool second = GATED || (mt * C::ROWS + 128 < a.NA);
      const int col_hi = min(rt.n_valid, col_lo + 64);
      float sA0 = 1.0f, sA1 = 1.0f, gb_lo = 1.0f, gb_hi = 1.0f;
      if constexpr (FMT == MOE_FMT_NVFP4) {
        sA0 = a.gA0[rt.e];
        sA1 = a.gA1[rt.e];
        if (col_lo + lane < col_hi) gb_lo = a.gB[rt.row + col_lo + lane];
        if (col_lo + 32 + lane < col_hi) gb_hi = a.gB[rt.row + col_lo + 32 + lane];
      }
      const int buf = it % C::ACC_BUFS;
      const uint32_t use = (uint32_t)(it / C::ACC_BUFS) & 1u;
      // the warp leaves together: tcgen05.ld and the shuffles below need all lanes
      if (!__all_sync(0xffffffffu, mbar_wait(&tmem_full[buf], use, abort_flag, a.status, ST_TIMEOUT_EPILOGUE,
                                             a.limit)))
        break;
      tc_fence_after();
      const uint32_t tacc = tq + buf * C::ACC_BUF;
      // one 16-column chunk of the gated epilogue: h = bf16(silu(cap g) cap u),
      // then (MXFP8, 64-row tiles) its codes and block scale, else the bf16 h.  Every element
      // of the chunk is computed (columns past n_valid hold stale accumulators
      // and are only discarded), so the 16 elements are straight-line code;
      // only the stores are predicated.
      auto gated_chunk = [&](const uint32_t (&c0)[16], const uint32_t (&c1)[16], int ch) {
        const float gbv = ch < 2 ? gb_lo : gb_hi;
        const bool capped = a.cap > 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = col_lo + ch * 16 + j;
          const bool valid = n < col_hi;  // warp-uniform
          float gb = 1.0f;
          if constexpr (FMT == MOE_FMT_NVFP4) gb = __shfl_sync(0xffffffffu, gbv, (ch * 16 + j) & 31);
          const int64_t row = (int64_t)rt.row + n;
          float g = __uint_as_float(c0[j]) * (sA0 * gb);
          float u = __uint_as_float(c1[j]) * (sA1 * gb);
          g = capped ? cap_soft(g, a.cap, a.inv_cap) : g;
          u = capped ? cap_soft(u, a.cap, a.inv_cap) : u;
          const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * u);
          if constexpr (FMT == MOE_FMT_MXFP8) {
            // the warp's 32 lanes are one 32-feature block of this token
            // row; |v| orders like its bit pattern
            const float v = __bfloat162float(hb);
            const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
            const uint32_t sc = m != 0.0f ? mx_scale_code(m, a.mx_mode) : 0u;
            const uint32_t code = m != 0.0f ? e4m3_encode(__fmul_rn(v, exp2i(127 - (int)sc))) : 0u;
            const bool ok = valid && MOE_IN_BOUNDS(row < a.R);
            if (ok) a.hq_codes[row * a.NA + f] = (uint8_t)code;
            if (ok && lane == 0) a.hq_scales[act_scale_offset(row, f >> 5, a.NA >> 5, C::NT)] = (uint8_t)sc;
          } else {
            if (valid && MOE_IN_BOUNDS(row < a.R)) a.h_out[row * a.NA + f] = hb;
          }
        }
      };
      uint32_t r0[4][16], r1[4][16];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if (col_lo + ch * 16 < col_hi) {
          tmem_ld16(tacc + col_lo + ch * 16, r0[ch]);
          tmem_ld16(tacc + C::ACC_COLS + col_lo + ch * 16, r1[ch]);
        }
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[buf]);
      if constexpr (GATED) {
        // The gated element is long (soft cap, SwiGLU, MXFP8 quantisation), so
        // only one 16-column chunk is unrolled (the chunks rotate through
        // r0[0] / r1[0]): a fully unrolled epilogue no longer fits the
        // instruction cache beside the producer and MMA loops.
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          if (col_lo + ch * 16 >= col_hi) break;
          gated_chunk(r0[0], r1[0], ch);
          // the next chunk moves to the front (register moves, no indexing)
#pragma unroll
          for (int i = 0; i < 3; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              r0[i][j] = r0[i + 1][j];
              r1[i][j] = r1[i + 1][j];
            }
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          if (col_lo + ch * 16 >= col_hi) continue;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = col_lo + ch * 16 + j;
            const float gb = __shfl_sync(0xffffffffu, ch < 2 ? gb_lo : gb_hi, (ch * 16 + j) & 31);
            if (n >= col_hi) continue;  // warp-uniform
            const float v0 = __uint_as_float(r0[ch][j]) * (sA0 * gb);
            const float v1 = __uint_as_float(r1[ch][j]) * (sA1 * gb);
            const bool ok = MOE_IN_BOUNDS(rt.canon + n < a.P);
            const int64_t prow = (int64_t)rt.canon + n;
            if (a.y16) {
              // the warp's 32 lanes are one 32-feature exponent block
              int e0, e1 = 0;
              const uint16_t c0 = y16_lane_code(v0, e0);
              const uint16_t c1 = second ? y16_lane_code(v1, e1) : (uint16_t)0;
              if (ok) {
                uint16_t* yrow = reinterpret_cast<uint16_t*>(a.y_out) + prow * a.NA;
                int8_t* erow = a.y_exp + prow * (a.NA >> 5);
                yrow[f] = c0;
                if (lane == 0) erow[f >> 5] = (int8_t)e0;
                if (second) {
                  yrow[f + 128] = c1;
                  if (lane == 0) erow[(f + 128) >> 5] = (int8_t)e1;
                }
              }
            } else if (ok) {
              float* yrow = reinterpret_cast<float*>(a.y_out) + prow * a.NA;
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

template <int FMT, bool GATED>
cudaError_t launch_t(const GemmLaunch& g, cudaStream_t st, bool pdl) {
  using C = Cfg<FMT, GATED>;
  static PerDeviceOnce attr;
  cudaError_t e = once_per_device(
      attr, [] { return cudaFuncSetAttribute(k_moe_gemm<FMT, GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM); });
  if (e != cudaSuccess) return e;
  const GemmArgs a = gemm_args(g);
  return launch_k(k_moe_gemm<FMT, GATED>, dim3(g.num_sms), dim3(C::THREADS), C::SMEM, st, pdl, *g.tmA0, *g.tmA1,
                  *g.tmB, a);
}

// ---------------------------------------------------------------------------
// Wide tiles, token-major.  For prefill batches the token rows of an expert
// fill the MMA's M = 128 and the tile's two 128-row weight blocks (gate and up
// rows of the same 128 features, or 256 consecutive W_down rows) form one
// N = 256 operand, so each k-step is one 128 x 256 MMA: the token operand is
// read from shared memory once instead of once per weight block, half as many
// MMAs are issued, and a thread of the epilogue (TMEM lane = token) holds the
// gate and up values of the same features side by side.
// ---------------------------------------------------------------------------
// 32 x 32 transpose across a warp, values v[0..15] = lo, v[16..31] = hi: on
// entry lane L holds row L (v[j] = M[L][j]), on exit column L (v[i] = M[i][L]).
// Five rounds; in the round of bit m, lanes L and L ^ m swap the elements
// whose index bit m differs from their lane bit m.
__device__ __forceinline__ void warp_transpose32(uint32_t (&lo)[16], uint32_t (&hi)[16], int lane) {
#pragma unroll
  for (int k = 4; k >= 0; --k) {
    const int m = 1 << k;
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i & m) continue;
      uint32_t& a = i < 16 ? lo[i & 15] : hi[i & 15];
      uint32_t& b = (i | m) < 16 ? lo[(i | m) & 15] : hi[(i | m) & 15];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, up ? a : b, m);
      if (up) a = recv;
      else b = recv;
    }
  }
}

// After warp_transpose32: row i of the 32-row group at base + i * stride,
// lane L writing element L (128 contiguous bytes per instruction); rows at or
// past nv are skipped (warp-uniform).
__device__ __forceinline__ void store_rows32(float* base, int stride, int nv, const uint32_t (&lo)[16],
                                             const uint32_t (&hi)[16]) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < nv) base[(int64_t)i * stride] = __uint_as_float(i < 16 ? lo[i] : hi[i - 16]);
}

// 4 x 4 transpose of 16-byte chunks within each group of four lanes: on
// entry lane 4g + j holds chunks 0..3 of its row (v[4c .. 4c + 3] = chunk c),
// on exit chunk j of rows 4g .. 4g + 3 (v[4r .. 4r + 3] = chunk j of row
// 4g + r).  Two rounds, as in warp_transpose32, four words per chunk.
__device__ __forceinline__ void quad_transpose4x4(uint32_t (&v)[16], int lane) {
#pragma unroll
  for (int m = 2; m >= 1; m >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c & m) continue;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t& a = v[4 * c + w];
        uint32_t& b = v[4 * (c | m) + w];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, up ? a : b, m);
        if (up) a = recv;
        else b = recv;
      }
    }
  }
}

// Token-major epilogue after the TMEM copy: r0 / r1 hold this thread's 64
// columns of weight block 0 / 1 (token row n of the tile, features
// 64 hc .. 64 hc + 63 of each block); s0 / s1 the global scales.  Gated:
// capped SwiGLU, bf16 h (MXFP8: quantised here); down: y rows, transposed
// across the warp so that each store writes 128 contiguous bytes.
template <int FMT, bool GATED>
__device__ __forceinline__ void tm_epilogue_math(const GemmArgs& a, uint32_t (&r0)[4][16], uint32_t (&r1)[4][16],
                                                 const RowTile& rt, int mt, int n, bool valid, int q, int hc,
                                                 int lane, float s0, float s1) {
  constexpr int ROWS = GATED ? 128 : 256;
  constexpr int NT = kNTWide;
  const bool second = GATED || (mt * ROWS + 128 < a.NA);
  // every lane stays on the same path below (the down epilogue shuffles
  // across the warp); lanes past n_valid only skip their stores
  if constexpr (GATED) {
    if (!valid) return;  // no warp-collective operation in the gated epilogue
    const bool capped = a.cap > 0.0f;
    const int64_t row = (int64_t)rt.row + n;
    if (!MOE_IN_BOUNDS(row < a.R)) return;
    const int f0 = mt * ROWS + 64 * hc;  // first feature of this thread's share
    // two 32-feature blocks (one MXFP8 scale block each), one unrolled
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      uint32_t pk[16];  // 32 bf16 h values
      float mh = 0.0f;  // their largest |h| before the bf16 rounding
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int c = j >> 4, jj = j & 15;
        // MXFP8 has no global scales (s0 = s1 = 1)
        float g0 = __uint_as_float(r0[c][jj]), g1 = __uint_as_float(r0[c][jj + 1]);
        float u0 = __uint_as_float(r1[c][jj]), u1 = __uint_as_float(r1[c][jj + 1]);
        if constexpr (FMT == MOE_FMT_NVFP4) {
          g0 *= s0;
          g1 *= s0;
          u0 *= s1;
          u1 *= s1;
        }
        if (capped) {
          g0 = cap_soft(g0, a.cap, a.inv_cap);
          g1 = cap_soft(g1, a.cap, a.inv_cap);
          u0 = cap_soft(u0, a.cap, a.inv_cap);
          u1 = cap_soft(u1, a.cap, a.inv_cap);
        }
        const float h0 = silu(g0) * u0, h1 = silu(g1) * u1;
        if constexpr (FMT == MOE_FMT_MXFP8) mh = fmaxf(mh, fmaxf(fabsf(h0), fabsf(h1)));
        const __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
        pk[j / 2] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      const int f = f0 + 32 * b;
      if constexpr (FMT == MOE_FMT_MXFP8) {
        // the block's 32 features are this thread's: amax, E8M0 scale and
        // E4M3 codes in registers.  The largest |bf16(h)| is bf16(largest
        // |h|): rounding to nearest even is monotone and symmetric.
        const float m = __bfloat162float(__float2bfloat16_rn(mh));
        uint32_t sc = 0, q[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (m != 0.0f) {
          sc = mx_scale_code(m, a.mx_mode);
          const float mul = exp2i(127 - (int)sc);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            q[i / 2] |= e4m3x2_encode(__fmul_rn(__uint_as_float(pk[i] << 16), mul),
                                      __fmul_rn(__uint_as_float(pk[i] & 0xFFFF0000u), mul))
                        << (16 * (i & 1));
        }
        uint4* dst = reinterpret_cast<uint4*>(a.hq_codes + row * a.NA + f);
        dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
        dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
        a.hq_scales[act_scale_offset(row, f >> 5, a.NA >> 5, NT)] = (uint8_t)sc;
      } else {
        uint4* dst = reinterpret_cast<uint4*>(a.h_out + row * a.NA + f);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
      // the next block moves to the front (register moves, no indexing)
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        r0[0][j] = r0[2][j];
        r0[1][j] = r0[3][j];
        r1[0][j] = r1[2][j];
        r1[1][j] = r1[3][j];
      }
    }
  } else if (a.y16) {
    // MOE_Y_FP16E: each thread's 64 features of a weight block are two whole
    // 32-feature exponent blocks of its own row, encoded by the thread (no
    // exchange for the exponent).  A block's codes are 64 bytes, four 16-byte
    // chunks; the four lanes of each group of four swap chunks (a 4 x 4
    // transpose) so that each store instruction writes whole 64-byte blocks
    // of eight rows instead of one 16-byte quarter of 32 rows.
    const int64_t prow = (int64_t)rt.canon + n;
    const bool row_ok = valid && MOE_IN_BOUNDS(prow < a.P);
    int nv = rt.n_valid - q * 32;  // token rows of this quadrant in the tile (warp-uniform)
    if (!MOE_IN_BOUNDS((int64_t)rt.canon + q * 32 + (nv > 32 ? 32 : nv) <= a.P)) nv = 0;
    if (nv <= 0) return;
    const int f0 = mt * ROWS + 64 * hc;
    const int g4 = lane & ~3;  // first row of this lane's group within the quadrant
    uint16_t* ybase = reinterpret_cast<uint16_t*>(a.y_out) + ((int64_t)rt.canon + q * 32 + g4) * a.NA + f0 +
                      8 * (lane & 3);
    uint16_t* erow = reinterpret_cast<uint16_t*>(a.y_exp + prow * (a.NA >> 5) + (f0 >> 5));
    uint32_t pk[16];
    int eb[2];
#pragma unroll
    for (int wb = 0; wb < 2; ++wb) {
      if (wb == 1 && !second) break;
      uint32_t(&ra)[4][16] = wb == 0 ? r0 : r1;
      const float sc = wb == 0 ? s0 : s1;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        eb[b] = y16_block_codes(ra[2 * b], ra[2 * b + 1], sc, pk);
        quad_transpose4x4(pk, lane);
        uint16_t* dst = ybase + 128 * wb + 32 * b;
#pragma unroll
        for (int r = 0; r < 4; ++r)
          if (g4 + r < nv)
            *reinterpret_cast<uint4*>(dst + (int64_t)r * a.NA) =
                make_uint4(pk[4 * r], pk[4 * r + 1], pk[4 * r + 2], pk[4 * r + 3]);
      }
      if (row_ok) erow[2 * wb] = (uint16_t)((eb[0] & 0xFF) | ((eb[1] & 0xFF) << 8));
    }
  } else {
    // y rows are written feature-contiguously: each 32 x 32 (token x
    // feature) group of the warp is transposed with xor shuffles, then
    // lane L stores feature L of one token row per instruction
    int nv = rt.n_valid - q * 32;  // token rows of this quadrant in the tile
    // (warp-uniform: the quadrant's rows are stored only if all are in range)
    if (!MOE_IN_BOUNDS((int64_t)rt.canon + q * 32 + (nv > 32 ? 32 : nv) <= a.P)) nv = 0;
    float* ybase = reinterpret_cast<float*>(a.y_out) + ((int64_t)rt.canon + q * 32) * a.NA + mt * ROWS + 64 * hc +
                   lane;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        r0[ch][j] = __float_as_uint(__uint_as_float(r0[ch][j]) * s0);
        r1[ch][j] = __float_as_uint(__uint_as_float(r1[ch][j]) * s1);
      }
    warp_transpose32(r0[0], r0[1], lane);
    warp_transpose32(r0[2], r0[3], lane);
    store_rows32(ybase, a.NA, nv, r0[0], r0[1]);
    store_rows32(ybase + 32, a.NA, nv, r0[2], r0[3]);
    if (second) {
      warp_transpose32(r1[0], r1[1], lane);
      warp_transpose32(r1[2], r1[3], lane);
      store_rows32(ybase + 128, a.NA, nv, r1[0], r1[1]);
      store_rows32(ybase + 160, a.NA, nv, r1[2], r1[3]);
    }
  }
}

template <int FMT, bool GATED>
struct CfgTM {
  static constexpr int NT = kNTWide;               // token rows per tile (MMA M)
  static constexpr int ROWS = GATED ? 128 : 256;   // output features per tile
  static constexpr int NB = 256;                   // weight rows per tile (MMA N)
  static constexpr int EPI_WARPS = 8;              // two warps per TMEM lane quadrant
  static constexpr int THREADS = (4 + EPI_WARPS) * 32;
  static constexpr int STAGES = 4;
  static constexpr int A_BYTES = NT * 128;         // tokens, 128 bytes of codes per row per stage
  static constexpr int B_BYTES = NB * 128;         // weights
  static constexpr int SF_ATOMS = FMT == MOE_FMT_NVFP4 ? 4 : 1;  // 512-byte atoms per 128 rows per stage
  static constexpr int SF_BYTES = SF_ATOMS * 512;
  static constexpr int RAW_STAGE = A_BYTES + B_BYTES + 3 * SF_BYTES;
  static constexpr int STAGE_BYTES = (RAW_STAGE + 1023) / 1024 * 1024;
  static constexpr int BAR_BYTES = 256;
  static constexpr int RTB_BYTES = (kMaxE + 1) * 4;
  static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + RTB_BYTES + 1024;
  static constexpr int ELEMS_PER_STAGE = FMT == MOE_FMT_NVFP4 ? 256 : 128;
  static constexpr int BLOCK = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  static constexpr int ACC_COLS = NB;              // 128 lanes (tokens) x 256 columns (weight rows)
  static constexpr int SFA_COLS = SF_ATOMS * 4;    // token scales
  static constexpr int SFB_COLS = 2 * SF_ATOMS * 4;  // weight scales: per MMA, rows 128..255 four columns on
  static constexpr int SF_COLS_STAGE = SFA_COLS + SFB_COLS;
  static constexpr int TMEM_SF = ACC_COLS;
  static constexpr int TMEM_COLS = 512;
  static_assert(TMEM_SF + STAGES * SF_COLS_STAGE <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(16 * STAGES + 64 <= BAR_BYTES, "barrier area");
};

template <int FMT, bool GATED>
__global__ void __launch_bounds__(CfgTM<FMT, GATED>::THREADS, 1)
    k_moe_gemm_tm(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                  const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
  using C = CfgTM<FMT, GATED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tmem_full = empty + C::STAGES;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* drain = tmem_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_rtb = reinterpret_cast<int32_t*>(smem + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, C::EPI_WARPS);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmA0);
    prefetch_tmap(&tmA1);
    prefetch_tmap(&tmB);
  }
  // the tile plan is read before the dependency wait, as in k_moe_gemm
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_rtb[i] = __ldcg(a.rt_base + i);
  tc_fence_before();
  const bool plan_ok = plan_ok_sync(s_rtb, a.E, a.max_tiles);
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // warp 0 stays out: a wait taken by some of its lanes would hold the
  // producer lane too (its other lanes read nothing the previous kernel wrote)
  if (warp != 0) pdl_wait();

  const int MT = (a.NA + C::ROWS - 1) / C::ROWS;
  const int total = plan_ok ? s_rtb[a.E] * MT : 0;
  const int KB = a.K / C::ELEMS_PER_STAGE;
  const int64_t atoms_per_row = (a.K / C::BLOCK) / 4;  // scale atoms per 128 rows over K

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      int mt = 0, rti = 0;
      RowTile rt{};
      if (blockIdx.x < total) {
        map_tile(blockIdx.x, MT, s_rtb, a.E, mt, rti);
        rt = load_tile(a.tiles + rti);
      }
      // the first tile's weight stages go out before the dependency wait
      const int pre = (blockIdx.x < total && !a.withhold_loads) ? min(KB, C::STAGES) : 0;
      if (pre > 0) {
        const int arow = rt.e * a.NA + mt * C::ROWS;
        const bool second = GATED || (mt * C::ROWS + 128 < a.NA);
        const int arow1 = (GATED || !second) ? arow : arow + 128;
        const uint8_t* sfw0 = a.sfA0 + (int64_t)(arow >> 7) * atoms_per_row * 512;
        const uint8_t* sfw1 = a.sfA1 + (int64_t)(arow1 >> 7) * atoms_per_row * 512;
        constexpr uint32_t bytes = C::A_BYTES + C::B_BYTES + 3 * C::SF_BYTES;
#pragma unroll 1
        for (int kb = 0; kb < pre; ++kb) {  // fresh stages, phase 0
          uint8_t* sW = smem + kb * C::STAGE_BYTES + C::A_BYTES;
          uint8_t* sSF = sW + C::B_BYTES;
          mbar_expect_tx(&full[kb], bytes);
          armed |= 1u << kb;
          tma_load_2d(sW, &tmA0, &full[kb], kb * 128, arow);
          tma_load_2d(sW + C::B_BYTES / 2, &tmA1, &full[kb], kb * 128, arow1);
          bulk_load(sSF + C::SF_BYTES, sfw0 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[kb]);
          bulk_load(sSF + 2 * C::SF_BYTES, sfw1 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[kb]);
        }
      }
      pdl_wait();
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        int mt_n = 0, rti_n = 0;
        RowTile rt_n{};
        if (t + (int)gridDim.x < total) {
          map_tile(t + gridDim.x, MT, s_rtb, a.E, mt_n, rti_n);
          rt_n = load_tile(a.tiles + rti_n);
        }
        const int arow = rt.e * a.NA + mt * C::ROWS;
        // down: the second block of the last tile lies past the expert when
        // NA % 256 == 128; it then re-reads the first block and the epilogue
        // drops its results
        const bool second = GATED || (mt * C::ROWS + 128 < a.NA);
        const int arow1 = (GATED || !second) ? arow : arow + 128;
        const uint8_t* sfw0 = a.sfA0 + (int64_t)(arow >> 7) * atoms_per_row * 512;
        const uint8_t* sfw1 = a.sfA1 + (int64_t)(arow1 >> 7) * atoms_per_row * 512;
        const uint8_t* sft = a.sfB + (int64_t)(rt.row / C::NT) * atoms_per_row * 512;
        constexpr uint32_t bytes = C::A_BYTES + C::B_BYTES + 3 * C::SF_BYTES;
        const bool first = t == (int)blockIdx.x;
        for (int kb = 0; kb < KB; ++kb) {
          if (first && kb < pre) {  // weights requested before the wait: now the token rows and scales
            uint8_t* sTok = smem + stage * C::STAGE_BYTES;
            uint8_t* sSF = sTok + C::A_BYTES + C::B_BYTES;
            tma_load_2d(sTok, &tmB, &full[stage], kb * 128, rt.row);
            bulk_load(sSF, sft + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.status, ST_TIMEOUT_PRODUCER, a.limit)) {
            ok = false;
            break;
          }
          uint8_t* sTok = smem + stage * C::STAGE_BYTES;
          uint8_t* sW = sTok + C::A_BYTES;
          uint8_t* sSF = sW + C::B_BYTES;  // token scales, weight block 0, weight block 1
          if (a.withhold_loads) {  // bounded-wait self-test: nothing arrives
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          mbar_expect_tx(&full[stage], bytes);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          tma_load_2d(sTok, &tmB, &full[stage], kb * 128, rt.row);
          tma_load_2d(sW, &tmA0, &full[stage], kb * 128, arow);
          tma_load_2d(sW + C::B_BYTES / 2, &tmA1, &full[stage], kb * 128, arow1);
          bulk_load(sSF, sft + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
          bulk_load(sSF + C::SF_BYTES, sfw0 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
          bulk_load(sSF + 2 * C::SF_BYTES, sfw1 + (int64_t)kb * C::SF_BYTES, C::SF_BYTES, &full[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        mt = mt_n;
        rt = rt_n;
      }
      if (!ok) {
        for (int s = 0; s < C::STAGES; ++s) {
          if (!((armed >> s) & 1u)) continue;
          const uint32_t par = (armed_par >> s) & 1u;
          const long long t0 = clock64();
          while (!mbar_try_wait(&full[s], par) && clock64() - t0 < a.limit) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++it) {
        if (!mbar_wait(tmem_empty, (it & 1) ^ 1, abort_flag, a.status, ST_TIMEOUT_MMA, a.limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.status, ST_TIMEOUT_MMA, a.limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* sTok = smem + stage * C::STAGE_BYTES;
          uint8_t* sW = sTok + C::A_BYTES;
          uint8_t* sSF = sW + C::B_BYTES;
          const uint32_t sfa_t = tmem + C::TMEM_SF + stage * C::SF_COLS_STAGE;
          const uint32_t sfb_t = sfa_t + C::SFA_COLS;
#pragma unroll
          for (int at = 0; at < C::SF_ATOMS; ++at) {
            tc_cp_32x128b_x4(sfa_t + 4 * at, sdesc_atom(smem_u32(sSF + at * 512)));
            tc_cp_32x128b_x4(sfb_t + 8 * at, sdesc_atom(smem_u32(sSF + C::SF_BYTES + at * 512)));
            tc_cp_32x128b_x4(sfb_t + 8 * at + 4, sdesc_atom(smem_u32(sSF + 2 * C::SF_BYTES + at * 512)));
          }
          const uint64_t dA = sdesc_sw128(smem_u32(sTok));
          const uint64_t dB = sdesc_sw128(smem_u32(sW));
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t accum = (kb | s) != 0;
            const uint64_t koff = (uint64_t)((s * 32) >> 4);
            if constexpr (FMT == MOE_FMT_NVFP4) {
              mma_nvfp4(tmem, dA + koff, dB + koff, idesc_nvfp4(C::NB), sfa_t + 4 * s, sfb_t + 8 * s, accum);
            } else {
              mma_mxfp8(tmem, dA + koff, dB + koff, idesc_mxfp8(C::NB, (uint32_t)s), sfa_t, sfb_t, accum);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(tmem_full);
      }
      tc_commit(drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(drain, 0) && clock64() - t0 < a.limit) {
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    // Warp (4 + i): TMEM lane quadrant i % 4 (tokens 32 (i % 4) + lane), and
    // columns [64 (i / 4), +64) of each weight block: the share is copied to
    // registers, TMEM is released, then the arithmetic and stores run.
    const int q = warp & 3;
    const int hc = (warp - 4) >> 2;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    const int n = q * 32 + lane;  // token row within the tile
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      int mt, rti;
      map_tile(t, MT, s_rtb, a.E, mt, rti);
      const RowTile rt = a.tiles[rti];
      const bool valid = n < rt.n_valid;
      float sA0 = 1.0f, sA1 = 1.0f, gb = 1.0f;
      if constexpr (FMT == MOE_FMT_NVFP4) {
        sA0 = a.gA0[rt.e];
        sA1 = a.gA1[rt.e];
        if (valid) gb = a.gB[rt.row + n];
      }
      // the warp leaves together: tcgen05.ld and the shuffles below need all lanes
      if (!__all_sync(0xffffffffu, mbar_wait(tmem_full, it & 1, abort_flag, a.status, ST_TIMEOUT_EPILOGUE, a.limit)))
        break;
      tc_fence_after();
      uint32_t r0[4][16], r1[4][16];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        tmem_ld16(tq + 64 * hc + 16 * ch, r0[ch]);
        tmem_ld16(tq + 128 + 64 * hc + 16 * ch, r1[ch]);
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
      tm_epilogue_math<FMT, GATED>(a, r0, r1, rt, mt, n, valid, q, hc, lane, sA0 * gb, sA1 * gb);
    }
  }
  __syncthreads();
  pdl_trigger();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int FMT, bool GATED>
cudaError_t launch_tm(const GemmLaunch& g, cudaStream_t st, bool pdl) {
  using C = CfgTM<FMT, GATED>;
  static PerDeviceOnce attr;
  cudaError_t e = once_per_device(
      attr, [] { return cudaFuncSetAttribute(k_moe_gemm_tm<FMT, GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM); });
  if (e != cudaSuccess) return e;
  const GemmArgs a = gemm_args(g);
  return launch_k(k_moe_gemm_tm<FMT, GATED>, dim3(g.num_sms), dim3(C::THREADS), C::SMEM, st, pdl, *g.tmA0, *g.tmA1,
                  *g.tmB, a);
}

}  // namespace

cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t st, bool pdl) {
  const bool wide = tile_rows(*g.cfg) == kNTWide;
  if (g.cfg->fmt == MOE_FMT_NVFP4) {
    if (wide) return g.gated ? launch_tm<MOE_FMT_NVFP4, true>(g, st, pdl) : launch_tm<MOE_FMT_NVFP4, false>(g, st, pdl);
    return g.gated ? launch_t<MOE_FMT_NVFP4, true>(g, st, pdl) : launch_t<MOE_FMT_NVFP4, false>(g, st, pdl);
  }
  if (wide) return g.gated ? launch_tm<MOE_FMT_MXFP8, true>(g, st, pdl) : launch_tm<MOE_FMT_MXFP8, false>(g, st, pdl);
  return g.gated ? launch_t<MOE_FMT_MXFP8, true>(g, st, pdl) : launch_t<MOE_FMT_MXFP8, false>(g, st, pdl);
}

}  // namespace moe
