// Internal (non-ABI) declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Token rows per expert tile (MMA N <= NT): 64 for decode batches (two TMEM
// accumulator buffers), 128 when the experts see 64 tokens or more on average
// (one buffer, twice the work per weight byte).  Each expert's rows start at a
// multiple of NT in the expert-grouped activation buffers.
constexpr int kNTDecode = 64;
constexpr int kNTWide = 128;

// One block of up to NT consecutive rows of one expert in padded row order.
struct RowTile {
  int e;        // expert
  int row;      // first padded row (multiple of NT)
  int n_valid;  // valid rows in the tile (1..NT)
  int canon;    // first canonical pair position (offsets[e] + NT*i)
};

constexpr int kTileRows = 128;     // weight rows (MMA M) per tile
constexpr int kMaxE = 1024;
constexpr int kMaxT = 65536;
constexpr int kMaxK = 32;

inline int block_elems(moe_format f) { return f == MOE_FMT_NVFP4 ? 16 : 32; }
inline int64_t code_bytes(moe_format f, int64_t K) { return f == MOE_FMT_NVFP4 ? K / 2 : K; }

inline int tile_rows(const moe_config& c) {
  return (int64_t)c.T * c.k >= (int64_t)64 * c.E ? kNTWide : kNTDecode;
}
// Rows of the token-operand TMA box: 16 for decode tiles (only the rows a
// tile holds are loaded), the whole tile for 128-row tiles (one copy per
// stage; a ragged tile reads rows of the next segment, which stay unused).
inline int b_box_rows(const moe_config& c) { return tile_rows(c) == kNTWide ? kNTWide : 16; }
// h goes through the bf16 buffer and a row-quantisation pass for NVFP4 (its
// global scale spans the whole row); MXFP8 h is quantised in GEMM1's epilogue.
inline bool h_row_pass(const moe_config& c) { return c.fmt == MOE_FMT_NVFP4; }
// Padded row capacity of the expert-grouped activation buffers.
inline int64_t padded_rows(const moe_config& c) {
  const int64_t P = (int64_t)c.T * c.k, nt = tile_rows(c);
  return ((P + nt - 1) / nt + c.E) * nt;
}
inline int64_t max_row_tiles(const moe_config& c) { return padded_rows(c) / tile_rows(c); }
// Bytes of activation block scales in the per-row-tile atom layout.
inline int64_t act_scale_bytes(int64_t R, int64_t scale_cols, int nt) { return (R / nt) * (scale_cols / 4) * 512; }

void ws_layout(const moe_config& c, moe_ws_layout* L);

// --- launches (all return cudaGetLastError() of their launches) -------------
// Launches after the first of an API call use programmatic dependent launch
// (`pdl` = true): the kernel may start while its predecessor drains and waits
// for it on the device.
// Router: logits + top-k + weights.  `scratch` holds router_scratch_floats(c)
// floats; `status` (nullable) is cleared by the router's first kernel.
// `fixed_scratch`: the caller's scratch is the static array of
// moe_route_noalloc, whose documented bound keeps the original split counts.
cudaError_t launch_router(const moe_config& c, const __nv_bfloat16* x, const __nv_bfloat16* wr,
                          const float* bias, float* scratch, int32_t* idx, float* w, uint32_t* status,
                          cudaStream_t st, bool pdl, bool fixed_scratch = false);
size_t router_scratch_floats(const moe_config& c, bool fixed_scratch = false);
int router_splits(const moe_config& c, bool fixed_scratch = false);
// Prefill router (tensor-core logits, exact re-check of the candidates).
bool router_uses_tc(const moe_config& c);
size_t router_tc_scratch_floats(const moe_config& c);
cudaError_t launch_router_tc(const moe_config& c, const __nv_bfloat16* x, const __nv_bfloat16* wr,
                             const float* bias, float* scratch, int32_t* idx, float* w, uint32_t* status,
                             cudaStream_t st, bool pdl);
// 2D u8 tensor map [rows, row_bytes] with 128-byte swizzle, box 128 bytes x box_rows.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int box_rows);

// bitmap [E, ceil(T/32)] and chunk_counts [dispatch_chunks(c), E]
int dispatch_chunks(const moe_config& c);
cudaError_t launch_dispatch(const moe_config& c, const int32_t* idx, uint32_t* bitmap, int32_t* chunk_counts,
                            cudaStream_t st, bool pdl);
// chunk_base: the chunk counts after launch_scan_plan replaced them by each
// expert's pairs in the earlier chunks
cudaError_t launch_dispatch_scatter(const moe_config& c, const int32_t* idx, const uint32_t* bitmap,
                                    const int32_t* chunk_base, const int32_t* offsets, int32_t* perm,
                                    int32_t* pair_pos, cudaStream_t st, bool pdl);
// Whole dispatch + tile plan in one CTA when the token bitmaps fit in shared
// memory (decode batches); returns cudaErrorNotSupported otherwise.
bool dispatch_fits_one_cta(const moe_config& c);
cudaError_t launch_dispatch_small(const moe_config& c, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                  int32_t* perm, int32_t* pair_pos, int32_t* seg_start, RowTile* tiles,
                                  int32_t* rt_base, uint32_t* status, int32_t* sync, cudaStream_t st, bool pdl);
// pair counts (the sum of chunk_counts, also written to counts_out; or from
// offsets_in when chunk_counts == nullptr) -> offsets_out (optional),
// seg_start [E+1], tiles, rt_base [E+1] (first row tile of each expert; the
// total at E); zeroes *status when given, and the fused decode FFN's
// counters (sync) when given and that kernel runs.  chunk_counts (if given)
// are replaced by each expert's pairs in the chunks before (launch_dispatch_scatter).
cudaError_t launch_scan_plan(const moe_config& c, int32_t* chunk_counts, int32_t* counts_out,
                             const int32_t* offsets_in, int32_t* offsets_out, int32_t* seg_start, RowTile* tiles,
                             int32_t* rt_base, uint32_t* status, int32_t* sync, cudaStream_t st, bool pdl);

// act_static: NVFP4 static activation globals fp32 [E, 2] (x, h) or nullptr
// (dynamic per-row globals).
cudaError_t launch_quant_x(const moe_config& c, const __nv_bfloat16* x, const int32_t* idx,
                           const int32_t* offsets, const int32_t* pair_pos, const int32_t* seg_start,
                           uint8_t* codes, uint8_t* scales, float* glob, const float* act_static, cudaStream_t st,
                           bool pdl);

cudaError_t launch_quant_h(const moe_config& c, const __nv_bfloat16* h, const int32_t* idx,
                           const int32_t* offsets, const int32_t* perm, const int32_t* seg_start,
                           uint8_t* codes, uint8_t* scales, float* glob, const float* act_static, cudaStream_t st,
                           bool pdl);

cudaError_t launch_quantize(moe_format fmt, int mx_mode, int src_fp32, const void* src, int64_t rows,
                            int64_t cols, int64_t group_rows, moe_scale_layout layout, uint8_t* codes,
                            uint8_t* scales, float* glob, float* amax_scratch, cudaStream_t st);

cudaError_t launch_pack_scales(const uint8_t* src, int64_t rows, int64_t cols, uint8_t* dst, cudaStream_t st);

cudaError_t launch_fake_quant(moe_format fmt, int mx_mode, int src_fp32, const void* src, int64_t rows, int64_t cols,
                              int64_t group_rows, float* out, float* glob, cudaStream_t st);

// MXFP8 KV-cache rows: bf16 [tokens, heads, head_dim] (token stride in
// elements) -> codes [num_slots, heads, head_dim], E8M0 scales
// [num_slots, heads, head_dim/32] at slot[t] (nullptr: slot t).
cudaError_t launch_kv_quant_mxfp8(const __nv_bfloat16* kv, int64_t tokens, int heads, int head_dim,
                                  int64_t token_stride, const int64_t* slot, int64_t num_slots, int mode,
                                  uint8_t* codes, uint8_t* scales, int sms, cudaStream_t st);

// Tensor-core peak microbenchmark (one CTA per SM; n_mma MMAs each).
int mma_peak_flops_per_mma(moe_format fmt);
cudaError_t launch_mma_peak(moe_format fmt, int ctas, long long n_mma, unsigned long long* cycles, uint32_t* status,
                            cudaStream_t st);

struct GemmLaunch {
  const moe_config* cfg;
  bool gated;          // GEMM1 (gate+up, SwiGLU epilogue) vs GEMM2 (down)
  const CUtensorMap* tmA0;
  const CUtensorMap* tmA1;
  const CUtensorMap* tmB;
  const uint8_t* sfA0;
  const uint8_t* sfA1;
  const uint8_t* sfB;
  const float* gA0;
  const float* gA1;
  const float* gB;
  const RowTile* tiles;
  const int32_t* rt_base;
  int E;
  int NA;              // rows of A per expert
  int K;               // reduction length (elements)
  __nv_bfloat16* h_out;   // gated, NVFP4: bf16 h [R, F]
  uint8_t* hq_codes = nullptr;   // gated, MXFP8: h codes [R, F] and scales, written by the epilogue
  uint8_t* hq_scales = nullptr;
  void* y_out;            // down:  y rows [P, H] in the config's y_format (fp32, or fp16 codes)
  int8_t* y_exp = nullptr; // down, MOE_Y_FP16E: exponents [P, H/32]
  uint32_t* status;
  int num_sms;
  long long wait_limit = 0;  // cycles per bounded wait; 0 = the default (~2 s)
  int withhold_loads = 0;    // self-test only: the producer issues no loads, so every wait runs out
};
cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t st, bool pdl);

// Decode batches (64-row tiles): GEMM1 (g1), the h quantisation and GEMM2
// (g2; its tmB is the h-code map) in one persistent launch.  sync:
// ffn_sync_ints(c) int32 (per row tile a completion count and a ready flag,
// then the tile counter, then per padded row the |h| maximum), zeroed by the
// tile-plan kernel.  NVFP4: the h row pass writes hq_codes / hq_scales /
// hq_global.
cudaError_t launch_ffn_decode(const GemmLaunch& g1, const GemmLaunch& g2, int32_t* sync, const float* act_static,
                              uint8_t* hq_codes, uint8_t* hq_scales, float* hq_global, int withhold_arrivals,
                              cudaStream_t st, bool pdl);
inline int64_t ffn_sync_ints(const moe_config& c) { return 2 * max_row_tiles(c) + 1 + padded_rows(c); }
// The expert FFN of this configuration runs as the fused decode kernel:
// decode tiles from 64 pairs on (measured on GB300: 6% faster at 64 pairs,
// 1.5% at 512, 2.3% at 1536; at 8 pairs, a single token, the separate
// kernels were 6 us faster).
constexpr int kFusedMinPairs = 64;
inline bool ffn_fused(const moe_config& c) {
  return tile_rows(c) == kNTDecode && c.ffn_schedule == 0 && (int64_t)c.T * c.k >= kFusedMinPairs;
}

// y rows of a configuration: bytes, and where the exponents of MOE_Y_FP16E
// start (after the P*H fp16 codes).
inline bool y16(const moe_config& c) { return c.y_format == MOE_Y_FP16E; }
inline int64_t y_bytes(const moe_config& c) {
  const int64_t P = (int64_t)c.T * c.k;
  return y16(c) ? P * c.H * 2 + P * (c.H / 32) : P * c.H * 4;
}
inline int8_t* y_exponents(const moe_config& c, void* y) {
  return y16(c) ? reinterpret_cast<int8_t*>(y) + (int64_t)c.T * c.k * c.H * 2 : nullptr;
}

cudaError_t launch_combine(const moe_config& c, const void* y, const float* w, const int32_t* pair_pos,
                           __nv_bfloat16* out, cudaStream_t st, bool pdl);

}  // namespace moe
