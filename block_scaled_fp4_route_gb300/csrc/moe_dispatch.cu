// Token dispatch: group the (token, slot) pairs by expert, in token order
// within an expert (cookbook page on Inkling-2-Small, MegaMoE paragraph:
// dispatch is the first step of the fused MoE unit), plus the expert tile
// plan the grouped GEMMs walk.
//
// Three small kernels, all deterministic:
//   1. one CTA per 256-token chunk sets the chunk's bits of every expert's
//      token bitmap (shared memory, then global) and counts them;
//   2. one CTA sums the chunk counts and scans counts -> offsets, padded
//      segment starts (each expert's rows begin at a multiple of nt) and the
//      list of nt-row tiles;
//   3. one CTA per expert ranks its tokens from the bitmap (popcount prefix)
//      and writes perm / pair_pos.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kDThreads = 256;

constexpr int kChunkTokens = 256;  // tokens per bitmap CTA: 8 bitmap words per expert

// One CTA per 256-token chunk: the chunk's token bits of every expert are
// set in shared memory, copied to the global bitmap [E, W], and counted per
// expert into chunk_counts [chunk, E].  idx is read once in total.
__global__ void __launch_bounds__(kDThreads) k_disp_bitmap(const int32_t* __restrict__ idx, int T, int k, int E,
                                                           uint32_t* __restrict__ bitmap,
                                                           int32_t* __restrict__ chunk_counts) {
  extern __shared__ uint32_t cbm[];  // [E][8]
  const int ch = blockIdx.x;
  const int t0 = ch * kChunkTokens, t1 = min(T, t0 + kChunkTokens);
  const int W = (T + 31) / 32, w0 = t0 / 32, nw = min(8, W - w0);
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) cbm[i] = 0u;
  __syncthreads();
  for (int p = t0 * k + threadIdx.x; p < t1 * k; p += blockDim.x) {
    const int t = p / k, e = idx[p];
    if ((unsigned)e < (unsigned)E) atomicOr(&cbm[e * 8 + ((t - t0) >> 5)], 1u << (t & 31));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) {
    const int e = i >> 3, j = i & 7;
    if (j < nw) bitmap[(int64_t)e * W + w0 + j] = cbm[i];
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) c += __popc(cbm[e * 8 + j]);
    chunk_counts[(int64_t)ch * E + e] = c;
  }
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int* total, int* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < nw ? sh[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) sh[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  int base = w > 0 ? sh[w - 1] : 0;
  *total = sh[nw - 1];
  __syncthreads();
  return base + x - v;
}

// counts (if non-null) or offsets_in -> offsets_out, seg_start, tile list.
// The pair counts come from per-chunk counts (summed here and written to
// counts_out), or from offsets_in.
__global__ void __launch_bounds__(1024) k_scan_plan(int32_t* __restrict__ chunk_counts, int nch,
                                                    int32_t* __restrict__ counts_out,
                                                    const int32_t* __restrict__ offsets_in, int E,
                                                    int32_t* __restrict__ offsets_out, int32_t* __restrict__ seg_start,
                                                    RowTile* __restrict__ tiles, int32_t* __restrict__ rt_base,
                                                    uint32_t* __restrict__ status, int nt,
                                                    int32_t* __restrict__ sync, int nsync, int max_tiles) {
  __shared__ int sh[32];
  const int e = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (status && e == 0) *status = 0u;
  // the fused decode FFN's completion counts start at zero
  for (int i = e; i < nsync; i += blockDim.x) sync[i] = 0;
  int c = 0;
  if (e < E) {
    if (chunk_counts) {
      // eight chunk counts requested at a time; each is replaced by the
      // expert's pairs in the chunks before it (the scatter's chunk base)
      int ch = 0;
      for (; ch + 8 <= nch; ch += 8) {
        int v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = chunk_counts[(int64_t)(ch + i) * E + e];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          chunk_counts[(int64_t)(ch + i) * E + e] = c;
          c += v[i];
        }
      }
      for (; ch < nch; ++ch) {
        const int v = chunk_counts[(int64_t)ch * E + e];
        chunk_counts[(int64_t)ch * E + e] = c;
        c += v;
      }
      if (counts_out) counts_out[e] = c;
    } else {
      c = offsets_in[e + 1] - offsets_in[e];
    }
  }
  int tot;
  int off = block_exclusive_scan(c, &tot, sh);
  if (offsets_out) {
    if (e < E) offsets_out[e] = off;
    if (e == 0) offsets_out[E] = tot;
  }
  int nrt = (c + nt - 1) / nt;
  int padded = nrt * nt;
  int ptot;
  int seg = block_exclusive_scan(padded, &ptot, sh);
  if (e < E) seg_start[e] = seg;
  if (e == 0) seg_start[E] = ptot;
  int rtot;
  int rt0 = block_exclusive_scan(nrt, &rtot, sh);
  if (e < E) {
    rt_base[e] = rt0;
    for (int i = 0; i < nrt; ++i) {
      RowTile t;
      t.e = e;
      t.row = seg + nt * i;
      t.n_valid = min(nt, c - nt * i);
      t.canon = off + nt * i;
      if (MOE_IN_BOUNDS(rt0 + i < max_tiles)) tiles[rt0 + i] = t;
    }
  }
  if (e == 0) rt_base[E] = rtot;
}

// One thread per pair (t, j), e = idx[t, j]: its position in the dispatch
// order is offsets[e] + the expert's pairs in the 256-token chunks before
// t's (chunk_base, from the tile-plan kernel) + the expert's tokens before t
// inside the chunk (popcounts of at most 8 bitmap words).  Every pair is
// independent, so a hot expert's pairs spread over the whole grid.
__global__ void __launch_bounds__(kDThreads) k_disp_scatter(const int32_t* __restrict__ idx, int T, int k, int E,
                                                            const uint32_t* __restrict__ bitmap,
                                                            const int32_t* __restrict__ chunk_base,
                                                            const int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ perm, int32_t* __restrict__ pair_pos) {
  const int W = (T + 31) / 32;
  const int64_t P = (int64_t)T * k;
  const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (p >= P) return;
  const int t = (int)(p / k);
  const int e = idx[p];
  if (!MOE_IN_BOUNDS((unsigned)e < (unsigned)E)) return;
  const int ch = t / kChunkTokens;
  const int wt = t >> 5;
  const uint32_t* bm = bitmap + (int64_t)e * W;
  int rank = 0;
  for (int w = ch * (kChunkTokens / 32); w < wt; ++w) rank += __popc(bm[w]);
  rank += __popc(bm[wt] & ((1u << (t & 31)) - 1u));
  const int64_t pos = (int64_t)offsets[e] + chunk_base[(int64_t)ch * E + e] + rank;
  if (MOE_IN_BOUNDS(pos >= 0 && pos < P)) {
    perm[pos] = (int32_t)p;
    pair_pos[p] = (int32_t)pos;
  }
}

constexpr int kSmallWords = 12288;  // 48 KB of token bitmaps
constexpr int kSmallPairs = 8192;   // 32 KB of staged expert ids (T <= 256, k <= 32)

// Whole dispatch for small batches in one CTA of 1024 threads: the expert ids
// and a token bitmap per expert in shared memory; counts and row tiles of all
// experts in one block scan (a packed (pairs, row tiles) sum); then every pair
// finds its rank among its expert's tokens by counting the bitmap bits below
// its token.
__global__ void __launch_bounds__(1024) k_dispatch_small(const int32_t* __restrict__ idx, int T, int k, int E,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ perm, int32_t* __restrict__ pair_pos,
                                                         int32_t* __restrict__ seg_start, RowTile* __restrict__ tiles,
                                                         int32_t* __restrict__ rt_base, uint32_t* __restrict__ status,
                                                         int nt, int32_t* __restrict__ sync, int nsync) {
  extern __shared__ uint32_t sbm[];  // [E][W] bitmaps, then the ids [T*k], then the offsets [E]
  __shared__ int sh[32];
  const int W = (T + 31) / 32;
  const int P = T * k;
  int32_t* sidx = reinterpret_cast<int32_t*>(sbm + E * W);
  int32_t* soff = sidx + P;
  pdl_wait();
  pdl_trigger();
  if (status && threadIdx.x == 0) *status = 0u;
  // the fused decode FFN's completion counts start at zero
  for (int i = threadIdx.x; i < nsync; i += blockDim.x) sync[i] = 0;
  for (int i = threadIdx.x; i < E * W; i += blockDim.x) sbm[i] = 0u;
  for (int p = threadIdx.x; p < P; p += blockDim.x) sidx[p] = idx[p];
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int t = p / k, e = sidx[p];
    if ((unsigned)e < (unsigned)E) atomicOr(&sbm[e * W + (t >> 5)], 1u << (t & 31));
  }
  __syncthreads();
  const int e = threadIdx.x;
  int c = 0;
  if (e < E)
    for (int i = 0; i < W; ++i) c += __popc(sbm[e * W + i]);
  const int nrt = (c + nt - 1) / nt;
  // pairs in the high half, row tiles in the low half: at most T*k <= 8192
  // pairs and T*k/nt + E <= 1152 row tiles, so the halves never carry
  int tot;
  const int pre = block_exclusive_scan((c << 16) | nrt, &tot, sh);
  const int off = pre >> 16, rt0 = pre & 0xFFFF;
  const int seg = rt0 * nt;  // each expert's rows start at its first row tile
  if (e < E) {
    counts[e] = c;
    offsets[e] = off;
    seg_start[e] = seg;
    rt_base[e] = rt0;
    soff[e] = off;
    for (int i = 0; i < nrt; ++i) {
      RowTile tl;
      tl.e = e;
      tl.row = seg + nt * i;
      tl.n_valid = min(nt, c - nt * i);
      tl.canon = off + nt * i;
      if (MOE_IN_BOUNDS(rt0 + i < (P + nt - 1) / nt + E)) tiles[rt0 + i] = tl;
    }
  }
  if (e == 0) {
    offsets[E] = tot >> 16;
    seg_start[E] = (tot & 0xFFFF) * nt;
    rt_base[E] = tot & 0xFFFF;
  }
  __syncthreads();
  // pair (t, j) of expert e: its rank is the number of e's tokens below t
  // (a token's first slot holding e; later duplicates are not dispatched)
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int ee = sidx[p];
    if ((unsigned)ee >= (unsigned)E) continue;
    const int t = p / k, j = p - t * k;
    bool first = true;
    for (int jj = 0; jj < j; ++jj) first = first && sidx[t * k + jj] != ee;
    if (!first) continue;
    const uint32_t* bm = sbm + ee * W;
    int rank = __popc(bm[t >> 5] & ((1u << (t & 31)) - 1u));
    for (int i = 0; i < (t >> 5); ++i) rank += __popc(bm[i]);
    const int pos = soff[ee] + rank;
    if (MOE_IN_BOUNDS(pos < P)) {
      perm[pos] = p;
      pair_pos[p] = pos;
    }
  }
}

}  // namespace

// The one-CTA path ranks each expert's tokens serially, so it is kept for
// decode batches (up to 256 tokens).
bool dispatch_fits_one_cta(const moe_config& c) {
  return c.T <= 256 && c.E <= 1024 && (int64_t)c.E * ((c.T + 31) / 32) <= kSmallWords &&
         (int64_t)c.T * c.k <= kSmallPairs;
}

cudaError_t launch_dispatch_small(const moe_config& c, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                  int32_t* perm, int32_t* pair_pos, int32_t* seg_start, RowTile* tiles,
                                  int32_t* rt_base, uint32_t* status, int32_t* sync, cudaStream_t st, bool pdl) {
  if (!dispatch_fits_one_cta(c)) return cudaErrorNotSupported;
  const size_t smem = ((size_t)c.E * ((c.T + 31) / 32) + (size_t)c.T * c.k + c.E) * 4;
  static PerDeviceOnce attr;
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(k_dispatch_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (kSmallWords + kSmallPairs + kMaxE) * 4);
  });
  if (e != cudaSuccess) return e;
  return launch_k(k_dispatch_small, dim3(1), dim3(1024), smem, st, pdl, idx, c.T, c.k, c.E, counts, offsets, perm,
                  pair_pos, seg_start, tiles, rt_base, status, tile_rows(c), sync,
                  sync && ffn_fused(c) ? (int)ffn_sync_ints(c) : 0);
}

int dispatch_chunks(const moe_config& c) { return (c.T + kChunkTokens - 1) / kChunkTokens; }

cudaError_t launch_dispatch(const moe_config& c, const int32_t* idx, uint32_t* bitmap, int32_t* chunk_counts,
                            cudaStream_t st, bool pdl) {
  return launch_k(k_disp_bitmap, dim3(dispatch_chunks(c)), dim3(kDThreads), (size_t)c.E * 8 * 4, st, pdl, idx, c.T,
                  c.k, c.E, bitmap, chunk_counts);
}

cudaError_t launch_dispatch_scatter(const moe_config& c, const int32_t* idx, const uint32_t* bitmap,
                                    const int32_t* chunk_base, const int32_t* offsets, int32_t* perm,
                                    int32_t* pair_pos, cudaStream_t st, bool pdl) {
  const int64_t P = (int64_t)c.T * c.k;
  return launch_k(k_disp_scatter, dim3((unsigned)((P + kDThreads - 1) / kDThreads)), dim3(kDThreads), 0, st, pdl,
                  idx, c.T, c.k, c.E, bitmap, chunk_base, offsets, perm, pair_pos);
}

cudaError_t launch_scan_plan(const moe_config& c, int32_t* chunk_counts, int32_t* counts_out,
                             const int32_t* offsets_in, int32_t* offsets_out, int32_t* seg_start, RowTile* tiles,
                             int32_t* rt_base, uint32_t* status, int32_t* sync, cudaStream_t st, bool pdl) {
  // the counters exist for the fused decode FFN only
  const int nsync = sync && ffn_fused(c) ? (int)ffn_sync_ints(c) : 0;
  return launch_k(k_scan_plan, dim3(1), dim3(1024), 0, st, pdl, chunk_counts, dispatch_chunks(c), counts_out,
                  offsets_in, c.E, offsets_out, seg_start, tiles, rt_base, status, tile_rows(c), sync, nsync,
                  (int)max_row_tiles(c));
}

}  // namespace moe
