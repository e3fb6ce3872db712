// Token dispatch: group the (token, slot) pairs by expert, in token order
// within an expert (cookbook page on Inkling-2-Small, MegaMoE paragraph:
// dispatch is the first step of the fused MoE unit), plus the expert tile
// plan the grouped GEMMs walk.
//
// Three small kernels, all deterministic:
//   1. one CTA per expert builds the expert's token bitmap in shared memory
//      from topk_idx and counts its pairs;
//   2. one CTA scans counts -> offsets, padded segment starts (each expert's
//      rows begin at a multiple of kNT) and the list of kNT-row tiles;
//   3. one CTA per expert ranks its tokens from the bitmap (popcount prefix)
//      and writes perm / pair_pos.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kDThreads = 256;
constexpr int kMaxWords = kMaxT / 32;

__global__ void __launch_bounds__(kDThreads) k_disp_bitmap(const int32_t* __restrict__ idx, int T, int k,
                                                           uint32_t* __restrict__ bitmap, int32_t* __restrict__ counts) {
  __shared__ uint32_t bm[kMaxWords];
  __shared__ int red[kDThreads / 32];
  const int e = blockIdx.x;
  const int W = (T + 31) / 32;
  for (int i = threadIdx.x; i < W; i += blockDim.x) bm[i] = 0u;
  __syncthreads();
  const int P = T * k;
  for (int p = threadIdx.x; p < P; p += blockDim.x)
    if (idx[p] == e) {
      int t = p / k;
      atomicOr(&bm[t >> 5], 1u << (t & 31));
    }
  __syncthreads();
  int c = 0;
  for (int i = threadIdx.x; i < W; i += blockDim.x) {
    uint32_t v = bm[i];
    bitmap[(int64_t)e * W + i] = v;
    c += __popc(v);
  }
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int i = 0; i < kDThreads / 32; ++i) s += red[i];
    counts[e] = s;
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
__global__ void __launch_bounds__(1024) k_scan_plan(const int32_t* __restrict__ counts,
                                                    const int32_t* __restrict__ offsets_in, int E,
                                                    int32_t* __restrict__ offsets_out, int32_t* __restrict__ seg_start,
                                                    RowTile* __restrict__ tiles, int32_t* __restrict__ rt_base,
                                                    uint32_t* __restrict__ status) {
  __shared__ int sh[32];
  const int e = threadIdx.x;
  if (status && e == 0) *status = 0u;
  int c = 0;
  if (e < E) c = counts ? counts[e] : (offsets_in[e + 1] - offsets_in[e]);
  int tot;
  int off = block_exclusive_scan(c, &tot, sh);
  if (offsets_out) {
    if (e < E) offsets_out[e] = off;
    if (e == 0) offsets_out[E] = tot;
  }
  int nrt = (c + kNT - 1) / kNT;
  int padded = nrt * kNT;
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
      t.row = seg + kNT * i;
      t.n_valid = min(kNT, c - kNT * i);
      t.canon = off + kNT * i;
      tiles[rt0 + i] = t;
    }
  }
  if (e == 0) rt_base[E] = rtot;
}

__global__ void __launch_bounds__(kDThreads) k_disp_scatter(const int32_t* __restrict__ idx, int T, int k,
                                                            const uint32_t* __restrict__ bitmap,
                                                            const int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ perm, int32_t* __restrict__ pair_pos) {
  __shared__ int sh[32];
  const int e = blockIdx.x;
  const int W = (T + 31) / 32;
  const int wpt = (W + blockDim.x - 1) / blockDim.x;
  const int w0 = threadIdx.x * wpt;
  int c = 0;
  for (int i = 0; i < wpt; ++i)
    if (w0 + i < W) c += __popc(bitmap[(int64_t)e * W + w0 + i]);
  int tot;
  int rank = block_exclusive_scan(c, &tot, sh);
  const int base = offsets[e];
  for (int i = 0; i < wpt; ++i) {
    if (w0 + i >= W) break;
    uint32_t v = bitmap[(int64_t)e * W + w0 + i];
    while (v) {
      int b = __ffs(v) - 1;
      v &= v - 1;
      int t = (w0 + i) * 32 + b;
      int j = 0;
      while (j < k && idx[t * k + j] != e) ++j;
      int p = base + rank;
      perm[p] = t * k + j;
      pair_pos[t * k + j] = p;
      ++rank;
    }
  }
}

}  // namespace

cudaError_t launch_dispatch(const moe_config& c, const int32_t* idx, int32_t* counts, int32_t* offsets,
                            int32_t* perm, int32_t* pair_pos, uint32_t* bitmap, cudaStream_t st) {
  k_disp_bitmap<<<c.E, kDThreads, 0, st>>>(idx, c.T, c.k, bitmap, counts);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_scatter(const moe_config& c, const int32_t* idx, const uint32_t* bitmap,
                                    const int32_t* offsets, int32_t* perm, int32_t* pair_pos, cudaStream_t st) {
  k_disp_scatter<<<c.E, kDThreads, 0, st>>>(idx, c.T, c.k, bitmap, offsets, perm, pair_pos);
  return cudaGetLastError();
}

cudaError_t launch_scan_plan(const moe_config& c, const int32_t* counts, const int32_t* offsets_in,
                             int32_t* offsets_out, int32_t* seg_start, RowTile* tiles, int32_t* rt_base,
                             uint32_t* status, cudaStream_t st) {
  k_scan_plan<<<1, 1024, 0, st>>>(counts, offsets_in, c.E, offsets_out, seg_start, tiles, rt_base, status);
  return cudaGetLastError();
}

}  // namespace moe
