// C ABI of the MoE layer (include/moe.h): argument validation, workspace
// layout, TMA descriptors, and the chaining of the kernels on the caller's
// stream.  Allocates no device memory.
#include <mutex>
#include <vector>

#include "moe_common.cuh"

namespace moe {

#ifdef MOE_DEBUG_BOUNDS
static std::vector<BoundsReader>& bounds_readers() {
  static std::vector<BoundsReader> v;
  return v;
}
void register_bounds_reader(BoundsReader r) { bounds_readers().push_back(r); }
#endif

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DevInfo {
  bool probed = false;
  bool ok = false;
  int sms = 0;
};
DevInfo g_dev[64];
std::mutex g_mu;

moe_status device_check(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.ok = (major == 10 && minor == 3);
    d.probed = true;
  }
  if (!d.ok) return MOE_ERR_ARCH;
  if (sms) *sms = d.sms;
  return MOE_OK;
}

moe_status check_cfg(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->fmt != MOE_FMT_NVFP4 && c->fmt != MOE_FMT_MXFP8) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->T > kMaxT || c->E < 1 || c->E > kMaxE || c->k < 1 || c->k > kMaxK || c->k > c->E)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const int q = c->fmt == MOE_FMT_NVFP4 ? 256 : 128;  // one 128-byte TMA box of codes along K
  if (c->H < q || c->F < q || c->H % q != 0 || c->F % q != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->H > 16384 || c->F > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;  // activation rows quantised in registers
  if ((int64_t)c->T * c->k > (1 << 30)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!(c->swiglu_cap >= 0.0f)) return MOE_ERR_INVALID_ARG;
  if (c->mx_scale_mode != 0 && c->mx_scale_mode != 1) return MOE_ERR_INVALID_ARG;
  if (c->act_global_mode != 0 && c->act_global_mode != 1) return MOE_ERR_INVALID_ARG;
  if (c->act_global_mode == 1 && c->fmt != MOE_FMT_NVFP4) return MOE_ERR_INVALID_ARG;  // MXFP8 has no global
  if (c->ffn_schedule != 0 && c->ffn_schedule != 1) return MOE_ERR_INVALID_ARG;
  if (c->y_format != MOE_Y_FP32 && c->y_format != MOE_Y_FP16E) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// act_static_scales: required (4-byte aligned) in act_global_mode 1, else ignored.
moe_status check_static(const moe_config* c, const float* act_static) {
  if (c->act_global_mode != 1) return MOE_OK;
  if (!act_static) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(act_static) & 3u) != 0) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_status check_qw(const moe_config* c, const moe_qweight* w) {
  if (!w || !w->codes || !w->scales) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w->codes) || !aligned16(w->scales)) return MOE_ERR_MISALIGNED;
  if (c->fmt == MOE_FMT_NVFP4) {
    if (!w->global_scale) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w->global_scale)) return MOE_ERR_MISALIGNED;
  }
  return MOE_OK;
}

moe_status check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  }
  return MOE_OK;
}

moe_status check_ws(const moe_config* c, const void* ws, size_t bytes) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  moe_ws_layout L;
  ws_layout(*c, &L);
  if (bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

// --- TMA descriptors ---------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(ws) + off);
}

void mark(cudaEvent_t* ev, int i, cudaStream_t st) {
  if (ev) cudaEventRecord(ev[i], st);
}

// Expert FFN after the tile plan exists in the workspace.  ev (optional)
// receives the stage boundaries 2..5 (x quantisation, GEMM1, h quantisation,
// GEMM2).
moe_status ffn_core(const moe_config& c, int sms, const __nv_bfloat16* x, const int32_t* idx, const int32_t* offsets,
                    const int32_t* perm, const int32_t* pair_pos, const moe_qweight* gate, const moe_qweight* up,
                    const moe_qweight* down, const float* act_static, void* y, void* ws, cudaStream_t st,
                    cudaEvent_t* ev = nullptr) {
  if (c.act_global_mode != 1) act_static = nullptr;
  moe_ws_layout L;
  ws_layout(c, &L);
  const int64_t R = L.R;
  uint8_t* xq = at<uint8_t>(ws, L.xq_codes);
  uint8_t* xs = at<uint8_t>(ws, L.xq_scales);
  float* xg = at<float>(ws, L.xq_global);
  __nv_bfloat16* h = at<__nv_bfloat16>(ws, L.h_bf16);
  uint8_t* hq = at<uint8_t>(ws, L.hq_codes);
  uint8_t* hs = at<uint8_t>(ws, L.hq_scales);
  float* hg = at<float>(ws, L.hq_global);
  const int32_t* seg = at<int32_t>(ws, L.seg_start);
  const RowTile* tiles = at<RowTile>(ws, L.tiles);
  const int32_t* rtb = at<int32_t>(ws, L.rt_base);
  uint32_t* status = at<uint32_t>(ws, L.status);

  mark(ev, 2, st);
  cudaError_t e = launch_quant_x(c, x, idx, offsets, pair_pos, seg, xq, xs, xg, act_static, st, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  const int64_t hb = code_bytes(c.fmt, c.H), fb = code_bytes(c.fmt, c.F);
  CUtensorMap mg, mu, md, mx, mh;
  if (!make_map(&mg, gate->codes, (int64_t)c.E * c.F, hb, 128) ||
      !make_map(&mu, up->codes, (int64_t)c.E * c.F, hb, 128) ||
      !make_map(&md, down->codes, (int64_t)c.E * c.H, fb, 128) || !make_map(&mx, xq, R, hb, b_box_rows(c)) ||
      !make_map(&mh, hq, R, fb, b_box_rows(c)))
    return MOE_ERR_CUDA;

  GemmLaunch g1{};
  g1.cfg = &c;
  g1.gated = true;
  g1.tmA0 = &mg;
  g1.tmA1 = &mu;
  g1.tmB = &mx;
  g1.sfA0 = (const uint8_t*)gate->scales;
  g1.sfA1 = (const uint8_t*)up->scales;
  g1.sfB = xs;
  g1.gA0 = gate->global_scale;
  g1.gA1 = up->global_scale;
  g1.gB = xg;
  g1.tiles = tiles;
  g1.rt_base = rtb;
  g1.E = c.E;
  g1.NA = c.F;
  g1.K = c.H;
  g1.h_out = h;
  g1.hq_codes = hq;
  g1.hq_scales = hs;
  g1.status = status;
  g1.num_sms = sms;

  GemmLaunch g2{};
  g2.cfg = &c;
  g2.gated = false;
  g2.tmA0 = &md;
  g2.tmA1 = &md;
  g2.tmB = &mh;
  g2.sfA0 = (const uint8_t*)down->scales;
  g2.sfA1 = (const uint8_t*)down->scales;
  g2.sfB = hs;
  g2.gA0 = down->global_scale;
  g2.gA1 = down->global_scale;
  g2.gB = hg;
  g2.tiles = tiles;
  g2.rt_base = rtb;
  g2.E = c.E;
  g2.NA = c.H;
  g2.K = c.F;
  g2.y_out = y;
  g2.y_exp = y_exponents(c, y);
  g2.status = status;
  g2.num_sms = sms;

  mark(ev, 3, st);
  if (ffn_fused(c)) {
    // decode batches: GEMM1, the h quantisation and GEMM2 in one launch (its
    // time is the GEMM1 stage; the h and GEMM2 stages are empty)
    if (launch_ffn_decode(g1, g2, at<int32_t>(ws, L.ffn_sync), act_static, hq, hs, hg, 0, st, true) != cudaSuccess)
      return MOE_ERR_CUDA;
    mark(ev, 4, st);
    mark(ev, 5, st);
    return MOE_OK;
  }
  if (launch_gemm(g1, st, true) != cudaSuccess) return MOE_ERR_CUDA;

  mark(ev, 4, st);
  if (h_row_pass(c) &&
      launch_quant_h(c, h, idx, offsets, perm, seg, hq, hs, hg, act_static, st, true) != cudaSuccess)
    return MOE_ERR_CUDA;

  mark(ev, 5, st);
  if (launch_gemm(g2, st, true) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

// Dispatch + tile plan into the workspace: one CTA for decode batches,
// bitmap / scan / scatter kernels otherwise.  `status` (optional) is cleared.
moe_status dispatch_impl(const moe_config& c, const int32_t* idx, int32_t* counts, int32_t* offsets, int32_t* perm,
                         int32_t* pair_pos, void* ws, uint32_t* status, cudaStream_t st, bool pdl) {
  moe_ws_layout L;
  ws_layout(c, &L);
  int32_t* seg = at<int32_t>(ws, L.seg_start);
  RowTile* tiles = at<RowTile>(ws, L.tiles);
  int32_t* rtb = at<int32_t>(ws, L.rt_base);
  if (dispatch_fits_one_cta(c))
    return cuda_status(launch_dispatch_small(c, idx, counts, offsets, perm, pair_pos, seg, tiles, rtb, status,
                                             at<int32_t>(ws, L.ffn_sync), st, pdl));
  uint32_t* bm = at<uint32_t>(ws, L.bitmap);
  int32_t* chunk_counts = reinterpret_cast<int32_t*>(bm + (size_t)c.E * ((c.T + 31) / 32));
  if (launch_dispatch(c, idx, bm, chunk_counts, st, pdl) != cudaSuccess ||
      launch_scan_plan(c, chunk_counts, counts, nullptr, offsets, seg, tiles, rtb, status, at<int32_t>(ws, L.ffn_sync),
                       st, true) != cudaSuccess ||
      launch_dispatch_scatter(c, idx, bm, chunk_counts, offsets, perm, pair_pos, st, true) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

void ws_layout(const moe_config& c, moe_ws_layout* L) {
  const int64_t T = c.T, E = c.E, P = T * c.k, R = padded_rows(c), W = (T + 31) / 32;
  const int bs = block_elems(c.fmt);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 1024);
    return o;
  };
  L->R = R;
  L->tile_rows = tile_rows(c);
  L->status = take(256);
  L->logits = take(router_scratch_floats(c) * 4);
  L->topk_idx = take(P * 4);
  L->topk_w = take(P * 4);
  L->counts = take(E * 4);
  L->offsets = take((E + 1) * 4);
  L->perm = take(P * 4);
  L->pair_pos = take(P * 4);
  L->bitmap = take((E * W + (int64_t)dispatch_chunks(c) * E) * 4);  // bitmap [E, W], then chunk counts
  L->seg_start = take((E + 1) * 4);
  L->tiles = take(max_row_tiles(c) * sizeof(RowTile));
  L->rt_base = take((E + 1) * 4);
  L->ffn_sync = take(ffn_sync_ints(c) * 4);
  L->xq_codes = take(R * code_bytes(c.fmt, c.H));
  L->xq_scales = take(act_scale_bytes(R, c.H / bs, tile_rows(c)));
  L->xq_global = take(R * 4);
  L->h_bf16 = take(h_row_pass(c) ? R * c.F * 2 : 0);
  L->hq_codes = take(R * code_bytes(c.fmt, c.F));
  L->hq_scales = take(act_scale_bytes(R, c.F / bs, tile_rows(c)));
  L->hq_global = take(R * 4);
  L->y_perm = take(y_bytes(c));
  L->total = off;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_ws_layout L;
  ws_layout(*cfg, &L);
  *bytes = L.total;
  return MOE_OK;
}

moe_status moe_workspace_layout(const moe_config* cfg, moe_ws_layout* layout) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!layout) return MOE_ERR_INVALID_ARG;
  ws_layout(*cfg, layout);
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x_dev, const void* w_router_dev, const float* bias_dev,
                     int32_t* topk_idx_dev, float* topk_w_dev, void* ws_dev, size_t ws_bytes, void* stream) {
  moe_status s = check_cfg(cfg);
  if (s == MOE_OK) s = check_ptrs({x_dev, w_router_dev, bias_dev, topk_idx_dev, topk_w_dev});
  if (s == MOE_OK) s = check_ws(cfg, ws_dev, ws_bytes);
  if (s == MOE_OK) s = device_check(nullptr);
  if (s != MOE_OK) return s;
  moe_ws_layout L;
  ws_layout(*cfg, &L);
  return cuda_status(launch_router(*cfg, (const __nv_bfloat16*)x_dev, (const __nv_bfloat16*)w_router_dev, bias_dev,
                                   at<float>(ws_dev, L.logits), topk_idx_dev, topk_w_dev,
                                   at<uint32_t>(ws_dev, L.status), (cudaStream_t)stream, false));
}

moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx_dev, int32_t* counts_dev, int32_t* offsets_dev,
                        int32_t* perm_dev, int32_t* pair_pos_dev, void* ws_dev, size_t ws_bytes, void* stream) {
  moe_status s = check_cfg(cfg);
  if (s == MOE_OK) s = check_ptrs({topk_idx_dev, counts_dev, offsets_dev, perm_dev, pair_pos_dev});
  if (s == MOE_OK) s = check_ws(cfg, ws_dev, ws_bytes);
  if (s == MOE_OK) s = device_check(nullptr);
  if (s != MOE_OK) return s;
  moe_ws_layout L;
  ws_layout(*cfg, &L);
  cudaStream_t st = (cudaStream_t)stream;
  return dispatch_impl(*cfg, topk_idx_dev, counts_dev, offsets_dev, perm_dev, pair_pos_dev, ws_dev, nullptr, st,
                       false);
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* x_dev, const int32_t* topk_idx_dev,
                          const int32_t* offsets_dev, const int32_t* perm_dev, const int32_t* pair_pos_dev,
                          const moe_qweight* gate, const moe_qweight* up, const moe_qweight* down,
                          const float* act_static_scales, void* y_perm_dev, void* ws_dev, size_t ws_bytes,
                          void* stream) {
  moe_status s = check_cfg(cfg);
  if (s == MOE_OK) s = check_ptrs({x_dev, topk_idx_dev, offsets_dev, perm_dev, pair_pos_dev, y_perm_dev});
  if (s == MOE_OK) s = check_static(cfg, act_static_scales);
  if (s == MOE_OK) s = check_qw(cfg, gate);
  if (s == MOE_OK) s = check_qw(cfg, up);
  if (s == MOE_OK) s = check_qw(cfg, down);
  if (s == MOE_OK) s = check_ws(cfg, ws_dev, ws_bytes);
  int sms = 0;
  if (s == MOE_OK) s = device_check(&sms);
  if (s != MOE_OK) return s;
  moe_ws_layout L;
  ws_layout(*cfg, &L);
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_scan_plan(*cfg, nullptr, nullptr, offsets_dev, nullptr, at<int32_t>(ws_dev, L.seg_start),
                       at<RowTile>(ws_dev, L.tiles), at<int32_t>(ws_dev, L.rt_base),
                       at<uint32_t>(ws_dev, L.status), at<int32_t>(ws_dev, L.ffn_sync), st, false) != cudaSuccess)
    return MOE_ERR_CUDA;
  return ffn_core(*cfg, sms, (const __nv_bfloat16*)x_dev, topk_idx_dev, offsets_dev, perm_dev, pair_pos_dev, gate, up,
                  down, act_static_scales, y_perm_dev, ws_dev, st);
}

moe_status moe_combine(const moe_config* cfg, const void* y_perm_dev, const float* topk_w_dev,
                       const int32_t* pair_pos_dev, void* out_dev, void* stream) {
  moe_status s = check_cfg(cfg);
  if (s == MOE_OK) s = check_ptrs({y_perm_dev, topk_w_dev, pair_pos_dev, out_dev});
  if (s == MOE_OK) s = device_check(nullptr);
  if (s != MOE_OK) return s;
  return cuda_status(launch_combine(*cfg, y_perm_dev, topk_w_dev, pair_pos_dev, (__nv_bfloat16*)out_dev,
                                    (cudaStream_t)stream, false));
}

moe_status moe_y_bytes(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = (size_t)y_bytes(*cfg);
  return MOE_OK;
}

static moe_status forward_impl(const moe_config* cfg, const void* x_dev, const void* w_router_dev,
                               const float* bias_dev, const moe_qweight* gate, const moe_qweight* up,
                               const moe_qweight* down, const float* act_static, void* out_dev, void* ws_dev,
                               size_t ws_bytes, void* stream, cudaEvent_t* ev) {
  moe_status s = check_cfg(cfg);
  if (s == MOE_OK) s = check_ptrs({x_dev, w_router_dev, bias_dev, out_dev});
  if (s == MOE_OK) s = check_static(cfg, act_static);
  if (s == MOE_OK) s = check_qw(cfg, gate);
  if (s == MOE_OK) s = check_qw(cfg, up);
  if (s == MOE_OK) s = check_qw(cfg, down);
  if (s == MOE_OK) s = check_ws(cfg, ws_dev, ws_bytes);
  int sms = 0;
  if (s == MOE_OK) s = device_check(&sms);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  moe_ws_layout L;
  ws_layout(c, &L);
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* idx = at<int32_t>(ws_dev, L.topk_idx);
  float* w = at<float>(ws_dev, L.topk_w);
  int32_t* counts = at<int32_t>(ws_dev, L.counts);
  int32_t* offsets = at<int32_t>(ws_dev, L.offsets);
  int32_t* perm = at<int32_t>(ws_dev, L.perm);
  int32_t* pair_pos = at<int32_t>(ws_dev, L.pair_pos);
  void* y = at<uint8_t>(ws_dev, L.y_perm);
  mark(ev, 0, st);
  // the router's first kernel clears the status word of the call.  It is
  // launched behind whatever precedes it on the stream (a previous layer's
  // combine, in a serving loop) and waits for it before its first access, so
  // its launch overlaps that kernel's tail.
  if (launch_router(c, (const __nv_bfloat16*)x_dev, (const __nv_bfloat16*)w_router_dev, bias_dev,
                    at<float>(ws_dev, L.logits), idx, w, at<uint32_t>(ws_dev, L.status), st, true) != cudaSuccess)
    return MOE_ERR_CUDA;
  mark(ev, 1, st);
  s = dispatch_impl(c, idx, counts, offsets, perm, pair_pos, ws_dev, nullptr, st, true);
  if (s != MOE_OK) return s;
  s = ffn_core(c, sms, (const __nv_bfloat16*)x_dev, idx, offsets, perm, pair_pos, gate, up, down, act_static, y, ws_dev,
               st, ev);
  if (s != MOE_OK) return s;
  mark(ev, 6, st);
  s = cuda_status(launch_combine(c, y, w, pair_pos, (__nv_bfloat16*)out_dev, st, true));
  mark(ev, 7, st);
  return s;
}

moe_status moe_forward_kernel_count(const moe_config* cfg, int* count) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!count) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  int n = router_uses_tc(c) ? 3 : 2;         // router: (norms,) logits, top-k
  n += dispatch_fits_one_cta(c) ? 1 : 3;      // dispatch: one CTA, or bitmap + scan + scatter
  n += 1;                                     // x quantisation
  if (ffn_fused(c)) {
    n += 2;                                   // the fused expert FFN, combine
  } else {
    n += 1;                                   // GEMM1
    n += h_row_pass(c) ? 1 : 0;               // h quantisation (else inside GEMM1)
    n += 2;                                   // GEMM2, combine
  }
  *count = n;
  return MOE_OK;
}

moe_status moe_forward(const moe_config* cfg, const void* x_dev, const void* w_router_dev, const float* bias_dev,
                       const moe_qweight* gate, const moe_qweight* up, const moe_qweight* down,
                       const float* act_static_scales, void* out_dev, void* ws_dev, size_t ws_bytes, void* stream) {
  return forward_impl(cfg, x_dev, w_router_dev, bias_dev, gate, up, down, act_static_scales, out_dev, ws_dev, ws_bytes,
                      stream, nullptr);
}

moe_status moe_forward_profiled(const moe_config* cfg, const void* x_dev, const void* w_router_dev,
                                const float* bias_dev, const moe_qweight* gate, const moe_qweight* up,
                                const moe_qweight* down, const float* act_static_scales, void* out_dev,
                                void* ws_dev, size_t ws_bytes, void* stream, void* const* events) {
  if (!events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_NUM_STAGES + 1; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  cudaEvent_t ev[MOE_NUM_STAGES + 1];
  for (int i = 0; i < MOE_NUM_STAGES + 1; ++i) ev[i] = (cudaEvent_t)events[i];
  return forward_impl(cfg, x_dev, w_router_dev, bias_dev, gate, up, down, act_static_scales, out_dev, ws_dev, ws_bytes,
                      stream, ev);
}

moe_status moe_quantize(moe_format fmt, int mx_scale_mode, int src_is_fp32, const void* src_dev, int64_t rows,
                        int64_t cols, int64_t group_rows, moe_scale_layout layout, void* codes_dev, void* scales_dev,
                        float* global_dev, void* stream) {
  if (fmt != MOE_FMT_NVFP4 && fmt != MOE_FMT_MXFP8) return MOE_ERR_INVALID_ARG;
  if (mx_scale_mode != 0 && mx_scale_mode != 1) return MOE_ERR_INVALID_ARG;
  if (layout != MOE_SCALES_ROWMAJOR && layout != MOE_SCALES_TILED) return MOE_ERR_INVALID_ARG;
  const int bs = fmt == MOE_FMT_NVFP4 ? 16 : 32;
  if (rows < 1 || rows > (int64_t)INT32_MAX || cols < bs || cols % bs != 0 || cols > (1 << 20))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (src_is_fp32 ? (cols % 4) : (cols % 8)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (layout == MOE_SCALES_TILED && (rows % 128 != 0 || (cols / bs) % 4 != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (fmt == MOE_FMT_NVFP4) {
    if (group_rows < 0 || (group_rows > 0 && rows % group_rows != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
    moe_status s = check_ptrs({src_dev, codes_dev, scales_dev, global_dev});
    if (s != MOE_OK) return s;
  } else {
    moe_status s = check_ptrs({src_dev, codes_dev, scales_dev});
    if (s != MOE_OK) return s;
  }
  moe_status s = device_check(nullptr);
  if (s != MOE_OK) return s;
  return cuda_status(launch_quantize(fmt, mx_scale_mode, src_is_fp32, src_dev, rows, cols, group_rows, layout,
                                     (uint8_t*)codes_dev, (uint8_t*)scales_dev, global_dev, nullptr,
                                     (cudaStream_t)stream));
}

moe_status moe_pack_scales(const void* rowmajor_dev, int64_t rows, int64_t scale_cols, void* tiled_dev, void* stream) {
  if (rows < 1 || rows % 128 != 0 || scale_cols < 4 || scale_cols % 4 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_status s = check_ptrs({rowmajor_dev, tiled_dev});
  if (s == MOE_OK) s = device_check(nullptr);
  if (s != MOE_OK) return s;
  return cuda_status(launch_pack_scales((const uint8_t*)rowmajor_dev, rows, scale_cols, (uint8_t*)tiled_dev,
                                        (cudaStream_t)stream));
}

moe_status moe_fake_quantize(moe_format fmt, int mx_scale_mode, int src_is_fp32, const void* src_dev, int64_t rows,
                             int64_t cols, int64_t group_rows, float* out_dev, float* global_dev, void* stream) {
  if (fmt != MOE_FMT_NVFP4 && fmt != MOE_FMT_MXFP8) return MOE_ERR_INVALID_ARG;
  if (mx_scale_mode != 0 && mx_scale_mode != 1) return MOE_ERR_INVALID_ARG;
  const int bs = fmt == MOE_FMT_NVFP4 ? 16 : 32;
  if (rows < 1 || rows > (int64_t)INT32_MAX || cols < bs || cols % bs != 0 || cols > (1 << 20))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (src_is_fp32 ? (cols % 4) : (cols % 8)) return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_status s;
  if (fmt == MOE_FMT_NVFP4) {
    if (group_rows < 0 || (group_rows > 0 && rows % group_rows != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
    s = check_ptrs({src_dev, out_dev, global_dev});
  } else {
    s = check_ptrs({src_dev, out_dev});
  }
  if (s == MOE_OK) s = device_check(nullptr);
  if (s != MOE_OK) return s;
  return cuda_status(launch_fake_quant(fmt, mx_scale_mode, src_is_fp32, src_dev, rows, cols, group_rows, out_dev,
                                       global_dev, (cudaStream_t)stream));
}

moe_status moe_kv_quantize_mxfp8(const void* kv_dev, int64_t tokens, int heads, int head_dim, int64_t token_stride,
                                 const int64_t* slot_dev, int64_t num_slots, int mx_scale_mode, void* codes_dev,
                                 void* scales_dev, void* stream) {
  if (tokens < 0 || tokens > (int64_t)INT32_MAX || heads < 1 || heads > 4096 || head_dim < 32 || head_dim > 1024 ||
      head_dim % 32 != 0)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (token_stride < (int64_t)heads * head_dim || token_stride % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (mx_scale_mode != 0 && mx_scale_mode != 1) return MOE_ERR_INVALID_ARG;
  if (num_slots < 0 || (!slot_dev && num_slots < tokens)) return MOE_ERR_INVALID_ARG;
  if (tokens == 0) return MOE_OK;
  moe_status s = check_ptrs({kv_dev, codes_dev});
  if (s == MOE_OK && !scales_dev) s = MOE_ERR_INVALID_ARG;
  if (s == MOE_OK && slot_dev && (reinterpret_cast<uintptr_t>(slot_dev) & 7u) != 0) s = MOE_ERR_MISALIGNED;
  int sms = 0;
  if (s == MOE_OK) s = device_check(&sms);
  if (s != MOE_OK) return s;
  return cuda_status(launch_kv_quant_mxfp8((const __nv_bfloat16*)kv_dev, tokens, heads, head_dim, token_stride,
                                           slot_dev, num_slots, mx_scale_mode, (uint8_t*)codes_dev,
                                           (uint8_t*)scales_dev, sms, (cudaStream_t)stream));
}

moe_status moe_bench_mma_peak(moe_format fmt, int64_t mmas_per_cta, unsigned long long* cycles_dev, void* status_dev,
                              int* ctas, double* flops_per_mma, void* stream) {
  if (fmt != MOE_FMT_NVFP4 && fmt != MOE_FMT_MXFP8) return MOE_ERR_INVALID_ARG;
  if (mmas_per_cta < 4 || mmas_per_cta % 4 != 0 || mmas_per_cta > ((int64_t)1 << 40)) return MOE_ERR_INVALID_ARG;
  if (!status_dev || !ctas || !flops_per_mma) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(status_dev) & 3u) != 0 || (reinterpret_cast<uintptr_t>(cycles_dev) & 7u) != 0)
    return MOE_ERR_MISALIGNED;
  int sms = 0;
  moe_status s = device_check(&sms);
  if (s != MOE_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(status_dev, 0, 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  *ctas = sms;
  *flops_per_mma = (double)mma_peak_flops_per_mma(fmt);
  return cuda_status(launch_mma_peak(fmt, sms, mmas_per_cta, cycles_dev, (uint32_t*)status_dev, st));
}

moe_status moe_selftest_bounded_wait(const moe_config* cfg, const moe_qweight* gate, const moe_qweight* up,
                                     void* ws_dev, size_t ws_bytes, int64_t limit_cycles, void* stream) {
  moe_status s = check_cfg(cfg);
  if (s == MOE_OK) s = check_qw(cfg, gate);
  if (s == MOE_OK) s = check_qw(cfg, up);
  if (s == MOE_OK) s = check_ws(cfg, ws_dev, ws_bytes);
  if (s == MOE_OK && (limit_cycles < 1000 || limit_cycles > 4000000000LL)) s = MOE_ERR_INVALID_ARG;
  int sms = 0;
  if (s == MOE_OK) s = device_check(&sms);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  moe_ws_layout L;
  ws_layout(c, &L);
  const int64_t hb = code_bytes(c.fmt, c.H);
  CUtensorMap mg, mu, mx;
  if (!make_map(&mg, gate->codes, (int64_t)c.E * c.F, hb, 128) || !make_map(&mu, up->codes, (int64_t)c.E * c.F, hb, 128) ||
      !make_map(&mx, at<uint8_t>(ws_dev, L.xq_codes), L.R, hb, b_box_rows(*cfg)))
    return MOE_ERR_CUDA;
  GemmLaunch g1{};
  g1.cfg = &c;
  g1.gated = true;
  g1.tmA0 = &mg;
  g1.tmA1 = &mu;
  g1.tmB = &mx;
  g1.sfA0 = (const uint8_t*)gate->scales;
  g1.sfA1 = (const uint8_t*)up->scales;
  g1.sfB = at<uint8_t>(ws_dev, L.xq_scales);
  g1.gA0 = gate->global_scale;
  g1.gA1 = up->global_scale;
  g1.gB = at<float>(ws_dev, L.xq_global);
  g1.tiles = at<RowTile>(ws_dev, L.tiles);
  g1.rt_base = at<int32_t>(ws_dev, L.rt_base);
  g1.E = c.E;
  g1.NA = c.F;
  g1.K = c.H;
  g1.h_out = at<__nv_bfloat16>(ws_dev, L.h_bf16);
  g1.status = at<uint32_t>(ws_dev, L.status);
  g1.num_sms = sms;
  g1.wait_limit = limit_cycles;
  g1.withhold_loads = 1;
  return cuda_status(launch_gemm(g1, (cudaStream_t)stream, false));
}

moe_status moe_selftest_dependency_wait(const moe_config* cfg, const moe_qweight* gate, const moe_qweight* up,
                                        const moe_qweight* down, void* ws_dev, size_t ws_bytes, int64_t limit_cycles,
                                        void* stream) {
  moe_status s = check_cfg(cfg);
  if (s == MOE_OK && tile_rows(*cfg) != kNTDecode) s = MOE_ERR_UNSUPPORTED_SHAPE;  // the fused kernel's shapes only
  if (s == MOE_OK) s = check_qw(cfg, gate);
  if (s == MOE_OK) s = check_qw(cfg, up);
  if (s == MOE_OK) s = check_qw(cfg, down);
  if (s == MOE_OK) s = check_ws(cfg, ws_dev, ws_bytes);
  if (s == MOE_OK && (limit_cycles < 1000 || limit_cycles > 4000000000LL)) s = MOE_ERR_INVALID_ARG;
  int sms = 0;
  if (s == MOE_OK) s = device_check(&sms);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  moe_ws_layout L;
  ws_layout(c, &L);
  const int64_t hb = code_bytes(c.fmt, c.H), fb = code_bytes(c.fmt, c.F);
  uint8_t* hq = at<uint8_t>(ws_dev, L.hq_codes);
  uint8_t* hs = at<uint8_t>(ws_dev, L.hq_scales);
  float* hg = at<float>(ws_dev, L.hq_global);
  CUtensorMap mg, mu, md, mx, mh;
  if (!make_map(&mg, gate->codes, (int64_t)c.E * c.F, hb, 128) ||
      !make_map(&mu, up->codes, (int64_t)c.E * c.F, hb, 128) ||
      !make_map(&md, down->codes, (int64_t)c.E * c.H, fb, 128) ||
      !make_map(&mx, at<uint8_t>(ws_dev, L.xq_codes), L.R, hb, b_box_rows(c)) || !make_map(&mh, hq, L.R, fb, b_box_rows(c)))
    return MOE_ERR_CUDA;
  GemmLaunch g1{}, g2{};
  g1.cfg = g2.cfg = &c;
  g1.gated = true;
  g1.tmA0 = &mg;
  g1.tmA1 = &mu;
  g1.tmB = &mx;
  g1.sfA0 = (const uint8_t*)gate->scales;
  g1.sfA1 = (const uint8_t*)up->scales;
  g1.sfB = at<uint8_t>(ws_dev, L.xq_scales);
  g1.gA0 = gate->global_scale;
  g1.gA1 = up->global_scale;
  g1.gB = at<float>(ws_dev, L.xq_global);
  g1.NA = c.F;
  g1.K = c.H;
  g1.h_out = at<__nv_bfloat16>(ws_dev, L.h_bf16);
  g1.hq_codes = hq;
  g1.hq_scales = hs;
  g2.gated = false;
  g2.tmA0 = g2.tmA1 = &md;
  g2.tmB = &mh;
  g2.sfA0 = g2.sfA1 = (const uint8_t*)down->scales;
  g2.sfB = hs;
  g2.gA0 = g2.gA1 = down->global_scale;
  g2.gB = hg;
  g2.NA = c.H;
  g2.K = c.F;
  g2.y_out = at<uint8_t>(ws_dev, L.y_perm);
  g2.y_exp = y_exponents(c, g2.y_out);
  for (GemmLaunch* g : {&g1, &g2}) {
    g->tiles = at<RowTile>(ws_dev, L.tiles);
    g->rt_base = at<int32_t>(ws_dev, L.rt_base);
    g->E = c.E;
    g->status = at<uint32_t>(ws_dev, L.status);
    g->num_sms = sms;
    g->wait_limit = limit_cycles;
  }
  // the counters are zeroed as the tile-plan kernel does (the self-test runs on its own)
  if (cudaMemsetAsync(at<int32_t>(ws_dev, L.ffn_sync), 0, ffn_sync_ints(c) * 4, (cudaStream_t)stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cuda_status(launch_ffn_decode(g1, g2, at<int32_t>(ws_dev, L.ffn_sync), nullptr, hq, hs, hg, 1,
                                       (cudaStream_t)stream, false));
}

moe_status moe_debug_bounds_status(void* stream, int* checked, int* site) {
  if (!checked) return MOE_ERR_INVALID_ARG;
  if (site) *site = 0;
#ifdef MOE_DEBUG_BOUNDS
  *checked = 1;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t any = 0;
  for (BoundsReader r : bounds_readers()) {
    uint32_t v = 0;
    if (r(&v) != cudaSuccess) return MOE_ERR_CUDA;
    any = v > any ? v : any;
  }
  if (site) *site = (int)any;
  return any ? MOE_ERR_BOUNDS : MOE_OK;
#else
  (void)stream;
  *checked = 0;
  return MOE_OK;
#endif
}

moe_status moe_poll_device_status(void* ws_dev, void* stream) {
  if (!ws_dev) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws_dev, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    if (cudaMemsetAsync(ws_dev, 0, sizeof(v), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_ERR_DEVICE_TIMEOUT;
  }
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "a device-side bounded wait ran out";
    case MOE_ERR_BOUNDS: return "an index check of the bounds-checked build failed (the access was skipped)";
  }
  return "unknown status";
}

}  // extern "C"
