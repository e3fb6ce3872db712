"""Routed block-scaled MoE layer for GB300 — Python binding of libmoe.so.

Thin ctypes marshalling over the C ABI in include/moe.h: every function here
has the name of its C entry point, takes torch tensors (device memory) and
passes their pointers and the current CUDA stream.  All arithmetic runs in the
library's CUDA kernels; there is no fallback path: if libmoe.so cannot be
built or loaded, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

FMT_NVFP4, FMT_MXFP8 = 0, 1
Y_FP32, Y_FP16E = 0, 1
SCALES_ROWMAJOR, SCALES_TILED = 0, 1

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_MISALIGNED",
          4: "MOE_ERR_WORKSPACE_TOO_SMALL", 5: "MOE_ERR_ARCH", 6: "MOE_ERR_CUDA", 7: "MOE_ERR_DEVICE_TIMEOUT",
          8: "MOE_ERR_BOUNDS"}

EXPORTED = ["moe_workspace_size", "moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_y_bytes",
            "moe_forward",
            "moe_forward_profiled", "moe_quantize", "moe_pack_scales", "moe_poll_device_status", "moe_workspace_layout",
            "moe_route_noalloc", "moe_route_noalloc_poll_status", "moe_fake_quantize", "moe_kv_quantize_mxfp8", "moe_bench_mma_peak", "moe_selftest_bounded_wait", "moe_selftest_dependency_wait", "moe_debug_bounds_status", "moe_forward_kernel_count",
            "moe_status_string"]


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("F", ctypes.c_int), ("fmt", ctypes.c_int), ("swiglu_cap", ctypes.c_float),
                ("act_global_mode", ctypes.c_int), ("mx_scale_mode", ctypes.c_int), ("bias_in_weights", ctypes.c_int),
                ("routed_scale", ctypes.c_float), ("ffn_schedule", ctypes.c_int), ("y_format", ctypes.c_int)]


class moe_qweight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


_LAYOUT_FIELDS = ["status", "logits", "topk_idx", "topk_w", "counts", "offsets", "perm", "pair_pos", "bitmap",
                  "seg_start", "tiles", "rt_base", "ffn_sync", "xq_codes", "xq_scales", "xq_global", "h_bf16", "hq_codes",
                  "hq_scales", "hq_global", "y_perm", "total"]


class moe_ws_layout(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int64), ("tile_rows", ctypes.c_int64)] + [(f, ctypes.c_size_t) for f in _LAYOUT_FIELDS]


_libs = {}
_lock = threading.Lock()
_debug_bounds = False


def use_debug_bounds_build(on: bool = True):
    """Route every entry point of this module to the bounds-checked build
    (libmoe_debug.so: kernels check the indices they derive from data and skip
    out-of-range accesses, reported by moe_debug_bounds_status) or back to the
    normal build."""
    global _debug_bounds
    _debug_bounds = bool(on)


def lib(debug_bounds=None):
    """Build (if stale) and load libmoe.so (or the bounds-checked build);
    raises if that is not possible."""
    db = _debug_bounds if debug_bounds is None else bool(debug_bounds)
    with _lock:
        if db not in _libs:
            path = _build.build(debug_bounds=db)
            L = ctypes.CDLL(path)
            P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
            cfgp = ctypes.POINTER(moe_config)
            qwp = ctypes.POINTER(moe_qweight)
            L.moe_workspace_size.argtypes = [cfgp, ctypes.POINTER(sz)]
            L.moe_route.argtypes = [cfgp, P, P, P, P, P, P, sz, P]
            L.moe_route_noalloc.argtypes = [cfgp, P, P, P, P, P, P]
            L.moe_route_noalloc_poll_status.argtypes = [P]
            L.moe_dispatch.argtypes = [cfgp, P, P, P, P, P, P, sz, P]
            L.moe_expert_ffn.argtypes = [cfgp, P, P, P, P, P, qwp, qwp, qwp, P, P, P, sz, P]
            L.moe_combine.argtypes = [cfgp, P, P, P, P, P]
            L.moe_y_bytes.argtypes = [cfgp, ctypes.POINTER(sz)]
            L.moe_forward.argtypes = [cfgp, P, P, P, qwp, qwp, qwp, P, P, P, sz, P]
            L.moe_forward_profiled.argtypes = [cfgp, P, P, P, qwp, qwp, qwp, P, P, P, sz, P,
                                               ctypes.POINTER(ctypes.c_void_p)]
            L.moe_quantize.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, i64, i64, i64, ctypes.c_int,
                                       P, P, P, P]
            L.moe_pack_scales.argtypes = [P, i64, i64, P, P]
            L.moe_fake_quantize.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, i64, i64, i64, P, P, P]
            L.moe_kv_quantize_mxfp8.argtypes = [P, i64, ctypes.c_int, ctypes.c_int, i64, P, i64, ctypes.c_int, P, P,
                                                P]
            L.moe_bench_mma_peak.argtypes = [ctypes.c_int, i64, P, P, ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_double), P]
            L.moe_selftest_bounded_wait.argtypes = [cfgp, qwp, qwp, P, sz, i64, P]
            L.moe_selftest_dependency_wait.argtypes = [cfgp, qwp, qwp, qwp, P, sz, i64, P]
            L.moe_poll_device_status.argtypes = [P, P]
            L.moe_workspace_layout.argtypes = [cfgp, ctypes.POINTER(moe_ws_layout)]
            L.moe_status_string.argtypes = [ctypes.c_int]
            L.moe_status_string.restype = ctypes.c_char_p
            L.moe_debug_bounds_status.argtypes = [P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
            for n in EXPORTED[:-1]:
                getattr(L, n).restype = ctypes.c_int
            _libs[db] = L
        return _libs[db]


def library_path() -> str:
    """Path of the in-tree library the entry points use (built by lib() when stale)."""
    return _build.LIB_DEBUG if _debug_bounds else _build.LIB


def _check(fn: str, st: int):
    if st != 0:
        raise MoeError(fn, st)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def make_config(T, H, E, k, F, fmt, swiglu_cap=10.0, mx_scale_mode=0, bias_in_weights=0, routed_scale=1.0,
                act_global_mode=0, ffn_schedule=0, y_format=None):
    """A moe_config: T tokens, hidden H, E experts, top-k, FFN width F; fmt "nvfp4" / "mxfp8" (or
    FMT_*); swiglu_cap c of c*tanh(v/c) (0 = none); mx_scale_mode 0 = OCP floor, 1 = round-up;
    bias_in_weights 0 = the bias steers selection only; act_global_mode 1 = static per-expert NVFP4
    activation globals; ffn_schedule 0 = decode batches run the expert FFN as one fused kernel,
    1 = separate kernels; y_format of the expert outputs, "fp16e" (default: fp16 codes with an
    exponent per 32 features) or "fp32" (or Y_*)."""
    if isinstance(fmt, str):
        fmt = {"nvfp4": FMT_NVFP4, "mxfp8": FMT_MXFP8}[fmt]
    if y_format is None:
        y_format = Y_FP16E
    if isinstance(y_format, str):
        y_format = {"fp32": Y_FP32, "fp16e": Y_FP16E}[y_format]
    return moe_config(T, H, E, k, F, fmt, swiglu_cap, act_global_mode, mx_scale_mode, bias_in_weights, routed_scale,
                      ffn_schedule, y_format)


def qweight(codes, scales, global_scale=None) -> moe_qweight:
    """One quantised expert matrix for all experts: codes u8 [E, N, K/2] (NVFP4) or [E, N, K]
    (MXFP8), block scales in the tiled layout, global_scale fp32 [E] (NVFP4) or None."""
    return moe_qweight(_ptr(codes), _ptr(scales), _ptr(global_scale))


# ----------------------------------------------------------------------------
# entry points (names of the C ABI)
# ----------------------------------------------------------------------------

def moe_workspace_size(cfg: moe_config) -> int:
    """Bytes of device workspace every call with this configuration needs."""
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size", lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_forward_kernel_count(cfg: moe_config) -> int:
    """Number of kernels one moe_forward launches for this configuration (host only)."""
    n = ctypes.c_int(0)
    _check("moe_forward_kernel_count", lib().moe_forward_kernel_count(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_workspace_layout(cfg: moe_config) -> dict:
    """Byte offsets of the intermediates inside the workspace, plus R and tile_rows."""
    L = moe_ws_layout()
    _check("moe_workspace_layout", lib().moe_workspace_layout(ctypes.byref(cfg), ctypes.byref(L)))
    return {f: getattr(L, f) for f in ["R", "tile_rows"] + _LAYOUT_FIELDS}


def moe_route(cfg, x, w_router, bias, topk_idx, topk_w, ws, stream=None):
    """Router: x bf16 [T, H], w_router bf16 [E, H], bias fp32 [E] -> topk_idx int32 [T, k]
    (descending key, ties to the lower expert) and topk_w fp32 [T, k]."""
    _check("moe_route", lib().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(topk_idx),
                                        _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_route_noalloc(cfg, x, w_router, bias, topk_idx, topk_w, stream=None):
    """moe_route without a workspace, for callers that cannot allocate device
    memory when they route: the library's own fixed scratch is used instead
    (see include/moe.h for its size limit and the one-time set-up)."""
    _check("moe_route_noalloc", lib().moe_route_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias),
                                                        _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


def moe_route_noalloc_poll_status(stream=None) -> int:
    """Synchronises the stream; the status of the allocation-free router's
    last calls on the current device (0 = no timeout; 7 = a bounded wait ran
    out), cleared by the read."""
    return int(lib().moe_route_noalloc_poll_status(_stream(stream)))


def moe_dispatch(cfg, topk_idx, counts, offsets, perm, pair_pos, ws, stream=None):
    """Dispatch: counts int32 [E], offsets int32 [E + 1], perm int32 [T * k] (pairs t * k + j
    sorted by expert, then token) and its inverse pair_pos int32 [T, k]; the tile plan goes to ws."""
    _check("moe_dispatch", lib().moe_dispatch(ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                                              _ptr(perm), _ptr(pair_pos), _ptr(ws), ws.numel() * ws.element_size(),
                                              _stream(stream)))


def moe_expert_ffn(cfg, x, topk_idx, offsets, perm, pair_pos, gate, up, down, y_perm, ws, stream=None,
                   act_static_scales=None):
    """Expert FFN of every pair: y_perm (out) the T * k rows in dispatch order in cfg.y_format
    (moe_y_bytes bytes: fp32 [T * k, H], or fp16 codes then int8 exponents, see y_rows); gate / up
    / down from qweight(); act_static_scales as for moe_forward."""
    _check("moe_expert_ffn", lib().moe_expert_ffn(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(offsets),
                                                  _ptr(perm), _ptr(pair_pos), ctypes.byref(gate), ctypes.byref(up),
                                                  ctypes.byref(down), _ptr(act_static_scales), _ptr(y_perm),
                                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_y_bytes(cfg) -> int:
    """Bytes of the T * k expert output rows in cfg.y_format."""
    n = ctypes.c_size_t(0)
    _check("moe_y_bytes", lib().moe_y_bytes(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def y_rows(cfg, buf):
    """Views of a y buffer (a uint8 / any tensor of moe_y_bytes bytes): fp32 [P, H] for Y_FP32,
    else (codes fp16 [P, H], exponents int8 [P, H / 32]).  Argument marshalling only."""
    import torch
    P, H = cfg.T * cfg.k, cfg.H
    b = buf.view(torch.uint8).reshape(-1)
    if cfg.y_format == Y_FP32:
        return b[:P * H * 4].view(torch.float32).view(P, H)
    return b[:P * H * 2].view(torch.float16).view(P, H), b[P * H * 2:P * H * 2 + P * (H // 32)].view(
        torch.int8).view(P, H // 32)


def moe_combine(cfg, y_perm, topk_w, pair_pos, out, stream=None):
    """out bf16 [T, H] = sum over slots (in slot order, fp32) of topk_w * y_perm[pair_pos], y_perm
    in cfg.y_format."""
    _check("moe_combine", lib().moe_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(topk_w), _ptr(pair_pos),
                                            _ptr(out), _stream(stream)))


def moe_forward(cfg, x, w_router, bias, gate, up, down, out, ws, stream=None, act_static_scales=None):
    """act_static_scales: fp32 [E, 2] (g_x, g_h) on the device when cfg.act_global_mode == 1."""
    _check("moe_forward", lib().moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias),
                                            ctypes.byref(gate), ctypes.byref(up), ctypes.byref(down),
                                            _ptr(act_static_scales), _ptr(out), _ptr(ws),
                                            ws.numel() * ws.element_size(), _stream(stream)))


NUM_STAGES = 7
STAGE_NAMES = ["router", "dispatch", "quant_x", "gemm1_gate_up_swiglu", "quant_h", "gemm2_down", "combine"]


def moe_forward_profiled(cfg, x, w_router, bias, gate, up, down, out, ws, events, stream=None,
                         act_static_scales=None):
    """events: NUM_STAGES + 1 torch.cuda.Event objects (created with timing)."""
    arr = (ctypes.c_void_p * (NUM_STAGES + 1))(*[e.cuda_event for e in events])
    _check("moe_forward_profiled", lib().moe_forward_profiled(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), ctypes.byref(gate), ctypes.byref(up),
        ctypes.byref(down), _ptr(act_static_scales), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream), arr))


def moe_quantize(fmt, src, codes, scales, global_scale=None, group_rows=0, layout=SCALES_TILED, mx_scale_mode=0,
                 stream=None):
    """src: fp32 or bf16 [rows, cols] (torch, on the device)."""
    import torch
    if isinstance(fmt, str):
        fmt = {"nvfp4": FMT_NVFP4, "mxfp8": FMT_MXFP8}[fmt]
    rows, cols = src.shape[-2] if src.dim() > 1 else 1, src.shape[-1]
    rows = src.numel() // cols
    _check("moe_quantize", lib().moe_quantize(fmt, mx_scale_mode, int(src.dtype == torch.float32), _ptr(src), rows,
                                              cols, group_rows, layout, _ptr(codes), _ptr(scales),
                                              _ptr(global_scale), _stream(stream)))


def moe_fake_quantize(fmt, src, out, global_scale=None, group_rows=0, mx_scale_mode=0, stream=None):
    """out (fp32, same shape as src) = decode(encode(src)); straight-through in training."""
    import torch
    if isinstance(fmt, str):
        fmt = {"nvfp4": FMT_NVFP4, "mxfp8": FMT_MXFP8}[fmt]
    cols = src.shape[-1]
    rows = src.numel() // cols
    _check("moe_fake_quantize", lib().moe_fake_quantize(fmt, mx_scale_mode, int(src.dtype == torch.float32), _ptr(src),
                                                        rows, cols, group_rows, _ptr(out), _ptr(global_scale),
                                                        _stream(stream)))


def moe_kv_quantize_mxfp8(kv, codes, scales, slots=None, token_stride=None, mx_scale_mode=0, stream=None):
    """New K or V rows kv bf16 [tokens, heads, head_dim] (a view whose token
    stride may exceed heads * head_dim) -> MXFP8 cache codes u8
    [num_slots, heads, head_dim] and E8M0 scales u8 [num_slots, heads,
    head_dim / 32] at slots int64 [tokens] (None: slot t; negative: skipped)."""
    tokens, heads, head_dim = kv.shape
    if token_stride is None:
        token_stride = kv.stride(0)
    num_slots = codes.shape[0]
    _check("moe_kv_quantize_mxfp8", lib().moe_kv_quantize_mxfp8(
        _ptr(kv), tokens, heads, head_dim, token_stride, _ptr(slots), num_slots, mx_scale_mode, _ptr(codes),
        _ptr(scales), _stream(stream)))


def moe_bench_mma_peak(fmt, mmas_per_cta, status, cycles=None, stream=None):
    """Launch the block-scaled MMA peak kernel (one CTA per SM, operands on
    chip); returns (ctas, flops_per_mma).  status: a device int32 tensor of
    >= 1 element; cycles: None or a device int64 tensor of >= ctas elements."""
    if isinstance(fmt, str):
        fmt = {"nvfp4": FMT_NVFP4, "mxfp8": FMT_MXFP8}[fmt]
    n, f = ctypes.c_int(0), ctypes.c_double(0.0)
    _check("moe_bench_mma_peak", lib().moe_bench_mma_peak(fmt, mmas_per_cta, _ptr(cycles), _ptr(status),
                                                          ctypes.byref(n), ctypes.byref(f), _stream(stream)))
    return n.value, f.value


def moe_selftest_bounded_wait(cfg, gate, up, ws, limit_cycles, stream=None):
    """Test hook: GEMM1 over the tile plan in ws with its loads withheld, so that every bounded wait
    runs out after limit_cycles; moe_poll_device_status then reports the timeout."""
    _check("moe_selftest_bounded_wait", lib().moe_selftest_bounded_wait(
        ctypes.byref(cfg), ctypes.byref(gate), ctypes.byref(up), _ptr(ws), ws.numel() * ws.element_size(),
        limit_cycles, _stream(stream)))


def moe_selftest_dependency_wait(cfg, gate, up, down, ws, limit_cycles, stream=None):
    """Test hook: the fused decode FFN over the tile plan in ws with its gate/up completion reports
    withheld, so that the down tiles' waits run out after limit_cycles; moe_poll_device_status then
    reports the timeout."""
    _check("moe_selftest_dependency_wait", lib().moe_selftest_dependency_wait(
        ctypes.byref(cfg), ctypes.byref(gate), ctypes.byref(up), ctypes.byref(down), _ptr(ws),
        ws.numel() * ws.element_size(), limit_cycles, _stream(stream)))


def moe_pack_scales(rowmajor, rows, scale_cols, tiled, stream=None):
    """Row-major block scales -> the tiled layout the GEMMs read (rows % 128 == 0, scale_cols % 4 == 0)."""
    _check("moe_pack_scales", lib().moe_pack_scales(_ptr(rowmajor), rows, scale_cols, _ptr(tiled), _stream(stream)))


def moe_poll_device_status(ws, stream=None) -> int:
    """Synchronises the stream; returns the status code (0 = no timeout)."""
    return int(lib().moe_poll_device_status(_ptr(ws), _stream(stream)))


def moe_debug_bounds_status(stream=None, with_site=False):
    """(status, checked[, site]): synchronises the stream and reads / clears the index-check flags
    of the bounds-checked build (status 8 = MOE_ERR_BOUNDS: a check failed and its access was
    skipped; site = the source line of a failed check); checked = 0 for the normal build, which
    has no checks."""
    c, site = ctypes.c_int(0), ctypes.c_int(0)
    st = int(lib().moe_debug_bounds_status(_stream(stream), ctypes.byref(c), ctypes.byref(site)))
    return (st, c.value, site.value) if with_site else (st, c.value)


def moe_status_string(status: int) -> str:
    """The library's text for a status code."""
    return lib().moe_status_string(status).decode()
