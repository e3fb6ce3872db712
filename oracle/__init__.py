"""CPU oracle of the routed block-scaled MoE layer — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and the
two share no code; only the seeded input generator (``synth``) serves both.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 accumulation, fp32
correctly rounded quantiser steps); this module marshals numpy arrays and
strings the steps together in the order the pages name them: route (sigmoid,
bias, top-k), dispatch, quantised expert GEMMs with the capped SwiGLU between
them, and the weighted combine.

Every function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_lib = None

FMT_NVFP4, FMT_MXFP8 = 0, 1


_CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared"]


def build() -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction).  The
    build is skipped only when a stamp beside the library holds the hash of
    the source, the flags and the machine it was built for."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "libmoe_oracle.so")
    src = os.path.join(_HERE, "moe_oracle.c")
    h = hashlib.sha256(open(src, "rb").read())
    h.update(" ".join(_CFLAGS + [platform.machine()]).encode())
    key, stamp = h.hexdigest(), out + ".key"
    if not (os.path.exists(out) and os.path.exists(stamp) and open(stamp).read().strip() == key):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
        with open(stamp, "w") as f:
            f.write(key + "\n")
    return out


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, i64, d, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
            u8 = ctypes.c_uint8
            L.orc_e2m1_value.argtypes = [u8]; L.orc_e2m1_value.restype = d
            L.orc_e2m1_encode.argtypes = [ctypes.c_float]; L.orc_e2m1_encode.restype = u8
            L.orc_e4m3_value.argtypes = [u8]; L.orc_e4m3_value.restype = d
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]; L.orc_e4m3_encode.restype = u8
            L.orc_e8m0_value.argtypes = [u8]; L.orc_e8m0_value.restype = d
            L.orc_bf16_value.argtypes = [ctypes.c_uint16]; L.orc_bf16_value.restype = d
            L.orc_bf16_from_f64.argtypes = [d]; L.orc_bf16_from_f64.restype = ctypes.c_uint16
            L.orc_nvfp4_quantize.argtypes = [P, i64, i64, c_int, P, P, P]
            L.orc_nvfp4_decode.argtypes = [P, P, P, i64, i64, c_int, P]
            L.orc_mxfp8_quantize.argtypes = [P, i64, i64, c_int, P, P]
            L.orc_mxfp8_decode.argtypes = [P, P, i64, i64, P]
            L.orc_router_logits.argtypes = [i64, i64, i64, P, P, P, P]
            L.orc_router_select.argtypes = [i64, i64, i64, P, P, c_int, d, P, P, P]
            L.orc_dispatch.argtypes = [i64, i64, i64, P, P, P, P, P]
            L.orc_expert_ffn.argtypes = [c_int, i64, i64, d, c_int, c_int, P, P, P, i64, P, P, P, P, P, P, P]
            L.orc_nvfp4_quantize_static.argtypes = [P, i64, i64, P, P, P, P]
            L.orc_combine.argtypes = [i64, i64, i64, P, P, P, P]
            L.orc_num_threads.restype = c_int
            _lib = L
        return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(lib().orc_num_threads())


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(v)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(v)


def e8m0_value(code: int) -> float:
    return lib().orc_e8m0_value(code)


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(bits)


def bf16_from_f64(v: float) -> int:
    return lib().orc_bf16_from_f64(v)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# quantisers
# ----------------------------------------------------------------------------

def nvfp4_quantize(v: np.ndarray, per_tensor: bool = False):
    v = _c(v, np.float32)
    rows, K = v.shape
    assert K % 16 == 0
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows, K // 16), np.uint8)
    g = np.empty(1 if per_tensor else rows, np.float32)
    lib().orc_nvfp4_quantize(_p(v), rows, K, int(per_tensor), _p(codes), _p(sf), _p(g))
    return codes, sf, g


def nvfp4_quantize_static(v: np.ndarray, g_rows):
    """Rows of v with given decode factors g_rows (static activation globals:
    G = 1/g in fp32, block maxima beyond 2688 g saturate)."""
    v = _c(v, np.float32)
    rows, K = v.shape
    assert K % 16 == 0
    g_rows = _c(np.broadcast_to(np.asarray(g_rows, np.float32), (rows,)), np.float32)
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows, K // 16), np.uint8)
    g = np.empty(rows, np.float32)
    lib().orc_nvfp4_quantize_static(_p(v), rows, K, _p(g_rows), _p(codes), _p(sf), _p(g))
    return codes, sf, g


def nvfp4_decode(codes, sf, g, per_tensor: bool = False) -> np.ndarray:
    codes, sf, g = _c(codes, np.uint8), _c(sf, np.uint8), _c(g, np.float32)
    rows = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    lib().orc_nvfp4_decode(_p(codes), _p(sf), _p(g), rows, K, int(per_tensor), _p(out))
    return out


def mxfp8_quantize(v: np.ndarray, mode: int = 0):
    v = _c(v, np.float32)
    rows, K = v.shape
    assert K % 32 == 0
    codes = np.empty((rows, K), np.uint8)
    sf = np.empty((rows, K // 32), np.uint8)
    lib().orc_mxfp8_quantize(_p(v), rows, K, int(mode), _p(codes), _p(sf))
    return codes, sf


def mxfp8_decode(codes, sf) -> np.ndarray:
    codes, sf = _c(codes, np.uint8), _c(sf, np.uint8)
    rows, K = codes.shape
    out = np.empty((rows, K), np.float64)
    lib().orc_mxfp8_decode(_p(codes), _p(sf), rows, K, _p(out))
    return out


def quantize(fmt: str, v: np.ndarray, per_tensor: bool = False, mx_mode: int = 0):
    """Quantise rows of v; returns (codes, scales, globals-or-None)."""
    if fmt == "nvfp4":
        return nvfp4_quantize(v, per_tensor)
    codes, sf = mxfp8_quantize(v, mx_mode)
    return codes, sf, None


def decode(fmt: str, codes, sf, g, per_tensor: bool = False) -> np.ndarray:
    if fmt == "nvfp4":
        return nvfp4_decode(codes, sf, g, per_tensor)
    return mxfp8_decode(codes, sf)


# ----------------------------------------------------------------------------
# router, dispatch, expert FFN, combine
# ----------------------------------------------------------------------------

def router_logits(x_bf16: np.ndarray, wr_bf16: np.ndarray):
    """fp64 logits [T,E] and sum_h |x_h * w_eh| [T,E] (for error bounds)."""
    x, wr = _c(x_bf16, np.uint16), _c(wr_bf16, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    logits = np.empty((T, E), np.float64)
    absdot = np.empty((T, E), np.float64)
    lib().orc_router_logits(T, H, E, _p(x), _p(wr), _p(logits), _p(absdot))
    return logits, absdot


def router_select(logits: np.ndarray, bias: np.ndarray, k: int, bias_in_weights: bool = False,
                  routed_scale: float = 1.0):
    logits, bias = _c(logits, np.float64), _c(bias, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    keys = np.empty((T, E), np.float64)
    lib().orc_router_select(T, E, k, _p(logits), _p(bias), int(bias_in_weights), routed_scale,
                            _p(idx), _p(w), _p(keys))
    return idx, w, keys


def route(x_bf16, wr_bf16, bias, k, bias_in_weights=False, routed_scale=1.0):
    logits, absdot = router_logits(x_bf16, wr_bf16)
    idx, w, keys = router_select(logits, bias, k, bias_in_weights, routed_scale)
    return dict(idx=idx, w=w, keys=keys, logits=logits, absdot=absdot)


def dispatch(idx: np.ndarray, E: int):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    pair_pos = np.empty((T, k), np.int32)
    lib().orc_dispatch(T, E, k, _p(idx), _p(counts), _p(offsets), _p(perm), _p(pair_pos))
    return dict(counts=counts, offsets=offsets, perm=perm, pair_pos=pair_pos)


def expert_ffn(fmt: str, Wg, Wu, Wd, a, cap: float = 10.0, h_round_bf16: bool = True, mx_mode: int = 0,
               h_static_g=None):
    """One expert over n pairs.  Wg, Wu [F,H], Wd [H,F], a [n,H] fp64 decoded.
    h_static_g: NVFP4 static h global of this expert (act_global_mode 1), or None.
    Returns y [n,H] fp64, h_bf16 [n,F], and h's codes / scales / globals."""
    Wg, Wu, Wd, a = (_c(m, np.float64) for m in (Wg, Wu, Wd, a))
    F, H = Wg.shape
    n = a.shape[0]
    f = FMT_NVFP4 if fmt == "nvfp4" else FMT_MXFP8
    y = np.empty((n, H), np.float64)
    hb = np.empty((n, F), np.uint16)
    hq_codes = np.empty((n, F // 2 if f == FMT_NVFP4 else F), np.uint8)
    hq_sf = np.empty((n, F // 16 if f == FMT_NVFP4 else F // 32), np.uint8)
    hq_g = np.empty(n, np.float32)
    hs = None if h_static_g is None else np.array([h_static_g], np.float32)
    lib().orc_expert_ffn(f, H, F, float(cap), int(h_round_bf16), int(mx_mode), _p(Wg), _p(Wu), _p(Wd), n,
                         _p(a), _p(y), _p(hb), _p(hq_codes), _p(hq_sf), _p(hq_g), _p(hs))
    return dict(y=y, h_bf16=hb, hq_codes=hq_codes, hq_sf=hq_sf, hq_g=hq_g)


def combine(w: np.ndarray, pair_pos: np.ndarray, y: np.ndarray) -> np.ndarray:
    w, pair_pos, y = _c(w, np.float64), _c(pair_pos, np.int32), _c(y, np.float64)
    T, k = w.shape
    H = y.shape[1]
    out = np.empty((T, H), np.float64)
    lib().orc_combine(T, k, H, _p(w), _p(pair_pos), _p(y), _p(out))
    return out


def encode_y16(y32: np.ndarray):
    """The expert outputs y (fp32 rows [n, H]) in the compact exchange format
    between the down GEMM and the combine.  The pages fix no format for y
    (the MegaMoE paragraph of the Inkling-2-Small cookbook keeps it inside
    the fused unit), so this is a reading of the library's own: per row and
    32-feature block, amax = max |y|; e = floor(log2 amax) - 14, not below
    -110, and 0 for an all-zero block; code = fp16(y * 2^-e), rounded to
    nearest even (the block maximum lands in [2^14, 2^15)).
    Returns (codes uint16 [n, H], exponents int8 [n, H/32])."""
    y = np.asarray(y32, np.float32)
    n, H = y.shape
    b = y.reshape(n, H // 32, 32).astype(np.float64)
    amax = np.abs(b).max(axis=2)
    _, ex = np.frexp(amax)                 # amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    e = np.where(amax > 0, np.maximum(ex - 1 - 14, -110), 0).astype(np.int32)
    scaled = b * np.exp2(-e.astype(np.float64))[..., None]      # exact: a power of two
    codes = scaled.astype(np.float16).view(np.uint16).reshape(n, H)
    return codes, e.astype(np.int8)


def decode_y16(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    """Values of encode_y16's format: code * 2^e (fp64, exact)."""
    codes = np.asarray(codes, np.uint16)
    n, H = codes.shape
    v = codes.view(np.float16).astype(np.float64).reshape(n, H // 32, 32)
    return (v * np.exp2(np.asarray(exps, np.float64))[..., None]).reshape(n, H)


# ----------------------------------------------------------------------------
# the layer over (a sample of) a seeded workload
# ----------------------------------------------------------------------------

def quantized_expert(w: dict, e: int, mx_mode: int = 0):
    """The encoded weights of one expert, from the seeded master values:
    dict(gate/up/down -> (codes, scales, global-or-None)).  NVFP4 uses one
    global per (expert, matrix)."""
    import synth
    out = {}
    for which in ("gate", "up", "down"):
        m = synth.expert_matrix(w, which, e)
        out[which] = quantize(w["fmt"], m, per_tensor=True, mx_mode=mx_mode)
    return out


def decoded_expert(w: dict, q: dict):
    return {which: decode(w["fmt"], *q[which], per_tensor=True) for which in ("gate", "up", "down")}


def quantize_x(w: dict, x_bf16: np.ndarray, mx_mode: int = 0):
    """Per-token activation quantisation over the full hidden width."""
    return quantize(w["fmt"], bf16_bits_to_f32(x_bf16), per_tensor=False, mx_mode=mx_mode)


def selected_weights(logits_row: np.ndarray, bias: np.ndarray, sel, bias_in_weights: bool = False,
                     routed_scale: float = 1.0) -> np.ndarray:
    """Routing weights of one token for a given ordered choice of experts
    (used where a certified near-tie replaces the oracle's own choice):
    routed_scale * v_j / sum_i v_i over the chosen experts, v = the sigmoid
    score s (bias steers selection only) or the key s + b with
    bias_in_weights.  The same rule as the selection's weights."""
    sel = np.asarray(sel, np.int64)
    s = 1.0 / (1.0 + np.exp(-np.asarray(logits_row, np.float64)[sel]))
    v = s + np.asarray(bias, np.float32)[sel].astype(np.float64) if bias_in_weights else s
    den = 0.0
    for x in v:          # slot order, as the selection sums them
        den += x
    return routed_scale * (v / den)


def moe_layer(w: dict, tokens=None, idx_override=None, cap: float = 10.0, mx_mode: int = 0,
              expert_cache=None, keep_pairs: bool = False, inputs=None, max_pairs=None, act_static=None,
              bias_in_weights: bool = False, routed_scale: float = 1.0):
    """Run the whole layer for the given token rows (default: all T).

    idx_override: optional {token_row_index_in_sample: int32[k]} replacing the
    oracle's own top-k for certified near-tie tokens (their weights follow
    the same rule, selected_weights).
    bias_in_weights, routed_scale: the router options of moe_config.
    expert_cache: optional dict e -> quantized_expert(...) to reuse encodings.
    inputs: optional (x rows of the tokens, W_r, bias) already generated.
    max_pairs: compute only the first max_pairs (token, slot) pairs of the
    sample's dispatch order (a bounded sample of the work; the output rows are
    then partial sums).
    act_static: NVFP4 static activation globals [E, 2] (decode factors g_x,
    g_h per expert; act_global_mode 1): the x rows routed to expert e are
    encoded with g_x[e] and its h rows with g_h[e].
    Returns dict with x codes, routing, dispatch (over the sample), y per pair
    and the fp64 output [n, H].
    """
    import synth
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens, np.int64)
    if inputs is None:
        x = synth.x_rows(w, tokens)
        wr = synth.router_weight(w)
        bias = synth.router_bias(w)
    else:
        x, wr, bias = inputs
    r = route(x, wr, bias, k, bias_in_weights, routed_scale)
    idx = r["idx"].copy()
    if idx_override:
        for i, sel in idx_override.items():
            idx[i] = np.asarray(sel, np.int32)
            r["w"][i] = selected_weights(r["logits"][i], bias, idx[i], bias_in_weights, routed_scale)
    d = dispatch(idx, E)
    xq = quantize_x(w, x, mx_mode)
    a_all = decode(w["fmt"], *xq, per_tensor=False)
    P = len(tokens) * k
    y = np.zeros((P, H), np.float64)
    pairs = {}
    budget = P if max_pairs is None else int(max_pairs)
    for e in np.nonzero(d["counts"])[0]:
        e = int(e)
        if d["offsets"][e] >= budget:
            break
        if expert_cache is not None and e in expert_cache:
            q = expert_cache[e]
        else:
            q = quantized_expert(w, e, mx_mode)
            if expert_cache is not None:
                expert_cache[e] = q
        dec = decoded_expert(w, q)
        lo, hi = d["offsets"][e], min(d["offsets"][e + 1], budget)
        pids = d["perm"][lo:hi]
        rows = pids // k
        if act_static is None:
            a_e = a_all[rows]
            hs = None
        else:
            xs = nvfp4_quantize_static(bf16_bits_to_f32(x[rows]), act_static[e, 0])
            a_e = decode("nvfp4", *xs, per_tensor=False)
            hs = float(act_static[e, 1])
        res = expert_ffn(w["fmt"], dec["gate"], dec["up"], dec["down"], a_e, cap=cap, mx_mode=mx_mode,
                         h_static_g=hs)
        y[lo:hi] = res["y"]
        if keep_pairs:
            pairs[e] = res
    out = combine(r["w"], d["pair_pos"], y)
    return dict(tokens=tokens, x=x, xq=xq, route=r, idx=idx, dispatch=d, y=y, out=out, pairs=pairs)
