"""Seeded synthetic inputs for the routed MoE layer (shared by the oracle side
and the GPU side; holds none of the layer's arithmetic).

The generator itself is defined once, in ``synth_gen.h``: a SplitMix64 hash of
(seed, tensor id, element index), and an Irwin-Hall(12) normal stand-in that is
an exact integer rounded to fp32 once.  ``synth_host.c`` fills host arrays,
``synth_dev.cu`` fills device arrays; both give the same bits.

Input recipe (the pages measure whole-model serving, not a layer, so these
seeded tensors stand in for real activations and trained weights):

* x[t,h] = bf16(z), z ~ Irwin-Hall stand-in for N(0,1); outlier rows (a seeded
  choice of round(frac*T) tokens) are bf16(20*z).
* W_r[e,h] = bf16(z * fp32(1/sqrt(H))).
* bias b[e] = fp32(-0.1 + 0.2*u), u a 24-bit uniform; or the Zipf recipe:
  b[e] = -c*s*ln(rank_e) with s = 1.1, rank a seeded permutation, and the 32
  least popular experts at -2 so that they receive no tokens; or "hot": the
  uniform bias + 10 on the first k experts (every token routes to them).
* expert master weights W[e,n,k] = z * fp32(1/sqrt(fan_in)), fp32, quantised
  afterwards by the method's own encoder.
"""
from __future__ import annotations

import ctypes
import hashlib
import math
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()

# Tensor ids (mirror of the enum in synth_gen.h).
T_X, T_ROUTER, T_BIAS, T_OUTLIER, T_RANK, T_GATE, T_UP, T_DOWN = 1, 2, 3, 4, 5, 10, 11, 12

# Zipf recipe constants.  ZIPF_C was picked once with the oracle's router
# (synth/calibrate_zipf.py) so that the most popular expert receives about ten
# times the mean load at T=16384.
ZIPF_S = 1.1
ZIPF_C = 0.036
ZIPF_N_COLD = 32
ZIPF_COLD_BIAS = -2.0
OUTLIER_SCALE = 20.0

# The five seeded workloads: a tiny correctness case, two decode batches and
# two prefill chunks in the layer shape of Inkling 2 Small.
WORKLOADS = {
    "tiny_mxfp8": dict(T=8, H=256, E=16, k=2, F=128, fmt="mxfp8", seed=0,
                       outlier_frac=0.0, bias="uniform"),
    "decode64_nvfp4": dict(T=64, H=4608, E=384, k=8, F=2304, fmt="nvfp4", seed=1,
                           outlier_frac=0.0, bias="uniform"),
    "decode192_mxfp8_outliers": dict(T=192, H=4608, E=384, k=8, F=2304, fmt="mxfp8", seed=2,
                                     outlier_frac=0.01, bias="uniform"),
    "prefill4096_nvfp4": dict(T=4096, H=4608, E=384, k=8, F=2304, fmt="nvfp4", seed=3,
                              outlier_frac=0.0, bias="uniform"),
    "prefill16384_mxfp8_zipf": dict(T=16384, H=4608, E=384, k=8, F=2304, fmt="mxfp8", seed=4,
                                    outlier_frac=0.0, bias="zipf"),
    # single-user and small-batch decode (latency-bound: few experts, few tiles)
    "decode1_nvfp4": dict(T=1, H=4608, E=384, k=8, F=2304, fmt="nvfp4", seed=31,
                          outlier_frac=0.0, bias="uniform"),
    "decode8_nvfp4": dict(T=8, H=4608, E=384, k=8, F=2304, fmt="nvfp4", seed=32,
                          outlier_frac=0.0, bias="uniform"),
    "decode32_mxfp8": dict(T=32, H=4608, E=384, k=8, F=2304, fmt="mxfp8", seed=33,
                           outlier_frac=0.0, bias="uniform"),
    # smaller cases of the same kernels for detailed profiler captures (a few
    # GB resident, touched weights still far above the L2 size)
    "profile_decode16_nvfp4_e96": dict(T=16, H=4608, E=96, k=8, F=2304, fmt="nvfp4", seed=21,
                                       outlier_frac=0.0, bias="uniform"),
    # one token: 8 touched experts, one wave of 144 gate/up and 144 down tiles
    "profile_decode1_nvfp4_e64": dict(T=1, H=4608, E=64, k=8, F=2304, fmt="nvfp4", seed=24,
                                      outlier_frac=0.0, bias="uniform"),
    "profile_prefill2048_mxfp8_e64": dict(T=2048, H=4608, E=64, k=8, F=2304, fmt="mxfp8", seed=22,
                                          outlier_frac=0.0, bias="uniform"),
    "profile_prefill2048_nvfp4_e64": dict(T=2048, H=4608, E=64, k=8, F=2304, fmt="nvfp4", seed=23,
                                          outlier_frac=0.0, bias="uniform"),
}


def workload_spec(spec) -> dict:
    """A workload dict: the name of one above, or a dict of the same keys."""
    return dict(WORKLOADS[spec]) if isinstance(spec, str) else dict(spec)


def inv_sqrt_f32(n: int) -> float:
    """fp32(1/sqrt(n)), computed in fp64 and rounded once."""
    return float(np.float32(1.0 / math.sqrt(n)))


def n_outliers(T: int, frac: float) -> int:
    return int(math.floor(frac * T + 0.5))


def _build_one(out_name: str, src_name: str, cmd: list, libs=()) -> str:
    """Build one library unless a stamp beside it holds the hash of its
    sources, the command and the machine it was built for."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, out_name)
    src = os.path.join(_HERE, src_name)
    h = hashlib.sha256()
    for f in (src, os.path.join(_HERE, "synth_gen.h")):
        h.update(open(f, "rb").read())
    h.update(" ".join(cmd + list(libs) + [platform.machine()]).encode())
    key, stamp = h.hexdigest(), out + ".key"
    if not (os.path.exists(out) and os.path.exists(stamp) and open(stamp).read().strip() == key):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(cmd + ["-o", tmp, src] + list(libs))
        os.replace(tmp, out)
        with open(stamp, "w") as f:
            f.write(key + "\n")
    return out


def _build_host() -> str:
    return _build_one("libsynth_host.so", "synth_host.c",
                      ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared"], libs=["-lm"])


def _build_dev() -> str:
    return _build_one("libsynth_dev.so", "synth_dev.cu",
                      ["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-Xcompiler", "-fPIC",
                       "-shared"])


_host = None
_dev = None


def host_lib():
    global _host
    with _lock:
        if _host is None:
            lib = ctypes.CDLL(_build_host())
            P = ctypes.c_void_p
            i64, u64 = ctypes.c_int64, ctypes.c_uint64
            lib.synth_host_x_rows.argtypes = [u64, i64, P, i64, P, ctypes.c_float, P]
            lib.synth_host_router.argtypes = [u64, i64, i64, ctypes.c_float, P]
            lib.synth_host_bias_uniform.argtypes = [u64, i64, ctypes.c_double, ctypes.c_double, P]
            lib.synth_host_expert_rank.argtypes = [u64, i64, P]
            lib.synth_host_bias_zipf.argtypes = [u64, i64, ctypes.c_double, ctypes.c_double, i64,
                                                 ctypes.c_double, P]
            lib.synth_host_outlier_flags.argtypes = [u64, i64, i64, P]
            lib.synth_host_expert_matrix.argtypes = [u64, ctypes.c_int, i64, i64, i64, ctypes.c_float, P]
            lib.synth_host_normals.argtypes = [u64, ctypes.c_int, i64, i64, P]
            _host = lib
        return _host


def dev_lib():
    global _dev
    with _lock:
        if _dev is None:
            lib = ctypes.CDLL(_build_dev())
            P = ctypes.c_void_p
            i64, u64 = ctypes.c_int64, ctypes.c_uint64
            lib.synth_dev_x.argtypes = [u64, i64, i64, P, ctypes.c_float, P, P]
            lib.synth_dev_router.argtypes = [u64, i64, i64, ctypes.c_float, P, P]
            lib.synth_dev_expert_matrices.argtypes = [u64, ctypes.c_int, i64, i64, i64, i64,
                                                      ctypes.c_float, P, P]
            for f in (lib.synth_dev_x, lib.synth_dev_router, lib.synth_dev_expert_matrices):
                f.restype = ctypes.c_int
            _dev = lib
        return _dev


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------
# host-side inputs (numpy)
# ----------------------------------------------------------------------------

def normals(seed: int, tensor: int, i0: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    host_lib().synth_host_normals(seed, tensor, i0, n, _ptr(out))
    return out


def outlier_flags(w: dict) -> np.ndarray:
    T = w["T"]
    flags = np.zeros(T, np.uint8)
    host_lib().synth_host_outlier_flags(w["seed"], T, n_outliers(T, w["outlier_frac"]), _ptr(flags))
    return flags


def x_rows(w: dict, rows) -> np.ndarray:
    """bf16 bit patterns (uint16) of x for the given token rows, [len(rows), H]."""
    rows = np.ascontiguousarray(np.asarray(rows, np.int64))
    flags = outlier_flags(w)
    out = np.empty((len(rows), w["H"]), np.uint16)
    host_lib().synth_host_x_rows(w["seed"], w["H"], _ptr(rows), len(rows), _ptr(flags),
                                 OUTLIER_SCALE, _ptr(out))
    return out


def router_weight(w: dict) -> np.ndarray:
    out = np.empty((w["E"], w["H"]), np.uint16)
    host_lib().synth_host_router(w["seed"], w["E"], w["H"], inv_sqrt_f32(w["H"]), _ptr(out))
    return out


def router_bias(w: dict) -> np.ndarray:
    out = np.empty(w["E"], np.float32)
    if w["bias"] == "uniform":
        host_lib().synth_host_bias_uniform(w["seed"], w["E"], -0.1, 0.1, _ptr(out))
    elif w["bias"] == "hot":
        # degenerate routing: the first k experts outrank every other key, so
        # each of them receives every token and the rest none
        host_lib().synth_host_bias_uniform(w["seed"], w["E"], -0.1, 0.1, _ptr(out))
        out[:w["k"]] += np.float32(10.0)
    elif w["bias"] == "zipf":
        host_lib().synth_host_bias_zipf(w["seed"], w["E"], ZIPF_C, ZIPF_S, ZIPF_N_COLD,
                                        ZIPF_COLD_BIAS, _ptr(out))
    else:
        raise ValueError(w["bias"])
    return out


def expert_rank(w: dict) -> np.ndarray:
    out = np.empty(w["E"], np.int32)
    host_lib().synth_host_expert_rank(w["seed"], w["E"], _ptr(out))
    return out


def expert_matrix(w: dict, which: str, e: int) -> np.ndarray:
    """fp32 master values of one expert matrix: gate/up [F,H], down [H,F]."""
    tensor, N, K = {"gate": (T_GATE, w["F"], w["H"]), "up": (T_UP, w["F"], w["H"]),
                    "down": (T_DOWN, w["H"], w["F"])}[which]
    out = np.empty((N, K), np.float32)
    host_lib().synth_host_expert_matrix(w["seed"], tensor, e, N, K, inv_sqrt_f32(K), _ptr(out))
    return out


# ----------------------------------------------------------------------------
# device-side inputs (torch tensors on cuda)
# ----------------------------------------------------------------------------

def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"synth device fill {what} failed: cuda error {rc}")


def dev_x(w: dict, torch, device="cuda"):
    T, H = w["T"], w["H"]
    x = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    flags = torch.from_numpy(outlier_flags(w)).to(device)
    st = torch.cuda.current_stream().cuda_stream
    _check(dev_lib().synth_dev_x(w["seed"], T, H, flags.data_ptr(), OUTLIER_SCALE, x.data_ptr(), st), "x")
    return x


def dev_router_weight(w: dict, torch, device="cuda"):
    E, H = w["E"], w["H"]
    out = torch.empty((E, H), dtype=torch.bfloat16, device=device)
    st = torch.cuda.current_stream().cuda_stream
    _check(dev_lib().synth_dev_router(w["seed"], E, H, inv_sqrt_f32(H), out.data_ptr(), st), "router")
    return out


def dev_expert_matrices(w: dict, which: str, e0: int, ne: int, torch, out=None, device="cuda"):
    tensor, N, K = {"gate": (T_GATE, w["F"], w["H"]), "up": (T_UP, w["F"], w["H"]),
                    "down": (T_DOWN, w["H"], w["F"])}[which]
    if out is None:
        out = torch.empty((ne, N, K), dtype=torch.float32, device=device)
    st = torch.cuda.current_stream().cuda_stream
    _check(dev_lib().synth_dev_expert_matrices(w["seed"], tensor, e0, ne, N, K, inv_sqrt_f32(K),
                                               out.data_ptr(), st), which)
    return out
