"""Parity rules between the CUDA path and the oracle, shared by the GPU tests,
the smoke check and the benchmark's correctness gate.

* Codes, scales, globals, dispatch and (outside certified near-ties) top-k
  indices: bit-exact.
* Top-k near-ties: the GPU's logits carry at most ROUTER_GAMMA * sum|x w| of
  rounding error (fp32 chunks of 32, Kahan across chunks: see the library's
  router); the sigmoid and bias add in fp32 add at most KEY_EPS.  A token may
  differ from the oracle only if the GPU's ordered choice is consistent with
  keys perturbed within those bounds; the oracle is then re-run with the GPU's
  choice for that token.
* Layer output (bf16) against the unrounded fp64 oracle: max|err| <=
  OUT_TOL * rms(reference).
"""
from __future__ import annotations

import numpy as np

U = 2.0 ** -24
ROUTER_GAMMA = 40 * U
KEY_EPS = 1e-6
OUT_TOL = 2e-2
W_TOL = 1e-4


def key_bounds(absdot_row: np.ndarray) -> np.ndarray:
    """Per-expert bound on |key_gpu - key| (sigmoid slope <= 1/4)."""
    return 0.25 * ROUTER_GAMMA * absdot_row + KEY_EPS


def consistent_choice(keys: np.ndarray, delta: np.ndarray, choice) -> bool:
    """Can keys perturbed by at most delta rank `choice` (ordered) as top-k?"""
    choice = [int(e) for e in choice]
    hi = keys + delta
    lo = keys - delta
    cur = np.inf
    for e in choice:
        v = min(hi[e], cur)
        if v < lo[e]:
            return False
        cur = v
    rest = np.ones(len(keys), bool)
    rest[choice] = False
    return bool(np.all(lo[rest] <= cur))


def check_topk(gpu_idx: np.ndarray, orc_idx: np.ndarray, keys: np.ndarray, absdot: np.ndarray, rows=None):
    """Returns {row: gpu_choice} of certified near-ties; raises on a real mismatch."""
    ties = {}
    rows = range(len(gpu_idx)) if rows is None else rows
    for i in rows:
        if np.array_equal(gpu_idx[i], orc_idx[i]):
            continue
        d = key_bounds(absdot[i])
        if not consistent_choice(keys[i], d, gpu_idx[i]):
            raise AssertionError(f"top-k mismatch at row {i}: gpu {list(gpu_idx[i])} oracle {list(orc_idx[i])} "
                                 f"keys gpu-choice {keys[i][gpu_idx[i]]} oracle-choice {keys[i][orc_idx[i]]}")
        ties[i] = gpu_idx[i].copy()
    return ties


def bf16_to_f64(t) -> np.ndarray:
    """torch bf16 tensor -> fp64 numpy."""
    import torch
    return t.to(torch.float32).cpu().numpy().astype(np.float64)


# the compact y rows keep 11 significant bits: |decoded - y| <= Y16_REL |y|
Y16_REL = 2.0 ** -11


def y_rows_f64(moe, cfg, raw, rows) -> np.ndarray:
    """fp64 values of the given y rows of a y buffer (bytes, on the device)
    in cfg.y_format: fp32 as stored, or the fp16 codes decoded with their
    exponents by the oracle's rule."""
    import torch
    import oracle
    idx = torch.as_tensor(np.asarray(rows, np.int64), device=raw.device)
    v = moe.y_rows(cfg, raw)
    if cfg.y_format == moe.Y_FP32:
        return v[idx].cpu().numpy().astype(np.float64)
    codes, ex = v
    return oracle.decode_y16(codes[idx].view(torch.int16).cpu().numpy().view(np.uint16), ex[idx].cpu().numpy())


def y_rel(moe, cfg) -> float:
    """Relative rounding of the y format (0 for fp32)."""
    return 0.0 if cfg.y_format == moe.Y_FP32 else Y16_REL


def out_error(gpu: np.ndarray, ref: np.ndarray):
    err = np.abs(gpu - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(err.max()), rms


def check_output(gpu: np.ndarray, ref: np.ndarray, tol: float = OUT_TOL):
    mx, rms = out_error(gpu, ref)
    assert mx <= tol * rms, f"max|err| {mx:.4g} > {tol} * rms {rms:.4g}"
    return mx / rms


def check_output_rowwise(gpu: np.ndarray, ref: np.ndarray, tol: float = OUT_TOL):
    worst = 0.0
    for r in range(ref.shape[0]):
        mx, rms = out_error(gpu[r], ref[r])
        worst = max(worst, mx / rms)
    assert worst <= tol, f"row-wise max|err|/rms {worst:.4g} > {tol}"
    return worst
