"""The prefill router (T > 256): tensor-core logits nominate the candidates,
which are recomputed on CUDA cores.  Checks that the tensor-core logits stay
far inside the error the candidate margin assumes (2^-11 ||x|| ||w_e||; the
candidates' entries of the scratch hold their recomputed logits, closer
still), that routing matches the oracle on small shapes with ragged token and
expert tiles, with outlier tokens, and through the standalone moe_route call,
and the degenerate case where every expert is a candidate."""
import numpy as np
import pytest

import oracle
import parity
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402
from synth.gpu_workload import GpuWorkload  # noqa: E402

ASSUMED_GAMMA = 2.0 ** -11   # the margin the library's candidate test assumes
U = dict(outlier_frac=0.0, bias="uniform")
TC_SMALL = {
    # 5 token tiles (the last one 88 rows), one 48-expert tile
    "tc_ragged_nvfp4": dict(T=600, H=512, E=48, k=4, F=256, fmt="nvfp4", seed=16, **U),
    # two expert tiles (128 + 32), 2% outlier tokens (x20): wide candidate sets
    "tc_outliers_mxfp8": dict(T=520, H=384, E=160, k=6, F=128, fmt="mxfp8", seed=17, outlier_frac=0.02,
                              bias="uniform"),
    # more than two waves of 128-expert tiles: 192-expert tiles (192 + 192 +
    # 16, the last one partial), 102 token tiles (the last one 72 rows)
    "tc_wide_nvfp4": dict(T=13000, H=256, E=400, k=8, F=256, fmt="nvfp4", seed=18, **U),
}


def tc_logits(gw):
    T, E = gw.w["T"], gw.w["E"]
    return gw.ws_view("logits", torch.float32, T * E).view(T, E).cpu().numpy().astype(np.float64)


def route_gpu(gw):
    T, k = gw.w["T"], gw.w["k"]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(gw.cfg, gw.x, gw.w_router, gw.bias, idx, wts, gw.ws)
    torch.cuda.synchronize()
    assert moe.moe_poll_device_status(gw.ws) == 0
    return idx.cpu().numpy(), wts.cpu().numpy()


@pytest.mark.parametrize("name", list(TC_SMALL) + ["prefill4096_nvfp4"])
def test_tc_logits_far_inside_assumed_bound(name):
    spec = TC_SMALL.get(name, name)
    gw = GpuWorkload(spec, torch, with_weights=False)
    w, T = gw.w, gw.w["T"]
    route_gpu(gw)
    rows = np.arange(T) if T <= 1024 else np.sort(np.random.default_rng(7).choice(T, 128, replace=False))
    x = synth.x_rows(w, rows)
    wr = synth.router_weight(w)
    ref = oracle.router_logits(x, wr)[0]
    xn = np.linalg.norm(oracle.bf16_bits_to_f32(x).astype(np.float64), axis=1)
    wn = np.linalg.norm(oracle.bf16_bits_to_f32(wr).astype(np.float64), axis=1)
    ratio = np.abs(tc_logits(gw)[rows] - ref) / (xn[:, None] * wn[None, :])
    print(name, "max |l_tc - l| / (||x|| ||w||) =", ratio.max(), "log2", np.log2(ratio.max()))
    assert ratio.max() < ASSUMED_GAMMA / 64


@pytest.mark.parametrize("name", list(TC_SMALL))
def test_tc_router_matches_oracle(name):
    gw = GpuWorkload(TC_SMALL[name], torch, with_weights=False)
    w, k = gw.w, gw.w["k"]
    idx, wts = route_gpu(gw)
    ro = oracle.route(synth.x_rows(w, np.arange(w["T"])), synth.router_weight(w), synth.router_bias(w), k)
    ties = parity.check_topk(idx, ro["idx"], ro["keys"], ro["absdot"])
    same = [i for i in range(w["T"]) if i not in ties]
    assert np.abs(wts[same] - ro["w"][same]).max() <= parity.W_TOL
    assert np.allclose(wts.sum(1), 1.0, atol=1e-5)
    print(name, "near ties", len(ties))


@pytest.mark.parametrize("E", [48, 384])
def test_tc_router_every_expert_a_candidate(E):
    # zero tokens and a zero bias: every logit is 0, every key 1/2, so every
    # expert is a candidate and the ties go to the lowest indices: experts
    # 0 .. k-1 with weight 1/k each (routed_scale 2: 2/k)
    spec = dict(T=300, H=512, E=E, k=8, F=256, fmt="nvfp4", seed=65, **U)
    gw = GpuWorkload(spec, torch, with_weights=False, routed_scale=2.0)
    gw.x.zero_()
    gw.bias.zero_()
    idx, wts = route_gpu(gw)
    assert (idx == np.arange(8, dtype=np.int32)[None, :]).all()
    assert np.allclose(wts, 2.0 / 8, rtol=0, atol=1e-7)
