"""moe_route_noalloc: the router for callers that cannot allocate device memory
when they route (captured graph regions, plugins without their host's
allocator, runtimes that forbid allocation after start-up).  On two calls in
a row (the second reuses the library's fixed scratch array) it must give the
same results as moe_route, which uses a caller workspace, and the oracle's
top-k (bit-exact outside certified near-ties, weights within W_TOL); its
status word must read clean; batches whose scratch would not fit are refused.

Kept in a file that pytest collects last: should it fail, a run that stops at
the first failure has already run every other test."""
import numpy as np
import pytest

import oracle
import parity
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402
from synth.gpu_workload import GpuWorkload  # noqa: E402


def shape(T, seed, **kw):
    return dict(T=T, H=4608, E=384, k=8, F=2304, fmt="nvfp4", seed=seed, outlier_frac=0.0, bias="uniform", **kw)


CASES = {
    "decode64_nvfp4": ("decode64_nvfp4", {}),
    "decode192_mxfp8_outliers": ("decode192_mxfp8_outliers", {}),
    "tiny_mxfp8": ("tiny_mxfp8", {}),
    "prefill2048": (shape(2048, 5), {}),
    # the largest batch the scratch holds at E = 384 (tensor-core router)
    "prefill2729_edge": (shape(2729, 6), {}),
    # the router options: weights from the biased keys, scaled
    "decode64_options": ("decode64_nvfp4", dict(bias_in_weights=1, routed_scale=2.5)),
    "prefill600_options": (shape(600, 7), dict(bias_in_weights=1, routed_scale=2.5)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_router_matches_moe_route_and_oracle_twice(name):
    spec, opts = CASES[name]
    gw = GpuWorkload(spec, torch, with_weights=False, **opts)
    w, T, k = gw.w, gw.w["T"], gw.w["k"]
    ref_idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ref_w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(gw.cfg, gw.x, gw.w_router, gw.bias, ref_idx, ref_w, gw.ws)
    # the oracle on every token (a seeded sample of 512 at the edge batch)
    rows = np.arange(T) if T <= 2048 else np.sort(np.random.default_rng(9).choice(T, 512, replace=False))
    ro = oracle.route(synth.x_rows(w, rows), synth.router_weight(w), synth.router_bias(w), k,
                      bias_in_weights=bool(opts.get("bias_in_weights", 0)),
                      routed_scale=opts.get("routed_scale", 1.0))
    for _ in range(2):
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        wt = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
        moe.moe_route_noalloc(gw.cfg, gw.x, gw.w_router, gw.bias, idx, wt)
        assert moe.moe_route_noalloc_poll_status() == 0
        assert torch.equal(idx, ref_idx)
        assert float((wt - ref_w).abs().max()) <= parity.W_TOL
        gi, gwt = idx.cpu().numpy()[rows], wt.cpu().numpy()[rows].astype(np.float64)
        ties = parity.check_topk(gi, ro["idx"], ro["keys"], ro["absdot"])
        same = [i for i in range(len(rows)) if i not in ties]
        assert np.abs(gwt[same] - ro["w"][same]).max() <= parity.W_TOL
        assert np.allclose(gwt.sum(1), opts.get("routed_scale", 1.0), atol=1e-5)


def test_noalloc_router_rejects_batches_beyond_its_scratch():
    big = moe.make_config(2730, 4608, 384, 8, 2304, "nvfp4")     # 64 + 2730*384 + 384 floats > 2^20
    x = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_noalloc(big, x, x, x, x, x)
    assert ei.value.status == 4     # MOE_ERR_WORKSPACE_TOO_SMALL
