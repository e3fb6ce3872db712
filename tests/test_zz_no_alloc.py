"""moe_route_noalloc: the router for callers that cannot allocate device memory
when they route (captured graph regions, plugins without their host's
allocator, runtimes that forbid allocation after start-up).  It must give the
same results as moe_route, which uses a caller workspace, on two calls in a
row (the second call reuses the library's fixed scratch array), and refuse
batches whose scratch would not fit.

Kept in a file that pytest collects last: should it fail, a run that stops at
the first failure has already run every other test."""
import numpy as np
import pytest

import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402
from synth.gpu_workload import GpuWorkload  # noqa: E402


PREFILL2048 = dict(T=2048, H=4608, E=384, k=8, F=2304, fmt="nvfp4", seed=5, outlier_frac=0.0, bias="uniform")


@pytest.mark.parametrize("name", ["decode64_nvfp4", "decode192_mxfp8_outliers", "tiny_mxfp8", "prefill2048"])
def test_noalloc_router_matches_moe_route_twice(name):
    gw = GpuWorkload(PREFILL2048 if name == "prefill2048" else name, torch, with_weights=False)
    T, k = gw.w["T"], gw.w["k"]
    ref_idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ref_w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(gw.cfg, gw.x, gw.w_router, gw.bias, ref_idx, ref_w, gw.ws)
    for _ in range(2):
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
        moe.moe_route_noalloc(gw.cfg, gw.x, gw.w_router, gw.bias, idx, w)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert float((w - ref_w).abs().max()) <= parity.W_TOL
        assert np.allclose(w.sum(1).cpu().numpy(), 1.0, atol=1e-5)


def test_noalloc_router_rejects_batches_beyond_its_scratch():
    big = moe.make_config(4096, 4608, 384, 8, 2304, "nvfp4")     # 1 x 4096 x 384 floats > 2^20
    x = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_noalloc(big, x, x, x, x, x)
    assert ei.value.status == 4     # MOE_ERR_WORKSPACE_TOO_SMALL
