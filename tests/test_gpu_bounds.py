"""The bounds-checked build (libmoe_debug.so, -DMOE_DEBUG_BOUNDS), standing in
for a memory checker: its kernels check every index they derive from data
(pair positions, padded activation rows, canonical pair rows, the row-tile
plan) before the access it addresses, skip the access when the check fails
and set a flag that moe_debug_bounds_status reports; nothing traps.  The
layer's small shapes (ragged, one token, k = E, several tiles per expert,
both routers, decode and prefill tiles, the fused decode kernel) and its
limit shapes run with no check failing and give the normal build's output bit
for bit.  An out-of-range pair position planted in the combine's input (this
build only) is flagged and its read skipped, and every other token is
unchanged."""
import numpy as np
import pytest

import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402
from synth.gpu_workload import GpuWorkload  # noqa: E402
from test_gpu_layer import SMALL  # noqa: E402
from test_gpu_limits import LIMITS  # noqa: E402

SHAPES = dict(SMALL)
SHAPES.update(LIMITS)
SHAPES["fused_decode_nvfp4"] = dict(T=40, H=256, E=16, k=2, F=256, fmt="nvfp4", seed=10, outlier_frac=0.0,
                                    bias="uniform")


@pytest.fixture
def checked_build():
    moe.use_debug_bounds_build(True)
    try:
        yield
    finally:
        moe.use_debug_bounds_build(False)


def test_checked_build_is_the_checked_one(checked_build):
    st, checked = moe.moe_debug_bounds_status()
    assert checked == 1 and st == 0
    moe.use_debug_bounds_build(False)
    assert moe.moe_debug_bounds_status() == (0, 0)


@pytest.mark.parametrize("name", list(SHAPES))
def test_checked_build_runs_clean_and_equals_the_normal_build(name, checked_build):
    gw = GpuWorkload(SHAPES[name], torch)      # weights encoded by the checked build's quantiser
    out = gw.forward().clone()
    assert moe.moe_poll_device_status(gw.ws) == 0
    st, checked = moe.moe_debug_bounds_status()
    assert checked == 1 and st == 0, "an index check failed"
    moe.use_debug_bounds_build(False)
    ref = gw.forward().clone()
    moe.use_debug_bounds_build(True)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_out_of_range_pair_position_is_flagged_and_skipped(checked_build):
    gw = GpuWorkload("tiny_mxfp8", torch)
    w, T, k, H = gw.w, gw.w["T"], gw.w["k"], gw.w["H"]
    gw.forward()
    assert moe.moe_debug_bounds_status()[0] == 0
    P = T * k
    y = gw.y_raw()
    wts = gw.ws_view("topk_w", torch.float32, P).view(T, k)
    pp = gw.ws_view("pair_pos", torch.int32, P).view(T, k)
    good = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(gw.cfg, y, wts, pp, good)
    assert moe.moe_debug_bounds_status()[0] == 0
    bad_pp = pp.clone()
    bad_pp[3, 1] = P + 1000                   # a pair that does not exist
    out = torch.empty_like(good)
    moe.moe_combine(gw.cfg, y, wts, bad_pp, out)
    st, _ = moe.moe_debug_bounds_status()
    assert st == 8                            # MOE_ERR_BOUNDS
    assert moe.moe_debug_bounds_status()[0] == 0   # read and cleared
    rows = [t for t in range(T) if t != 3]
    assert torch.equal(out[rows].view(torch.int16), good[rows].view(torch.int16))
    # token 3 is the sum of its other slot only
    y3 = parity.y_rows_f64(moe, gw.cfg, y, [pp[3, 0].item()])[0] * float(wts[3, 0])
    assert np.allclose(out[3].double().cpu().numpy(), y3, rtol=2 ** -7, atol=1e-6)
