"""The fused decode expert FFN (moe_config.ffn_schedule = 0: GEMM1, the h
quantisation and GEMM2 in one persistent cooperative kernel, a down tile
starting when its h rows exist) against the separate kernels (ffn_schedule =
1): the layer output, the expert outputs y and the h codes are identical bit
for bit, on small ragged shapes, the full-size decode batches and NVFP4
static globals.  (Both schedules are checked against the oracle by the layer
tests, which run the default.)  And the fused kernel's dependency wait: with
the gate/up tiles' completion reports withheld and a short limit, the down
tiles' waits run out, the timeout is reported, and the next forward is
unchanged."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402
from synth.gpu_workload import GpuWorkload  # noqa: E402

U = dict(outlier_frac=0.0, bias="uniform")
SHAPES = {
    "tiny_mxfp8": dict(T=36, H=256, E=16, k=2, F=128, fmt="mxfp8", seed=60, **U),
    "tiny_nvfp4": dict(T=40, H=256, E=16, k=2, F=256, fmt="nvfp4", seed=10, **U),
    "ragged_mxfp8": dict(T=37, H=256, E=8, k=3, F=128, fmt="mxfp8", seed=11, **U),
    "h384_mxfp8": dict(T=40, H=384, E=6, k=2, F=384, fmt="mxfp8", seed=61, **U),   # last down tile: one block
    "one_token_nvfp4": dict(T=1, H=512, E=16, k=4, F=256, fmt="nvfp4", seed=14, **U),   # separate: 4 pairs
    "sixteen_tokens_nvfp4": dict(T=16, H=512, E=16, k=4, F=256, fmt="nvfp4", seed=62, **U),  # 64 pairs: fused
    "tc_router_decode_tiles_nvfp4": dict(T=600, H=512, E=48, k=4, F=256, fmt="nvfp4", seed=16, **U),
    "decode1_nvfp4": "decode1_nvfp4",
    "decode8_nvfp4": "decode8_nvfp4",
    "decode32_mxfp8": "decode32_mxfp8",
    "decode64_nvfp4": "decode64_nvfp4",
    "decode192_mxfp8_outliers": "decode192_mxfp8_outliers",
}


def config_with(c, **kw):
    f = {n: getattr(c, n) for n, _ in c._fields_}
    f.update(kw)
    return moe.moe_config(*[f[n] for n, _ in c._fields_])


def run(gw, cfg):
    out = torch.empty_like(gw.out)
    moe.moe_forward(cfg, gw.x, gw.w_router, gw.bias, gw.qw["gate"], gw.qw["up"], gw.qw["down"], out, gw.ws,
                    act_static_scales=gw.act_static)
    assert moe.moe_poll_device_status(gw.ws) == 0
    P, H, R, F = gw.w["T"] * gw.w["k"], gw.w["H"], gw.layout["R"], gw.w["F"]
    cb = F // 2 if gw.w["fmt"] == "nvfp4" else F
    y = gw.y_raw().clone()
    hq = gw.ws_view("hq_codes", torch.uint8, R * cb).view(R, cb).clone()
    return out, y, hq


def check_same(gw):
    assert gw.layout["tile_rows"] == 64
    fused, sep = config_with(gw.cfg, ffn_schedule=0), config_with(gw.cfg, ffn_schedule=1)
    if gw.w["T"] * gw.w["k"] >= 64:     # the fused kernel runs from 64 pairs
        assert moe.moe_forward_kernel_count(fused) < moe.moe_forward_kernel_count(sep)
    else:
        assert moe.moe_forward_kernel_count(fused) == moe.moe_forward_kernel_count(sep)
    of, yf, hf = run(gw, fused)
    os_, ys, hs = run(gw, sep)
    # h codes: the rows the tiles hold (the padding rows of a tile are never written)
    r = gw.routing()
    rows = np.concatenate([np.arange(s, s + c) for s, c in zip(r["seg_start"][:-1], r["counts"])])
    rows_t = torch.from_numpy(rows).cuda()
    assert torch.equal(hf[rows_t], hs[rows_t])
    assert torch.equal(yf, ys)
    assert torch.equal(of.view(torch.int16), os_.view(torch.int16))
    of2, _, _ = run(gw, fused)   # the counters restart at zero on every call
    assert torch.equal(of2.view(torch.int16), of.view(torch.int16))


@pytest.mark.parametrize("name", list(SHAPES))
def test_fused_decode_ffn_equals_separate_kernels(name):
    check_same(GpuWorkload(SHAPES[name], torch))
    torch.cuda.empty_cache()


def test_fused_decode_ffn_static_nvfp4_globals():
    spec = SHAPES["tiny_nvfp4"]
    rng = np.random.default_rng(3)
    act_static = np.stack([rng.uniform(2e-3, 4e-3, spec["E"]), rng.uniform(1e-3, 3e-3, spec["E"])], 1)
    check_same(GpuWorkload(spec, torch, act_static=act_static.astype(np.float32)))


@pytest.mark.parametrize("spec", [SHAPES["tiny_mxfp8"], SHAPES["tiny_nvfp4"]], ids=["mxfp8", "nvfp4"])
def test_fused_dependency_wait_timeout_is_reported_and_device_stays_usable(spec):
    gw = GpuWorkload(spec, torch)
    ref = gw.forward().clone()
    assert moe.moe_poll_device_status(gw.ws) == 0
    # ~1 ms of SM clock per wait: the down tiles' waits for their h rows run out
    moe.moe_selftest_dependency_wait(gw.cfg, gw.qw["gate"], gw.qw["up"], gw.qw["down"], gw.ws, 2_000_000)
    assert moe.moe_poll_device_status(gw.ws) == 7      # MOE_ERR_DEVICE_TIMEOUT
    assert moe.moe_poll_device_status(gw.ws) == 0      # polling clears it
    again = gw.forward()
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_dependency_wait(gw.cfg, gw.qw["gate"], gw.qw["up"], gw.qw["down"], gw.ws, 10)
