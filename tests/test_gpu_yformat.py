"""The compact expert-output rows (y_format MOE_Y_FP16E: fp16 codes with a
power-of-two exponent per 32 features) against the fp32 rows.

The down GEMM accumulates the same fp32 values in both formats, so on the
same workload the compact rows must be exactly the oracle's encoding
(oracle.encode_y16) of the fp32 rows, code for code and exponent for
exponent, on every pair row.  The combine over the compact rows must be the
weighted slot sum of the decoded values (within half a bf16 ulp and the fp32
summation error), and the fp32 format must still pass the layer's parity
against the oracle.  Covered: weight-major decode tiles (separate and fused
kernels), token-major 128-row tiles with and without the second weight block
of the last down tile (H % 256 == 128), both formats' full-size decode
batch."""
import numpy as np
import pytest

import oracle
import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402
from synth.gpu_workload import GpuWorkload  # noqa: E402
from test_gpu_layer import SMALL, check_combine_rows, check_layer  # noqa: E402

U = dict(outlier_frac=0.0, bias="uniform")
SHAPES = {
    "tiny_mxfp8": (SMALL["tiny_mxfp8"], 0),
    "fused_nvfp4": (dict(T=40, H=256, E=16, k=2, F=256, fmt="nvfp4", seed=30, **U), 0),
    "separate_nvfp4": (dict(T=40, H=256, E=16, k=2, F=256, fmt="nvfp4", seed=30, **U), 1),
    "deep_mxfp8_h384": (SMALL["deep_mxfp8"], 0),
    "deep_nvfp4": (SMALL["deep_nvfp4"], 0),
    "tc_router_mxfp8_outliers": (SMALL["tc_router_mxfp8_outliers"], 0),
    "decode64_nvfp4": ("decode64_nvfp4", 0),
}


def config_with(c, **kw):
    f = {n: getattr(c, n) for n, _ in c._fields_}
    f.update(kw)
    return moe.moe_config(*[f[n] for n, _ in c._fields_])


@pytest.mark.parametrize("name", list(SHAPES))
def test_compact_rows_are_the_encoding_of_the_fp32_rows(name):
    spec, sched = SHAPES[name]
    gw = GpuWorkload(spec, torch, ffn_schedule=sched)
    assert gw.cfg.y_format == moe.Y_FP16E
    T, k, H = gw.w["T"], gw.w["k"], gw.w["H"]
    P = T * k
    # the fp32 rows of the same workload, in a workspace of their own
    c32 = config_with(gw.cfg, y_format=moe.Y_FP32)
    ws32 = torch.empty(moe.moe_workspace_size(c32), dtype=torch.uint8, device="cuda")
    out32 = torch.empty_like(gw.out)
    moe.moe_forward(c32, gw.x, gw.w_router, gw.bias, gw.qw["gate"], gw.qw["up"], gw.qw["down"], out32, ws32)
    assert moe.moe_poll_device_status(ws32) == 0
    L32 = moe.moe_workspace_layout(c32)
    y32 = moe.y_rows(c32, ws32[L32["y_perm"]:L32["y_perm"] + moe.moe_y_bytes(c32)]).cpu().numpy()
    out16 = gw.forward()
    torch.cuda.synchronize()
    assert moe.moe_poll_device_status(gw.ws) == 0
    assert moe.moe_y_bytes(gw.cfg) == P * H * 2 + P * (H // 32)
    codes, ex = moe.y_rows(gw.cfg, gw.y_raw())
    codes = codes.view(torch.int16).cpu().numpy().view(np.uint16)
    ex = ex.cpu().numpy()
    ref_codes, ref_ex = oracle.encode_y16(y32)
    assert np.array_equal(ex, ref_ex), f"exponents differ in {int((ex != ref_ex).sum())} blocks"
    assert np.array_equal(codes, ref_codes), f"codes differ at {int((codes != ref_codes).sum())} elements"
    # the combine on the compact rows: the weighted slot sum of the decoded values
    r = gw.routing()
    check_combine_rows(gw, r, parity.bf16_to_f64(out16), np.arange(min(T, 1024)))
    # the two outputs differ only through y's rounding (2^-11 relative) and bf16
    d = np.abs(parity.bf16_to_f64(out16) - parity.bf16_to_f64(out32))
    scale = np.abs(parity.bf16_to_f64(out32))
    ymax = np.abs(y32).max()
    assert np.all(d <= 2.0 ** -7 * scale + 2.0 ** -10 * ymax + 1e-30)


@pytest.mark.parametrize("name", ["tiny_nvfp4", "ragged_mxfp8", "multitile_mxfp8", "deep_nvfp4", "tc_router_nvfp4"])
def test_fp32_rows_layer_parity(name):
    gw = GpuWorkload(SMALL[name], torch, y_format="fp32")
    assert gw.cfg.y_format == moe.Y_FP32
    check_layer(gw)
