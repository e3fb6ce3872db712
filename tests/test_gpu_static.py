"""NVFP4 with static per-expert activation globals (act_global_mode 1): the x
rows routed to expert e are encoded with the caller's decode factor g_x[e],
its h rows with g_h[e] (block maxima beyond 2688 g saturate).  The x codes,
block scales and globals of every (token, slot) row must equal the oracle's
bit for bit; the layer output is held to the usual tolerance.  The factors are
chosen so that the largest values of some experts' rows saturate."""
import numpy as np
import pytest

import oracle
import parity
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402
from synth.gpu_workload import GpuWorkload, untile_scales  # noqa: E402

U = dict(outlier_frac=0.0, bias="uniform")
SHAPES = {
    "static_decode_tiles": dict(T=37, H=512, E=8, k=3, F=256, fmt="nvfp4", seed=18, **U),
    "static_wide_tiles": dict(T=300, H=512, E=4, k=2, F=256, fmt="nvfp4", seed=19, **U),
}


def static_scales(w):
    x = oracle.bf16_bits_to_f32(synth.x_rows(w, np.arange(w["T"])))
    f = 0.5 + 0.25 * (np.arange(w["E"]) % 4)
    gx = (f * float(np.abs(x).max()) / 2688).astype(np.float32)
    gh = (f * 40.0 / 2688).astype(np.float32)
    return np.stack([gx, gh], 1)


@pytest.mark.parametrize("name", list(SHAPES))
def test_static_activation_globals(name):
    w = SHAPES[name]
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    st = static_scales(w)
    gw = GpuWorkload(w, torch, act_static=st)
    out = parity.bf16_to_f64(gw.forward())
    assert moe.moe_poll_device_status(gw.ws) == 0
    r = gw.routing()
    x = synth.x_rows(w, np.arange(T))
    ro = oracle.route(x, synth.router_weight(w), synth.router_bias(w), k)
    ties = parity.check_topk(r["idx"], ro["idx"], ro["keys"], ro["absdot"])

    # x codes, scales and globals at every (token, slot) row, each with its expert's factor
    R, nt = gw.layout["R"], gw.layout["tile_rows"]
    codes = gw.ws_view("xq_codes", torch.uint8, R * H // 2).view(R, H // 2).cpu().numpy()
    scales = untile_scales(gw.ws_view("xq_scales", torch.uint8, (R // nt) * (H // 64) * 512).cpu().numpy(),
                           R, H // 16, tile_rows=nt)
    glob = gw.ws_view("xq_global", torch.float32, R).cpu().numpy()
    hglob = gw.ws_view("hq_global", torch.float32, R).cpu().numpy()
    xf = oracle.bf16_bits_to_f32(x)
    sat = 0
    for t in range(T):
        for j in range(k):
            e = int(r["idx"][t, j])
            row = r["seg_start"][e] + r["pair_pos"][t, j] - r["offsets"][e]
            q = oracle.nvfp4_quantize_static(xf[t:t + 1], st[e, 0])
            assert np.array_equal(codes[row], q[0][0]) and np.array_equal(scales[row], q[1][0]), (t, j)
            assert glob[row].view(np.uint32) == st[e, 0].view(np.uint32)
            assert hglob[row].view(np.uint32) == st[e, 1].view(np.uint32)
            sat += int((q[1][0] == 0x7E).sum())
    assert sat > 0  # some block scales saturated

    res = oracle.moe_layer(w, np.arange(T), idx_override=ties, act_static=st)
    print(name, "err/rms", parity.check_output(out, res["out"]), "saturated x blocks", sat)
