"""GPU tests of the layer's extra entry points and modes: fake quantisation
(bit-exact against the oracle's encode + decode), CUDA-graph capture of the
whole forward (the small-T decode path replays as one graph), and the
bounded-wait failure detection (a GEMM whose loads are withheld reports a
timeout through the workspace status word and leaves the device usable)."""
import numpy as np
import pytest

import oracle
import parity
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402
from synth.gpu_workload import GpuWorkload  # noqa: E402


@pytest.mark.parametrize("fmt,group_rows,mx_mode", [("nvfp4", 0, 0), ("nvfp4", 128, 0), ("mxfp8", 0, 0),
                                                     ("mxfp8", 0, 1)])
def test_fake_quantize_bit_exact(fmt, group_rows, mx_mode):
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((256, 512)) * rng.uniform(1e-2, 1e2, (256, 1))).astype(np.float32)
    src = torch.from_numpy(v).cuda()
    out = torch.empty_like(src)
    ng = (256 // group_rows) if group_rows else 256
    glob = torch.empty(ng, dtype=torch.float32, device="cuda") if fmt == "nvfp4" else None
    moe.moe_fake_quantize(fmt, src, out, glob, group_rows=group_rows, mx_scale_mode=mx_mode)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    if fmt == "nvfp4" and group_rows:
        want = np.concatenate([oracle.decode(fmt, *oracle.quantize(fmt, v[i:i + group_rows], per_tensor=True),
                                             per_tensor=True) for i in range(0, 256, group_rows)])
    else:
        want = oracle.decode(fmt, *oracle.quantize(fmt, v, mx_mode=mx_mode))
    assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("name", ["tiny_mxfp8", "decode64_nvfp4"])
def test_forward_replays_as_cuda_graph(name):
    gw = GpuWorkload(name, torch)
    eager = gw.forward().clone()
    out2 = torch.empty_like(eager)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        moe.moe_forward(gw.cfg, gw.x, gw.w_router, gw.bias, gw.qw["gate"], gw.qw["up"], gw.qw["down"], out2, gw.ws,
                        stream=st)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(st)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_forward(gw.cfg, gw.x, gw.w_router, gw.bias, gw.qw["gate"], gw.qw["up"], gw.qw["down"], out2, gw.ws)
    out2.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), eager.view(torch.int16))
    # the graph reads its inputs on every replay
    x_saved = gw.x.clone()
    gw.x.mul_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    neg = out2.clone()
    gw.x.copy_(x_saved)
    eager_neg_check = gw.forward()
    assert not torch.equal(neg.view(torch.int16), eager_neg_check.view(torch.int16))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), eager.view(torch.int16))


WIDE_MXFP8 = dict(T=1100, H=384, E=5, k=3, F=384, fmt="mxfp8", seed=19, outlier_frac=0.0, bias="uniform")


# tiny: 64-row weight-major tiles; WIDE_MXFP8: 128-row token-major tiles
@pytest.mark.parametrize("spec", ["tiny_mxfp8", WIDE_MXFP8], ids=["decode_tiles", "token_major_tiles"])
def test_bounded_wait_timeout_is_reported_and_device_stays_usable(spec):
    gw = GpuWorkload(spec, torch)
    ref = gw.forward().clone()
    assert moe.moe_poll_device_status(gw.ws) == 0
    # ~1 ms of SM clock per wait; every wait of the kernel runs out
    moe.moe_selftest_bounded_wait(gw.cfg, gw.qw["gate"], gw.qw["up"], gw.ws, 2_000_000)
    assert moe.moe_poll_device_status(gw.ws) == 7      # MOE_ERR_DEVICE_TIMEOUT
    assert moe.moe_poll_device_status(gw.ws) == 0      # polling clears it
    again = gw.forward()
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_bounded_wait(gw.cfg, gw.qw["gate"], gw.qw["up"], gw.ws, 10)   # limit out of range
