"""The block-scaled tensor-core peak microbenchmark (moe_bench_mma_peak): it
runs on every SM, reports no timeout, and its rate per SM cycle is that of a
tensor core doing the work (above a tenth of the nominal dense rate, below
1.5x of it).  The nominal rates (13.5 PFLOP/s NVFP4, 4.5 PFLOP/s MXFP8 dense
at 2070 MHz on 152 SMs) give the expected FLOP per SM cycle."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402

NOMINAL_FLOP_PER_SM_CYCLE = {"nvfp4": 13.5e15 / (152 * 2070e6), "mxfp8": 4.5e15 / (152 * 2070e6)}


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
def test_mma_peak_runs_on_every_sm(fmt):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    status = torch.zeros(64, dtype=torch.int32, device="cuda")
    cycles = torch.zeros(sms, dtype=torch.int64, device="cuda")
    n = 1 << 14
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    ctas, fpm = moe.moe_bench_mma_peak(fmt, n, status, cycles)
    end.record()
    assert moe.moe_poll_device_status(status) == 0
    assert ctas == sms and fpm == 2 * 128 * 256 * (64 if fmt == "nvfp4" else 32)
    cyc = cycles.cpu().numpy()
    assert (cyc > 0).all()
    per_cycle = n * fpm / float(cyc.max())
    nominal = NOMINAL_FLOP_PER_SM_CYCLE[fmt]
    assert 0.1 * nominal < per_cycle < 1.5 * nominal, (per_cycle, nominal)
    tflops = ctas * n * fpm / (start.elapsed_time(end) * 1e-3) / 1e12
    print(fmt, f"{per_cycle:.0f} FLOP/SM/cycle ({per_cycle / nominal:.2f} of nominal), {tflops:.0f} TFLOP/s")
