"""The largest shapes the API accepts, each in one dimension at a time: 1024
experts with k = 32 (and with the tensor-core router's selection), hidden
and FFN widths of 16384 (rows quantised in registers by one CTA), and 65536
tokens; and degenerate routing (every token on the same k experts).  Same
checks as the layer tests: routing against the oracle, dispatch and x codes
bit-exact, h near-exact, the output within tolerance (sampled tokens for the
largest batch)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from synth.gpu_workload import GpuWorkload  # noqa: E402
from test_gpu_layer import check_layer, sample_tokens  # noqa: E402

U = dict(outlier_frac=0.0, bias="uniform")
LIMITS = {
    "E1024_k32_mxfp8": dict(T=40, H=256, E=1024, k=32, F=128, fmt="mxfp8", seed=40, **U),
    # T > 256: the tensor-core router's selection with 32 experts a lane
    "E1024_tc_router_mxfp8": dict(T=300, H=256, E=1024, k=8, F=128, fmt="mxfp8", seed=46, **U),
    "H16384_nvfp4": dict(T=3, H=16384, E=4, k=2, F=256, fmt="nvfp4", seed=41, **U),
    "F16384_nvfp4": dict(T=2, H=256, E=2, k=1, F=16384, fmt="nvfp4", seed=42, **U),
    "F16384_mxfp8": dict(T=5, H=256, E=2, k=2, F=16384, fmt="mxfp8", seed=43, **U),
    # degenerate routing: all 300 tokens on the same 4 of 64 experts (one
    # expert with every token, 60 with none; 128-row tiles)
    "all_tokens_4_experts_nvfp4": dict(T=300, H=512, E=64, k=4, F=256, fmt="nvfp4", seed=45, outlier_frac=0.0,
                                       bias="hot"),
}


@pytest.mark.parametrize("name", list(LIMITS))
def test_limit_shapes(name):
    gw = GpuWorkload(LIMITS[name], torch)
    print(name, check_layer(gw))


def test_65536_tokens():
    w = dict(T=65536, H=256, E=16, k=1, F=128, fmt="mxfp8", seed=44, **U)
    gw = GpuWorkload(w, torch)
    print("T65536", check_layer(gw, sample_tokens(w, 16)))
