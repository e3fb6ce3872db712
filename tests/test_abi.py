"""Host-side tests of the C ABI: the library builds, loads and exports every
entry point include/moe.h declares; argument validation returns the
documented status codes before anything is enqueued (no GPU needed: the
pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

import block_scaled_fp4_route_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ["moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward", "moe_workspace_size",
              "moe_quantize", "moe_poll_device_status", "moe_status_string"]:
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    L = moe.lib()
    for n in declared_functions():
        assert hasattr(L, n), n
        assert ctypes.cast(getattr(L, n), ctypes.c_void_p).value
    assert sorted(declared_functions()) == sorted(moe.EXPORTED)


def test_status_strings():
    for s in range(8):
        assert moe.moe_status_string(s)


def cfg(**kw):
    base = dict(T=64, H=4608, E=384, k=8, F=2304, fmt="nvfp4")
    base.update(kw)
    return moe.make_config(**base)


def test_workspace_size_and_layout():
    c = cfg()
    n = moe.moe_workspace_size(c)
    L = moe.moe_workspace_layout(c)
    assert L["total"] == n
    offs = [L[f] for f in ["status", "logits", "topk_idx", "topk_w", "counts", "offsets", "perm", "pair_pos",
                           "bitmap", "seg_start", "tiles", "rt_base", "xq_codes", "xq_scales", "xq_global",
                           "h_bf16", "hq_codes", "hq_scales", "hq_global", "y_perm", "total"]]
    assert offs == sorted(offs) and all(o % 1024 == 0 for o in offs)
    # padded rows: one token tile per expert on top of the pairs
    assert L["tile_rows"] == 64 and L["R"] == ((64 * 8 + 63) // 64 + 384) * 64
    Lp = moe.moe_workspace_layout(cfg(T=4096))      # >= 64 tokens per expert: 128-row tiles
    assert Lp["tile_rows"] == 128 and Lp["R"] == ((4096 * 8 + 127) // 128 + 384) * 128
    assert L["hq_codes"] - L["h_bf16"] >= L["R"] * 2304 * 2
    for T in (64, 4096):  # MXFP8: h quantised inside GEMM1 (64- and 128-row tiles), no bf16 h
        Lm = moe.moe_workspace_layout(cfg(fmt="mxfp8", T=T))
        assert Lm["hq_codes"] == Lm["h_bf16"]
    # larger T needs no less workspace
    assert moe.moe_workspace_size(cfg(T=4096)) > n
    # the y rows: fp16 codes then one exponent byte per 32 features (default), or fp32
    P, H = 64 * 8, 4608
    assert c.y_format == moe.Y_FP16E and moe.moe_y_bytes(c) == P * H * 2 + P * H // 32
    c32 = cfg(y_format="fp32")
    assert moe.moe_y_bytes(c32) == P * H * 4
    L32 = moe.moe_workspace_layout(c32)
    assert L32["total"] - L32["y_perm"] >= P * H * 4 and L["total"] - L["y_perm"] >= P * H * 2 + P * H // 32
    assert L32["total"] > L["total"]


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), 2), (dict(T=70000), 2), (dict(k=0), 2), (dict(k=33), 2), (dict(E=4, k=8), 2),
    (dict(E=2000), 2), (dict(H=4608 + 128), 2), (dict(F=128), 2), (dict(fmt="mxfp8", F=128 + 64), 2),
    (dict(swiglu_cap=-1.0), 1), (dict(mx_scale_mode=2), 1), (dict(act_global_mode=2), 1),
    (dict(fmt="mxfp8", act_global_mode=1), 1), (dict(ffn_schedule=2), 1), (dict(y_format=2), 1),
])
def test_config_validation(kw, status):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(cfg(**kw))
    assert ei.value.status == status


class FakeTensor:
    """Stands in for a device tensor: an address and a size, never dereferenced."""

    def __init__(self, addr, nbytes=1 << 40):
        self.addr, self.nbytes = addr, nbytes

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.nbytes

    def element_size(self):
        return 1


def test_argument_validation_without_a_device():
    c = cfg()
    ok = FakeTensor(0x10000)
    mis = FakeTensor(0x10008)
    ws = FakeTensor(0x100000)
    with pytest.raises(moe.MoeError) as ei:   # null pointer
        moe.moe_route(c, ok, ok, 0, ok, ok, ws, stream=0)
    assert ei.value.status == 1
    with pytest.raises(moe.MoeError) as ei:   # misaligned pointer
        moe.moe_route(c, mis, ok, ok, ok, ok, ws, stream=0)
    assert ei.value.status == 3
    with pytest.raises(moe.MoeError) as ei:   # workspace too small
        moe.moe_route(c, ok, ok, ok, ok, ok, FakeTensor(0x100000, 1024), stream=0)
    assert ei.value.status == 4
    with pytest.raises(moe.MoeError) as ei:   # workspace not 256-byte aligned
        moe.moe_route(c, ok, ok, ok, ok, ok, FakeTensor(0x100010), stream=0)
    assert ei.value.status == 3
    qw = moe.qweight(0x20000, 0x30000, None)   # NVFP4 needs globals
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward(c, ok, ok, ok, qw, qw, qw, ok, ws, stream=0)
    assert ei.value.status == 1
    cs = cfg(act_global_mode=1)                # static activation globals: the scales are required
    qg = moe.qweight(0x20000, 0x30000, 0x40000)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward(cs, ok, ok, ok, qg, qg, qg, ok, ws, stream=0)
    assert ei.value.status == 1
    with pytest.raises(moe.MoeError) as ei:   # and 4-byte aligned
        moe.moe_forward(cs, ok, ok, ok, qg, qg, qg, ok, ws, stream=0, act_static_scales=0x10002)
    assert ei.value.status == 3
    with pytest.raises(moe.MoeError) as ei:   # tiled scales need rows % 128 == 0
        moe.lib()
        st = moe.lib().moe_quantize(0, 0, 1, 0x10000, 100, 256, 0, 1, 0x20000, 0x30000, 0x40000, 0)
        moe._check("moe_quantize", st)
    assert ei.value.status == 2
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_pack_scales(ok, 100, 16, ok, stream=0)
    assert ei.value.status == 2


def test_forward_kernel_count():
    # router (2 for decode batches, 3 with tensor-core logits) + dispatch (1 for decode batches, else 3)
    # + x quant + (decode batches: the fused expert FFN | GEMM1 + h quant (unless GEMM1 quantises h)
    # + GEMM2) + combine
    assert moe.moe_forward_kernel_count(cfg()) == 6
    assert moe.moe_forward_kernel_count(cfg(fmt="mxfp8", T=192)) == 6
    assert moe.moe_forward_kernel_count(cfg(ffn_schedule=1)) == 8
    assert moe.moe_forward_kernel_count(cfg(fmt="mxfp8", T=192, ffn_schedule=1)) == 7
    assert moe.moe_forward_kernel_count(cfg(T=1024)) == 9         # tensor-core router, 3 dispatch kernels, fused
    assert moe.moe_forward_kernel_count(cfg(T=7)) == 8            # 56 pairs: separate kernels
    assert moe.moe_forward_kernel_count(cfg(T=8)) == 6            # 64 pairs: fused
    assert moe.moe_forward_kernel_count(cfg(T=4096)) == 11
    assert moe.moe_forward_kernel_count(cfg(fmt="mxfp8", T=16384)) == 10
    assert moe.moe_forward_kernel_count(cfg(T=4096, E=376)) == 10  # E % 16 != 0: CUDA-core router
    with pytest.raises(moe.MoeError):
        moe.moe_forward_kernel_count(cfg(T=0))


def test_noalloc_router_refuses_batches_beyond_its_scratch_before_any_launch():
    # moe_route_noalloc's fixed scratch holds 2^20 floats: a 64-float status
    # area, then the router's scratch.  For T > 256 (tensor-core router) that
    # is the logits [T, E] and ||w_e|| padded to 64: at E = 384 the largest
    # batch is T = 2729 (64 + 2729*384 + 384 = 1,048,384 <= 1,048,576), and
    # T = 2730 needs 1,048,768.  The refusal comes before the device is
    # touched (these addresses are never dereferenced).
    ok = FakeTensor(0x10000)
    for T in (2730, 4096):
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_route_noalloc(cfg(T=T), ok, ok, ok, ok, ok, stream=0)
        assert ei.value.status == 4
    assert 64 + 2729 * 384 + 384 <= 1 << 20 < 64 + 2730 * 384 + 384
    # E not a multiple of 16: the CUDA-core router (one K split above 256
    # tokens), 64 + T*E floats; E = 376: T <= 2788
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_noalloc(cfg(T=2789, E=376), ok, ok, ok, ok, ok, stream=0)
    assert ei.value.status == 4
    assert 64 + 2788 * 376 <= 1 << 20 < 64 + 2789 * 376
    with pytest.raises(moe.MoeError) as ei:   # pointers are validated first
        moe.moe_route_noalloc(cfg(T=64), ok, ok, FakeTensor(0x10004), ok, ok, stream=0)
    assert ei.value.status == 3


def test_kv_quantize_validation_without_a_device():
    L = moe.lib()
    ok = 0x10000
    call = lambda **kw: L.moe_kv_quantize_mxfp8(*[kw.get(n, d) for n, d in [
        ("kv", ok), ("tokens", 16), ("heads", 8), ("head_dim", 128), ("stride", 8 * 128), ("slot", None),
        ("num_slots", 16), ("mode", 0), ("codes", ok), ("scales", ok), ("stream", None)]])
    assert call(head_dim=100) == 2 and call(head_dim=16) == 2 and call(head_dim=2048) == 2
    assert call(stride=8 * 128 - 8) == 2 and call(stride=8 * 128 + 4) == 2
    assert call(heads=0) == 2 and call(tokens=-1) == 2
    assert call(mode=2) == 1
    assert call(num_slots=15) == 1                  # identity slots need num_slots >= tokens
    assert call(tokens=0) == 0                      # nothing to do, nothing enqueued
    assert call(kv=ok + 8) == 3 and call(codes=ok + 4) == 3 and call(scales=None) == 1
    assert call(slot=ok + 4) == 3                   # int64 slots, 8-byte aligned


def test_bounds_checked_build_exports_the_same_symbols():
    D = moe.lib(debug_bounds=True)
    for n in declared_functions():
        assert hasattr(D, n), n
    c = ctypes.c_int(-1)
    site = ctypes.c_int(-1)
    assert moe.lib().moe_debug_bounds_status(None, ctypes.byref(c), ctypes.byref(site)) == 0
    assert c.value == 0 and site.value == 0
