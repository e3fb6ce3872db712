"""GPU block quantiser (moe_quantize, moe_pack_scales) against the oracle:
codes, scales and globals must match bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden
from synth.gpu_workload import untile_scales

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402


def gpu_quant(fmt, v, group_rows=0, layout=moe.SCALES_ROWMAJOR, mx_mode=0, src_dtype=torch.float32):
    rows, cols = v.shape
    nv = fmt == "nvfp4"
    bs = 16 if nv else 32
    src = torch.from_numpy(np.ascontiguousarray(v)).to(src_dtype).cuda()
    codes = torch.empty((rows, cols // 2 if nv else cols), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, cols // bs), dtype=torch.uint8, device="cuda")
    ng = rows if group_rows == 0 else rows // group_rows
    glob = torch.empty(ng, dtype=torch.float32, device="cuda") if nv else None
    moe.moe_quantize(fmt, src, codes, scales, glob, group_rows=group_rows, layout=layout, mx_scale_mode=mx_mode)
    torch.cuda.synchronize()
    sc = scales.cpu().numpy()
    if layout == moe.SCALES_TILED:
        sc = untile_scales(sc, rows, cols // bs)
    return codes.cpu().numpy(), sc, (glob.cpu().numpy() if nv else None)


def oracle_quant(fmt, v, per_tensor=False, mx_mode=0):
    return oracle.quantize(fmt, v.astype(np.float32), per_tensor=per_tensor, mx_mode=mx_mode)


def assert_same(gq, oq):
    assert np.array_equal(gq[0], oq[0]), f"codes differ at {np.argwhere(gq[0] != oq[0])[:5]}"
    assert np.array_equal(gq[1], oq[1]), f"scales differ at {np.argwhere(gq[1] != oq[1])[:5]}"
    if oq[2] is not None:
        assert np.array_equal(gq[2].view(np.uint32), np.asarray(oq[2]).view(np.uint32))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
@pytest.mark.parametrize("layout", [moe.SCALES_ROWMAJOR, moe.SCALES_TILED])
def test_random_rows_bit_exact(fmt, layout):
    rng = np.random.default_rng(1)
    v = (rng.standard_normal((256, 512)) * rng.uniform(1e-3, 1e3, (256, 1))).astype(np.float32)
    v[3] = 0.0                                     # an all-zero row
    v[5, :40] = 0.0                                # zero blocks
    v[7] = -0.0
    assert_same(gpu_quant(fmt, v, layout=layout), oracle_quant(fmt, v))


@pytest.mark.parametrize("mx_mode", [0, 1])
def test_mxfp8_scale_modes(mx_mode):
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((64, 256)) * 3.9).astype(np.float32)
    assert_same(gpu_quant("mxfp8", v, mx_mode=mx_mode), oracle_quant("mxfp8", v, mx_mode=mx_mode))


def test_nvfp4_group_globals_bit_exact():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((3 * 128, 256)) * np.repeat([0.01, 1.0, 55.0], 128)[:, None]).astype(np.float32)
    g = gpu_quant("nvfp4", v, group_rows=128, layout=moe.SCALES_TILED)
    for i in range(3):
        o = oracle_quant("nvfp4", v[128 * i:128 * (i + 1)], per_tensor=True)
        assert np.array_equal(g[0][128 * i:128 * (i + 1)], o[0])
        assert np.array_equal(g[1][128 * i:128 * (i + 1)], o[1])
        assert g[2][i].view(np.uint32) == o[2][0].view(np.uint32)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
@pytest.mark.parametrize("mul", [1.0, 3.0, 1e-30])
def test_every_finite_bf16_pattern(fmt, mul):
    # all 2^16 bf16 bit patterns except NaN/Inf, in rows of 256, from a bf16
    # source (the activation path) and scaled copies from fp32
    bits = np.arange(1 << 16, dtype=np.uint32)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]
    bits = np.concatenate([bits, np.zeros((-len(bits)) % 256, np.uint32)])
    vals = (bits << 16).view(np.float32).reshape(-1, 256)
    with np.errstate(over="ignore"):
        vals = (vals * np.float32(mul)).astype(np.float32)
    # the documented domain: finite inputs; for NVFP4 a row maximum whose
    # global 2688/amax stays finite in fp32
    amax = np.abs(vals).max(1)
    keep = np.isfinite(vals).all(1)
    if fmt == "nvfp4":
        keep &= amax >= 1e-32   # G and G/scale stay finite
    vals = np.ascontiguousarray(vals[keep])
    assert len(vals) > 16
    if mul == 1.0:
        src = torch.from_numpy(vals.copy()).to(torch.bfloat16)
        assert np.array_equal(src.float().numpy().view(np.uint32), vals.view(np.uint32))
        g = gpu_quant(fmt, vals, src_dtype=torch.bfloat16)
    else:
        g = gpu_quant(fmt, vals)
    assert_same(g, oracle_quant(fmt, vals))


def test_worked_blocks_on_device():
    gold = read_golden("nvfp4_block_roundtrip.txt")
    v = np.array([float(s) for s in gold["values"]], np.float32)[None, :]
    v = np.tile(v, (1, 8))                                   # 256 columns
    codes, sf, g = gpu_quant("nvfp4", v)
    nib = []
    for b in codes[0][:16]:
        nib += [b & 15, b >> 4]
    assert [f"{q:X}" for q in nib] == gold["codes_hex"]
    assert [f"{b:02X}" for b in sf[0][:2]] == gold["scales_hex"]
    assert g[0] == float(gold["global"][0])
    gm = read_golden("mxfp8_block_roundtrip.txt")
    a = np.array([float(s) for s in gm["blockA_values"]] * 4, np.float32)[None, :]
    codes, sf, _ = gpu_quant("mxfp8", a)
    assert [f"{c:02X}" for c in codes[0][:32]] == gm["blockA_codes_hex"]
    assert f"{sf[0, 0]:02X}" == gm["blockA_scale_hex"][0]


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
def test_pack_scales_matches_tiled_quantiser(fmt):
    rng = np.random.default_rng(4)
    v = rng.standard_normal((256, 1024)).astype(np.float32)
    bs = 16 if fmt == "nvfp4" else 32
    src = torch.from_numpy(v).cuda()
    nv = fmt == "nvfp4"
    c = torch.empty((256, 512 if nv else 1024), dtype=torch.uint8, device="cuda")
    s_rm = torch.empty((256, 1024 // bs), dtype=torch.uint8, device="cuda")
    s_t = torch.empty_like(s_rm)
    s_p = torch.empty_like(s_rm)
    g = torch.empty(256, dtype=torch.float32, device="cuda") if nv else None
    moe.moe_quantize(fmt, src, c, s_rm, g, layout=moe.SCALES_ROWMAJOR)
    moe.moe_quantize(fmt, src, c, s_t, g, layout=moe.SCALES_TILED)
    moe.moe_pack_scales(s_rm, 256, 1024 // bs, s_p)
    torch.cuda.synchronize()
    assert torch.equal(s_t, s_p)
    assert np.array_equal(untile_scales(s_t.cpu().numpy(), 256, 1024 // bs), s_rm.cpu().numpy())


@pytest.mark.parametrize("name", ["decode64_nvfp4", "decode192_mxfp8_outliers"])
def test_full_size_expert_encoding_bit_exact(name):
    # one expert of each matrix, generated on the device and encoded by the
    # library, against the oracle's encoding of the same seeded values
    w = synth.WORKLOADS[name]
    e = 37
    nv = w["fmt"] == "nvfp4"
    q = oracle.quantized_expert(w, e)
    for which, N, K in (("gate", w["F"], w["H"]), ("down", w["H"], w["F"])):
        m = synth.dev_expert_matrices(w, which, e, 1, torch)
        bs = 16 if nv else 32
        codes = torch.empty((N, K // 2 if nv else K), dtype=torch.uint8, device="cuda")
        sc = torch.empty((N, K // bs), dtype=torch.uint8, device="cuda")
        gl = torch.empty(1, dtype=torch.float32, device="cuda") if nv else None
        moe.moe_quantize(w["fmt"], m.view(N, K), codes, sc, gl, group_rows=N if nv else 0, layout=moe.SCALES_TILED)
        torch.cuda.synchronize()
        # the device fill equals the host fill
        host = synth.expert_matrix(w, which, e)
        assert np.array_equal(m.view(N, K).cpu().numpy().view(np.uint32), host.view(np.uint32))
        oc, osf, og = q[which]
        assert np.array_equal(codes.cpu().numpy(), oc)
        assert np.array_equal(untile_scales(sc.cpu().numpy(), N, K // bs), osf)
        if nv:
            assert gl.cpu().numpy()[0].view(np.uint32) == og[0].view(np.uint32)


def test_device_inputs_match_host_generator():
    w = synth.WORKLOADS["decode192_mxfp8_outliers"]
    x = synth.dev_x(w, torch).view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(x[[0, 5, 191]], synth.x_rows(w, [0, 5, 191]))
    flags = synth.outlier_flags(w)
    t = int(np.nonzero(flags)[0][0])
    assert np.array_equal(x[t], synth.x_rows(w, [t])[0])
    wr = synth.dev_router_weight(w, torch).view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(wr, synth.router_weight(w))
