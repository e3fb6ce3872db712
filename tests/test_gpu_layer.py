"""The whole layer on the GPU (moe_forward and the staged calls) against the
oracle.  Small shapes are compared on every token; the full-size seeded
workloads, in the launch configuration the benchmark times, on all routing /
dispatch / activation-code results and on the output rows of a seeded token
sample (the oracle regenerates the touched experts itself)."""
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
SMALL = {
    "tiny_mxfp8": "tiny_mxfp8",
    "tiny_nvfp4": dict(T=8, H=256, E=16, k=2, F=256, fmt="nvfp4", seed=10, **U),
    "ragged_mxfp8": dict(T=37, H=256, E=8, k=3, F=128, fmt="mxfp8", seed=11, **U),
    "multitile_nvfp4": dict(T=300, H=256, E=2, k=1, F=256, fmt="nvfp4", seed=12, **U),
    "multitile_mxfp8": dict(T=290, H=384, E=3, k=2, F=256, fmt="mxfp8", seed=15, **U),
    "k_eq_E_mxfp8": dict(T=5, H=256, E=4, k=4, F=128, fmt="mxfp8", seed=13, **U),
    "one_token_nvfp4": dict(T=1, H=512, E=16, k=4, F=256, fmt="nvfp4", seed=14, **U),
    # T > 256: the tensor-core router; ragged token and expert tiles
    "tc_router_nvfp4": dict(T=600, H=512, E=48, k=4, F=256, fmt="nvfp4", seed=16, **U),
    "tc_router_mxfp8_outliers": dict(T=520, H=384, E=160, k=6, F=128, fmt="mxfp8", seed=17, outlier_frac=0.02,
                                     bias="uniform"),
    # hundreds of tokens per expert on 128-row token tiles: 4-10 tiles per
    # expert with ragged tails, H % 256 == 128 (down: no second weight block
    # in the last tile), empty experts ("hot": two experts take every token)
    "deep_nvfp4": dict(T=1200, H=512, E=4, k=2, F=256, fmt="nvfp4", seed=18, **U),
    "deep_mxfp8": dict(T=1100, H=384, E=5, k=3, F=384, fmt="mxfp8", seed=19, **U),
    "deep_hot_nvfp4": dict(T=1100, H=512, E=8, k=2, F=256, fmt="nvfp4", seed=20, outlier_frac=0.0, bias="hot"),
    # T >= 2048: x quantised a warp per row, the row held in registers (H =
    # 1024: four 32-lane slots; H = 384: the last slot half full)
    "warp_x_nvfp4": dict(T=2100, H=1024, E=8, k=2, F=256, fmt="nvfp4", seed=21, **U),
    "warp_x_mxfp8": dict(T=2080, H=384, E=6, k=3, F=128, fmt="mxfp8", seed=22, **U),
}


def padded_rows_of(r, tokens, k):
    """Padded expert-grouped row of every (token, slot) of the sample."""
    idx, pp, off, seg = r["idx"], r["pair_pos"], r["offsets"], r["seg_start"]
    rows = np.empty((len(tokens), k), np.int64)
    for i, t in enumerate(tokens):
        for j in range(k):
            e = idx[t, j]
            rows[i, j] = seg[e] + pp[t, j] - off[e]
    return rows


def check_layer(gw, tokens=None, cap=10.0, mx_mode=0, check_h=True, out_rowwise=False, route_all=True,
                expert_cache=None):
    w, T, k, E, H, F = gw.w, gw.w["T"], gw.w["k"], gw.w["E"], gw.w["H"], gw.w["F"]
    out = gw.forward()
    assert moe.moe_poll_device_status(gw.ws) == 0
    gpu_out = parity.bf16_to_f64(out)
    r = gw.routing()
    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens, np.int64)
    stats = {}

    # routing: all tokens (or the sample), near-ties certified against the bound
    rows_r = np.arange(T) if route_all else tokens
    x_r = synth.x_rows(w, rows_r)
    ro = oracle.route(x_r, synth.router_weight(w), synth.router_bias(w), k, **gw.route_opts)
    ties_all = parity.check_topk(r["idx"][rows_r], ro["idx"], ro["keys"], ro["absdot"])
    stats["near_ties"] = len(ties_all)
    same = [i for i in range(len(rows_r)) if i not in ties_all]
    assert np.abs(r["w"][rows_r][same] - ro["w"][same]).max() <= parity.W_TOL

    # dispatch of the GPU's own indices: bit-exact
    d = oracle.dispatch(r["idx"], E)
    for key in ("counts", "offsets", "perm", "pair_pos"):
        assert np.array_equal(r[key].ravel(), d[key].ravel()), key

    # activation codes of the sample at every expert-grouped row: bit-exact
    xq = oracle.quantize_x(w, synth.x_rows(w, tokens), mx_mode)
    prow = padded_rows_of(r, tokens, k)
    R = gw.layout["R"]
    nv = w["fmt"] == "nvfp4"
    cb, bs = (H // 2, 16) if nv else (H, 32)
    codes = gw.ws_view("xq_codes", torch.uint8, R * cb).view(R, cb)
    nt = gw.layout["tile_rows"]
    scales = gw.ws_view("xq_scales", torch.uint8, (R // nt) * (H // bs // 4) * 512).cpu().numpy()
    gcodes = codes[torch.from_numpy(prow.ravel()).cuda()].cpu().numpy().reshape(len(tokens), k, cb)
    gsc = untile_scales(scales, R, H // bs, tile_rows=nt)[prow.ravel()].reshape(len(tokens), k, H // bs)
    for j in range(k):
        assert np.array_equal(gcodes[:, j], xq[0])
        assert np.array_equal(gsc[:, j], xq[1])
    if nv:
        gg = gw.ws_view("xq_global", torch.float32, R).cpu().numpy()[prow]
        for j in range(k):
            assert np.array_equal(gg[:, j].view(np.uint32), xq[2].view(np.uint32))

    # the layer on the sample, with the GPU's choice on certified near-ties
    pos = {int(t): i for i, t in enumerate(rows_r)}
    override = {i: ties_all[pos[int(t)]] for i, t in enumerate(tokens) if pos.get(int(t)) in ties_all}
    res = oracle.moe_layer(w, tokens, idx_override=override, cap=cap, mx_mode=mx_mode, keep_pairs=check_h,
                           expert_cache=expert_cache, **gw.route_opts)
    if out_rowwise:
        stats["literal"] = parity.out_error(gpu_out[tokens], res["out"])[0] / parity.out_error(
            gpu_out[tokens], res["out"])[1]
        stats["rowwise"] = parity.check_output_rowwise(gpu_out[tokens], res["out"])
    else:
        stats["err_over_rms"] = parity.check_output(gpu_out[tokens], res["out"])

    if check_h:
        # h = bf16(silu(cap g) cap u) as GEMM1 writes it, or, where GEMM1's
        # epilogue quantises h itself (MXFP8, 64-row tiles), the h codes and
        # block scales.  Near-exact: the GEMM accumulation order differs from
        # the oracle's.
        h_in_ws = gw.layout["hq_codes"] > gw.layout["h_bf16"]
        # NVFP4 with per-row globals: the row pass's codes, block scales and
        # global of the GPU's own h rows, bit-exact against the oracle's
        # quantiser of the same bf16 values
        hq_exact = h_in_ws and gw.act_static is None
        if hq_exact:
            hqc = gw.ws_view("hq_codes", torch.uint8, R * (F // 2)).view(R, F // 2)
            hqs = untile_scales(gw.ws_view("hq_scales", torch.uint8, (R // nt) * (F // 16 // 4) * 512).cpu().numpy(),
                                R, F // 16, tile_rows=nt)
            hqg = gw.ws_view("hq_global", torch.float32, R).cpu().numpy()
        if h_in_ws:
            hbuf = gw.ws_view("h_bf16", torch.int16, R * F).view(R, F)
        else:
            hbuf = gw.ws_view("hq_codes", torch.uint8, R * F).view(R, F)
            hs = untile_scales(gw.ws_view("hq_scales", torch.uint8, (R // nt) * (F // 32 // 4) * 512).cpu().numpy(),
                               R, F // 32, tile_rows=nt)
        flips, total, sflips, stotal = 0, 0, 0, 0
        od = res["dispatch"]
        for e, pr in res["pairs"].items():
            lo, hi = od["offsets"][e], od["offsets"][e + 1]
            pids = od["perm"][lo:hi]
            grow = prow[pids // k, pids % k]
            gh = hbuf[torch.from_numpy(grow).cuda()].cpu().numpy()
            if h_in_ws:
                flips += int((gh.view(np.uint16) != pr["h_bf16"]).sum())
                if hq_exact:
                    q = oracle.quantize("nvfp4", oracle.bf16_bits_to_f32(gh.view(np.uint16)))
                    gi = torch.from_numpy(grow).cuda()
                    assert np.array_equal(hqc[gi].cpu().numpy(), q[0])
                    assert np.array_equal(hqs[grow], q[1])
                    assert np.array_equal(hqg[grow].view(np.uint32), q[2].view(np.uint32))
            else:
                flips += int((gh != pr["hq_codes"]).sum())
                sflips += int((hs[grow] != pr["hq_sf"]).sum())
                stotal += pr["hq_sf"].size
            total += gh.size
        stats["h_flip_rate"] = flips / max(total, 1)
        assert stats["h_flip_rate"] < 0.01
        if not h_in_ws:
            stats["h_scale_flip_rate"] = sflips / max(stotal, 1)
            assert stats["h_scale_flip_rate"] < 0.01
    return stats


@pytest.mark.parametrize("name", list(SMALL))
def test_small_layer_all_tokens(name):
    gw = GpuWorkload(SMALL[name], torch)
    st = check_layer(gw, out_rowwise=gw.w["outlier_frac"] > 0)
    print(name, st)


def test_small_layer_uncapped_and_mx_round_up():
    gw = GpuWorkload("tiny_mxfp8", torch, cap=0.0, mx_scale_mode=1)
    print(check_layer(gw, cap=0.0, mx_mode=1))
    gw = GpuWorkload(SMALL["tiny_nvfp4"], torch, cap=0.0)
    print(check_layer(gw, cap=0.0))


@pytest.mark.parametrize("name", ["tiny_nvfp4", "ragged_mxfp8", "tc_router_nvfp4", "tc_router_mxfp8_outliers"])
@pytest.mark.parametrize("opts", [dict(bias_in_weights=1), dict(routed_scale=2.5),
                                  dict(bias_in_weights=1, routed_scale=2.5)])
def test_router_options_through_the_layer(name, opts):
    # moe_config.bias_in_weights (weights from the biased keys) and
    # routed_scale, on the decode router (T <= 256) and the tensor-core
    # router (T > 256): routing bit-exact, weights within W_TOL, the output
    # within tolerance
    gw = GpuWorkload(SMALL[name], torch, **opts)
    st = check_layer(gw, out_rowwise=gw.w["outlier_frac"] > 0, check_h=False)
    w = gw.routing()["w"].astype(np.float64)
    assert np.allclose(w.sum(1), opts.get("routed_scale", 1.0), atol=1e-5)
    print(name, opts, st)


@pytest.mark.parametrize("name", ["ragged_mxfp8", "tc_router_nvfp4"])
def test_staged_calls_equal_forward(name):
    gw = GpuWorkload(SMALL[name], torch)
    ref = gw.forward().clone()
    c, T, k, E, H = gw.cfg, gw.w["T"], gw.w["k"], gw.w["E"], gw.w["H"]
    dev = "cuda"
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    pp = torch.empty((T, k), dtype=torch.int32, device=dev)
    y = torch.empty(moe.moe_y_bytes(c), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty_like(gw.ws)
    moe.moe_route(c, gw.x, gw.w_router, gw.bias, idx, wts, ws)
    moe.moe_dispatch(c, idx, counts, offsets, perm, pp, ws)
    moe.moe_expert_ffn(c, gw.x, idx, offsets, perm, pp, gw.qw["gate"], gw.qw["up"], gw.qw["down"], y, ws)
    moe.moe_combine(c, y, wts, pp, out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # deterministic across runs
    again = gw.forward()
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))


def sample_tokens(w, n, extra=()):
    rng = np.random.default_rng(1000 + w["seed"])
    toks = set(int(t) for t in extra)
    toks.add(0)
    toks.add(w["T"] - 1)
    while len(toks) < min(n, w["T"]):
        toks.add(int(rng.integers(0, w["T"])))
    return np.array(sorted(toks))


def tile_focus(r, nt, n_tail=4):
    """The most loaded expert and n_tail more experts (the most loaded first)
    whose last token tile is ragged (count % nt != 0) and which span more
    than one tile."""
    counts = r["counts"]
    order = [int(e) for e in np.argsort(-counts, kind="stable")]
    hot = order[0]
    tails = [e for e in order[1:] if counts[e] > nt and counts[e] % nt][:n_tail]
    if len(tails) < n_tail:
        tails += [e for e in order[1:] if counts[e] % nt and e not in tails][:n_tail - len(tails)]
    return hot, tails


def focus_sample(w, r, nt, n=48):
    """>= n tokens for the output check of a large batch: rows of the most
    loaded expert (its first tile, a middle row, its last ragged tile), the
    last ragged tile of four more experts, the outlier rows, the first and
    last token; the rest filled with tokens (from a seeded pool) that add the
    fewest experts not yet in the sample, so that the oracle decodes few
    experts."""
    T, k = w["T"], r["idx"].shape[1]
    counts, offsets, perm, idx = r["counts"], r["offsets"], r["perm"], r["idx"]
    hot, tails = tile_focus(r, nt)
    toks = {0, T - 1}
    c = int(counts[hot])
    for p in sorted({0, 1, min(2, c - 1), c // 2, (c - 1) // nt * nt, c - 1}):
        toks.add(int(perm[offsets[hot] + p]) // k)
    for e in tails:
        c = int(counts[e])
        for p in ((c - 1) // nt * nt, c - 1):
            toks.add(int(perm[offsets[e] + p]) // k)
    if w["outlier_frac"] > 0:
        toks.update(int(t) for t in np.nonzero(synth.outlier_flags(w))[0])
    experts = set(int(e) for t in toks for e in idx[t])
    pool = [int(t) for t in np.random.default_rng(2000 + w["seed"]).permutation(T)[:4096]]
    while len(toks) < min(n, T):
        best = min((t for t in pool if t not in toks), key=lambda t: len(set(idx[t].tolist()) - experts))
        toks.add(best)
        experts.update(int(e) for e in idx[best])
    return np.array(sorted(toks)), hot, tails


def check_pair_rows(gw, r, experts, cache, max_rows=256):
    """GEMM2 on the GPU's own h: y of the pairs in the first and the last
    token tile of each expert (every row of a ragged tail) against
    W_down_e . h^, with h^ the decoded h codes / scales (/ globals) that the
    GPU wrote for those rows and W_down_e the oracle's decoded expert (fp64).
    The products of the two encodings are exact, so the GPU's y differs only
    by its fp32 accumulation over F and the epilogue's scale multiply:
    |dy| <= 2^-12 sum_f |h^_f w_of| (the bound of an fp32 sum of F = 2304
    terms is below 2^-12 even with truncating adds), plus, for the compact y
    rows, their rounding to 11 significant bits (2^-11 of the fp32 value).
    (The h codes themselves are checked against the oracle by their flip
    rate, and the layer output end to end.)"""
    w, k, H, F = gw.w, gw.w["k"], gw.w["H"], gw.w["F"]
    nt = gw.layout["tile_rows"]
    R = gw.layout["R"]
    P = w["T"] * k
    nv = w["fmt"] == "nvfp4"
    yraw = gw.y_raw()
    rel = parity.y_rel(moe, gw.cfg)
    cb, bs = (F // 2, 16) if nv else (F, 32)
    hq = gw.ws_view("hq_codes", torch.uint8, R * cb).view(R, cb)
    hs_all = untile_scales(gw.ws_view("hq_scales", torch.uint8, (R // nt) * (F // bs // 4) * 512).cpu().numpy(),
                           R, F // bs, tile_rows=nt)
    hg_all = gw.ws_view("hq_global", torch.float32, R).cpu().numpy() if nv else None
    worst = 0.0
    for e in experts:
        c, lo, seg = int(r["counts"][e]), int(r["offsets"][e]), int(r["seg_start"][e])
        ps = sorted(set(range(min(c, nt))) | set(range((c - 1) // nt * nt, c)))[:max_rows]
        ps = np.asarray(ps, np.int64)
        rows = seg + ps                                  # padded expert-grouped rows
        hc = hq[torch.from_numpy(rows).cuda()].cpu().numpy()
        h = oracle.decode(w["fmt"], hc, hs_all[rows], hg_all[rows] if nv else None)
        if e not in cache:
            cache[e] = oracle.quantized_expert(w, e)
        wd = oracle.decode(w["fmt"], *cache[e]["down"], per_tensor=True)
        y_ref = h @ wd.T
        acc = 2.0 ** -12 * (np.abs(h) @ np.abs(wd).T)
        bound = acc + rel * (np.abs(y_ref) + acc) + 1e-30
        y_gpu = parity.y_rows_f64(moe, gw.cfg, yraw, ps + lo)
        err = np.abs(y_gpu - y_ref)
        assert np.all(err <= bound), f"expert {e}: |dy| above the accumulation bound at {np.argmax(err / bound)}"
        worst = max(worst, float((err / bound).max()))
    return worst


def check_combine_rows(gw, r, out_gpu, tokens):
    """The combine on the GPU's own y and weights: out[t] = bf16(sum_j w y)
    within half a bf16 ulp plus the fp32 summation error."""
    k, H = gw.w["k"], gw.w["H"]
    pp = r["pair_pos"][tokens]
    y = parity.y_rows_f64(moe, gw.cfg, gw.y_raw(), pp.ravel()).reshape(len(tokens), k, H)
    wt = r["w"][tokens].astype(np.float64)
    ref = np.einsum("tj,tjh->th", wt, y)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-6 * np.einsum("tj,tjh->th", np.abs(wt), np.abs(y)) + 1e-30
    assert np.all(np.abs(out_gpu[tokens] - ref) <= bound)


FULL = ["decode1_nvfp4", "decode8_nvfp4", "decode32_mxfp8", "decode64_nvfp4", "decode192_mxfp8_outliers",
        "prefill4096_nvfp4", "prefill16384_mxfp8_zipf"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    # every token's routing and dispatch; x codes, output rows (and, above
    # 1000 tokens, GEMM2's y rows of the most loaded expert and of four
    # ragged tile tails, and the combine of 1024 tokens) of a sample
    w = synth.WORKLOADS[name]
    gw = GpuWorkload(name, torch)
    big = w["T"] > 1000
    cache = {}
    if big:
        gw.forward()
        r = gw.routing()
        tokens, hot, tails = focus_sample(w, r, gw.layout["tile_rows"], 48)
    else:
        extra = list(np.nonzero(synth.outlier_flags(w))[0]) if w["outlier_frac"] > 0 else []
        tokens = sample_tokens(w, 8, extra)
    st = check_layer(gw, tokens, out_rowwise=w["outlier_frac"] > 0, route_all=True, expert_cache=cache)
    st["sample_tokens"] = len(tokens)
    if big:
        r = gw.routing()
        st["gemm2_err_over_bound"] = check_pair_rows(gw, r, [hot] + tails, cache)
        out = parity.bf16_to_f64(gw.out)
        check_combine_rows(gw, r, out, np.sort(np.random.default_rng(3).choice(w["T"], 1024, replace=False)))
        st["experts_decoded"] = len(cache)
    print(name, st)
    del gw
    torch.cuda.empty_cache()
