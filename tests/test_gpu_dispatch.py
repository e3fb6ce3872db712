"""moe_dispatch on its own, on expert choices built directly (every row k
distinct experts): counts, offsets, perm and pair_pos bit-exact against the
oracle's dispatch, and the tile plan the library keeps in the workspace
against its plain definition.  Covers the one-CTA path at its limits
(T = 256 with E = 1024 and k = 32; heavy skew; a single token) and the
chunked path."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402


def choices(T, E, k, seed, skew=False):
    """[T, k] distinct experts per row; skew: low expert ids are far more likely."""
    rng = np.random.default_rng(seed)
    idx = np.empty((T, k), np.int32)
    p = None
    if skew:
        p = 1.0 / (np.arange(E) + 1.0) ** 1.5
        p /= p.sum()
    for t in range(T):
        idx[t] = rng.choice(E, size=k, replace=False, p=p)
    return idx


def ws_ints(ws, off, n):
    return ws[off:off + 4 * n].view(torch.int32).cpu().numpy()


CASES = {
    "one_cta_limit": dict(T=256, E=1024, k=32, seed=1),
    "one_cta_skewed": dict(T=256, E=16, k=8, seed=2, skew=True),
    "one_token": dict(T=1, E=384, k=8, seed=3),
    "ragged_small": dict(T=37, E=8, k=3, seed=4),
    "chunked": dict(T=3000, E=384, k=8, seed=5, skew=True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_dispatch_and_tile_plan(name):
    cs = CASES[name]
    T, E, k = cs["T"], cs["E"], cs["k"]
    idx_h = choices(T, E, k, cs["seed"], cs.get("skew", False))
    c = moe.make_config(T, 256, E, k, 256, "nvfp4")
    dev = "cuda"
    idx = torch.from_numpy(idx_h).to(dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    pp = torch.empty((T, k), dtype=torch.int32, device=dev)
    ws = torch.empty(moe.moe_workspace_size(c), dtype=torch.uint8, device=dev)
    moe.moe_dispatch(c, idx, counts, offsets, perm, pp, ws)
    torch.cuda.synchronize()
    d = oracle.dispatch(idx_h, E)
    assert np.array_equal(counts.cpu().numpy(), d["counts"])
    assert np.array_equal(offsets.cpu().numpy(), d["offsets"])
    assert np.array_equal(perm.cpu().numpy(), d["perm"])
    assert np.array_equal(pp.cpu().numpy(), d["pair_pos"])

    # tile plan: each expert's rows start at a multiple of nt, one tile per
    # nt of its pairs, in expert order
    L = moe.moe_workspace_layout(c)
    nt = L["tile_rows"]
    cnt = d["counts"].astype(np.int64)
    nrt = (cnt + nt - 1) // nt
    rt_base = np.concatenate([[0], np.cumsum(nrt)])
    seg = rt_base * nt
    assert np.array_equal(ws_ints(ws, L["rt_base"], E + 1), rt_base)
    assert np.array_equal(ws_ints(ws, L["seg_start"], E + 1), seg)
    tiles = ws_ints(ws, L["tiles"], 4 * int(rt_base[-1])).reshape(-1, 4)
    want = []
    for e in range(E):
        for i in range(int(nrt[e])):
            want.append((e, seg[e] + nt * i, min(nt, cnt[e] - nt * i), d["offsets"][e] + nt * i))
    assert np.array_equal(tiles, np.array(want, np.int64).reshape(-1, 4))
