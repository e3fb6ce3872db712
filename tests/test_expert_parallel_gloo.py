"""Expert-parallel partition plan (block_scaled_fp4_route_gb300.expert_parallel)
on the CPU: the plan's orders against the oracle's dispatch, and 2 and 4 gloo
ranks that each route their own tokens, exchange the encoded activation rows
with all_to_all, run the oracle's expert FFN on the experts they own, send the
outputs back and combine: the result equals the single-process oracle layer
bit for bit, and every receiver's regrouped rows are exactly the oracle's
dispatch order of the whole batch restricted to its experts.  No GPU."""
import os
import socket

import numpy as np
import pytest

import oracle
import synth
from block_scaled_fp4_route_gb300 import expert_parallel as ep

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def test_expert_ranges_cover_every_expert_once():
    for E, G in [(384, 4), (384, 8), (15, 4), (16, 16), (7, 1)]:
        r = ep.expert_ranges(E, G)
        assert r[0][0] == 0 and r[-1][1] == E and all(a[1] == b[0] for a, b in zip(r, r[1:]))
        sizes = [hi - lo for lo, hi in r]
        assert max(sizes) - min(sizes) <= 1
        own = ep.expert_owner(E, G)
        assert all((own[lo:hi] == g).all() for g, (lo, hi) in enumerate(r))
    with pytest.raises(ValueError):
        ep.expert_ranges(4, 5)


def test_local_dispatch_is_the_oracle_dispatch():
    rng = np.random.default_rng(3)
    for T, E, k in [(1, 4, 2), (37, 16, 3), (200, 384, 8)]:
        idx = np.array([rng.choice(E, k, replace=False) for _ in range(T)], np.int32)
        mine, ref = ep.local_dispatch(idx, E), oracle.dispatch(idx, E)
        for key in ("counts", "offsets", "perm", "pair_pos"):
            assert np.array_equal(mine[key], ref[key]), key


def test_plan_receive_regroups_by_expert_then_source():
    # two sources, three experts; received rows labelled (source, expert, n)
    cm = np.array([[2, 0, 1], [1, 3, 0]])
    labels = [(s, e, i) for s in range(2) for e in range(3) for i in range(cm[s, e])]
    p = ep.plan_receive(cm)
    assert list(p["recv_counts"]) == [3, 4]
    grouped = [labels[j] for j in p["grouped_from_recv"]]
    assert grouped == sorted(labels, key=lambda x: (x[1], x[0], x[2]))
    assert list(p["expert_offsets"]) == [0, 3, 6, 7]
    assert [grouped[i] for i in p["recv_from_grouped"]] == labels


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


SPEC = dict(H=256, E=15, k=3, F=128, fmt="mxfp8", seed=51, outlier_frac=0.0, bias="uniform")
T_PER_RANK = 7


def _exchange(send: np.ndarray, send_counts, recv_counts):
    """all_to_all of rows (any dtype, viewed as bytes) with the given splits."""
    width = send.dtype.itemsize * int(np.prod(send.shape[1:]))
    src = torch.from_numpy(np.ascontiguousarray(send).view(np.uint8).reshape(-1, width))
    out = torch.empty((int(sum(recv_counts)), width), dtype=torch.uint8)
    dist.all_to_all_single(out, src, [int(c) for c in recv_counts], [int(c) for c in send_counts])
    return out.numpy().view(send.dtype).reshape((-1,) + send.shape[1:])


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = dict(SPEC, T=T_PER_RANK * world)
        E, k, H = w["E"], w["k"], w["H"]
        lo, hi = ep.expert_ranges(E, world)[rank]
        gtok = np.arange(rank * T_PER_RANK, (rank + 1) * T_PER_RANK)      # this rank's global token ids
        x = synth.x_rows(w, gtok)
        r = oracle.route(x, synth.router_weight(w), synth.router_bias(w), k)
        # encode each token once (its activation global is per row, expert-independent)
        codes, scales, _ = oracle.quantize_x(w, x)
        plan = ep.plan_send(r["idx"], E, world)
        # the small exchange first: per-expert counts of every destination's block
        n_max = max(h - l for l, h in ep.expert_ranges(E, world))
        cm_send = np.zeros((world, n_max), np.int64)
        for d in range(world):
            cm_send[d, :len(plan["expert_counts"][d])] = plan["expert_counts"][d]
        cm_recv = torch.empty((world, n_max), dtype=torch.int64)
        dist.all_to_all_single(cm_recv, torch.from_numpy(cm_send))
        recv = ep.plan_receive(cm_recv.numpy()[:, :hi - lo])
        # the rows: encoded codes and scales, and (for the check) global token ids
        st = plan["send_tokens"]
        rc, rs = _exchange(codes[st], plan["send_counts"], recv["recv_counts"]), \
            _exchange(scales[st], plan["send_counts"], recv["recv_counts"])
        rt = _exchange(gtok[st].astype(np.int64), plan["send_counts"], recv["recv_counts"])
        g = recv["grouped_from_recv"]
        gc, gs, gt = rc[g], rs[g], rt[g]
        # the receiver's grouped order is the whole batch's dispatch order on its experts
        full_idx = oracle.route(synth.x_rows(w, np.arange(w["T"])), synth.router_weight(w),
                                synth.router_bias(w), k)["idx"]
        fd = oracle.dispatch(full_idx, E)
        assert np.array_equal(gt, fd["perm"][fd["offsets"][lo]:fd["offsets"][hi]] // k)
        assert np.array_equal(recv["expert_offsets"], fd["offsets"][lo:hi + 1] - fd["offsets"][lo])
        # the experts this rank owns, on the rows it received
        a = oracle.decode(w["fmt"], gc, gs, None)
        y = np.zeros((len(g), H))
        for e in range(lo, hi):
            s0, s1 = recv["expert_offsets"][e - lo], recv["expert_offsets"][e - lo + 1]
            if s1 > s0:
                dec = oracle.decoded_expert(w, oracle.quantized_expert(w, e))
                y[s0:s1] = oracle.expert_ffn(w["fmt"], dec["gate"], dec["up"], dec["down"], a[s0:s1])["y"]
        # outputs back in received order; they arrive in this rank's dispatch order
        y_back = _exchange(y[recv["recv_from_grouped"]], recv["recv_counts"], plan["send_counts"])
        out = oracle.combine(r["w"], plan["pair_pos"], y_back)
        ref = oracle.moe_layer(w)["out"][gtok]
        q.put((rank, bool(np.array_equal(out, ref)), float(np.abs(out - ref).max()), len(g)))
    except Exception as ex:  # report, so that the parent does not wait for a result that never comes
        q.put((rank, False, repr(ex), -1))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_expert_parallel_exchange_reproduces_the_layer(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ok, err, rows in sorted(out):
        assert ok, (rank, err)
    assert sum(rows for _, _, _, rows in out) == T_PER_RANK * world * SPEC["k"]
