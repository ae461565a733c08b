"""Host side of expert parallelism over several processes (no GPU): the exchange plan and the
slice exchange between rank windows.

The plan (moe_exchange_plan, host code of libmoe_ep) is built from the oracle's layout of the
gathered routing and checked slice by slice against the oracle's send and receive buffers;
two gloo processes then gather their routing, plan, and move the oracle's rows between
their windows with the sharded driver's transport, and each checks that the rows it
received are the oracle's."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import workloads

CASES = [
    workloads.Workload("shard-uniform", 4, 9, 128, 16, 3, "bf16", "uniform", 501),
    workloads.Workload("shard-zipf", 6, 7, 256, 24, 4, "bf16", "zipf", 502),
    workloads.Workload("shard-skew", 4, 8, 128, 8, 2, "bf16", "skew0", 503),
    workloads.Workload("shard-fp8", 4, 6, 256, 8, 2, "fp8", "uniform", 504),
]


def _local(buf: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """The window-local part of a whole-group buffer [N, rows, ...] as [n * rows, ...]."""
    return buf[lo:hi].reshape((-1,) + buf.shape[2:])


def _oracle(orc, wl, inp):
    return orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])


def _dims(wl):
    from combine_routing_count_gb300 import MoeDims, MOE_PAYLOAD_BF16, MOE_PAYLOAD_FP8_E4M3_B128
    return MoeDims(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap,
                   MOE_PAYLOAD_FP8_E4M3_B128 if wl.payload == "fp8" else MOE_PAYLOAD_BF16)


@pytest.mark.parametrize("G", [1, 2, 3])
@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_exchange_plan_against_oracle_buffers(orc, wl, G):
    """Every remote (s, d) slice is listed once by its sender and once by its receiver, with
    C[s][d] rows at the window-local rows where the oracle's send, receive, combine-send and
    combine-receive buffers hold that slice; local slices are listed by no one."""
    _check_plan(orc, wl, G)


def _check_plan(orc, wl, G):
    from combine_routing_count_gb300.sharded import exchange_plan, window_bounds
    inp = workloads.make_inputs(wl)
    o = _oracle(orc, wl, inp)
    lay = o["layout"]
    C, soff, roff = lay["C"], lay["soff"], lay["roff"]
    b = window_bounds(wl.N, G)
    win = np.repeat(np.arange(G), np.diff(b))
    dims = _dims(wl)
    send, recv, csend, crecv = o["send"], o["recv"], o["csend"], o["crecv"]
    for direction in (0, 1):
        sent, got = {}, {}
        for me in range(G):
            lo, hi = b[me], b[me + 1]
            src_buf = _local(send if direction == 0 else csend, lo, hi)
            dst_buf = _local(recv if direction == 0 else crecv, lo, hi)
            for peer, s, d, rows, r0 in exchange_plan(dims, C, soff, roff, b, me, direction, 1):
                assert rows == C[s, d] > 0 and win[s] != win[d]
                assert peer == (win[d] if direction == 0 else win[s]) and me == (win[s] if direction == 0 else win[d])
                assert (s, d) not in sent
                sent[(s, d)] = (me, peer, src_buf[r0:r0 + rows])
            for peer, s, d, rows, r0 in exchange_plan(dims, C, soff, roff, b, me, direction, 0):
                assert rows == C[s, d] > 0 and (s, d) not in got
                got[(s, d)] = (peer, me, dst_buf[r0:r0 + rows])
        remote = {(s, d) for s in range(wl.N) for d in range(wl.N) if C[s, d] > 0 and win[s] != win[d]}
        assert set(sent) == remote and set(got) == remote
        for key in remote:
            p, q, rows_sent = sent[key]
            assert (p, q) == got[key][:2]
            np.testing.assert_array_equal(rows_sent, got[key][2], err_msg=f"slice {key} direction {direction}")
        # order: the k-th slice p sends to q is the k-th q receives from p
        for p in range(G):
            for q in range(G):
                a = [k for k in sorted(sent) if sent[k][:2] == (p, q)]
                c = [k for k in sorted(got) if got[k][:2] == (p, q)]
                assert a == c


def test_exchange_plan_rejects_bad_windows():
    from combine_routing_count_gb300 import lib
    from combine_routing_count_gb300.sharded import exchange_plan
    wl = CASES[0]
    dims = _dims(wl)
    z = np.zeros((wl.N, wl.N), np.int32)
    so = np.zeros((wl.N, wl.E), np.int32)
    for bounds, me in (([0, 2, 3], 0), ([1, 2, wl.N], 0), ([0, 3, 2, wl.N], 1), ([0, wl.N], 1)):
        with pytest.raises(ValueError):
            exchange_plan(dims, z, so, z, bounds, me, 0, 1)
    assert lib().moe_exchange_plan(None, None, None, None, 1, None, 0, 0, 0, None, 0) == -1


def _gloo_worker(rank, port, wl_i, q):
    import torch.distributed as dist

    import oracle
    from combine_routing_count_gb300.sharded import DistTransport, exchange_plan, window_bounds
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        wl = CASES[wl_i]
        inp = workloads.make_inputs(wl)
        b = window_bounds(wl.N, 2)
        lo, hi = b[rank], b[rank + 1]
        # routing exchange: each process holds only its window's ids
        mine = torch.from_numpy(inp["idx"][lo:hi].copy())
        full = torch.empty((wl.N,) + mine.shape[1:], dtype=torch.int32)
        dist.all_gather_into_tensor(full, mine)
        assert np.array_equal(full.numpy(), inp["idx"])
        o = oracle.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], full.numpy(), inp["w"])
        lay = o["layout"]
        dims = _dims(wl)
        tr = DistTransport()
        ok = True
        for direction, src_all, dst_all in ((0, o["send"], o["recv"]), (1, o["csend"], o["crecv"])):
            src = torch.from_numpy(np.ascontiguousarray(_local(src_all, lo, hi)))
            dst = torch.zeros_like(torch.from_numpy(np.ascontiguousarray(_local(dst_all, lo, hi))))
            sends = [(p, src[r0:r0 + rows]) for p, s, d, rows, r0 in
                     exchange_plan(dims, lay["C"], lay["soff"], lay["roff"], b, rank, direction, 1)]
            plan_in = exchange_plan(dims, lay["C"], lay["soff"], lay["roff"], b, rank, direction, 0)
            tr.exchange_views(sends, [(p, dst[r0:r0 + rows]) for p, s, d, rows, r0 in plan_in])
            ref = _local(dst_all, lo, hi)
            for p, s, d, rows, r0 in plan_in:
                ok = ok and np.array_equal(dst[r0:r0 + rows].numpy(), ref[r0:r0 + rows])
        q.put((rank, ok, sum(1 for _ in plan_in)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("wl_i", [0, 2, 3], ids=lambda i: CASES[i].name)
def test_sharded_exchange_gloo_two_ranks(wl_i):
    """Two gloo processes, one window each: routing all-gathered, slices planned and moved
    with the sharded driver's transport; every received slice equals the oracle's rows."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + (os.getpid() + 17 * wl_i) % 1000
    ps = [ctx.Process(target=_gloo_worker, args=(r, port, wl_i, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1] and all(g[1] for g in got)
    assert sum(g[2] for g in got) > 0   # slices crossed windows


def _fuzz_plan_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        N = int(rng.integers(1, 10))
        L = int(rng.integers(1, 5))
        R = int(rng.integers(1, min(6, N * L) + 1))
        T = int(rng.integers(0, 12))
        routing = str(rng.choice(["uniform", "zipf"]))
        G = int(rng.integers(1, N + 1))
        out.append((workloads.Workload(f"pfuzz{i}-N{N}-G{G}", N, T, 64, N * L, R, "bf16", routing, 800 + i), G))
    return out


@pytest.mark.parametrize("wl,G", _fuzz_plan_cases(40, 91), ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_fuzz_exchange_plan(orc, wl, G):
    """Random shapes and window counts (including empty batches and one-rank windows): the
    plan's slices are exactly the remote (s, d) pairs with rows, with matching rows and order."""
    _check_plan(orc, wl, G)
