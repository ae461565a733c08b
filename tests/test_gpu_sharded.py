"""Expert parallelism over rank windows on the GPU: the sharded pass (combine_routing_count_gb300
.sharded) against the oracle, bit for bit.

G windows of one group run on one GPU in one process (LocalTransport moves the slices
between them); every window's receive, grouped and combine rows and its output must be the
oracle's rows for its ranks. The single-window case runs through a one-process
torch.distributed group (DistTransport), the code path of one process per GPU."""
import ctypes
import os
import socket

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import to_dev, u8, u16

pytestmark = pytest.mark.gpu

W = workloads.Workload
CASES = [
    W("shard-uniform", 4, 24, 1024, 16, 4, "bf16", "uniform", 601),
    W("shard-zipf", 6, 20, 2048, 24, 6, "bf16", "zipf", 602),
    W("shard-skew", 4, 32, 512, 16, 4, "bf16", "skew0", 603),
    W("shard-fp8", 4, 16, 1024, 32, 4, "fp8", "uniform", 604),
    W("shard-fp8-row660", 3, 10, 640, 12, 3, "fp8", "zipf", 605),
    W("shard-cap", 4, 16, 256, 8, 4, "bf16", "zipf", 606, cap=9),
    W("shard-ep8-shape", 8, 32, 7168, 256, 8, "bf16", "uniform", 607),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_routing_count_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _inputs(wl, bad_id=False):
    inp = workloads.make_inputs(wl)
    if bad_id:
        inp["idx"] = inp["idx"].copy()
        inp["idx"][1, 2, 0] = -1
        inp["idx"][0, 0, 1] = wl.E + 3
    return inp


def _check_window(o, wl, sh, lo, hi):
    lay = o["layout"]
    rtot, ecnt, cap = lay["rtot"], np.minimum(lay["ecnt"], lay["cap"]), lay["cap"]
    np.testing.assert_array_equal(u16(sh.out.cpu()), o["out"][lo:hi], err_msg="output")
    recv = u8(sh.recv.cpu())
    for i, d in enumerate(range(lo, hi)):
        np.testing.assert_array_equal(recv[i, :rtot[d]], o["recv"][d, :rtot[d]], err_msg=f"receive rows of rank {d}")
    if wl.payload == "fp8":
        ex, exs = u8(sh.expert_x.cpu()), u8(sh.expert_scale.cpu())
        exs_o = o["exs"].view(np.uint8).reshape(o["exs"].shape[:3] + (-1,))
        ey = u16(sh.expert_y.cpu())
        for i, d in enumerate(range(lo, hi)):
            for l in range(wl.L):
                n = ecnt[d, l]
                np.testing.assert_array_equal(ex[i, l, :n], o["exq"][d, l, :n], err_msg="expert codes")
                np.testing.assert_array_equal(exs[i, l, :n], exs_o[d, l, :n], err_msg="expert scales")
                np.testing.assert_array_equal(ey[i, l, :n], o["ey"][d, l, :n], err_msg="dequantised rows")
    else:
        ex = u16(sh.expert_x.cpu())
        for i, d in enumerate(range(lo, hi)):
            for l in range(wl.L):
                n = ecnt[d, l]
                np.testing.assert_array_equal(ex[i, l, :n], o["ex"][d, l, :n], err_msg=f"grouped rows {d}/{l}")
    crecv = u16(sh.crecv.cpu())
    pos, slot = lay["pos"], lay["slot"]
    for i, s in enumerate(range(lo, hi)):
        rows = pos[s][(slot[s] >= 0)]
        np.testing.assert_array_equal(crecv[i][rows], o["crecv"][s][rows], err_msg=f"combine rows of rank {s}")


def _run_local(wl, inp, G):
    from combine_routing_count_gb300.sharded import LocalTransport, ShardedEP, sharded_forward, window_bounds
    b = window_bounds(wl.N, G)
    shards = [ShardedEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, bounds=b, me=g) for g in range(G)]
    x = to_dev(inp["x"]).view(torch.bfloat16)
    idx, w = to_dev(inp["idx"]), to_dev(inp["w"])
    parts = lambda t: [t[b[g]:b[g + 1]].contiguous() for g in range(G)]   # noqa: E731
    for _ in range(2):   # a second pass on the same buffers: counters and plans start over
        sharded_forward(shards, LocalTransport(), parts(x), parts(idx), parts(w))
    return shards, b


@pytest.mark.parametrize("G", [2, 3, 4])
@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_windows_on_one_gpu_match_oracle(orc, wl, G):
    if G > wl.N:
        pytest.skip("more windows than ranks")
    inp = _inputs(wl, bad_id=(wl.name == "shard-cap"))
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    shards, b = _run_local(wl, inp, G)
    for g, sh in enumerate(shards):
        code, bits = sh.status()
        assert bits == o["layout"]["status"], (bits, o["layout"]["status"])
        _check_window(o, wl, sh, b[g], b[g + 1])


def test_one_window_through_a_process_group(orc):
    """G = 1 through torch.distributed (NCCL, one process): the path of one process per GPU."""
    import torch.distributed as dist

    from combine_routing_count_gb300.sharded import DistTransport, ShardedEP, sharded_forward, window_bounds
    wl = CASES[3]
    inp = _inputs(wl)
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        b = window_bounds(wl.N, 1)
        sh = ShardedEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, bounds=b, me=0)
        sharded_forward([sh], DistTransport(), [to_dev(inp["x"]).view(torch.bfloat16)], [to_dev(inp["idx"])],
                        [to_dev(inp["w"])])
        code, _ = sh.status()
        assert code == 0
        _check_window(o, wl, sh, 0, wl.N)
        assert all(len(v) == 0 for v in sh.plans.values()), "one window exchanges nothing"
    finally:
        dist.destroy_process_group()


def test_window_rejections():
    """A rank window works only with the calls that support it, and never with direct push."""
    from combine_routing_count_gb300 import MoeEP, lib
    ep = MoeEP(4, 8, 256, 8, 2)
    L = lib()
    x = torch.zeros((4, 8, 256), dtype=torch.bfloat16, device="cuda")
    ep.layout.win_lo, ep.layout.win_hi = 1, 3
    b = ep.buffers(x, torch.zeros((4, 8, 2), dtype=torch.int32, device="cuda"),
                   torch.zeros((4, 8, 2), dtype=torch.float32, device="cuda"))
    n0 = L.moe_launch_count()
    assert L.moe_forward(ctypes.byref(ep.dims), ctypes.byref(ep.layout), ctypes.byref(b), None) == 1
    assert L.moe_dispatch(ctypes.byref(ep.dims), ctypes.byref(ep.layout), x.data_ptr(), ep.send.data_ptr(),
                          ep.recv.data_ptr(), ep.expert_x.data_ptr(), None, None) == 1
    assert L.moe_dispatch_split(ctypes.byref(ep.dims), ctypes.byref(ep.layout), x.data_ptr(), ep.recv.data_ptr(),
                                ep.expert_x.data_ptr(), None, -1, None) == 1
    ep.layout.flags = 8   # direct push with a window
    assert L.moe_dispatch_send(ctypes.byref(ep.dims), ctypes.byref(ep.layout), x.data_ptr(), ep.send.data_ptr(),
                               ep.recv.data_ptr(), None) == 1
    ep.layout.flags = 0
    for lo, hi in ((2, 2), (3, 1), (-1, 2), (0, 5)):
        ep.layout.win_lo, ep.layout.win_hi = lo, hi
        assert L.moe_dispatch_send(ctypes.byref(ep.dims), ctypes.byref(ep.layout), x.data_ptr(),
                                   ep.send.data_ptr(), ep.recv.data_ptr(), None) == 1
    assert L.moe_launch_count() == n0


def _fuzz_window_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        N = int(rng.integers(2, 9))
        L = int(rng.integers(1, 6))
        R = int(rng.integers(1, min(8, N * L) + 1))
        T = int(rng.integers(1, 24))
        payload = "fp8" if rng.random() < 0.3 else "bf16"
        H = int(rng.choice([128, 256, 640, 1024])) if payload == "fp8" else int(rng.choice([64, 136, 512, 1024]))
        routing = str(rng.choice(["uniform", "zipf", "skew0"])) if R <= L else str(rng.choice(["uniform", "zipf"]))
        cap = int(rng.integers(1, N * T + 1)) if rng.random() < 0.25 else 0
        G = int(rng.integers(2, N + 1))
        out.append((W(f"wfuzz{i}-N{N}-G{G}", N, T, H, N * L, R, payload, routing, 700 + i, cap=cap), G))
    return out


@pytest.mark.parametrize("wl,G", _fuzz_window_cases(30, 71), ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_fuzz_windows_match_oracle(orc, wl, G):
    """Random shapes (ranks, experts per rank, R, tokens, row sizes including 16-byte-unaligned
    fp8 rows, routing, capacity drops) split into 2..N windows on one GPU: every window bit
    for bit against the oracle."""
    inp = _inputs(wl)
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    shards, b = _run_local(wl, inp, G)
    for g, sh in enumerate(shards):
        _, bits = sh.status()
        assert bits == o["layout"]["status"]
        _check_window(o, wl, sh, b[g], b[g + 1])
