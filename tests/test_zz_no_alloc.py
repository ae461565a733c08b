"""The allocation-free dispatch send against the oracle and the regular one (GPU).

moe_dispatch_send_noalloc serves callers that cannot allocate device memory: code that
runs under a memory plan fixed before serving starts, allocator hooks that must not call
back into the allocator, and hosts that hand the library only tensors they already own.
It keeps its send buffer in a device array built into the library instead of taking one
from the caller. This file is named to be collected last, so a stop at its first failure
has already run every other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

CASES = [
    (workloads.Workload("noalloc-bf16", 8, 32, 2048, 64, 8, "bf16", "uniform", 201), 0),
    (workloads.Workload("noalloc-fp8", 8, 24, 1024, 32, 4, "fp8", "zipf", 202), 0),
    # fp8 rows of 660 bytes (not a multiple of 16): the 4-byte register mover through the array
    (workloads.Workload("noalloc-fp8-row660", 4, 40, 640, 32, 6, "fp8", "uniform", 203), 0),
    # the direct-push flag on the layout: this entry point still packs and scatters
    (workloads.Workload("noalloc-bf16-pushflag", 4, 48, 1024, 16, 4, "bf16", "skew0", 204), 8),
]


def _recv_of(ep, fn):
    ep.recv.fill_(0x5A)
    fn()
    code, _ = ep.status()
    assert code == 0
    n = ep.layout_arrays()["rtot"].cpu().numpy()
    r = ep.recv.cpu().numpy()
    return [r[d, :n[d]].copy() for d in range(ep.N)], r, n


@pytest.mark.parametrize("wl,flags", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_noalloc_dispatch_send_matches_oracle_twice(orc, wl, flags):
    from combine_routing_count_gb300 import MoeEP, build, lib
    build.build()
    L = lib()
    inp = workloads.make_inputs(wl)
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload=wl.payload)
    x = torch.from_numpy(inp["x"]).view(torch.bfloat16).cuda()
    ep.layout_step(torch.from_numpy(inp["idx"]).cuda())
    if wl.payload == "fp8":
        ep.quantize(x)
        xin = ep.xq
    else:
        xin = x
    ref, _, _ = _recv_of(ep, lambda: ep.dispatch_send(xin))
    ep.layout.flags = flags
    for _ in range(2):   # two calls in a row share (and overwrite) the library's send array
        got, full, n = _recv_of(ep, lambda: L.moe_dispatch_send_noalloc(
            ctypes.byref(ep.dims), ctypes.byref(ep.layout), xin.data_ptr(), ep.recv.data_ptr(),
            torch.cuda.current_stream().cuda_stream))
        for d in range(wl.N):
            np.testing.assert_array_equal(got[d], o["recv"][d, :n[d]], err_msg=f"receive rows of rank {d} (oracle)")
            np.testing.assert_array_equal(got[d], ref[d], err_msg=f"receive rows of rank {d} (moe_dispatch_send)")
            assert (full[d, n[d]:] == 0x5A).all(), "write beyond the received rows"


def test_noalloc_rejects_sizes_beyond_its_buffer():
    from combine_routing_count_gb300 import MoeEP, lib
    ep = MoeEP(8, 128, 7168, 256, 8)       # 8*128*8 rows of 14336 bytes = 117 MB > 64 MiB
    x = torch.zeros((8, 128, 7168), dtype=torch.bfloat16, device="cuda")
    rc = lib().moe_dispatch_send_noalloc(ctypes.byref(ep.dims), ctypes.byref(ep.layout), x.data_ptr(),
                                         ep.recv.data_ptr(), None)
    assert rc == 1   # MOE_ERR_INVALID_ARG
