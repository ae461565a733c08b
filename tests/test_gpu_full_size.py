"""GPU parity at the full sizes of the benchmark workloads, in the launch configuration the
benchmark times (default mover choice, programmatic dependent launch, the micro-batched
moe_forward, and direct push).

Every buffer is compared with the oracle in full, with no sampling: the layout arrays and
the output on the host; the send, receive, grouped (codes and scales for fp8), dequantised,
combine-send and combine rows on the device, each used row against the oracle's row
(uploaded a rank at a time) and every unused row against the poison it was filled with, so
a stray write anywhere in the hundreds of MB of padding fails. A second pass runs with the
benchmark's aliased buffers (combine reusing the dispatch buffers) and compares the output
again."""
import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import POISON, to_dev, u16

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28   # bytes of oracle rows uploaded per comparison


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_routing_count_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _bytes(t: torch.Tensor) -> torch.Tensor:
    """The tensor's rows as a [rows, bytes] uint8 view (first dimension kept)."""
    return t.contiguous().view(torch.uint8).reshape(t.shape[0], -1)


def _same_rows(dev: torch.Tensor, host: np.ndarray, what: str):
    """dev [n, ...] on the GPU equals host [n, ...] byte for byte (uploaded in chunks)."""
    assert dev.shape[0] == host.shape[0], (what, dev.shape, host.shape)
    if dev.shape[0] == 0:
        return
    d = _bytes(dev)
    h = np.ascontiguousarray(host).view(np.uint8).reshape(d.shape[0], -1)
    assert d.shape == h.shape, (what, d.shape, h.shape)
    step = max(1, CHUNK // max(1, d.shape[1]))
    for i in range(0, d.shape[0], step):
        hc = torch.from_numpy(h[i:i + step]).to(d.device)
        if not torch.equal(d[i:i + step], hc):
            bad = (d[i:i + step] != hc).any(dim=1).nonzero()[:5, 0].cpu().numpy() + i
            raise AssertionError(f"{what}: rows {bad.tolist()} differ from the oracle")


def _poisoned(dev: torch.Tensor, what: str):
    """Every byte of dev still holds the poison (no stray write)."""
    if dev.numel() == 0:
        return
    b = dev.contiguous().view(torch.uint8)
    assert bool((b == POISON).all()), f"{what}: stray write into unused rows"


def _check_buffers(ep, o, wl, push: bool):
    N, L = wl.N, wl.L
    lay = o["layout"]
    rtot, cap = lay["rtot"], lay["cap"]
    nvalid = (lay["pos"] >= 0).reshape(N, -1).sum(axis=1)
    ecnt = np.minimum(lay["ecnt"], cap)
    for s in range(N):
        nv = int(nvalid[s])
        if push:
            _poisoned(ep.send[s], "send (direct push must not write it)")
        else:
            _same_rows(ep.send[s, :nv], o["send"][s, :nv], f"send rank {s}")
            _poisoned(ep.send[s, nv:], f"send rank {s}")
    for d in range(N):
        n = int(rtot[d])
        _same_rows(ep.recv[d, :n], o["recv"][d, :n], f"recv rank {d}")
        _poisoned(ep.recv[d, n:], f"recv rank {d}")
    for d in range(N):
        for l in range(L):
            n = int(ecnt[d, l])
            if wl.payload == "fp8":
                _same_rows(ep.expert_x[d, l, :n], o["exq"][d, l, :n], f"expert codes {d}/{l}")
                _same_rows(ep.expert_scale[d, l, :n], o["exs"][d, l, :n], f"expert scales {d}/{l}")
                _poisoned(ep.expert_x[d, l, n:], f"expert codes {d}/{l}")
                _poisoned(ep.expert_scale[d, l, n:], f"expert scales {d}/{l}")
                _same_rows(ep.expert_y[d, l, :n], o["ey"][d, l, :n], f"dequantised expert rows {d}/{l}")
            else:
                _same_rows(ep.expert_x[d, l, :n], o["ex"][d, l, :n], f"grouped rows {d}/{l}")
                _poisoned(ep.expert_x[d, l, n:], f"grouped rows {d}/{l}")
    kept = (lay["slot"] >= 0).reshape(N, -1)
    assert kept.sum() == (lay["pos"] >= 0).sum(), "full-size workloads drop no pair"
    for d in range(N):
        n = int(rtot[d])
        if push:
            _poisoned(ep.csend[d], "combine send (direct push must not write it)")
        else:
            _same_rows(ep.csend[d, :n], o["csend"][d, :n], f"combine send rank {d}")
            _poisoned(ep.csend[d, n:], f"combine send rank {d}")
    for s in range(N):
        nv = int(nvalid[s])
        _same_rows(ep.crecv[s, :nv], o["crecv"][s, :nv], f"combine rows rank {s}")
        _poisoned(ep.crecv[s, nv:], f"combine rows rank {s}")


@pytest.mark.parametrize("push", [False, True], ids=["scatter", "push"])
@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_matches_oracle(orc, cfg, push):
    from combine_routing_count_gb300 import MoeEP
    wl = workloads.config(cfg)
    inp = workloads.make_inputs(wl)
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    lay_o = o["layout"]
    x, idx, w = to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"])

    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, flags=8 if push else 0)
    for t in (ep.send, ep.recv, ep.expert_x, ep.csend, ep.crecv):
        t.view(torch.uint8).fill_(POISON)
    if ep.expert_scale is not None:
        ep.expert_scale.view(torch.uint8).fill_(POISON)
    ep.forward(x, idx, w)
    code, bits = ep.status()
    assert bits == lay_o["status"] and code == 0
    np.testing.assert_array_equal(u16(ep.out.cpu()), o["out"], err_msg="combine output")
    got = {k: v.cpu().numpy() for k, v in ep.layout_arrays().items()}
    for k in ("cnt", "C", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow", "slot", "slot_src", "recv_src"):
        np.testing.assert_array_equal(got[k], lay_o[k], err_msg=k)
    _check_buffers(ep, o, wl, push)

    # the benchmark's buffer reuse: combine writes into the dispatch buffers
    if wl.payload == "bf16":
        del ep
        torch.cuda.empty_cache()
        ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, alias_buffers=True, flags=8 if push else 0)
        for _ in range(2):
            ep.forward(x, idx, w)
        code, _ = ep.status()
        assert code == 0
        np.testing.assert_array_equal(u16(ep.out.cpu()), o["out"], err_msg="combine output (aliased buffers)")
