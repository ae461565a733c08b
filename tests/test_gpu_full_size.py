"""GPU parity at the full sizes of the benchmark workloads, in the launch configuration the
benchmark times (default mover choice, programmatic dependent launch, and direct push).

The whole output and every layout array are compared bit for bit with the oracle; the
receive, grouped and combine rows (hundreds of MB) are compared on a seeded sample of rows.
A second pass runs with the benchmark's aliased buffers (combine reusing the dispatch
buffers) and compares the output again."""
import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import to_dev, u8, u16

pytestmark = pytest.mark.gpu

SAMPLE = 768


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_routing_count_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _rows(t: torch.Tensor, index: tuple) -> np.ndarray:
    """Gathers rows t[index] on the device, then copies only those to the host."""
    return t[tuple(torch.as_tensor(i, device=t.device, dtype=torch.long) for i in index)].cpu()


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
    ep.forward(x, idx, w)
    code, bits = ep.status()
    assert bits == lay_o["status"] and code == 0
    np.testing.assert_array_equal(u16(ep.out.cpu()), o["out"], err_msg="combine output")
    got = {k: v.cpu().numpy() for k, v in ep.layout_arrays().items()}
    for k in ("cnt", "C", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow", "slot", "slot_src", "recv_src"):
        np.testing.assert_array_equal(got[k], lay_o[k], err_msg=k)

    rng = np.random.default_rng(1000 + cfg)
    # receive rows: sampled (d, i) with i < rtot[d]
    rtot = lay_o["rtot"]
    ds = rng.choice(np.flatnonzero(rtot > 0), SAMPLE)
    iis = (rng.random(SAMPLE) * rtot[ds]).astype(np.int64)
    np.testing.assert_array_equal(u8(_rows(ep.recv, (ds, iis))), o["recv"][ds, iis], err_msg="receive rows")
    # grouped rows: sampled (d, l, j) with j < min(ecnt, cap)
    ecnt = np.minimum(lay_o["ecnt"], lay_o["cap"]).reshape(-1)
    es = rng.choice(np.flatnonzero(ecnt > 0), SAMPLE)
    js = (rng.random(SAMPLE) * ecnt[es]).astype(np.int64)
    dd, ll = es // wl.L, es % wl.L
    if wl.payload == "fp8":
        np.testing.assert_array_equal(u8(_rows(ep.expert_x, (dd, ll, js))), o["exq"][dd, ll, js], err_msg="codes")
        exs_o = o["exs"].view(np.uint8).reshape(o["exs"].shape[:3] + (-1,))
        np.testing.assert_array_equal(u8(_rows(ep.expert_scale, (dd, ll, js))), exs_o[dd, ll, js], err_msg="scales")
    else:
        np.testing.assert_array_equal(u16(_rows(ep.expert_x, (dd, ll, js))), o["ex"][dd, ll, js], err_msg="grouped rows")
    # combine rows back at the sources: sampled kept pairs (s, pos)
    pos, slot = lay_o["pos"].reshape(wl.N, -1), lay_o["slot"].reshape(wl.N, -1)
    kept = np.argwhere(slot >= 0)
    pick = kept[rng.integers(0, len(kept), SAMPLE)]
    ss, pp = pick[:, 0], pos[pick[:, 0], pick[:, 1]]
    np.testing.assert_array_equal(u16(_rows(ep.crecv, (ss, pp))), o["crecv"][ss, pp], err_msg="combine rows")

    # the benchmark's buffer reuse: combine writes into the dispatch buffers
    if wl.payload == "bf16":
        del ep
        ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, alias_buffers=True, flags=8 if push else 0)
        for _ in range(2):
            ep.forward(x, idx, w)
        code, _ = ep.status()
        assert code == 0
        np.testing.assert_array_equal(u16(ep.out.cpu()), o["out"], err_msg="combine output (aliased buffers)")
