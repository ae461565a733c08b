"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element."""
import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import compare_all, run_gpu, to_dev, u8, u16

pytestmark = pytest.mark.gpu

W = workloads.Workload
# Sizes the oracle finishes in seconds that still span many CTAs and end in ragged tails.
CASES = [
    workloads.config(0),
    W("ragged-bf16-H7168", 4, 37, 7168, 32, 8, "bf16", "uniform", 101),
    W("zipf-bf16-H4096", 6, 23, 4096, 48, 8, "bf16", "zipf", 102),
    W("skew-bf16-H2048", 8, 19, 2048, 64, 8, "bf16", "skew0", 103),
    W("fp8-H7168", 8, 9, 7168, 48, 8, "fp8", "uniform", 104),
    W("fp8-H384-unaligned", 3, 11, 384, 12, 3, "fp8", "uniform", 105),     # rows of 396 bytes
    W("R1-bf16", 5, 13, 1024, 10, 1, "bf16", "uniform", 106),
    W("R3-E-small", 2, 40, 136, 4, 3, "bf16", "uniform", 107),              # H not a multiple of 16
    W("cap-overflow", 4, 16, 512, 8, 2, "bf16", "uniform", 108, cap=5),
    W("R12-gather-batches", 4, 9, 512, 32, 12, "bf16", "uniform", 109),  # R > 8: gathers in batches
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_routing_count_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("flags", [0, 1, 4, 6], ids=["auto", "ldg", "tma", "tma-nopdl"])
@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_path_matches_oracle(orc, wl, flags):
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags)
    compare_all(orc, wl, inp, res)


@pytest.mark.parametrize("flags", [8, 9, 12], ids=["push-auto", "push-ldg", "push-tma"])
@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_direct_push_matches_oracle(orc, wl, flags):
    """Direct push (pack into the owners' receive rows, combine into the sources' rows)
    leaves exactly the canonical receive, grouped and combine contents."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags)
    compare_all(orc, wl, inp, res, push=True)


@pytest.mark.parametrize("flags", [1, 4, 12], ids=["ldg", "tma", "push-tma"])
def test_duplicates_and_bad_ids(orc, flags):
    wl = W("dups", 3, 21, 256, 12, 4, "bf16", "uniform", 110)
    inp = workloads.make_inputs(wl)
    rng = np.random.default_rng(0)
    idx = rng.integers(0, wl.E, size=(wl.N, wl.T, wl.R)).astype(np.int32)   # duplicates allowed
    idx[0, 3, 1] = -1
    idx[2, 5, 0] = wl.E
    idx[1, 7, 3] = 1 << 30
    inp["idx"] = idx
    _, res = run_gpu(wl, inp, flags=flags)
    assert res["status_code"] == 2                      # MOE_ERR_EXPERT_RANGE, no trap
    compare_all(orc, wl, inp, res, push=bool(flags & 8))


@pytest.mark.parametrize("mode", ["forward", "phases"])
@pytest.mark.parametrize("flags", [0, 4, 8], ids=["auto", "tma", "push"])
@pytest.mark.parametrize("payload", ["bf16", "fp8"])
def test_duplicates_and_bad_ids_in_token_batches(orc, payload, flags, mode):
    """Duplicate experts in a token and ids outside [0, E), with the pass split into 3 token
    batches (moe_forward's micro-batches, or moe_dispatch / moe_combine): status bit, no
    trap, every buffer as the oracle's."""
    wl = W("dups-mb", 3, 21, 512, 12, 4, payload, "uniform", 111)
    inp = workloads.make_inputs(wl)
    rng = np.random.default_rng(1)
    idx = rng.integers(0, wl.E, size=(wl.N, wl.T, wl.R)).astype(np.int32)   # duplicates allowed
    idx[0, 3, 1] = -1
    idx[2, 20, 0] = wl.E
    idx[1, 9, 3] = 1 << 30
    inp["idx"] = idx
    _, res = run_gpu(wl, inp, flags=flags, batches=3, **{mode: True})
    assert res["status_code"] == 2                      # MOE_ERR_EXPERT_RANGE, no trap
    compare_all(orc, wl, inp, res, push=bool(flags & 8), fused_quant=True)


def test_random_tiny_layouts_bit_exact(orc):
    from combine_routing_count_gb300 import MoeEP
    rng = np.random.default_rng(1234)
    for i in range(40):
        N = int(rng.integers(1, 6))
        L = int(rng.integers(1, 7))
        E, T, R = N * L, int(rng.integers(0, 40)), int(rng.integers(1, 9))
        cap = int(rng.integers(1, N * T + 1)) if (T and rng.random() < 0.3) else 0
        idx = rng.integers(0, E, size=(N, T, R)).astype(np.int32)
        ep = MoeEP(N, T, 64, E, R, cap)
        ep.layout_step(to_dev(idx))
        code, bits = ep.status()
        got = {k: v.cpu().numpy() for k, v in ep.layout_arrays().items()}
        o = orc.layout(N, T, E, R, cap, idx)
        for k in ("cnt", "C", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow", "slot", "slot_src", "recv_src"):
            np.testing.assert_array_equal(got[k], o[k], err_msg=f"case {i} {k}")
        assert bits == o["status"]


def test_large_pairs_per_rank_layout(orc):
    """T*R well above one 1024-pair chunk per rank (prefill-sized), with duplicates."""
    from combine_routing_count_gb300 import MoeEP
    rng = np.random.default_rng(5)
    N, T, E, R = 4, 1500, 64, 6
    idx = rng.integers(0, E, size=(N, T, R)).astype(np.int32)
    ep = MoeEP(N, T, 64, E, R, 0)
    ep.layout_step(to_dev(idx))
    ep.status()
    got = {k: v.cpu().numpy() for k, v in ep.layout_arrays().items()}
    o = orc.layout(N, T, E, R, 0, idx)
    for k in ("cnt", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow", "slot", "slot_src", "recv_src"):
        np.testing.assert_array_equal(got[k], o[k], err_msg=k)


def test_empty_batch():
    from combine_routing_count_gb300 import MoeEP, lib
    ep = MoeEP(4, 0, 256, 8, 2)
    x = torch.empty((4, 0, 256), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((4, 0, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((4, 0, 2), dtype=torch.float32, device="cuda")
    ep.forward(x, idx, w)
    code, bits = ep.status()
    assert code == 0 and bits == 0
    assert (ep.layout_arrays()["cnt"] == 0).all()


def test_invalid_arguments_launch_nothing():
    import ctypes
    from combine_routing_count_gb300 import MoeEP, lib
    ep = MoeEP(2, 4, 128, 4, 2)
    L = lib()
    n0 = L.moe_launch_count()
    x = torch.zeros((2, 4, 128), dtype=torch.bfloat16, device="cuda")
    # misaligned pointer
    rc = L.moe_dispatch_send(ctypes.byref(ep.dims), ctypes.byref(ep.layout), x.data_ptr() + 2,
                             ep.send.data_ptr(), ep.recv.data_ptr(), None)
    assert rc == 1
    rc = L.moe_combine_recv(ctypes.byref(ep.dims), ctypes.byref(ep.layout), None, None, None, None)
    assert rc == 1
    assert L.moe_launch_count() == n0


# mode: (flags, batches, capacity, pinned, identity expert by aliasing)
HOST_MODES = {
    "pipelined": (0, 0, 0, True, True),              # copy-engine pipeline, automatic batches
    "pipelined-7": (0, 7, 0, True, True),            # 7 uneven batches of 29 tokens
    "pipelined-29": (0, 29, 0, True, True),          # one token per batch
    "pipelined-cap": (0, 5, 9, True, True),          # capacity drops
    "pipelined-copy-expert": (0, 3, 0, True, False), # ranged identity expert into its own buffer
    "pipelined-push": (0x8, 4, 0, True, True),       # direct push in every batch
    "one-batch": (0x40, 0, 0, True, True),
    "pageable": (0, 4, 0, False, True),
    "mapped": (0x20, 0, 0, True, True),              # kernels on the pinned memory, two batches
    "mapped-one-batch": (0x60, 0, 0, True, True),
    "mapped-cap": (0x20, 0, 9, True, True),
}


@pytest.mark.parametrize("mode", list(HOST_MODES))
@pytest.mark.parametrize("payload", ["bf16", "fp8"])
def test_forward_host_matches_device_path(orc, mode, payload):
    """Host inputs and output: copied by the copy-engine pipeline in token batches (default;
    several batch counts, pageable memory too), in one batch (MOE_FLAG_ONE_BATCH), or
    read and written by the kernels directly (MOE_FLAG_HOST_MAPPED); an odd token count,
    with and without capacity drops."""
    flags, nb, cap, pinned, alias = HOST_MODES[mode]
    wl = W("host-e2e", 4, 29, 2048, 16, 4, payload, "zipf", 120, cap=cap)
    inp = workloads.make_inputs(wl)
    from combine_routing_count_gb300 import MoeEP
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, payload=payload, alias_buffers=(payload == "bf16" and alias),
               separate_expert_y=(payload == "bf16" and not alias), flags=flags, batches=nb)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    h_x = pin(torch.from_numpy(inp["x"]).view(torch.bfloat16))
    h_idx = pin(torch.from_numpy(inp["idx"]))
    h_w = pin(torch.from_numpy(inp["w"]))
    h_out = pin(torch.empty((wl.N, wl.T, wl.H), dtype=torch.bfloat16))
    x = torch.empty_like(h_x, device="cuda")
    idx = torch.empty_like(h_idx, device="cuda")
    w = torch.empty_like(h_w, device="cuda")
    for _ in range(2):
        h_out.view(torch.int16).fill_(-1)
        ep.forward_host(h_x, h_idx, h_w, h_out, x, idx, w)
        code, _ = ep.status()
        assert code == (3 if cap else 0)   # 3: capacity drops
        o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, payload, inp["x"], inp["idx"], inp["w"])
        np.testing.assert_array_equal(u16(h_out), o["out"])


def test_launch_counter_counts_kernels():
    from combine_routing_count_gb300 import MoeEP, lib
    wl = workloads.config(0)
    inp = workloads.make_inputs(wl)
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R)
    n0 = lib().moe_launch_count()
    ep.forward(to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"]))
    torch.cuda.synchronize()
    # layout (3) + dispatch (pack, write, shuffle) + combine (pack, write, sum); bf16 identity aliases
    assert lib().moe_launch_count() - n0 == 5
    ep.layout.flags |= 0x80   # MOE_FLAG_SEPARATE_MOVES: the four moves apart
    n0 = lib().moe_launch_count()
    ep.forward(to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"]))
    torch.cuda.synchronize()
    assert lib().moe_launch_count() - n0 == 9


def test_profiling_events_bracket_each_kernel():
    import ctypes
    from combine_routing_count_gb300 import KERNEL_NAMES, MoeEP, MoeProf, lib
    wl = W("prof", 4, 16, 1024, 16, 4, "fp8", "uniform", 130)
    inp = workloads.make_inputs(wl)
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload="fp8")
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(64)]
    prof = MoeProf()
    for i, e in enumerate(evs):
        e.record()  # materialise the handle
        prof.events[i] = e.cuda_event
    prof.n = 0
    ep.layout.prof = ctypes.pointer(prof)
    ep.forward(to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"]))
    torch.cuda.synchronize()
    names = [KERNEL_NAMES[prof.kernel[i]] for i in range(prof.n)]
    assert names == ["route_count", "route_scan", "layout_maps", "quant_dispatch_fused", "expert", "combine_fused"]
    for i in range(prof.n):
        assert evs[2 * i].elapsed_time(evs[2 * i + 1]) >= 0.0
    out0 = ep.out.clone()
    # cold timing: the library reads a flush buffer before each bracketed launch; same
    # brackets, one extra launch per kernel, same results
    flush = torch.ones(1 << 22, dtype=torch.float32, device="cuda")
    prof.n = 0
    prof.flush, prof.flush_bytes = flush.data_ptr(), flush.numel() * 4
    ep.out.zero_()
    n0 = lib().moe_launch_count()
    ep.forward(to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"]))
    torch.cuda.synchronize()
    assert [KERNEL_NAMES[prof.kernel[i]] for i in range(prof.n)] == names
    assert lib().moe_launch_count() - n0 == 2 * len(names)
    assert torch.equal(ep.out, out0)
    assert bool((flush == 1.0).all()), "the flush read must leave its buffer as it was"
    for i in range(prof.n):
        assert evs[2 * i].elapsed_time(evs[2 * i + 1]) >= 0.0


@pytest.mark.parametrize("wl", CASES + [workloads.config(4).replace(T=24, H=1024, seed=140)], ids=lambda w: w.name)
def test_partial_combine_matches_oracle(orc, wl):
    """Expert-side partial sums (one row per token and destination rank) and the source-side
    sum, bit for bit against the oracle."""
    inp = workloads.make_inputs(wl)
    ep, res = run_gpu(wl, inp)
    ep.cpart = torch.full((wl.N, wl.T, min(wl.R, wl.N), wl.H), -1.0, dtype=torch.bfloat16, device="cuda")
    poison = u16(ep.cpart[:1, :1, :1].cpu())[0, 0, 0, 0]
    ep.combine_partial(to_dev(inp["w"]))
    code, _ = ep.status()
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    cpart_o, out_o = orc.combine_partial(wl.N, wl.T, wl.E, wl.R, wl.cap, wl.H, o["ey"], inp["w"], inp["idx"],
                                         o["layout"], fill=poison)
    np.testing.assert_array_equal(u16(ep.cpart.cpu()), cpart_o)
    np.testing.assert_array_equal(u16(ep.out.cpu()), out_o)


@pytest.mark.parametrize("nb", [0, 3, 7], ids=lambda b: f"batches{b}")
@pytest.mark.parametrize("wl", CASES + [workloads.config(1).replace(T=16, seed=150)], ids=lambda w: w.name)
def test_split_dispatch_matches_oracle(orc, wl, nb):
    """Split-phase dispatch (push, per-(batch, source) arrival counters, bounded waits,
    shuffle in one cooperative launch over token batches: automatic, 3 and 7) leaves exactly
    the receive and grouped rows of the two-step path."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=8, split=True, batches=nb)
    compare_all(orc, wl, inp, res, push=True)


@pytest.mark.parametrize("nb", [1, 5], ids=lambda b: f"batches{b}")
def test_split_dispatch_withheld_source_times_out_and_recovers(orc, nb):
    """A source whose arrival signals never come: the waits for its rows end after the bound
    with the timeout status, every other row is still placed, and the next call on the same
    layout (counters reset by the call itself) is exact again."""
    wl = W("split-timeout", 4, 33, 1024, 16, 4, "bf16", "uniform", 151)
    inp = workloads.make_inputs(wl)
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    lay_o = o["layout"]
    s = 1
    ep, res = run_gpu(wl, inp, flags=8, split=True, withhold_source=s, batches=nb)
    assert res["status_code"] == 6                      # MOE_ERR_TIMEOUT
    recv = u8(res["recv"])
    for dd in range(wl.N):
        n = lay_o["rtot"][dd]
        np.testing.assert_array_equal(recv[dd, :n], o["recv"][dd, :n], err_msg="recv")
    # grouped rows: those from source s are unwritten, every other one is exact
    ex = u16(res["expert_x"])
    slot_src = lay_o["slot_src"].reshape(wl.E, -1)
    TR = wl.T * wl.R
    for e in range(wl.E):
        dd, l = divmod(e, wl.L)
        for j in range(min(lay_o["ecnt"][dd, l], lay_o["cap"])):
            src = slot_src[e, j] // TR
            if src == s:
                assert (ex[dd, l, j].view(np.uint8) == 0xA5).all(), "withheld row was written"
            else:
                np.testing.assert_array_equal(ex[dd, l, j], o["ex"][dd, l, j])
    # the context is still usable and the counters start from zero again
    ep.expert_x.view(torch.uint8).fill_(0xA5)
    ep.dispatch_split(ep.x)
    code, bits = ep.status()
    assert code == 0 and bits == 0
    ex = u16(ep.expert_x.cpu())
    ecnt = np.minimum(lay_o["ecnt"], lay_o["cap"])
    for dd in range(wl.N):
        for l in range(wl.L):
            np.testing.assert_array_equal(ex[dd, l, :ecnt[dd, l]], o["ex"][dd, l, :ecnt[dd, l]])


def test_split_dispatch_rejects_bad_withhold_source():
    import ctypes
    from combine_routing_count_gb300 import MoeEP, lib
    ep = MoeEP(2, 4, 128, 4, 2)
    x = torch.zeros((2, 4, 128), dtype=torch.bfloat16, device="cuda")
    n0 = lib().moe_launch_count()
    for bad in (-2, 2):
        rc = lib().moe_dispatch_split(ctypes.byref(ep.dims), ctypes.byref(ep.layout), x.data_ptr(),
                                      ep.recv.data_ptr(), ep.expert_x.data_ptr(), None, bad, None)
        assert rc == 1
    assert lib().moe_launch_count() == n0


def _quant_boundary_rows(H: int) -> np.ndarray:
    """bf16 rows whose 128-blocks put x / scale on the e4m3 rounding boundaries: exact ties at
    the normal-range midpoints and at the subnormal-range odd multiples of 2^-10 (scales 1.5
    and 1.25, exact in fp32, so the quotients are exact), their e4m3 neighbours, zeros of
    both signs, subnormal scales, and a wide log-normal spread of magnitudes."""
    rng = np.random.default_rng(77)
    mids = [(1 + (2 * j + 1) / 16) * 2.0 ** e for e in range(-6, 9) for j in range(8)]
    mids += [(2 * k + 1) * 2.0 ** -10 for k in range(8)]                       # subnormal-range ties
    vals = mids + [(1 + j / 8) * 2.0 ** e for e in range(-6, 9) for j in range(8)] + [m * 2.0 ** -9 for m in range(8)]
    rows = []
    for scale in (1.5, 1.25):
        cand = np.array([s * v * scale for v in vals for s in (1.0, -1.0)], np.float32)
        cand = cand[np.abs(cand) <= 448 * scale]
        exact = workloads.from_bf16_bits(workloads.to_bf16_bits(cand)) == cand
        cand = cand[exact]
        nblk = -(-len(cand) // 127)
        blocks = np.zeros((nblk, 128), np.float32)
        flat = np.concatenate([cand, np.zeros(nblk * 127 - len(cand), np.float32)])
        blocks[:, 1:] = flat.reshape(nblk, 127)
        blocks[:, 0] = 448 * scale                                              # amax -> this scale
        rows.append(blocks.reshape(-1))
    z = np.zeros(128, np.float32)
    z[::2] = -0.0
    rows.append(z)                                                              # amax 0 -> scale 1
    tiny = (rng.standard_normal(128 * 4) * 1e-37).astype(np.float32)            # subnormal scales
    rows.append(tiny)
    spread = rng.standard_normal(128 * 2048) * np.exp(rng.normal(0, 12, size=(2048, 1))).repeat(128, 1).reshape(-1)
    rows.append(np.clip(spread, -3e38, 3e38).astype(np.float32))
    flat = np.concatenate(rows)
    flat = np.concatenate([flat, np.zeros(-len(flat) % H, np.float32)])
    return workloads.to_bf16_bits(flat).reshape(1, -1, H)


def test_quantize_fp8_rounding_boundaries(orc):
    from combine_routing_count_gb300 import MoeEP
    H = 1024
    xb = _quant_boundary_rows(H)
    T = xb.shape[1]
    ep = MoeEP(1, T, H, 2, 1, payload="fp8")
    ep.quantize(to_dev(xb).view(torch.bfloat16))
    code, _ = ep.status()
    assert code == 0
    np.testing.assert_array_equal(u8(ep.xq.cpu()), orc.quantize_fp8(xb))


FP8_CASES = [c for c in CASES if c.payload == "fp8"] + [
    W("fp8-H1152-R12", 5, 17, 1152, 20, 12, "fp8", "zipf", 160),           # 9 blocks: a ragged warp unit
    W("fp8-skew", 4, 40, 2048, 32, 8, "fp8", "skew0", 161),
]


@pytest.mark.parametrize("flags", [0, 8], ids=["scatter", "push"])
@pytest.mark.parametrize("wl", FP8_CASES, ids=lambda w: w.name)
def test_fused_quantize_dispatch_matches_oracle(orc, wl, flags):
    """Quantisation inside the pack: send, receive and grouped rows (codes and scales) are
    those of the staged path, bit for bit."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags, fused_quant=True)
    compare_all(orc, wl, inp, res, push=bool(flags & 8), fused_quant=True)


def test_fused_quantize_rejects_bf16_payload():
    import ctypes
    from combine_routing_count_gb300 import MoeEP, lib
    ep = MoeEP(2, 4, 128, 4, 2)
    x = torch.zeros((2, 4, 128), dtype=torch.bfloat16, device="cuda")
    rc = lib().moe_quantize_dispatch_send(ctypes.byref(ep.dims), ctypes.byref(ep.layout), x.data_ptr(),
                                          ep.send.data_ptr(), ep.recv.data_ptr(), None)
    assert rc == 1


@pytest.mark.parametrize("payload", ["bf16", "fp8"])
def test_forward_variants_agree(orc, payload):
    """moe_forward by default, with staged fp8 quantisation, and pushed: the same output and
    layout, twice in a row on the same layout workspace."""
    wl = W("forward-variants", 8, 24, 7168, 64, 8, payload, "uniform", 162)
    inp = workloads.make_inputs(wl)
    from combine_routing_count_gb300 import MoeEP
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    for flags in (0, 0x10, 0x18, 0x8):
        ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload=payload, flags=flags)
        for _ in range(2):
            ep.out.fill_(0)
            ep.forward(to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"]))
            code, _ = ep.status()
            assert code == 0
            np.testing.assert_array_equal(u16(ep.out.cpu()), o["out"], err_msg=f"flags {flags:#x}")
            got = {k: v.cpu().numpy() for k, v in ep.layout_arrays().items()}
            for k in ("pos", "rrow", "slot", "slot_src", "recv_src", "soff", "roff", "eoff"):
                np.testing.assert_array_equal(got[k], o["layout"][k], err_msg=f"flags {flags:#x} {k}")


@pytest.mark.parametrize("batches", [1, 3])
@pytest.mark.parametrize("flags", [0, 4, 8], ids=["auto", "tma", "push"])
@pytest.mark.parametrize("payload", ["bf16", "fp8"])
def test_forward_replays_under_cuda_graph(orc, flags, payload, batches):
    """The whole pass captures into a CUDA graph (no synchronisation or allocation on the
    path; programmatic dependent launches become graph edges; micro-batches on the library's
    second stream fork from and join back into the captured stream) and replays on new
    inputs written into the captured tensors."""
    from combine_routing_count_gb300 import MoeEP
    wl = W("graph", 4, 64, 2048, 32, 8, payload, "uniform", 170)
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload=payload, alias_buffers=(payload == "bf16"), flags=flags,
               batches=batches)
    inp = workloads.make_inputs(wl)
    x, idx, w = to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ep.forward(x, idx, w)          # first launches set kernel attributes outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ep.forward(x, idx, w)
    for seed in (171, 172):
        inp = workloads.make_inputs(wl.replace(seed=seed))
        x.copy_(to_dev(inp["x"]).view(torch.bfloat16))
        idx.copy_(to_dev(inp["idx"]))
        w.copy_(to_dev(inp["w"]))
        graph.replay()
        code, _ = ep.status()
        assert code == 0
        o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, 0, payload, inp["x"], inp["idx"], inp["w"])
        np.testing.assert_array_equal(u16(ep.out.cpu()), o["out"], err_msg=f"seed {seed}")


MB_CASES = [
    W("mb-bf16", 8, 40, 2048, 64, 8, "bf16", "uniform", 230),
    W("mb-fp8", 4, 33, 1024, 32, 6, "fp8", "zipf", 231),
    W("mb-skew-cap", 4, 24, 1024, 16, 4, "bf16", "skew0", 232, cap=7),   # capacity drops
    W("mb-fp8-H384", 3, 17, 384, 6, 3, "fp8", "uniform", 233),          # 396-byte fp8 rows
    W("mb-H136", 2, 21, 136, 8, 3, "bf16", "zipf", 234),                # 272-byte rows
]


@pytest.mark.parametrize("batches", [2, 3, 7])
@pytest.mark.parametrize("flags", [0, 1, 4, 8], ids=["auto", "ldg", "tma", "push"])
@pytest.mark.parametrize("wl", MB_CASES, ids=lambda w: w.name)
def test_forward_micro_batches_match_oracle(orc, wl, flags, batches):
    """moe_forward in micro-batches (token ranges of every rank; odd ones on the library's
    second stream): every buffer bit for bit as the oracle's, unused rows untouched, with
    each mover, direct push, capacity drops and rows that are not 16-byte multiples."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags, forward=True, batches=batches)
    assert res["status_code"] == (3 if wl.cap else 0)
    compare_all(orc, wl, inp, res, push=bool(flags & 8), fused_quant=True)


@pytest.mark.parametrize("batches", [1, 2, 3, 7])
@pytest.mark.parametrize("flags", [0, 1, 4, 8], ids=["auto", "ldg", "tma", "push"])
@pytest.mark.parametrize("wl", MB_CASES, ids=lambda w: w.name)
def test_dispatch_and_combine_phases_match_oracle(orc, wl, flags, batches):
    """moe_dispatch and moe_combine (whole phases, in token batches on two streams when asked)
    around the identity expert: every buffer bit for bit as the oracle's."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags, phases=True, batches=batches)
    assert res["status_code"] == (3 if wl.cap else 0)
    compare_all(orc, wl, inp, res, push=bool(flags & 8), fused_quant=True)


@pytest.mark.parametrize("flags", [0, 1, 4, 0x80, 0x81, 0x84], ids=["fused-auto", "fused-ldg", "fused-tma",
                                                                   "separate-auto", "separate-ldg", "separate-tma"])
@pytest.mark.parametrize("wl", CASES + MB_CASES, ids=lambda w: w.name)
def test_fused_and_separate_moves_match_oracle(orc, wl, flags):
    """moe_forward in one batch with one kernel per phase (pack, write and shuffle; combine
    pack, write and sum) and with the phases' kernels apart (MOE_FLAG_SEPARATE_MOVES): in
    both, every buffer, the send, receive and combine-send rows included, bit for bit as the
    oracle's, unused rows untouched; each mover, fp8 rows that are not 16-byte multiples,
    capacity drops."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags | 0x40, forward=True)
    assert res["status_code"] == (3 if wl.cap else 0)
    compare_all(orc, wl, inp, res, fused_quant=True)


@pytest.mark.parametrize("mode", ["forward", "phases"])
@pytest.mark.parametrize("flags", [0x80, 0x88], ids=["separate", "separate-push"])
@pytest.mark.parametrize("wl", MB_CASES, ids=lambda w: w.name)
def test_separate_kernels_in_token_batches_match_oracle(orc, wl, flags, mode):
    """MOE_FLAG_SEPARATE_MOVES in token batches (moe_forward's micro-batches and the
    moe_dispatch / moe_combine phases, 3 batches), with and without direct push: every buffer
    bit for bit as the oracle's."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags, batches=3, **{mode: True})
    assert res["status_code"] == (3 if wl.cap else 0)
    compare_all(orc, wl, inp, res, push=bool(flags & 8), fused_quant=True)


@pytest.mark.parametrize("batches", [1, 3])
@pytest.mark.parametrize("payload", ["bf16", "fp8"])
def test_forward_direct_push_without_send_buffers(orc, payload, batches):
    """Direct push never touches the send and combine-send buffers, so moe_forward accepts
    NULL for both, in one batch and in micro-batches."""
    import ctypes
    from combine_routing_count_gb300 import MoeEP, lib
    wl = W("push-null", 4, 30, 1024, 16, 4, payload, "zipf", 236)
    inp = workloads.make_inputs(wl)
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload=payload, alias_buffers=(payload == "bf16"), flags=0x8,
               batches=batches)
    x, idx, w = to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"])
    b = ep.buffers(x, idx, w)
    b.send, b.csend = None, None
    assert lib().moe_forward(ctypes.byref(ep.dims), ctypes.byref(ep.layout), ctypes.byref(b), None) == 0
    code, _ = ep.status()
    assert code == 0
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, 0, payload, inp["x"], inp["idx"], inp["w"])
    np.testing.assert_array_equal(u16(ep.out.cpu()), o["out"])


LIMIT_CASES = [
    W("E1536-max", 8, 64, 256, 1536, 8, "bf16", "uniform", 180),      # largest E: 48 KB count tables
    W("N1536-L1", 1536, 2, 128, 1536, 2, "bf16", "uniform", 181),     # 1536 ranks, one expert each
    W("R40", 4, 16, 256, 64, 40, "bf16", "uniform", 182),             # R > 32: pair data past one warp
    W("fp8-E1536-zipf", 8, 32, 1024, 1536, 8, "fp8", "zipf", 183),
]


@pytest.mark.parametrize("mode", ["forward", "phases"])
@pytest.mark.parametrize("flags", [0, 8], ids=["auto", "push"])
@pytest.mark.parametrize("wl", LIMIT_CASES + [W("fp8-R36", 4, 12, 512, 64, 36, "fp8", "uniform", 184)],
                         ids=lambda w: w.name)
def test_limits_one_kernel_phases_match_oracle(orc, wl, flags, mode):
    """The one-kernel dispatch and combine (and their direct-push instances) at the limits: the
    largest E, 1536 ranks, R > 32 (pair rows held past one warp's lanes, bf16 and fp8): every
    buffer bit for bit as the oracle's."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags, forward=(mode == "forward"), phases=(mode == "phases"))
    assert res["status_code"] == 0
    compare_all(orc, wl, inp, res, push=bool(flags & 8), fused_quant=True)


@pytest.mark.parametrize("flags", [0, 8], ids=["auto", "push"])
@pytest.mark.parametrize("wl", LIMIT_CASES, ids=lambda w: w.name)
def test_limits_match_oracle(orc, wl, flags):
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags)
    compare_all(orc, wl, inp, res, push=bool(flags & 8))


RANDOM_EXPERT_CASES = [CASES[1], CASES[2], CASES[4], CASES[8], CASES[9],
                       W("dups-bad-ids", 3, 21, 256, 12, 4, "bf16", "uniform", 190)]


@pytest.mark.parametrize("flags", [0, 1, 4, 8], ids=["auto", "ldg", "tma", "push"])
@pytest.mark.parametrize("wl", RANDOM_EXPERT_CASES, ids=lambda w: w.name)
def test_combine_with_random_expert_outputs(orc, wl, flags):
    """Experts that return their own random rows (not the identity), so every pair of a
    token brings a different row: combine rows, output, and the partial combine must
    match the oracle on the same expert outputs bit for bit."""
    from workloads import to_bf16_bits
    inp = workloads.make_inputs(wl)
    if wl.name == "dups-bad-ids":
        rng0 = np.random.default_rng(191)
        inp["idx"] = rng0.integers(0, wl.E, size=(wl.N, wl.T, wl.R)).astype(np.int32)
        inp["idx"][1, 4, 2] = -3
    ep, _ = run_gpu(wl, inp, flags=flags)
    lay_o = orc.layout(wl.N, wl.T, wl.E, wl.R, wl.cap, inp["idx"])
    cap = lay_o["cap"]
    ey = to_bf16_bits(np.random.default_rng(192).standard_normal((wl.N, wl.L, cap, wl.H)).astype(np.float32))
    ep.expert_y.copy_(to_dev(ey).view(torch.bfloat16))
    w = to_dev(inp["w"])
    ep.combine_send()
    ep.combine_recv(w)
    ep.status()
    _, crecv_o = orc.combine_send(wl.N, wl.T, wl.E, wl.R, cap, wl.H, ey, lay_o)
    out_o, _ = orc.combine_recv(wl.N, wl.T, wl.R, wl.H, crecv_o, inp["w"], lay_o)
    np.testing.assert_array_equal(u16(ep.out.cpu()), out_o, err_msg="combine output")
    crecv = u16(ep.crecv.cpu())
    for s in range(wl.N):
        rows = lay_o["pos"][s][lay_o["slot"][s] >= 0]
        np.testing.assert_array_equal(crecv[s][rows], crecv_o[s][rows], err_msg="combine rows")
    if wl.R <= 32:
        ep.combine_partial(w)
        ep.status()
        cpart_o, pout_o = orc.combine_partial(wl.N, wl.T, wl.E, wl.R, cap, wl.H, ey, inp["w"], inp["idx"], lay_o)
        np.testing.assert_array_equal(u16(ep.out.cpu()), pout_o, err_msg="partial combine output")
        ngroups = [[len({int(inp["idx"][s, t, k]) // wl.L for k in range(wl.R) if lay_o["slot"][s, t, k] >= 0})
                    for t in range(wl.T)] for s in range(wl.N)]
        cpart = u16(ep.cpart.cpu())
        for s in range(wl.N):
            for t in range(wl.T):
                g = ngroups[s][t]
                np.testing.assert_array_equal(cpart[s, t, :g], cpart_o[s, t, :g], err_msg="partial rows")


def test_concurrent_passes_on_two_streams(orc):
    """Two host threads, each with its own stream and layout, run whole passes at the same
    time (different workloads, TMA and register movers, bf16 and fp8): the library keeps
    no per-call state outside the caller's layout and buffers."""
    import threading
    from combine_routing_count_gb300 import MoeEP
    cases = [(W("conc-a", 8, 64, 4096, 64, 8, "bf16", "uniform", 210), 4),
             (W("conc-b", 4, 48, 2048, 32, 6, "fp8", "zipf", 211), 0)]
    results, errors = {}, []

    def run(wl, flags):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                inp = workloads.make_inputs(wl)
                ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload=wl.payload, flags=flags)
                x, idx, w = to_dev(inp["x"]).view(torch.bfloat16), to_dev(inp["idx"]), to_dev(inp["w"])
                outs = []
                for _ in range(6):
                    ep.forward(x, idx, w)
                    code, _ = ep.status()
                    assert code == 0
                    outs.append(u16(ep.out.cpu()))
                results[wl.name] = (inp, outs)
        except Exception as e:   # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=c) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for wl, _ in cases:
        inp, outs = results[wl.name]
        o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, 0, wl.payload, inp["x"], inp["idx"], inp["w"])
        for out in outs:
            np.testing.assert_array_equal(out, o["out"], err_msg=wl.name)


def _host_tensors(inp, wl):
    h_x = torch.from_numpy(inp["x"]).view(torch.bfloat16).pin_memory()
    h_idx = torch.from_numpy(inp["idx"]).pin_memory()
    h_w = torch.from_numpy(inp["w"]).pin_memory()
    h_out = torch.empty((wl.N, wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    return h_x, h_idx, h_w, h_out


def test_forward_host_concurrent_callers(orc):
    """Two host threads, each with its own stream, layout and pinned buffers, run host passes
    at the same time through the library's shared copy streams (pipelines of 3 and 4 batches)
    and, in a third thread, the pass on mapped host memory: every output is the oracle's."""
    import threading
    from combine_routing_count_gb300 import MoeEP
    cases = [(W("hconc-a", 8, 40, 2048, 64, 8, "bf16", "uniform", 214), 0, 3),
             (W("hconc-b", 4, 33, 2048, 32, 6, "fp8", "zipf", 215), 0, 4),
             (W("hconc-c", 4, 20, 1024, 16, 4, "bf16", "zipf", 216), 0x20, 0)]
    results, errors = {}, []

    def run(wl, flags, nb):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                inp = workloads.make_inputs(wl)
                ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload=wl.payload, alias_buffers=(wl.payload == "bf16"),
                           flags=flags, batches=nb)
                h_x, h_idx, h_w, h_out = _host_tensors(inp, wl)
                x = torch.empty_like(h_x, device="cuda")
                idx = torch.empty_like(h_idx, device="cuda")
                w = torch.empty_like(h_w, device="cuda")
                outs = []
                for _ in range(6):
                    h_out.view(torch.int16).fill_(-1)
                    ep.forward_host(h_x, h_idx, h_w, h_out, x, idx, w)
                    code, _ = ep.status()
                    assert code == 0
                    outs.append(u16(h_out).copy())
                results[wl.name] = (inp, outs)
        except Exception as e:   # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=c) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for wl, _, _ in cases:
        inp, outs = results[wl.name]
        o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, 0, wl.payload, inp["x"], inp["idx"], inp["w"])
        for out in outs:
            np.testing.assert_array_equal(out, o["out"], err_msg=wl.name)


def test_forward_host_pipeline_large_batches_one_stream(orc):
    """Batches whose combine rows exceed 40% of L2 stay on the caller's stream, with half-size
    first and last batches (8 batches of about 4096 pairs of 14 KB rows here); the output is
    still the oracle's."""
    import ctypes
    from combine_routing_count_gb300 import MoeEP, lib
    wl = W("host-large", 8, 512, 7168, 64, 8, "bf16", "uniform", 222)
    inp = workloads.make_inputs(wl)
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload="bf16", alias_buffers=True, batches=8)
    assert lib().moe_batches(ctypes.byref(ep.dims), ctypes.byref(ep.layout), 1) == 8
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    assert wl.N * wl.T * wl.R // 8 * 2 * wl.H > 0.4 * l2
    h_x, h_idx, h_w, h_out = _host_tensors(inp, wl)
    x = torch.empty_like(h_x, device="cuda")
    idx = torch.empty_like(h_idx, device="cuda")
    w = torch.empty_like(h_w, device="cuda")
    h_out.view(torch.int16).fill_(-1)
    ep.forward_host(h_x, h_idx, h_w, h_out, x, idx, w)
    code, _ = ep.status()
    assert code == 0
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, 0, "bf16", inp["x"], inp["idx"], inp["w"])
    np.testing.assert_array_equal(u16(h_out), o["out"])


@pytest.mark.parametrize("payload", ["bf16", "fp8"])
def test_forward_host_pipeline_replays_under_cuda_graph(orc, payload):
    """The copy-engine pipeline (its two library streams fork from and join back into the
    caller's stream) captures into a CUDA graph and replays on new host inputs written into
    the captured pinned tensors."""
    from combine_routing_count_gb300 import MoeEP
    wl = W("hgraph", 4, 24, 2048, 16, 4, payload, "uniform", 217)
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, payload=payload, alias_buffers=(payload == "bf16"), batches=3)
    inp = workloads.make_inputs(wl)
    h_x, h_idx, h_w, h_out = _host_tensors(inp, wl)
    x = torch.empty_like(h_x, device="cuda")
    idx = torch.empty_like(h_idx, device="cuda")
    w = torch.empty_like(h_w, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ep.forward_host(h_x, h_idx, h_w, h_out, x, idx, w)   # streams, events, attributes set up here
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ep.forward_host(h_x, h_idx, h_w, h_out, x, idx, w)
    for seed in (218, 219):
        inp = workloads.make_inputs(wl.replace(seed=seed))
        h_x.copy_(torch.from_numpy(inp["x"]).view(torch.bfloat16))
        h_idx.copy_(torch.from_numpy(inp["idx"]))
        h_w.copy_(torch.from_numpy(inp["w"]))
        h_out.view(torch.int16).fill_(-1)
        graph.replay()
        code, _ = ep.status()
        assert code == 0
        o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, 0, payload, inp["x"], inp["idx"], inp["w"])
        np.testing.assert_array_equal(u16(h_out), o["out"], err_msg=f"seed {seed}")


def _run_dedicated(orc, wl, inp, K, withhold=-1):
    from combine_routing_count_gb300 import MoeEP
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload)
    for t in (ep.recv, ep.expert_x):
        t.view(torch.uint8).fill_(0xA5)
    if ep.expert_scale is not None:
        ep.expert_scale.view(torch.uint8).fill_(0xA5)
    x = to_dev(inp["x"]).view(torch.bfloat16)
    idx = to_dev(inp["idx"])
    ep.layout_step(idx)
    if wl.payload == "fp8":
        ep.quantize(x)
        x = ep.xq
    ep.dispatch_dedicated(x, idx, K, withhold)
    code, _ = ep.status()
    return ep, code


def _check_dedicated(orc, wl, inp, ep, K, skip_slice=None):
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    lay = o["layout"]
    C, roff = lay["C"], lay["roff"]
    ded, main = u8(ep.ded.cpu()), u8(ep.recv.cpu())
    for d in range(wl.N):
        moff = 0
        for s in range(wl.N):
            c = int(C[s, d])
            rows = o["recv"][d, roff[d, s]:roff[d, s] + c]
            if skip_slice != d * wl.N + s:
                nd = min(c, K)
                np.testing.assert_array_equal(ded[d, s, :nd], rows[:nd], err_msg=f"dedicated ({d},{s})")
                np.testing.assert_array_equal(main[d, moff:moff + c - nd], rows[nd:], err_msg=f"shared ({d},{s})")
            moff += max(c - K, 0)
    ecnt = np.minimum(lay["ecnt"], lay["cap"])
    slot_src = lay["slot_src"]
    TR = wl.T * wl.R
    if wl.payload == "fp8":
        ex, ex_o = u8(ep.expert_x.cpu()), o["exq"]
        exs, exs_o = u8(ep.expert_scale.cpu()), o["exs"].view(np.uint8).reshape(o["exs"].shape[:3] + (-1,))
    else:
        ex, ex_o = u16(ep.expert_x.cpu()), o["ex"]
    for d in range(wl.N):
        for l in range(wl.L):
            for j in range(ecnt[d, l]):
                src = slot_src[d, l, j] // TR
                if skip_slice == d * wl.N + src:
                    continue
                np.testing.assert_array_equal(ex[d, l, j], ex_o[d, l, j], err_msg=f"grouped ({d},{l},{j})")
                if wl.payload == "fp8":
                    np.testing.assert_array_equal(exs[d, l, j], exs_o[d, l, j])


DEDICATED_CASES = [CASES[1], CASES[3], CASES[4], CASES[5], CASES[8], W("dups-ded", 3, 21, 256, 12, 4, "bf16", "uniform", 220)]


@pytest.mark.parametrize("K", [0, 3, 16])
@pytest.mark.parametrize("wl", DEDICATED_CASES, ids=lambda w: w.name)
def test_dedicated_dispatch_matches_oracle(orc, wl, K):
    """Split-phase dispatch with K dedicated rows per (receiver, sender) and piggybacked
    counts: dedicated and shared regions hold the slices' rows where the layout puts them,
    and the grouped rows are the oracle's."""
    inp = workloads.make_inputs(wl)
    if wl.name == "dups-ded":
        rng = np.random.default_rng(221)
        inp["idx"] = rng.integers(0, wl.E, size=(wl.N, wl.T, wl.R)).astype(np.int32)
        inp["idx"][2, 3, 0] = -1
    ep, code = _run_dedicated(orc, wl, inp, K)
    assert code in (0, 2, 3)   # ok, or the data errors of the case (bad id, capacity)
    _check_dedicated(orc, wl, inp, ep, K)


def test_dedicated_dispatch_withheld_slice_times_out_and_recovers(orc):
    wl = W("ded-timeout", 4, 33, 1024, 16, 4, "bf16", "uniform", 222)
    inp = workloads.make_inputs(wl)
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    s, d = 2, 1
    assert o["layout"]["C"][s, d] > 0
    ep, code = _run_dedicated(orc, wl, inp, 5, withhold=d * wl.N + s)
    assert code == 6                                   # MOE_ERR_TIMEOUT
    _check_dedicated(orc, wl, inp, ep, 5, skip_slice=d * wl.N + s)
    ep.expert_x.view(torch.uint8).fill_(0xA5)
    ep.dispatch_dedicated(ep.x, to_dev(inp["idx"]), 5)
    code, _ = ep.status()
    assert code == 0
    _check_dedicated(orc, wl, inp, ep, 5)


def _fuzz_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        fp8 = rng.random() < 0.35
        N = int(rng.integers(1, 9))
        L = int(rng.integers(1, 13))
        E = N * L
        R = int(rng.integers(1, min(E, 12) + 1))
        T = int(rng.integers(0, 40))
        H = int(rng.choice([128, 256, 384, 1024, 1152])) if fp8 else int(8 * rng.integers(1, 160))
        routing = str(rng.choice(["uniform", "zipf"] + (["skew0"] if R <= L else [])))
        cap = int(rng.integers(1, N * T + 1)) if (T and rng.random() < 0.3) else 0
        flags = int(rng.choice([0, 1, 4, 2, 8, 9, 12]))
        out.append((W(f"fuzz{i}", N, T, H, E, R, "fp8" if fp8 else "bf16", routing, 300 + i, cap=cap), flags))
    return out


@pytest.mark.parametrize("wl,flags", _fuzz_cases(120, 31), ids=lambda v: v.name if hasattr(v, "name") else f"f{v}")
def test_fuzz_shapes_and_flags(orc, wl, flags):
    """Seeded random shapes (ranks, tokens incl. none, hidden sizes incl. rows that are not
    16-byte multiples, experts, R, capacity, routing) and launch options (movers, no PDL,
    direct push): every buffer bit for bit against the oracle."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags)
    compare_all(orc, wl, inp, res, push=bool(flags & 8))


def _fuzz_batch_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for wl, flags in _fuzz_cases(n, seed):
        mode = str(rng.choice(["forward", "phases"]))
        batches = int(rng.choice([2, 3, 5, 7]))
        out.append((wl.replace(name=wl.name.replace("fuzz", f"fuzzb-{mode}{batches}-")), flags, mode, batches))
    return out


@pytest.mark.parametrize("wl,flags,mode,batches", _fuzz_batch_cases(80, 37),
                         ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_fuzz_token_batches(orc, wl, flags, mode, batches):
    """The fuzz shapes and launch options again, with the pass split into 2-7 token batches
    (moe_forward's micro-batches or the moe_dispatch / moe_combine phases, fp8 quantised in
    the pack): every buffer bit for bit against the oracle."""
    inp = workloads.make_inputs(wl)
    _, res = run_gpu(wl, inp, flags=flags, batches=batches, **{mode: True})
    compare_all(orc, wl, inp, res, push=bool(flags & 8), fused_quant=True)


def _fuzz_host_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for wl, flags in _fuzz_cases(n, seed):
        if wl.T == 0:
            continue
        nb = int(rng.choice([0, 2, 3, 6]))
        out.append((wl.replace(name=wl.name.replace("fuzz", f"fuzzh{nb}-")), flags & ~0x2, nb))
    return out


@pytest.mark.parametrize("wl,flags,nb", _fuzz_host_cases(40, 41),
                         ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_fuzz_host_pipeline(orc, wl, flags, nb):
    """Random shapes through moe_forward_host's copy-engine pipeline (automatic, 2, 3 or 6
    token batches; each mover, direct push): the host output bit for bit the oracle's."""
    from combine_routing_count_gb300 import MoeEP
    inp = workloads.make_inputs(wl)
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, payload=wl.payload, alias_buffers=(wl.payload == "bf16"),
               flags=flags, batches=nb)
    h_x, h_idx, h_w, h_out = _host_tensors(inp, wl)
    x = torch.empty_like(h_x, device="cuda")
    idx = torch.empty_like(h_idx, device="cuda")
    w = torch.empty_like(h_w, device="cuda")
    h_out.view(torch.int16).fill_(-1)
    ep.forward_host(h_x, h_idx, h_w, h_out, x, idx, w)
    code, bits = ep.status()
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    assert bits == o["layout"]["status"], (code, bits, o["layout"]["status"])
    np.testing.assert_array_equal(u16(h_out), o["out"])
