"""Helpers for the GPU parity tests: run the CUDA path step by step through the C ABI and
compare every buffer with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import workloads

POISON = 0xA5


def to_dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def run_gpu(wl: workloads.Workload, inp: dict, flags: int = 0, poison: bool = True, split: bool = False,
            withhold_source: int = -1, fused_quant: bool = False, forward: bool = False, phases: bool = False,
            **kw):
    """Runs every step separately on the GPU; returns (MoeEP, host copies of every buffer).
    With split, dispatch is the one-launch split-phase dispatch (direct push) instead of
    dispatch send + receive; withhold_source is passed to it. With fused_quant (fp8), the
    quantisation runs inside the pack (the quantised token rows are not kept). With forward,
    the whole pass is one moe_forward call (micro-batched as the layout's settings say); with
    phases, moe_dispatch, the identity expert and moe_combine (fp8 quantised in the pack)."""
    from combine_routing_count_gb300 import MoeEP
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, flags=flags, separate_expert_y=True, **kw)
    if poison:
        for t in (ep.send, ep.recv, ep.expert_x, ep.csend, ep.crecv):
            t.view(torch.uint8).fill_(POISON)
        if ep.expert_scale is not None:
            ep.expert_scale.view(torch.uint8).fill_(POISON)
    x = to_dev(inp["x"]).view(torch.bfloat16) if "x" in inp else None
    idx = to_dev(inp["idx"])
    w = to_dev(inp["w"])
    res = {}
    if forward:
        ep.forward(x, idx, w)
    elif phases:
        ep.layout_step(idx)
        ep.dispatch(x)
        ep.expert_identity()
        ep.combine(w)
    else:
        ep.layout_step(idx)
        if fused_quant:
            ep.quantize_dispatch_send(x)
            ep.dispatch_recv()
        else:
            if wl.payload == "fp8":
                ep.quantize(x)
                x = ep.xq
            if split:
                ep.dispatch_split(x, withhold_source)
            else:
                ep.dispatch_send(x)
                ep.dispatch_recv()
        ep.expert_identity()
        ep.combine_send()
        ep.combine_recv(w)
    code, bits = ep.status()
    torch.cuda.synchronize()
    res["status_code"], res["status_bits"] = code, bits
    res["layout"] = {k: v.cpu().numpy() for k, v in ep.layout_arrays().items()}
    for k in ("xq", "send", "recv", "expert_x", "expert_scale", "expert_y", "csend", "crecv", "out"):
        t = getattr(ep, k)
        res[k] = None if t is None else t.cpu()
    return ep, res


def u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy()


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def compare_all(orc, wl, inp, res, check_poison=True, push=False, fused_quant=False):
    """Bit-exact comparison of every buffer's used rows with the oracle; padding untouched.
    With push (direct-push mode) the send and combine-send buffers must stay untouched."""
    N, T, H, E, R, L = wl.N, wl.T, wl.H, wl.E, wl.R, wl.L
    o = orc.forward(N, T, H, E, R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    lay_o = o["layout"]
    for k in ("cnt", "C", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow", "slot", "slot_src", "recv_src"):
        np.testing.assert_array_equal(res["layout"][k], lay_o[k], err_msg=f"layout {k}")
    bits_o = lay_o["status"]
    assert res["status_bits"] == bits_o, (res["status_bits"], bits_o)
    cap, RB = lay_o["cap"], lay_o["RB"]
    pos, slot = lay_o["pos"], lay_o["slot"]
    valid = pos >= 0
    kept = slot >= 0
    if wl.payload == "fp8" and not fused_quant:
        np.testing.assert_array_equal(u8(res["xq"]), o["xq"], err_msg="fp8 quantised rows")
    # send rows of every valid pair
    send = u8(res["send"])
    if push:
        assert (send == POISON).all(), "direct push wrote the send buffer"
    for s in ([] if push else range(N)):
        rows = pos[s][valid[s]]
        np.testing.assert_array_equal(send[s][rows], o["send"][s][rows], err_msg="send")
        if check_poison:
            assert (send[s][valid[s].sum():] == POISON).all(), "stray send write"
    recv = u8(res["recv"])
    for d in range(N):
        n = lay_o["rtot"][d]
        np.testing.assert_array_equal(recv[d, :n], o["recv"][d, :n], err_msg="recv")
        if check_poison:
            assert (recv[d, n:] == POISON).all(), "stray recv write"
    ecnt = np.minimum(lay_o["ecnt"], cap)
    if wl.payload == "fp8":
        ex, exs = u8(res["expert_x"]), u8(res["expert_scale"])
        exs_o = o["exs"].view(np.uint8).reshape(exs.shape)
        for d in range(N):
            for l in range(L):
                n = ecnt[d, l]
                np.testing.assert_array_equal(ex[d, l, :n], o["exq"][d, l, :n], err_msg="expert codes")
                np.testing.assert_array_equal(exs[d, l, :n], exs_o[d, l, :n], err_msg="expert scales")
                if check_poison:
                    assert (ex[d, l, n:] == POISON).all() and (exs[d, l, n:] == POISON).all()
        ey = u16(res["expert_y"])
        for d in range(N):
            for l in range(L):
                n = ecnt[d, l]
                np.testing.assert_array_equal(ey[d, l, :n], o["ey"][d, l, :n], err_msg="dequantised expert rows")
    else:
        ex = u16(res["expert_x"])
        for d in range(N):
            for l in range(L):
                n = ecnt[d, l]
                np.testing.assert_array_equal(ex[d, l, :n], o["ex"][d, l, :n], err_msg="expert rows")
                if check_poison:
                    assert (ex[d, l, n:].view(np.uint8) == POISON).all(), "stray expert write"
        ey = u16(res["expert_y"])
        for d in range(N):
            for l in range(L):
                n = ecnt[d, l]
                np.testing.assert_array_equal(ey[d, l, :n], o["ex"][d, l, :n], err_msg="identity expert copy")
    csend = u16(res["csend"])
    crecv = u16(res["crecv"])
    if push:
        assert (csend.view(np.uint8) == POISON).all(), "direct push wrote the combine send buffer"
    for d in ([] if push else range(N)):
        rows = lay_o["rrow"][kept & (np.asarray(inp["idx"]) // L == d)] if L > 0 else []
        np.testing.assert_array_equal(csend[d][rows], o["csend"][d][rows], err_msg="combine send rows")
    for s in range(N):
        rows = pos[s][kept[s]]
        np.testing.assert_array_equal(crecv[s][rows], o["crecv"][s][rows], err_msg="combine recv rows")
    out = u16(res["out"])
    # bit-exact with the oracle's fp32 path (same order, separate rounding) ...
    np.testing.assert_array_equal(out, o["out"], err_msg="combine output (fp32 path)")
    # ... and within the stated tolerance of the fp64 sum
    xmax = float(np.abs(workloads.from_bf16_bits(inp["x"])).max()) if inp["x"].size else 0.0
    outf = workloads.from_bf16_bits(out).astype(np.float64)
    if out.size:
        assert np.abs(outf - o["out64"]).max() <= 2.0 ** -7 * xmax
    return o
