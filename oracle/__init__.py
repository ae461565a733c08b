"""CPU oracle for MoE expert-parallel dispatch/combine (numpy front end of moe_oracle.c).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline
leg may import this package. The CUDA library never calls it and shares no code with it.

Every function follows "Enabling trillion-parameter models on AWS EFA" (Perplexity),
sections "Send and receive buffers" (전송 및 수신 버퍼), "Dispatch and combine"
(디스패치 및 결합) and "Evaluation" (평가); the readings taken where the page is silent
are listed at the top of moe_oracle.c. Pins: tests/test_oracle_*.py check every
function against brute force, invariants, closed forms and the OCP FP8 definition.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from ctypes import POINTER, c_double, c_float, c_int, c_int64, c_uint8, c_uint16, c_uint32

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

BIT_EXPERT_RANGE = 1 << 2
BIT_CAPACITY = 1 << 3
BIT_RECV_BOUND = 1 << 4


def compile_source(src: str, out: str) -> str:
    """gcc the C source file src into the shared library out (no FMA contraction, no
    fast-math)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile moe_oracle.c."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


_lib = None


def _P(t):
    return POINTER(t)


@contextlib.contextmanager
def library(path: str):
    """Runs every function of this module on another build of moe_oracle.c (the tests that
    plant a mistake in a copy of the oracle, to show that its pins catch it)."""
    global _lib
    saved = _lib
    _lib = _load(path)
    try:
        yield
    finally:
        _lib = saved


def lib():
    global _lib
    if _lib is None:
        _lib = _load(build())
    return _lib


def _load(path: str):
    L = ctypes.CDLL(path)
    i32p = _P(ctypes.c_int32)
    L.orc_bf16_to_f32.argtypes = [c_uint16]
    L.orc_bf16_to_f32.restype = c_float
    L.orc_f32_to_bf16.argtypes = [c_float]
    L.orc_f32_to_bf16.restype = c_uint16
    L.orc_e4m3_decode.argtypes = [c_uint8]
    L.orc_e4m3_decode.restype = c_double
    L.orc_e4m3_encode.argtypes = [c_float]
    L.orc_e4m3_encode.restype = c_uint8
    L.orc_layout.argtypes = [c_int] * 5 + [i32p] * 13
    L.orc_layout.restype = c_uint32
    L.orc_quantize_fp8.argtypes = [c_int, c_int, c_int, _P(c_uint16), _P(c_uint8)]
    L.orc_quantize_fp8.restype = None
    L.orc_dispatch_send.argtypes = [c_int] * 4 + [c_int64, _P(c_uint8)] + [i32p] * 4 + [_P(c_uint8)] * 2
    L.orc_dispatch_send.restype = None
    L.orc_dispatch_recv.argtypes = [c_int] * 5 + [c_int64, c_int, _P(c_uint8)] + [i32p] * 4 + [_P(c_uint8), _P(c_float)]
    L.orc_dispatch_recv.restype = None
    L.orc_expert_dequant.argtypes = [c_int] * 4 + [i32p, _P(c_uint8), _P(c_float), _P(c_uint16)]
    L.orc_expert_dequant.restype = None
    L.orc_combine_send.argtypes = [c_int] * 6 + [_P(c_uint16)] + [i32p] * 5 + [_P(c_uint16)] * 2
    L.orc_combine_send.restype = None
    L.orc_combine_recv.argtypes = [c_int] * 4 + [_P(c_uint16), _P(c_float), i32p, i32p, _P(c_uint16), _P(c_double)]
    L.orc_combine_recv.restype = None
    L.orc_combine_partial_send.argtypes = [c_int] * 6 + [_P(c_uint16), _P(c_float), i32p, i32p, _P(c_uint16)]
    L.orc_combine_partial_send.restype = None
    L.orc_combine_partial_recv.argtypes = [c_int] * 4 + [i32p, i32p, c_int, _P(c_uint16), _P(c_uint16)]
    L.orc_combine_partial_recv.restype = None
    return L


def _ptr(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(POINTER(t))


def _i32(a):
    return _ptr(a, ctypes.c_int32)


# ------------------------------------------------------------------ scalar formats

def bf16_to_f32(b: int) -> float:
    return lib().orc_bf16_to_f32(int(b))


def f32_to_bf16(f: float) -> int:
    return int(lib().orc_f32_to_bf16(float(f)))


def e4m3_decode(c: int) -> float:
    return float(lib().orc_e4m3_decode(int(c)))


def e4m3_encode(f: float) -> int:
    return int(lib().orc_e4m3_encode(float(f)))


# ------------------------------------------------------------------ the path

def recv_rows(N, T, E, R) -> int:
    """N*T*max(R, E/N): rows a rank can receive ("Send and receive buffers")."""
    return N * T * max(R, E // N)


def layout(N: int, T: int, E: int, R: int, cap: int, idx: np.ndarray) -> dict:
    """Counts, scans and per-pair placements; returns a dict of int32 arrays + 'status'."""
    L = E // N
    cap = cap if cap > 0 else N * T
    RB = recv_rows(N, T, E, R)
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(N, T, R)
    o = {
        "cnt": np.zeros((N, E), np.int32), "C": np.zeros((N, N), np.int32),
        "soff": np.zeros((N, E), np.int32), "roff": np.zeros((N, N), np.int32),
        "rtot": np.zeros((N,), np.int32), "ecnt": np.zeros((N, L), np.int32),
        "eoff": np.zeros((N, L, N), np.int32), "pos": np.zeros((N, T, R), np.int32),
        "rrow": np.zeros((N, T, R), np.int32), "slot": np.zeros((N, T, R), np.int32),
        "slot_src": np.zeros((N, L, cap), np.int32), "recv_src": np.zeros((N, RB), np.int32),
    }
    st = lib().orc_layout(N, T, E, R, cap, _i32(idx), *[_i32(o[k]) for k in
                          ("cnt", "C", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow",
                           "slot", "slot_src", "recv_src")])
    o["status"] = int(st)
    o["cap"] = cap
    o["RB"] = RB
    return o


def quantize_fp8(x: np.ndarray) -> np.ndarray:
    """x uint16 bf16 bits [..., H] -> uint8 rows [..., H + 4*(H/128)] (codes then fp32 scales)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    H = x.shape[-1]
    assert H % 128 == 0
    rows = int(np.prod(x.shape[:-1]))
    B = H + 4 * (H // 128)
    out = np.zeros(x.shape[:-1] + (B,), np.uint8)
    lib().orc_quantize_fp8(rows, 1, H, _ptr(x, c_uint16), _ptr(out, c_uint8))
    return out


def dispatch_send(N, T, E, R, xrows: np.ndarray, lay: dict, recv_fill: int = 0):
    """xrows uint8 [N,T,B] -> (send uint8 [N,T*R,B], recv uint8 [N,RB,B]). Unused rows hold recv_fill."""
    xrows = np.ascontiguousarray(xrows, dtype=np.uint8)
    B = xrows.shape[-1]
    RB = recv_rows(N, T, E, R)
    send = np.full((N, T * R, B), recv_fill, np.uint8)
    recv = np.full((N, RB, B), recv_fill, np.uint8)
    lib().orc_dispatch_send(N, T, E, R, B, _ptr(xrows, c_uint8), _i32(lay["pos"]), _i32(lay["C"]),
                            _i32(lay["soff"]), _i32(lay["roff"]), _ptr(send, c_uint8), _ptr(recv, c_uint8))
    return send, recv


def dispatch_recv(N, T, E, R, cap, recv: np.ndarray, lay: dict, payload: str, H: int, fill: int = 0):
    """recv -> grouped rows. bf16: uint16 [N,L,cap,H]. fp8: (uint8 [N,L,cap,H], fp32 [N,L,cap,H/128])."""
    L = E // N
    cap = cap if cap > 0 else N * T
    recv = np.ascontiguousarray(recv, dtype=np.uint8)
    B = recv.shape[-1]
    if payload == "fp8":
        exq = np.full((N, L, cap, H), fill, np.uint8)
        exs = np.zeros((N, L, cap, H // 128), np.float32)
        lib().orc_dispatch_recv(N, T, E, R, cap, B, H, _ptr(recv, c_uint8), _i32(lay["cnt"]), _i32(lay["soff"]),
                                _i32(lay["roff"]), _i32(lay["eoff"]), _ptr(exq, c_uint8), _ptr(exs, c_float))
        return exq, exs
    ex = np.full((N, L, cap, B), fill, np.uint8)
    lib().orc_dispatch_recv(N, T, E, R, cap, B, 0, _ptr(recv, c_uint8), _i32(lay["cnt"]), _i32(lay["soff"]),
                            _i32(lay["roff"]), _i32(lay["eoff"]), _ptr(ex, c_uint8), None)
    return ex.view(np.uint16)


def expert_dequant(N, L, cap, H, exq: np.ndarray, exs: np.ndarray, lay: dict) -> np.ndarray:
    ey = np.zeros((N, L, cap, H), np.uint16)
    lib().orc_expert_dequant(N, L, cap, H, _i32(lay["ecnt"]), _ptr(np.ascontiguousarray(exq), c_uint8),
                             _ptr(np.ascontiguousarray(exs, dtype=np.float32), c_float), _ptr(ey, c_uint16))
    return ey


def combine_send(N, T, E, R, cap, H, ey: np.ndarray, lay: dict, fill: int = 0):
    """ey uint16 [N,L,cap,H] -> (csend uint16 [N,RB,H], crecv uint16 [N,T*R,H])."""
    cap = cap if cap > 0 else N * T
    RB = recv_rows(N, T, E, R)
    ey = np.ascontiguousarray(ey, dtype=np.uint16)
    csend = np.full((N, RB, H), fill, np.uint16)
    crecv = np.full((N, T * R, H), fill, np.uint16)
    lib().orc_combine_send(N, T, E, R, cap, H, _ptr(ey, c_uint16), _i32(lay["cnt"]), _i32(lay["C"]),
                           _i32(lay["soff"]), _i32(lay["roff"]), _i32(lay["eoff"]),
                           _ptr(csend, c_uint16), _ptr(crecv, c_uint16))
    return csend, crecv


def combine_recv(N, T, R, H, crecv: np.ndarray, w: np.ndarray, lay: dict):
    """-> (out uint16 bf16 [N,T,H], out64 fp64 [N,T,H])."""
    crecv = np.ascontiguousarray(crecv, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.zeros((N, T, H), np.uint16)
    out64 = np.zeros((N, T, H), np.float64)
    lib().orc_combine_recv(N, T, R, H, _ptr(crecv, c_uint16), _ptr(w, c_float), _i32(lay["pos"]),
                           _i32(lay["slot"]), _ptr(out, c_uint16), _ptr(out64, c_double))
    return out, out64


def forward(N, T, H, E, R, cap, payload, x: np.ndarray, idx: np.ndarray, w: np.ndarray) -> dict:
    """The whole path: layout -> [fp8 quantise] -> dispatch send/recv -> identity expert -> combine."""
    lay = layout(N, T, E, R, cap, idx)
    cap = lay["cap"]
    L = E // N
    res = {"layout": lay}
    if payload == "fp8":
        xrows = quantize_fp8(x)
        res["xq"] = xrows
    else:
        xrows = np.ascontiguousarray(x, dtype=np.uint16).view(np.uint8)
    send, recv = dispatch_send(N, T, E, R, xrows, lay)
    res["send"], res["recv"] = send, recv
    if payload == "fp8":
        exq, exs = dispatch_recv(N, T, E, R, cap, recv, lay, "fp8", H)
        res["exq"], res["exs"] = exq, exs
        ey = expert_dequant(N, L, cap, H, exq, exs, lay)
    else:
        ey = dispatch_recv(N, T, E, R, cap, recv, lay, "bf16", H)
        res["ex"] = ey
    res["ey"] = ey
    csend, crecv = combine_send(N, T, E, R, cap, H, ey, lay)
    res["csend"], res["crecv"] = csend, crecv
    out, out64 = combine_recv(N, T, R, H, crecv, w, lay)
    res["out"], res["out64"] = out, out64
    return res


def alloc_step(N, T, H, E, R, cap, payload) -> dict:
    """Buffers for run_step, allocated once (np.empty: pages are touched only where written)."""
    L = E // N
    cap = cap if cap > 0 else N * T
    RB = recv_rows(N, T, E, R)
    B = H + 4 * (H // 128) if payload == "fp8" else 2 * H
    b = {"dims": (N, T, H, E, R, cap, payload), "B": B}
    for k in ("cnt", "soff"):
        b[k] = np.empty((N, E), np.int32)
    b["C"], b["roff"] = np.empty((N, N), np.int32), np.empty((N, N), np.int32)
    b["rtot"], b["ecnt"], b["eoff"] = np.empty(N, np.int32), np.empty((N, L), np.int32), np.empty((N, L, N), np.int32)
    for k in ("pos", "rrow", "slot"):
        b[k] = np.empty((N, T, R), np.int32)
    b["slot_src"], b["recv_src"] = np.empty((N, L, cap), np.int32), np.empty((N, RB), np.int32)
    b["xq"] = np.empty((N, T, B), np.uint8) if payload == "fp8" else None
    b["send"], b["recv"] = np.empty((N, T * R, B), np.uint8), np.empty((N, RB, B), np.uint8)
    if payload == "fp8":
        b["exq"], b["exs"] = np.empty((N, L, cap, H), np.uint8), np.empty((N, L, cap, H // 128), np.float32)
        b["ey"] = np.empty((N, L, cap, H), np.uint16)
    else:
        b["ex"] = np.empty((N, L, cap, B), np.uint8)
    b["csend"], b["crecv"] = np.empty((N, RB, H), np.uint16), np.empty((N, T * R, H), np.uint16)
    b["out"], b["out64"] = np.empty((N, T, H), np.uint16), np.empty((N, T, H), np.float64)
    return b


def run_step(b: dict, x: np.ndarray, idx: np.ndarray, w: np.ndarray) -> int:
    """One whole pass into preallocated buffers (same arithmetic as forward()); returns the status bits."""
    N, T, H, E, R, cap, payload = b["dims"]
    L_ = lib()
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    st = L_.orc_layout(N, T, E, R, cap, _i32(idx), *[_i32(b[k]) for k in
                       ("cnt", "C", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow", "slot", "slot_src",
                        "recv_src")])
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if payload == "fp8":
        L_.orc_quantize_fp8(N, T, H, _ptr(x, c_uint16), _ptr(b["xq"], c_uint8))
        xrows = b["xq"]
    else:
        xrows = x.view(np.uint8)
    L_.orc_dispatch_send(N, T, E, R, b["B"], _ptr(xrows, c_uint8), _i32(b["pos"]), _i32(b["C"]), _i32(b["soff"]),
                         _i32(b["roff"]), _ptr(b["send"], c_uint8), _ptr(b["recv"], c_uint8))
    if payload == "fp8":
        L_.orc_dispatch_recv(N, T, E, R, cap, b["B"], H, _ptr(b["recv"], c_uint8), _i32(b["cnt"]), _i32(b["soff"]),
                             _i32(b["roff"]), _i32(b["eoff"]), _ptr(b["exq"], c_uint8), _ptr(b["exs"], c_float))
        L_.orc_expert_dequant(N, E // N, cap, H, _i32(b["ecnt"]), _ptr(b["exq"], c_uint8), _ptr(b["exs"], c_float),
                              _ptr(b["ey"], c_uint16))
        ey = b["ey"]
    else:
        L_.orc_dispatch_recv(N, T, E, R, cap, b["B"], 0, _ptr(b["recv"], c_uint8), _i32(b["cnt"]), _i32(b["soff"]),
                             _i32(b["roff"]), _i32(b["eoff"]), _ptr(b["ex"], c_uint8), None)
        ey = b["ex"]
    L_.orc_combine_send(N, T, E, R, cap, H, ey.ctypes.data_as(POINTER(c_uint16)), _i32(b["cnt"]), _i32(b["C"]),
                        _i32(b["soff"]), _i32(b["roff"]), _i32(b["eoff"]), _ptr(b["csend"], c_uint16),
                        _ptr(b["crecv"], c_uint16))
    L_.orc_combine_recv(N, T, R, H, _ptr(b["crecv"], c_uint16), _ptr(np.ascontiguousarray(w, np.float32), c_float),
                        _i32(b["pos"]), _i32(b["slot"]), _ptr(b["out"], c_uint16), _ptr(b["out64"], c_double))
    return int(st)


def combine_partial(N, T, E, R, cap, H, ey: np.ndarray, w: np.ndarray, idx: np.ndarray, lay: dict, fill: int = 0):
    """Expert-side partial sums then source-side sum -> (cpart uint16 [N,T,J,H], out uint16 [N,T,H])."""
    cap = cap if cap > 0 else N * T
    J = min(R, N)
    ey = np.ascontiguousarray(ey, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    cpart = np.full((N, T, J, H), fill, np.uint16)
    out = np.zeros((N, T, H), np.uint16)
    lib().orc_combine_partial_send(N, T, E, R, cap, H, _ptr(ey, c_uint16), _ptr(w, c_float), _i32(idx),
                                   _i32(lay["slot"]), _ptr(cpart, c_uint16))
    lib().orc_combine_partial_recv(N, T, E, R, _i32(idx), _i32(lay["slot"]), H, _ptr(cpart, c_uint16),
                                   _ptr(out, c_uint16))
    return cpart, out
