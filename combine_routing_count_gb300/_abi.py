"""ctypes mirror of include/moe_ep.h. Argument marshalling only; every step runs in libmoe_ep.so."""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_int32, c_size_t, c_uint32, c_uint64, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_ep.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_EXPERT_RANGE = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_RECV_BOUND = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6

MOE_PAYLOAD_BF16 = 0
MOE_PAYLOAD_FP8_E4M3_B128 = 1

MOE_FLAG_LDG_MOVER = 0x1
MOE_FLAG_NO_PDL = 0x2
MOE_FLAG_TMA_MOVER = 0x4
MOE_FLAG_DIRECT_PUSH = 0x8
MOE_FLAG_STAGED_QUANT = 0x10
MOE_FLAG_HOST_MAPPED = 0x20
MOE_FLAG_ONE_BATCH = 0x40
MOE_FLAG_SEPARATE_MOVES = 0x80
MOE_PROF_MAX = 32

KERNEL_NAMES = ["route_count", "layout_maps", "quant_fp8", "pack", "scatter", "unpack", "expert",
                "combine_pack", "combine_scatter", "combine_reduce", "route_scan", "pack_push", "combine_push",
                "combine_partial", "combine_sum", "dispatch_split", "quant_pack", "dispatch_dedicated",
                "dispatch_fused", "quant_dispatch_fused", "combine_fused"]

LAYOUT_FIELDS = ("cnt", "C", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow", "slot", "slot_src",
                 "recv_src", "gsend", "grecv", "gslot", "status", "scratch")


class MoeDims(ctypes.Structure):
    _fields_ = [("N", c_int32), ("T", c_int32), ("H", c_int32), ("E", c_int32), ("R", c_int32),
                ("cap", c_int32), ("payload", c_int32)]


class MoeProf(ctypes.Structure):
    _fields_ = [("events", c_void_p * (2 * MOE_PROF_MAX)), ("kernel", c_int32 * MOE_PROF_MAX), ("n", c_int32),
                ("flush", c_void_p), ("flush_bytes", ctypes.c_size_t)]


class MoeLayout(ctypes.Structure):
    _fields_ = [(f, c_void_p) for f in LAYOUT_FIELDS] + [
        ("flags", c_uint32), ("prof", POINTER(MoeProf)), ("tma_stages", c_int32), ("ctas_per_sm", c_int32),
        ("batches", c_int32), ("win_lo", c_int32), ("win_hi", c_int32)]


BUFFER_FIELDS = ("x", "xq", "idx", "w", "send", "recv", "expert_x", "expert_scale", "expert_y", "csend",
                 "crecv", "out")


class MoeBuffers(ctypes.Structure):
    _fields_ = [(f, c_void_p) for f in BUFFER_FIELDS]


class MoeSlice(ctypes.Structure):
    _fields_ = [("peer", c_int32), ("s", c_int32), ("d", c_int32), ("rows", c_int32), ("local_row", ctypes.c_int64)]


_lib = None


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


def lib():
    """Loads libmoe_ep.so. There is no fallback: a missing library is an error."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m combine_routing_count_gb300.build` "
                               "or __graft_entry__.build()")
        import torch  # noqa: F401  (load torch's libcudart first so both share one CUDA runtime)
        L = ctypes.CDLL(LIB_PATH)
        D, Lp, B = POINTER(MoeDims), POINTER(MoeLayout), POINTER(MoeBuffers)
        sig = {
            "moe_check_dims": (c_int32, [D]),
            "moe_recv_capacity_rows": (c_size_t, [D]),
            "moe_row_bytes": (c_size_t, [D]),
            "moe_capacity": (c_int32, [D]),
            "moe_layout_workspace_bytes": (c_size_t, [D]),
            "moe_layout_init": (c_int32, [D, c_void_p, c_size_t, Lp, c_void_p]),
            "moe_layout": (c_int32, [D, c_void_p, Lp, c_void_p]),
            "moe_quantize_fp8_b128": (c_int32, [D, c_void_p, c_void_p, Lp, c_void_p]),
            "moe_dispatch_send": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_dispatch_send_noalloc": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p]),
            "moe_quantize_dispatch_send": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_dedicated_exchange_bytes": (c_size_t, [D]),
            "moe_dispatch_dedicated": (c_int32, [D, Lp, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                                 c_void_p, c_void_p, c_int32, c_void_p]),
            "moe_dispatch_split": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_void_p]),
            "moe_dispatch_recv": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_expert_identity": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_combine_send": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_combine_recv": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_dispatch": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_combine": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_combine_send_partial": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_combine_recv_partial": (c_int32, [D, Lp, c_void_p, c_void_p, c_void_p]),
            "moe_forward": (c_int32, [D, Lp, B, c_void_p]),
            "moe_forward_host": (c_int32, [D, Lp, B, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
            "moe_batches": (c_int32, [D, Lp, c_int32]),
            "moe_exchange_plan": (ctypes.c_int64, [D, c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_int32,
                                                   c_int32, c_int32, POINTER(MoeSlice), ctypes.c_int64]),
            "moe_status_sync": (c_int32, [Lp, c_void_p, POINTER(c_uint32)]),
            "moe_status_string": (c_char_p, [c_int32]),
            "moe_launch_count": (c_uint64, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def check(code: int, what: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, what)


# Names a symbol-export test checks against include/moe_ep.h.
EXPORTED = ("moe_check_dims", "moe_recv_capacity_rows", "moe_row_bytes", "moe_capacity",
            "moe_layout_workspace_bytes", "moe_layout_init", "moe_layout", "moe_quantize_fp8_b128",
            "moe_dispatch_send", "moe_dispatch_send_noalloc", "moe_quantize_dispatch_send", "moe_dispatch_split",
            "moe_dedicated_exchange_bytes", "moe_dispatch_dedicated", "moe_dispatch_recv",
            "moe_expert_identity", "moe_combine_send", "moe_combine_recv", "moe_dispatch", "moe_combine",
            "moe_combine_send_partial",
            "moe_combine_recv_partial", "moe_forward", "moe_forward_host", "moe_batches", "moe_exchange_plan",
            "moe_status_sync",
            "moe_status_string", "moe_launch_count")
