"""GB300-native MoE expert-parallel dispatch and combine.

The path of "Enabling trillion-parameter models on AWS EFA" (Perplexity): routing-count
histogram and scans, collision-free contiguous placement, pack, per-peer write, receive
shuffle into per-expert grouped rows, and the combine back with a weighted sum per token.
All N simulated ranks live in one GPU's HBM. Every step runs in hand-written sm_103a CUDA
kernels of libmoe_ep.so behind the C ABI in include/moe_ep.h; this package only marshals
arguments and uses PyTorch for device memory and streams. There is no CPU fallback.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import (MOE_FLAG_DIRECT_PUSH, MOE_FLAG_ONE_BATCH, MOE_FLAG_HOST_MAPPED, MOE_FLAG_LDG_MOVER,
                   MOE_FLAG_NO_PDL, MOE_FLAG_SEPARATE_MOVES, MOE_FLAG_STAGED_QUANT,
                   MOE_FLAG_TMA_MOVER, MOE_PAYLOAD_BF16, MOE_PAYLOAD_FP8_E4M3_B128, KERNEL_NAMES, MoeBuffers,
                   MoeDims, MoeError, MoeLayout, MoeProf, check, lib)

__all__ = ["MoeEP", "MoeDims", "MoeLayout", "MoeBuffers", "MoeProf", "MoeError", "lib", "check",
           "MOE_FLAG_LDG_MOVER", "MOE_FLAG_NO_PDL", "MOE_FLAG_TMA_MOVER", "MOE_FLAG_DIRECT_PUSH",
           "MOE_FLAG_STAGED_QUANT", "MOE_FLAG_HOST_MAPPED", "MOE_FLAG_ONE_BATCH", "MOE_FLAG_SEPARATE_MOVES",
           "KERNEL_NAMES"]


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class MoeEP:
    """One expert-parallel group of N simulated ranks on the current CUDA device.

    Owns the layout workspace and every dispatch/combine buffer (torch allocations). Shapes
    (B = row bytes, RB = N*T*max(R,E/N) receive rows per rank, L = E/N):
      send [N, T*R, B] u8, recv [N, RB, B] u8,
      expert_x [N, L, cap, H] bf16 (bf16 payload) or u8 e4m3 codes + expert_scale [N, L, cap, H/128] f32,
      expert_y [N, L, cap, H] bf16 (aliases expert_x for bf16 unless separate_expert_y),
      csend [N, RB, H] bf16, crecv [N, T*R, H] bf16, out [N, T, H] bf16.
    With alias_buffers=True (bf16 only) csend reuses recv and crecv reuses send, the buffer
    reuse between dispatch and combine of the page's section "Dispatch and combine".
    """

    def __init__(self, N, T, H, E, R, cap=0, payload="bf16", *, alias_buffers=False, separate_expert_y=False,
                 flags=0, tma_stages=0, ctas_per_sm=0, batches=0):
        L_ = lib()
        self.payload = payload
        self.fp8 = payload == "fp8"
        self.dims = MoeDims(N, T, H, E, R, cap, MOE_PAYLOAD_FP8_E4M3_B128 if self.fp8 else MOE_PAYLOAD_BF16)
        check(L_.moe_check_dims(ctypes.byref(self.dims)), "moe_check_dims")
        self.N, self.T, self.H, self.E, self.R, self.L = N, T, H, E, R, E // N
        self.cap = L_.moe_capacity(ctypes.byref(self.dims))
        self.RB = L_.moe_recv_capacity_rows(ctypes.byref(self.dims))
        self.B = L_.moe_row_bytes(ctypes.byref(self.dims))
        dev = torch.device("cuda", torch.cuda.current_device())
        u8, bf16 = torch.uint8, torch.bfloat16
        ws_bytes = L_.moe_layout_workspace_bytes(ctypes.byref(self.dims))
        self.workspace = torch.empty(ws_bytes, dtype=u8, device=dev)
        self.layout = MoeLayout()
        check(L_.moe_layout_init(ctypes.byref(self.dims), self.workspace.data_ptr(), ws_bytes,
                                 ctypes.byref(self.layout), _stream()), "moe_layout_init")
        self.layout.flags = flags
        self.layout.tma_stages = tma_stages
        self.layout.ctas_per_sm = ctas_per_sm
        self.layout.batches = batches
        L = self.L
        self.xq = torch.empty((N, T, self.B), dtype=u8, device=dev) if self.fp8 else None
        self.send = torch.empty((N, T * R, self.B), dtype=u8, device=dev)
        self.recv = torch.empty((N, self.RB, self.B), dtype=u8, device=dev)
        if self.fp8:
            self.expert_x = torch.empty((N, L, self.cap, H), dtype=u8, device=dev)
            self.expert_scale = torch.empty((N, L, self.cap, H // 128), dtype=torch.float32, device=dev)
            self.expert_y = torch.empty((N, L, self.cap, H), dtype=bf16, device=dev)
        else:
            self.expert_x = torch.empty((N, L, self.cap, H), dtype=bf16, device=dev)
            self.expert_scale = None
            self.expert_y = (torch.empty_like(self.expert_x) if separate_expert_y else self.expert_x)
        if alias_buffers and not self.fp8:
            self.csend = self.recv.view(bf16).view(N, self.RB, H)
            self.crecv = self.send.view(bf16).view(N, T * R, H)
        else:
            self.csend = torch.empty((N, self.RB, H), dtype=bf16, device=dev)
            self.crecv = torch.empty((N, T * R, H), dtype=bf16, device=dev)
        self.out = torch.empty((N, T, H), dtype=bf16, device=dev)
        self.x = None
        self.idx = None
        self.w = None

    # ------------------------------------------------------------------ steps
    def layout_step(self, idx: torch.Tensor, stream=None):
        self.idx = idx
        check(lib().moe_layout(ctypes.byref(self.dims), idx.data_ptr(), ctypes.byref(self.layout),
                               _stream(stream)), "moe_layout")

    def quantize(self, x: torch.Tensor, stream=None):
        check(lib().moe_quantize_fp8_b128(ctypes.byref(self.dims), x.data_ptr(), self.xq.data_ptr(),
                                          ctypes.byref(self.layout), _stream(stream)), "moe_quantize_fp8_b128")

    def dispatch_send(self, x: torch.Tensor, stream=None):
        """x: [N,T,H] bf16 (bf16 payload) or [N,T,B] u8 rows from quantize (fp8)."""
        self.x = x
        check(lib().moe_dispatch_send(ctypes.byref(self.dims), ctypes.byref(self.layout), x.data_ptr(),
                                      self.send.data_ptr(), self.recv.data_ptr(), _stream(stream)),
              "moe_dispatch_send")

    def quantize_dispatch_send(self, x: torch.Tensor, stream=None):
        """fp8 payload: quantise the bf16 token rows x [N,T,H] inside the pack (xq is not written)."""
        self.x = x
        check(lib().moe_quantize_dispatch_send(ctypes.byref(self.dims), ctypes.byref(self.layout), x.data_ptr(),
                                               self.send.data_ptr(), self.recv.data_ptr(), _stream(stream)),
              "moe_quantize_dispatch_send")

    def dispatch(self, x: torch.Tensor, stream=None):
        """Whole dispatch phase (send + recv; fp8: the bf16 token rows x are quantised inside
        the pack), in token batches when moe_batches(..., 2) says so."""
        self.x = x
        check(lib().moe_dispatch(ctypes.byref(self.dims), ctypes.byref(self.layout), x.data_ptr(),
                                 self.send.data_ptr(), self.recv.data_ptr(), self.expert_x.data_ptr(),
                                 _ptr(self.expert_scale), _stream(stream)), "moe_dispatch")

    def combine(self, w: torch.Tensor, stream=None) -> torch.Tensor:
        """Whole combine phase (send + recv) from self.expert_y into self.out."""
        self.w = w
        check(lib().moe_combine(ctypes.byref(self.dims), ctypes.byref(self.layout), self.expert_y.data_ptr(),
                                self.csend.data_ptr(), self.crecv.data_ptr(), w.data_ptr(), self.out.data_ptr(),
                                _stream(stream)), "moe_combine")
        return self.out

    def dispatch_split(self, x: torch.Tensor, withhold_source: int = -1, stream=None):
        """Split-phase dispatch: receive rows and grouped expert rows in one launch.
        withhold_source (tests only) names a source rank whose arrival signals are not sent."""
        self.x = x
        check(lib().moe_dispatch_split(ctypes.byref(self.dims), ctypes.byref(self.layout), x.data_ptr(),
                                       self.recv.data_ptr(), self.expert_x.data_ptr(), _ptr(self.expert_scale),
                                       int(withhold_source), _stream(stream)), "moe_dispatch_split")

    def dispatch_dedicated(self, x: torch.Tensor, idx: torch.Tensor, K: int, withhold_slice: int = -1, stream=None):
        """Split-phase dispatch with K dedicated rows per (receiver, sender) and the routing
        counts piggybacked on the first writes. The shared region is self.recv; the
        dedicated rows are self.ded [N,N,K,B]. withhold_slice (tests only) names a slice
        d*N + s whose row signals are not sent."""
        self.x = x
        if getattr(self, "ded", None) is None or self.ded.shape[2] != K:
            self.ded = torch.empty((self.N, self.N, max(K, 1), self.B), dtype=torch.uint8, device=self.recv.device)
            nbytes = lib().moe_dedicated_exchange_bytes(ctypes.byref(self.dims))
            self.xchg = torch.empty(nbytes, dtype=torch.uint8, device=self.recv.device)
        check(lib().moe_dispatch_dedicated(ctypes.byref(self.dims), ctypes.byref(self.layout), idx.data_ptr(),
                                           x.data_ptr(), int(K), self.ded.data_ptr(), self.xchg.data_ptr(),
                                           self.recv.data_ptr(), self.expert_x.data_ptr(), _ptr(self.expert_scale),
                                           int(withhold_slice), _stream(stream)), "moe_dispatch_dedicated")

    def dispatch_recv(self, stream=None):
        check(lib().moe_dispatch_recv(ctypes.byref(self.dims), ctypes.byref(self.layout), self.recv.data_ptr(),
                                      self.expert_x.data_ptr(), _ptr(self.expert_scale), _stream(stream)),
              "moe_dispatch_recv")

    def expert_identity(self, stream=None):
        check(lib().moe_expert_identity(ctypes.byref(self.dims), ctypes.byref(self.layout),
                                        self.expert_x.data_ptr(), _ptr(self.expert_scale),
                                        self.expert_y.data_ptr(), _stream(stream)), "moe_expert_identity")

    def combine_send(self, stream=None):
        check(lib().moe_combine_send(ctypes.byref(self.dims), ctypes.byref(self.layout), self.expert_y.data_ptr(),
                                     self.csend.data_ptr(), self.crecv.data_ptr(), _stream(stream)),
              "moe_combine_send")

    def combine_recv(self, w: torch.Tensor, stream=None):
        self.w = w
        check(lib().moe_combine_recv(ctypes.byref(self.dims), ctypes.byref(self.layout), self.crecv.data_ptr(),
                                     w.data_ptr(), self.out.data_ptr(), _stream(stream)), "moe_combine_recv")

    def combine_partial(self, w: torch.Tensor, stream=None) -> torch.Tensor:
        """Combine with expert-side partial sums (one row per token and destination rank):
        moe_combine_send_partial into self.cpart, then moe_combine_recv_partial into self.out."""
        if getattr(self, "cpart", None) is None:
            J = min(self.R, self.N)
            self.cpart = torch.empty((self.N, self.T, J, self.H), dtype=torch.bfloat16, device=self.out.device)
        self.w = w
        check(lib().moe_combine_send_partial(ctypes.byref(self.dims), ctypes.byref(self.layout),
                                             self.expert_y.data_ptr(), w.data_ptr(), self.cpart.data_ptr(),
                                             _stream(stream)), "moe_combine_send_partial")
        check(lib().moe_combine_recv_partial(ctypes.byref(self.dims), ctypes.byref(self.layout),
                                             self.cpart.data_ptr(), self.out.data_ptr(), _stream(stream)),
              "moe_combine_recv_partial")
        return self.out

    def buffers(self, x, idx, w) -> MoeBuffers:
        b = MoeBuffers()
        b.x, b.xq, b.idx, b.w = _ptr(x), _ptr(self.xq), _ptr(idx), _ptr(w)
        b.send, b.recv = self.send.data_ptr(), self.recv.data_ptr()
        b.expert_x, b.expert_scale, b.expert_y = self.expert_x.data_ptr(), _ptr(self.expert_scale), \
            self.expert_y.data_ptr()
        b.csend, b.crecv, b.out = self.csend.data_ptr(), self.crecv.data_ptr(), self.out.data_ptr()
        return b

    def forward(self, x, idx, w, stream=None) -> torch.Tensor:
        """The whole pass on device tensors (one C call): returns self.out."""
        self.x, self.idx, self.w = x, idx, w
        self._bufs = self.buffers(x, idx, w)
        check(lib().moe_forward(ctypes.byref(self.dims), ctypes.byref(self.layout), ctypes.byref(self._bufs),
                                _stream(stream)), "moe_forward")
        return self.out

    def forward_host(self, h_x, h_idx, h_w, h_out, x, idx, w, stream=None):
        """The whole pass from host tensors (pinned) into h_out; x/idx/w are the device staging tensors
        (copy-engine pipeline by default; with MOE_FLAG_HOST_MAPPED the kernels use the pinned
        tensors directly)."""
        self._bufs = self.buffers(x, idx, w)
        check(lib().moe_forward_host(ctypes.byref(self.dims), ctypes.byref(self.layout), ctypes.byref(self._bufs),
                                     h_x.data_ptr(), h_idx.data_ptr(), h_w.data_ptr(), h_out.data_ptr(),
                                     _stream(stream)), "moe_forward_host")

    def status(self, stream=None) -> tuple[int, int]:
        """Synchronises, returns (first error code, all status bits) and clears the status word."""
        bits = ctypes.c_uint32(0)
        code = lib().moe_status_sync(ctypes.byref(self.layout), _stream(stream), ctypes.byref(bits))
        return int(code), int(bits.value)

    # ------------------------------------------------------------------ inspection
    def layout_arrays(self) -> dict:
        """Torch views of the layout arrays inside the workspace (device, int32)."""
        base = self.workspace.data_ptr()
        N, T, E, R, L, cap, RB = self.N, self.T, self.E, self.R, self.L, self.cap, self.RB
        shapes = {"cnt": (N, E), "C": (N, N), "soff": (N, E), "roff": (N, N), "rtot": (N,), "ecnt": (N, L),
                  "eoff": (N, L, N), "pos": (N, T, R), "rrow": (N, T, R), "slot": (N, T, R),
                  "slot_src": (N, L, cap), "recv_src": (N, RB), "gsend": (N, T, R), "grecv": (N, T, R),
                  "gslot": (N, T, R)}
        out = {}
        for k, shp in shapes.items():
            off = getattr(self.layout, k) - base
            n = 1
            for d in shp:
                n *= d
            out[k] = self.workspace[off:off + 4 * n].view(torch.int32).view(shp)
        return out
