"""Seeded synthetic inputs for MoE expert-parallel dispatch/combine.

This module only draws inputs: token activations, top-R expert ids and
router weights. It holds none of the dispatch/combine arithmetic, so both the
CUDA path and the CPU oracle can take their inputs from here without sharing
any code of the method.

Shapes follow the evaluation of "Enabling trillion-parameter models on AWS
EFA" (Perplexity), section "Evaluation": hidden size 7168, R = 8 experts per
token, block-scaled fp8 dispatch and bf16 combine, DeepSeek-V3 / Kimi-K2 sized
expert counts. The pages use live model traffic; these seeded draws stand in
for it:

* x      bf16, each element an fp32 draw from N(0,1) rounded to nearest-even;
* idx    int32 [N,T,R], R distinct experts per token, one of
           "uniform": a uniformly random ordered R-subset of the E experts,
           "zipf":    sequential sampling without replacement with expert
                      popularity p ∝ (i+1)^-s over a seeded permutation of
                      the experts (Gumbel top-R, which equals that sequential
                      sampling exactly),
           "skew0":   every token routed only to experts of rank 0 (a seeded
                      random order of R of rank 0's E/N experts per token);
* w      fp32 [N,T,R], a softmax over R N(0,1) logits, computed in fp32.

All draws come from numpy's counter-based Philox generator keyed by `seed`,
in a fixed order (routing, then logits, then x).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

__all__ = ["Workload", "CONFIGS", "config", "make_inputs", "to_bf16_bits", "from_bf16_bits"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic dispatch/combine problem (all N simulated ranks)."""

    name: str
    N: int          # simulated expert-parallel ranks
    T: int          # tokens per rank
    H: int          # hidden size
    E: int          # experts in total, E % N == 0
    R: int          # experts per token
    payload: str    # "bf16" or "fp8" (e4m3 + fp32 scale per 128 elements)
    routing: str    # "uniform", "zipf" or "skew0"
    seed: int
    zipf_s: float = 1.2
    cap: int = 0    # per-expert slots; 0 means N*T

    @property
    def L(self) -> int:
        return self.E // self.N

    @property
    def cap_eff(self) -> int:
        return self.cap if self.cap > 0 else self.N * self.T

    @property
    def RB(self) -> int:
        """Receive rows per rank, N*T*max(R, E/N) (section "Send and receive buffers")."""
        return self.N * self.T * max(self.R, self.L)

    @property
    def row_bytes(self) -> int:
        if self.payload == "fp8":
            return self.H + 4 * (self.H // 128)
        return 2 * self.H

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny parity case, then DeepSeek-V3 / Kimi-K2 shaped cases
# (decode batch 128 and 32 tokens per rank, EP8 / EP32 / EP64) and a worst-case skew
# that fills rank 0's receive buffer to its N*T*max(R,E/N) bound.
CONFIGS = {
    0: Workload("tiny-N2-T16-H128-E8-R2", 2, 16, 128, 8, 2, "bf16", "uniform", 0),
    1: Workload("ep8-T128-H7168-E256-R8-bf16", 8, 128, 7168, 256, 8, "bf16", "uniform", 1),
    2: Workload("ep32-T128-H7168-E384-R8-bf16-zipf1.2", 32, 128, 7168, 384, 8, "bf16", "zipf", 2),
    3: Workload("ep64-T32-H7168-E384-R8-fp8", 64, 32, 7168, 384, 8, "fp8", "uniform", 3),
    4: Workload("ep16-T512-H4096-E128-R8-skew-rank0", 16, 512, 4096, 128, 8, "bf16", "skew0", 4),
}


def config(i: int) -> Workload:
    return CONFIGS[int(i)]


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even, by torch) returned as uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _routing(rng: np.random.Generator, wl: Workload) -> np.ndarray:
    N, T, E, R, L = wl.N, wl.T, wl.E, wl.R, wl.L
    ntok = N * T
    if wl.routing == "uniform":
        if R > E:
            raise ValueError("uniform distinct routing needs R <= E")
        keys = rng.random((ntok, E))
        idx = np.argsort(keys, axis=1, kind="stable")[:, :R]
    elif wl.routing == "zipf":
        if R > E:
            raise ValueError("zipf distinct routing needs R <= E")
        perm = rng.permutation(E)
        logp = np.empty(E)
        logp[perm] = -wl.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        u = rng.random((ntok, E))
        gumbel = -np.log(-np.log(np.clip(u, 1e-300, 1.0)))
        idx = np.argsort(-(logp[None, :] + gumbel), axis=1, kind="stable")[:, :R]
    elif wl.routing == "skew0":
        if R > L:
            raise ValueError("skew0 routing needs R <= E/N")
        keys = rng.random((ntok, L))
        idx = np.argsort(keys, axis=1, kind="stable")[:, :R]
    else:
        raise ValueError(f"unknown routing {wl.routing!r}")
    return idx.astype(np.int32).reshape(N, T, R)


def _softmax_f32(logits: np.ndarray) -> np.ndarray:
    m = logits.max(axis=-1, keepdims=True)
    e = np.exp(logits - m, dtype=np.float32)
    return (e / e.sum(axis=-1, keepdims=True, dtype=np.float32)).astype(np.float32)


def make_inputs(wl: Workload, with_x: bool = True) -> dict:
    """Draw one problem: {"x": uint16 [N,T,H] bf16 bits, "idx": int32 [N,T,R], "w": fp32 [N,T,R]}."""
    rng = np.random.Generator(np.random.Philox(wl.seed))
    idx = _routing(rng, wl)
    logits = rng.standard_normal((wl.N, wl.T, wl.R), dtype=np.float32)
    w = _softmax_f32(logits)
    out = {"idx": np.ascontiguousarray(idx), "w": np.ascontiguousarray(w)}
    if with_x:
        x = rng.standard_normal((wl.N, wl.T, wl.H), dtype=np.float32)
        out["x"] = np.ascontiguousarray(to_bf16_bits(x))
    return out
