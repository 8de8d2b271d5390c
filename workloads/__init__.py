"""Seeded synthetic inputs for jagged GDPA.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark.  It holds only the recipe for drawing inputs (lengths, offsets,
tensors, bias tables, upstream gradients) and none of the attention
arithmetic, so that the oracle and the CUDA path stay independent of each
other.

The five named workloads follow the shapes given for the method on the pages
("GEM Training: How Meta Doubled the Efficiency of Its ...", section "What to
watch": self-attention, PMA and cross-attention share one GDPA kernel;
"Meta redesigns AI training infrastructure ...", section "Eliminating Compute
Waste in Asymmetric Workloads": a production jagged sparsity of 0.5).  No
dataset is named there, so these distributions stand in for production traffic.
A sixth workload runs the long-tail batch under a sliding window of 1024
(the same page, section "Custom Kernels and 5D Parallelism ...": sliding
window attention for long sequences).

Draw order for one workload, from ``numpy.random.default_rng(seed)``:
query lengths, key/value lengths, Q, K, V (float32 standard normal), the bias
table (0.1 * standard normal, float32 [H, 257]) when the workload has one,
and finally dO (float32 standard normal).  Q, K, V and dO are then rounded to
bfloat16 (round to nearest even).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

ACTS = ("gelu", "silu", "softmax")
ACT_CODE = {"gelu": 0, "silu": 1, "softmax": 2}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    head_dim: int
    act: str
    causal: bool
    bias_len: int          # 0: no bias table
    seed: int
    lq: tuple              # ("uniform", lo, hi) inclusive, ("fixed", n), ("same",), ("lognormal", mu, sigma, lo, hi)
    lkv: tuple
    shared_q: int = 0      # >0: that many seed queries per head, shared by every segment (PMA)
    window: int = 0        # >0: sliding window, pairs with |i - j| < window


WORKLOADS = {
    1: Workload("tiny jagged GDPA", 4, 2, 32, "silu", False, 0, 0,
                ("uniform", 1, 64), ("uniform", 1, 48)),
    2: Workload("JFA causal self-attention", 256, 4, 128, "softmax", True, 0, 1,
                ("uniform", 1, 1024), ("same",)),
    3: Workload("GDPA short-K/V cross-attention", 1024, 4, 128, "gelu", False, 257, 2,
                ("uniform", 1, 2048), ("uniform", 32, 128)),
    4: Workload("PMA-style pooling", 512, 8, 64, "silu", False, 0, 3,
                ("fixed", 16), ("uniform", 1, 4096), shared_q=16),
    5: Workload("long-tail jagged GDPA", 64, 8, 128, "gelu", False, 257, 4,
                ("lognormal", math.log(1500.0), 1.0, 100, 16384), ("same",)),
    # the long-tail batch (same seed, same draws) under a sliding window
    6: Workload("long-tail jagged GDPA, sliding window 1024", 64, 8, 128, "gelu", False, 257, 4,
                ("lognormal", math.log(1500.0), 1.0, 100, 16384), ("same",), window=1024),
}


def _draw_lengths(rng: np.random.Generator, spec: tuple, n: int) -> np.ndarray:
    kind = spec[0]
    if kind == "uniform":
        return rng.integers(spec[1], spec[2] + 1, size=n).astype(np.int64)
    if kind == "fixed":
        return np.full(n, spec[1], dtype=np.int64)
    if kind == "lognormal":
        x = rng.lognormal(spec[1], spec[2], size=n)
        return np.clip(np.round(x), spec[3], spec[4]).astype(np.int64)
    raise ValueError(f"unknown length spec {spec}")


def offsets_from_lengths(lengths) -> torch.Tensor:
    """Exclusive prefix sum of segment lengths as int32 [B+1] (offsets[0] = 0)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lengths)
    if off[-1] > np.iinfo(np.int32).max:
        raise ValueError("total length exceeds int32 offsets")
    return torch.from_numpy(off.astype(np.int32))


def lengths_for(w: Workload, rng: Optional[np.random.Generator] = None):
    """The realized (Lq, Lkv) arrays of a workload, drawn first from its seed."""
    rng = rng if rng is not None else np.random.default_rng(w.seed)
    lq = _draw_lengths(rng, w.lq, w.batch)
    lkv = lq.copy() if w.lkv[0] == "same" else _draw_lengths(rng, w.lkv, w.batch)
    return lq, lkv


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


@dataclasses.dataclass
class Inputs:
    """One batch of jagged GDPA inputs on the CPU (move with ``.to(device)``)."""
    q: torch.Tensor            # bf16 [total_q, H, d]
    k: torch.Tensor            # bf16 [total_kv, H, d]
    v: torch.Tensor            # bf16 [total_kv, H, d]
    dout: torch.Tensor         # bf16 [total_q, H, d]
    q_offsets: torch.Tensor    # int32 [B+1]
    kv_offsets: torch.Tensor   # int32 [B+1]
    bias: Optional[torch.Tensor]  # float32 [H, bias_len] or None
    lq: np.ndarray
    lkv: np.ndarray
    heads: int
    head_dim: int
    act: str
    causal: bool
    scale: float               # float32 value 1/sqrt(d)
    q_seed: Optional[torch.Tensor] = None  # PMA: the shared bf16 [n_seed, H, d] queries
    window: int = 0            # >0: only pairs with |i - j| < window (segment-local)

    @property
    def batch(self) -> int:
        return len(self.lq)

    @property
    def bias_len(self) -> int:
        return 0 if self.bias is None else int(self.bias.shape[1])

    def to(self, device) -> "Inputs":
        def mv(t):
            return None if t is None else t.to(device)
        return dataclasses.replace(
            self, q=mv(self.q), k=mv(self.k), v=mv(self.v), dout=mv(self.dout),
            q_offsets=mv(self.q_offsets), kv_offsets=mv(self.kv_offsets),
            bias=mv(self.bias), q_seed=mv(self.q_seed))


def make_inputs(lq, lkv, heads: int, head_dim: int, act: str, causal: bool = False,
                bias_len: int = 0, seed: int = 0, rng: Optional[np.random.Generator] = None,
                shared_q: int = 0, window: int = 0) -> Inputs:
    """Draw Q, K, V, bias and dO for given segment lengths (draw order in the module doc)."""
    if act not in ACTS:
        raise ValueError(f"act must be one of {ACTS}")
    rng = rng if rng is not None else np.random.default_rng(seed)
    lq = np.asarray(lq, dtype=np.int64)
    lkv = np.asarray(lkv, dtype=np.int64)
    tq, tkv = int(lq.sum()), int(lkv.sum())
    h, d = heads, head_dim
    q_seed = None
    if shared_q:
        if not np.all(lq == shared_q):
            raise ValueError("shared queries need every Lq equal to the seed count")
        q_seed = _bf16(rng.standard_normal((shared_q, h, d), dtype=np.float32))
        q = q_seed.repeat(len(lq), 1, 1).contiguous()
    else:
        q = _bf16(rng.standard_normal((tq, h, d), dtype=np.float32))
    k = _bf16(rng.standard_normal((tkv, h, d), dtype=np.float32))
    v = _bf16(rng.standard_normal((tkv, h, d), dtype=np.float32))
    bias = None
    if bias_len:
        bias = torch.from_numpy(
            (0.1 * rng.standard_normal((h, bias_len), dtype=np.float32)).astype(np.float32))
    dout = _bf16(rng.standard_normal((tq, h, d), dtype=np.float32))
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    return Inputs(q=q, k=k, v=v, dout=dout, q_offsets=offsets_from_lengths(lq),
                  kv_offsets=offsets_from_lengths(lkv), bias=bias, lq=lq, lkv=lkv,
                  heads=h, head_dim=d, act=act, causal=causal, scale=scale, q_seed=q_seed,
                  window=int(window))


def select_segments(x: Inputs, segs) -> Inputs:
    """A compact Inputs holding only the listed segments (in the given order),
    with their rows copied and the offsets rebuilt; used to run the oracle on a
    sample of a large batch."""
    segs = [int(b) for b in segs]
    qo, ko = x.q_offsets.numpy(), x.kv_offsets.numpy()
    qi = np.concatenate([np.arange(qo[b], qo[b + 1]) for b in segs]) if segs else np.zeros(0, np.int64)
    ki = np.concatenate([np.arange(ko[b], ko[b + 1]) for b in segs]) if segs else np.zeros(0, np.int64)
    qi = torch.from_numpy(qi.astype(np.int64))
    ki = torch.from_numpy(ki.astype(np.int64))
    lq, lkv = x.lq[segs], x.lkv[segs]
    return dataclasses.replace(
        x, q=x.q[qi].contiguous(), k=x.k[ki].contiguous(), v=x.v[ki].contiguous(),
        dout=x.dout[qi].contiguous(), q_offsets=offsets_from_lengths(lq),
        kv_offsets=offsets_from_lengths(lkv), lq=lq, lkv=lkv)


def workload_inputs(index: int) -> Inputs:
    """The full-size inputs of workload ``index`` (1..6)."""
    w = WORKLOADS[index]
    rng = np.random.default_rng(w.seed)
    lq, lkv = lengths_for(w, rng)
    return make_inputs(lq, lkv, w.heads, w.head_dim, w.act, w.causal, w.bias_len,
                       rng=rng, shared_q=w.shared_q, window=w.window)


def random_case(seed: int, batch: int, heads: int, head_dim: int, act: str,
                lq_range=(1, 20), lkv_range=(1, 20), causal: bool = False,
                bias_len: int = 0, allow_empty: bool = False, window: int = 0) -> Inputs:
    """A small random jagged case; with ``allow_empty`` lengths may be 0."""
    rng = np.random.default_rng(seed)
    lo_q = 0 if allow_empty else lq_range[0]
    lo_k = 0 if allow_empty else lkv_range[0]
    lq = rng.integers(lo_q, lq_range[1] + 1, size=batch)
    lkv = rng.integers(lo_k, lkv_range[1] + 1, size=batch)
    return make_inputs(lq, lkv, heads, head_dim, act, causal, bias_len, rng=rng, window=window)
