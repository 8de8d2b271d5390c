"""Helpers shared by the GPU parity tests."""

from __future__ import annotations

import dataclasses
import functools

import numpy as np
import torch

import oracle
import workloads

# Per-output-tensor bar: max|gpu - ref| <= TOL * max|ref| (bf16 inputs, fp32
# accumulation, bf16 P / dS operands).
TOL = 2e-2


def rel_err(gpu, ref) -> float:
    g = gpu.detach().float().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64)
    if r.size == 0:
        return 0.0
    den = float(np.max(np.abs(r)))
    num = float(np.max(np.abs(g.astype(np.float64) - r)))
    if den == 0.0:
        return num
    return num / den


def assert_close(name, gpu, ref, tol=TOL):
    g = gpu.detach().float().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    e = rel_err(g, ref)
    assert e <= tol, f"{name}: max|err|/max|ref| = {e:.3e} > {tol}"
    return e


def unit_rows(x, units, which="q"):
    """Row indices (token index, head) of the given (segment, head) units."""
    off = (x.q_offsets if which == "q" else x.kv_offsets).numpy()
    rows, heads = [], []
    for u in units:
        b, h = divmod(int(u), x.heads)
        r = np.arange(off[b], off[b + 1])
        rows.append(r)
        heads.append(np.full(r.shape, h))
    if not rows:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.concatenate(rows), np.concatenate(heads)


def sample_units(x, n_random: int, seed: int, max_pairs=None, include_longest=True):
    """A few (segment, head) units: the longest segment (if cheap enough), the
    shortest, and random ones, each with at most max_pairs valid pairs."""
    rng = np.random.default_rng(seed)
    pairs = x.lq.astype(np.int64) * x.lkv.astype(np.int64)
    ok = np.ones(x.batch, bool) if max_pairs is None else pairs <= max_pairs
    cand = np.nonzero(ok & (x.lq > 0))[0]
    chosen = set()
    if include_longest and len(cand):
        chosen.add(int(cand[np.argmax(pairs[cand])]))
        chosen.add(int(cand[np.argmin(pairs[cand])]))
    if len(cand):
        for b in rng.choice(cand, size=min(n_random, len(cand)), replace=False):
            chosen.add(int(b))
    units = []
    for b in sorted(chosen):
        units.append(b * x.heads + int(rng.integers(0, x.heads)))
    return units


def oracle_fwd(x, units=None):
    return oracle.fwd_inputs(x, units=units)


def oracle_bwd(x, units=None):
    return oracle.bwd_inputs(x, units=units)


def sampled_oracle(x, units, backward: bool):
    """Oracle results for the (segment, head) units b*H + h of a large batch,
    computed on a compact copy holding only those segments.  Returns a list of
    (b, h, q_rows, kv_rows, results) where q_rows / kv_rows index the full
    batch and results are the oracle arrays restricted to that unit's rows."""
    import workloads
    segs = [u // x.heads for u in units]
    sub = workloads.select_segments(x, segs)
    sub_units = [i * x.heads + (u % x.heads) for i, u in enumerate(units)]
    res = oracle.bwd_inputs(sub, units=sub_units) if backward else oracle.fwd_inputs(sub, units=sub_units)
    qo, ko = x.q_offsets.numpy(), x.kv_offsets.numpy()
    sqo, sko = sub.q_offsets.numpy(), sub.kv_offsets.numpy()
    out = []
    for i, u in enumerate(units):
        b, h = divmod(u, x.heads)
        q_rows = np.arange(qo[b], qo[b + 1])
        kv_rows = np.arange(ko[b], ko[b + 1])
        sq = slice(sqo[i], sqo[i + 1])
        sk = slice(sko[i], sko[i + 1])
        if backward:
            dq, dk, dv, _ = res
            out.append((b, h, q_rows, kv_rows, (dq[sq, h], dk[sk, h], dv[sk, h])))
        else:
            o, lse = res
            out.append((b, h, q_rows, kv_rows, (o[sq, h], lse[h, sq])))
    return out


@functools.lru_cache(maxsize=2)
def _workload(idx: int):
    return workloads.workload_inputs(idx)


def full_workload(idx: int):
    """The full-size inputs of a named workload, generated once per process
    (the sliding-window workload 6 reuses the draws of workload 5)."""
    if idx == 6:
        return dataclasses.replace(_workload(5), window=workloads.WORKLOADS[6].window)
    return _workload(idx)
