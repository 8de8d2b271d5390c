"""Pins of the fp64 CPU oracle against things other than itself.

Each check is chosen so that a plausible slip in the oracle (a dropped bias
term, a wrong sign in the bias index, a transposed operand, a wrong
derivative, a missing mask) fails at least one of them:

* a padded-and-masked dense brute force written independently here (numpy +
  scipy's erf/expit, not the C library's);
* torch autograd on that dense formulation for the gradients;
* central finite differences of L = sum(O * dO) through the oracle forward;
* the identity-activation associativity (s Q K^T) V = s Q (K^T V);
* invariance under permutation of the segments;
* softmax mode against torch.softmax per segment (a library routine);
* sliding window: the dense references above with a band mask |i - j| < w,
  a window of 1 against its closed form, a window no shorter than any
  segment against the unwindowed oracle, and rows left without any key;
* closed forms (tests/golden/activation_closed_forms.json and hand-derived
  single-key / zero-query cases).
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special as sps
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "activation_closed_forms.json")


# ----------------------------------------------------------------------------
# Independent dense brute force (padded to the longest segment, then masked).
# ----------------------------------------------------------------------------

def _pad(x: np.ndarray, off: np.ndarray, lmax: int) -> np.ndarray:
    b = len(off) - 1
    out = np.zeros((b, lmax) + x.shape[1:], dtype=np.float64)
    for s in range(b):
        n = off[s + 1] - off[s]
        out[s, :n] = x[off[s]:off[s + 1]]
    return out


def _unpad(xp: np.ndarray, off: np.ndarray) -> np.ndarray:
    return np.concatenate([xp[s, : off[s + 1] - off[s]] for s in range(len(off) - 1)], axis=0)


def dense_reference(x: workloads.Inputs, act: str = None):
    """O [total_q, H, d] by a dense masked computation per padded segment."""
    act = act or x.act
    q = x.q.double().numpy()
    k = x.k.double().numpy()
    v = x.v.double().numpy()
    qo = x.q_offsets.numpy().astype(np.int64)
    ko = x.kv_offsets.numpy().astype(np.int64)
    lqm = max(1, int(x.lq.max(initial=0)))
    lkm = max(1, int(x.lkv.max(initial=0)))
    qp, kp, vp = _pad(q, qo, lqm), _pad(k, ko, lkm), _pad(v, ko, lkm)  # [B, L, H, d]
    i = np.arange(lqm)[:, None]
    j = np.arange(lkm)[None, :]
    mask = (j[None] < x.lkv[:, None, None]) & (i[None] < x.lq[:, None, None])
    if x.causal:
        mask = mask & (j <= i)[None]
    if x.window:
        mask = mask & (np.abs(i - j) < x.window)[None]
    s = np.einsum("bihc,bjhc->bhij", qp, kp) * x.scale
    if x.bias is not None:
        t = x.bias.shape[1]
        r = (t - 1) // 2
        idx = np.clip(i - j, -r, r) + r                        # [Lq, Lkv]
        s = s + x.bias.double().numpy()[:, idx][None]          # [1, H, Lq, Lkv]
    m4 = mask[:, None]
    if act == "softmax":
        sm = np.where(m4, s, -np.inf)
        mx = np.max(sm, axis=-1, keepdims=True)
        mx = np.where(np.isfinite(mx), mx, 0.0)
        e = np.where(m4, np.exp(sm - mx), 0.0)
        den = e.sum(-1, keepdims=True)
        p = np.where(den > 0, e / np.where(den > 0, den, 1.0), 0.0)
    elif act == "gelu":
        p = np.where(m4, s * 0.5 * (1.0 + sps.erf(s / math.sqrt(2.0))), 0.0)
    elif act == "silu":
        p = np.where(m4, s * sps.expit(s), 0.0)
    elif act == "identity":
        p = np.where(m4, s, 0.0)
    else:
        raise ValueError(act)
    o = np.einsum("bhij,bjhc->bihc", p, vp)
    return _unpad(o, qo)


def dense_torch_grads(x: workloads.Inputs):
    """dQ, dK, dV, dbias of L = sum(O * dO) by torch autograd on the dense form."""
    qo = x.q_offsets.numpy().astype(np.int64)
    ko = x.kv_offsets.numpy().astype(np.int64)
    lqm = max(1, int(x.lq.max(initial=0)))
    lkm = max(1, int(x.lkv.max(initial=0)))
    qp = torch.tensor(_pad(x.q.double().numpy(), qo, lqm), requires_grad=True)
    kp = torch.tensor(_pad(x.k.double().numpy(), ko, lkm), requires_grad=True)
    vp = torch.tensor(_pad(x.v.double().numpy(), ko, lkm), requires_grad=True)
    dop = torch.tensor(_pad(x.dout.double().numpy(), qo, lqm))
    i = torch.arange(lqm)[:, None]
    j = torch.arange(lkm)[None, :]
    lq = torch.tensor(x.lq)
    lkv = torch.tensor(x.lkv)
    mask = (j[None] < lkv[:, None, None]) & (i[None] < lq[:, None, None])
    if x.causal:
        mask = mask & (j <= i)[None]
    if x.window:
        mask = mask & ((i - j).abs() < x.window)[None]
    m4 = mask[:, None]
    s = torch.einsum("bihc,bjhc->bhij", qp, kp) * x.scale
    bias = None
    if x.bias is not None:
        bias = x.bias.double().clone().requires_grad_(True)
        t = bias.shape[1]
        r = (t - 1) // 2
        idx = torch.clamp(i - j, -r, r) + r
        s = s + bias[:, idx][None]
    if x.act == "softmax":
        sm = torch.where(m4, s, torch.full_like(s, -torch.inf))
        rowvalid = m4.any(-1, keepdim=True)
        sm = torch.where(rowvalid, sm, torch.zeros_like(sm))
        p = torch.softmax(sm, dim=-1)
        p = torch.where(m4, p, torch.zeros_like(p))
    elif x.act == "gelu":
        p = torch.where(m4, torch.nn.functional.gelu(s), torch.zeros_like(s))
    else:
        p = torch.where(m4, torch.nn.functional.silu(s), torch.zeros_like(s))
    o = torch.einsum("bhij,bjhc->bihc", p, vp)
    (o * dop).sum().backward()
    dq = _unpad(qp.grad.numpy(), qo)
    dk = _unpad(kp.grad.numpy(), ko)
    dv = _unpad(vp.grad.numpy(), ko)
    db = None if bias is None else bias.grad.numpy()
    return dq, dk, dv, db


def _rel(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    den = max(np.max(np.abs(b)) if b.size else 0.0, 1e-300)
    return float(np.max(np.abs(a - b)) / den) if a.size else 0.0


MODES = [(a, bl, c) for a in ("gelu", "silu", "softmax") for bl in (0, 7) for c in (False, True)]


@pytest.mark.parametrize("act,bias_len,causal", MODES)
def test_forward_matches_dense_bruteforce(act, bias_len, causal):
    for seed in range(12):
        d = (4, 8, 32)[seed % 3]
        x = workloads.random_case(100 + seed, batch=1 + seed % 6, heads=1 + seed % 3,
                                  head_dim=d, act=act, lq_range=(1, 20), lkv_range=(1, 20),
                                  causal=causal, bias_len=bias_len, allow_empty=(seed % 4 == 3))
        o, _ = oracle.fwd_inputs(x)
        ref = dense_reference(x)
        assert o.shape == ref.shape
        if o.size:
            assert _rel(o, ref) <= 1e-12, (seed, _rel(o, ref))


@pytest.mark.parametrize("act,bias_len,causal", MODES)
def test_backward_matches_torch_autograd(act, bias_len, causal):
    for seed in range(6):
        d = (4, 8)[seed % 2]
        x = workloads.random_case(200 + seed, batch=1 + seed % 4, heads=1 + seed % 2,
                                  head_dim=d, act=act, lq_range=(1, 12), lkv_range=(1, 12),
                                  causal=causal, bias_len=bias_len, allow_empty=(seed % 3 == 2))
        dq, dk, dv, db = oracle.bwd_inputs(x)
        rq, rk, rv, rb = dense_torch_grads(x)
        for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
            assert got.shape == ref.shape
            if ref.size and np.max(np.abs(ref)) > 0:
                assert _rel(got, ref) <= 1e-10, (seed, _rel(got, ref))
        if bias_len:
            assert _rel(db, rb) <= 1e-10


@pytest.mark.parametrize("act", ["gelu", "silu", "softmax"])
def test_backward_finite_differences(act):
    """Central differences (h = 1e-6) of L = sum(O * dO) on every input element."""
    x = workloads.random_case(7, batch=2, heads=2, head_dim=4, act=act, lq_range=(1, 5),
                              lkv_range=(1, 5), causal=(act == "softmax"), bias_len=5)
    q = x.q.double().numpy()
    k = x.k.double().numpy()
    v = x.v.double().numpy()
    bias = x.bias.double().numpy()
    dout = x.dout.double().numpy()

    def loss(q_, k_, v_, b_):
        o, _ = oracle.fwd(q_, k_, v_, x.q_offsets, x.kv_offsets, x.heads, x.head_dim, act,
                          x.scale, bias=b_, causal=x.causal)
        return float(np.sum(o * dout))

    dq, dk, dv, db = oracle.bwd(q, k, v, dout, x.q_offsets, x.kv_offsets, x.heads, x.head_dim,
                                act, x.scale, bias=bias, causal=x.causal)
    h = 1e-6
    args = [q, k, v, bias]
    grads = [dq, dk, dv, db]
    for which in range(4):
        base = args[which]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        scale = max(np.max(np.abs(fd)), 1e-3)
        assert np.max(np.abs(fd - grads[which])) / scale <= 1e-6, which


def test_identity_activation_associativity():
    """With act(x) = x, no bias, non-causal: (s Q K^T) V == s Q (K^T V) per segment."""
    for seed in range(10):
        x = workloads.random_case(300 + seed, batch=3, heads=2, head_dim=8, act="gelu",
                                  lq_range=(1, 16), lkv_range=(1, 16))
        o, _ = oracle.fwd(x.q, x.k, x.v, x.q_offsets, x.kv_offsets, x.heads, x.head_dim,
                          "identity", x.scale)
        q = x.q.double().numpy()
        k = x.k.double().numpy()
        v = x.v.double().numpy()
        qo, ko = x.q_offsets.numpy(), x.kv_offsets.numpy()
        for b in range(x.batch):
            for h in range(x.heads):
                qs = q[qo[b]:qo[b + 1], h]
                ks = k[ko[b]:ko[b + 1], h]
                vs = v[ko[b]:ko[b + 1], h]
                ref = x.scale * (qs @ (ks.T @ vs))
                got = o[qo[b]:qo[b + 1], h]
                assert _rel(got, ref) <= 1e-12


@pytest.mark.parametrize("act", ["gelu", "silu", "softmax"])
def test_segment_permutation_invariance(act):
    x = workloads.random_case(11, batch=6, heads=2, head_dim=8, act=act, lq_range=(0, 9),
                              lkv_range=(0, 9), causal=(act == "softmax"), bias_len=9)
    perm = np.random.default_rng(5).permutation(x.batch)
    qo, ko = x.q_offsets.numpy(), x.kv_offsets.numpy()
    qidx = np.concatenate([np.arange(qo[b], qo[b + 1]) for b in perm]).astype(np.int64)
    kidx = np.concatenate([np.arange(ko[b], ko[b + 1]) for b in perm]).astype(np.int64)
    y = workloads.make_inputs(x.lq[perm], x.lkv[perm], x.heads, x.head_dim, act, x.causal, 9)
    y.q, y.k, y.v, y.dout = x.q[qidx], x.k[kidx], x.v[kidx], x.dout[qidx]
    y.bias = x.bias
    o1, l1 = oracle.fwd_inputs(x)
    o2, l2 = oracle.fwd_inputs(y)
    assert np.array_equal(o1[qidx], o2)
    assert np.array_equal(l1[:, qidx], l2)
    g1 = oracle.bwd_inputs(x)
    g2 = oracle.bwd_inputs(y)
    assert np.array_equal(g1[0][qidx], g2[0])
    assert np.array_equal(g1[1][kidx], g2[1])
    assert np.array_equal(g1[2][kidx], g2[2])
    assert np.allclose(g1[3], g2[3], rtol=1e-12, atol=1e-14)


def test_softmax_matches_torch_softmax():
    """Softmax mode, no bias, Lq = Lkv: each segment is textbook causal attention."""
    for seed in range(5):
        rng = np.random.default_rng(seed)
        lens = rng.integers(1, 24, size=4)
        x = workloads.make_inputs(lens, lens, 3, 16, "softmax", causal=True, rng=rng)
        o, lse = oracle.fwd_inputs(x)
        qo = x.q_offsets.numpy()
        for b in range(x.batch):
            for h in range(x.heads):
                qs = x.q[qo[b]:qo[b + 1], h].double()
                ks = x.k[qo[b]:qo[b + 1], h].double()
                vs = x.v[qo[b]:qo[b + 1], h].double()
                s = x.scale * qs @ ks.T
                n = s.shape[0]
                s = s.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), -torch.inf)
                ref = torch.softmax(s, dim=-1) @ vs
                assert _rel(o[qo[b]:qo[b + 1], h], ref.numpy()) <= 1e-12
                assert np.allclose(lse[h, qo[b]:qo[b + 1]], torch.logsumexp(s, -1).numpy(),
                                   rtol=1e-13, atol=1e-13)


def test_activation_closed_forms():
    g = json.load(open(GOLDEN))
    for name, key in (("gelu", "gelu"), ("silu", "silu")):
        pts = [float(t) for t in g[key] if not t.startswith("_")]
        y, dy = oracle.act(name, pts)
        for t, val in zip(pts, y):
            assert abs(val - g[key][repr(t)]) <= 1e-14, (name, t)
        dk = key + "_prime"
        dpts = [float(t) for t in g[dk]]
        _, dyy = oracle.act(name, dpts)
        for t, val in zip(dpts, dyy):
            assert abs(val - g[dk][repr(t)]) <= 1e-14, (name, "prime", t)


def test_single_key_closed_form():
    """Lkv = 1: O_i = act(s q_i.k_0 + bias[h][clamp(i)+R]) v_0 for every row i."""
    g = json.load(open(GOLDEN))
    d = 2
    q = np.zeros((3, 1, d))
    q[:, 0, 0] = [1.0, 2.0, -1.0]        # q_i . k_0 = q_i[0] with k_0 = e_0
    k = np.zeros((1, 1, d))
    k[0, 0, 0] = 1.0
    v = np.zeros((1, 1, d))
    v[0, 0] = [3.0, -2.0]
    qo = np.array([0, 3], np.int32)
    ko = np.array([0, 1], np.int32)
    o, _ = oracle.fwd(q, k, v, qo, ko, 1, d, "gelu", 1.0)
    expect = [g["gelu"]["1.0"], g["gelu"]["2.0"], g["gelu"]["-1.0"]]
    for i in range(3):
        assert np.allclose(o[i, 0], np.array([3.0, -2.0]) * expect[i], rtol=1e-14, atol=0)
    # A bias table of 3 entries (R = 1): row i uses entry clamp(i - 0, -1, 1) + 1.
    # Choose the table so that x_i hits the golden points 1, 2, 1 after the bias.
    bias = np.array([[0.0, 0.0, 0.0]])
    q2 = q.copy()
    q2[:, 0, 0] = [1.0, 3.0, 2.0]
    bias[0] = [5.0, 0.0, -1.0]           # i=0 -> entry 1 (0.0); i=1,2 -> entry 2 (-1.0)
    o, _ = oracle.fwd(q2, k, v, qo, ko, 1, d, "silu", 1.0, bias=bias)
    expect = [g["silu"]["1.0"], 2.0 / (1.0 + math.exp(-2.0)), g["silu"]["1.0"]]
    for i in range(3):
        assert np.allclose(o[i, 0], np.array([3.0, -2.0]) * expect[i], rtol=1e-14, atol=0)


def test_zero_query_closed_forms():
    """Q = 0, no bias: GELU/SiLU give O = 0; softmax gives the mean of the valid v_j."""
    x = workloads.random_case(3, batch=3, heads=2, head_dim=8, act="softmax",
                              lq_range=(1, 9), lkv_range=(1, 9), causal=True)
    x.q = torch.zeros_like(x.q)
    for act in ("gelu", "silu"):
        o, _ = oracle.fwd(x.q, x.k, x.v, x.q_offsets, x.kv_offsets, x.heads, x.head_dim, act,
                          x.scale)
        assert np.all(o == 0.0)
    o, lse = oracle.fwd_inputs(x)
    v = x.v.double().numpy()
    qo, ko = x.q_offsets.numpy(), x.kv_offsets.numpy()
    for b in range(x.batch):
        for i in range(x.lq[b]):
            n = min(i + 1, x.lkv[b])
            ref = v[ko[b]:ko[b] + n].mean(axis=0)
            assert np.allclose(o[qo[b] + i], ref, rtol=1e-13, atol=1e-13)
            assert np.allclose(lse[:, qo[b] + i], math.log(n), rtol=1e-13)
    # causal softmax row 0 attends to key 0 only: O_0 = v_0
    for b in range(x.batch):
        assert np.allclose(o[qo[b]], v[ko[b]], rtol=0, atol=1e-15)


def test_empty_segments():
    """Lkv = 0 gives O = 0 (LSE = -inf in softmax mode) and zero gradients."""
    x = workloads.make_inputs([3, 0, 2], [0, 4, 2], 2, 8, "softmax", bias_len=5, seed=1)
    o, lse = oracle.fwd_inputs(x)
    assert np.all(o[:3] == 0.0)
    assert np.all(np.isneginf(lse[:, :3]))
    dq, dk, dv, db = oracle.bwd_inputs(x)
    assert np.all(dq[:3] == 0.0)
    assert np.all(dk[0:4] == 0.0) and np.all(dv[0:4] == 0.0)   # segment 1 has no queries
    assert np.all(np.isfinite(db))


def test_workload_lengths_are_reproduced():
    """The realized lengths of the workloads and the offsets derived from them
    (the sliding-window workload draws the long-tail batch)."""
    expect_tot = {1: (147, 22), 2: (133254, 133254), 3: (1054174, 82241),
                  4: (8192, 1039300), 5: (147612, 147612), 6: (147612, 147612)}
    for idx, w in workloads.WORKLOADS.items():
        lq, lkv = workloads.lengths_for(w)
        assert (int(lq.sum()), int(lkv.sum())) == expect_tot[idx]
        qo = workloads.offsets_from_lengths(lq).numpy()
        assert qo[0] == 0 and np.array_equal(np.diff(qo), lq)
    lq, lkv = workloads.lengths_for(workloads.WORKLOADS[1])
    assert lq.tolist() == [55, 41, 33, 18] and lkv.tolist() == [15, 2, 4, 1]
    lq, _ = workloads.lengths_for(workloads.WORKLOADS[5])
    assert int(lq.max()) == 14270 and int(lq.min()) >= 100


def test_unit_subset_equals_full_run():
    """Restricting the oracle to some (segment, head) units reproduces those rows."""
    x = workloads.random_case(21, batch=4, heads=3, head_dim=8, act="gelu",
                              lq_range=(1, 10), lkv_range=(1, 10), bias_len=7)
    o, _ = oracle.fwd_inputs(x)
    dq, dk, dv, db = oracle.bwd_inputs(x)
    units = [1 * 3 + 2, 3 * 3 + 0]
    os_, _ = oracle.fwd_inputs(x, units=units)
    gq, gk, gv, _ = oracle.bwd_inputs(x, units=units)
    qo, ko = x.q_offsets.numpy(), x.kv_offsets.numpy()
    for u in units:
        b, h = divmod(u, 3)
        assert np.array_equal(os_[qo[b]:qo[b + 1], h], o[qo[b]:qo[b + 1], h])
        assert np.array_equal(gq[qo[b]:qo[b + 1], h], dq[qo[b]:qo[b + 1], h])
        assert np.array_equal(gk[ko[b]:ko[b + 1], h], dk[ko[b]:ko[b + 1], h])
        assert np.array_equal(gv[ko[b]:ko[b + 1], h], dv[ko[b]:ko[b + 1], h])


# ----------------------------------------------------------------------------
# Sliding window (|i - j| < w, segment-local)
# ----------------------------------------------------------------------------

WINDOW_MODES = [(a, c, w) for a in ("gelu", "softmax") for c in (False, True) for w in (1, 3, 8)]


@pytest.mark.parametrize("act,causal,window", WINDOW_MODES)
def test_window_forward_matches_dense_bruteforce(act, causal, window):
    for seed in range(8):
        x = workloads.random_case(700 + seed, batch=1 + seed % 5, heads=1 + seed % 2,
                                  head_dim=(4, 8)[seed % 2], act=act, lq_range=(1, 20),
                                  lkv_range=(1, 20), causal=causal, bias_len=(0, 7)[seed % 2],
                                  allow_empty=(seed % 4 == 3), window=window)
        o, _ = oracle.fwd_inputs(x)
        ref = dense_reference(x)
        if o.size:
            assert _rel(o, ref) <= 1e-12, (seed, _rel(o, ref))


@pytest.mark.parametrize("act,causal,window", WINDOW_MODES)
def test_window_backward_matches_torch_autograd(act, causal, window):
    for seed in range(4):
        x = workloads.random_case(800 + seed, batch=1 + seed % 3, heads=1 + seed % 2,
                                  head_dim=4, act=act, lq_range=(1, 12), lkv_range=(1, 12),
                                  causal=causal, bias_len=(0, 5)[seed % 2], window=window)
        dq, dk, dv, db = oracle.bwd_inputs(x)
        rq, rk, rv, rb = dense_torch_grads(x)
        for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
            if ref.size and np.max(np.abs(ref)) > 0:
                assert _rel(got, ref) <= 1e-10, (seed, _rel(got, ref))
        if x.bias is not None:
            assert _rel(db, rb) <= 1e-10


def test_window_finite_differences():
    """Central differences of L = sum(O * dO) under a window, GELU with bias."""
    x = workloads.random_case(901, batch=2, heads=1, head_dim=3, act="gelu", lq_range=(2, 6),
                              lkv_range=(2, 6), bias_len=5, window=2)
    q, k, v = x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy()
    do, bias = x.dout.double().numpy(), x.bias.double().numpy()

    def loss(q_, k_, v_, b_):
        o, _ = oracle.fwd(q_, k_, v_, x.q_offsets, x.kv_offsets, x.heads, x.head_dim, "gelu",
                          x.scale, bias=b_, window=x.window)
        return float(np.sum(o * do))

    dq, dk, dv, db = oracle.bwd(q, k, v, do, x.q_offsets, x.kv_offsets, x.heads, x.head_dim,
                                "gelu", x.scale, bias=bias, window=x.window)
    h = 1e-6
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2), (bias, db, 3)):
        num = np.zeros_like(arr)
        flat, nflat = arr.reshape(-1), num.reshape(-1)
        for e in range(flat.size):
            keep = flat[e]
            args = [q, k, v, bias]
            flat[e] = keep + h
            lp = loss(*args)
            flat[e] = keep - h
            lm = loss(*args)
            flat[e] = keep
            nflat[e] = (lp - lm) / (2 * h)
        assert _rel(grad, num) <= 1e-6, (which, _rel(grad, num))


@pytest.mark.parametrize("act", ["gelu", "silu", "softmax"])
def test_window_of_one_closed_form(act):
    """w = 1 leaves the diagonal only: O_i = act(s q_i.k_i + B[h][R]) v_i for
    GELU / SiLU, and O_i = v_i with LSE_i = x_ii for softmax (Lq = Lkv)."""
    lens = np.array([5, 1, 9])
    x = workloads.make_inputs(lens, lens, 2, 8, act, bias_len=7, seed=31, window=1)
    o, lse = oracle.fwd_inputs(x)
    q, k, v = x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy()
    bias = x.bias.double().numpy()
    off = x.q_offsets.numpy()
    for b in range(len(lens)):
        for i in range(lens[b]):
            r = off[b] + i
            for h in range(2):
                xi = x.scale * float(q[r, h] @ k[r, h]) + bias[h, 3]
                if act == "softmax":
                    assert np.allclose(o[r, h], v[r, h], rtol=0, atol=1e-12)
                    assert abs(lse[h, r] - xi) <= 1e-12
                else:
                    a = xi * 0.5 * (1 + math.erf(xi / math.sqrt(2))) if act == "gelu" else xi * sps.expit(xi)
                    assert np.allclose(o[r, h], a * v[r, h], rtol=0, atol=1e-12)


@pytest.mark.parametrize("act", ["gelu", "softmax"])
def test_window_covering_every_pair_equals_no_window(act):
    x = workloads.random_case(950, batch=4, heads=2, head_dim=8, act=act, lq_range=(1, 20),
                              lkv_range=(1, 20), causal=(act == "softmax"), bias_len=7)
    import dataclasses
    y = dataclasses.replace(x, window=20)
    o0, l0 = oracle.fwd_inputs(x)
    o1, l1 = oracle.fwd_inputs(y)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    g0, g1 = oracle.bwd_inputs(x), oracle.bwd_inputs(y)
    for a, b in zip(g0, g1):
        assert np.array_equal(a, b)


def test_window_rows_without_keys():
    """Lq > Lkv + w - 1: rows i >= Lkv + w - 1 see no key: O_i = 0, LSE_i = -inf,
    and those rows contribute nothing to any gradient."""
    x = workloads.make_inputs([12], [3], 1, 4, "softmax", seed=5, window=2)
    o, lse = oracle.fwd_inputs(x)
    assert np.all(o[4:] == 0.0) and np.all(np.isneginf(lse[0, 4:]))
    assert np.all(np.isfinite(lse[0, :4]))
    dq, dk, dv, _ = oracle.bwd_inputs(x)
    assert np.all(dq[4:] == 0.0)
    y = workloads.make_inputs([4], [3], 1, 4, "softmax", seed=5, window=2)
    y = type(y)(**{**y.__dict__, "q": x.q[:4], "dout": x.dout[:4], "k": x.k, "v": x.v})
    _, dk4, dv4, _ = oracle.bwd_inputs(y)
    assert np.allclose(dk, dk4, rtol=0, atol=1e-14) and np.allclose(dv, dv4, rtol=0, atol=1e-14)


# ----------------------------------------------------------------------------
# Shared query rows (PMA-style pooling): q_shared = S
# ----------------------------------------------------------------------------

def _shared_case(seed, act, batch=4, s=5, heads=2, d=8, bias_len=7, causal=False):
    rng = np.random.default_rng(seed)
    lkv = rng.integers(0, 14, size=batch)
    return workloads.make_inputs(np.full(batch, s), lkv, heads, d, act, causal=causal, bias_len=bias_len,
                                 rng=rng, shared_q=s)


@pytest.mark.parametrize("act,causal", [("gelu", False), ("silu", True), ("softmax", False), ("softmax", True)])
def test_shared_queries_equal_the_expanded_batch(act, causal):
    """Shared rows read by every segment give the expanded batch's O, LSE, dK,
    dV exactly, and dQ equal to the expanded dQ summed over segments."""
    x = _shared_case(60 + len(act) + int(causal), act, causal=causal)
    s = x.q_seed.shape[0]
    o_e, l_e = oracle.fwd_inputs(x)
    dq_e, dk_e, dv_e, db_e = oracle.bwd_inputs(x)
    args = (x.k, x.v)
    o_s, l_s = oracle.fwd(x.q_seed, *args, x.q_offsets, x.kv_offsets, x.heads, x.head_dim, act, x.scale,
                          bias=x.bias, causal=causal, q_shared=s)
    dq_s, dk_s, dv_s, db_s = oracle.bwd(x.q_seed, *args, x.dout, x.q_offsets, x.kv_offsets, x.heads,
                                        x.head_dim, act, x.scale, bias=x.bias, causal=causal, q_shared=s)
    assert np.array_equal(o_s, o_e) and np.array_equal(l_s, l_e)
    assert np.array_equal(dk_s, dk_e) and np.array_equal(dv_s, dv_e)
    assert np.allclose(db_s, db_e, rtol=1e-13, atol=1e-15)
    want = dq_e.reshape(x.batch, s, x.heads, x.head_dim).sum(axis=0)
    assert dq_s.shape == (s, x.heads, x.head_dim)
    assert _rel(dq_s, want) <= 1e-12


@pytest.mark.parametrize("act", ["gelu", "softmax"])
def test_shared_query_gradient_matches_autograd_through_the_broadcast(act):
    """dQ of the shared rows against torch autograd on a dense formulation in
    which one [S, H, d] leaf is broadcast to every segment."""
    x = _shared_case(71, act, batch=3, s=4, d=4, bias_len=5)
    s, b = x.q_seed.shape[0], x.batch
    lkm = max(1, int(x.lkv.max()))
    ko = x.kv_offsets.numpy().astype(np.int64)
    qs = torch.tensor(x.q_seed.double().numpy(), requires_grad=True)            # [S, H, d]
    kp = torch.tensor(_pad(x.k.double().numpy(), ko, lkm))
    vp = torch.tensor(_pad(x.v.double().numpy(), ko, lkm))
    dop = torch.tensor(x.dout.double().numpy().reshape(b, s, x.heads, x.head_dim))
    i = torch.arange(s)[:, None]
    j = torch.arange(lkm)[None, :]
    mask = (j[None] < torch.tensor(x.lkv)[:, None, None]).expand(b, s, lkm)
    m4 = mask[:, None]
    sc = torch.einsum("ihc,bjhc->bhij", qs, kp) * x.scale
    r = (x.bias.shape[1] - 1) // 2
    sc = sc + x.bias.double()[:, torch.clamp(i - j, -r, r) + r][None]
    if act == "softmax":
        sm = torch.where(m4, sc, torch.full_like(sc, -torch.inf))
        sm = torch.where(m4.any(-1, keepdim=True), sm, torch.zeros_like(sm))
        p = torch.where(m4, torch.softmax(sm, dim=-1), torch.zeros_like(sm))
    else:
        p = torch.where(m4, torch.nn.functional.gelu(sc), torch.zeros_like(sc))
    o = torch.einsum("bhij,bjhc->bihc", p, vp)
    (o * dop).sum().backward()
    dq_s, _, _, _ = oracle.bwd(x.q_seed, x.k, x.v, x.dout, x.q_offsets, x.kv_offsets, x.heads, x.head_dim,
                               act, x.scale, bias=x.bias, q_shared=s)
    assert _rel(dq_s, qs.grad.numpy()) <= 1e-10


def test_shared_queries_need_equal_segment_lengths():
    x = workloads.make_inputs([3, 4], [5, 5], 1, 4, "gelu", seed=2)
    with pytest.raises(ValueError):
        oracle.fwd(x.q[:3], x.k, x.v, x.q_offsets, x.kv_offsets, 1, 4, "gelu", x.scale, q_shared=3)


# ----------------------------------------------------------------------------
# Row-restricted backward (single rows of long units)
# ----------------------------------------------------------------------------

ROW_MODES = [(a, c, w, bl) for a in ("gelu", "silu", "softmax") for c in (False, True) for w in (0, 5)
             for bl in (0, 7)]


@pytest.mark.parametrize("act,causal,window,bias_len", ROW_MODES)
def test_backward_rows_equal_the_full_backward(act, causal, window, bias_len):
    """dQ / dK / dV of selected rows equal the full backward's rows bit for bit
    (same per-pair quantities, same summation order), and match torch
    autograd on the dense form."""
    x = workloads.random_case(900 + window + bias_len + int(causal), batch=3, heads=2, head_dim=8, act=act,
                              lq_range=(1, 15), lkv_range=(1, 15), causal=causal, bias_len=bias_len,
                              window=window)
    dq, dk, dv, _ = oracle.bwd_inputs(x)
    rq, rk, rv, _ = dense_torch_grads(x)
    qo, ko = x.q_offsets.numpy(), x.kv_offsets.numpy()
    rng = np.random.default_rng(3)
    for b in range(x.batch):
        for h in range(x.heads):
            qr = np.sort(rng.choice(int(x.lq[b]), size=min(4, int(x.lq[b])), replace=False))
            kr = np.sort(rng.choice(int(x.lkv[b]), size=min(4, int(x.lkv[b])), replace=False))
            gq, gk, gv = oracle.bwd_rows_inputs(x, b, h, qr, kr)
            assert np.array_equal(gq, dq[qo[b] + qr, h])
            assert np.array_equal(gk, dk[ko[b] + kr, h])
            assert np.array_equal(gv, dv[ko[b] + kr, h])
            for got, ref in ((gq, rq[qo[b] + qr, h]), (gk, rk[ko[b] + kr, h]), (gv, rv[ko[b] + kr, h])):
                if np.max(np.abs(ref), initial=0) > 0:
                    assert _rel(got, ref) <= 1e-10


def test_backward_rows_reject_rows_outside_the_segment():
    x = workloads.random_case(5, batch=2, heads=1, head_dim=4, act="gelu", lq_range=(3, 5), lkv_range=(3, 5))
    with pytest.raises(ValueError):
        oracle.bwd_rows_inputs(x, 0, 0, [int(x.lq[0])], [])
    with pytest.raises(ValueError):
        oracle.bwd_rows_inputs(x, 0, 0, [], [-1])
    with pytest.raises(ValueError):
        oracle.bwd_rows_inputs(x, 2, 0, [0], [0])
