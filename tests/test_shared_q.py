"""GPU parity of the shared-query (PMA-style pooling) entry points against
the fp64 oracle's shared-query mode.

Every segment attends with the same S query rows (learned seed queries
shared across the batch, "GEM Training: How Meta Doubled the Efficiency of
Its ...", section "What to watch"); O, dO and LSE keep one block of S rows per
segment, and dQ of the shared rows is the sum over segments.  The kernels
read Q once per segment from the S-row tensor (no expanded copy) and the
summed dQ comes from a fixed-order reduction, so no caller-side expand or sum
is involved.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_close, full_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jg():
    import __graft_entry__
    __graft_entry__.build()
    import jagged_gdpa_gb300 as m
    return m


def shared_case(seed, s, batch, heads, d, act, bias_len=0, causal=False, lkv_range=(1, 300), window=0):
    rng = np.random.default_rng(seed)
    lkv = rng.integers(lkv_range[0], lkv_range[1] + 1, size=batch)
    lkv[rng.integers(0, batch)] = 0  # one segment without keys
    return workloads.make_inputs(np.full(batch, s), lkv, heads, d, act, causal=causal, bias_len=bias_len,
                                 rng=rng, shared_q=s, window=window)


def run(jg, x, stored):
    d = x.to("cuda")
    out, lse = jg.jgdpa_fwd_shared_q(d.q_seed, d.k, d.v, d.kv_offsets, x.act, x.scale, bias_table=d.bias,
                                     causal=x.causal, window=x.window)
    scratch = None
    if stored:
        n = jg.jgdpa_ds_scratch_bytes(x.q_offsets, x.kv_offsets, x.heads)
        scratch = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    s = x.q_seed.shape[0]
    ws = torch.empty(jg.jgdpa_shared_q_workspace_bytes(x.batch, s, x.k.shape[0], x.heads, x.head_dim, x.act,
                                                       x.bias_len, True), dtype=torch.uint8, device="cuda")
    dq, dk, dv, db = jg.jgdpa_bwd_shared_q(d.q_seed, d.k, d.v, out, lse, d.dout, d.kv_offsets, x.act, x.scale,
                                           bias_table=d.bias, causal=x.causal, workspace=ws, ds_scratch=scratch,
                                           window=x.window)
    torch.cuda.synchronize()
    assert jg.jgdpa_read_device_status(ws) == 0
    return out.cpu(), (None if lse is None else lse.cpu()), dq.cpu(), dk.cpu(), dv.cpu(), \
        (None if db is None else db.cpu())


def reference(x, units=None):
    s = x.q_seed.shape[0]
    o, lse = oracle.fwd(x.q_seed, x.k, x.v, x.q_offsets, x.kv_offsets, x.heads, x.head_dim, x.act, x.scale,
                        bias=x.bias, causal=x.causal, q_shared=s, units=units, window=x.window)
    dq, dk, dv, db = oracle.bwd(x.q_seed, x.k, x.v, x.dout, x.q_offsets, x.kv_offsets, x.heads, x.head_dim,
                                x.act, x.scale, bias=x.bias, causal=x.causal, q_shared=s, units=units,
                                window=x.window)
    return o, lse, dq, dk, dv, db


CASES = [(d, act, s, bias_len, causal) for d in (32, 64, 128) for act in ("gelu", "silu", "softmax")
         for (s, bias_len, causal) in ((16, 0, False), (130, 7, True))]


@pytest.mark.parametrize("stored", [False, True])
@pytest.mark.parametrize("d,act,s,bias_len,causal", CASES)
def test_shared_queries_match_the_oracle(jg, d, act, s, bias_len, causal, stored):
    x = shared_case(7000 + d + s, s, batch=6, heads=2, d=d, act=act, bias_len=bias_len, causal=causal)
    out, lse, dq, dk, dv, db = run(jg, x, stored)
    ro, rl, rq, rk, rv, rb = reference(x)
    tag = f"d={d} {act} S={s} bias={bias_len} causal={causal}{' stored-dS' if stored else ''}"
    assert_close(f"O {tag}", out, ro)
    if act == "softmax":
        fin = np.isfinite(rl)
        assert np.array_equal(np.isfinite(lse.numpy()), fin)
        assert_close(f"LSE {tag}", lse.numpy()[fin], rl[fin])
    assert dq.shape == (s, x.heads, d)
    assert_close(f"dQ (sum over segments) {tag}", dq, rq)
    assert_close(f"dK {tag}", dk, rk)
    assert_close(f"dV {tag}", dv, rv)
    if bias_len:
        assert_close(f"dbias {tag}", db, rb)


# the short-query forward and backward (keys on the MMA's rows; GELU / SiLU,
# S <= 64) at each of their widths NQ = 16, 32, 64, with bias, causal masking
# and a window
SHORT = [(d, act, s, causal, w) for d in (32, 64, 128) for act in ("gelu", "silu") for (s, causal, w) in
         ((5, False, 0), (20, True, 0), (40, False, 0), (64, False, 37), (33, True, 130))]


@pytest.mark.parametrize("d,act,s,causal,w", SHORT)
def test_short_query_widths(jg, d, act, s, causal, w):
    x = shared_case(7100 + d + s + w, s, batch=7, heads=2, d=d, act=act, bias_len=7, causal=causal,
                    lkv_range=(1, 400), window=w)
    out, _, dq, dk, dv, db = run(jg, x, stored=True)
    ro, _, rq, rk, rv, rb = reference(x)
    tag = f"short-query d={d} {act} S={s} causal={causal} window={w}"
    assert_close(f"O {tag}", out, ro)
    assert_close(f"dQ {tag}", dq, rq)
    assert_close(f"dK {tag}", dk, rk)
    assert_close(f"dV {tag}", dv, rv)
    assert_close(f"dbias {tag}", db, rb)


# segments of more than one chunk of key tiles (16 tiles = 2048 keys): each
# chunk writes its own dQ contribution; the first two key tiles of every
# segment meet the bias table's band (R = 128), the rest its first entry
CHUNKS = [(d, act, s) for d in (32, 64, 128) for (act, s) in (("gelu", 16), ("silu", 48))]


@pytest.mark.parametrize("d,act,s", CHUNKS)
def test_short_query_backward_chunks(jg, d, act, s):
    x = shared_case(7200 + d + s, s, batch=3, heads=2, d=d, act=act, bias_len=257, lkv_range=(1500, 5000))
    out, _, dq, dk, dv, db = run(jg, x, stored=False)
    ro, _, rq, rk, rv, rb = reference(x)
    tag = f"short-query chunks d={d} {act} S={s}"
    assert_close(f"O {tag}", out, ro)
    assert_close(f"dQ {tag}", dq, rq)
    assert_close(f"dK {tag}", dk, rk)
    assert_close(f"dV {tag}", dv, rv)
    assert_close(f"dbias {tag}", db, rb)


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_short_query_backward_chunk_edges(jg, act):
    """Key counts at the short-query backward's edges: one and two tiles
    around 128, exactly one chunk of 16 tiles (2048 keys), one key past it
    (a second chunk of one tile), two full chunks, and no keys."""
    rng = np.random.default_rng(7300)
    lkv = np.array([2048, 2049, 1, 128, 129, 4096, 0])
    x = workloads.make_inputs(np.full(len(lkv), 16), lkv, 2, 64, act, bias_len=257, rng=rng, shared_q=16)
    out, _, dq, dk, dv, db = run(jg, x, stored=False)
    ro, _, rq, rk, rv, rb = reference(x)
    tag = f"short-query chunk edges {act}"
    assert_close(f"O {tag}", out, ro)
    assert_close(f"dQ {tag}", dq, rq)
    assert_close(f"dK {tag}", dk, rk)
    assert_close(f"dV {tag}", dv, rv)
    assert_close(f"dbias {tag}", db, rb)


def test_shared_queries_equal_the_expanded_batch(jg):
    """The shared-query call matches the regular call on the expanded batch:
    O, dK and dV within the parity bar (the short-query kernels sum over the
    16 query rows in another order than the 128-row tiles) and dQ equal to
    the expanded dQ summed over segments."""
    x = shared_case(77, 16, batch=9, heads=3, d=64, act="silu")
    out, _, dq, dk, dv, _ = run(jg, x, stored=True)
    d = x.to("cuda")
    o2, _ = jg.jgdpa_fwd(d.q, d.k, d.v, d.q_offsets, d.kv_offsets, x.act, x.scale)
    n = jg.jgdpa_ds_scratch_bytes(x.q_offsets, x.kv_offsets, x.heads)
    dq2, dk2, dv2, _ = jg.jgdpa_bwd(d.q, d.k, d.v, None, None, d.dout, d.q_offsets, d.kv_offsets, x.act, x.scale,
                                   ds_scratch=torch.empty(n, dtype=torch.uint8, device="cuda"))
    assert_close("O vs expanded O", out, o2.double().cpu().numpy())
    assert_close("dK vs expanded dK", dk, dk2.double().cpu().numpy())
    assert_close("dV vs expanded dV", dv, dv2.double().cpu().numpy())
    summed = dq2.float().cpu().view(x.batch, 16, x.heads, 64).sum(0)
    assert_close("dQ vs expanded dQ summed", dq, summed.double().numpy())


@pytest.mark.parametrize("stored", [False, True])
def test_pma_workload_full_size(jg, stored):
    """The PMA workload at full size (B=512, H=8, d=64, S=16 shared seed
    queries, Lkv ~ U[1, 4096], SiLU): O and dK / dV on sampled segments, and
    the summed dQ against the oracle over the whole batch."""
    x = full_workload(4)
    out, _, dq, dk, dv, _ = run(jg, x, stored)
    rng = np.random.default_rng(4 + int(stored))
    segs = sorted(int(b) for b in rng.choice(x.batch, size=6, replace=False))
    units = [b * x.heads + int(rng.integers(0, x.heads)) for b in segs]
    ro, _, rq, rk, rv, _ = reference(x)
    qo, ko = x.q_offsets.numpy(), x.kv_offsets.numpy()
    got_o, want_o, got_k, want_k, got_v, want_v = [], [], [], [], [], []
    for u in units:
        b, h = divmod(u, x.heads)
        got_o.append(out.float().numpy()[qo[b]:qo[b + 1], h])
        want_o.append(ro[qo[b]:qo[b + 1], h])
        got_k.append(dk.float().numpy()[ko[b]:ko[b + 1], h])
        want_k.append(rk[ko[b]:ko[b + 1], h])
        got_v.append(dv.float().numpy()[ko[b]:ko[b + 1], h])
        want_v.append(rv[ko[b]:ko[b + 1], h])
    tag = f"PMA full size{' stored-dS' if stored else ''}"
    assert_close(f"O {tag}", np.concatenate(got_o), np.concatenate(want_o))
    assert_close(f"dK {tag}", np.concatenate(got_k), np.concatenate(want_k))
    assert_close(f"dV {tag}", np.concatenate(got_v), np.concatenate(want_v))
    assert_close(f"dQ summed over 512 segments {tag}", dq, rq)
