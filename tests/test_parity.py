"""GPU parity: libjgdpa.so (through the C ABI) against the fp64 CPU oracle.

Bar (per output tensor): max|gpu - oracle| <= 2e-2 * max|oracle|; offsets
and lengths are integers and must be reproduced exactly.  Small cases run the
oracle on everything; the named workloads run at full size on the GPU
and the oracle recomputes a sample of (segment, head) units, whose rows are
compared (each unit is independent of the others).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_close, full_workload, oracle_bwd, oracle_fwd, sample_units, sampled_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jg():
    import __graft_entry__
    __graft_entry__.build()
    import jagged_gdpa_gb300 as m
    return m


def run_fwd(jg, x, lib=None):
    d = x.to("cuda")
    out, lse = jg.jgdpa_fwd(d.q, d.k, d.v, d.q_offsets, d.kv_offsets, x.act, x.scale,
                            bias_table=d.bias, causal=x.causal, window=x.window, lib=lib)
    torch.cuda.synchronize()
    return out.cpu(), (None if lse is None else lse.cpu())


def run_bwd(jg, x, out=None, lse=None, stored=False, lib=None):
    """Backward through the C ABI; stored=True takes the stored-dS path
    (jgdpa_bwd_ex with a scratch of exactly jgdpa_ds_scratch_bytes)."""
    d = x.to("cuda")
    if x.act == "softmax":
        out, lse = jg.jgdpa_fwd(d.q, d.k, d.v, d.q_offsets, d.kv_offsets, x.act, x.scale,
                                bias_table=d.bias, causal=x.causal, window=x.window, lib=lib)
    scratch = None
    if stored:
        nbytes = jg.jgdpa_ds_scratch_bytes(x.q_offsets, x.kv_offsets, x.heads, x.window)
        scratch = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    ws = torch.empty(jg.jgdpa_workspace_bytes(x.batch, x.q.shape[0], x.k.shape[0], x.heads, x.head_dim, x.act,
                                              x.bias_len, True), dtype=torch.uint8, device="cuda")
    dq, dk, dv, db = jg.jgdpa_bwd(d.q, d.k, d.v, out, lse, d.dout, d.q_offsets, d.kv_offsets, x.act,
                                  x.scale, bias_table=d.bias, causal=x.causal, workspace=ws, ds_scratch=scratch,
                                  window=x.window, lib=lib)
    torch.cuda.synchronize()
    assert jg.jgdpa_read_device_status(ws, lib=lib) == 0, "device status"
    return dq.cpu(), dk.cpu(), dv.cpu(), (None if db is None else db.cpu())


def check_fwd_full(jg, x, tag="", lib=None):
    out, lse = run_fwd(jg, x, lib=lib)
    ref, rlse = oracle_fwd(x)
    assert_close(f"O {tag}", out, ref)
    if x.act == "softmax":
        valid = np.isfinite(rlse)
        assert np.array_equal(np.isfinite(lse.numpy()), valid), f"LSE -inf pattern {tag}"
        assert_close(f"LSE {tag}", lse.numpy()[valid], rlse[valid])


def check_bwd_full(jg, x, tag="", stored=False, lib=None):
    dq, dk, dv, db = run_bwd(jg, x, stored=stored, lib=lib)
    tag = f"{tag}{' stored-dS' if stored else ''}"
    rq, rk, rv, rb = oracle_bwd(x)
    assert_close(f"dQ {tag}", dq, rq)
    assert_close(f"dK {tag}", dk, rk)
    assert_close(f"dV {tag}", dv, rv)
    if rb is not None:
        assert_close(f"dbias {tag}", db, rb)


# ---------------------------------------------------------------- small cases
SMALL = []
for d in (32, 64, 128):
    for act in ("gelu", "silu", "softmax"):
        for bias_len in (0, 257):
            for causal in (False, True):
                SMALL.append((d, act, bias_len, causal))


@pytest.mark.parametrize("d,act,bias_len,causal", SMALL)
def test_forward_small(jg, d, act, bias_len, causal):
    # several tiles and ragged tails: lengths up to ~3 tiles, some empty segments
    x = workloads.random_case(1000 + d + bias_len + int(causal), batch=5, heads=2, head_dim=d, act=act,
                              lq_range=(1, 300), lkv_range=(1, 300), causal=causal, bias_len=bias_len)
    check_fwd_full(jg, x, f"d={d} {act} bias={bias_len} causal={causal}")


@pytest.mark.parametrize("stored", [False, True])
@pytest.mark.parametrize("d,act,bias_len,causal", SMALL)
def test_backward_small(jg, d, act, bias_len, causal, stored):
    x = workloads.random_case(2000 + d + bias_len + int(causal), batch=4, heads=2, head_dim=d, act=act,
                              lq_range=(1, 300), lkv_range=(1, 300), causal=causal, bias_len=bias_len)
    check_bwd_full(jg, x, f"d={d} {act} bias={bias_len} causal={causal}", stored=stored)


@pytest.mark.parametrize("act", ["gelu", "softmax"])
def test_edge_lengths(jg, act):
    """Empty segments, length 1, multiples of 128 and +-1 around them."""
    lq = [0, 1, 127, 128, 129, 255, 256, 257, 3, 0, 384]
    lkv = [5, 1, 128, 127, 129, 256, 0, 257, 0, 7, 385]
    rng = np.random.default_rng(9)
    x = workloads.make_inputs(lq, lkv, 3, 64, act, causal=False, bias_len=7, rng=rng)
    check_fwd_full(jg, x, "edge fwd")
    check_bwd_full(jg, x, "edge bwd")
    check_bwd_full(jg, x, "edge bwd", stored=True)
    x = workloads.make_inputs(lq, lkv, 3, 64, act, causal=True, bias_len=0, rng=rng)
    check_fwd_full(jg, x, "edge fwd causal")
    check_bwd_full(jg, x, "edge bwd causal")
    check_bwd_full(jg, x, "edge bwd causal", stored=True)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act,causal,bias_len", [("gelu", False, 257), ("softmax", True, 0), ("silu", True, 7)])
def test_key_value_resident_forward(jg, d, act, causal, bias_len):
    """Segments whose keys fit one tile (the key/value-resident forward and
    the direct-dQ backward): one to 128 keys, query counts from one row to
    across one and two chunks of 16 query tiles (2048 / 2049 rows), next to
    segments that take the general kernels."""
    lq = [129, 256, 2048, 2049, 300, 4096, 1, 5000, 200, 128, 77]
    lkv = [1, 64, 127, 128, 128, 33, 100, 300, 0, 128, 5]
    rng = np.random.default_rng(11 + d)
    x = workloads.make_inputs(lq, lkv, 2, d, act, causal=causal, bias_len=bias_len, rng=rng)
    check_fwd_full(jg, x, f"kv-resident fwd d={d} {act} causal={causal}")
    check_bwd_full(jg, x, f"kv-resident bwd d={d} {act} causal={causal}")


@pytest.mark.parametrize("d,act", [(128, "softmax"), (64, "softmax"), (32, "gelu")])
def test_forward_output_16_byte_aligned(jg, d, act):
    """O written through a pointer that is 16- but not 32-byte aligned: the
    epilogues that store 32 bytes at a time where they can (softmax, d = 32)
    fall back to 16-byte stores, in the general and the key/value-resident
    kernels."""
    lq = [300, 77, 1, 2049, 128]
    lkv = [300, 5, 100, 64, 513]
    rng = np.random.default_rng(21 + d)
    x = workloads.make_inputs(lq, lkv, 2, d, act, causal=act == "softmax", bias_len=7, rng=rng)
    dev = x.to("cuda")
    n = x.q.shape[0] * x.heads * d
    buf = torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(x.q.shape[0], x.heads, d)
    assert out.data_ptr() % 32 == 16
    o, _ = jg.jgdpa_fwd(dev.q, dev.k, dev.v, dev.q_offsets, dev.kv_offsets, x.act, x.scale, bias_table=dev.bias,
                        causal=x.causal, out=out)
    torch.cuda.synchronize()
    ref, _ = oracle_fwd(x)
    assert_close(f"O, 16-byte aligned out, d={d} {act}", o.cpu(), ref)
    assert torch.count_nonzero(buf[:8]).item() == 0, "bytes before out written"


# ------------------------------------------------------------ sliding window
WINDOW_FWD = [(d, act, causal, w) for d in (64, 128) for act in ("gelu", "silu", "softmax")
              for causal in (False, True) for w in (1, 129, 300)]
WINDOW_BWD = [(d, act, causal, w) for d in (64, 128) for act in ("gelu", "softmax")
              for causal in (False, True) for w in (1, 129, 300)]


def _window_case(seed, d, act, causal, w, batch):
    # lengths up to ~5.5 tiles, so that whole tiles fall outside the band
    return workloads.random_case(seed, batch=batch, heads=2, head_dim=d, act=act, lq_range=(1, 700),
                                 lkv_range=(1, 700), causal=causal, bias_len=257, window=w)


@pytest.mark.parametrize("d,act,causal,w", WINDOW_FWD)
def test_forward_window(jg, d, act, causal, w):
    x = _window_case(3000 + d + w + int(causal), d, act, causal, w, batch=5)
    check_fwd_full(jg, x, f"d={d} {act} causal={causal} window={w}")


@pytest.mark.parametrize("stored", [False, True])
@pytest.mark.parametrize("d,act,causal,w", WINDOW_BWD)
def test_backward_window(jg, d, act, causal, w, stored):
    x = _window_case(4000 + d + w + int(causal), d, act, causal, w, batch=4)
    check_bwd_full(jg, x, f"d={d} {act} causal={causal} window={w}", stored=stored)


@pytest.mark.parametrize("act", ["gelu", "softmax"])
def test_window_rows_without_keys(jg, act):
    """Lq far beyond Lkv + w: the later query rows (and whole query tiles)
    meet no key: O = 0, LSE = -inf, no gradient from them."""
    lq = [600, 300, 1, 129]
    lkv = [40, 1, 5, 129]
    rng = np.random.default_rng(21)
    for w in (1, 7, 130):
        x = workloads.make_inputs(lq, lkv, 2, 128, act, bias_len=257, rng=rng, window=w)
        check_fwd_full(jg, x, f"no-key rows fwd window={w}")
        check_bwd_full(jg, x, f"no-key rows bwd window={w}")
        check_bwd_full(jg, x, f"no-key rows bwd window={w}", stored=True)


def test_window_covering_every_pair_equals_no_window(jg):
    """A window at least as long as every segment changes nothing (bitwise)."""
    x = workloads.random_case(77, batch=4, heads=2, head_dim=128, act="gelu", lq_range=(1, 400),
                              lkv_range=(1, 400), bias_len=257)
    import dataclasses
    y = dataclasses.replace(x, window=400)
    o0, _ = run_fwd(jg, x)
    o1, _ = run_fwd(jg, y)
    assert torch.equal(o0, o1)
    g0, g1 = run_bwd(jg, x), run_bwd(jg, y)
    for a, b in zip(g0[:3], g1[:3]):
        assert torch.equal(a, b)


def test_workload_1_tiny_full(jg):
    x = workloads.workload_inputs(1)
    check_fwd_full(jg, x, "w1")
    check_bwd_full(jg, x, "w1")
    check_bwd_full(jg, x, "w1", stored=True)


# ------------------------------------------------------ full-size workloads
def check_sampled(jg, x, units_fwd, units_bwd, tag, stored=False):
    """Full-size GPU run; oracle on the sampled units; compare those units' rows
    (each tensor gathered over all sampled units, then one max-relative check).
    The forward is checked on the recompute run only."""
    out, lse = run_fwd(jg, x)
    if stored:
        units_fwd = []
    got, want, got_l, want_l = [], [], [], []
    for b, h, qr, kr, (o, l) in sampled_oracle(x, units_fwd, backward=False):
        got.append(out.float().numpy()[qr, h])
        want.append(o)
        if x.act == "softmax":
            got_l.append(lse.numpy()[h, qr])
            want_l.append(l)
    if got:
        assert_close(f"O {tag}", np.concatenate(got), np.concatenate(want))
    if got_l:
        assert_close(f"LSE {tag}", np.concatenate(got_l), np.concatenate(want_l))
    dq, dk, dv, db = run_bwd(jg, x, stored=stored)
    tag = f"{tag}{' stored-dS' if stored else ''}"
    g = {"dQ": [], "dK": [], "dV": []}
    w = {"dQ": [], "dK": [], "dV": []}
    for b, h, qr, kr, (rq, rk, rv) in sampled_oracle(x, units_bwd, backward=True):
        g["dQ"].append(dq.float().numpy()[qr, h])
        w["dQ"].append(rq)
        g["dK"].append(dk.float().numpy()[kr, h])
        w["dK"].append(rk)
        g["dV"].append(dv.float().numpy()[kr, h])
        w["dV"].append(rv)
    for k in g:
        assert_close(f"{k} {tag}", np.concatenate(g[k]), np.concatenate(w[k]))
    for t in (out, dq, dk, dv):
        assert torch.isfinite(t.float()).all(), f"non-finite output {tag}"


@pytest.mark.parametrize("idx,n_random,max_pairs_fwd,max_pairs_bwd", [
    (2, 6, None, None),
    (3, 6, None, None),
    (4, 6, None, None),
    (5, 4, None, 3e7),
    (6, 4, 4e7, 4e7),
])
def test_full_size_workloads_sampled(jg, idx, n_random, max_pairs_fwd, max_pairs_bwd):
    x = full_workload(idx)
    uf = sample_units(x, n_random, seed=idx, max_pairs=max_pairs_fwd)
    ub = sample_units(x, n_random, seed=100 + idx, max_pairs=max_pairs_bwd)
    check_sampled(jg, x, uf, ub, f"w{idx}")
    check_sampled(jg, x, uf, ub, f"w{idx}", stored=True)


@pytest.mark.parametrize("stored", [False, True])
@pytest.mark.parametrize("idx", [5, 6])
def test_longest_unit_backward_rows(jg, idx, stored):
    """The backward of the workload's longest segment (14,270 tokens, about a
    quarter of the long-tail batch's pairs), one head, at full size in the
    launch configuration the benchmark times: dQ rows of three query tiles
    (first, middle, and the ragged last one) and dK / dV rows of three key
    tiles, against the oracle restricted to those rows."""
    x = full_workload(idx)
    dq, dk, dv, _ = run_bwd(jg, x, stored=stored)
    pairs = x.lq.astype(np.int64) * x.lkv.astype(np.int64)
    b = int(np.argmax(pairs))
    h = (idx + int(stored)) % x.heads
    sub = workloads.select_segments(x, [b])
    rows = []
    for n in (int(x.lq[b]), int(x.lkv[b])):
        last = (n - 1) // 128 * 128
        mid = (n // 2) // 128 * 128
        rows.append(np.unique(np.concatenate([np.arange(0, min(128, n)), np.arange(mid, min(mid + 128, n)),
                                              np.arange(last, n)])))
    qr, kr = rows
    rq, rk, rv = oracle.bwd_rows_inputs(sub, 0, h, qr, kr)
    q0, k0 = int(x.q_offsets[b]), int(x.kv_offsets[b])
    tag = f"w{idx} longest segment b={b} h={h}{' stored-dS' if stored else ''}"
    assert_close(f"dQ {tag}", dq.float().numpy()[q0 + qr, h], rq)
    assert_close(f"dK {tag}", dk.float().numpy()[k0 + kr, h], rk)
    assert_close(f"dV {tag}", dv.float().numpy()[k0 + kr, h], rv)


# ---------------------------------------------- ALU-only activation route
# The same library built with every GELU / SiLU element of the forward and of
# the backward on the ALU polynomial route (no special-function unit), the
# activation design of the GDPA kernel redesign ("Meta redesigns AI training
# infrastructure ...", section "Custom Kernels and 5D Parallelism ...").
ALU_GRID = [(d, act, causal) for d in (32, 64, 128) for act in ("gelu", "silu") for causal in (False, True)]


@pytest.fixture(scope="module")
def alu_lib(jg):
    return jg.load(jg.ALU_LIB_PATH)


@pytest.mark.parametrize("d,act,causal", ALU_GRID)
def test_alu_route_forward_small(jg, alu_lib, d, act, causal):
    x = workloads.random_case(5000 + d + int(causal), batch=5, heads=2, head_dim=d, act=act,
                              lq_range=(1, 300), lkv_range=(1, 300), causal=causal, bias_len=257)
    check_fwd_full(jg, x, f"ALU route d={d} {act} causal={causal}", lib=alu_lib)


@pytest.mark.parametrize("stored", [False, True])
@pytest.mark.parametrize("d,act,causal", ALU_GRID)
def test_alu_route_backward_small(jg, alu_lib, d, act, causal, stored):
    x = workloads.random_case(6000 + d + int(causal), batch=4, heads=2, head_dim=d, act=act,
                              lq_range=(1, 300), lkv_range=(1, 300), causal=causal, bias_len=257)
    check_bwd_full(jg, x, f"ALU route d={d} {act} causal={causal}", stored=stored, lib=alu_lib)


def test_alu_route_long_tail_sampled(jg, alu_lib):
    """The ALU-route kernels on the full long-tail batch, sampled units."""
    x = full_workload(5)
    out, _ = run_fwd(jg, x, lib=alu_lib)
    units = sample_units(x, 3, seed=77, max_pairs=3e7)
    got, want = [], []
    for b, h, qr, kr, (o, _) in sampled_oracle(x, units, backward=False):
        got.append(out.float().numpy()[qr, h])
        want.append(o)
    assert_close("O ALU route w5", np.concatenate(got), np.concatenate(want))
    dq, dk, dv, _ = run_bwd(jg, x, stored=True, lib=alu_lib)
    g = {"dQ": [], "dK": [], "dV": []}
    w = {"dQ": [], "dK": [], "dV": []}
    for b, h, qr, kr, (rq, rk, rv) in sampled_oracle(x, units, backward=True):
        for name, t, rows, ref in (("dQ", dq, qr, rq), ("dK", dk, kr, rk), ("dV", dv, kr, rv)):
            g[name].append(t.float().numpy()[rows, h])
            w[name].append(ref)
    for name in g:
        assert_close(f"{name} ALU route w5 stored-dS", np.concatenate(g[name]), np.concatenate(w[name]))


def test_largest_bias_table_and_more_heads(jg):
    """The largest accepted bias table (4095 entries, R = 2047) on segments
    longer than R, so both clamped ends and the band are hit, with 16 heads."""
    lq = [2600, 5, 300]
    lkv = [2500, 2100, 1]
    rng = np.random.default_rng(41)
    x = workloads.make_inputs(lq, lkv, 16, 64, "gelu", bias_len=4095, rng=rng)
    check_fwd_full(jg, x, "bias 4095, H=16")
    check_bwd_full(jg, x, "bias 4095, H=16", stored=True)


def test_cuda_graph_capture_replays_the_step(jg):
    """Forward + stored-dS backward captured in a CUDA graph and replayed give
    the eager results bit for bit (the library allocates nothing and issues
    only stream-ordered work; buffers and the scratch size are set up first)."""
    x = workloads.random_case(55, batch=4, heads=2, head_dim=128, act="gelu", lq_range=(1, 300),
                              lkv_range=(1, 300), bias_len=257)
    d = x.to("cuda")
    tq, tkv = x.q.shape[0], x.k.shape[0]
    out = torch.empty_like(d.q)
    dq, dk, dv = torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)
    db = torch.empty((x.heads, x.bias_len), dtype=torch.float32, device="cuda")
    ws_f = torch.empty(jg.jgdpa_workspace_bytes(x.batch, tq, tkv, x.heads, x.head_dim, x.act, x.bias_len, False),
                       dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(jg.jgdpa_workspace_bytes(x.batch, tq, tkv, x.heads, x.head_dim, x.act, x.bias_len, True),
                       dtype=torch.uint8, device="cuda")
    scratch = torch.empty(jg.jgdpa_ds_scratch_bytes(x.q_offsets, x.kv_offsets, x.heads), dtype=torch.uint8,
                          device="cuda")

    def step():
        jg.jgdpa_fwd(d.q, d.k, d.v, d.q_offsets, d.kv_offsets, x.act, x.scale, bias_table=d.bias, out=out,
                     workspace=ws_f)
        jg.jgdpa_bwd(d.q, d.k, d.v, out, None, d.dout, d.q_offsets, d.kv_offsets, x.act, x.scale,
                     bias_table=d.bias, dq=dq, dk=dk, dv=dv, dbias=db, workspace=ws_b, ds_scratch=scratch)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (out, dq, dk, dv, db)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (out, dq, dk, dv, db):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert jg.jgdpa_read_device_status(ws_f) == 0 and jg.jgdpa_read_device_status(ws_b) == 0
    for a, b in zip((out, dq, dk, dv, db), ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("stored", [False, True])
def test_backward_is_bitwise_reproducible_including_dbias(jg, stored):
    """Repeated backward calls give identical bits for dQ, dK, dV and dbias.
    The dbias partial sums are 64-bit fixed-point integers, so their totals do
    not depend on which CTA ran which unit or in which order the warps added
    them (the scheduler's order among equal-cost units is not fixed)."""
    x = workloads.random_case(66, batch=6, heads=3, head_dim=128, act="gelu", lq_range=(1, 900),
                              lkv_range=(1, 900), bias_len=257)
    first = run_bwd(jg, x, stored=stored)
    for _ in range(3):
        again = run_bwd(jg, x, stored=stored)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
