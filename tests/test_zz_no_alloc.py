"""jgdpa_fwd_noalloc: the forward entry point for callers that cannot allocate
device memory at call time (it takes no workspace and uses a fixed array
compiled into the library).

Called through the C ABI (ctypes, raw device pointers) and compared with the
regular jgdpa_fwd on the same inputs, within the parity tolerance, on two
calls in a row with different shapes -- the second call runs on scratch that
still holds the first call's contents.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""

import ctypes

import pytest
import torch

import workloads
from tests._util import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jg():
    import __graft_entry__
    __graft_entry__.build()
    import jagged_gdpa_gb300 as m
    return m


def _noalloc_c(lib, d, x, out, lse):
    P = ctypes.c_void_p
    total_q, heads, hd = d.q.shape
    rc = lib.jgdpa_fwd_noalloc(
        P(d.q.data_ptr()), P(d.k.data_ptr()), P(d.v.data_ptr()), P(d.q_offsets.data_ptr()),
        P(d.kv_offsets.data_ptr()), x.batch, total_q, d.k.shape[0], heads, hd,
        {"gelu": 0, "silu": 1, "softmax": 2}[x.act], ctypes.c_float(x.scale),
        None if d.bias is None else P(d.bias.data_ptr()), x.bias_len, int(x.causal),
        P(out.data_ptr()), None if lse is None else P(lse.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))
    return rc


CASES = [
    # (seed, batch, heads, d, act, lq, lkv, causal, bias_len)
    (11, 5, 2, 128, "gelu", (1, 600), (1, 400), False, 257),
    (12, 9, 3, 64, "softmax", (1, 300), (1, 300), True, 0),
]


def test_noalloc_matches_fwd_on_two_calls_in_a_row(jg):
    lib = jg.load()
    for seed, b, h, d, act, lqr, lkvr, causal, bl in CASES:
        x = workloads.random_case(seed, batch=b, heads=h, head_dim=d, act=act, lq_range=lqr,
                                  lkv_range=lkvr, causal=causal, bias_len=bl)
        dx = x.to("cuda")
        ref, ref_lse = jg.jgdpa_fwd(dx.q, dx.k, dx.v, dx.q_offsets, dx.kv_offsets, x.act, x.scale,
                                    bias_table=dx.bias, causal=x.causal)
        out = torch.full_like(dx.q, float("nan"))
        lse = None if act != "softmax" else torch.full_like(ref_lse, float("nan"))
        assert _noalloc_c(lib, dx, x, out, lse) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert rel_err(out, ref.double().cpu().numpy()) <= TOL
        if lse is not None:
            fin = torch.isfinite(ref_lse)
            assert torch.equal(torch.isfinite(lse), fin)
            assert rel_err(lse[fin], ref_lse[fin].double().cpu().numpy()) <= TOL


def test_noalloc_rejects_sizes_beyond_its_scratch(jg):
    lib = jg.load()
    # batch of 600,000 one-token segments needs more unit entries than 4 MiB hold;
    # the call must fail on the host before any pointer is used
    P = ctypes.c_void_p
    fake = P(1 << 20)
    rc = lib.jgdpa_fwd_noalloc(fake, fake, fake, fake, fake, 600000, 600000, 600000, 1, 64, 0,
                               ctypes.c_float(0.125), None, 0, 0, fake, None,
                               P(torch.cuda.current_stream().cuda_stream))
    assert rc == 4  # JGDPA_ERR_WORKSPACE_TOO_SMALL
