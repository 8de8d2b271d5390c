"""The C ABI: the library loads, exports every declared entry point, and the
host-side checks reject bad arguments before touching the GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "jgdpa.h")


@pytest.fixture(scope="module")
def lib():
    from jagged_gdpa_gb300 import build as b
    b.build()
    import jagged_gdpa_gb300 as jg
    return jg.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"JGDPA_API\s+[\w\s\*]+?\b(jgdpa_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("jgdpa_fwd", "jgdpa_bwd", "jgdpa_workspace_bytes", "jgdpa_read_device_status",
              "jgdpa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    import jagged_gdpa_gb300 as jg
    assert set(jg.EXPORTS) >= set(declared_functions())


def test_status_strings(lib):
    import jagged_gdpa_gb300 as jg
    assert jg.jgdpa_status_string(0) == "ok"
    assert "offsets" in jg.jgdpa_status_string(6)
    assert jg.jgdpa_status_string(99) == "unknown status"


def _fwd_args(**kw):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, qo=1 << 20, ko=1 << 20, batch=1, tq=4, tkv=4, heads=1,
             d=64, act=0, scale=0.125, bias=None, blen=0, causal=0, out=1 << 20, lse=None, ws=1 << 20,
             wsb=1 << 30, stream=None)
    a.update(kw)
    return [a["q"], a["k"], a["v"], a["qo"], a["ko"], a["batch"], a["tq"], a["tkv"], a["heads"], a["d"],
            a["act"], ctypes.c_float(a["scale"]), a["bias"], a["blen"], a["causal"], a["out"], a["lse"],
            a["ws"], a["wsb"], a["stream"]]


@pytest.mark.parametrize("kw,code", [
    (dict(d=48), 2),                    # head_dim not supported
    (dict(d=256), 2),
    (dict(act=3), 1),                   # bad enum
    (dict(blen=4, bias=1 << 20), 1),    # even bias table
    (dict(blen=5, bias=None), 1),       # table length without a table
    (dict(causal=2), 1),
    (dict(heads=0), 1),
    (dict(batch=-1), 1),
    (dict(qo=None), 1),                 # null offsets
    (dict(act=2, lse=None), 1),         # softmax needs lse
    (dict(act=0, lse=1 << 20), 1),      # lse only in softmax mode
    (dict(scale=float("nan")), 1),
    (dict(blen=8191, bias=1 << 20), 2), # table too long
])
def test_fwd_rejects_bad_arguments_without_a_launch(lib, kw, code):
    # fake (never dereferenced) device addresses: every case fails host validation
    assert lib.jgdpa_fwd(*_fwd_args(**kw)) == code


def test_workspace_query_rejects_invalid_sizes(lib):
    import jagged_gdpa_gb300 as jg
    assert jg.jgdpa_workspace_bytes(1, 4, 4, 1, 48, "gelu") == 0
    assert jg.jgdpa_workspace_bytes(-1, 4, 4, 1, 64, "gelu") == 0


@pytest.mark.parametrize("window,code", [(-1, 1), (-1000, 1)])
def test_fwd_ex_rejects_a_negative_window_without_a_launch(lib, window, code):
    args = _fwd_args()
    args.insert(15, window)  # after causal
    assert lib.jgdpa_fwd_ex(*args) == code
    # a valid window still meets the other checks first: bad head_dim
    args = _fwd_args(d=48)
    args.insert(15, 5)
    assert lib.jgdpa_fwd_ex(*args) == 2


def test_ds_scratch_size_follows_the_band(lib):
    """Stored-dS scratch: heads * sum_b nk_b * span_b tiles of 32 KB, span = nq
    without a window, else min(nq, 2e + 1) with e = ceil((w - 1) / 128)."""
    import numpy as np
    import torch
    import jagged_gdpa_gb300 as jg
    import workloads
    rng = np.random.default_rng(3)
    lq = rng.integers(0, 3000, size=9)
    lkv = rng.integers(0, 3000, size=9)
    qo, ko = workloads.offsets_from_lengths(lq), workloads.offsets_from_lengths(lkv)
    for heads in (1, 3):
        for w in (0, 1, 2, 128, 129, 300, 1000, 5000):
            nq, nk = -(-lq // 128), -(-lkv // 128)
            e = -(-(w - 1) // 128) if w > 0 else 0
            span = nq if w == 0 else np.minimum(nq, 2 * e + 1)
            want = int(heads * np.sum(nk * span)) * 32768
            assert jg.jgdpa_ds_scratch_bytes(qo, ko, heads, w) == want, (heads, w)
    assert jg.jgdpa_ds_scratch_bytes(qo, ko, 1, -1) == 0
    # the band never holds more than the unwindowed scratch
    assert jg.jgdpa_ds_scratch_bytes(qo, ko, 2, 300) <= jg.jgdpa_ds_scratch_bytes(qo, ko, 2, 0)
