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


# ---------------------------------------------------------------- binding checks
# The Python wrappers check dtypes and shapes before any pointer reaches the
# library (the library builds V's tensor map from K's row count and dO's from
# Q's, so a short tensor would be read past its end).  These run on the CPU:
# the checks come before the device check.

def _bundle(tq=10, tkv=7, h=2, d=64, bias=5):
    import torch
    return dict(q=torch.zeros(tq, h, d, dtype=torch.bfloat16), k=torch.zeros(tkv, h, d, dtype=torch.bfloat16),
                v=torch.zeros(tkv, h, d, dtype=torch.bfloat16), q_offsets=torch.tensor([0, tq], dtype=torch.int32),
                kv_offsets=torch.tensor([0, tkv], dtype=torch.int32),
                bias_table=torch.zeros(h, bias, dtype=torch.float32) if bias else None)


@pytest.mark.parametrize("field,bad,match", [
    ("q", "float32", "q must have dtype"),
    ("k", "float16", "k must have dtype"),
    ("v", "short", "v must have shape"),
    ("k", "heads", "k must have shape"),
    ("q_offsets", "int64", "q_offsets must have dtype"),
    ("kv_offsets", "long", "kv_offsets must have shape"),
    ("bias_table", "float64", "bias_table must have dtype"),
    ("bias_table", "heads", "bias_table must have shape"),
])
def test_forward_wrapper_rejects_bad_tensors(lib, field, bad, match):
    import torch
    import jagged_gdpa_gb300 as jg
    b = _bundle()
    t = b[field]
    if bad in ("float32", "float16", "int64", "float64"):
        b[field] = t.to(getattr(torch, bad))
    elif bad == "short":
        b[field] = t[:-1]
    elif bad == "heads":  # one head too many: dimension 1 of [rows, H, d], dimension 0 of [H, T]
        shape = list(t.shape)
        shape[1 if t.dim() == 3 else 0] += 1
        b[field] = torch.zeros(shape, dtype=t.dtype)
    elif bad == "long":
        b[field] = torch.zeros(t.numel() + 1, dtype=t.dtype)
    with pytest.raises(ValueError, match=match):
        jg.jgdpa_fwd(b["q"], b["k"], b["v"], b["q_offsets"], b["kv_offsets"], "gelu", 0.125,
                     bias_table=b["bias_table"])


def test_forward_wrapper_rejects_bad_outputs(lib):
    import torch
    import jagged_gdpa_gb300 as jg
    b = _bundle()
    args = (b["q"], b["k"], b["v"], b["q_offsets"], b["kv_offsets"])
    with pytest.raises(ValueError, match="out must have shape"):
        jg.jgdpa_fwd(*args, "gelu", 0.125, out=torch.zeros(9, 2, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out must have dtype"):
        jg.jgdpa_fwd(*args, "gelu", 0.125, out=torch.zeros(10, 2, 64, dtype=torch.float32))
    with pytest.raises(ValueError, match="lse must have shape"):
        jg.jgdpa_fwd(*args, "softmax", 0.125, lse=torch.zeros(2, 9, dtype=torch.float32))
    with pytest.raises(ValueError, match="lse is written in softmax mode only"):
        jg.jgdpa_fwd(*args, "gelu", 0.125, lse=torch.zeros(2, 10, dtype=torch.float32))
    with pytest.raises(ValueError, match="workspace must have dtype"):
        jg.jgdpa_fwd(*args, "gelu", 0.125, workspace=torch.zeros(1024, dtype=torch.float32))
    # everything valid: the wrapper gets as far as the device check
    with pytest.raises(ValueError, match="CUDA device"):
        jg.jgdpa_fwd(*args, "gelu", 0.125, bias_table=b["bias_table"])


@pytest.mark.parametrize("field,shape,dtype,match", [
    ("dout", (9, 2, 64), "bfloat16", "dout must have shape"),
    ("dq", (10, 2, 64), "float32", "dq must have dtype"),
    ("dk", (6, 2, 64), "bfloat16", "dk must have shape"),
    ("dv", (7, 2, 32), "bfloat16", "dv must have shape"),
    ("dbias", (2, 4), "float32", "dbias must have shape"),
    ("lse", (2, 11), "float32", "lse must have shape"),
    ("out", (10, 2, 64), "float16", "out must have dtype"),
    ("ds_scratch", (64,), "int32", "ds_scratch must have dtype"),
])
def test_backward_wrapper_rejects_bad_tensors(lib, field, shape, dtype, match):
    import torch
    import jagged_gdpa_gb300 as jg
    b = _bundle()
    kw = dict(dq=None, dk=None, dv=None, dbias=None, ds_scratch=None)
    out = torch.zeros(10, 2, 64, dtype=torch.bfloat16)
    lse = torch.zeros(2, 10, dtype=torch.float32)
    dout = torch.zeros(10, 2, 64, dtype=torch.bfloat16)
    bad = torch.zeros(shape, dtype=getattr(torch, dtype))
    if field == "dout":
        dout = bad
    elif field == "lse":
        lse = bad
    elif field == "out":
        out = bad
    else:
        kw[field] = bad
    with pytest.raises(ValueError, match=match):
        jg.jgdpa_bwd(b["q"], b["k"], b["v"], out, lse, dout, b["q_offsets"], b["kv_offsets"], "softmax", 0.125,
                     bias_table=b["bias_table"], **kw)


def test_backward_wrapper_rejects_dbias_without_a_table(lib):
    import torch
    import jagged_gdpa_gb300 as jg
    b = _bundle(bias=0)
    with pytest.raises(ValueError, match="dbias needs a bias table"):
        jg.jgdpa_bwd(b["q"], b["k"], b["v"], None, None, torch.zeros(10, 2, 64, dtype=torch.bfloat16),
                     b["q_offsets"], b["kv_offsets"], "gelu", 0.125, dbias=torch.zeros(2, 5))


def test_alu_route_library_is_built_and_exports_the_same_symbols(lib):
    import jagged_gdpa_gb300 as jg
    alu = jg.load(jg.ALU_LIB_PATH)
    assert alu is not lib
    for n in declared_functions():
        assert hasattr(alu, n), n
