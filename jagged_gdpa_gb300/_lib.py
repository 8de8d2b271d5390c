"""ctypes binding of libjgdpa.so (include/jgdpa.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Tensors are torch tensors on the current CUDA device;
torch supplies device memory and the stream.  If the library is missing the
import fails loudly -- there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libjgdpa.so")
# the same library with GELU/SiLU on the ALU-only polynomial route everywhere
ALU_LIB_PATH = os.path.join(_HERE, "_build", "alu", "libjgdpa.so")

ACT = {"gelu": 0, "silu": 1, "softmax": 2}
STATUS = {
    0: "JGDPA_OK", 1: "JGDPA_ERR_INVALID_ARGUMENT", 2: "JGDPA_ERR_UNSUPPORTED",
    3: "JGDPA_ERR_MISALIGNED", 4: "JGDPA_ERR_WORKSPACE_TOO_SMALL", 5: "JGDPA_ERR_CUDA",
    6: "JGDPA_ERR_BAD_OFFSETS", 7: "JGDPA_ERR_DEVICE_TIMEOUT",
}
EXPORTS = ("jgdpa_workspace_bytes", "jgdpa_fwd", "jgdpa_fwd_ex", "jgdpa_bwd", "jgdpa_bwd_ex",
           "jgdpa_ds_scratch_bytes",
           "jgdpa_read_device_status", "jgdpa_status_string", "jgdpa_eval_activation", "jgdpa_fwd_noalloc",
           "jgdpa_set_wait_limit_ns", "jgdpa_shared_q_workspace_bytes", "jgdpa_fwd_shared_q", "jgdpa_bwd_shared_q")


class JgdpaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


_libs: dict = {}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libjgdpa.so (raises if it has not been built).  Each path is
    loaded once; the wrappers below take ``lib=`` to use another build."""
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with jagged_gdpa_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.jgdpa_workspace_bytes.argtypes = [i32, i64, i64, i32, i32, ctypes.c_int, i32, i32]
    lib.jgdpa_workspace_bytes.restype = sz
    lib.jgdpa_fwd.argtypes = [P, P, P, P, P, i32, i64, i64, i32, i32, ctypes.c_int, f32, P, i32, i32,
                              P, P, P, sz, P]
    lib.jgdpa_fwd.restype = ctypes.c_int
    lib.jgdpa_fwd_ex.argtypes = lib.jgdpa_fwd.argtypes[:15] + [i32] + lib.jgdpa_fwd.argtypes[15:]
    lib.jgdpa_fwd_ex.restype = ctypes.c_int
    lib.jgdpa_bwd.argtypes = [P, P, P, P, P, P, P, P, i32, i64, i64, i32, i32, ctypes.c_int, f32, P, i32,
                              i32, P, P, P, P, P, sz, P]
    lib.jgdpa_bwd.restype = ctypes.c_int
    lib.jgdpa_bwd_ex.argtypes = (lib.jgdpa_bwd.argtypes[:18] + [i32] + lib.jgdpa_bwd.argtypes[18:-1]
                                 + [P, sz, P, P])
    lib.jgdpa_bwd_ex.restype = ctypes.c_int
    lib.jgdpa_ds_scratch_bytes.argtypes = [P, P, i32, i32, i32]
    lib.jgdpa_ds_scratch_bytes.restype = sz
    lib.jgdpa_read_device_status.argtypes = [P, P]
    lib.jgdpa_read_device_status.restype = ctypes.c_int
    lib.jgdpa_status_string.argtypes = [ctypes.c_int]
    lib.jgdpa_status_string.restype = ctypes.c_char_p
    lib.jgdpa_eval_activation.argtypes = [ctypes.c_int, i32, P, i64, P, P, P]
    lib.jgdpa_eval_activation.restype = ctypes.c_int
    lib.jgdpa_fwd_noalloc.argtypes = [P, P, P, P, P, i32, i64, i64, i32, i32, ctypes.c_int, f32, P, i32, i32,
                                      P, P, P]
    lib.jgdpa_fwd_noalloc.restype = ctypes.c_int
    lib.jgdpa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.jgdpa_set_wait_limit_ns.restype = None
    lib.jgdpa_shared_q_workspace_bytes.argtypes = [i32, i32, i64, i32, i32, ctypes.c_int, i32, i32]
    lib.jgdpa_shared_q_workspace_bytes.restype = sz
    lib.jgdpa_fwd_shared_q.argtypes = [P, i32, P, P, P, i32, i64, i32, i32, ctypes.c_int, f32, P, i32, i32, i32,
                                       P, P, P, sz, P]
    lib.jgdpa_fwd_shared_q.restype = ctypes.c_int
    lib.jgdpa_bwd_shared_q.argtypes = [P, i32, P, P, P, P, P, P, i32, i64, i32, i32, ctypes.c_int, f32, P, i32,
                                       i32, i32, P, P, P, P, P, sz, P, sz, P, P]
    lib.jgdpa_bwd_shared_q.restype = ctypes.c_int
    _libs[path] = lib
    return lib


def _check(t, name: str, dtype, shape, device=None, optional: bool = False):
    """Raise ValueError unless t is a tensor of this dtype and shape (None
    entries of shape match any size) on `device`.  Run before any pointer is
    taken: the library builds its TMA maps from the shapes it is given, so a
    short tensor would be read past its end."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if t.dim() != len(shape) or any(w is not None and g != w for g, w in zip(t.shape, shape)):
        want = "[" + ", ".join("*" if w is None else str(w) for w in shape) + "]"
        raise ValueError(f"{name} must have shape {want}, got {list(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _check_common(q, k, v, q_offsets, kv_offsets, bias_table):
    """Shapes and dtypes shared by the forward and backward wrappers; returns
    (total_q, heads, head_dim, total_kv, batch, bias_len)."""
    if not isinstance(q, torch.Tensor) or q.dim() != 3:
        raise ValueError("q must be a bf16 tensor [total_q, heads, head_dim]")
    total_q, heads, d = q.shape
    _check(q, "q", torch.bfloat16, (None, None, None))
    _check(k, "k", torch.bfloat16, (None, heads, d), q.device)
    total_kv = k.shape[0]
    _check(v, "v", torch.bfloat16, (total_kv, heads, d), q.device)
    _check(q_offsets, "q_offsets", torch.int32, (None,), q.device)
    batch = q_offsets.numel() - 1
    if batch < 0:
        raise ValueError("q_offsets must hold batch + 1 >= 1 entries")
    _check(kv_offsets, "kv_offsets", torch.int32, (batch + 1,), q.device)
    _check(bias_table, "bias_table", torch.float32, (heads, None), q.device, optional=True)
    bias_len = 0 if bias_table is None else int(bias_table.shape[1])
    return total_q, heads, d, total_kv, batch, bias_len


def _check_bytes(t, name: str, device):
    if t is None:
        return
    _check(t, name, torch.uint8, (None,), device)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libjgdpa must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libjgdpa must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _events(pass_events):
    """Three torch.cuda.Event (or None) as a C array of cudaEvent_t, or None."""
    if pass_events is None:
        return None
    return (ctypes.c_void_p * 3)(*[None if e is None else e.cuda_event for e in pass_events])


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _rc(rc: int, where: str):
    if rc != 0:
        raise JgdpaError(rc, where)


def _act(act) -> int:
    return ACT[act] if isinstance(act, str) else int(act)


def jgdpa_status_string(code: int, lib=None) -> str:
    return (lib or load()).jgdpa_status_string(int(code)).decode()


def jgdpa_workspace_bytes(batch: int, total_q: int, total_kv: int, heads: int, head_dim: int, act,
                          bias_len: int = 0, for_backward: bool = False, lib=None) -> int:
    return int((lib or load()).jgdpa_workspace_bytes(batch, total_q, total_kv, heads, head_dim, _act(act),
                                                     bias_len, int(bool(for_backward))))


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is not None:
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def jgdpa_fwd(q, k, v, q_offsets, kv_offsets, act, scale: float, bias_table=None, causal: bool = False,
              out=None, lse=None, workspace=None, stream=None, window: int = 0, lib=None):
    """Forward pass; returns (out, lse) with lse None unless act == 'softmax'.
    window > 0 takes the sliding-window entry point (jgdpa_fwd_ex).  Shapes
    and dtypes are checked here (ValueError) before the library sees any
    pointer."""
    lib = lib or load()
    total_q, heads, d, total_kv, batch, bias_len = _check_common(q, k, v, q_offsets, kv_offsets, bias_table)
    a = _act(act)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and a == ACT["softmax"]:
        lse = torch.empty((heads, total_q), dtype=torch.float32, device=q.device)
    _check(out, "out", torch.bfloat16, (total_q, heads, d), q.device)
    if a == ACT["softmax"]:
        _check(lse, "lse", torch.float32, (heads, total_q), q.device)
    elif lse is not None:
        raise ValueError("lse is written in softmax mode only; pass None")
    _check_bytes(workspace, "workspace", q.device)
    nbytes = jgdpa_workspace_bytes(batch, total_q, total_kv, heads, d, a, bias_len, False, lib=lib)
    ws = _workspace(nbytes, q.device, workspace)
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(q_offsets), _ptr(kv_offsets), batch, total_q, total_kv, heads, d,
            a, float(scale), _ptr(bias_table), bias_len, int(bool(causal)))
    tail = (_ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    if window:
        rc = lib.jgdpa_fwd_ex(*head, int(window), *tail)
        _rc(rc, "jgdpa_fwd_ex")
    else:
        rc = lib.jgdpa_fwd(*head, *tail)
        _rc(rc, "jgdpa_fwd")
    return out, lse


def jgdpa_ds_scratch_bytes(q_offsets, kv_offsets, heads: int, window: int = 0, lib=None) -> int:
    """Stored-dS scratch bytes for these offsets (copied to the host here)."""
    lib = lib or load()
    qo = q_offsets.detach().to("cpu", torch.int32).contiguous()
    ko = kv_offsets.detach().to("cpu", torch.int32).contiguous()
    return int(lib.jgdpa_ds_scratch_bytes(qo.data_ptr(), ko.data_ptr(), qo.numel() - 1, int(heads), int(window)))


def jgdpa_bwd(q, k, v, out, lse, dout, q_offsets, kv_offsets, act, scale: float, bias_table=None,
              causal: bool = False, dq=None, dk=None, dv=None, dbias=None, want_dbias: bool = True,
              workspace=None, stream=None, ds_scratch=None, pass_events=None, window: int = 0, lib=None):
    """Backward pass; returns (dq, dk, dv, dbias) with dbias None without a bias table.

    ds_scratch: optional uint8 device tensor of at least jgdpa_ds_scratch_bytes
    bytes -- selects the stored-dS backward (jgdpa_bwd_ex).  pass_events:
    optional three torch.cuda.Event (timing enabled, already recorded once),
    recorded before the dK/dV pass, between the passes and after the dQ pass.
    window: the forward's sliding window (jgdpa_bwd_ex); 0 for none.  Shapes
    and dtypes are checked here (ValueError) before the library sees any
    pointer."""
    lib = lib or load()
    total_q, heads, d, total_kv, batch, bias_len = _check_common(q, k, v, q_offsets, kv_offsets, bias_table)
    a = _act(act)
    _check(dout, "dout", torch.bfloat16, (total_q, heads, d), q.device)
    if a == ACT["softmax"]:
        _check(out, "out", torch.bfloat16, (total_q, heads, d), q.device)
        _check(lse, "lse", torch.float32, (heads, total_q), q.device)
    else:
        _check(out, "out", torch.bfloat16, (total_q, heads, d), q.device, optional=True)
        _check(lse, "lse", torch.float32, (heads, total_q), q.device, optional=True)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dbias is None and bias_len and want_dbias:
        dbias = torch.empty((heads, bias_len), dtype=torch.float32, device=q.device)
    _check(dq, "dq", torch.bfloat16, (total_q, heads, d), q.device)
    _check(dk, "dk", torch.bfloat16, (total_kv, heads, d), q.device)
    _check(dv, "dv", torch.bfloat16, (total_kv, heads, d), q.device)
    if dbias is not None:
        if not bias_len:
            raise ValueError("dbias needs a bias table")
        _check(dbias, "dbias", torch.float32, (heads, bias_len), q.device)
    _check_bytes(workspace, "workspace", q.device)
    _check_bytes(ds_scratch, "ds_scratch", q.device)
    nbytes = jgdpa_workspace_bytes(batch, total_q, total_kv, heads, d, a, bias_len, True, lib=lib)
    ws = _workspace(nbytes, q.device, workspace)
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(q_offsets),
            _ptr(kv_offsets), batch, total_q, total_kv, heads, d, a, float(scale),
            _ptr(bias_table), bias_len, int(bool(causal)))
    tail = (_ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias), _ptr(ws), ws.numel())
    if ds_scratch is None and pass_events is None and not window:
        rc = lib.jgdpa_bwd(*head, *tail, _stream(stream))
        _rc(rc, "jgdpa_bwd")
    else:
        rc = lib.jgdpa_bwd_ex(*head, int(window), *tail, _ptr(ds_scratch),
                              0 if ds_scratch is None else ds_scratch.numel(), _stream(stream),
                              _events(pass_events))
        _rc(rc, "jgdpa_bwd_ex")
    return dq, dk, dv, dbias


def jgdpa_fwd_noalloc(q, k, v, q_offsets, kv_offsets, act, scale: float, bias_table=None,
                      causal: bool = False, out=None, lse=None, stream=None, lib=None):
    """Forward pass using the library's built-in scratch (no workspace
    argument; for callers that cannot allocate device memory at call time).
    out / lse must be passed by such callers; they are created here only for
    convenience when omitted.  Returns (out, lse)."""
    lib = lib or load()
    total_q, heads, d, total_kv, batch, bias_len = _check_common(q, k, v, q_offsets, kv_offsets, bias_table)
    a = _act(act)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and a == ACT["softmax"]:
        lse = torch.empty((heads, total_q), dtype=torch.float32, device=q.device)
    _check(out, "out", torch.bfloat16, (total_q, heads, d), q.device)
    if a == ACT["softmax"]:
        _check(lse, "lse", torch.float32, (heads, total_q), q.device)
    rc = lib.jgdpa_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(q_offsets), _ptr(kv_offsets),
                               q_offsets.numel() - 1, total_q, k.shape[0], heads, d, a, float(scale),
                               _ptr(bias_table), bias_len, int(bool(causal)), _ptr(out), _ptr(lse),
                               _stream(stream))
    _rc(rc, "jgdpa_fwd_noalloc")
    return out, lse


def jgdpa_read_device_status(workspace, stream=None, lib=None) -> int:
    return int((lib or load()).jgdpa_read_device_status(_ptr(workspace), _stream(stream)))


def jgdpa_eval_activation(act, x, path: int = 0, stream=None, lib=None):
    """Device act(x), act'(x) for fp32 x (test hook); path 0 = SFU route, 1 = ALU route."""
    _check(x, "x", torch.float32, (None,))
    y = torch.empty_like(x)
    dy = torch.empty_like(x)
    rc = (lib or load()).jgdpa_eval_activation(_act(act), int(path), _ptr(x), x.numel(), _ptr(y), _ptr(dy),
                                      _stream(stream))
    _rc(rc, "jgdpa_eval_activation")
    return y, dy


def jgdpa_set_wait_limit_ns(limit_ns: int, lib=None) -> None:
    """Test hook: limit of one internal device wait for later launches (0 =
    the default of 2 s)."""
    (lib or load()).jgdpa_set_wait_limit_ns(int(limit_ns))


# ------------------------------------------------------------ shared queries
def jgdpa_shared_q_workspace_bytes(batch: int, n_shared: int, total_kv: int, heads: int, head_dim: int, act,
                                   bias_len: int = 0, for_backward: bool = False, lib=None) -> int:
    return int((lib or load()).jgdpa_shared_q_workspace_bytes(batch, n_shared, total_kv, heads, head_dim,
                                                              _act(act), bias_len, int(bool(for_backward))))


def _check_shared(q, k, v, kv_offsets, bias_table):
    if not isinstance(q, torch.Tensor) or q.dim() != 3:
        raise ValueError("q must be a bf16 tensor [n_shared, heads, head_dim]")
    n_shared, heads, d = q.shape
    _check(q, "q", torch.bfloat16, (None, None, None))
    _check(k, "k", torch.bfloat16, (None, heads, d), q.device)
    total_kv = k.shape[0]
    _check(v, "v", torch.bfloat16, (total_kv, heads, d), q.device)
    _check(kv_offsets, "kv_offsets", torch.int32, (None,), q.device)
    batch = kv_offsets.numel() - 1
    if batch < 0:
        raise ValueError("kv_offsets must hold batch + 1 >= 1 entries")
    _check(bias_table, "bias_table", torch.float32, (heads, None), q.device, optional=True)
    bias_len = 0 if bias_table is None else int(bias_table.shape[1])
    return n_shared, heads, d, total_kv, batch, bias_len


def jgdpa_fwd_shared_q(q, k, v, kv_offsets, act, scale: float, bias_table=None, causal: bool = False,
                       out=None, lse=None, workspace=None, stream=None, window: int = 0, lib=None):
    """Forward with query rows shared by every segment: q is [S, H, d]; out is
    [batch S, H, d] (segment b's rows b S .. b S + S - 1); returns (out, lse)."""
    lib = lib or load()
    n_shared, heads, d, total_kv, batch, bias_len = _check_shared(q, k, v, kv_offsets, bias_table)
    a = _act(act)
    total_q = batch * n_shared
    if out is None:
        out = torch.empty((total_q, heads, d), dtype=q.dtype, device=q.device)
    if lse is None and a == ACT["softmax"]:
        lse = torch.empty((heads, total_q), dtype=torch.float32, device=q.device)
    _check(out, "out", torch.bfloat16, (total_q, heads, d), q.device)
    if a == ACT["softmax"]:
        _check(lse, "lse", torch.float32, (heads, total_q), q.device)
    elif lse is not None:
        raise ValueError("lse is written in softmax mode only; pass None")
    _check_bytes(workspace, "workspace", q.device)
    nbytes = jgdpa_shared_q_workspace_bytes(batch, n_shared, total_kv, heads, d, a, bias_len, False, lib=lib)
    ws = _workspace(nbytes, q.device, workspace)
    rc = lib.jgdpa_fwd_shared_q(_ptr(q), n_shared, _ptr(k), _ptr(v), _ptr(kv_offsets), batch, total_kv, heads, d,
                                a, float(scale), _ptr(bias_table), bias_len, int(bool(causal)), int(window),
                                _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _rc(rc, "jgdpa_fwd_shared_q")
    return out, lse


def jgdpa_bwd_shared_q(q, k, v, out, lse, dout, kv_offsets, act, scale: float, bias_table=None,
                       causal: bool = False, dq=None, dk=None, dv=None, dbias=None, want_dbias: bool = True,
                       workspace=None, stream=None, ds_scratch=None, window: int = 0, pass_events=None,
                       lib=None):
    """Backward with shared query rows; dq [S, H, d] is the sum over segments.
    pass_events as in jgdpa_bwd.  Returns (dq, dk, dv, dbias)."""
    lib = lib or load()
    n_shared, heads, d, total_kv, batch, bias_len = _check_shared(q, k, v, kv_offsets, bias_table)
    a = _act(act)
    total_q = batch * n_shared
    _check(dout, "dout", torch.bfloat16, (total_q, heads, d), q.device)
    opt = a != ACT["softmax"]
    _check(out, "out", torch.bfloat16, (total_q, heads, d), q.device, optional=opt)
    _check(lse, "lse", torch.float32, (heads, total_q), q.device, optional=opt)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dbias is None and bias_len and want_dbias:
        dbias = torch.empty((heads, bias_len), dtype=torch.float32, device=q.device)
    _check(dq, "dq", torch.bfloat16, (n_shared, heads, d), q.device)
    _check(dk, "dk", torch.bfloat16, (total_kv, heads, d), q.device)
    _check(dv, "dv", torch.bfloat16, (total_kv, heads, d), q.device)
    if dbias is not None:
        if not bias_len:
            raise ValueError("dbias needs a bias table")
        _check(dbias, "dbias", torch.float32, (heads, bias_len), q.device)
    _check_bytes(workspace, "workspace", q.device)
    _check_bytes(ds_scratch, "ds_scratch", q.device)
    nbytes = jgdpa_shared_q_workspace_bytes(batch, n_shared, total_kv, heads, d, a, bias_len, True, lib=lib)
    ws = _workspace(nbytes, q.device, workspace)
    rc = lib.jgdpa_bwd_shared_q(_ptr(q), n_shared, _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                _ptr(kv_offsets), batch, total_kv, heads, d, a, float(scale), _ptr(bias_table),
                                bias_len, int(bool(causal)), int(window), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(dbias), _ptr(ws), ws.numel(), _ptr(ds_scratch),
                                0 if ds_scratch is None else ds_scratch.numel(), _stream(stream),
                                _events(pass_events))
    _rc(rc, "jgdpa_bwd_shared_q")
    return dq, dk, dv, dbias
