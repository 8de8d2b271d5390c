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

ACT = {"gelu": 0, "silu": 1, "softmax": 2}
STATUS = {
    0: "JGDPA_OK", 1: "JGDPA_ERR_INVALID_ARGUMENT", 2: "JGDPA_ERR_UNSUPPORTED",
    3: "JGDPA_ERR_MISALIGNED", 4: "JGDPA_ERR_WORKSPACE_TOO_SMALL", 5: "JGDPA_ERR_CUDA",
    6: "JGDPA_ERR_BAD_OFFSETS", 7: "JGDPA_ERR_DEVICE_TIMEOUT",
}
EXPORTS = ("jgdpa_workspace_bytes", "jgdpa_fwd", "jgdpa_fwd_ex", "jgdpa_bwd", "jgdpa_bwd_ex",
           "jgdpa_ds_scratch_bytes",
           "jgdpa_read_device_status", "jgdpa_status_string", "jgdpa_eval_activation", "jgdpa_fwd_noalloc")


class JgdpaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libjgdpa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
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
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libjgdpa must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libjgdpa must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != 0:
        raise JgdpaError(rc, where)


def _act(act) -> int:
    return ACT[act] if isinstance(act, str) else int(act)


def jgdpa_status_string(code: int) -> str:
    return load().jgdpa_status_string(int(code)).decode()


def jgdpa_workspace_bytes(batch: int, total_q: int, total_kv: int, heads: int, head_dim: int, act,
                          bias_len: int = 0, for_backward: bool = False) -> int:
    return int(load().jgdpa_workspace_bytes(batch, total_q, total_kv, heads, head_dim, _act(act),
                                            bias_len, int(bool(for_backward))))


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is not None:
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def jgdpa_fwd(q, k, v, q_offsets, kv_offsets, act, scale: float, bias_table=None, causal: bool = False,
              out=None, lse=None, workspace=None, stream=None, window: int = 0):
    """Forward pass; returns (out, lse) with lse None unless act == 'softmax'.
    window > 0 takes the sliding-window entry point (jgdpa_fwd_ex)."""
    lib = load()
    total_q, heads, d = q.shape
    total_kv = k.shape[0]
    batch = q_offsets.numel() - 1
    a = _act(act)
    bias_len = 0 if bias_table is None else int(bias_table.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if lse is None and a == ACT["softmax"]:
        lse = torch.empty((heads, total_q), dtype=torch.float32, device=q.device)
    nbytes = jgdpa_workspace_bytes(batch, total_q, total_kv, heads, d, a, bias_len, False)
    ws = _workspace(nbytes, q.device, workspace)
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(q_offsets), _ptr(kv_offsets), batch, total_q, total_kv, heads, d,
            a, float(scale), _ptr(bias_table), bias_len, int(bool(causal)))
    tail = (_ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    if window:
        rc = lib.jgdpa_fwd_ex(*head, int(window), *tail)
        _check(rc, "jgdpa_fwd_ex")
    else:
        rc = lib.jgdpa_fwd(*head, *tail)
        _check(rc, "jgdpa_fwd")
    return out, lse


def jgdpa_ds_scratch_bytes(q_offsets, kv_offsets, heads: int, window: int = 0) -> int:
    """Stored-dS scratch bytes for these offsets (copied to the host here)."""
    lib = load()
    qo = q_offsets.detach().to("cpu", torch.int32).contiguous()
    ko = kv_offsets.detach().to("cpu", torch.int32).contiguous()
    return int(lib.jgdpa_ds_scratch_bytes(qo.data_ptr(), ko.data_ptr(), qo.numel() - 1, int(heads), int(window)))


def jgdpa_bwd(q, k, v, out, lse, dout, q_offsets, kv_offsets, act, scale: float, bias_table=None,
              causal: bool = False, dq=None, dk=None, dv=None, dbias=None, want_dbias: bool = True,
              workspace=None, stream=None, ds_scratch=None, pass_events=None, window: int = 0):
    """Backward pass; returns (dq, dk, dv, dbias) with dbias None without a bias table.

    ds_scratch: optional uint8 device tensor of at least jgdpa_ds_scratch_bytes
    bytes -- selects the stored-dS backward (jgdpa_bwd_ex).  pass_events:
    optional three torch.cuda.Event (timing enabled, already recorded once),
    recorded before the dK/dV pass, between the passes and after the dQ pass.
    window: the forward's sliding window (jgdpa_bwd_ex); 0 for none."""
    lib = load()
    total_q, heads, d = q.shape
    total_kv = k.shape[0]
    batch = q_offsets.numel() - 1
    a = _act(act)
    bias_len = 0 if bias_table is None else int(bias_table.shape[1])
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dbias is None and bias_len and want_dbias:
        dbias = torch.empty((heads, bias_len), dtype=torch.float32, device=q.device)
    nbytes = jgdpa_workspace_bytes(batch, total_q, total_kv, heads, d, a, bias_len, True)
    ws = _workspace(nbytes, q.device, workspace)
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(q_offsets),
            _ptr(kv_offsets), batch, total_q, total_kv, heads, d, a, float(scale),
            _ptr(bias_table), bias_len, int(bool(causal)))
    tail = (_ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias), _ptr(ws), ws.numel())
    if ds_scratch is None and pass_events is None and not window:
        rc = lib.jgdpa_bwd(*head, *tail, _stream(stream))
        _check(rc, "jgdpa_bwd")
    else:
        ev = None
        if pass_events is not None:
            ev = (ctypes.c_void_p * 3)(*[None if e is None else e.cuda_event for e in pass_events])
        rc = lib.jgdpa_bwd_ex(*head, int(window), *tail, _ptr(ds_scratch),
                              0 if ds_scratch is None else ds_scratch.numel(), _stream(stream), ev)
        _check(rc, "jgdpa_bwd_ex")
    return dq, dk, dv, dbias


def jgdpa_fwd_noalloc(q, k, v, q_offsets, kv_offsets, act, scale: float, bias_table=None,
                      causal: bool = False, out=None, lse=None, stream=None):
    """Forward pass using the library's built-in scratch (no workspace
    argument; for callers that cannot allocate device memory at call time).
    out / lse must be passed by such callers; they are created here only for
    convenience when omitted.  Returns (out, lse)."""
    lib = load()
    total_q, heads, d = q.shape
    a = _act(act)
    bias_len = 0 if bias_table is None else int(bias_table.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if lse is None and a == ACT["softmax"]:
        lse = torch.empty((heads, total_q), dtype=torch.float32, device=q.device)
    rc = lib.jgdpa_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(q_offsets), _ptr(kv_offsets),
                               q_offsets.numel() - 1, total_q, k.shape[0], heads, d, a, float(scale),
                               _ptr(bias_table), bias_len, int(bool(causal)), _ptr(out), _ptr(lse),
                               _stream(stream))
    _check(rc, "jgdpa_fwd_noalloc")
    return out, lse


def jgdpa_read_device_status(workspace, stream=None) -> int:
    return int(load().jgdpa_read_device_status(_ptr(workspace), _stream(stream)))


def jgdpa_eval_activation(act, x, path: int = 0, stream=None):
    """Device act(x), act'(x) for fp32 x (test hook); path 0 = SFU route, 1 = ALU route."""
    y = torch.empty_like(x)
    dy = torch.empty_like(x)
    rc = load().jgdpa_eval_activation(_act(act), int(path), _ptr(x), x.numel(), _ptr(y), _ptr(dy),
                                      _stream(stream))
    _check(rc, "jgdpa_eval_activation")
    return y, dy
