"""Python wrapper of the fp64 CPU oracle for jagged GDPA.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The library path never imports it.

The oracle is plain C (``oracle.c``), compiled here with gcc into
``oracle/_build/liboracle.so``.  It takes the bf16 inputs decoded exactly to
float64 and returns float64 outputs.  Definitions and the readings of the
pages are in the header comment of ``oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")

ACT_CODE = {"gelu": 0, "silu": 1, "softmax": 2, "identity": 3}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, OpenMP, no fast-math) into _build/."""
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-fopenmp",
                    "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_fwd.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, P, i32, i32, i32, i32,
                                   P, i32, i32, P, P]
        lib.oracle_fwd.restype = ctypes.c_int
        lib.oracle_bwd.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, f64, P, i32, i32, i32, i32,
                                   P, i32, i32, P, P, P, P]
        lib.oracle_bwd.restype = ctypes.c_int
        lib.oracle_bwd_rows.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, f64, P, i32, i32, i32,
                                        i32, i32, P, i32, P, i32, i32, P, P, P]
        lib.oracle_bwd_rows.restype = ctypes.c_int
        lib.oracle_act_eval.argtypes = [i32, P, i64, P, P]
        lib.oracle_act_eval.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu").to(torch.float64).numpy()
    return np.ascontiguousarray(t, dtype=np.float64)


def _i32(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu").numpy()
    return np.ascontiguousarray(t, dtype=np.int32)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def act(name: str, x) -> tuple[np.ndarray, np.ndarray]:
    """act(x) and act'(x) in fp64 for 'gelu', 'silu' or 'identity'."""
    x = _f64(x).ravel()
    y = np.empty_like(x)
    dy = np.empty_like(x)
    if _load().oracle_act_eval(ACT_CODE[name], _ptr(x), x.size, _ptr(y), _ptr(dy)):
        raise ValueError(f"oracle has no element-wise activation {name!r}")
    return y, dy


def _units(units: Optional[Sequence[int]]):
    if units is None:
        return None, 0
    u = np.ascontiguousarray(units, dtype=np.int32)
    return u, int(u.size)


def fwd(q, k, v, q_offsets, kv_offsets, heads: int, head_dim: int, act: str, scale: float,
        bias=None, causal: bool = False, units: Optional[Sequence[int]] = None,
        threads: int = 0, window: int = 0, q_shared: int = 0):
    """O (float64 [total_q, H, d]) and LSE (float64 [H, total_q]).

    ``window`` > 0 keeps only the pairs with |i - j| < window (segment-local).
    ``q_shared`` = S > 0: q is [S, H, d], read by every segment as its query
    rows (each segment has Lq = S; q_offsets still place O and LSE).

    ``units`` restricts the work to (segment, head) units b*H + h; rows of
    other units are returned as NaN.
    """
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    bf = None if bias is None else _f64(bias)
    bias_len = 0 if bf is None else int(bf.shape[1])
    total_q = int(qo[-1])
    out = np.full((total_q, heads, head_dim), np.nan)
    lse = np.full((heads, total_q), np.nan)
    u, nu = _units(units)
    rc = _load().oracle_fwd(_ptr(qf), _ptr(kf), _ptr(vf), _ptr(qo), _ptr(ko), len(qo) - 1,
                            heads, head_dim, ACT_CODE[act], float(scale), _ptr(bf), bias_len,
                            int(bool(causal)), int(window), int(q_shared), _ptr(u), nu, int(threads),
                            _ptr(out), _ptr(lse))
    if rc:
        raise ValueError("oracle_fwd rejected its arguments" if rc == 1 else "oracle_fwd: out of memory")
    return out, lse


def bwd(q, k, v, dout, q_offsets, kv_offsets, heads: int, head_dim: int, act: str,
        scale: float, bias=None, causal: bool = False,
        units: Optional[Sequence[int]] = None, threads: int = 0, window: int = 0,
        q_shared: int = 0):
    """dQ, dK, dV (float64, layouts of q/k/v) and dbias (float64 [H, T] or None).
    With ``q_shared`` = S > 0, dQ is [S, H, d]: the sum over segments."""
    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(dout)
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    bf = None if bias is None else _f64(bias)
    bias_len = 0 if bf is None else int(bf.shape[1])
    dq = np.full(qf.shape, np.nan)
    dk = np.full(kf.shape, np.nan)
    dv = np.full(vf.shape, np.nan)
    dbias = None if bf is None else np.zeros_like(bf)
    u, nu = _units(units)
    rc = _load().oracle_bwd(_ptr(qf), _ptr(kf), _ptr(vf), _ptr(dof), _ptr(qo), _ptr(ko),
                            len(qo) - 1, heads, head_dim, ACT_CODE[act], float(scale), _ptr(bf),
                            bias_len, int(bool(causal)), int(window), int(q_shared), _ptr(u), nu,
                            int(threads),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias))
    if rc:
        raise ValueError("oracle_bwd rejected its arguments" if rc == 1 else "oracle_bwd: out of memory")
    return dq, dk, dv, dbias


def bwd_rows(q, k, v, dout, q_offsets, kv_offsets, heads: int, head_dim: int, act: str,
             scale: float, segment: int, head: int, q_rows, kv_rows, bias=None,
             causal: bool = False, window: int = 0, threads: int = 0):
    """The backward of one (segment, head) unit restricted to some of its rows:
    dQ of the segment-local query rows ``q_rows`` ([n_q, d]) and dK, dV of the
    key rows ``kv_rows`` ([n_kv, d]), equal to those rows of ``bwd``.  The work
    is O(rows x partner length), spread over threads, so single rows of very
    long segments can be checked."""
    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(dout)
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    bf = None if bias is None else _f64(bias)
    bias_len = 0 if bf is None else int(bf.shape[1])
    qr = np.ascontiguousarray(q_rows, dtype=np.int32)
    kr = np.ascontiguousarray(kv_rows, dtype=np.int32)
    dq = np.full((qr.size, head_dim), np.nan)
    dk = np.full((kr.size, head_dim), np.nan)
    dv = np.full((kr.size, head_dim), np.nan)
    rc = _load().oracle_bwd_rows(_ptr(qf), _ptr(kf), _ptr(vf), _ptr(dof), _ptr(qo), _ptr(ko),
                                 len(qo) - 1, heads, head_dim, ACT_CODE[act], float(scale), _ptr(bf),
                                 bias_len, int(bool(causal)), int(window), int(segment), int(head),
                                 _ptr(qr), int(qr.size), _ptr(kr), int(kr.size), int(threads),
                                 _ptr(dq), _ptr(dk), _ptr(dv))
    if rc:
        raise ValueError("oracle_bwd_rows rejected its arguments" if rc == 1 else "oracle_bwd_rows: out of memory")
    return dq, dk, dv


def fwd_inputs(x, units=None, threads: int = 0):
    """``fwd`` on a ``workloads.Inputs`` bundle."""
    return fwd(x.q, x.k, x.v, x.q_offsets, x.kv_offsets, x.heads, x.head_dim, x.act, x.scale,
               bias=x.bias, causal=x.causal, units=units, threads=threads, window=x.window)


def bwd_inputs(x, units=None, threads: int = 0):
    """``bwd`` on a ``workloads.Inputs`` bundle."""
    return bwd(x.q, x.k, x.v, x.dout, x.q_offsets, x.kv_offsets, x.heads, x.head_dim, x.act,
               x.scale, bias=x.bias, causal=x.causal, units=units, threads=threads, window=x.window)


def bwd_rows_inputs(x, segment: int, head: int, q_rows, kv_rows, threads: int = 0):
    """``bwd_rows`` on a ``workloads.Inputs`` bundle."""
    return bwd_rows(x.q, x.k, x.v, x.dout, x.q_offsets, x.kv_offsets, x.heads, x.head_dim, x.act,
                    x.scale, segment, head, q_rows, kv_rows, bias=x.bias, causal=x.causal,
                    window=x.window, threads=threads)
