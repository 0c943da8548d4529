"""ctypes wrapper of the FP64 token-recurrence oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable flags only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("n_seq", ctypes.c_int),
        ("seq_start", ctypes.c_void_p),
        ("H", ctypes.c_int), ("K", ctypes.c_int), ("V", ctypes.c_int),
        ("gate", ctypes.c_int),
        ("scale", ctypes.c_double),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("g", ctypes.c_void_p), ("h0", ctypes.c_void_p),
        ("dout", ctypes.c_void_p), ("dht", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("ht", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dbeta", ctypes.c_void_p), ("dg", ctypes.c_void_p), ("dh0", ctypes.c_void_p),
        ("backward", ctypes.c_int),
        ("items", ctypes.c_void_p),
        ("n_items", ctypes.c_int),
        ("erase", ctypes.c_void_p), ("write", ctypes.c_void_p),
        ("derase", ctypes.c_void_p), ("dwrite", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.kda_oracle_run.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int]
            lib.kda_oracle_run.restype = ctypes.c_int
            _lib = lib
    return _lib


_GATES = {"none": 0, "scalar": 1, "channel": 2}


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def run_recurrence(q, k, v, beta, g, seq_start, *, gate: str, scale: float, h0=None,
                   do=None, dht=None, backward: bool = True, nthreads: int | None = None,
                   items=None, erase=None, write=None) -> dict:
    """Run the oracle on packed arrays.

    q, k: [T, H, K]; v, do: [T, H, V]; beta: [T, H]; g: [T, H] (scalar),
    [T, H, K] (channel) or None; h0, dht: [N, H, K, V] or None;
    seq_start: N + 1 token offsets. ``items``: optional list of (seq, head)
    pairs to compute (outputs of other pairs are left at zero).
    Returns float64 arrays o, ht and, with ``backward``, dq, dk, dv, dbeta, dg
    (None without a gate) and dh0. GatedDeltaNet-2: ``erase`` [T, H, K] and
    ``write`` [T, H, V] replace beta (which may then be None); the backward
    then returns derase and dwrite in place of dbeta.
    """
    lib = _load()
    q, k, v, beta = _c64(q), _c64(k), _c64(v), _c64(beta)
    g, h0, do, dht = _c64(g), _c64(h0), _c64(do), _c64(dht)
    erase, write = _c64(erase), _c64(write)
    T, H, K = q.shape
    V = v.shape[2]
    ss = np.ascontiguousarray(np.asarray(seq_start, dtype=np.int64))
    N = ss.size - 1
    out = dict(o=np.zeros((T, H, V)), ht=np.zeros((N, H, K, V)))
    if backward:
        if do is None:
            raise ValueError("backward needs do")
        out.update(dq=np.zeros((T, H, K)), dk=np.zeros((T, H, K)), dv=np.zeros((T, H, V)),
                   dbeta=None if erase is not None else np.zeros((T, H)), dh0=np.zeros((N, H, K, V)),
                   dg=None if gate == "none" else np.zeros(g.shape))
        if erase is not None:
            out.update(derase=np.zeros((T, H, K)), dwrite=np.zeros((T, H, V)))
    it = None
    n_items = 0
    if items is not None:
        it = np.ascontiguousarray(np.asarray(items, dtype=np.int32).reshape(-1, 2))
        n_items = it.shape[0]
    p = _Problem()
    p.n_seq, p.seq_start, p.H, p.K, p.V = N, ss.ctypes.data, H, K, V
    p.gate, p.scale = _GATES[gate], float(scale)
    p.q, p.k, p.v, p.beta, p.g, p.h0 = _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0)
    p.dout, p.dht = _ptr(do), _ptr(dht)
    p.erase, p.write = _ptr(erase), _ptr(write)
    p.o, p.ht = _ptr(out["o"]), _ptr(out["ht"])
    if backward:
        p.dq, p.dk, p.dv = _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"])
        p.dbeta, p.dg, p.dh0 = _ptr(out["dbeta"]), _ptr(out["dg"]), _ptr(out["dh0"])
        if erase is not None:
            p.derase, p.dwrite = _ptr(out["derase"]), _ptr(out["dwrite"])
    p.backward = 1 if backward else 0
    p.items = None if it is None else it.ctypes.data
    p.n_items = n_items
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib.kda_oracle_run(ctypes.byref(p), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle failed with status %d" % rc)
    return out
