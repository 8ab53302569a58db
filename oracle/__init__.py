"""float64 CPU oracle for GDN speculative-tree verification.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  Nothing here is imported by
the CUDA library or its Python binding, and this package imports nothing from
them.

The arithmetic lives in ``gdn_oracle.c`` (plain C, float64, one sequential path
walk per node; see its header for the passages it follows).  This module
compiles it with gcc into ``oracle/_build/`` and marshals numpy arrays.

Parity pins (tests/test_oracle_pins.py): delta-rule write property, the
beta = 0 closed form, a hand-worked scalar example (tests/golden), brute force
over every forest with N <= 6 against a numpy.linalg.solve of the matrix form,
sibling independence, relabelling invariance, commit = walked state, and the
descriptor against networkx.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, IEEE float64, no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    P = ctypes.c_void_p
    lib.gdn_oracle_build_desc.argtypes = [P, P, i32, i32, P, P]
    lib.gdn_oracle_build_desc.restype = ctypes.c_int
    lib.gdn_oracle_verify.argtypes = [i32] * 5 + [P] * 8 + [f64, P, i32]
    lib.gdn_oracle_verify.restype = i32
    lib.gdn_oracle_verify_sel.argtypes = [i32] * 5 + [P] * 8 + [f64, P, i64, P, i32]
    lib.gdn_oracle_verify_sel.restype = i32
    lib.gdn_oracle_commit.argtypes = [i32] * 5 + [P] * 9 + [P, i32]
    lib.gdn_oracle_commit.restype = i32
    lib.gdn_oracle_state_at.argtypes = [i32] * 5 + [P] * 7 + [i32, i32, i32, P]
    lib.gdn_oracle_state_at.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(build()))
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def build_desc(parent, offsets, words: int):
    """Ancestor bitmask [T, words] (uint32) and depth [T] (int32, root = 1).
    Returns (mask, depth, status); status 1 marks a parent outside [-1, i)."""
    parent, offsets = _i32(parent), _i32(offsets)
    T = int(offsets[-1]) if len(offsets) else 0
    mask = np.zeros((max(T, 0), words), np.uint32)
    depth = np.zeros(max(T, 0), np.int32)
    st = _load().gdn_oracle_build_desc(_p(parent), _p(offsets), len(offsets) - 1, words,
                                       _p(mask), _p(depth))
    return mask, depth, int(st)


def _dims(tb):
    return (tb.batch, tb.n_k_heads, tb.n_v_heads, tb.d_k, tb.d_v)


def verify(tb, nthreads: Optional[int] = None) -> np.ndarray:
    """Every node's output o [T, Hv, d_v] in float64 (sequential path walk per node)."""
    o = np.zeros((tb.total_nodes, tb.n_v_heads, tb.d_v), np.float64)
    keep = [_i32(tb.node_offsets), _i32(tb.parent), _f64(tb.q), _f64(tb.k), _f64(tb.v),
            _f64(tb.g), _f64(tb.beta), _f64(tb.S0)]
    st = _load().gdn_oracle_verify(*_dims(tb), *[_p(a) for a in keep], float(tb.scale), _p(o),
                                   nthreads or default_threads())
    if st:
        raise ValueError("oracle: malformed tree")
    return o


def prepare(tb):
    """The workload's arrays in the oracle's own layout (int32 / float64 copies),
    so that repeated calls on one workload convert them once."""
    return [_i32(tb.node_offsets), _i32(tb.parent), _f64(tb.q), _f64(tb.k), _f64(tb.v),
            _f64(tb.g), _f64(tb.beta), _f64(tb.S0)]


def verify_selected(tb, sel, nthreads: Optional[int] = None, prepared=None) -> np.ndarray:
    """Outputs [len(sel), d_v] of the selected (request, value head, local node) triples.
    `prepared` is the result of prepare(tb), when the caller holds one."""
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int64).reshape(-1, 3))
    o = np.zeros((len(sel), tb.d_v), np.float64)
    keep = prepared if prepared is not None else prepare(tb)
    st = _load().gdn_oracle_verify_sel(*_dims(tb), *[_p(a) for a in keep], float(tb.scale),
                                       _p(sel), len(sel), _p(o), nthreads or default_threads())
    if st:
        raise ValueError("oracle: malformed tree")
    return o


def commit(tb, nthreads: Optional[int] = None, path_offsets=None, path_idx=None):
    """New state [B, Hv, d_v, d_k] after each request's accepted path.
    Returns (S_new, status); status 2 marks an invalid path."""
    poff = _i32(tb.path_offsets if path_offsets is None else path_offsets)
    pidx = _i32(tb.path_idx if path_idx is None else path_idx)
    S = np.zeros(tb.S0.shape, np.float64)
    keep = [_i32(tb.node_offsets), _i32(tb.parent), _f64(tb.k), _f64(tb.v), _f64(tb.g),
            _f64(tb.beta), _f64(tb.S0), poff, pidx if len(pidx) else np.zeros(1, np.int32)]
    st = _load().gdn_oracle_commit(*_dims(tb), *[_p(a) for a in keep], _p(S),
                                   nthreads or default_threads())
    return S, int(st)


def state_at(tb, b: int, h: int, i: int) -> np.ndarray:
    """The state [d_v, d_k] after walking node i's path (request b, value head h)."""
    S = np.zeros((tb.d_v, tb.d_k), np.float64)
    keep = [_i32(tb.node_offsets), _i32(tb.parent), _f64(tb.k), _f64(tb.v), _f64(tb.g),
            _f64(tb.beta), _f64(tb.S0)]
    st = _load().gdn_oracle_state_at(*_dims(tb), *[_p(a) for a in keep], b, h, i, _p(S))
    if st:
        raise ValueError("oracle: malformed tree")
    return S
