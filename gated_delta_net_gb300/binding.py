"""Thin Python binding of ``include/gdn_tree.h``: argument marshalling only.

Every function has the name of the C entry point it calls.  Tensors are torch
tensors on the CUDA device (torch provides memory and streams; every step of
the computation runs in the library's kernels).  The library is loaded on
first use from ``_build/libgdn_tree.so``; if it is missing the call raises,
there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED = 0, 1, 2
GDN_ERR_INVALID_TREE, GDN_ERR_INVALID_PATH, GDN_ERR_CUDA, GDN_ERR_DEVICE = 3, 4, 5, 6
GDN_F32, GDN_BF16 = 0, 1
DEV_BITS = {1: "BAD_TREE", 2: "BAD_PATH", 4: "TOO_MANY", 8: "TOO_DEEP", 16: "TIMEOUT", 64: "INTERNAL",
            32: "BAD_DESC"}

_P = ctypes.c_void_p
_I = ctypes.c_int32


class VerifyArgs(ctypes.Structure):
    _fields_ = [("batch", _I), ("n_k_heads", _I), ("n_v_heads", _I), ("d_k", _I), ("d_v", _I),
                ("total_nodes", _I), ("max_nodes", _I), ("max_depth", _I), ("scale", ctypes.c_float),
                ("qkv_dtype", _I), ("out_dtype", _I), ("node_offsets", _P), ("q", _P), ("k", _P),
                ("v", _P), ("g", _P), ("beta", _P), ("S0", _P), ("parent", _P), ("anc_mask", _P),
                ("mask_words", _I), ("depth", _P), ("o", _P), ("dev_status", _P)]


class CommitArgs(ctypes.Structure):
    _fields_ = [("batch", _I), ("n_k_heads", _I), ("n_v_heads", _I), ("d_k", _I), ("d_v", _I),
                ("total_nodes", _I), ("max_nodes", _I), ("max_path", _I), ("qkv_dtype", _I),
                ("node_offsets", _P),
                ("k", _P), ("v", _P),
                ("g", _P), ("beta", _P), ("S0", _P), ("parent", _P), ("path_offsets", _P),
                ("path_idx", _P), ("S_new", _P), ("dev_status", _P)]


class StatesArgs(ctypes.Structure):
    _fields_ = [("batch", _I), ("n_k_heads", _I), ("n_v_heads", _I), ("d_k", _I), ("d_v", _I),
                ("total_nodes", _I), ("max_nodes", _I), ("qkv_dtype", _I),
                ("node_offsets", _P), ("k", _P), ("v", _P), ("g", _P), ("beta", _P), ("S0", _P),
                ("parent", _P), ("anc_mask", _P), ("mask_words", _I), ("n_sel", _I),
                ("sel_request", _P), ("sel_node", _P), ("S_sel", _P), ("dev_status", _P)]


class GdnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"gdn status {code}: {msg}")
        self.code = code


class GdnDeviceError(RuntimeError):
    def __init__(self, bits: int):
        names = [n for b, n in DEV_BITS.items() if bits & b]
        super().__init__(f"device status {bits} ({', '.join(names)})")
        self.bits = bits


_lib = None


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with gated_delta_net_gb300.build.build()")
        L = ctypes.CDLL(path)
        L.gdn_tree_build_desc.argtypes = [_P, _P, _I, _I, _P, _I, _P, _P, _P]
        L.gdn_tree_build_desc.restype = ctypes.c_int
        for fn in (L.gdn_tree_verify, L.gdn_tree_verify_branches):
            fn.argtypes = [ctypes.POINTER(VerifyArgs), _P]
            fn.restype = ctypes.c_int
        L.gdn_tree_commit.argtypes = [ctypes.POINTER(CommitArgs), _P]
        L.gdn_tree_commit.restype = ctypes.c_int
        L.gdn_tree_commit_verify.argtypes = [ctypes.POINTER(CommitArgs), ctypes.POINTER(VerifyArgs), _P]
        L.gdn_tree_commit_verify.restype = ctypes.c_int
        L.gdn_tree_states.argtypes = [ctypes.POINTER(StatesArgs), _P]
        L.gdn_tree_states.restype = ctypes.c_int
        L.gdn_tree_grow.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]
        L.gdn_tree_grow.restype = ctypes.c_int
        L.gdn_tree_relabel.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P]
        L.gdn_tree_relabel.restype = ctypes.c_int
        L.gdn_gather_rows.argtypes = [_P, _P, _P, _P, _I, _I, ctypes.c_int64, _P, _P]
        L.gdn_gather_rows.restype = ctypes.c_int
        L.gdn_last_error.restype = ctypes.c_char_p
        L.gdn_tree_version.restype = ctypes.c_int
        L.gdn_test_set_wait_probe.argtypes = [_I]
        L.gdn_test_set_wait_probe.restype = None
        _lib = L
    return _lib


def _check(code: int):
    if code != GDN_OK:
        raise GdnError(code, lib().gdn_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return GDN_F32
    if dtype == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"unsupported dtype {dtype}")


def gdn_test_set_wait_probe(polls: int) -> None:
    """Test hook: later tensor-core verify/commit launches make one bounded wait of
    ``polls`` polls that runs out (GDN_DEV_TIMEOUT); 0 turns it off."""
    lib().gdn_test_set_wait_probe(int(polls))


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_status(dev_status: torch.Tensor):
    """Synchronise on the status word and raise GdnDeviceError if any bit is set."""
    bits = int(dev_status.item())
    if bits:
        raise GdnDeviceError(bits)


def gdn_tree_build_desc(parent: torch.Tensor, node_offsets: torch.Tensor, max_nodes: int,
                        anc_mask: Optional[torch.Tensor] = None,
                        depth: Optional[torch.Tensor] = None, mask_words: Optional[int] = None,
                        dev_status: Optional[torch.Tensor] = None, stream=None):
    """Ancestor bitmask [T, mask_words] (int32 storage of uint32 words) and depth [T]."""
    _dev(parent, "parent", torch.int32)
    _dev(node_offsets, "node_offsets", torch.int32)
    T = parent.numel()
    words = mask_words or max(1, (max_nodes + 31) // 32)
    if anc_mask is None:
        anc_mask = torch.empty((T, words), dtype=torch.int32, device=parent.device)
    if depth is None:
        depth = torch.empty(T, dtype=torch.int32, device=parent.device)
    _dev(anc_mask, "anc_mask", torch.int32)
    _dev(depth, "depth", torch.int32)
    if anc_mask.shape != (T, words) or depth.numel() != T:
        raise ValueError("anc_mask must be [T, mask_words] and depth [T]")
    _check(lib().gdn_tree_build_desc(_ptr(parent), _ptr(node_offsets), node_offsets.numel() - 1,
                                     int(max_nodes), _ptr(anc_mask), words, _ptr(depth),
                                     _ptr(dev_status), _stream(stream)))
    return anc_mask, depth


def gdn_tree_states(k, v, g, beta, S0, node_offsets, parent, anc_mask, sel_request, sel_node,
                    max_nodes: int, out=None, dev_status=None, stream=None) -> torch.Tensor:
    """The state at each selected node [n_sel, Hv, d_v, d_k] (fp32)."""
    for name, t in (("k", k), ("v", v)):
        _dev(t, name)
    for name, t in (("g", g), ("beta", beta), ("S0", S0)):
        _dev(t, name, torch.float32)
    for name, t in (("node_offsets", node_offsets), ("parent", parent), ("anc_mask", anc_mask),
                    ("sel_request", sel_request), ("sel_node", sel_node)):
        _dev(t, name, torch.int32)
    T, Hk, dk = k.shape
    Hv, dv = v.shape[1], v.shape[2]
    B = node_offsets.numel() - 1
    n_sel = sel_request.numel()
    if sel_node.numel() != n_sel or S0.shape != (B, Hv, dv, dk):
        raise ValueError("inconsistent selection / S0 shapes")
    if out is None:
        out = torch.empty((n_sel, Hv, dv, dk), dtype=torch.float32, device=S0.device)
    _dev(out, "out", torch.float32)
    if out.shape != (n_sel, Hv, dv, dk):
        raise ValueError("out must be [n_sel, Hv, d_v, d_k]")
    a = StatesArgs(B, Hk, Hv, dk, dv, T, int(max_nodes), _code(k.dtype), _ptr(node_offsets), _ptr(k),
                   _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(parent), _ptr(anc_mask),
                   anc_mask.shape[1] if anc_mask.dim() == 2 else 1, n_sel, _ptr(sel_request),
                   _ptr(sel_node), _ptr(out), _ptr(dev_status))
    _check(lib().gdn_tree_states(ctypes.byref(a), _stream(stream)))
    return out


def gdn_tree_grow(node_offsets: torch.Tensor, n_children: torch.Tensor, draws: torch.Tensor,
                  width: int, max_depth: int = 16, dev_status=None, stream=None):
    """Top-w best-first trees: (parent [T] int32, score [T] float32, n_nodes [B] int32)."""
    _dev(node_offsets, "node_offsets", torch.int32)
    _dev(n_children, "n_children", torch.int32)
    _dev(draws, "draws", torch.float32)
    T = n_children.numel()
    if draws.dim() != 2 or draws.shape[0] != T or not draws.is_contiguous():
        raise ValueError("draws must be a contiguous [T, max_children] tensor")
    B = node_offsets.numel() - 1
    parent = torch.empty(T, dtype=torch.int32, device=draws.device)
    score = torch.empty(T, dtype=torch.float32, device=draws.device)
    n_nodes = torch.empty(B, dtype=torch.int32, device=draws.device)
    _check(lib().gdn_tree_grow(_ptr(node_offsets), B, T, int(width), int(max_depth), draws.shape[1],
                               _ptr(n_children), _ptr(draws), _ptr(parent), _ptr(score), _ptr(n_nodes),
                               _ptr(dev_status), _stream(stream)))
    return parent, score, n_nodes


def gdn_tree_relabel(parent: torch.Tensor, node_offsets: torch.Tensor, max_nodes: int,
                     dev_status: Optional[torch.Tensor] = None, stream=None):
    """Topological relabelling by (depth, old id): (order, rank, parent_out), each [T] int32
    with request-local ids."""
    _dev(parent, "parent", torch.int32)
    _dev(node_offsets, "node_offsets", torch.int32)
    T = parent.numel()
    order = torch.empty(T, dtype=torch.int32, device=parent.device)
    rank = torch.empty_like(order)
    parent_out = torch.empty_like(order)
    _check(lib().gdn_tree_relabel(_ptr(parent), _ptr(node_offsets), node_offsets.numel() - 1, T,
                                  int(max_nodes), _ptr(order), _ptr(rank), _ptr(parent_out),
                                  _ptr(dev_status), _stream(stream)))
    return order, rank, parent_out


def gdn_gather_rows(src: torch.Tensor, index: torch.Tensor, node_offsets: torch.Tensor,
                    out: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """Rows permuted within each request: out[lo + j] = src[lo + index[lo + j]]."""
    _dev(src, "src")
    _dev(index, "index", torch.int32)
    _dev(node_offsets, "node_offsets", torch.int32)
    if not src.is_contiguous():
        raise ValueError("src must be contiguous")
    T = src.shape[0]
    if index.numel() != T:
        raise ValueError("index must have one entry per row")
    if out is None:
        out = torch.empty_like(src)
    _dev(out, "out", src.dtype)
    if out.shape != src.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like src")
    row_bytes = src[0].numel() * src.element_size() if T else 16
    _check(lib().gdn_gather_rows(_ptr(src), _ptr(out), _ptr(index), _ptr(node_offsets),
                                 node_offsets.numel() - 1, T, row_bytes, _ptr(dev_status),
                                 _stream(stream)))
    return out


def _verify_args(q, k, v, g, beta, S0, node_offsets, parent, anc_mask, depth, max_nodes,
                 max_depth, scale, out, out_dtype, dev_status):
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    for name, t in (("g", g), ("beta", beta), ("S0", S0)):
        _dev(t, name, torch.float32)
    for name, t in (("node_offsets", node_offsets), ("parent", parent), ("anc_mask", anc_mask),
                    ("depth", depth)):
        _dev(t, name, torch.int32)
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    B = node_offsets.numel() - 1
    if k.shape != q.shape or v.shape[0] != T or g.shape != (T, Hv) or beta.shape != (T, Hv):
        raise ValueError("inconsistent token shapes")
    if S0.shape != (B, Hv, dv, dk) or parent.numel() != T or depth.numel() != T:
        raise ValueError("inconsistent S0 / tree shapes")
    od = out_dtype or q.dtype
    if out is None:
        out = torch.empty((T, Hv, dv), dtype=od, device=q.device)
    _dev(out, "out", od)
    if out.shape != (T, Hv, dv):
        raise ValueError("out must be [T, Hv, d_v]")
    a = VerifyArgs(B, Hk, Hv, dk, dv, T, int(max_nodes), int(max_depth), float(scale), _code(q.dtype),
                   _code(od), _ptr(node_offsets), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                   _ptr(S0), _ptr(parent), _ptr(anc_mask), anc_mask.shape[1] if anc_mask.dim() == 2 else 1,
                   _ptr(depth), _ptr(out), _ptr(dev_status))
    return a, out


def gdn_tree_verify(q, k, v, g, beta, S0, node_offsets, parent, anc_mask, depth, max_nodes: int,
                    max_depth: int = 0, scale: float = 1.0, out=None, out_dtype=None,
                    dev_status=None, stream=None) -> torch.Tensor:
    """Every node's output o [T, Hv, d_v]; S0 is only read."""
    a, out = _verify_args(q, k, v, g, beta, S0, node_offsets, parent, anc_mask, depth, max_nodes,
                          max_depth, scale, out, out_dtype, dev_status)
    _check(lib().gdn_tree_verify(ctypes.byref(a), _stream(stream)))
    return out


def gdn_tree_verify_branches(q, k, v, g, beta, S0, node_offsets, parent, anc_mask, depth,
                             max_nodes: int, max_depth: int = 0, scale: float = 1.0, out=None,
                             out_dtype=None, dev_status=None, stream=None) -> torch.Tensor:
    """Per-branch recurrent baseline; same results as gdn_tree_verify up to rounding."""
    a, out = _verify_args(q, k, v, g, beta, S0, node_offsets, parent, anc_mask, depth, max_nodes,
                          max_depth, scale, out, out_dtype, dev_status)
    _check(lib().gdn_tree_verify_branches(ctypes.byref(a), _stream(stream)))
    return out


def _commit_args(k, v, g, beta, S0, node_offsets, parent, path_offsets, path_idx, max_nodes,
                 max_path, out, dev_status):
    for name, t in (("k", k), ("v", v)):
        _dev(t, name)
    for name, t in (("g", g), ("beta", beta), ("S0", S0)):
        _dev(t, name, torch.float32)
    for name, t in (("node_offsets", node_offsets), ("parent", parent),
                    ("path_offsets", path_offsets), ("path_idx", path_idx)):
        _dev(t, name, torch.int32)
    T, Hk, dk = k.shape
    Hv, dv = v.shape[1], v.shape[2]
    B = node_offsets.numel() - 1
    if S0.shape != (B, Hv, dv, dk) or path_offsets.numel() != B + 1:
        raise ValueError("inconsistent S0 / path shapes")
    if out is None:
        out = torch.empty_like(S0)
    _dev(out, "out", torch.float32)
    if out.shape != S0.shape:
        raise ValueError("out must match S0")
    pidx = path_idx if path_idx.numel() else torch.zeros(1, dtype=torch.int32, device=k.device)
    a = CommitArgs(B, Hk, Hv, dk, dv, T, int(max_nodes), int(max_path), _code(k.dtype),
                   _ptr(node_offsets), _ptr(k),
                   _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(parent), _ptr(path_offsets),
                   _ptr(pidx), _ptr(out), _ptr(dev_status))
    return a, out, pidx


def gdn_tree_commit(k, v, g, beta, S0, node_offsets, parent, path_offsets, path_idx,
                    max_nodes: int, max_path: int = 0, out=None, dev_status=None,
                    stream=None) -> torch.Tensor:
    """State after each request's accepted path [B, Hv, d_v, d_k]; ``out`` may be ``S0``."""
    a, out, _keep = _commit_args(k, v, g, beta, S0, node_offsets, parent, path_offsets, path_idx,
                                 max_nodes, max_path, out, dev_status)
    _check(lib().gdn_tree_commit(ctypes.byref(a), _stream(stream)))
    return out


def gdn_tree_commit_verify(prev: dict, S0, max_nodes_prev: int, max_path: int,
                           q, k, v, g, beta, node_offsets, parent, anc_mask, depth, max_nodes: int,
                           max_depth: int = 16, scale: float = 1.0, S_new=None, out=None,
                           out_dtype=None, dev_status=None, stream=None):
    """Commit S0 along the previous tree's accepted path (``prev``: k, v, g, beta,
    node_offsets, parent, path_offsets, path_idx), write it to ``S_new`` (may be
    ``S0``), and verify the new tree from it.  Returns (o, S_new)."""
    c, S_new, _keep = _commit_args(prev["k"], prev["v"], prev["g"], prev["beta"], S0,
                                   prev["node_offsets"], prev["parent"], prev["path_offsets"],
                                   prev["path_idx"], max_nodes_prev, max_path, S_new, dev_status)
    a, out = _verify_args(q, k, v, g, beta, S_new, node_offsets, parent, anc_mask, depth, max_nodes,
                          max_depth, scale, out, out_dtype, dev_status)
    _check(lib().gdn_tree_commit_verify(ctypes.byref(c), ctypes.byref(a), _stream(stream)))
    return out, S_new


# ----------------------------------------------------------------------------
# upload of a seeded workload (marshalling only)
# ----------------------------------------------------------------------------

def upload(tb, device="cuda", pin: bool = False) -> dict:
    """Copy a ``workloads.TreeBatch`` into tensors (device, or pinned host if ``pin``)."""
    qdt = torch.bfloat16 if tb.qkv_dtype == "bf16" else torch.float32

    def put(x, dtype):
        t = torch.from_numpy(x).to(dtype)
        if pin:
            return t.pin_memory()
        return t.to(device)

    return {
        "q": put(tb.q, qdt), "k": put(tb.k, qdt), "v": put(tb.v, qdt),
        "g": put(tb.g, torch.float32), "beta": put(tb.beta, torch.float32),
        "S0": put(tb.S0, torch.float32),
        "node_offsets": put(tb.node_offsets, torch.int32), "parent": put(tb.parent, torch.int32),
        "path_offsets": put(tb.path_offsets, torch.int32),
        "path_idx": put(tb.path_idx if len(tb.path_idx) else tb.path_idx.reshape(0), torch.int32),
    }
