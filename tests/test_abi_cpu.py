"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every entry point the header declares, and rejects bad
arguments with the documented status codes before launching anything."""
import ctypes
import os
import re

import pytest

from gated_delta_net_gb300 import binding, build

HEADER = os.path.join(build.INCLUDE, "gdn_tree.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_symbols() == sorted(["gdn_gather_rows", "gdn_last_error", "gdn_tree_build_desc",
                                         "gdn_tree_commit", "gdn_tree_commit_verify", "gdn_tree_grow",
                                         "gdn_tree_relabel",
                                         "gdn_tree_states",
                                         "gdn_tree_verify", "gdn_tree_verify_branches",
                                         "gdn_tree_version", "gdn_test_set_wait_probe"])


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name
    assert L.gdn_tree_version() == 200


def _verify_args(**kw):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: every case fails validation first
    base = dict(batch=1, n_k_heads=1, n_v_heads=1, d_k=16, d_v=16, total_nodes=12, max_nodes=12,
                max_depth=0,
                scale=1.0, qkv_dtype=0, out_dtype=0, node_offsets=fake, q=fake, k=fake, v=fake,
                g=fake, beta=fake, S0=fake, parent=fake, anc_mask=fake, mask_words=1, depth=fake,
                o=fake, dev_status=fake)
    base.update(kw)
    return binding.VerifyArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(batch=-1), binding.GDN_ERR_INVALID_ARG),
    (dict(n_k_heads=0), binding.GDN_ERR_INVALID_ARG),
    (dict(n_k_heads=2, n_v_heads=3), binding.GDN_ERR_INVALID_ARG),
    (dict(d_k=48), binding.GDN_ERR_UNSUPPORTED),
    (dict(d_v=256), binding.GDN_ERR_UNSUPPORTED),
    (dict(max_nodes=0), binding.GDN_ERR_INVALID_ARG),
    (dict(max_nodes=257, mask_words=9), binding.GDN_ERR_UNSUPPORTED),
    (dict(max_nodes=64, mask_words=1), binding.GDN_ERR_INVALID_ARG),
    (dict(qkv_dtype=7), binding.GDN_ERR_UNSUPPORTED),
    (dict(max_depth=-1), binding.GDN_ERR_INVALID_ARG),
    (dict(total_nodes=-1), binding.GDN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.GDN_ERR_INVALID_ARG),
    (dict(q=None), binding.GDN_ERR_INVALID_ARG),
    (dict(o=None), binding.GDN_ERR_INVALID_ARG),
])
def test_verify_rejects_bad_arguments(L, kw, code):
    a = _verify_args(**kw)
    for fn in (L.gdn_tree_verify, L.gdn_tree_verify_branches):
        assert fn(ctypes.byref(a), None) == code
        assert L.gdn_last_error().decode() != ""


def test_verify_empty_batch_is_a_no_op(L):
    a = _verify_args(batch=0, q=None, k=None)
    assert L.gdn_tree_verify(ctypes.byref(a), None) == binding.GDN_OK


def test_commit_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    base = dict(batch=1, n_k_heads=1, n_v_heads=1, d_k=16, d_v=16, total_nodes=12, max_nodes=12,
                max_path=0, qkv_dtype=0,
                node_offsets=fake, k=fake, v=fake, g=fake, beta=fake, S0=fake, parent=fake,
                path_offsets=fake, path_idx=fake, S_new=fake, dev_status=fake)
    for kw, code in ((dict(S_new=None), binding.GDN_ERR_INVALID_ARG),
                     (dict(d_k=8), binding.GDN_ERR_UNSUPPORTED),
                     (dict(max_nodes=300), binding.GDN_ERR_UNSUPPORTED),
                     (dict(qkv_dtype=3), binding.GDN_ERR_UNSUPPORTED),
                     (dict(max_path=-1), binding.GDN_ERR_INVALID_ARG)):
        a = binding.CommitArgs(**{**base, **kw})
        assert L.gdn_tree_commit(ctypes.byref(a), None) == code
    assert L.gdn_tree_commit(None, None) == binding.GDN_ERR_INVALID_ARG


def test_commit_verify_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    cbase = dict(batch=1, n_k_heads=1, n_v_heads=1, d_k=16, d_v=16, total_nodes=12, max_nodes=12,
                 max_path=0, qkv_dtype=0,
                 node_offsets=fake, k=fake, v=fake, g=fake, beta=fake, S0=fake, parent=fake,
                 path_offsets=fake, path_idx=fake, S_new=fake, dev_status=fake)
    f = L.gdn_tree_commit_verify
    v = _verify_args(S0=None)  # the verify side's S0 is not read: the committed state is
    for ckw, vkw, code in ((dict(S_new=None), {}, binding.GDN_ERR_INVALID_ARG),
                           ({}, dict(q=None), binding.GDN_ERR_INVALID_ARG),
                           (dict(n_v_heads=2), dict(n_v_heads=1), binding.GDN_ERR_INVALID_ARG),
                           (dict(batch=2), {}, binding.GDN_ERR_INVALID_ARG),
                           (dict(d_k=32, d_v=32), {}, binding.GDN_ERR_INVALID_ARG),
                           (dict(d_k=8), {}, binding.GDN_ERR_UNSUPPORTED),
                           ({}, dict(d_v=48), binding.GDN_ERR_UNSUPPORTED),
                           (dict(max_path=-1), {}, binding.GDN_ERR_INVALID_ARG)):
        c = binding.CommitArgs(**{**cbase, **ckw})
        vv = _verify_args(S0=None, **vkw)
        assert f(ctypes.byref(c), ctypes.byref(vv), None) == code, (ckw, vkw)
        assert L.gdn_last_error().decode() != ""
    c = binding.CommitArgs(**cbase)
    assert f(None, ctypes.byref(v), None) == binding.GDN_ERR_INVALID_ARG
    assert f(ctypes.byref(c), None, None) == binding.GDN_ERR_INVALID_ARG
    c0 = binding.CommitArgs(**{**cbase, "batch": 0})
    v0 = _verify_args(batch=0, S0=None, q=None)
    assert f(ctypes.byref(c0), ctypes.byref(v0), None) == binding.GDN_OK


def test_build_desc_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    f = L.gdn_tree_build_desc
    assert f(fake, fake, -1, 12, fake, 1, fake, fake, None) == binding.GDN_ERR_INVALID_ARG
    assert f(fake, fake, 1, 300, fake, 8, fake, fake, None) == binding.GDN_ERR_UNSUPPORTED
    assert f(fake, fake, 1, 100, fake, 2, fake, fake, None) == binding.GDN_ERR_INVALID_ARG
    assert f(None, fake, 1, 12, fake, 1, fake, fake, None) == binding.GDN_ERR_INVALID_ARG
    assert f(None, None, 0, 12, None, 1, None, None, None) == binding.GDN_OK


def _states_args(**kw):
    fake = 0x1000
    a = dict(batch=1, n_k_heads=1, n_v_heads=2, d_k=128, d_v=128, total_nodes=4, max_nodes=4,
             qkv_dtype=binding.GDN_BF16, node_offsets=fake, k=fake, v=fake, g=fake, beta=fake,
             S0=fake, parent=fake, anc_mask=fake, mask_words=1, n_sel=2, sel_request=fake,
             sel_node=fake, S_sel=fake, dev_status=None)
    a.update(kw)
    return binding.StatesArgs(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(n_sel=-1), binding.GDN_ERR_INVALID_ARG),
    (dict(sel_node=None), binding.GDN_ERR_INVALID_ARG),
    (dict(mask_words=0), binding.GDN_ERR_INVALID_ARG),
    (dict(d_k=64, d_v=64), binding.GDN_ERR_UNSUPPORTED),
    (dict(qkv_dtype=binding.GDN_F32), binding.GDN_ERR_UNSUPPORTED),
    (dict(n_v_heads=3, n_k_heads=2), binding.GDN_ERR_INVALID_ARG),
    (dict(n_sel=0, S_sel=None), binding.GDN_OK),
])
def test_states_rejects_bad_arguments(L, kw, code):
    a = _states_args(**kw)
    assert L.gdn_tree_states(ctypes.byref(a), None) == code
    assert L.gdn_tree_states(None, None) == binding.GDN_ERR_INVALID_ARG


def test_grow_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    f = L.gdn_tree_grow
    ok = [fake, 1, 8, 2, 16, 8, fake, fake, fake, fake, fake, None, None]
    for pos, bad in ((1, -1), (2, -1), (3, 0), (4, 0), (5, 0), (5, 65), (6, None), (9, None)):
        args = list(ok)
        args[pos] = bad
        assert f(*args) == binding.GDN_ERR_INVALID_ARG, pos
    assert f(None, 0, 0, 1, 16, 8, None, None, None, None, None, None, None) == binding.GDN_OK


def test_relabel_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    f = L.gdn_tree_relabel
    assert f(fake, fake, -1, 4, 12, fake, fake, fake, fake, None) == binding.GDN_ERR_INVALID_ARG
    assert f(fake, fake, 1, -1, 12, fake, fake, fake, fake, None) == binding.GDN_ERR_INVALID_ARG
    assert f(fake, fake, 1, 4, 0, fake, fake, fake, fake, None) == binding.GDN_ERR_INVALID_ARG
    assert f(fake, fake, 1, 4, 300, fake, fake, fake, fake, None) == binding.GDN_ERR_UNSUPPORTED
    assert f(fake, fake, 1, 4, 12, None, fake, fake, fake, None) == binding.GDN_ERR_INVALID_ARG
    assert f(None, None, 0, 0, 12, None, None, None, None, None) == binding.GDN_OK


def test_gather_rejects_bad_arguments(L):
    a, b = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x100000)
    f = L.gdn_gather_rows
    assert f(a, b, a, a, 1, 4, 24, None, None) == binding.GDN_ERR_INVALID_ARG      # not a multiple of 16
    assert f(a, b, a, a, 1, 4, 0, None, None) == binding.GDN_ERR_INVALID_ARG
    assert f(a, ctypes.c_void_p(0x1008), a, a, 1, 4, 32, None, None) == binding.GDN_ERR_INVALID_ARG
    assert f(a, ctypes.c_void_p(0x1010), a, a, 1, 4, 32, None, None) == binding.GDN_ERR_INVALID_ARG  # overlap
    assert f(None, b, a, a, 1, 4, 32, None, None) == binding.GDN_ERR_INVALID_ARG
    assert f(None, None, None, None, 0, 0, 32, None, None) == binding.GDN_OK


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()
