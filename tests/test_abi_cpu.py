"""The C-ABI library builds, loads and exports every declared entry point, and
rejects bad arguments synchronously (host-only checks; no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fz():
    from learned_group_sparse_focus_gb300 import _build
    if not os.path.exists(_build.LIB):
        _build.build()
    from learned_group_sparse_focus_gb300 import focus
    return focus


def _declared():
    src = open(os.path.join(ROOT, "include", "focus.h")).read()
    return re.findall(r"FOCUS_API\s+[\w\s\*]+?\b(focus_\w+)\s*\(", src)


def test_header_declares_the_hot_path():
    names = set(_declared())
    assert {"focus_assign", "focus_build_index", "focus_attention_fwd",
            "focus_dense_causal_fwd", "focus_workspace_bytes", "focus_check_errors"} <= names


def test_every_declared_symbol_is_exported(fz):
    lib = ctypes.CDLL(fz.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(fz.EXPORTED) == set(_declared())
    assert lib.focus_abi_version() == 3


def test_struct_layouts_match_header(fz):
    assert ctypes.sizeof(fz.Params) == 12 * 4
    assert ctypes.sizeof(fz.Item) == 8 * 4
    assert ctypes.sizeof(fz.Index) == 9 * 8 + 2 * 4
    assert ctypes.sizeof(fz.IndexTopk) == 2 * ctypes.sizeof(fz.Index) + 2 * 8 + 2 * 4 + 8


def test_status_strings(fz):
    lib = fz.lib()
    for s in range(7):
        assert lib.focus_status_string(s)
    assert lib.focus_status_string(3) == b"workspace too small"


def test_workspace_size_is_host_arithmetic(fz):
    p = fz.make_params(B=1, H=32, H_kv=8, n=32768, d=128, D=4096, d_g=64, K=64, A=1, w=512)
    nb = fz.focus_workspace_bytes(p)
    # at least the group partial (O_far bf16 + LSE) and the sorted K/V copies
    assert nb >= 32 * 32768 * 128 * 2 + 32 * 32768 * 4 + 2 * 8 * 32768 * 128 * 2
    assert nb % 256 == 0
    bad = fz.make_params(B=1, H=3, H_kv=2, n=10, d=64, D=8, d_g=32, K=2, A=1, w=1)
    assert fz.focus_workspace_bytes(bad) == 0


@pytest.mark.parametrize("field,value", [
    ("H_kv", 5), ("n", 0), ("K", 0), ("K", 5000), ("A", 3), ("w", -1), ("scale", 0.0),
    ("dtype", 7), ("n", (1 << 20) + 1),
])
def test_invalid_params_rejected_before_any_launch(fz, field, value):
    kw = dict(B=1, H=4, H_kv=2, n=64, d=64, D=64, d_g=32, K=4, A=1, w=8)
    p = fz.make_params(**kw)
    setattr(p, field, value)
    lib = fz.lib()
    fake = ctypes.c_void_p(1 << 20)
    st = lib.focus_assign(ctypes.byref(p), fake, fake, fake, fake, fake, 1 << 30, None)
    assert st == 1
    idx = fz.Index()
    assert lib.focus_build_index(ctypes.byref(p), fake, ctypes.byref(idx), fake, 1 << 30, None) == 1


def test_null_misaligned_and_small_workspace(fz):
    lib = fz.lib()
    p = fz.make_params(B=1, H=4, H_kv=2, n=64, d=64, D=64, d_g=32, K=4, A=1, w=8)
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    need = fz.focus_workspace_bytes(p)
    assert lib.focus_assign(ctypes.byref(p), None, ok, ok, ok, ok, need, None) == 1
    assert lib.focus_assign(ctypes.byref(p), mis, ok, ok, ok, ok, need, None) == 1
    assert lib.focus_assign(ctypes.byref(p), ok, ok, ok, ok, ok, need - 256, None) == 3
    assert lib.focus_assign(ctypes.byref(p), ok, ok, ok, ok, mis, need, None) == 1
    idx = fz.Index()
    assert lib.focus_build_index(ctypes.byref(p), ok, None, ok, need, None) == 1
    assert lib.focus_attention_fwd(ctypes.byref(p), ok, ok, ok, None, ok, None, ok, need, None) == 1
    assert lib.focus_dense_causal_fwd(ctypes.byref(p), ok, ok, ok, ok, None, ok, need - 256, None) == 3
    p.d = 96
    assert lib.focus_dense_causal_fwd(ctypes.byref(p), ok, ok, ok, ok, None, ok, need, None) == 2
    assert lib.focus_workspace_init(mis, None) == 1
    assert lib.focus_attention_two_call_fwd(ctypes.byref(p), ok, ok, ok, None, ok, None, ok, need, None) == 1
    del idx


# ------------------------------------------------------- top-k membership ---

def test_topk_workspace_sizes(fz):
    p = fz.make_params(B=1, H=32, H_kv=8, n=32768, d=128, D=4096, d_g=64, K=4, A=1, w=512)
    one, two = fz.focus_workspace_bytes_topk(p, 1), fz.focus_workspace_bytes_topk(p, 2)
    # k = 1 holds the top-1 index and partials (not the two-call comparator's LSE)
    assert one >= fz.focus_workspace_bytes(p) - 32 * 32768 * 4 - 256 and one % 256 == 0
    # entry partials (2n rows), pair and merged partials (n rows each), bf16
    assert two >= 4 * 32 * 32768 * 128 * 2 and two > one
    assert fz.focus_workspace_bytes_topk(p, 0) == 0
    assert fz.focus_workspace_bytes_topk(p, 3) == 0
    p.K = 91                                    # 4095 group pairs: the largest K for k = 2
    assert fz.focus_workspace_bytes_topk(p, 2) > 0
    p.K = 92
    assert fz.focus_workspace_bytes_topk(p, 2) == 0
    assert fz.focus_workspace_bytes_topk(p, 1) > 0
    p.K = 1                                     # two distinct groups need K >= 2
    assert fz.focus_workspace_bytes_topk(p, 2) == 0


def test_topk_argument_checks(fz):
    lib = fz.lib()
    p = fz.make_params(B=1, H=4, H_kv=2, n=64, d=64, D=64, d_g=32, K=4, A=1, w=8)
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    need = fz.focus_workspace_bytes_topk(p, 2)
    assert lib.focus_assign_topk(ctypes.byref(p), 3, ok, ok, ok, ok, ok, need, None) == 1
    assert lib.focus_assign_topk(ctypes.byref(p), 2, mis, ok, ok, ok, ok, need, None) == 1
    assert lib.focus_assign_topk(ctypes.byref(p), 2, ok, ok, ok, ok, ok, need - 256, None) == 3
    idx = fz.IndexTopk()
    assert lib.focus_build_index_topk(ctypes.byref(p), 2, ok, None, ok, need, None) == 1
    assert lib.focus_build_index_topk(ctypes.byref(p), 2, mis, ctypes.byref(idx), ok, need, None) == 1
    assert lib.focus_build_index_topk(ctypes.byref(p), 2, ok, ctypes.byref(idx), ok, need - 256, None) == 3
    q = fz.make_params(B=1, H=4, H_kv=2, n=64, d=64, D=64, d_g=32, K=100, A=1, w=8)
    assert lib.focus_build_index_topk(ctypes.byref(q), 2, ok, ctypes.byref(idx), ok, 1 << 40, None) == 2
    # attention: an index that is not one (k outside {1, 2}, null arrays) is refused
    assert lib.focus_attention_topk_fwd(ctypes.byref(p), ok, ok, ok, None, ok, None, ok, need, None) == 1
    idx.k = 3
    assert lib.focus_attention_topk_fwd(ctypes.byref(p), ok, ok, ok, ctypes.byref(idx), ok, None, ok, need,
                                        None) == 1
    idx.k = 2
    assert lib.focus_attention_topk_fwd(ctypes.byref(p), ok, ok, ok, ctypes.byref(idx), ok, None, ok, need,
                                        None) == 1


def test_sinkhorn_argument_checks(fz):
    lib = fz.lib()
    p = fz.make_params(B=1, H=2, H_kv=2, n=1000, d=64, D=64, d_g=32, K=16, A=2, w=8)
    need = lib.focus_sinkhorn_workspace_bytes(ctypes.byref(p))
    # error word + u [2, 1000] + v [2, 16] + chunk partials [2, 8, 16] float2 + a
    # ticket per problem, each 256-aligned
    assert need == 256 + 8192 + 256 + 2048 + 256
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    f = lib.focus_sinkhorn_fwd
    assert f(ctypes.byref(p), 0, 1.0, ok, ok, ok, need, None) == 1           # no rounds
    assert f(ctypes.byref(p), 10001, 1.0, ok, ok, ok, need, None) == 1
    assert f(ctypes.byref(p), 3, 0.0, ok, ok, ok, need, None) == 1           # tau
    assert f(ctypes.byref(p), 3, float("inf"), ok, ok, ok, need, None) == 1
    assert f(ctypes.byref(p), 3, 1.0, mis, ok, ok, need, None) == 1
    assert f(ctypes.byref(p), 3, 1.0, ok, ok, ok, need - 256, None) == 3
    assert lib.focus_assign_scores(ctypes.byref(p), ok, ok, ok, None, ok, need, None) == 1
    assert lib.focus_assign_scores(ctypes.byref(p), ok, ok, ok, ok, ok, need - 256, None) == 3


def test_backward_argument_checks(fz):
    lib = fz.lib()
    p = fz.make_params(B=1, H=4, H_kv=2, n=64, d=64, D=64, d_g=32, K=4, A=1, w=8)
    need = lib.focus_backward_workspace_bytes(ctypes.byref(p))
    # error word + Delta [4*64] + dQ part [4*64*64] + dK, dV parts [2*64*64] fp32,
    # and for bf16 the index-ordered copies: Q, dO [4*64*64], K, V [2*64*64] bf16,
    # LSE and Delta [4*64] fp32, and the far dK/dV unit order [2 KV heads x 1 tile]
    # int32 (one 256-byte block)
    assert need == 256 + 1024 + 65536 + 2 * 32768 + 2 * 32768 + 2 * 16384 + 2 * 1024 + 256
    q = fz.make_params(B=1, H=4, H_kv=2, n=64, d=64, D=64, d_g=32, K=4, A=1, w=8, dtype="f32")
    assert lib.focus_backward_workspace_bytes(ctypes.byref(q)) == 256 + 1024 + 65536 + 2 * 32768
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    f = lib.focus_attention_bwd
    assert f(ctypes.byref(p), ok, ok, ok, ok, ok, ok, None, ok, ok, ok, ok, need, None) == 1
    idx = fz.Index()
    for name in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot", "items", "order", "n_items"):
        setattr(idx, name, 1 << 21)
    idx.max_items = 1 + 4          # ceil(64/128) + min(K, n) for one problem
    idx.w_eff = 8
    assert f(ctypes.byref(p), mis, ok, ok, ok, ok, ok, ctypes.byref(idx), ok, ok, ok, ok, need, None) == 1
    assert f(ctypes.byref(p), ok, ok, ok, ok, ok, ok, ctypes.byref(idx), ok, ok, ok, ok, need - 256, None) == 3
    idx.w_eff = 9                  # an index built for another window
    assert f(ctypes.byref(p), ok, ok, ok, ok, ok, ok, ctypes.byref(idx), ok, ok, ok, ok, need, None) == 1
