"""The C-ABI library loads and exports every symbol ``include/tv.h`` declares; host-side
argument checks reject bad calls before any device work (CPU only: no call here reaches the
GPU)."""
import ctypes
import os
import re

import pytest
import torch

import tree_speculative_verification_gdn_gb300 as tv

# These tests pass host addresses where device pointers belong and rely on the host-side checks
# rejecting the call first; they never run where a GPU could receive such a pointer.
cpu_only = pytest.mark.skipif(torch.cuda.is_available(), reason="host-address stand-ins; CPU only")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "tv.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"TV_API\s+[\w\s\*]*?\b(tv_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported_and_bound():
    names = _declared()
    assert len(names) >= 10
    lib = ctypes.CDLL(tv.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
        assert name in tv.EXPORTED, name
    assert sorted(tv.EXPORTED) == names


def test_enum_values_match_header():
    with open(os.path.join(ROOT, "include", "tv.h")) as f:
        text = f.read()
    for name in ("TV_OK", "TV_ERR_INVALID_ARG", "TV_ERR_BAD_TREE", "TV_ERR_BAD_PATH", "TV_ERR_UNSUPPORTED",
                 "TV_ERR_CUDA", "TV_ERR_TIMEOUT", "TV_ERR_CAPACITY", "TV_ERR_BAD_BLOCK", "TV_F32", "TV_BF16",
                 "TV_MODE_FORK", "TV_MODE_WY"):
        m = re.search(rf"\b{name}\s*=\s*(-?\d+)", text)
        assert m and int(m.group(1)) == getattr(tv, name), name
    for name in ("TV_MAX_NODES", "TV_BLOCK_SIZE"):
        m = re.search(rf"#define\s+{name}\s+(\d+)", text)
        assert m and int(m.group(1)) == getattr(tv, name)


def test_status_strings_and_version():
    assert tv.status_string(0) == "ok"
    for code in range(-9, 0):
        assert tv.status_string(code) and tv.status_string(code) != "unknown status"
    assert tv.status_string(99) == "unknown status"
    assert tv.lib.tv_version() >= 100


def test_null_pointers_are_rejected_before_launch():
    L = tv.lib
    assert L.tv_tree_prepare(None, 1, 4, None, None, None, 0, None, None, None) == tv.TV_ERR_INVALID_ARG
    args = [None] * 7 + [1, 7, 2, 64, 64, tv.TV_F32, tv.TV_F32, 1.0, None, None, None, None]
    assert L.tv_gdn_tree_verify_fork(*args) == tv.TV_ERR_INVALID_ARG
    args = [None] * 7 + [1, 7, 2, 64, 64, tv.TV_F32, tv.TV_F32, 1.0, None, None, None, None, None]
    assert L.tv_gdn_tree_verify_wy(*args) == tv.TV_ERR_INVALID_ARG
    assert L.tv_gdn_commit(tv.TV_MODE_FORK, None, None, 3, None, None, None, None, None, None, 1, 7, 2, 64,
                           64, 0, 0, None, None) == tv.TV_ERR_INVALID_ARG


def _fake(n=1 << 20):
    """A 256-byte-aligned host address standing in for a device pointer; the checks below fail
    on sizes before anything dereferences it."""
    buf = ctypes.create_string_buffer(n + 256)
    addr = (ctypes.addressof(buf) + 255) & ~255
    return buf, ctypes.c_void_p(addr)


@cpu_only
@pytest.mark.parametrize("dk,dv,io,st,want", [
    (96, 64, 0, 0, tv.TV_ERR_UNSUPPORTED),
    (64, 32, 0, 0, tv.TV_ERR_UNSUPPORTED),
    (64, 64, 0, 1, tv.TV_ERR_UNSUPPORTED),   # fp32 I/O with a bf16 state has no kernel
    (64, 64, 5, 0, tv.TV_ERR_INVALID_ARG),
])
def test_unsupported_sizes_and_dtypes(dk, dv, io, st, want):
    keep, p = _fake()
    args = [p] * 7 + [1, 7, 2, dk, dv, io, st, 1.0, p, p, p, None]
    assert tv.lib.tv_gdn_tree_verify_fork(*args) == want
    del keep


@cpu_only
def test_size_limits():
    keep, p = _fake()
    args = [p] * 7 + [1, 257, 2, 64, 64, 0, 0, 1.0, p, p, p, None]
    assert tv.lib.tv_gdn_tree_verify_fork(*args) == tv.TV_ERR_UNSUPPORTED
    args = [p] * 7 + [0, 7, 2, 64, 64, 0, 0, 1.0, p, p, p, None]
    assert tv.lib.tv_gdn_tree_verify_fork(*args) == tv.TV_ERR_INVALID_ARG
    # misaligned q
    q = ctypes.c_void_p(p.value + 4)
    args = [q] + [p] * 6 + [1, 7, 2, 64, 64, 0, 0, 1.0, p, p, p, None]
    assert tv.lib.tv_gdn_tree_verify_fork(*args) == tv.TV_ERR_INVALID_ARG
    # attention: unsupported head dim / block size, Hq not a multiple of Hkv
    a = [p] * 5 + [4, p, 2, p, p, 1, 3, 4, 2, 96, 16, 1e6, 0.1, p, p, 1 << 20, p, None]
    assert tv.lib.tv_tree_attn(*a) == tv.TV_ERR_UNSUPPORTED
    a = [p] * 5 + [4, p, 2, p, p, 1, 3, 4, 2, 64, 32, 1e6, 0.1, p, p, 1 << 20, p, None]
    assert tv.lib.tv_tree_attn(*a) == tv.TV_ERR_UNSUPPORTED
    a = [p] * 5 + [4, p, 2, p, p, 1, 3, 3, 2, 64, 16, 1e6, 0.1, p, p, 1 << 20, p, None]
    assert tv.lib.tv_tree_attn(*a) == tv.TV_ERR_INVALID_ARG
    del keep


def test_workspace_size_is_host_only_and_monotone():
    s1 = tv.tv_tree_attn_workspace_size(1, 15, 16, 4, 128, 258)
    s2 = tv.tv_tree_attn_workspace_size(32, 40, 16, 4, 256, 2053)
    assert 0 < s1 < s2
    assert tv.tv_tree_attn_workspace_size(1, 15, 16, 3, 128, 258) == 0   # Hq % Hkv != 0


@cpu_only
def test_stack_commit_and_selective_snapshot_argument_checks():
    keep, p = _fake()
    L = tv.lib
    # tv_gdn_commit_layers: the layer count and the mode are checked on the host
    base = [tv.TV_MODE_FORK, p, p, 4, p, p, None, None, None, p]
    assert L.tv_gdn_commit_layers(*base, 0, 2, 7, 2, 64, 64, 0, 0, p, None) == tv.TV_ERR_INVALID_ARG
    assert L.tv_gdn_commit_layers(*base, 3, 2, 300, 2, 64, 64, 0, 0, p, None) == tv.TV_ERR_UNSUPPORTED
    assert L.tv_gdn_commit_layers(*base, 1 << 20, 1 << 10, 7, 1 << 10, 64, 64, 0, 0, p, None) == \
        tv.TV_ERR_UNSUPPORTED                                        # layers * B * H overflows an int
    wy = [tv.TV_MODE_WY, p, p, 4, p, None, p, p, p, p]
    assert L.tv_gdn_commit_layers(*wy, 2, 2, 7, 2, 96, 64, 0, 0, p, None) == tv.TV_ERR_UNSUPPORTED
    assert L.tv_gdn_commit_layers(7, p, p, 4, p, p, p, p, p, p, 2, 2, 7, 2, 64, 64, 0, 0, p, None) == \
        tv.TV_ERR_INVALID_ARG                                        # no such mode
    # tv_gdn_fork_materialize_selective: capacity, threshold and pointers
    sel = [p, p, p, p, p, p]
    assert L.tv_gdn_fork_materialize_selective(*sel, 0.95, 0, 2, 7, 2, 64, 64, 0, 0, 0, p, p, p, None) == \
        tv.TV_ERR_INVALID_ARG                                        # capacity 0
    assert L.tv_gdn_fork_materialize_selective(*sel, 0.95, 8, 2, 7, 2, 64, 64, 0, 0, 0, p, p, p, None) == \
        tv.TV_ERR_INVALID_ARG                                        # capacity > N
    assert L.tv_gdn_fork_materialize_selective(*sel, float("nan"), 3, 2, 7, 2, 64, 64, 0, 0, 0, p, p, p, None) == \
        tv.TV_ERR_INVALID_ARG
    assert L.tv_gdn_fork_materialize_selective(p, p, p, p, p, None, 0.95, 3, 2, 7, 2, 64, 64, 0, 0, 0, p, p, p,
                                               None) == tv.TV_ERR_INVALID_ARG   # no confidence
    assert L.tv_gdn_fork_materialize_selective(*sel, 0.95, 3, 2, 7, 2, 64, 64, 0, 0, -1, p, p, p, None) == \
        tv.TV_ERR_INVALID_ARG                                        # negative CTA cap
    assert L.tv_gdn_fork_materialize(p, p, p, p, p, 2, 300, 2, 64, 64, 0, 0, 0, p, p, None) == tv.TV_ERR_UNSUPPORTED
    # tv_tree_prepare: paths need a positive row length
    assert L.tv_tree_prepare(p, 2, 7, p, p, p, 0, None, p, None) == tv.TV_ERR_INVALID_ARG
    del keep


@cpu_only
def test_block_table_compaction_argument_checks():
    keep, p = _fake()
    out = ctypes.c_void_p(p.value + 4096)
    base = [p, p, 8, p, out, 4, p, p, 40, p, p, 5, 2, 4, 128, 16, p, p, p, p, None]

    def call(**changes):
        a = list(base)
        for i, v in changes.items():
            a[int(i[1:])] = v
        return tv.lib.tv_kv_compact_remap(*a)

    assert call(a4=ctypes.c_void_p(p.value + 16)) == tv.TV_ERR_INVALID_ARG   # output overlaps the table
    assert call(a4=p) == tv.TV_ERR_INVALID_ARG
    assert call(a4=None) == tv.TV_ERR_INVALID_ARG
    assert call(a18=None) == tv.TV_ERR_INVALID_ARG                           # no exchange counts
    assert call(a12=0) == tv.TV_ERR_INVALID_ARG
    assert call(a14=96) == tv.TV_ERR_UNSUPPORTED
    assert call(a15=32) == tv.TV_ERR_UNSUPPORTED
    assert call(a8=257) == tv.TV_ERR_UNSUPPORTED
    del keep


def test_static_attention_rejects_bad_arguments_before_any_cuda_call():
    # Hq % Hkv != 0 (the workspace size is then 0) and null pointers: refused by the host-side
    # checks of tv_tree_attn, which run before the scratch lookup (no CUDA call is made, so this
    # holds without a GPU).
    L = tv.lib
    assert L.tv_tree_attn_static(None, None, None, None, None, 8, None, 4, None, None,
                                 1, 3, 3, 2, 64, 16, 1e6, 0.125, None, None, None) == tv.TV_ERR_INVALID_ARG
    assert L.tv_tree_attn_static(None, None, None, None, None, 8, None, 4, None, None,
                                 1, 3, 4, 2, 64, 16, 1e6, 0.125, None, None, None) == tv.TV_ERR_INVALID_ARG


@cpu_only
def test_static_attention_rejects_unsupported_sizes_before_any_cuda_call():
    keep, p = _fake()
    a = [p] * 5 + [4, p, 2, p, p, 1, 3, 4, 2, 96, 16, 1e6, 0.1, p, p, None]
    assert tv.lib.tv_tree_attn_static(*a) == tv.TV_ERR_UNSUPPORTED
    a = [p] * 5 + [4, p, 2, p, p, 1, 3, 4, 2, 64, 16, 0.0, 0.1, p, p, None]     # rope_theta <= 0
    assert tv.lib.tv_tree_attn_static(*a) == tv.TV_ERR_INVALID_ARG
    del keep


def test_bounded_wait_probe_rejects_null_outputs():
    assert tv.lib.tv_test_bounded_wait(100, 0, None, None, None) == tv.TV_ERR_INVALID_ARG
    assert tv.status_string(tv.TV_ERR_TIMEOUT) == "device wait timed out"
