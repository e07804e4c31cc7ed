"""tv_tree_attn_static: tree attention on the library's static scratch, through the C ABI.

Its results must equal tv_tree_attn's (same kernels, same split plan) bit for bit.  The
module runs last (file name) and also on its own: it builds everything it uses.
"""
import gc

import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W

DEV = "cuda:0"


def test_oversize_request_is_refused_before_any_cuda_call():
    # The paged batch-32 hd-256 shape needs ~350 MB of scratch: refused on the host, so null
    # pointers never reach a check that would dereference them.
    need = tv.tv_tree_attn_workspace_size(32, 40, 16, 4, 256, 2053)
    assert need > tv.TV_STATIC_SCRATCH_BYTES
    st = tv.lib.tv_tree_attn_static(None, None, None, None, None, 4000, None, 2053, None, None,
                                    32, 40, 16, 4, 256, 16, 1e6, 0.0625, None, None, None)
    assert st == tv.TV_ERR_SCRATCH
    assert "static scratch" in tv.status_string(tv.TV_ERR_SCRATCH)


def test_scratch_constant_matches_header():
    import os
    import re
    with open(os.path.join(os.path.dirname(__file__), "..", "include", "tv.h")) as f:
        text = f.read()
    m = re.search(r"#define\s+TV_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == tv.TV_STATIC_SCRATCH_BYTES
    m = re.search(r"\bTV_ERR_SCRATCH\s*=\s*(-?\d+)", text)
    assert m and int(m.group(1)) == tv.TV_ERR_SCRATCH


def _device_inputs(case):
    B, N, Hq, Hkv, hd = case.shape
    d = {k: _gpu.to_dev(getattr(case, k)) for k in
         ("q", "k_new", "v_new", "k_cache", "v_cache", "block_table", "prefix_len", "parents")}
    return d, (B, N, Hq, hd)


def _run(case, static: bool):
    d, (B, N, Hq, hd) = _device_inputs(case)
    out = torch.full((B, N, Hq, hd), float("nan"), dtype=torch.bfloat16, device=DEV)
    err = torch.full((B,), 12345, dtype=torch.int32, device=DEV)
    args = (d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_table"],
            d["prefix_len"], d["parents"], out)
    if static:
        tv.tv_tree_attn_static(*args, err, rope_theta=case.rope_theta)
    else:
        ws = torch.empty(tv.tv_tree_attn_workspace_size(B, N, Hq, case.shape[3], hd, d["block_table"].shape[1]),
                         dtype=torch.uint8, device=DEV)
        tv.tv_tree_attn(*args, ws, err, rope_theta=case.rope_theta)
    torch.cuda.synchronize()
    return out.cpu(), d["k_cache"].cpu(), d["v_cache"].cpu(), err.cpu()


def _cases():
    rng = np.random.default_rng(11)
    a = W.single_layer_attn_case("tree")                                        # hd 128, P 4096
    b = W.attn_case([W.random_tree(33, rng) for _ in range(4)], [0, 17, 300, 2049],
                    Hq=8, Hkv=2, hd=256, seed=5)                                # hd 256, ragged
    c = W.attn_case([W.random_tree(7, rng) for _ in range(3)], [0, 5, 70],
                    Hq=4, Hkv=2, hd=64, seed=6)                                 # hd 64: CUDA-core partials
    return a, b, c


@pytest.mark.gpu
def test_two_calls_in_a_row_equal_the_workspace_entry_point():
    cases = _cases()
    for c in cases:
        B, N, Hq, Hkv, hd = c.shape
        assert tv.tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, c.block_table.shape[1]) <= tv.TV_STATIC_SCRATCH_BYTES
    got = [_run(c, static=True) for c in cases]          # two static calls back to back
    want = [_run(c, static=False) for c in cases]
    for (o, kc, vc, e), (o_w, kc_w, vc_w, e_w) in zip(got, want):
        assert (e == 0).all() and (e_w == 0).all(), (e, e_w)
        assert torch.equal(o.view(torch.int16), o_w.view(torch.int16))
        assert torch.equal(kc.view(torch.int16), kc_w.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), vc_w.view(torch.int16))
        assert not torch.isnan(o.float()).any()


@pytest.mark.gpu
def test_repeat_call_gives_same_result_and_allocates_nothing():
    case = _cases()[1]
    first = _run(case, static=True)                       # also does the per-device set-up
    d, (B, N, Hq, hd) = _device_inputs(case)
    out = torch.empty((B, N, Hq, hd), dtype=torch.bfloat16, device=DEV)
    err = torch.empty((B,), dtype=torch.int32, device=DEV)
    args = (d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_table"],
            d["prefix_len"], d["parents"], out, err)
    tv.tv_tree_attn_static(*args, rope_theta=case.rope_theta)
    torch.cuda.synchronize()
    gc.collect()  # tensors of earlier tests must not be freed inside the measured call
    gc.disable()
    try:
        free_before, _ = torch.cuda.mem_get_info()
        alloc_before = torch.cuda.memory_allocated()
        tv.tv_tree_attn_static(*args, rope_theta=case.rope_theta)
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()
        alloc_after = torch.cuda.memory_allocated()
    finally:
        gc.enable()
    assert free_after == free_before
    assert alloc_after == alloc_before
    assert (err.cpu() == 0).all()
    assert torch.equal(out.cpu().view(torch.int16), first[0].view(torch.int16))
