"""GPU vs fp64 oracle: one verify round of a synthetic 3:1 hybrid stack through the C ABI, in
the order a serving step issues it -- 24 independent GDN layers verified in both modes (fork
as its two passes, TreeWY), the accept walk on the device, one stacked commit per mode, then 8
tree-attention layers and the compaction of each layer's cache.  The shapes are the wide-tree
sweep's (GDN H=16, d=128; attention 16q/4kv, hd 128, prefix 8192; random dynamic trees of 40
nodes, bf16) at batch 2, so that the oracle checks every layer: every committed state, every
attention output, every compacted cache, and sampled GDN outputs of every layer."""
import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import attention as A
from oracle import gdn as G

pytestmark = pytest.mark.gpu
DEV = "cuda"
GDN_LAYERS, ATTN_LAYERS, B, N = 24, 8, 2, 40


def test_hybrid_stack_round_matches_the_oracle():
    trees = W.sweep_trees(N, B, seed=7)
    gdn = [W.gdn_case(trees, H=16, dk=128, dv=128, io="bf16", state="bf16", seed=7000 + l, path_max_len=4)
           for l in range(GDN_LAYERS)]
    attn = [W.attn_case(trees, [8192] * B, Hq=16, Hkv=4, hd=128, seed=7100 + l, rope_theta=1e6, path_max_len=4)
            for l in range(ATTN_LAYERS)]
    c0 = gdn[0]
    H, dk, dv = 16, 128, 128
    parents = _gpu.to_dev(c0.parents)
    # the accept walk takes the first layer's sampled paths (one path per sequence for the stack)
    draft, target = W.walk_tokens(trees, c0.path.numpy(), c0.path_len.numpy(), seed=3)
    Lmax = c0.path.shape[1]
    i32 = dict(dtype=torch.int32, device=DEV)
    path, plen, nxt = torch.full((B, Lmax), 777, **i32), torch.full((B,), 777, **i32), torch.full((B,), 777, **i32)
    err = torch.full((6 + GDN_LAYERS, B), 777, **i32)

    x = [_gpu.gdn_inputs(c) for c in gdn]
    k_all = torch.stack([xi["k"] for xi in x]).contiguous()
    S0_fork = torch.stack([xi["S0"] for xi in x]).contiguous()
    S0_wy = S0_fork.clone()
    o_fork = torch.full((GDN_LAYERS, B, N, H, dv), float("nan"), dtype=torch.bfloat16, device=DEV)
    o_wy = torch.full_like(o_fork, float("nan"))
    states = torch.full((GDN_LAYERS, B, N, H, dv, dk), float("nan"), dtype=torch.bfloat16, device=DEV)
    pv = torch.full((GDN_LAYERS, B, N, H, dv), float("nan"), device=DEV)
    lg = torch.full((GDN_LAYERS, B, N, H), float("nan"), device=DEV)
    w_scratch = torch.empty((B, N, H, dv), device=DEV)
    lg_scratch = torch.empty((B, N, H), device=DEV)
    for l in range(GDN_LAYERS):
        xi = x[l]
        tv.tv_gdn_tree_verify_wy(xi["q"], k_all[l], xi["v"], xi["alpha"], xi["beta"], S0_fork[l], parents,
                                 o_fork[l], w_scratch, lg_scratch, err[6 + l])
        tv.tv_gdn_fork_materialize(k_all[l], xi["alpha"], S0_fork[l], parents, w_scratch, states[l], err[6 + l])
        tv.tv_gdn_tree_verify_wy(xi["q"], k_all[l], xi["v"], xi["alpha"], xi["beta"], S0_wy[l], parents,
                                 o_wy[l], pv[l], lg[l], err[0])
    tv.tv_accept_walk(parents, _gpu.to_dev(draft), _gpu.to_dev(target), path, plen, nxt, err[1])
    tv.tv_gdn_commit_layers(tv.TV_MODE_FORK, path, plen, parents, S0_fork, err[2], node_states=states)
    tv.tv_gdn_commit_layers(tv.TV_MODE_WY, path, plen, parents, S0_wy, err[3], pseudo_v=pv, log_gamma=lg, k=k_all)

    a_res = []
    for c in attn:
        q, kn, vn = _gpu.to_dev(c.q), _gpu.to_dev(c.k_new), _gpu.to_dev(c.v_new)
        kc, vc = _gpu.to_dev(c.k_cache), _gpu.to_dev(c.v_cache)
        table, pl = _gpu.to_dev(c.block_table), _gpu.to_dev(c.prefix_len)
        out = torch.full((B, N, 16, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        ws = torch.empty(tv.tv_tree_attn_workspace_size(B, N, 16, 4, 128, table.shape[1]), dtype=torch.uint8,
                         device=DEV)
        tv.tv_tree_attn(q, kn, vn, kc, vc, table, pl, parents, out, ws, err[4], rope_theta=1e6)
        o_after = out.clone()
        kc_after, vc_after = kc.clone(), vc.clone()
        smap, new_len = torch.full((B, Lmax), 777, **i32), torch.full((B,), 777, **i32)
        tv.tv_kv_compact(kc, vc, table, pl, parents, path, plen, smap, new_len, err[5])
        a_res.append(dict(out=o_after, kc_after=kc_after, vc_after=vc_after, kc=kc, vc=vc, smap=smap,
                          new_len=new_len))
    torch.cuda.synchronize()
    assert (err.cpu() == 0).all(), err.cpu().tolist()

    # the walk took the sampled paths
    p_np, L_np = path.cpu().numpy(), plen.cpu().numpy()
    assert np.array_equal(L_np, c0.path_len.numpy())
    for b in range(B):
        assert list(p_np[b, :L_np[b]]) == list(c0.path.numpy()[b, :L_np[b]])

    rng = np.random.default_rng(11)
    for l, c in enumerate(gdn):
        inp = c.oracle_inputs()
        # committed state of every layer and sequence, both modes
        for b in range(B):
            S_ref = G.node_state(inp, b, int(p_np[b, L_np[b] - 1]))[0]
            _gpu.assert_close(S0_fork[l, b].cpu(), S_ref, "bf16", "stack fork commit")
            _gpu.assert_close(S0_wy[l, b].cpu(), S_ref, "bf16", "stack wy commit")
        # sampled outputs and snapshots of every layer
        b = int(rng.integers(0, B))
        for i in sorted(set([0, N - 1, int(rng.integers(1, N - 1))])):
            S, o = G.node_state(inp, b, i)
            _gpu.assert_close(o_fork[l, b, i].cpu(), o, "bf16", "stack fork o")
            _gpu.assert_close(o_wy[l, b, i].cpu(), o, "bf16", "stack wy o")
            _gpu.assert_close(states[l, b, i].cpu(), S, "bf16", "stack fork snapshot")

    for c, r in zip(attn, a_res):
        f = _gpu.attn_f64(c)
        o_ref, kr_ref = _gpu.assert_attention_close(r["out"].cpu(), f, list(range(B)), "stack attention o")
        kc_ref, vc_ref = A.cache_after_attention(f, kr_ref)
        kc_got, vc_got = _gpu.f32np(r["kc_after"]), _gpu.f32np(r["vc_after"])
        kc2, vc2, smap, new_len = A.kv_compact(kc_got, vc_got, f["block_table"], f["prefix_len"], f["parents"],
                                               p_np, L_np)
        assert np.array_equal(r["smap"].cpu().numpy(), smap)
        assert np.array_equal(r["new_len"].cpu().numpy(), new_len)
        kc3, vc3 = _gpu.f32np(r["kc"]), _gpu.f32np(r["vc"])
        for b in range(B):
            n, tab = int(new_len[b]), f["block_table"][b]
            P = int(f["prefix_len"][b])
            # values are copied exactly; rotated keys within the bf16 rule of the oracle's
            assert np.array_equal(A.logical_rows(vc3, tab, n), A.logical_rows(vc2, tab, n))
            assert np.array_equal(A.logical_rows(kc3, tab, n), A.logical_rows(kc2, tab, n))
            assert np.array_equal(A.logical_rows(vc_got, tab, P + N)[P:], f["v_new"][b])
            _gpu.assert_close(A.logical_rows(kc_got, tab, P + N)[P:], kr_ref[b], "bf16",
                              "stack rotated node keys", stored="bf16")
