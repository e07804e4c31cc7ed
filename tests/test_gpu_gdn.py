"""GPU vs fp64 oracle: GDN tree verify (fork and TreeWY modes) and commit, through the C ABI.

Small cases are compared element by element over every output; the full-size batch-64 stack layer and
the wide-tree sweep cases (the launch configuration the benchmark times) are compared on sampled
(sequence, node) outputs the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import gdn as G

pytestmark = pytest.mark.gpu


def _caterpillar(n):
    """Spine nodes each with one leaf and one spine child: every spine node branches."""
    parents, spine = [-1], 0
    while len(parents) < n:
        parents.append(spine)           # leaf
        if len(parents) < n:
            parents.append(spine)       # next spine node
            spine = len(parents) - 1
    return parents


def _forest(n, rng):
    """Several roots (children of the committed state) with random subtrees."""
    parents = []
    for i in range(n):
        parents.append(-1 if i == 0 or rng.random() < 0.2 else int(rng.integers(0, i)))
    return parents


def _check_all(case, modes=("fork", "wy")):
    io = case.io
    inp = case.oracle_inputs()
    o_ref, S_ref = G.verify(inp)
    res = {}
    if "fork" in modes:
        f = _gpu.run_fork(case)
        assert (f["err"] == 0).all()
        _gpu.assert_close(f["out"], o_ref, io, "fork o")
        _gpu.assert_close(f["states"], S_ref, io if case.state == io else "bf16", "fork states")
        res["fork"] = f
    if "wy" in modes:
        w = _gpu.run_wy(case)
        assert (w["err"] == 0).all()
        _gpu.assert_close(w["out"], o_ref, io, "wy o")
        for b in range(case.q.shape[0]):
            w_ref, lg_ref = G.pseudo_values(inp, b)
            _gpu.assert_close(w["pseudo_v"][b], w_ref, io, f"wy pseudo-values b={b}")
            _gpu.assert_close(w["log_gamma"][b], lg_ref, io, f"wy log-gamma b={b}")
        res["wy"] = w
    commit_ref = G.commit(inp, case.path.numpy(), case.path_len.numpy())
    for mode, r in res.items():
        S0 = _gpu.run_commit(case, mode, r)
        assert (r["commit_err"] == 0).all()
        _gpu.assert_close(S0, commit_ref, io if case.state == io else "bf16", f"{mode} commit")
    return res


def test_small_fp32_layer():
    _check_all(W.small_fp32_case())


@pytest.mark.parametrize("tree", ["chain", "tree"])
def test_single_layer_bf16(tree):
    _check_all(W.single_layer_gdn_case(tree))


@pytest.mark.parametrize("io,state", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("d", [64, 128])
def test_small_random_trees(io, state, d):
    rng = np.random.default_rng(d + len(io))
    trees = [W.random_tree(33, rng) for _ in range(3)]
    _check_all(W.gdn_case(trees, H=2, dk=d, dv=d, io=io, state=state, seed=d))


@pytest.mark.parametrize("n", [1, 2, 3])
def test_tiny_trees(n):
    trees = [W.chain(n), [-1] * n]
    _check_all(W.gdn_case(trees, H=3, dk=64, dv=64, io="f32", state="f32", seed=n))


def test_mixed_dims():
    rng = np.random.default_rng(7)
    trees = [W.random_tree(20, rng) for _ in range(2)]
    _check_all(W.gdn_case(trees, H=2, dk=128, dv=64, io="f32", state="f32", seed=3))
    _check_all(W.gdn_case(trees, H=2, dk=64, dv=128, io="bf16", state="bf16", seed=4))


def test_stack_stress_shapes():
    """Caterpillar (every spine node branches), complete binary tree of depth 7 (deepest light
    nesting for 255 nodes), forest, deep chain."""
    rng = np.random.default_rng(11)
    trees = [_caterpillar(64), W.full_tree(2, 5)[:63] + [0], _forest(64, rng), W.chain(64)]
    _check_all(W.gdn_case(trees, H=1, dk=64, dv=64, io="f32", state="f32", seed=5))


def test_max_nodes_complete_binary():
    trees = [W.full_tree(2, 7) + [0]]  # 255 + 1 = 256 nodes, depth 7
    case = W.gdn_case(trees, H=1, dk=64, dv=64, io="f32", state="f32", seed=6)
    inp = case.oracle_inputs()
    f = _gpu.run_fork(case)
    w = _gpu.run_wy(case)
    assert int(f["err"][0]) == 0 and int(w["err"][0]) == 0
    rng = np.random.default_rng(0)
    for i in list(rng.choice(256, 24, replace=False)) + [255, 254, 127]:
        S, o = G.node_state(inp, 0, int(i))
        _gpu.assert_close(f["states"][0, i], S, "f32", f"fork state {i}")
        _gpu.assert_close(f["out"][0, i], o, "f32", f"fork o {i}")
        _gpu.assert_close(w["out"][0, i], o, "f32", f"wy o {i}")


def test_fork_and_wy_agree_and_commits_agree():
    rng = np.random.default_rng(21)
    trees = [W.random_tree(40, rng) for _ in range(4)]
    case = W.gdn_case(trees, H=4, dk=128, dv=128, io="bf16", state="f32", seed=8)
    f = _gpu.run_fork(case)
    w = _gpu.run_wy(case)
    o_f, o_w = W.f64(f["out"]), W.f64(w["out"])
    _gpu.assert_close(o_w, o_f, "bf16", "wy vs fork", stored="bf16", ref_rounded=True)
    S_f = _gpu.run_commit(case, "fork", f)
    S_w = _gpu.run_commit(case, "wy", w)
    _gpu.assert_close(S_w, W.f64(S_f), "bf16", "wy commit vs fork commit", ref_rounded=S_f.dtype == torch.bfloat16)


def _sampled_check(case, n_seq, n_nodes, seed):
    inp = case.oracle_inputs()
    B, N = case.q.shape[:2]
    io = case.io
    f = _gpu.run_fork(case, keep_device=True)   # the snapshots stay on the device: sampled rows only
    w = _gpu.run_wy(case)
    assert (f["err"].cpu() == 0).all() and (w["err"] == 0).all()
    f_out = f["out"].cpu()
    rng = np.random.default_rng(seed)
    seqs = sorted(set([0, B - 1] + list(rng.choice(B, n_seq, replace=False))))
    S_got, S_ref, o_got_f, o_got_w, o_ref = [], [], [], [], []
    for b in seqs:
        for i in sorted(set([0, N - 1] + list(rng.choice(N, n_nodes, replace=False)))):
            S, o = G.node_state(inp, b, int(i))
            S_ref.append(S); o_ref.append(o)
            S_got.append(W.f64(f["states"][b, int(i)].cpu())); o_got_f.append(W.f64(f_out[b, i]))
            o_got_w.append(W.f64(w["out"][b, i]))
    _gpu.assert_close(np.stack(S_got), np.stack(S_ref), io, "fork states (sampled)", stored=case.state)
    _gpu.assert_close(np.stack(o_got_f), np.stack(o_ref), io, "fork o (sampled)", stored=io)
    _gpu.assert_close(np.stack(o_got_w), np.stack(o_ref), io, "wy o (sampled)", stored=io)
    pv_got, pv_ref, lg_got, lg_ref = [], [], [], []
    for b in seqs[:2]:
        for i in sorted(set([0, N - 1] + list(rng.choice(N, n_nodes, replace=False)))):
            wr, lr = G.pseudo_value_node(inp, b, int(i))
            pv_ref.append(wr); lg_ref.append(lr)
            pv_got.append(W.f64(w["pseudo_v"][b, i])); lg_got.append(W.f64(w["log_gamma"][b, i]))
    _gpu.assert_close(np.stack(pv_got), np.stack(pv_ref), io, "wy pseudo-values (sampled)", stored="f32")
    _gpu.assert_close(np.stack(lg_got), np.stack(lg_ref), io, "wy log-gamma (sampled)", stored="f32")
    commit_ref = {bb: G.node_state(inp, bb, int(case.path[bb, int(case.path_len[bb]) - 1]))[0]
                  for bb in seqs[:3]}
    for mode, r in (("fork", f), ("wy", w)):
        S0 = _gpu.run_commit(case, mode, r)
        assert (r["commit_err"] == 0).all()
        for bb, ref in commit_ref.items():
            _gpu.assert_close(S0[bb], ref, io, f"{mode} commit b={bb}")
    # fork and WY agree on every output, not only the sampled ones
    _gpu.assert_close(w["out"], W.f64(f_out), io, "wy vs fork, all outputs", ref_rounded=True)


def test_stack_layer_full_size_sampled():
    """One layer of the batch-64 GDN stack at its full size: B=64, N=40 (k=3 d=3), H=16, d=128, bf16."""
    _sampled_check(W.stack_b64_layer(layer=0), n_seq=3, n_nodes=5, seed=2)


@pytest.mark.parametrize("N,B", [(15, 8), (64, 8), (256, 4), (40, 128), (256, 128)])
def test_wide_tree_sweep_sampled(N, B):
    """GDN layers of the wide-tree sweep, up to its largest shape (B=128, N=256: 16 GiB of
    fork snapshots on the device)."""
    _sampled_check(W.sweep_gdn_layer(N, B), n_seq=2, n_nodes=4, seed=N)


def test_malformed_tree_only_fails_its_sequence():
    rng = np.random.default_rng(3)
    trees = [W.random_tree(12, rng) for _ in range(3)]
    case = W.gdn_case(trees, H=2, dk=64, dv=64, io="f32", state="f32", seed=9)
    case.parents[1, 5] = 7          # a later node: not allowed
    inp = case.oracle_inputs()
    for run in (_gpu.run_fork, _gpu.run_wy):
        r = run(case)
        assert r["err"].tolist() == [0, tv.TV_ERR_BAD_TREE, 0]
        for b in (0, 2):
            for i in range(12):
                _, o = G.node_state(inp, b, i)
                _gpu.assert_close(r["out"][b, i], o, "f32", f"healthy sequence {b}")
        assert torch.isnan(r["out"][1]).all()     # the failed sequence is left unwritten


def test_wy_path_capacity_is_reported():
    case = W.gdn_case([W.chain(256)], H=1, dk=64, dv=64, io="f32", state="f32", seed=1)
    r = _gpu.run_wy(case)
    assert int(r["err"][0]) == tv.TV_ERR_UNSUPPORTED
    f = _gpu.run_fork(case)   # fork mode has no such limit
    assert int(f["err"][0]) == 0
    inp = case.oracle_inputs()
    S, o = G.node_state(inp, 0, 255)
    _gpu.assert_close(f["states"][0, 255], S, "f32", "deep chain fork state")


def test_commit_rejects_bad_paths_and_leaves_state():
    tree = [-1, 0, 0, 1, 1, 2, 2]
    case = W.gdn_case([tree] * 4, H=2, dk=64, dv=64, io="f32", state="f32", seed=2,
                      paths=[[0, 2, 6], [0, 3], [1, 3], [0]])
    path = case.path.clone()
    L = case.path_len.clone()
    L[3] = 0                                   # empty path
    inp = case.oracle_inputs()
    for mode, run in (("fork", _gpu.run_fork), ("wy", _gpu.run_wy)):
        r = run(case)
        S0 = _gpu.run_commit(case, mode, r, path=path, path_len=L)
        assert r["commit_err"].tolist() == [0, tv.TV_ERR_BAD_PATH, tv.TV_ERR_BAD_PATH, tv.TV_ERR_BAD_PATH]
        _gpu.assert_close(S0[0], G.node_state(inp, 0, 6)[0], "f32", f"{mode} good commit")
        for b in (1, 2, 3):
            assert torch.equal(S0[b], case.S0[b])


def test_host_side_argument_errors():
    case = W.small_fp32_case()
    x = _gpu.gdn_inputs(case)
    out = torch.empty_like(x["v"])
    st = torch.empty((1, 7, 2, 64, 64), device="cuda")
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(tv.TVError) as e:
        tv.tv_gdn_tree_verify_fork(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"],
                                   out, st, err, q_scale=float("nan"))
    assert e.value.status == tv.TV_ERR_INVALID_ARG
    q96 = torch.zeros((1, 7, 2, 96), device="cuda")
    with pytest.raises(tv.TVError) as e:
        tv.tv_gdn_tree_verify_fork(q96, q96, x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], out, st,
                                   err)
    assert e.value.status == tv.TV_ERR_UNSUPPORTED


def _stack_cases(kind):
    if kind == "bf16":
        return [W.stack_b64_layer(layer=l, B=8) for l in range(3)]
    rng = np.random.default_rng(31)
    trees = [W.random_tree(21, rng) for _ in range(4)]
    return [W.gdn_case(trees, H=3, dk=64, dv=64, io="f32", state="f32", seed=40 + l, path_max_len=6)
            for l in range(2)]


@pytest.mark.parametrize("kind", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["fork", "wy"])
def test_commit_of_a_layer_stack_in_one_launch_equals_per_layer_commits(mode, kind):
    # Independent layers sharing the trees and the accepted paths: tv_gdn_commit_layers on the
    # stacked tensors gives each layer's tv_gdn_commit result, bit for bit (bf16 d=128 and
    # fp32 d=64, so both element sizes enter the layer offsets).
    cases = _stack_cases(kind)
    c0 = cases[0]
    runs = [(_gpu.run_fork(c, keep_device=True) if mode == "fork" else _gpu.run_wy(c)) for c in cases]
    want = [_gpu.run_commit(c, mode, r, path=c0.path, path_len=c0.path_len) for c, r in zip(cases, runs)]
    S0 = torch.stack([r["inputs"]["S0"] for r in runs]).contiguous()
    err = torch.full((c0.shape[0],), 777, dtype=torch.int32, device="cuda:0")
    path, plen = _gpu.to_dev(c0.path), _gpu.to_dev(c0.path_len)
    parents = runs[0]["inputs"]["parents"]
    if mode == "fork":
        states = torch.stack([r["states"] for r in runs]).contiguous()
        tv.tv_gdn_commit_layers(tv.TV_MODE_FORK, path, plen, parents, S0, err, node_states=states)
    else:
        pv = torch.stack([r["pv_dev"] for r in runs]).contiguous()
        lg = torch.stack([r["lg_dev"] for r in runs]).contiguous()
        k = torch.stack([r["inputs"]["k"] for r in runs]).contiguous()
        tv.tv_gdn_commit_layers(tv.TV_MODE_WY, path, plen, parents, S0, err, pseudo_v=pv, log_gamma=lg, k=k)
    torch.cuda.synchronize()
    assert (err.cpu() == 0).all()
    for l in range(len(cases)):
        assert torch.equal(S0[l].cpu(), want[l])


@pytest.mark.parametrize("shape", ["shallow", "depth9", "depth15", "chain20", "chain64", "forest", "single"])
def test_small_tree_solve_variants(shape):
    """bf16, d=128 trees of at most 64 nodes (the row-per-thread TreeWY kernel): root paths held
    in registers for depths below 4, 10 and 16, the shared-memory solve of deeper trees, a forest
    and a single node, every output against the oracle."""
    rng = np.random.default_rng(77)
    if shape == "shallow":
        trees = [W.full_tree(3, 3)[:33], W.full_tree(2, 3)]
        trees = [t + [0] * (33 - len(t)) if len(t) < 33 else t for t in trees]
    elif shape == "depth9":
        trees = [W.chain(10) + [3, 4, 5], W.chain(10) + [0, 10, 11]]
    elif shape == "depth15":
        trees = [W.chain(16) + [2, 7], W.chain(16) + [0, 16]]
    elif shape == "chain20":
        trees = [W.chain(20), W.chain(20)]
    elif shape == "chain64":
        trees = [W.chain(64)]
    elif shape == "forest":
        trees = [[-1, -1, 0, 1, -1, 2, 3, 4, 4], [-1, 0, -1, 2, 1, -1, 5, 6, 0]]
    else:
        trees = [[-1], [-1]]
    case = W.gdn_case(trees, H=3, dk=128, dv=128, io="bf16", state="bf16", seed=len(shape))
    _check_all(case)


def test_wy_commit_with_a_wide_path_table_equals_the_staged_form():
    """The WY commit stages the S_0 tile and the path's rows in shared memory when both fit, and
    streams the tile through registers when a wide path table (min(Lmax, N) rows staged) leaves
    no room for it.  Both forms compute the same arithmetic: equal bit for bit, and equal to
    the oracle's commit within the bf16 rule."""
    rng = np.random.default_rng(21)
    trees = [W.random_tree(256, rng, max_children=4, max_depth=8) for _ in range(2)]
    # bf16 keys, fp32 state: a 64 KB tile, and 256 staged rows of 768 bytes with the wide table
    case = W.gdn_case(trees, H=2, dk=128, dv=128, io="bf16", state="f32", seed=21)
    w = _gpu.run_wy(case)
    assert (w["err"] == 0).all()
    narrow = _gpu.run_commit(case, "wy", w)
    B, Lmax = case.path.shape
    wide = torch.full((B, 256), -1, dtype=torch.int32)
    wide[:, :Lmax] = case.path
    wide_S0 = _gpu.run_commit(case, "wy", w, path=wide)
    assert (w["commit_err"] == 0).all()
    assert torch.equal(narrow, wide_S0)
    inp = case.oracle_inputs()
    for b in range(B):
        ref = G.node_state(inp, b, int(case.path[b, int(case.path_len[b]) - 1]))[0]
        _gpu.assert_close(narrow[b], ref, "bf16", "wy commit, staged and register forms", stored="f32")


def test_malformed_trees_in_a_wide_batch_fail_only_their_sequences():
    """At the batch-64 layer the fork walks plan their units as groups of CTAs tiling every
    sequence, so CTAs start and end inside sequences.  Two malformed trees -- one of them the
    last sequence -- fail alone, in the one-pass call and in both passes of the two-pass call;
    every other sequence equals a run without the faults bit for bit."""
    case = W.stack_b64_layer()
    clean = _gpu.run_fork(case, keep_device=True)
    bad = W.stack_b64_layer()
    for b in (17, 63):
        bad.parents[b, 20] = 30         # a later node: not allowed
    got = _gpu.run_fork(bad, keep_device=True)
    want_err = [tv.TV_ERR_BAD_TREE if b in (17, 63) else 0 for b in range(64)]
    assert got["err"].cpu().tolist() == want_err
    keep = [b for b in range(64) if b not in (17, 63)]
    assert torch.equal(got["out"][keep], clean["out"][keep])
    assert torch.equal(got["states"][keep], clean["states"][keep])
    x = _gpu.gdn_inputs(bad)
    B, N, H, dk, dv = bad.shape
    ws = torch.empty(tv.tv_gdn_fork_workspace_size(B, N, H, dv), dtype=torch.uint8, device="cuda")
    out = torch.full((B, N, H, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    states = torch.full((B, N, H, dv, dk), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.full((B,), 12345, dtype=torch.int32, device="cuda")
    tv.tv_gdn_tree_verify_fork_ws(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], out, states,
                                  ws, err)
    torch.cuda.synchronize()
    assert err.cpu().tolist() == want_err
    for b in (16, 18, 62):              # the neighbours of the malformed trees
        _gpu.assert_close(states[b].cpu(), W.f64(clean["states"][b].cpu()), "bf16",
                          "two-pass snapshots next to malformed trees", ref_rounded=True)
        assert not torch.isnan(out[b].float()).any()
    assert torch.isnan(states[17].float()).all() and torch.isnan(states[63].float()).all()
