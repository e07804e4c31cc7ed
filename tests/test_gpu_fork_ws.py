"""GPU vs fp64 oracle: the two-pass fork verify (TreeWY outputs and w, then every snapshot from its
parent's), through the C ABI."""
import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import gdn as G

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run_ws(case):
    x = _gpu.gdn_inputs(case)
    B, N, H, dk, dv = case.shape
    out = torch.full((B, N, H, dv), float("nan"), dtype=x["q"].dtype, device=DEV)
    states = torch.full((B, N, H, dv, dk), float("nan"), dtype=x["S0"].dtype, device=DEV)
    ws = torch.empty(tv.tv_gdn_fork_workspace_size(B, N, H, dv), dtype=torch.uint8, device=DEV)
    err = torch.full((B,), 12345, dtype=torch.int32, device=DEV)
    tv.tv_gdn_tree_verify_fork_ws(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], out,
                                  states, ws, err, q_scale=case.q_scale)
    torch.cuda.synchronize()
    return dict(out=out.cpu(), states=states.cpu(), err=err.cpu(), inputs=x)


def _check(case):
    io = case.io
    inp = case.oracle_inputs()
    o_ref, S_ref = G.verify(inp)
    r = _run_ws(case)
    assert (r["err"] == 0).all(), r["err"]
    _gpu.assert_close(r["out"], o_ref, io, "two-pass fork o")
    _gpu.assert_close(r["states"], S_ref, io if case.state == io else "bf16", "two-pass fork states")
    # the commit of fork mode takes its snapshots
    S0 = _gpu.run_commit(case, "fork", dict(states=r["states"], inputs=r["inputs"]))
    _gpu.assert_close(S0, G.commit(inp, case.path.numpy(), case.path_len.numpy()), io, "commit")


def test_small_fp32_layer():
    _check(W.small_fp32_case())


@pytest.mark.parametrize("io,state", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("d", [64, 128])
def test_random_trees(io, state, d):
    rng = np.random.default_rng(d)
    trees = [W.random_tree(37, rng) for _ in range(3)]
    _check(W.gdn_case(trees, H=2, dk=d, dv=d, io=io, state=state, seed=d + 1))


def test_stack_layer_sampled_and_against_the_one_pass_fork():
    case = W.stack_b64_layer()
    r = _run_ws(case)
    f = _gpu.run_fork(case)
    assert (r["err"] == 0).all()
    # both forms of the same snapshots: within the tolerance of each other and of the oracle
    _gpu.assert_close(r["states"][:4], W.f64(f["states"][:4]), "bf16", "two-pass vs one-pass states",
                      ref_rounded=True)
    inp = case.oracle_inputs()
    rng = np.random.default_rng(3)
    got, ref = [], []
    for b in (0, 17, 63):
        for i in sorted(set([0, 39] + list(rng.choice(40, 5, replace=False)))):
            S, o = G.node_state(inp, b, int(i))
            got.append(W.f64(r["states"][b, i]))
            ref.append(S)
    _gpu.assert_close(np.stack(got), np.stack(ref), "bf16", "two-pass states (sampled)", stored="bf16")


def test_treewy_path_capacity_limit_is_reported():
    case = W.gdn_case([W.chain(256)], H=1, dk=64, dv=64, io="f32", state="f32", seed=1)
    r = _run_ws(case)
    assert int(r["err"][0]) == tv.TV_ERR_UNSUPPORTED


def _run_split(case, max_ctas_per_sm, side_stream=True):
    """tv_gdn_tree_verify_wy on the current stream, tv_gdn_fork_materialize on a second one."""
    x = _gpu.gdn_inputs(case)
    B, N, H, dk, dv = case.shape
    out = torch.full((B, N, H, dv), float("nan"), dtype=x["q"].dtype, device=DEV)
    states = torch.full((B, N, H, dv, dk), float("nan"), dtype=x["S0"].dtype, device=DEV)
    pv = torch.empty((B, N, H, dv), dtype=torch.float32, device=DEV)
    lg = torch.empty((B, N, H), dtype=torch.float32, device=DEV)
    err = torch.full((B,), 12345, dtype=torch.int32, device=DEV)
    tv.tv_gdn_tree_verify_wy(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], out, pv, lg,
                             err, q_scale=case.q_scale)
    side = torch.cuda.Stream() if side_stream else torch.cuda.current_stream()
    side.wait_stream(torch.cuda.current_stream())
    tv.tv_gdn_fork_materialize(x["k"], x["alpha"], x["S0"], x["parents"], pv, states, err,
                               max_ctas_per_sm=max_ctas_per_sm, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    return dict(out=out.cpu(), states=states.cpu(), err=err.cpu())


@pytest.mark.parametrize("io,state,d", [("f32", "f32", 64), ("bf16", "bf16", 128), ("bf16", "f32", 128)])
@pytest.mark.parametrize("max_ctas_per_sm", [0, 1, 3])
def test_split_passes_equal_the_two_pass_call(io, state, d, max_ctas_per_sm):
    # Same kernels as tv_gdn_tree_verify_fork_ws: outputs and snapshots bit for bit, whatever
    # the CTA cap (it only changes how items are spread over CTAs).
    rng = np.random.default_rng(5 + d)
    trees = [W.random_tree(41, rng) for _ in range(5)]
    case = W.gdn_case(trees, H=3, dk=d, dv=d, io=io, state=state, seed=9)
    want = _run_ws(case)
    got = _run_split(case, max_ctas_per_sm)
    assert (got["err"] == 0).all() and (want["err"] == 0).all()
    assert torch.equal(got["out"], want["out"])
    assert torch.equal(got["states"], want["states"])


def test_split_stack_layer_on_a_side_stream_matches_the_oracle_sampled():
    case = W.stack_b64_layer()
    got = _run_split(case, 2)
    want = _run_ws(case)
    assert (got["err"] == 0).all()
    assert torch.equal(got["states"], want["states"])
    inp = case.oracle_inputs()
    ref = [G.node_state(inp, b, i)[0] for b, i in ((0, 0), (31, 12), (63, 39))]
    _gpu.assert_close(torch.stack([got["states"][b, i] for b, i in ((0, 0), (31, 12), (63, 39))]),
                      np.stack(ref), "bf16", "split fork states (sampled)")


def test_materialize_skips_sequences_the_verify_rejected():
    rng = np.random.default_rng(8)
    case = W.gdn_case([W.random_tree(12, rng) for _ in range(3)], H=2, dk=64, dv=64, io="f32", state="f32",
                      seed=4)
    case.parents[1, 5] = 7          # a later node: not allowed
    r = _run_split(case, 0)
    assert list(r["err"].numpy()) == [0, tv.TV_ERR_BAD_TREE, 0]
    assert torch.isnan(r["states"][1]).all()                 # untouched
    assert not torch.isnan(r["states"][0]).any() and not torch.isnan(r["states"][2]).any()
    want = _run_ws(case)
    assert torch.equal(r["states"][0], want["states"][0]) and torch.equal(r["states"][2], want["states"][2])


def test_materialize_argument_errors():
    L = tv.lib
    p = torch.zeros(64, dtype=torch.int32, device=DEV)
    ok = [p.data_ptr()] * 5
    assert L.tv_gdn_fork_materialize(None, *ok[1:], 1, 4, 1, 64, 64, 0, 0, 0, p.data_ptr(), p.data_ptr(),
                                     None) == tv.TV_ERR_INVALID_ARG
    assert L.tv_gdn_fork_materialize(*ok, 1, 4, 1, 64, 64, 0, 0, -1, p.data_ptr(), p.data_ptr(),
                                     None) == tv.TV_ERR_INVALID_ARG
    assert L.tv_gdn_fork_materialize(*ok, 1, 257, 1, 64, 64, 0, 0, 0, p.data_ptr(), p.data_ptr(),
                                     None) == tv.TV_ERR_UNSUPPORTED
    assert L.tv_gdn_fork_materialize(*ok, 1, 4, 1, 64, 64, 0, 1, 0, p.data_ptr(), p.data_ptr(),
                                     None) == tv.TV_ERR_UNSUPPORTED
