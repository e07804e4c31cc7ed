"""GPU vs oracle: fork mode with selective snapshots and its replaying commit, through the C ABI.

Outputs and the kept snapshots are those of the plain fork verify, bit for bit (same kernel,
same arithmetic); the slot map is exact; the commit is the accepted node's state, checked
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import gdn as G

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _confidence(B, N, seed, frac_high=0.5):
    rng = np.random.default_rng(seed)
    c = np.where(rng.random((B, N)) < frac_high, rng.uniform(0.951, 1.0, (B, N)), rng.uniform(0.0, 0.95, (B, N)))
    return torch.from_numpy(c.astype(np.float32))


def _run_selective(case, conf, threshold, capacity):
    x = _gpu.gdn_inputs(case)
    B, N, H, dk, dv = case.shape
    out = torch.full((B, N, H, dv), float("nan"), dtype=x["q"].dtype, device=DEV)
    states = torch.full((B, capacity, H, dv, dk), float("nan"), dtype=x["S0"].dtype, device=DEV)
    slot = torch.full((B, N), 777, dtype=torch.int32, device=DEV)
    err = torch.full((B,), 12345, dtype=torch.int32, device=DEV)
    tv.tv_gdn_tree_verify_fork_selective(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"],
                                         conf.to(DEV), threshold, out, states, slot, err, q_scale=case.q_scale)
    S0 = x["S0"].clone()
    cerr = torch.full((B,), 12345, dtype=torch.int32, device=DEV)
    tv.tv_gdn_commit_selective(_gpu.to_dev(case.path), _gpu.to_dev(case.path_len), x["parents"], states, slot,
                               x["k"], x["v"], x["alpha"], x["beta"], S0, cerr)
    torch.cuda.synchronize()
    return dict(out=out.cpu(), states=states.cpu(), slot=slot.cpu().numpy(), err=err.cpu().numpy(),
                S0=S0.cpu(), commit_err=cerr.cpu().numpy())


def _check(case, conf, threshold, io):
    B, N = case.shape[0], case.shape[1]
    slots = [G.selective_slots(conf[b].numpy(), threshold, N)[0] for b in range(B)]
    capacity = max(1, max(sum(s >= 0 for s in row) for row in slots))
    sel = _run_selective(case, conf, threshold, capacity)
    full = _gpu.run_fork(case)
    assert (sel["err"] == 0).all(), sel["err"]
    assert (sel["commit_err"] == 0).all(), sel["commit_err"]
    assert torch.equal(sel["out"], full["out"])                           # outputs: same kernel
    for b in range(B):
        assert list(sel["slot"][b]) == slots[b]
        for i in range(N):
            if slots[b][i] >= 0:
                assert torch.equal(sel["states"][b, slots[b][i]], full["states"][b, i])
    ref = G.commit(case.oracle_inputs(), case.path.numpy(), case.path_len.numpy())
    _gpu.assert_close(sel["S0"], ref, io, "selective commit")


@pytest.mark.parametrize("io,state", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
def test_random_trees_half_confident(io, state):
    rng = np.random.default_rng(7)
    N = 47
    trees = [W.random_tree(N, rng) for _ in range(6)]
    case = W.gdn_case(trees, H=3, dk=64, dv=64, io=io, state=state, seed=11, path_max_len=8)
    _check(case, _confidence(6, N, 3), 0.95, io)


def test_stack_layer_shapes_all_kept_and_none_kept():
    case = W.stack_b64_layer(B=8)
    N = case.shape[1]
    _check(case, _confidence(8, N, 5), 0.95, "bf16")
    _check(case, torch.full((8, N), 0.5), 0.95, "bf16")     # every node keeps its snapshot
    _check(case, torch.full((8, N), 0.99), 0.95, "bf16")    # none does: commits replay from S_0


def test_capacity_overflow_skips_the_sequence_and_commit_replays_from_s0():
    case = W.small_fp32_case()
    B, N = case.shape[0], case.shape[1]
    conf = torch.zeros((B, N))                                # all 7 nodes want a snapshot
    sel = _run_selective(case, conf, 0.95, 3)
    assert (sel["err"] == tv.TV_ERR_CAPACITY).all()
    assert (sel["slot"] == -1).all()
    assert (sel["commit_err"] == 0).all()
    ref = G.commit(case.oracle_inputs(), case.path.numpy(), case.path_len.numpy())
    _gpu.assert_close(sel["S0"], ref, "f32", "commit after a skipped verify")


def _run_selective_two_pass(case, conf, threshold, capacity):
    """tv_gdn_tree_verify_wy, then the selective snapshot pass on a second stream."""
    x = _gpu.gdn_inputs(case)
    B, N, H, dk, dv = case.shape
    out = torch.full((B, N, H, dv), float("nan"), dtype=x["q"].dtype, device=DEV)
    pv = torch.empty((B, N, H, dv), dtype=torch.float32, device=DEV)
    lg = torch.empty((B, N, H), dtype=torch.float32, device=DEV)
    states = torch.full((B, capacity, H, dv, dk), float("nan"), dtype=x["S0"].dtype, device=DEV)
    slot = torch.full((B, N), 777, dtype=torch.int32, device=DEV)
    err = torch.full((B,), 12345, dtype=torch.int32, device=DEV)
    tv.tv_gdn_tree_verify_wy(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], out, pv, lg, err,
                             q_scale=case.q_scale)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    tv.tv_gdn_fork_materialize_selective(x["k"], x["alpha"], x["S0"], x["parents"], pv, conf.to(DEV), threshold,
                                         states, slot, err, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    S0 = x["S0"].clone()
    cerr = torch.full((B,), 12345, dtype=torch.int32, device=DEV)
    tv.tv_gdn_commit_selective(_gpu.to_dev(case.path), _gpu.to_dev(case.path_len), x["parents"], states, slot,
                               x["k"], x["v"], x["alpha"], x["beta"], S0, cerr)
    torch.cuda.synchronize()
    return dict(out=out.cpu(), states=states.cpu(), slot=slot.cpu().numpy(), err=err.cpu().numpy(), S0=S0.cpu(),
                commit_err=cerr.cpu().numpy())


def _run_fork_ws(case):
    x = _gpu.gdn_inputs(case)
    B, N, H, dk, dv = case.shape
    out = torch.empty((B, N, H, dv), dtype=x["q"].dtype, device=DEV)
    states = torch.empty((B, N, H, dv, dk), dtype=x["S0"].dtype, device=DEV)
    ws = torch.empty(tv.tv_gdn_fork_workspace_size(B, N, H, dv), dtype=torch.uint8, device=DEV)
    err = torch.zeros((B,), dtype=torch.int32, device=DEV)
    tv.tv_gdn_tree_verify_fork_ws(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], out, states,
                                  ws, err, q_scale=case.q_scale)
    torch.cuda.synchronize()
    return dict(out=out.cpu(), states=states.cpu())


@pytest.mark.parametrize("io,state", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
def test_two_pass_selective_equals_the_two_pass_fork_at_kept_nodes(io, state):
    rng = np.random.default_rng(17)
    N = 47
    trees = [W.random_tree(N, rng) for _ in range(6)]
    case = W.gdn_case(trees, H=3, dk=64, dv=64, io=io, state=state, seed=12, path_max_len=8)
    conf = _confidence(6, N, 4)
    slots = [G.selective_slots(conf[b].numpy(), 0.95, N)[0] for b in range(6)]
    capacity = max(1, max(sum(s >= 0 for s in row) for row in slots))
    sel = _run_selective_two_pass(case, conf, 0.95, capacity)
    full = _run_fork_ws(case)
    assert (sel["err"] == 0).all() and (sel["commit_err"] == 0).all()
    assert torch.equal(sel["out"], full["out"])
    for b in range(6):
        assert list(sel["slot"][b]) == slots[b]
        for i in range(N):
            if slots[b][i] >= 0:
                assert torch.equal(sel["states"][b, slots[b][i]], full["states"][b, i])
    ref = G.commit(case.oracle_inputs(), case.path.numpy(), case.path_len.numpy())
    _gpu.assert_close(sel["S0"], ref, io, "two-pass selective commit")


def test_two_pass_selective_stack_layer_and_capacity_overflow():
    case = W.stack_b64_layer(B=8)
    N = case.shape[1]
    conf = _confidence(8, N, 6)
    slots = [G.selective_slots(conf[b].numpy(), 0.95, N)[0] for b in range(8)]
    kept = [sum(s >= 0 for s in row) for row in slots]
    capacity = sorted(kept)[3]                     # the fuller half of the sequences overflows
    sel = _run_selective_two_pass(case, conf, 0.95, capacity)
    ref = G.commit(case.oracle_inputs(), case.path.numpy(), case.path_len.numpy())
    for b in range(8):
        if kept[b] > capacity:
            assert sel["err"][b] == tv.TV_ERR_CAPACITY and (sel["slot"][b] == -1).all()
        else:
            assert sel["err"][b] == 0 and list(sel["slot"][b]) == slots[b]
    assert (sel["commit_err"] == 0).all()          # every commit replays from what was kept
    _gpu.assert_close(sel["S0"], ref, "bf16", "two-pass selective commit, overflow included")


def test_two_pass_selective_sequence_rejected_by_the_verify_keeps_nothing():
    rng = np.random.default_rng(21)
    case = W.gdn_case([W.random_tree(12, rng) for _ in range(3)], H=2, dk=64, dv=64, io="f32", state="f32", seed=2)
    case.parents[1, 5] = 7
    sel = _run_selective_two_pass(case, torch.zeros((3, 12)), 0.95, 12)
    assert list(sel["err"]) == [0, tv.TV_ERR_BAD_TREE, 0]
    assert (sel["slot"][1] == -1).all()
    assert list(sel["slot"][0]) == list(range(12)) and list(sel["slot"][2]) == list(range(12))
