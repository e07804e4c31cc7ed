"""GPU: TreeWY verify with the previous round's commit fused in, through the C ABI.

The fused call must equal tv_gdn_commit (WY mode) followed by tv_gdn_tree_verify_wy bit for bit
(same arithmetic), and the fp64 oracle's commit-then-verify within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import gdn as G

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _rounds(B=8, seed=0):
    prev = W.stack_b64_layer(B=B, seed=seed)
    rng = np.random.default_rng(seed + 17)
    trees = [W.random_tree(40, rng) for _ in range(B)]
    cur = W.gdn_case(trees, H=16, dk=128, dv=128, io="bf16", state="bf16", seed=seed + 9)
    return prev, cur


def _prev_round(prev):
    r = _gpu.run_wy(prev)
    assert (r["err"] == 0).all()
    return r


def _lazy(prev, r_prev, cur, S0, pv=None, lg=None, path=None):
    x = _gpu.gdn_inputs(cur)
    B, N, H, dk, dv = cur.shape
    out = torch.full((B, N, H, dv), float("nan"), dtype=torch.bfloat16, device=DEV)
    pv = torch.full((B, N, H, dv), float("nan"), dtype=torch.float32, device=DEV) if pv is None else pv
    lg = torch.full((B, N, H), float("nan"), dtype=torch.float32, device=DEV) if lg is None else lg
    err = torch.full((B,), 12345, dtype=torch.int32, device=DEV)
    tv.tv_gdn_tree_verify_wy_lazy(_gpu.to_dev(prev.path if path is None else path), _gpu.to_dev(prev.path_len),
                                  r_prev["inputs"]["parents"], r_prev["pv_dev"], r_prev["lg_dev"],
                                  r_prev["inputs"]["k"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], S0,
                                  x["parents"], out, pv, lg, err, q_scale=cur.q_scale)
    torch.cuda.synchronize()
    return dict(out=out.cpu(), pv=pv.cpu(), lg=lg.cpu(), err=err.cpu(), S0=S0.cpu())


def _reference(prev, r_prev, cur):
    S0 = r_prev["inputs"]["S0"].clone()
    err = torch.full((S0.shape[0],), 12345, dtype=torch.int32, device=DEV)
    tv.tv_gdn_commit(tv.TV_MODE_WY, _gpu.to_dev(prev.path), _gpu.to_dev(prev.path_len), r_prev["inputs"]["parents"],
                     S0, err, pseudo_v=r_prev["pv_dev"], log_gamma=r_prev["lg_dev"], k=r_prev["inputs"]["k"])
    x = _gpu.gdn_inputs(cur)
    x["S0"] = S0
    r = _gpu.run_wy(cur, inputs=x)
    return dict(out=r["out"], pv=r["pseudo_v"], lg=r["log_gamma"], S0=S0.cpu(), err=err.cpu())


def test_fused_commit_equals_commit_then_verify_and_the_oracle():
    prev, cur = _rounds()
    r_prev = _prev_round(prev)
    ref = _reference(prev, r_prev, cur)
    lz = _lazy(prev, r_prev, cur, r_prev["inputs"]["S0"].clone())
    assert (lz["err"] == 0).all() and (ref["err"] == 0).all()
    for key in ("S0", "out", "pv", "lg"):
        assert torch.equal(lz[key], ref[key]), key
    S0_ref, o_ref = G.verify_after_commit(prev.oracle_inputs(), prev.path.numpy(), prev.path_len.numpy(),
                                          cur.oracle_inputs())
    _gpu.assert_close(lz["S0"], S0_ref, "bf16", "committed S0")
    _gpu.assert_close(lz["out"], o_ref, "bf16", "outputs after the fused commit")


def test_outputs_may_share_memory_with_the_previous_round():
    prev, cur = _rounds(seed=3)
    r_prev = _prev_round(prev)
    ref = _reference(prev, r_prev, cur)
    pv_prev, lg_prev = r_prev["pv_dev"], r_prev["lg_dev"]
    lz = _lazy(prev, r_prev, cur, r_prev["inputs"]["S0"].clone(), pv=pv_prev, lg=lg_prev)  # in place
    assert torch.equal(lz["out"], ref["out"]) and torch.equal(lz["S0"], ref["S0"])
    assert torch.equal(lz["pv"], ref["pv"]) and torch.equal(lz["lg"], ref["lg"])


def test_bad_previous_path_skips_the_sequence():
    prev, cur = _rounds(B=3, seed=5)
    r_prev = _prev_round(prev)
    path = prev.path.clone()
    path[1, 0] = 5                                      # not a root of the previous tree
    S0 = r_prev["inputs"]["S0"].clone()
    before = S0.cpu()
    lz = _lazy(prev, r_prev, cur, S0, path=path)
    assert list(lz["err"]) == [0, tv.TV_ERR_BAD_PATH, 0]
    assert torch.equal(lz["S0"][1], before[1])


def test_unsupported_shapes_are_refused():
    case = W.small_fp32_case()                          # fp32, d = 64: no fused path
    x = _gpu.gdn_inputs(case)
    B, N, H, dk, dv = case.shape
    o = torch.empty((B, N, H, dv), dtype=torch.float32, device=DEV)
    pv = torch.empty((B, N, H, dv), dtype=torch.float32, device=DEV)
    lg = torch.empty((B, N, H), dtype=torch.float32, device=DEV)
    err = torch.empty((B,), dtype=torch.int32, device=DEV)
    path = _gpu.to_dev(case.path)
    with pytest.raises(tv.TVError) as e:
        tv.tv_gdn_tree_verify_wy_lazy(path, _gpu.to_dev(case.path_len), x["parents"], pv, lg, x["k"], x["q"], x["k"],
                                      x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], o, pv, lg, err)
    assert e.value.status == tv.TV_ERR_UNSUPPORTED
