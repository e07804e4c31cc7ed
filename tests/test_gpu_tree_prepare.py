"""GPU vs oracle: tree topology (depth, packed tree-mask bits, root-to-node paths, maximum depth),
bit-exact."""
import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import tree as T

pytestmark = pytest.mark.gpu


def _pad(trees):
    n = max(len(t) for t in trees)
    assert all(len(t) == n for t in trees)
    return torch.tensor(trees, dtype=torch.int32)


def test_printed_example(golden):
    lines = golden("tree_mask_6node.txt")
    parents = [int(x) for x in lines[0].split(":")[1].split()]
    depths = [int(x) for x in lines[1].split(":")[1].split()]
    mask = np.array([[int(x) for x in ln.split()] for ln in lines[2:]], dtype=bool)
    r = _gpu.run_tree_prepare(_pad([parents]))
    assert int(r["err"][0]) == 0
    assert r["depth"][0].tolist() == depths
    got = np.array([[(int(r["mask_bits"][0, i, 0]) >> j) & 1 for j in range(6)] for i in range(6)], dtype=bool)
    assert np.array_equal(got, mask)


@pytest.mark.parametrize("n", [1, 2, 3, 31, 32, 33, 64, 255, 256])
def test_random_trees_bit_exact(n):
    rng = np.random.default_rng(n)
    trees = [W.random_tree(n, rng) for _ in range(3)] + [W.chain(n), [-1] * n]
    r = _gpu.run_tree_prepare(_pad(trees))
    assert (r["err"] == 0).all()
    for b, t in enumerate(trees):
        assert r["depth"][b].tolist() == T.depths(t)
        assert np.array_equal(r["mask_bits"][b], T.mask_bits(t))


def test_malformed_trees_flagged():
    good = [-1, 0, 0, 1]
    trees = [good, [-1, 0, 3, 1], [-1, -2, 0, 1], [0, 0, 0, 0], [-1, 0, 1, 3]]
    r = _gpu.run_tree_prepare(_pad(trees))
    assert r["err"].tolist() == [0] + [tv.TV_ERR_BAD_TREE] * 4
    assert r["depth"][0].tolist() == [0, 1, 1, 2]


def _check_paths(trees, r, cap):
    for b, t in enumerate(trees):
        assert int(r["max_depth"][b]) == max(T.depths(t))
        for i in range(len(t)):
            want = T.path_to(t, i)
            assert list(r["paths"][b, i, :len(want)]) == want
            assert (r["paths"][b, i, len(want):cap] == -1).all()


@pytest.mark.parametrize("n", [1, 7, 40, 100, 256])
def test_paths_and_max_depth_bit_exact(n):
    rng = np.random.default_rng(100 + n)
    trees = [W.random_tree(n, rng) for _ in range(3)] + [[-1] * n]
    cap = max(max(T.depths(t)) for t in trees) + 1
    r = _gpu.run_tree_prepare(_pad(trees), path_cap=cap + 2)    # room to spare: -1 padded
    assert (r["err"] == 0).all()
    _check_paths(trees, r, cap + 2)
    r = _gpu.run_tree_prepare(_pad(trees), path_cap=cap)        # exactly deep enough
    assert (r["err"] == 0).all()
    _check_paths(trees, r, cap)


def test_path_capacity_too_small_only_fails_that_sequence():
    trees = [W.chain(9), W.full_tree(2, 3)[:9]]                 # depths 8 and 3
    r = _gpu.run_tree_prepare(_pad(trees), path_cap=4)
    assert r["err"].tolist() == [tv.TV_ERR_UNSUPPORTED, 0]
    assert r["depth"][0].tolist() == list(range(9))             # still written
    assert r["max_depth"].tolist() == [8, 3]
    for i in range(9):
        want = T.path_to(trees[1], i)
        assert list(r["paths"][1, i, :len(want)]) == want


def test_optional_outputs_argument_checks():
    L = tv.lib
    p = torch.zeros((1, 4), dtype=torch.int32, device="cuda:0")
    o = torch.zeros(64, dtype=torch.int32, device="cuda:0")
    P, O = p.data_ptr(), o.data_ptr()
    assert L.tv_tree_prepare(P, 1, 4, O, O, O, 0, None, O, None) == tv.TV_ERR_INVALID_ARG   # paths, cap 0
    assert L.tv_tree_prepare(P, 1, 4, O, O, O + 2, 3, None, O, None) == tv.TV_ERR_INVALID_ARG  # misaligned
    assert L.tv_tree_prepare(P, 1, 4, O, O, None, 0, None, O, None) == tv.TV_OK
    torch.cuda.synchronize()
