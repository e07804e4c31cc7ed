"""GPU vs oracle: tree topology (depth and packed tree-mask bits), bit-exact."""
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
