"""Pins of the oracle's tree topology and of the synthetic tree shapes (CPU only)."""
import numpy as np
import pytest

import workloads as W
from oracle import tree as T


def _mask_fixture(golden):
    lines = golden("tree_mask_6node.txt")
    parents = [int(x) for x in lines[0].split(":")[1].split()]
    depths = [int(x) for x in lines[1].split(":")[1].split()]
    mask = np.array([[int(x) for x in ln.split()] for ln in lines[2:]], dtype=bool)
    return parents, depths, mask


def test_tree_mask_matches_printed_example(golden):
    parents, _, mask = _mask_fixture(golden)
    assert np.array_equal(T.tree_mask(parents), mask)


def test_depths_match_printed_example(golden):
    parents, depths, _ = _mask_fixture(golden)
    assert T.depths(parents) == depths


def test_mask_bits_pack_the_mask(golden):
    parents, _, mask = _mask_fixture(golden)
    bits = T.mask_bits(parents)
    assert bits.shape == (6, 1)
    for i in range(6):
        assert [(int(bits[i, 0]) >> j) & 1 for j in range(6)] == [int(x) for x in mask[i]]


def test_mask_bits_multiword():
    parents = W.chain(70)
    bits = T.mask_bits(parents)
    assert bits.shape == (70, 3)
    # a chain sees every earlier node: row i has exactly i+1 bits set, the low ones
    for i in range(70):
        total = sum(bin(int(w)).count("1") for w in bits[i])
        assert total == i + 1
        assert (int(bits[i, i // 32]) >> (i % 32)) & 1 == 1


def test_tree_sizes_from_pages(golden):
    for ln in golden("tree_sizes.txt"):
        br, without_root, with_root = [x.strip() for x in ln.split("|")]
        parents = W.branching_tree([int(x) for x in br.split(",")])
        assert len(parents) == int(with_root)
        assert len(parents) - 1 == int(without_root)
        assert T.is_valid_tree(parents)


def test_full_trees_match_workload_sizes():
    assert W.full_tree(2, 2) == [-1, 0, 0, 1, 1, 2, 2]
    assert len(W.full_tree(2, 3)) == 15
    assert len(W.full_tree(3, 3)) == 40
    assert T.depths(W.full_tree(3, 3)).count(3) == 27


def test_path_and_mask_agree_by_brute_force():
    rng = np.random.default_rng(3)
    for n in (1, 2, 3, 17, 40):
        parents = W.random_tree(n, rng)
        m = T.tree_mask(parents)
        d = T.depths(parents)
        for i in range(n):
            p = T.path_to(parents, i)
            assert p[-1] == i and parents[p[0]] == -1
            assert len(p) == d[i] + 1
            assert sorted(p) == list(np.nonzero(m[i])[0])
            # j visible to i  <=>  following parents from i reaches j
            for j in range(n):
                x, hit = i, False
                while x != -1:
                    hit |= x == j
                    x = parents[x]
                assert hit == m[i, j]


def test_random_tree_generator_shapes():
    rng = np.random.default_rng(0)
    for n in (15, 40, 64, 128, 256):
        t = W.random_tree(n, rng)
        assert len(t) == n and T.is_valid_tree(t)
        assert max(T.depths(t)) <= 8
        kids = T.children(t)
        assert all(1 <= len(v) <= 4 for p, v in kids.items() if p >= 0)


@pytest.mark.parametrize("parents,ok", [
    ([-1], True), ([-1, 0, 0, 1], True), ([-1, -1, 1], True),
    ([0], False), ([-1, 1], False), ([-1, 0, 3, 1], False), ([-2, 0], False), ([], False),
])
def test_tree_validity(parents, ok):
    assert T.is_valid_tree(parents) == ok


def test_path_validity():
    parents = [-1, 0, 0, 1, 1, 2]
    assert T.is_valid_path(parents, [0, 1, 3], 3)
    assert T.is_valid_path(parents, [0, 2, 5], 2)
    assert T.is_valid_path(parents, [0, -1, -1], 1)
    assert not T.is_valid_path(parents, [0, 2, 3], 3)      # 3 is not a child of 2
    assert not T.is_valid_path(parents, [1, 3], 2)         # does not start at a root
    assert not T.is_valid_path(parents, [0, 1], 0)         # empty
    assert not T.is_valid_path(parents, [0, 1], 3)         # longer than the buffer
    assert not T.is_valid_path(parents, [0, 9], 2)         # out of range


def test_accepted_path_generator_gives_valid_paths():
    rng = np.random.default_rng(1)
    t = W.full_tree(3, 3)
    for _ in range(50):
        p = W.random_accepted_path(t, rng, 4)
        assert 1 <= len(p) <= 4 and T.is_valid_path(t, p, len(p))


def test_candidate_chains_and_their_paths():
    """A root with chains numbered depth-first: a valid tree whose chain c starts at node
    1 + (lengths before c) and runs one node deeper per index; the generated paths run down
    one chain from the root."""
    lengths = W.CHAIN_LENGTHS
    t = W.candidate_chains(lengths)
    assert T.is_valid_tree(t) and len(t) == 1 + sum(lengths) == 40
    start = 1
    for n in lengths:
        assert t[start] == 0
        assert T.depths(t)[start:start + n] == list(range(1, n + 1))
        start += n
    rng = np.random.default_rng(2)
    for p in W.candidate_chain_paths(lengths, 200, rng):
        assert p[0] == 0 and T.is_valid_path(t, p, len(p))
        assert all(b == a + 1 for a, b in zip(p[1:], p[2:]))


# ----------------------------------------------------------------------------- accept walk
def test_accept_walk_hand_example():
    # 6-node tree of the handbook's printed example; tokens chosen so that the target at the
    # root predicts node 2's token, at node 2 predicts node 5's token, at node 5 nothing.
    parents = [-1, 0, 0, 1, 1, 2]
    draft = [9, 5, 6, 7, 8, 7]
    target = [6, 0, 7, 0, 0, 1]
    path, nxt = T.accept_walk(parents, draft, target, 8)
    assert path == [0, 2, 5] and nxt == 1


def test_accept_walk_chain_and_no_match():
    chain = [-1, 0, 1, 2, 3]
    draft = [10, 11, 12, 13, 14]
    assert T.accept_walk(chain, draft, [11, 12, 13, 14, 99], 8) == ([0, 1, 2, 3, 4], 99)
    assert T.accept_walk(chain, draft, [50, 12, 13, 14, 99], 8) == ([0], 50)   # nothing at the root
    assert T.accept_walk(chain, draft, [11, 12, 13, 14, 99], 3) == ([0, 1, 2], 13)  # stops at lmax
    assert T.accept_walk([-1], [3], [4], 1) == ([0], 4)


def test_accept_walk_prefers_lowest_numbered_matching_child():
    parents = [-1, 0, 0, 0, 2, 3]
    draft = [0, 7, 5, 5, 1, 2]     # nodes 2 and 3 both carry token 5
    target = [5, 0, 9, 2, 0, 0]    # the root predicts 5: node 2 wins over node 3
    assert T.accept_walk(parents, draft, target, 8) == ([0, 2], 9)


def test_accept_walk_properties_on_random_trees():
    rng = np.random.default_rng(5)
    for trial in range(60):
        n = int(rng.integers(1, 80))
        parents = W.random_tree(n, rng)
        draft = rng.integers(0, 4, size=n)     # small vocabulary: ties among siblings happen
        target = rng.integers(0, 4, size=n)
        lmax = int(rng.integers(1, 10))
        path, nxt = T.accept_walk(parents, draft, target, lmax)
        assert T.is_valid_path(parents, path, len(path)) and path[0] == 0 and len(path) <= lmax
        for a, b in zip(path, path[1:]):
            assert draft[b] == target[a]
            assert b == min(c for c in range(n) if parents[c] == a and draft[c] == target[a])
        last = path[-1]
        no_match = not any(parents[c] == last and draft[c] == target[last] for c in range(n))
        assert len(path) == lmax or no_match
        assert nxt == target[last]
