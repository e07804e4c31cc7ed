"""Pins of the oracle's block-table compaction (CPU only).

The handbook chapter 树形草稿与 EAGLE (note after the listing) allows keeping the accepted
path's KV by updating only the block table.  The oracle's ``kv_compact_remap`` exchanges the
table entries of whole destination blocks whose kept entries all come from one source block
at the same rows, and moves the rest.  Its pins:

* hand-worked cases (``golden/kv_remap_two_chains.txt``);
* on random trees, prefixes and tables, the logical contents of slots [0, new length) read
  through the new table equal those of the moving compaction (itself pinned in
  ``test_oracle_attention``) read through the old table;
* the new table row is a permutation of the old one and leaves the prefix's blocks alone;
* the plan agrees with a second statement of the rule, written from the physical slots.
"""
import os

import numpy as np
import pytest

import workloads as W
from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kv_remap_two_chains.txt")


def _ints(spec: str) -> list[int]:
    out = []
    for part in spec.split(","):
        if not part:
            continue
        if ".." in part:
            lo, hi = part.split("..")
            out.extend(range(int(lo), int(hi) + 1))
        else:
            out.append(int(part))
    return out


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for ln in f:
            if not ln.startswith("case "):
                continue
            fields = dict(kv.split("=", 1) for kv in ln.split()[1:])
            cases.append(fields)
    return cases


def _tree(spec: str) -> list[int]:
    """``chains:a,b,...`` = a root with chains of those lengths; ``forest:a,b`` = two chains,
    each its own root; ``parents:...`` = the parents array itself."""
    kind, lengths = spec.split(":")
    if kind == "parents":
        return _ints(lengths)
    lengths = [int(x) for x in lengths.split(",")]
    if kind == "forest":
        n1, n2 = lengths
        return W.chain(n1) + [-1] + [n1 + j for j in range(n2 - 1)]
    return W.candidate_chains(lengths)


def _case(tree, P, path, table_row, Hkv=2, hd=4, seed=0):
    """One sequence with a given table row; every physical row holds distinct values."""
    nb = max(table_row) + 2
    rng = np.random.default_rng(seed)
    kc = rng.standard_normal((nb, Hkv, 16, hd))
    vc = rng.standard_normal((nb, Hkv, 16, hd))
    return (kc, vc, np.array([table_row], dtype=np.int64), np.array([P]), np.array([tree]),
            np.array([path]), np.array([len(path)]))


@pytest.mark.parametrize("fields", _golden_cases(), ids=lambda f: f"{f['tree']}-P{f['P']}-{f['path']}")
def test_golden_cases(fields):
    tree = _tree(fields["tree"])
    P = int(fields["P"])
    path = _ints(fields["path"])
    before = _ints(fields["before"])
    kc, vc, table, plen, par, pth, L = _case(tree, P, path, before)
    kc2, vc2, new_table, smap, new_len, remapped = A.kv_compact_remap(kc, vc, table, plen, par, pth, L)
    assert new_table[0].tolist() == _ints(fields["after"])
    assert int(remapped[0]) == int(fields["remapped"])
    assert int(new_len[0]) == int(fields["new_len"])
    taken = {m for m, _ in A.remap_plan(P, path, len(path))}
    moved = [r for r in range(len(path)) if (P + r) // 16 not in taken]
    assert moved == _ints(fields["moved"])
    # the logical view equals the moving compaction's
    kc3, vc3, smap3, new_len3 = A.kv_compact(kc, vc, table, plen, par, pth, L)
    n = int(new_len[0])
    assert np.array_equal(A.logical_rows(kc2, new_table[0], n), A.logical_rows(kc3, table[0], n))
    assert np.array_equal(A.logical_rows(vc2, new_table[0], n), A.logical_rows(vc3, table[0], n))
    assert np.array_equal(smap, smap3) and np.array_equal(new_len, new_len3)


def _random_cases(seed: int, count: int):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        kind = i % 4
        if kind == 0:
            lengths = rng.choice([5, 15, 16, 17, 32, 40], size=int(rng.integers(1, 4)))
            tree = W.candidate_chains([int(x) for x in lengths])
        elif kind == 1:
            tree = W.random_tree(int(rng.integers(2, 90)), rng)
        elif kind == 2:     # a forest of chains, each chain its own root
            n1, n2 = int(rng.integers(1, 40)), int(rng.integers(1, 40))
            tree = W.chain(n1) + [-1] + [n1 + j for j in range(n2 - 1)]
        else:
            tree = W.candidate_chains([16 * int(rng.integers(1, 3)), int(rng.choice([16, 33, 48, 60]))])
        N = len(tree)
        roots = [i for i, p in enumerate(tree) if p == -1]
        path = [int(rng.choice(roots))]
        stop = int(rng.integers(1, N + 1))
        while len(path) < stop:
            kids = [c for c in range(N) if tree[c] == path[-1]]
            if not kids:
                break
            path.append(int(rng.choice(kids)))
        P = int(rng.choice([0, 1, 7, 15, 16, 17, 31, 32, 33, int(rng.integers(0, 200))]))
        nblk = (P + N + 15) // 16 + int(rng.integers(0, 3))
        table_row = rng.permutation(nblk + 4)[:nblk].tolist()
        out.append((tree, P, path, table_row, i))
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_logical_view_equals_moving_compaction(seed):
    exchanged = 0
    for tree, P, path, table_row, i in _random_cases(seed, 60):
        kc, vc, table, plen, par, pth, L = _case(tree, P, path, table_row, seed=i)
        kc2, vc2, new_table, smap, new_len, remapped = A.kv_compact_remap(kc, vc, table, plen, par, pth, L)
        kc3, vc3, smap3, new_len3 = A.kv_compact(kc, vc, table, plen, par, pth, L)
        n = int(new_len[0])
        assert n == P + len(path) and n == int(new_len3[0])
        assert np.array_equal(A.logical_rows(kc2, new_table[0], n), A.logical_rows(kc3, table[0], n))
        assert np.array_equal(A.logical_rows(vc2, new_table[0], n), A.logical_rows(vc3, table[0], n))
        assert np.array_equal(smap, smap3)
        # a permutation of the row that leaves the blocks holding prefix slots alone
        assert sorted(new_table[0].tolist()) == sorted(table_row)
        first = -(-P // 16)
        assert new_table[0][:first].tolist() == table_row[:first]
        exchanged += int(remapped[0])
    assert exchanged > 0


def _plan_from_slots(P, path, L, table_row):
    """The rule restated on physical slots: block m (wholly past the prefix) is taken over when
    all its kept entries' source slots lie in one other block at the destination's rows."""
    plan = []
    for m in range(len(table_row)):
        if 16 * m < P:
            continue
        rows = [r for r in range(L) if (P + r) // 16 == m]
        if not rows:
            continue
        srcs = {A.physical_slot(table_row, P + path[r]) // 16 for r in rows}
        same_rows = all((P + path[r]) % 16 == (P + r) % 16 for r in rows)
        src_logical = {(P + path[r]) // 16 for r in rows}
        if len(srcs) == 1 and same_rows and src_logical != {m}:
            plan.append((m, src_logical.pop() - m))
    return plan


@pytest.mark.parametrize("seed", [3, 4])
def test_plan_matches_physical_statement(seed):
    for tree, P, path, table_row, _ in _random_cases(seed, 80):
        assert A.remap_plan(P, path, len(path)) == _plan_from_slots(P, path, len(path), table_row)


def test_invalid_path_leaves_everything():
    tree = W.candidate_chains([16, 16])
    kc, vc, table, plen, par, pth, L = _case(tree, 15, [0, 17, 19], [5, 3, 9])
    kc2, vc2, new_table, smap, new_len, remapped = A.kv_compact_remap(kc, vc, table, plen, par, pth, L)
    assert np.array_equal(kc2, kc) and np.array_equal(vc2, vc)
    assert np.array_equal(new_table, table) and int(new_len[0]) == 15 and int(remapped[0]) == 0
    assert (smap == -1).all()
