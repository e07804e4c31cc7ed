"""GPU vs fp64 oracle: compaction that exchanges whole blocks of the block table
(``tv_kv_compact_remap``), through the C ABI.

Every output is compared exactly: the new table rows, the exchange counts, the slot map, the
new lengths and the caches (bf16 rows are copied, never computed).
"""
import numpy as np
import pytest
import torch

import _gpu
import test_oracle_compact_remap as PR
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import attention as A

pytestmark = pytest.mark.gpu


def _single(tree, P, path, table_row, Hkv, hd, seed):
    """One sequence over its own small cache pool (bf16), the table row given."""
    nb = max(table_row) + 2
    rng = np.random.default_rng(seed)
    kc = W.round_to(rng.standard_normal((nb, Hkv, 16, hd)), "bf16")
    vc = W.round_to(rng.standard_normal((nb, Hkv, 16, hd)), "bf16")
    Lmax = len(path) + 2
    return dict(k_cache=kc, v_cache=vc, block_table=torch.tensor([table_row], dtype=torch.int32),
                prefix_len=torch.tensor([P], dtype=torch.int32),
                parents=torch.tensor([tree], dtype=torch.int32),
                path=torch.tensor([path + [-1] * (Lmax - len(path))], dtype=torch.int32),
                path_len=torch.tensor([len(path)], dtype=torch.int32))


def _oracle(x):
    return A.kv_compact_remap(W.f64(x["k_cache"]), W.f64(x["v_cache"]), x["block_table"].numpy(),
                              x["prefix_len"].numpy(), x["parents"].numpy(), x["path"].numpy(),
                              x["path_len"].numpy())


def _run(x):
    return _gpu.run_compact_remap(x["k_cache"], x["v_cache"], x["block_table"], x["prefix_len"],
                                  x["parents"], x["path"], x["path_len"])


def _compare(res, ref):
    kc, vc, table, smap, new_len, remapped = ref
    assert np.array_equal(res["table"], table)
    assert np.array_equal(res["remapped"], remapped)
    assert np.array_equal(res["new_len"], new_len)
    assert np.array_equal(res["slot_map"], smap)
    assert np.array_equal(_gpu.f32np(res["k_cache"].cpu()), kc)
    assert np.array_equal(_gpu.f32np(res["v_cache"].cpu()), vc)


@pytest.mark.parametrize("hd", [64, 256])
@pytest.mark.parametrize("fields", PR._golden_cases(), ids=lambda f: f"{f['tree']}-P{f['P']}")
def test_hand_worked_cases(fields, hd):
    tree = PR._tree(fields["tree"])
    x = _single(tree, int(fields["P"]), PR._ints(fields["path"]), PR._ints(fields["before"]), Hkv=4, hd=hd,
                seed=int(fields["P"]))
    res = _run(x)
    assert (res["err"] == 0).all()
    assert res["table"][0].tolist() == PR._ints(fields["after"])
    assert int(res["remapped"][0]) == int(fields["remapped"])
    _compare(res, _oracle(x))


def _pad_tree(tree, N):
    """Extra leaves under the root up to N nodes (the shape stays a valid tree)."""
    return list(tree) + [0] * (N - len(tree))


@pytest.mark.parametrize("seed", [0, 1])
def test_mixed_batch_shared_pool(seed):
    """Twelve sequences over one permuted block pool: candidate chains, forests and random
    trees, prefixes on and off block boundaries; every output against the oracle."""
    rng = np.random.default_rng(seed + 50)
    N = 72
    trees, paths, prefix = [], [], []
    for i in range(12):
        kind = i % 4
        if kind == 0:
            t = W.candidate_chains([16, 16, 16, 16])
            c = int(rng.integers(0, 4))
            L = int(rng.integers(1, 18))
            path = [0] + list(range(1 + 16 * c, 1 + 16 * c + L - 1))
        elif kind == 1:
            t = W.candidate_chains([16, 48])
            L = int(rng.integers(10, 50))
            path = [0] + list(range(17, 17 + L - 1))
        elif kind == 2:
            t = W.chain(32) + [-1] + [32 + j for j in range(31)]
            L = int(rng.integers(1, 33))
            path = list(range(32, 32 + L))
        else:
            t = W.random_tree(N, rng)
            path = W.random_accepted_path(t, rng)
        trees.append(_pad_tree(t, N))
        paths.append(path)
        prefix.append(int(rng.choice([0, 1, 15, 16, 17, int(rng.integers(2, 300))])))
    case = W.attn_case(trees, prefix, Hq=4, Hkv=4, hd=128, seed=seed, paths=paths)
    x = dict(k_cache=case.k_cache, v_cache=case.v_cache, block_table=case.block_table,
             prefix_len=case.prefix_len, parents=case.parents, path=case.path, path_len=case.path_len)
    res = _run(x)
    assert (res["err"] == 0).all()
    ref = _oracle(x)
    _compare(res, ref)
    assert ref[5].sum() >= 4


def test_errors_leave_the_sequence_alone():
    tree = W.candidate_chains([16, 16])
    rows = [[5, 3, 9], [0, 1, 2], [4, 6, 7], [8, 10, 11]]
    x = _single(tree, 15, list(range(17, 33)), rows[0], Hkv=2, hd=64, seed=1)   # not from a root
    nb = 12
    rng = np.random.default_rng(3)
    x["k_cache"] = W.round_to(rng.standard_normal((nb, 2, 16, 64)), "bf16")
    x["v_cache"] = W.round_to(rng.standard_normal((nb, 2, 16, 64)), "bf16")
    x["block_table"] = torch.tensor(rows, dtype=torch.int32)
    x["prefix_len"] = torch.tensor([15, 15, 15, 15], dtype=torch.int32)
    x["parents"] = torch.tensor([tree] * 4, dtype=torch.int32)
    good = [0] + list(range(17, 33))
    bad = list(range(17, 33)) + [-1]
    x["path"] = torch.tensor([bad, good, good, good], dtype=torch.int32)
    x["path_len"] = torch.tensor([16, 17, 17, 17], dtype=torch.int32)
    x["block_table"][2, 2] = nb + 4                         # block outside the pool
    x["prefix_len"][3] = 3 * 16 - 33 + 1                   # one slot short for the tree
    res = _run(x)
    assert res["err"].tolist() == [tv.TV_ERR_BAD_PATH, 0, tv.TV_ERR_BAD_BLOCK, tv.TV_ERR_CAPACITY]
    assert res["remapped"].tolist() == [0, 1, 0, 0]
    assert res["table"][1].tolist() == [0, 2, 1]
    for b in (0, 2, 3):
        assert res["table"][b].tolist() == x["block_table"][b].tolist()
        assert int(res["new_len"][b]) == int(x["prefix_len"][b])
        assert (res["slot_map"][b] == -1).all()
    # only sequence 1's blocks (0, 1, 2) may change, and they do as the oracle says
    ok = dict(x)
    for key in ("block_table", "prefix_len", "parents", "path", "path_len"):
        ok[key] = x[key][1:2]
    ref = _oracle(ok)
    assert np.array_equal(_gpu.f32np(res["k_cache"].cpu()), ref[0])
    assert np.array_equal(_gpu.f32np(res["v_cache"].cpu()), ref[1])


def test_overlapping_output_table_is_rejected():
    x = _single(W.candidate_chains([16, 16]), 15, [0] + list(range(17, 33)), [5, 3, 9], Hkv=1, hd=64, seed=0)
    d = {k: _gpu.to_dev(v) for k, v in x.items()}
    B = 1
    out = [torch.zeros(s, dtype=torch.int32, device="cuda") for s in ((B, 19), (B,), (B,), (B,))]
    with pytest.raises(tv.TVError) as e:
        tv.tv_kv_compact_remap(d["k_cache"], d["v_cache"], d["block_table"], d["block_table"], d["prefix_len"],
                               d["parents"], d["path"], d["path_len"], *out)
    assert e.value.status == tv.TV_ERR_INVALID_ARG


def _gather_logical(cache_dev, table_row, slots):
    """Rows of logical ``slots`` of one sequence from a device cache, on the CPU (indexing only)."""
    s = torch.as_tensor(slots, dtype=torch.int64)
    blk = torch.as_tensor(np.asarray(table_row), dtype=torch.int64)[s // 16]
    return cache_dev[blk.to(cache_dev.device), :, (s % 16).to(cache_dev.device)].cpu()


@pytest.mark.parametrize("workload", ["chains", "b32"])
def test_full_size_paged_batch(workload):
    """The paged batch-32 shapes (hd 256, 4 KV heads, P ~ U[2048, 32768], 2.4 GB of KV): every
    sequence's kept slots and the blocks around them, and the new rows, against the oracle's
    plan and the compaction's definition."""
    case = W.paged_chains_case() if workload == "chains" else W.paged_attn_b32_case()
    res = _gpu.run_compact_remap(case.k_cache, case.v_cache, case.block_table, case.prefix_len, case.parents,
                                 case.path, case.path_len)
    assert (res["err"] == 0).all()
    path, L = case.path.numpy(), case.path_len.numpy()
    tables = case.block_table.numpy()
    total = 0
    for b in range(case.q.shape[0]):
        P, Lb = int(case.prefix_len[b]), int(L[b])
        plan = A.remap_plan(P, path[b], Lb)
        want = tables[b].copy()
        for m, j in plan:
            want[m], want[m + j] = want[m + j], want[m]
        assert res["table"][b].tolist() == want.tolist()
        assert int(res["remapped"][b]) == len(plan)
        assert int(res["new_len"][b]) == P + Lb
        total += len(plan)
        # kept slots, and the prefix rows of the first and last prefix block
        lo = max(0, P - 16 - P % 16)
        before_slots = list(range(lo, P)) + [P + int(path[b][r]) for r in range(Lb)]
        after_slots = list(range(lo, P + Lb))
        for cache, name in ((case.k_cache, "k"), (case.v_cache, "v")):
            before = cache[torch.as_tensor(tables[b][np.asarray(before_slots) // 16], dtype=torch.int64), :,
                           torch.as_tensor(np.asarray(before_slots) % 16, dtype=torch.int64)]
            dev = res["k_cache"] if name == "k" else res["v_cache"]
            after = _gather_logical(dev, res["table"][b], after_slots)
            assert torch.equal(after, before), (workload, b, name)
        assert np.array_equal(res["slot_map"][b, :Lb],
                              [A.physical_slot(tables[b], P + int(path[b][r])) for r in range(Lb)])
    if workload == "chains":
        assert total > 0
    else:
        assert total == 0


@pytest.mark.parametrize("hd", [128, 256])
def test_long_paths_move_in_several_rounds(hd):
    """Paths of up to 101 entries: more than one load/store round at hd 256 (32 entries per
    round) and hd 128 (64).  Both kernels, the whole caches, against the oracle."""
    t = W.candidate_chains([32, 100])
    paths = [[0] + list(range(33, 33 + L - 1)) for L in (101, 70, 40, 33)]
    case = W.attn_case([t] * 4, [0, 15, 17, 33], Hq=2, Hkv=2, hd=hd, seed=9, paths=paths)
    x = dict(k_cache=case.k_cache, v_cache=case.v_cache, block_table=case.block_table,
             prefix_len=case.prefix_len, parents=case.parents, path=case.path, path_len=case.path_len)
    res = _run(x)
    assert (res["err"] == 0).all()
    ref = _oracle(x)
    _compare(res, ref)
    assert ref[5].sum() >= 4
    comp = _gpu.run_compact(case, case.k_cache, case.v_cache)
    assert (comp["err"] == 0).all()
    kc2, vc2, smap, new_len = A.kv_compact(W.f64(case.k_cache), W.f64(case.v_cache), case.block_table.numpy(),
                                           case.prefix_len.numpy(), case.parents.numpy(), case.path.numpy(),
                                           case.path_len.numpy())
    assert np.array_equal(comp["slot_map"], smap) and np.array_equal(comp["new_len"], new_len)
    assert np.array_equal(_gpu.f32np(comp["k_cache"]), kc2)
    assert np.array_equal(_gpu.f32np(comp["v_cache"]), vc2)
