"""GPU vs oracle: the greedy accept walk, bit-exact, through the C ABI."""
import numpy as np
import pytest
import torch

import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import tree as T

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pad(trees):
    N = max(len(t) for t in trees)
    return np.array([t + [-1] * (N - len(t)) for t in trees], dtype=np.int32)


def _run(parents, draft, target, lmax):
    B = parents.shape[0]
    path = torch.full((B, lmax), 777, dtype=torch.int32, device=DEV)
    ln = torch.full((B,), 777, dtype=torch.int32, device=DEV)
    nxt = torch.full((B,), 777, dtype=torch.int32, device=DEV)
    err = torch.full((B,), 777, dtype=torch.int32, device=DEV)
    tv.tv_accept_walk(torch.as_tensor(parents, device=DEV), torch.as_tensor(draft, device=DEV),
                      torch.as_tensor(target, device=DEV), path, ln, nxt, err)
    torch.cuda.synchronize()
    return path.cpu().numpy(), ln.cpu().numpy(), nxt.cpu().numpy(), err.cpu().numpy()


def _check(trees, draft, target, lmax):
    path, ln, nxt, err = _run(_pad(trees), draft, target, lmax)
    for b, parents in enumerate(trees):
        n = len(parents)
        ref_path, ref_next = T.accept_walk(parents, draft[b, :n], target[b, :n], lmax)
        assert err[b] == 0
        assert ln[b] == len(ref_path)
        assert list(path[b, :ln[b]]) == ref_path
        assert (path[b, ln[b]:] == -1).all()
        assert nxt[b] == ref_next


@pytest.mark.parametrize("n", [1, 2, 7, 33, 64, 255, 256])
def test_random_trees_small_vocabulary(n):
    rng = np.random.default_rng(n)
    trees = [W.random_tree(n, rng) if n > 1 else [-1] for _ in range(9)]
    draft = rng.integers(0, 3, size=(9, n)).astype(np.int32)    # sibling ties are frequent
    target = rng.integers(0, 3, size=(9, n)).astype(np.int32)
    for lmax in (1, 3, 9):
        _check(trees, draft, target, lmax)


def test_chains_accept_to_the_limit():
    n = 200
    chain = W.chain(n)
    draft = np.arange(n, dtype=np.int32)[None] + 5
    target = np.concatenate([draft[:, 1:], [[-7]]], axis=1).astype(np.int32)   # every step matches
    _check([chain], draft, target, 256)
    _check([chain], draft, target, 17)


def test_walk_reproduces_the_benchmark_paths():
    case = W.stack_b64_layer()
    draft, target = W.walk_tokens(case.trees, case.path.numpy(), case.path_len.numpy(), seed=3)
    path, ln, nxt, err = _run(_pad(case.trees), draft.numpy(), target.numpy(), case.path.shape[1])
    assert (err == 0).all()
    assert np.array_equal(ln, case.path_len.numpy())
    for b in range(len(case.trees)):
        assert list(path[b, :ln[b]]) == list(case.path[b, :ln[b]].numpy())


def test_malformed_tree_only_fails_its_sequence():
    trees = [[-1, 0, 0], [-1, 2, 0], [-1, 0, 1]]        # sequence 1: parents[1] = 2 is not earlier
    draft = np.array([[1, 2, 3]] * 3, dtype=np.int32)
    target = np.array([[2, 9, 9]] * 3, dtype=np.int32)
    path, ln, nxt, err = _run(_pad(trees), draft, target, 4)
    assert list(err) == [0, tv.TV_ERR_BAD_TREE, 0]
    assert ln[1] == 0 and nxt[1] == -1 and (path[1] == -1).all()
    assert list(path[0, :ln[0]]) == [0, 1] and list(path[2, :ln[2]]) == [0, 1]


def test_host_side_argument_errors():
    L = tv.lib
    assert L.tv_accept_walk(None, None, None, 1, 4, 4, None, None, None, None, None) == tv.TV_ERR_INVALID_ARG
    p = torch.zeros((1, 4), dtype=torch.int32, device=DEV)
    o = torch.zeros(8, dtype=torch.int32, device=DEV)
    args = [p.data_ptr()] * 3 + [1, 257, 4] + [o.data_ptr()] * 4 + [None]
    assert L.tv_accept_walk(*args) == tv.TV_ERR_UNSUPPORTED
    args = [p.data_ptr()] * 3 + [1, 4, 0] + [o.data_ptr()] * 4 + [None]
    assert L.tv_accept_walk(*args) == tv.TV_ERR_INVALID_ARG
