"""The bounded device wait, driven to its limit on the GPU (no copy or MMA in flight): the wait
gives up, TV_ERR_TIMEOUT comes back, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
from oracle import tree as T

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _wait(max_polls, arrive):
    status = torch.full((1,), 777, dtype=torch.int32, device=DEV)
    ns = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    t0 = time.perf_counter()
    tv.tv_test_bounded_wait(max_polls, arrive, status, ns)
    torch.cuda.synchronize()
    return int(status.item()), int(ns.item()), time.perf_counter() - t0


def test_a_wait_nothing_arrives_on_gives_up_with_timeout():
    st, ns, _ = _wait(1000, arrive=False)
    assert st == tv.TV_ERR_TIMEOUT
    assert ns > 0


def test_a_wait_whose_phase_completes_succeeds():
    st, ns, _ = _wait(1000, arrive=True)
    assert st == tv.TV_OK
    assert 0 <= ns < 1_000_000


def test_the_kernels_default_limit_ends_within_seconds_and_the_context_stays_usable():
    st, ns, wall = _wait(0, arrive=False)
    assert st == tv.TV_ERR_TIMEOUT
    assert 0 < ns < 10_000_000_000 and wall < 20.0
    # more polls wait longer
    _, ns_short, _ = _wait(1 << 12, arrive=False)
    assert ns_short < ns
    # the context still runs kernels: tree topology against the oracle
    parents = [-1, 0, 0, 1, 1, 2]
    r = _gpu.run_tree_prepare(torch.tensor([parents], dtype=torch.int32))
    assert int(r["err"][0]) == 0 and r["depth"][0].tolist() == T.depths(parents)
    assert np.array_equal(r["mask_bits"][0], T.mask_bits(parents))
