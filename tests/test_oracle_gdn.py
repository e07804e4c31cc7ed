"""Pins of the oracle's gated delta rule over trees (CPU only).

Every pin checks the oracle against something other than itself: a closed form of the rule,
a property the pages require (sibling isolation, node = its path as a plain chain), a second
algorithm (the depth-by-depth schedule), or a library triangular solve (pseudo-values).
Shapes use dk != dv where it matters so that a transposed operand fails.
"""
import numpy as np
import pytest
import scipy.linalg

import workloads as W
from oracle import gdn as G
from oracle import tree as T


def _inputs(trees, H=2, dk=6, dv=4, seed=0, **over):
    case = W.gdn_case(trees, H=H, dk=dk, dv=dv, io="f32", state="f32", seed=seed)
    inp = case.oracle_inputs()
    inp.update(over)
    return inp


def _trees():
    rng = np.random.default_rng(5)
    return [[-1, 0, 0, 1, 1, 2, 2], W.random_tree(7, rng)]


def test_no_write_no_decay_keeps_state():
    inp = _inputs(_trees())
    inp["alpha"] = np.ones_like(inp["alpha"])
    inp["beta"] = np.zeros_like(inp["beta"])
    o, S = G.verify(inp)
    for b in range(2):
        for i in range(7):
            assert np.allclose(S[b, i], inp["S0"][b], atol=1e-15)
            assert np.allclose(o[b, i], np.einsum("hvk,hk->hv", inp["S0"][b], inp["q"][b, i]))


def test_pure_decay_scales_by_path_product():
    inp = _inputs(_trees())
    inp["beta"] = np.zeros_like(inp["beta"])
    _, S = G.verify(inp)
    for b in range(2):
        for i in range(7):
            gamma = np.prod([inp["alpha"][b, j] for j in T.path_to(inp["parents"][b], i)], axis=0)
            assert np.allclose(S[b, i], gamma[:, None, None] * inp["S0"][b], rtol=1e-13)


@pytest.mark.parametrize("beta_val", [1.0, 0.3])
def test_write_interpolates_key_prediction_towards_value(beta_val):
    """For a unit key the transition I - beta k k^T shrinks k by (1 - beta), so
    S_i k_i = (1 - beta_i) alpha_i S_p k_i + beta_i v_i; with beta = 1 the state maps the key
    exactly to the value (delta-rule write)."""
    inp = _inputs(_trees())
    inp["beta"] = np.full_like(inp["beta"], beta_val)
    _, S = G.verify(inp)
    for b in range(2):
        par = inp["parents"][b]
        for i in range(7):
            p = par[i]
            Sp = inp["S0"][b] if p == -1 else S[b, p]
            k = inp["k"][b, i]
            lhs = np.einsum("hvk,hk->hv", S[b, i], k)
            pred = np.einsum("hvk,hk->hv", Sp, k)
            a = inp["alpha"][b, i][:, None]
            rhs = (1 - beta_val) * a * pred + beta_val * inp["v"][b, i]
            assert np.allclose(lhs, rhs, atol=1e-13)


def test_directions_orthogonal_to_key_only_decay():
    inp = _inputs(_trees(), dk=7, dv=3)
    inp["v"] = np.zeros_like(inp["v"])
    _, S = G.verify(inp)
    rng = np.random.default_rng(9)
    for b in range(2):
        par = inp["parents"][b]
        for i in range(7):
            p = par[i]
            Sp = inp["S0"][b] if p == -1 else S[b, p]
            for h in range(2):
                k = inp["k"][b, i, h]
                u = rng.standard_normal(7)
                u -= (u @ k) * k
                a = inp["alpha"][b, i, h]
                assert np.allclose(S[b, i, h] @ u, a * (Sp[h] @ u), atol=1e-13)
                assert np.allclose(S[b, i, h] @ k,
                                   a * (1 - inp["beta"][b, i, h]) * (Sp[h] @ k), atol=1e-13)


def test_orthonormal_keys_closed_form():
    """alpha = beta = 1 with mutually orthonormal keys: S_i = S_0 + sum_j (v_j - S_0 k_j) k_j^T
    over the path (each write lands in a fresh direction)."""
    n, dk, dv, H = 7, 9, 5, 2
    trees = [[-1, 0, 0, 1, 1, 2, 2]]
    inp = _inputs(trees, H=H, dk=dk, dv=dv)
    rng = np.random.default_rng(2)
    for h in range(H):
        Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
        inp["k"][0, :, h, :] = Qm[:n]
    inp["alpha"] = np.ones_like(inp["alpha"])
    inp["beta"] = np.ones_like(inp["beta"])
    _, S = G.verify(inp)
    for i in range(n):
        expect = inp["S0"][0].copy()
        for j in T.path_to(trees[0], i):
            for h in range(H):
                k = inp["k"][0, j, h]
                expect[h] += np.outer(inp["v"][0, j, h] - inp["S0"][0, h] @ k, k)
        assert np.allclose(S[0, i], expect, atol=1e-13)


def test_every_node_equals_its_path_run_as_a_plain_chain():
    """Brute force: node i's state/output equals the rule run over its root-to-node path as an
    ordinary sequence (a chain tree holding only the path's inputs)."""
    rng = np.random.default_rng(11)
    tree = W.random_tree(12, rng)
    inp = _inputs([tree], dk=5, dv=3, seed=4)
    o, S = G.verify(inp)
    for i in range(12):
        path = T.path_to(tree, i)
        sub = {key: (val[:, path] if key in ("q", "k", "v", "alpha", "beta") else val)
               for key, val in inp.items()}
        sub["q"] = inp["q"][:, [i] * len(path)]
        sub["parents"] = np.array([W.chain(len(path))])
        o2, S2 = G.verify(sub)
        assert np.allclose(S2[0, -1], S[0, i], atol=1e-14)
        assert np.allclose(o2[0, -1], o[0, i], atol=1e-14)


def test_siblings_do_not_contaminate_each_other():
    tree = [-1, 0, 0, 1, 1, 2, 2]
    inp = _inputs([tree])
    o, _ = G.verify(inp)
    for i in range(7):
        off = [j for j in range(7) if j not in T.path_to(tree, i)]
        pert = {k: v.copy() for k, v in inp.items() if isinstance(v, np.ndarray)}
        pert["q_scale"] = 1.0
        for j in off:
            pert["k"][0, j] *= -1.0
            pert["v"][0, j] += 3.0
            pert["alpha"][0, j] *= 0.5
        o2, _ = G.verify(pert)
        assert np.allclose(o2[0, i], o[0, i], atol=1e-15)


def test_depth_schedule_equals_path_replay():
    rng = np.random.default_rng(8)
    trees = [W.random_tree(15, rng) for _ in range(3)]
    inp = _inputs(trees, dk=5, dv=4)
    o1, S1 = G.verify(inp)
    o2, S2 = G.verify_by_depth(inp)
    assert np.allclose(o1, o2, atol=1e-14) and np.allclose(S1, S2, atol=1e-14)


def test_q_scale_scales_outputs():
    inp = _inputs(_trees())
    o1, _ = G.verify(inp)
    inp["q_scale"] = 0.125
    o2, _ = G.verify(inp)
    assert np.allclose(o2, 0.125 * o1, atol=1e-15)


def test_pseudo_values_rebuild_states_and_solve_the_triangular_system():
    """The TreeWY reading: S_i = gamma_i S_0 + sum_{j in path(i)} (gamma_i/gamma_j) w_j k_j^T, and
    W solves (I + diag(beta)(A o Gamma o K K^T)) W = diag(beta)(V - diag(gamma) K S_0^T), A the
    strict-ancestor mask; the solve is done here by scipy's triangular solver."""
    rng = np.random.default_rng(12)
    tree = W.random_tree(14, rng)
    inp = _inputs([tree], H=2, dk=6, dv=4, seed=3)
    _, S = G.verify(inp)
    w, lg = G.pseudo_values(inp, 0)
    n = len(tree)
    A = T.tree_mask(tree) & ~np.eye(n, dtype=bool)
    for h in range(2):
        gamma = np.exp(lg[:, h])
        K = inp["k"][0, :, h]
        V = inp["v"][0, :, h]
        S0 = inp["S0"][0, h]
        beta = inp["beta"][0, :, h]
        for i in range(n):
            rebuilt = gamma[i] * S0
            for j in T.path_to(tree, i):
                rebuilt = rebuilt + (gamma[i] / gamma[j]) * np.outer(w[j, h], K[j])
            assert np.allclose(rebuilt, S[0, i, h], atol=1e-13)
        Gam = gamma[:, None] / gamma[None, :]
        Lmat = np.eye(n) + beta[:, None] * (A * Gam * (K @ K.T))
        rhs = beta[:, None] * (V - gamma[:, None] * (K @ S0.T))
        Wsol = scipy.linalg.solve_triangular(Lmat, rhs, lower=True, unit_diagonal=True)
        assert np.allclose(Wsol, w[:, h], atol=1e-12)
        # log(gamma) is the running sum of log(alpha): gamma_i = alpha_i * gamma_parent
        for i in range(n):
            p = tree[i]
            parent_gamma = 1.0 if p == -1 else gamma[p]
            assert np.isclose(gamma[i], inp["alpha"][0, i, h] * parent_gamma, rtol=1e-14)


def test_commit_takes_last_accepted_state_and_skips_bad_paths():
    tree = [-1, 0, 0, 1, 1, 2, 2]
    inp = _inputs([tree, tree, tree])
    _, S = G.verify(inp)
    path = np.array([[0, 2, 6], [0, 1, -1], [0, 3, -1]])
    L = np.array([3, 1, 2])
    out = G.commit(inp, path, L)
    assert np.allclose(out[0], S[0, 6], atol=1e-15)
    assert np.allclose(out[1], S[1, 0], atol=1e-15)
    assert np.array_equal(out[2], inp["S0"][2])     # 3 is not a child of 0: unchanged


def test_selective_slots_number_kept_snapshots_in_node_order():
    # the page's rule: confidence above the threshold -> no snapshot; at the threshold -> kept
    slots, kept, fits = G.selective_slots([0.5, 0.99, 0.2, 0.96, 0.95, 0.951], 0.95, 3)
    assert slots == [0, -1, 1, -1, 2, -1] and kept == 3 and fits
    assert G.selective_slots([0.5, 0.2, 0.1], 0.95, 2)[2] is False       # 3 kept > capacity 2
    assert G.selective_slots([0.99, 0.97], 0.95, 0) == ([-1, -1], 0, True)  # nothing kept
    assert G.selective_slots([0.3] * 4, 1.0, 4) == ([0, 1, 2, 3], 4, True)  # threshold 1: all kept


def test_commit_then_verify_continues_the_sequence():
    # Round 1 verifies a chain of m nodes and accepts all of them; round 2 verifies a chain of n
    # nodes from the committed state.  Round 2's outputs must be those of nodes m .. m+n-1 of a
    # single chain over both rounds' inputs -- the plain sequential recurrence.
    m, n, H, d = 3, 4, 2, 8
    long = W.gdn_case([W.chain(m + n)], H=H, dk=d, dv=d, io="f32", state="f32", seed=4)
    li = long.oracle_inputs()
    first = {k: (v[:, :m] if k in ("q", "k", "v", "alpha", "beta") else v) for k, v in li.items()}
    first["parents"] = np.array([W.chain(m)])
    second = {k: (v[:, m:] if k in ("q", "k", "v", "alpha", "beta") else v) for k, v in li.items()}
    second["parents"] = np.array([W.chain(n)])
    path = np.array([list(range(m))])
    S0, o = G.verify_after_commit(first, path, np.array([m]), second)
    # the sequential recurrence over all m + n tokens, written out
    S = li["S0"][0].copy()
    outs = []
    for t in range(m + n):
        for h in range(H):
            kk, vv, a_, b_ = li["k"][0, t, h], li["v"][0, t, h], li["alpha"][0, t, h], li["beta"][0, t, h]
            S[h] = a_ * S[h] @ (np.eye(d) - b_ * np.outer(kk, kk)) + b_ * np.outer(vv, kk)
        outs.append(np.einsum("hvk,hk->hv", S, li["q"][0, t]))
        if t == m - 1:
            assert np.allclose(S0[0], S, atol=1e-12)
    assert np.allclose(o[0], np.stack(outs[m:]), atol=1e-12)
