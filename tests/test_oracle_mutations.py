"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch them.

Each mutant replaces one oracle function with a near miss (a dropped term, a wrong sign or
index, a transposed operand).  The pins of ``test_oracle_gdn`` / ``test_oracle_attention``
are then run against the mutant; at least one must fail.
"""
import numpy as np
import pytest

import test_oracle_attention as PA
import test_oracle_compact_remap as PR
import test_oracle_gdn as PG
from oracle import attention as A
from oracle import gdn as G
from oracle import tree as T

_GDN_PINS = [f for n, f in vars(PG).items() if n.startswith("test_")]
_ATTN_PINS = [f for n, f in vars(PA).items() if n.startswith("test_")]


def _run_pins(pins):
    failed = 0
    for pin in pins:
        params = pin.__code__.co_varnames[:pin.__code__.co_argcount]
        kwargs = {}
        if "beta_val" in params:
            kwargs["beta_val"] = 0.3
        if "hd" in params:
            kwargs["hd"] = 8
        try:
            pin(**kwargs)
        except (AssertionError, ValueError, IndexError, KeyError, TypeError):
            failed += 1
    return failed


def _step_no_alpha_on_state(S, k, v, alpha, beta):
    return G._orig_step(S, k, v, np.ones_like(np.asarray(alpha)), beta)


def _step_alpha_on_write_too(S, k, v, alpha, beta):
    a = np.asarray(alpha).reshape(-1, 1, 1)
    return a * G._orig_step(S, k, v, np.ones_like(np.asarray(alpha)), beta)


def _step_transition_on_left(S, k, v, alpha, beta):
    H, dv, dk = S.shape
    a = np.asarray(alpha).reshape(H, 1, 1)
    b = np.asarray(beta).reshape(H, 1, 1)
    t = np.eye(dv)[None] - b * (v[:, :, None] * v[:, None, :])
    return a * np.matmul(t, S) + b * (v[:, :, None] * k[:, None, :])


def _step_plus_sign(S, k, v, alpha, beta):
    H = S.shape[0]
    a = np.asarray(alpha).reshape(H, 1, 1)
    b = np.asarray(beta).reshape(H, 1, 1)
    t = np.eye(S.shape[2])[None] + b * (k[:, :, None] * k[:, None, :])
    return a * np.matmul(S, t) + b * (v[:, :, None] * k[:, None, :])


def _step_no_beta_on_write(S, k, v, alpha, beta):
    H = S.shape[0]
    a = np.asarray(alpha).reshape(H, 1, 1)
    b = np.asarray(beta).reshape(H, 1, 1)
    t = np.eye(S.shape[2])[None] - b * (k[:, :, None] * k[:, None, :])
    return a * np.matmul(S, t) + (v[:, :, None] * k[:, None, :])


def _step_write_key_reversed(S, k, v, alpha, beta):
    H = S.shape[0]
    a = np.asarray(alpha).reshape(H, 1, 1)
    b = np.asarray(beta).reshape(H, 1, 1)
    t = np.eye(S.shape[2])[None] - b * (k[:, :, None] * k[:, None, :])
    return a * np.matmul(S, t) + b * (v[:, :, None] * k[:, None, ::-1])


@pytest.mark.parametrize("mutant", [_step_no_alpha_on_state, _step_alpha_on_write_too,
                                    _step_transition_on_left, _step_plus_sign,
                                    _step_no_beta_on_write, _step_write_key_reversed])
def test_gdn_step_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(G, "_orig_step", G.gdn_step, raising=False)
    monkeypatch.setattr(G, "gdn_step", mutant)
    assert _run_pins(_GDN_PINS) >= 1


_ORIG_PATH = T.path_to


def _path_skips_root(parents, i):
    return _ORIG_PATH(parents, i)[1:] or [i]


def _path_wrong_order(parents, i):
    return _ORIG_PATH(parents, i)[::-1]


@pytest.mark.parametrize("mutant", [_path_skips_root, _path_wrong_order])
def test_path_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(G, "path_to", mutant)
    assert _run_pins(_GDN_PINS) >= 1


def _rope_interleaved(x, pos, theta):
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-2.0 * np.arange(half) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    out = x.copy()
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return out


def _rope_sign(x, pos, theta):
    return A._orig_rope(x, -np.asarray(pos), theta)


def _rope_freq(x, pos, theta):
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-1.0 * np.arange(half) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


@pytest.mark.parametrize("mutant", [_rope_interleaved, _rope_sign, _rope_freq])
def test_rope_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(A, "_orig_rope", A.rope, raising=False)
    monkeypatch.setattr(A, "rope", mutant)
    assert _run_pins(_ATTN_PINS) >= 1


def _mask_no_self(parents):
    return T.tree_mask(parents) & ~np.eye(len(parents), dtype=bool)


def _mask_causal(parents):
    n = len(parents)
    return np.tril(np.ones((n, n), dtype=bool))


def _depths_off_by_one(parents):
    return [d + 1 for d in T.depths(parents)]


@pytest.mark.parametrize("name,mutant", [("tree_mask", _mask_no_self),
                                         ("tree_mask", _mask_causal),
                                         ("depths", _depths_off_by_one)])
@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_attention_topology_mutants_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(A, name, mutant)
    assert _run_pins(_ATTN_PINS) >= 1


def _compact_descending_in_place(k_cache, v_cache, block_table, prefix_len, parents, path,
                                 path_len, block_size=16):
    """Copies in place from the last kept entry down, reading slots an earlier copy of the same
    call may already have overwritten."""
    kc, vc = k_cache.copy(), v_cache.copy()
    B, Lmax = path.shape
    slot_map = np.full((B, Lmax), -1, dtype=np.int64)
    new_len = np.asarray(prefix_len, dtype=np.int64).copy()
    for b in range(B):
        P, L, row = int(prefix_len[b]), int(path_len[b]), block_table[b]
        if not T.is_valid_path(parents[b], path[b], L):
            continue
        for r in reversed(range(L)):
            src = A.physical_slot(row, P + int(path[b][r]), block_size)
            dst = A.physical_slot(row, P + r, block_size)
            kc[dst // block_size, :, dst % block_size] = kc[src // block_size, :, src % block_size]
            vc[dst // block_size, :, dst % block_size] = vc[src // block_size, :, src % block_size]
            slot_map[b, r] = src
        new_len[b] = P + L
    return kc, vc, slot_map, new_len


def test_compaction_mutant_is_caught(monkeypatch):
    monkeypatch.setattr(A, "kv_compact", _compact_descending_in_place)
    assert _run_pins(_ATTN_PINS) >= 1


# ----------------------------------------------------------------------------- accept walk
import test_oracle_tree as PT  # noqa: E402

_WALK_PINS = [f for n, f in vars(PT).items() if n.startswith("test_accept_walk")]
_WALK = T.accept_walk  # the unmutated walk, for mutants that alter only its result


def _walk_highest_child(parents, draft_tokens, target_tokens, lmax):
    path, node = [0], 0
    while len(path) < lmax:
        cs = [c for c in range(len(parents)) if parents[c] == node and draft_tokens[c] == target_tokens[node]]
        if not cs:
            break
        node = cs[-1]
        path.append(node)
    return path, int(target_tokens[node])


def _walk_target_at_child(parents, draft_tokens, target_tokens, lmax):
    path, node = [0], 0
    while len(path) < lmax:
        cs = [c for c in range(len(parents)) if parents[c] == node and draft_tokens[c] == target_tokens[c]]
        if not cs:
            break
        node = cs[0]
        path.append(node)
    return path, int(target_tokens[node])


def _walk_next_token_at_root(parents, draft_tokens, target_tokens, lmax):
    path, _ = _WALK(parents, draft_tokens, target_tokens, lmax)
    return path, int(target_tokens[0])


def _walk_ignores_lmax(parents, draft_tokens, target_tokens, lmax):
    return _WALK(parents, draft_tokens, target_tokens, 10 ** 6)


@pytest.mark.parametrize("mutant", [_walk_highest_child, _walk_target_at_child, _walk_next_token_at_root,
                                    _walk_ignores_lmax])
def test_accept_walk_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(T, "accept_walk", mutant)
    assert _run_pins(_WALK_PINS) >= 1


_PLAN = A.remap_plan


def _run_remap_pins():
    """Every remap pin with each of its parameters; returns how many failed."""
    calls = [lambda f=f: PR.test_golden_cases(f) for f in PR._golden_cases()]
    calls += [lambda s=s: PR.test_logical_view_equals_moving_compaction(s) for s in (0, 1, 2)]
    calls += [lambda s=s: PR.test_plan_matches_physical_statement(s) for s in (3, 4)]
    calls += [PR.test_invalid_path_leaves_everything]
    failed = 0
    for call in calls:
        try:
            call()
        except (AssertionError, IndexError):
            failed += 1
    return failed


def _plan_floor(P, path, L, block_size=16):
    """Also considers the block that holds the last prefix slots."""
    bs = block_size
    plan = []
    for m in range(P // bs, (P + L - 1) // bs + 1):
        rows = [r for r in range(L) if m * bs <= P + r < (m + 1) * bs]
        shifts = {int(path[r]) - r for r in rows}
        if len(shifts) == 1:
            d = shifts.pop()
            if d > 0 and d % bs == 0:
                plan.append((m, d // bs))
    return plan


def _plan_any_shift(P, path, L, block_size=16):
    """Takes over blocks whose shift is not a whole number of blocks."""
    bs = block_size
    plan = []
    for m in range(-(-P // bs), (P + L - 1) // bs + 1):
        rows = [r for r in range(L) if m * bs <= P + r < (m + 1) * bs]
        shifts = {int(path[r]) - r for r in rows}
        if len(shifts) == 1 and min(shifts) > 0:
            plan.append((m, max(1, min(shifts) // bs)))
    return plan


def _plan_first_row_only(P, path, L, block_size=16):
    """Decides each block from its first kept entry alone."""
    bs = block_size
    plan = []
    for m in range(-(-P // bs), (P + L - 1) // bs + 1):
        r = max(m * bs - P, 0)
        d = int(path[r]) - r
        if d > 0 and d % bs == 0:
            plan.append((m, d // bs))
    return plan


def _plan_descending(P, path, L, block_size=16):
    """Right blocks, exchanged from the last to the first."""
    return _PLAN(P, path, L, block_size)[::-1]


@pytest.mark.parametrize("mutant", [_plan_floor, _plan_any_shift, _plan_first_row_only, _plan_descending])
def test_remap_plan_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(A, "remap_plan", mutant)
    assert _run_remap_pins() >= 1


def test_remap_pins_pass_on_the_oracle():
    assert _run_remap_pins() == 0
