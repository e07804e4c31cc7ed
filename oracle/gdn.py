"""Gated delta rule over a draft tree, by root-to-node path replay (fp64 oracle).

Test infrastructure only: see the package docstring.

Sources
-------
* The recurrence.  The qwen35-tree-spec post (§三, 混合架构的挑战) introduces the GDN state
  update, but its formula was lost in extraction; the surviving text says the state is one
  global matrix per head that every token changes irreversibly, and that a decay factor
  scales the whole state.  The reading used here is the gated delta rule

      S_i = alpha_i * S_p @ (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,     o_i = S_i q_i,

  with S a [dv, dk] matrix per head, alpha_i and beta_i scalars per (node, head), p the
  parent of i (the committed state S_0 for a root) and q scaled by ``q_scale`` (1.0 unless
  a caller asks otherwise).
* Per-path semantics.  The same post (§三 and §四) requires every node to see only its own
  root-to-node path: siblings must not contaminate each other, so each branch evolves from
  a snapshot of its parent's state.  ``node_state`` replays the path from S_0, which is the
  plainest statement of that requirement; ``verify_by_depth`` is the post's own
  depth-by-depth schedule (§四, 逐深度处理), kept as a second, independent algorithm.
* Commit.  After verification the state goes back to that of the last accepted node and
  the other snapshots are dropped (§五 用途 2, §七 Step 4).
* Selective fork.  The same post (§六, 选择性 Fork) skips the snapshot of a node whose draft
  confidence exceeds a threshold (0.95 on the page): such a node is processed but keeps no
  rollback point.  ``selective_slots`` numbers the kept snapshots in node order; a commit
  whose accepted node kept no snapshot resumes from the deepest kept one on its path (or
  S_0) -- which ``commit`` already states, since it replays the path.
* Lazy commit.  ``verify_after_commit`` is the previous round's commit followed by this
  round's verify from the committed state: the TreeWY kernel that fuses the two must equal it.
* Pseudo-values.  The TreeWY abstract (TreeWY: Speculative Verification for Gated DeltaNet
  Hybrids) keeps a small pseudo-value matrix instead of per-node states and rebuilds only
  the accepted state on commit.  Its derivation is not on the page.  The reading used
  here: unrolling the rule gives S_i = gamma_i S_0 + sum_{j on path(i)} (gamma_i/gamma_j)
  w_j k_j^T with gamma_i the product of alpha along path(i) and the pseudo-value
  w_i = beta_i (v_i - alpha_i S_p k_i).  ``pseudo_values`` computes w and log(gamma) from
  those definitions, from the replayed states, not by the triangular solve.
"""
from __future__ import annotations

import numpy as np

from .tree import depths, is_valid_path, is_valid_tree, path_to


def gdn_step(S: np.ndarray, k: np.ndarray, v: np.ndarray, alpha, beta) -> np.ndarray:
    """One gated delta rule update for every head at once.

    ``S [H, dv, dk]``, ``k [H, dk]``, ``v [H, dv]``, ``alpha, beta [H]``; returns
    ``alpha * S @ (I - beta k k^T) + beta v k^T``, with the transition matrix formed
    explicitly.
    """
    H, dv, dk = S.shape
    alpha = np.asarray(alpha, dtype=np.float64).reshape(H, 1, 1)
    beta = np.asarray(beta, dtype=np.float64).reshape(H, 1, 1)
    eye = np.eye(dk)[None, :, :]
    transition = eye - beta * (k[:, :, None] * k[:, None, :])
    return alpha * np.matmul(S, transition) + beta * (v[:, :, None] * k[:, None, :])


def gdn_output(S: np.ndarray, q: np.ndarray, q_scale: float = 1.0) -> np.ndarray:
    """o = S (q_scale q) for every head: ``S [H, dv, dk]``, ``q [H, dk]`` -> ``[H, dv]``."""
    return np.matmul(S, (q_scale * q)[:, :, None])[:, :, 0]


def node_state(inp: dict, b: int, i: int) -> tuple[np.ndarray, np.ndarray]:
    """State ``[H, dv, dk]`` and output ``[H, dv]`` of node i of sequence b, replaying the
    gated delta rule from S_0 along the node's root-to-node path."""
    parents = inp["parents"][b]
    S = inp["S0"][b].copy()
    for j in path_to(parents, i):
        S = gdn_step(S, inp["k"][b, j], inp["v"][b, j], inp["alpha"][b, j], inp["beta"][b, j])
    return S, gdn_output(S, inp["q"][b, i], inp.get("q_scale", 1.0))


def verify(inp: dict, want_states: bool = True):
    """Outputs ``o [B,N,H,dv]`` and (optionally) every node's state ``[B,N,H,dv,dk]`` by path
    replay."""
    B, N, H, dk = inp["q"].shape
    dv = inp["v"].shape[-1]
    o = np.zeros((B, N, H, dv))
    states = np.zeros((B, N, H, dv, dk)) if want_states else None
    for b in range(B):
        for i in range(N):
            S, oi = node_state(inp, b, i)
            o[b, i] = oi
            if want_states:
                states[b, i] = S
    return o, states


def verify_by_depth(inp: dict):
    """The depth-by-depth schedule of the qwen35-tree-spec post (§四, 逐深度处理): all nodes of
    depth d evolve, each from its parent's snapshot (S_0 for a root), before any node of depth
    d+1.  Returns ``o [B,N,H,dv]`` and the states ``[B,N,H,dv,dk]``."""
    B, N, H, dk = inp["q"].shape
    dv = inp["v"].shape[-1]
    o = np.zeros((B, N, H, dv))
    states = np.zeros((B, N, H, dv, dk))
    q_scale = inp.get("q_scale", 1.0)
    for b in range(B):
        parents = inp["parents"][b]
        dep = depths(parents)
        for d in range(max(dep) + 1):
            for i in [n for n in range(N) if dep[n] == d]:
                p = int(parents[i])
                S_parent = inp["S0"][b] if p == -1 else states[b, p]
                states[b, i] = gdn_step(S_parent, inp["k"][b, i], inp["v"][b, i],
                                        inp["alpha"][b, i], inp["beta"][b, i])
                o[b, i] = gdn_output(states[b, i], inp["q"][b, i], q_scale)
    return o, states


def pseudo_value_node(inp: dict, b: int, i: int):
    """TreeWY quantities of node i of sequence b from their definitions (reading stated in the
    module docstring): ``w_i [H, dv]`` = beta_i (v_i - alpha_i S_parent k_i) and
    ``log_gamma_i [H]`` = sum of log(alpha) along the root-to-node path."""
    parents = inp["parents"][b]
    p = int(parents[i])
    S_parent = inp["S0"][b] if p == -1 else node_state(inp, b, p)[0]
    Sk = np.matmul(S_parent, inp["k"][b, i][:, :, None])[:, :, 0]
    a = inp["alpha"][b, i][:, None]
    w = inp["beta"][b, i][:, None] * (inp["v"][b, i] - a * Sk)
    log_gamma = sum(np.log(inp["alpha"][b, j]) for j in path_to(parents, i))
    return w, log_gamma


def pseudo_values(inp: dict, b: int):
    """``w [N, H, dv]`` and ``log_gamma [N, H]`` of every node of sequence b."""
    N = inp["q"].shape[1]
    pairs = [pseudo_value_node(inp, b, i) for i in range(N)]
    return np.stack([w for w, _ in pairs]), np.stack([lg for _, lg in pairs])


def commit(inp: dict, path: np.ndarray, path_len: np.ndarray) -> np.ndarray:
    """Committed state ``[B,H,dv,dk]`` after acceptance: the state of the last accepted node
    (qwen35-tree-spec §五 用途 2).  A sequence whose tree is malformed or whose path is not a
    root-to-node path keeps S_0."""
    out = inp["S0"].copy()
    for b in range(out.shape[0]):
        L = int(path_len[b])
        if not (is_valid_tree(inp["parents"][b]) and is_valid_path(inp["parents"][b], path[b], L)):
            continue
        out[b] = node_state(inp, b, int(path[b][L - 1]))[0]
    return out


def selective_slots(confidence, threshold: float, capacity: int):
    """Snapshot slots of one tree under selective fork: node i keeps its snapshot unless its
    confidence is above ``threshold``; kept snapshots take slots 0, 1, ... in node order.
    Returns (slot per node, -1 where skipped; number kept; whether it fits ``capacity``)."""
    slots, kept = [], 0
    for c in confidence:
        if float(c) > threshold:
            slots.append(-1)
        else:
            slots.append(kept)
            kept += 1
    return slots, kept, kept <= capacity


def verify_after_commit(prev_inp: dict, prev_path: np.ndarray, prev_len: np.ndarray, inp: dict):
    """The previous round's commit, then this round's verify from the committed state.
    Returns (committed S_0 [B,H,dv,dk], outputs [B,N,H,dv])."""
    S0 = commit(prev_inp, prev_path, prev_len)
    cur = dict(inp)
    cur["S0"] = S0
    o, _ = verify(cur, want_states=False)
    return S0, o

