"""Draft-tree topology: depth, tree mask, root-to-node paths, validity (fp64 oracle).

Test infrastructure only: see the package docstring.

Sources
-------
* Tree mask: the handbook chapter 树形草稿与 EAGLE, §实现, ``tree_mask``: node i sees
  itself and every ancestor; its printed 6-node example is a golden fixture.
* Depth: same chapter and section, ``depths``: 0 for a root, else parent depth + 1; the
  RoPE position of a node is prefix length + depth (same chapter, opening summary).
* Node ordering: ``parents[i] < i`` (the chapter's ``depths`` walks nodes in index order and
  needs every parent first; its breadth-first draft builder produces such numbering).
* Accepted path: the chapter's accept walk starts at a root and steps from parent to child
  (§实现, ``tree_speculative_generate``); the qwen35-tree-spec post restores the state of the
  last accepted token (§五, 用途 2).  ``accept_walk`` is that walk on given target tokens.
"""
from __future__ import annotations

import numpy as np


def is_valid_tree(parents) -> bool:
    """Every entry is -1 (a root, child of the committed state) or an earlier node."""
    return len(parents) >= 1 and all(-1 <= int(p) < i for i, p in enumerate(parents))


def depths(parents) -> list[int]:
    """depth[i] = 0 for a root, depth[parent] + 1 otherwise (handbook §实现, ``depths``)."""
    d: list[int] = []
    for p in parents:
        p = int(p)
        d.append(0 if p == -1 else d[p] + 1)
    return d


def path_to(parents, i: int) -> list[int]:
    """Root-to-node path of node i, inclusive, by following parents upward."""
    out = []
    j = int(i)
    while j != -1:
        out.append(j)
        j = int(parents[j])
    return out[::-1]


def tree_mask(parents) -> np.ndarray:
    """Boolean [N, N]: row i is True at i and at every ancestor of i (handbook §实现,
    ``tree_mask``)."""
    n = len(parents)
    mask = np.zeros((n, n), dtype=bool)
    for i in range(n):
        for j in path_to(parents, i):
            mask[i, j] = True
    return mask


def mask_bits(parents) -> np.ndarray:
    """The tree mask packed into uint32 words: [N, ceil(N/32)], bit (j % 32) of word j // 32."""
    m = tree_mask(parents)
    n = len(parents)
    words = (n + 31) // 32
    out = np.zeros((n, words), dtype=np.uint32)
    for i in range(n):
        for j in range(n):
            if m[i, j]:
                out[i, j // 32] |= np.uint32(1) << np.uint32(j % 32)
    return out


def children(parents) -> dict[int, list[int]]:
    out: dict[int, list[int]] = {}
    for i, p in enumerate(parents):
        out.setdefault(int(p), []).append(i)
    return out


def is_valid_path(parents, path, length: int) -> bool:
    """``path[0]`` is a root and ``path[r]`` is a child of ``path[r-1]`` for r < length;
    ``1 <= length <= len(path)``."""
    n = len(parents)
    if length < 1 or length > len(path):
        return False
    for r in range(length):
        node = int(path[r])
        if node < 0 or node >= n:
            return False
        want = -1 if r == 0 else int(path[r - 1])
        if int(parents[node]) != want:
            return False
    return True


def accept_walk(parents, draft_tokens, target_tokens, lmax: int):
    """Greedy acceptance of one draft tree (handbook chapter 树形草稿与 EAGLE, §实现,
    ``tree_speculative_generate``): start at node 0; while the target's token at the current
    node equals the draft token of one of its children, step to the lowest-numbered such child.
    Stops when no child matches or the path holds ``lmax`` nodes.

    ``target_tokens[i]`` is the target model's chosen token at node i (its argmax).  Returns
    (path as a list of nodes, next token = the target's token at the last accepted node).
    """
    path = [0]
    node = 0
    while len(path) < lmax:
        want = int(target_tokens[node])
        nxt = None
        for c in range(len(parents)):          # lowest index first
            if int(parents[c]) == node and int(draft_tokens[c]) == want:
                nxt = c
                break
        if nxt is None:
            break
        path.append(nxt)
        node = nxt
    return path, int(target_tokens[node])
