"""Tree-masked GQA attention over a paged KV prefix, and KV compaction (fp64 oracle).

Test infrastructure only: see the package docstring.

Sources
-------
* The handbook chapter 树形草稿与 EAGLE, §实现, ``forward_with_mask``: node queries and keys
  are rotated at their positions, keys and values are the cached prefix followed by the new
  nodes', the mask is "all prefix visible" beside the tree mask, KV heads are repeated to
  the query heads (``repeat_interleave``, so query head h reads KV head h // (Hq/Hkv)), and
  softmax uses the default scale 1/sqrt(head_dim).  The cache holds already-rotated keys.
* Positions: prefix length + depth; siblings share a position (same chapter, opening
  summary and §实现).
* RoPE: the chapter's ``rope_cos_sin`` / ``apply_rope`` come from a module that is not on the
  page.  Reading: rotate-half pairs (x_i, x_{i+hd/2}) over the full head dim, frequency
  theta^(-2i/hd), applied to q and k only.
* KV keep/discard: the accepted path's KV is reused, not recomputed, by moving it to the
  contiguous slots after the prefix; rejected slots become void (same chapter, note after
  the listing; qwen35-tree-spec §七 Step 4).  Reading: node i's KV sits at logical slot
  prefix_len + i; after compaction slots prefix_len + r hold node path[r] for r < L and the
  new length is prefix_len + L.
* Block-table compaction: the same note allows updating the block table instead of moving
  the slots.  Reading: a logical block that lies wholly at or past the prefix and whose kept
  entries all come from one other block, each at its own row, takes that block by an exchange
  of the two table entries; every other kept entry is moved as above.  The logical contents
  of slots [0, new length) are those of the moving compaction.
* Query operand precision: the handbook chapter's ``forward_with_mask`` runs on the model's
  bf16 tensors, and a tensor-core score product takes the rotated query as a bf16 operand.  Everything here is
  fp64 by default; ``query_bf16=True`` rounds the rotated query, and nothing else, to bf16
  (nearest, ties to even) before the score product, so that a comparison can separate the
  effect of that one rounding from every other error.
"""
from __future__ import annotations

import numpy as np

from .tree import depths, is_valid_path, is_valid_tree, tree_mask


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE in fp64.  ``x [T, heads, hd]``, ``pos [T]`` integer positions."""
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def logical_rows(cache: np.ndarray, table_row: np.ndarray, n_slots: int,
                 block_size: int = 16) -> np.ndarray:
    """Logical slots 0..n_slots-1 of one sequence from a paged cache ``[num_blocks, Hkv, bs,
    hd]`` -> ``[n_slots, Hkv, hd]``: slot s lives in block ``table_row[s // bs]`` at row
    ``s % bs``."""
    slots = np.arange(n_slots)
    blocks = np.asarray(table_row)[slots // block_size].astype(np.int64)
    return np.asarray(cache[blocks, :, slots % block_size, :], dtype=np.float64)


def physical_slot(table_row: np.ndarray, s: int, block_size: int = 16) -> int:
    """Physical slot index block * block_size + row of logical slot s."""
    return int(table_row[s // block_size]) * block_size + s % block_size


def bf16_round(x: np.ndarray) -> np.ndarray:
    """x rounded to the nearest bf16 value (8 significant bits, ties to even), as fp64."""
    x = np.asarray(x, dtype=np.float64)
    mant, expo = np.frexp(x)                    # x = mant * 2^expo, 0.5 <= |mant| < 1
    return np.ldexp(np.round(mant * 256.0) / 256.0, expo)   # np.round: half to even


def attend_one(q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray, prefix_k: np.ndarray,
               prefix_v: np.ndarray, parents, theta: float, sm_scale: float | None = None,
               query_bf16: bool = False):
    """One sequence: ``q [N,Hq,hd]``, ``k_new, v_new [N,Hkv,hd]``, ``prefix_k, prefix_v
    [P,Hkv,hd]`` (prefix keys already rotated).  Returns ``o [N,Hq,hd]`` and the rotated node
    keys ``[N,Hkv,hd]`` that the cache receives."""
    N, Hq, hd = q.shape
    Hkv = k_new.shape[1]
    P = prefix_k.shape[0]
    scale = hd ** -0.5 if sm_scale is None else sm_scale
    pos = P + np.asarray(depths(parents))
    qr = rope(q, pos, theta)
    if query_bf16:
        qr = bf16_round(qr)
    kr = rope(k_new, pos, theta)
    K = np.concatenate([prefix_k, kr], axis=0)
    V = np.concatenate([prefix_v, v_new], axis=0)
    visible = np.concatenate([np.ones((N, P), dtype=bool), tree_mask(parents)], axis=1)
    group = Hq // Hkv
    o = np.zeros((N, Hq, hd))
    for h in range(Hq):
        g = h // group
        scores = (qr[:, h, :] @ K[:, g, :].T) * scale
        scores = np.where(visible, scores, -np.inf)
        scores = scores - scores.max(axis=1, keepdims=True)
        p = np.exp(scores)
        p = p / p.sum(axis=1, keepdims=True)
        o[:, h, :] = p @ V[:, g, :]
    return o, kr


def tree_attention(case_f64: dict, batch=None, query_bf16: bool = False):
    """Paged form.  ``case_f64`` holds fp64 numpy arrays ``q, k_new, v_new, k_cache, v_cache``
    and int arrays ``block_table, prefix_len, parents`` plus ``rope_theta``.  Returns
    ``o [B,N,Hq,hd]`` (NaN rows for sequences not computed) and the rotated node keys."""
    q = case_f64["q"]
    B, N, Hq, hd = q.shape
    Hkv = case_f64["k_new"].shape[2]
    bs = case_f64.get("block_size", 16)
    o = np.full((B, N, Hq, hd), np.nan)
    kr_all = np.full((B, N, Hkv, hd), np.nan)
    for b in (range(B) if batch is None else batch):
        P = int(case_f64["prefix_len"][b])
        row = case_f64["block_table"][b]
        pk = logical_rows(case_f64["k_cache"], row, P, bs)
        pv = logical_rows(case_f64["v_cache"], row, P, bs)
        o[b], kr_all[b] = attend_one(q[b], case_f64["k_new"][b], case_f64["v_new"][b], pk, pv,
                                     case_f64["parents"][b], case_f64["rope_theta"],
                                     case_f64.get("sm_scale"), query_bf16)
    return o, kr_all


def cache_after_attention(case_f64: dict, rotated_k: np.ndarray, batch=None):
    """Expected caches after the attention call: logical slot prefix_len + i of each sequence
    holds node i's rotated key and its value; every other slot is unchanged."""
    kc = case_f64["k_cache"].copy()
    vc = case_f64["v_cache"].copy()
    bs = case_f64.get("block_size", 16)
    N = case_f64["q"].shape[1]
    for b in (range(case_f64["q"].shape[0]) if batch is None else batch):
        P = int(case_f64["prefix_len"][b])
        row = case_f64["block_table"][b]
        for i in range(N):
            s = P + i
            kc[int(row[s // bs]), :, s % bs, :] = rotated_k[b, i]
            vc[int(row[s // bs]), :, s % bs, :] = case_f64["v_new"][b, i]
    return kc, vc


def kv_compact(k_cache: np.ndarray, v_cache: np.ndarray, block_table: np.ndarray,
               prefix_len: np.ndarray, parents: np.ndarray, path: np.ndarray,
               path_len: np.ndarray, block_size: int = 16):
    """Compaction of the accepted path: for r < L, logical slot P + r receives the contents
    logical slot P + path[r] had before the call.  Returns the new caches, ``slot_map
    [B, Lmax]`` (physical source slot of each kept entry, -1 past L) and ``new_len [B]``
    (P + L; P for a sequence with an invalid path, whose cache is left unchanged)."""
    kc = k_cache.copy()
    vc = v_cache.copy()
    B, Lmax = path.shape
    slot_map = np.full((B, Lmax), -1, dtype=np.int64)
    new_len = np.asarray(prefix_len, dtype=np.int64).copy()
    for b in range(B):
        P = int(prefix_len[b])
        L = int(path_len[b])
        row = block_table[b]
        if not (is_valid_tree(parents[b]) and is_valid_path(parents[b], path[b], L)):
            continue
        src = [physical_slot(row, P + int(path[b][r]), block_size) for r in range(L)]
        saved_k = [k_cache[s // block_size, :, s % block_size, :].copy() for s in src]
        saved_v = [v_cache[s // block_size, :, s % block_size, :].copy() for s in src]
        for r in range(L):
            dst = physical_slot(row, P + r, block_size)
            kc[dst // block_size, :, dst % block_size, :] = saved_k[r]
            vc[dst // block_size, :, dst % block_size, :] = saved_v[r]
            slot_map[b, r] = src[r]
        new_len[b] = P + L
    return kc, vc, slot_map, new_len


def remap_plan(P: int, path, L: int, block_size: int = 16):
    """Destination blocks taken over by a table exchange, in ascending order: pairs (m, j) where
    logical block m lies wholly at or past P (m * bs >= P), holds kept entries r (P + r in
    block m, r < L), and every one of them comes from P + path[r] = P + r + j * bs with the
    same j >= 1.  Such a block's kept entries are exactly block m + j's entries at the same
    rows, so block m may take block m + j's physical block."""
    bs = block_size
    plan = []
    first = -(-P // bs)
    last = (P + L - 1) // bs
    for m in range(first, last + 1):
        rows = [r for r in range(L) if m * bs <= P + r < (m + 1) * bs]
        shifts = {int(path[r]) - r for r in rows}
        if len(shifts) == 1:
            d = shifts.pop()
            if d > 0 and d % bs == 0:
                plan.append((m, d // bs))
    return plan


def kv_compact_remap(k_cache: np.ndarray, v_cache: np.ndarray, block_table: np.ndarray,
                     prefix_len: np.ndarray, parents: np.ndarray, path: np.ndarray,
                     path_len: np.ndarray, block_size: int = 16):
    """Compaction that exchanges block-table entries where a whole destination block can be
    taken from one source block (``remap_plan``), and moves the remaining kept entries.

    For each valid sequence: the table row's entries m and m + j are exchanged for every
    (m, j) of the plan, in ascending m; then for every kept entry r < L outside the planned
    blocks, physical slot (new table, P + r) receives what physical slot (old table,
    P + path[r]) held before the call.  Returns the new caches, the new block table, ``slot_map
    [B, Lmax]`` (physical source slot under the old table, -1 past L), ``new_len [B]`` and
    ``remapped [B]`` (the number of exchanges).  A sequence with an invalid tree or path keeps
    its cache and table; its new length is P."""
    kc = k_cache.copy()
    vc = v_cache.copy()
    table = np.asarray(block_table).copy()
    B, Lmax = path.shape
    slot_map = np.full((B, Lmax), -1, dtype=np.int64)
    new_len = np.asarray(prefix_len, dtype=np.int64).copy()
    remapped = np.zeros(B, dtype=np.int64)
    for b in range(B):
        P = int(prefix_len[b])
        L = int(path_len[b])
        if not (is_valid_tree(parents[b]) and is_valid_path(parents[b], path[b], L)):
            continue
        old_row = np.asarray(block_table[b])
        new_row = table[b]
        plan = remap_plan(P, path[b], L, block_size)
        for m, j in plan:
            new_row[m], new_row[m + j] = new_row[m + j], new_row[m]
        taken = {m for m, _ in plan}
        src = [physical_slot(old_row, P + int(path[b][r]), block_size) for r in range(L)]
        saved_k = [k_cache[s // block_size, :, s % block_size, :].copy() for s in src]
        saved_v = [v_cache[s // block_size, :, s % block_size, :].copy() for s in src]
        for r in range(L):
            slot_map[b, r] = src[r]
            if (P + r) // block_size in taken:
                continue
            dst = physical_slot(new_row, P + r, block_size)
            kc[dst // block_size, :, dst % block_size, :] = saved_k[r]
            vc[dst // block_size, :, dst % block_size, :] = saved_v[r]
        new_len[b] = P + L
        remapped[b] = len(plan)
    return kc, vc, table, slot_map, new_len, remapped
