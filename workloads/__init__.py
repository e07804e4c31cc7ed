"""Seeded synthetic inputs shaped like the pages' workloads.

This module is shared by the fp64 oracle's tests and by the CUDA path's tests and
benchmark.  It holds none of the method's arithmetic: it only draws random numbers
(numpy PCG64, explicit seed, fixed draw order), shapes them into trees, paths and
tensors, and rounds them to the storage dtype.  Both sides consume exactly the
arrays built here; the oracle upcasts the rounded values to fp64.

Shapes follow the two pages' workloads:

* draft trees given by a ``parents`` array, ``parents[i] < i``, root ``-1``, numbered in
  breadth-first order like the draft-tree builder of the handbook chapter
  (树形草稿与 EAGLE, §实现, ``build_draft_tree``);
* gated-DeltaNet inputs per (sequence, node, head): unit-norm q and k, v ~ N(0,1),
  decay ``alpha = exp(-softplus(x))`` and write strength ``beta = sigmoid(x)`` with
  x ~ N(0,1), committed state ``S_0`` ~ N(0, 0.02^2);
* tree attention inputs: node q / k / v ~ N(0,1), a committed KV prefix ~ N(0,1)
  (stored already rotated) in a paged cache of 16-token blocks reached through a
  randomly permuted block table.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


# ----------------------------------------------------------------------------- trees
def chain(n: int) -> list[int]:
    """A single chain of ``n`` nodes: ``[-1, 0, 1, ..., n-2]``."""
    return [-1] + list(range(n - 1))


def branching_tree(branching: list[int]) -> list[int]:
    """Root plus, at level l, ``branching[l]`` children under every node of level l-1.

    This is the shape the handbook chapter's draft builder produces (树形草稿与 EAGLE,
    §实现, ``build_draft_tree``): node 0 is the root and nodes are numbered level by level.
    """
    parents, frontier = [-1], [0]
    for width in branching:
        nxt = []
        for node in frontier:
            for _ in range(width):
                parents.append(node)
                nxt.append(len(parents) - 1)
        frontier = nxt
    return parents


def candidate_chains(lengths: list[int]) -> list[int]:
    """A root with one draft chain per entry of ``lengths`` under it, each chain numbered
    contiguously (depth-first order, so ``parents[i] < i`` still holds)."""
    parents = [-1]
    for length in lengths:
        parents.append(0)
        for _ in range(length - 1):
            parents.append(len(parents) - 1)
    return parents


def full_tree(k: int, d: int) -> list[int]:
    """Full k-ary tree of depth ``d`` below the root, numbered breadth-first."""
    return branching_tree([k] * d)


def random_tree(n: int, rng: np.random.Generator, max_children: int = 4,
                max_depth: int = 8) -> list[int]:
    """Random dynamic tree of exactly ``n`` nodes, numbered breadth-first.

    Nodes are expanded in breadth-first order; each expanded node draws c ~ U{1..max_children}
    children until ``n`` nodes exist; nodes at ``max_depth`` are not expanded.  If the
    frontier empties first the caller's generator simply draws again (at most 1000 times).
    """
    for _ in range(1000):
        parents, depth = [-1], [0]
        head = 0
        while len(parents) < n and head < len(parents):
            node = head
            head += 1
            if depth[node] >= max_depth:
                continue
            c = int(rng.integers(1, max_children + 1))
            for _ in range(c):
                if len(parents) == n:
                    break
                parents.append(node)
                depth.append(depth[node] + 1)
        if len(parents) == n:
            return parents
    raise ValueError(f"no tree of {n} nodes with <= {max_children} children and depth <= {max_depth}")


def random_accepted_path(parents: list[int], rng: np.random.Generator,
                         max_len: int | None = None) -> list[int]:
    """A random root-to-node path: walk from node 0 to a leaf choosing a uniform child at
    each step, then keep a prefix of uniform length in 1..len (capped at ``max_len``)."""
    children: dict[int, list[int]] = {}
    for i, p in enumerate(parents):
        children.setdefault(p, []).append(i)
    path = [0]
    while path[-1] in children:
        kids = children[path[-1]]
        path.append(kids[int(rng.integers(0, len(kids)))])
    hi = len(path) if max_len is None else min(len(path), max_len)
    length = int(rng.integers(1, hi + 1))
    return path[:length]


def walk_tokens(trees: list[list[int]], paths: np.ndarray, path_len: np.ndarray, seed: int,
                vocab: int = 151936) -> tuple[torch.Tensor, torch.Tensor]:
    """Draft and target tokens ``[B, N]`` int32 under which the greedy accept walk takes exactly
    the given paths: draft tokens are distinct within a tree; along the path the target token
    of each node is the draft token of the next path node; at the path's last node it matches
    no child; elsewhere it is random."""
    rng = np.random.default_rng(seed)
    B, N = len(trees), max(len(t) for t in trees)
    draft = np.zeros((B, N), dtype=np.int32)
    target = np.zeros((B, N), dtype=np.int32)
    for b, parents in enumerate(trees):
        n = len(parents)
        draft[b, :n] = rng.choice(vocab, size=n, replace=False)
        target[b, :n] = rng.integers(0, vocab, size=n)
        L = int(path_len[b])
        for r in range(L - 1):
            target[b, paths[b, r]] = draft[b, paths[b, r + 1]]
        last = int(paths[b, L - 1])
        kids = {int(draft[b, c]) for c in range(n) if parents[c] == last}
        t = int(rng.integers(0, vocab))
        while t in kids:
            t = int(rng.integers(0, vocab))
        target[b, last] = t
    return torch.from_numpy(draft), torch.from_numpy(target)


# ----------------------------------------------------------------------------- dtypes
def round_to(x: np.ndarray, dtype: str) -> torch.Tensor:
    """fp32 numpy -> CPU torch tensor in the storage dtype (round-to-nearest-even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(_TORCH_DTYPES[dtype])


def f64(t: torch.Tensor) -> np.ndarray:
    """The stored values of a CPU tensor, upcast exactly to fp64."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def _unit(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def _pad_int(rows: list[list[int]], fill: int) -> np.ndarray:
    width = max(1, max(len(r) for r in rows))
    out = np.full((len(rows), width), fill, dtype=np.int32)
    for b, r in enumerate(rows):
        out[b, :len(r)] = r
    return out


# ----------------------------------------------------------------------------- GDN
@dataclass
class GDNCase:
    """Inputs of one gated-DeltaNet tree-verify layer.

    ``q, k [B,N,H,dk]``, ``v [B,N,H,dv]`` in the I/O dtype; ``alpha, beta [B,N,H]`` fp32;
    ``S0 [B,H,dv,dk]`` in the state dtype; ``parents [B,N]`` int32; ``path [B,Lmax]``
    int32 (-1 padded) with ``path_len [B]``.
    """
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    alpha: torch.Tensor
    beta: torch.Tensor
    S0: torch.Tensor
    parents: torch.Tensor
    path: torch.Tensor
    path_len: torch.Tensor
    io: str
    state: str
    q_scale: float = 1.0
    trees: list = field(default_factory=list)

    @property
    def shape(self):
        B, N, H, dk = self.q.shape
        return B, N, H, dk, self.v.shape[-1]

    def oracle_inputs(self) -> dict:
        """fp64 numpy views of the stored (rounded) values."""
        return dict(q=f64(self.q), k=f64(self.k), v=f64(self.v), alpha=f64(self.alpha),
                    beta=f64(self.beta), S0=f64(self.S0), parents=self.parents.numpy().copy(),
                    q_scale=float(self.q_scale))


def gdn_case(trees: list[list[int]], H: int, dk: int, dv: int, io: str, state: str,
             seed: int, paths: list[list[int]] | None = None, q_scale: float = 1.0,
             path_max_len: int | None = None) -> GDNCase:
    """Draw one GDN layer's inputs for ``B = len(trees)`` sequences with ``N`` nodes each.

    Draw order: q, k, v, x_alpha, x_beta, S_0, then one accepted path per sequence.
    """
    B, N = len(trees), len(trees[0])
    assert all(len(t) == N for t in trees)
    rng = np.random.default_rng(seed)
    q = _unit(rng.standard_normal((B, N, H, dk)))
    k = _unit(rng.standard_normal((B, N, H, dk)))
    v = rng.standard_normal((B, N, H, dv))
    alpha = np.exp(-_softplus(rng.standard_normal((B, N, H))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, N, H))))
    S0 = 0.02 * rng.standard_normal((B, H, dv, dk))
    if paths is None:
        paths = [random_accepted_path(t, rng, path_max_len) for t in trees]
    return GDNCase(q=round_to(q, io), k=round_to(k, io), v=round_to(v, io),
                   alpha=round_to(alpha, "f32"), beta=round_to(beta, "f32"),
                   S0=round_to(S0, state), parents=torch.from_numpy(_pad_int(trees, -1)),
                   path=torch.from_numpy(_pad_int(paths, -1)),
                   path_len=torch.tensor([len(p) for p in paths], dtype=torch.int32),
                   io=io, state=state, q_scale=q_scale, trees=trees)


# ----------------------------------------------------------------------------- attention
@dataclass
class AttnCase:
    """Inputs of one tree-masked GQA attention layer over a paged KV prefix.

    ``q [B,N,Hq,hd]``, ``k_new, v_new [B,N,Hkv,hd]`` (pre-RoPE q and k); the caches
    ``k_cache, v_cache [num_blocks,Hkv,16,hd]`` hold each sequence's committed prefix
    (k already rotated) at logical slots ``0..prefix_len-1`` through ``block_table
    [B,max_blocks]``; the table has room for ``prefix_len + N`` slots.
    """
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    prefix_len: torch.Tensor
    parents: torch.Tensor
    path: torch.Tensor
    path_len: torch.Tensor
    rope_theta: float
    block_size: int = BLOCK_SIZE
    trees: list = field(default_factory=list)

    @property
    def shape(self):
        B, N, Hq, hd = self.q.shape
        return B, N, Hq, self.k_new.shape[2], hd


def attn_case(trees: list[list[int]], prefix_lens: list[int], Hq: int, Hkv: int, hd: int,
              seed: int, rope_theta: float = 1e6, dtype: str = "bf16",
              paths: list[list[int]] | None = None, path_max_len: int | None = None,
              spare_blocks: int = 3) -> AttnCase:
    """Draw one attention layer's inputs.

    Draw order: q, k_new, v_new, the block-table permutation, the prefix K and V (per
    logical slot, sequence by sequence), then one accepted path per sequence.  Cache
    slots that hold no prefix token are filled with N(0,1) garbage so that a kernel that
    reads past the prefix is caught.
    """
    B, N = len(trees), len(trees[0])
    bs = BLOCK_SIZE
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, N, Hq, hd))
    k_new = rng.standard_normal((B, N, Hkv, hd))
    v_new = rng.standard_normal((B, N, Hkv, hd))
    need = [(P + N + bs - 1) // bs for P in prefix_lens]
    max_blocks = max(need)
    num_blocks = sum(need) + spare_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    table = np.zeros((B, max_blocks), dtype=np.int32)
    cursor = 0
    for b in range(B):
        table[b, :need[b]] = perm[cursor:cursor + need[b]]
        table[b, need[b]:] = perm[cursor + need[b] - 1] if need[b] else 0
        cursor += need[b]
    kc = np.empty((num_blocks, Hkv, bs, hd), dtype=np.float32)
    vc = np.empty((num_blocks, Hkv, bs, hd), dtype=np.float32)
    for b in range(B):
        n_slots = need[b] * bs
        kb = rng.standard_normal((n_slots, Hkv, hd), dtype=np.float32)
        vb = rng.standard_normal((n_slots, Hkv, hd), dtype=np.float32)
        for s in range(n_slots):
            blk = table[b, s // bs]
            kc[blk, :, s % bs] = kb[s]
            vc[blk, :, s % bs] = vb[s]
    used = set(int(x) for b in range(B) for x in table[b, :need[b]])
    for blk in range(num_blocks):
        if blk not in used:
            kc[blk] = rng.standard_normal((Hkv, bs, hd), dtype=np.float32)
            vc[blk] = rng.standard_normal((Hkv, bs, hd), dtype=np.float32)
    if paths is None:
        paths = [random_accepted_path(t, rng, path_max_len) for t in trees]
    return AttnCase(q=round_to(q, dtype), k_new=round_to(k_new, dtype), v_new=round_to(v_new, dtype),
                    k_cache=round_to(kc, dtype), v_cache=round_to(vc, dtype),
                    block_table=torch.from_numpy(table),
                    prefix_len=torch.tensor(prefix_lens, dtype=torch.int32),
                    parents=torch.from_numpy(_pad_int(trees, -1)),
                    path=torch.from_numpy(_pad_int(paths, -1)),
                    path_len=torch.tensor([len(p) for p in paths], dtype=torch.int32),
                    rope_theta=rope_theta, trees=trees)


# ----------------------------------------------------------------------------- configs
def small_fp32_case(seed: int = 0) -> GDNCase:
    """Single GDN layer, batch 1, H=2, d=64, fp32, tree k=2 d=2 (7 nodes)."""
    return gdn_case([[-1, 0, 0, 1, 1, 2, 2]], H=2, dk=64, dv=64, io="f32", state="f32", seed=seed)


def single_layer_gdn_case(tree: str = "tree", seed: int = 0) -> GDNCase:
    """One GDN layer, H=16, d=128, bf16, batch 1; ``tree`` = "chain" (5 nodes) or "tree" (k=2 d=3)."""
    t = chain(5) if tree == "chain" else full_tree(2, 3)
    return gdn_case([t], H=16, dk=128, dv=128, io="bf16", state="bf16", seed=seed)


def single_layer_attn_case(tree: str = "tree", seed: int = 0) -> AttnCase:
    """One tree attention layer on the single-layer workload's tree (or chain): 16q/4kv, hd 128, prefix 4096, theta 1e6."""
    t = chain(5) if tree == "chain" else full_tree(2, 3)
    return attn_case([t], [4096], Hq=16, Hkv=4, hd=128, seed=seed, rope_theta=1e6)


def stack_b64_layer(layer: int = 0, B: int = 64, seed: int = 0) -> GDNCase:
    """One of the 24 independent GDN layers of the batch-64 stack: B=64, H=16, d=128, bf16, k=3 d=3 trees."""
    t = full_tree(3, 3)
    return gdn_case([t] * B, H=16, dk=128, dv=128, io="bf16", state="bf16",
                    seed=seed * 1000 + layer)


def paged_attn_b32_case(B: int = 32, seed: int = 0, pmin: int = 2048, pmax: int = 32768) -> AttnCase:
    """Tree attention + compaction: B=32, 16q/4kv, hd 256, bf16, P ~ U{2048..32768}, k=3 d=3,
    accepted length 1..4."""
    rng = np.random.default_rng(seed + 7)
    prefix = [int(x) for x in rng.integers(pmin, pmax + 1, size=B)]
    t = full_tree(3, 3)
    return attn_case([t] * B, prefix, Hq=16, Hkv=4, hd=256, seed=seed, rope_theta=1e6,
                     path_max_len=4)


def paged_chains_case(B: int = 32, seed: int = 0, pmin: int = 2048, pmax: int = 32768) -> AttnCase:
    """Compaction on candidate chains: the paged batch-32 shapes (16q/4kv, hd 256, bf16,
    P ~ U{2048..32768}) with a root and chains of 16, 16 and 7 nodes (N = 40) in depth-first
    order; each accepted path runs down one chain, chosen uniformly, for a uniform length
    (1 .. chain length + 1)."""
    rng = np.random.default_rng(seed + 11)
    prefix = [int(x) for x in rng.integers(pmin, pmax + 1, size=B)]
    lengths = CHAIN_LENGTHS
    paths = candidate_chain_paths(lengths, B, rng)
    return attn_case([candidate_chains(lengths)] * B, prefix, Hq=16, Hkv=4, hd=256, seed=seed,
                     rope_theta=1e6, paths=paths)


CHAIN_LENGTHS = [16, 16, 7]


def candidate_chain_paths(lengths: list[int], B: int, rng: np.random.Generator) -> list[list[int]]:
    """One accepted path per sequence of a ``candidate_chains(lengths)`` tree: down one chain,
    chosen uniformly, for a uniform length 1 .. chain length + 1 (root included)."""
    starts = [1 + sum(lengths[:c]) for c in range(len(lengths))]
    paths = []
    for _ in range(B):
        c = int(rng.integers(0, len(lengths)))
        L = int(rng.integers(1, lengths[c] + 2))
        paths.append([0] + list(range(starts[c], starts[c] + L - 1)))
    return paths


def sweep_trees(N: int, B: int, seed: int = 0) -> list[list[int]]:
    """Wide-tree sweep: random dynamic trees (1..4 children per node, depth <= 8), one per sequence."""
    rng = np.random.default_rng(seed + 4000 + N)
    return [random_tree(N, rng) for _ in range(B)]


def sweep_gdn_layer(N: int, B: int, layer: int = 0, seed: int = 0) -> GDNCase:
    return gdn_case(sweep_trees(N, B, seed), H=16, dk=128, dv=128, io="bf16", state="bf16",
                    seed=seed * 1000 + 100 + layer)


def sweep_attn_layer(N: int, B: int, layer: int = 0, seed: int = 0) -> AttnCase:
    return attn_case(sweep_trees(N, B, seed), [8192] * B, Hq=16, Hkv=4, hd=128,
                     seed=seed * 1000 + 500 + layer, rope_theta=1e6)


# ----------------------------------------------------------------------------- device-drawn stacks
# The wide-tree sweep's largest stacks (24 GDN layers at B=128, N=256: ~10 GB of inputs, and 8
# paged attention layers of ~2 GB each) take too long to draw with numpy, so the benchmark draws
# them on the device with a seeded torch generator, in the same distributions as gdn_case and
# attn_case.  Only the benchmark uses these; the parity tests use the numpy cases above.
def _device_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def device_gdn_stack(layers: int, B: int, N: int, H: int, d: int, seed: int, device) -> dict:
    """Stacked inputs of ``layers`` independent GDN layers, bf16 I/O and state: q, k
    [layers,B,N,H,d] unit-norm per (node, head); v [layers,B,N,H,d] ~ N(0,1); alpha =
    exp(-softplus(x)), beta = sigmoid(x) [layers,B,N,H] fp32 with x ~ N(0,1); S0
    [layers,B,H,d,d] ~ N(0, 0.02^2).  Draw order: q, k, v, x_alpha, x_beta, S0."""
    g = _device_gen(seed, device)
    f32 = dict(device=device, dtype=torch.float32, generator=g)

    def unit(shape):
        x = torch.randn(shape, **f32)
        return (x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)).to(torch.bfloat16)

    shape = (layers, B, N, H, d)
    q = unit(shape)
    k = unit(shape)
    v = torch.randn(shape, **f32).to(torch.bfloat16)
    alpha = torch.exp(-torch.nn.functional.softplus(torch.randn((layers, B, N, H), **f32)))
    beta = torch.sigmoid(torch.randn((layers, B, N, H), **f32))
    S0 = (0.02 * torch.randn((layers, B, H, d, d), **f32)).to(torch.bfloat16)
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0)


def device_attn_layer(B: int, N: int, prefix: int, Hq: int, Hkv: int, hd: int, seed: int, device) -> dict:
    """One paged attention layer, bf16: q [B,N,Hq,hd], k_new, v_new [B,N,Hkv,hd] ~ N(0,1); the
    caches [num_blocks,Hkv,16,hd] ~ N(0,1) (the prefix's keys taken as already rotated); a
    block table [B, max_blocks] that hands each sequence ceil((prefix + N) / 16) blocks of a
    random permutation; prefix_len [B] = prefix.  Draw order: q, k_new, v_new, permutation,
    K cache, V cache."""
    g = _device_gen(seed, device)
    f32 = dict(device=device, dtype=torch.float32, generator=g)
    q = torch.randn((B, N, Hq, hd), **f32).to(torch.bfloat16)
    k_new = torch.randn((B, N, Hkv, hd), **f32).to(torch.bfloat16)
    v_new = torch.randn((B, N, Hkv, hd), **f32).to(torch.bfloat16)
    need = (prefix + N + BLOCK_SIZE - 1) // BLOCK_SIZE
    num_blocks = B * need
    perm = torch.randperm(num_blocks, device=device, generator=g).to(torch.int32)
    table = perm.view(B, need).contiguous()
    cache = (num_blocks, Hkv, BLOCK_SIZE, hd)
    k_cache = torch.empty(cache, device=device, dtype=torch.bfloat16)
    v_cache = torch.empty(cache, device=device, dtype=torch.bfloat16)
    for c in (k_cache, v_cache):           # drawn in slices: fp32 staging of one slice at a time
        step = max(1, (1 << 28) // (Hkv * BLOCK_SIZE * hd))
        for s in range(0, num_blocks, step):
            e = min(num_blocks, s + step)
            c[s:e] = torch.randn((e - s,) + cache[1:], **f32).to(torch.bfloat16)
    prefix_len = torch.full((B,), prefix, device=device, dtype=torch.int32)
    return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache, block_table=table,
                prefix_len=prefix_len)
