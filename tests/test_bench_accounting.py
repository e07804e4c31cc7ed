"""The benchmark's algorithmic bytes and FLOPs (the numerators of its roofline figures), checked
against counts written out tensor by tensor at the workload's sizes, and against brute force on
small trees (CPU only)."""
import numpy as np

import bench
import workloads as W
from oracle import tree as T

# the batch-64 GDN layer: B=64, N=40, H=16, dk=dv=128, bf16 inputs and states
B, N, H, D = 64, 40, 16, 128
STATE = B * H * D * D * 2                 # S_0, bf16
NODE_STATE = B * N * H * D * D * 2        # one snapshot per node, bf16


def test_snapshot_pass_bytes():
    """S_0, k (bf16), w (fp32), alpha (fp32) and parents in; every snapshot out."""
    want = STATE + B * N * H * D * 2 + B * N * H * D * 4 + B * N * H * 4 + B * N * 4 + NODE_STATE
    assert bench.gdn_bytes(B, N, H, D, D, 2, 2, "materialize") == want == 1_407_363_072


def test_fork_verify_bytes():
    """S_0, q, k, v (bf16), alpha and beta (fp32), parents in; outputs and snapshots out."""
    inputs = STATE + B * N * H * 3 * D * 2 + B * N * H * 8 + B * N * 4
    want = inputs + B * N * H * D * 2 + NODE_STATE
    assert bench.gdn_bytes(B, N, H, D, D, 2, 2, "fork") == want == 1_418_012_672


def test_treewy_bytes():
    """The same inputs; outputs (bf16), W (fp32) and log gamma (fp32) out."""
    inputs = STATE + B * N * H * 3 * D * 2 + B * N * H * 8 + B * N * 4
    want = inputs + B * N * H * D * 2 + B * N * H * D * 4 + B * N * H * 4
    assert bench.gdn_bytes(B, N, H, D, D, 2, 2, "wy") == want == 96_970_752


def test_commit_bytes():
    """Fork: S_0 written, the accepted snapshot read, the path read.  TreeWY: S_0 read and
    written, plus w (fp32), k (bf16) and log gamma of every accepted entry."""
    assert bench.gdn_bytes(B, N, H, D, D, 2, 2, "commit_fork") == 2 * STATE + B * N * 4 == 67_119_104
    L_sum = 159
    want = 2 * STATE + L_sum * H * (D * 4 + D * 2 + 4) + B * N * 4
    assert bench.gdn_bytes(B, N, H, D, D, 2, 2, "commit_wy", L_sum) == want


def test_checkpoint_bytes_match_the_pages_accounting():
    # one checkpoint of the 24-layer, 16-head, 128 x 128 bf16 stack: 12,582,912 bytes
    assert bench.checkpoint_bytes(24, 16, 128, 128, 2) == 12_582_912


def test_attention_bytes_by_tensor():
    P = [2048, 5000, 32768]
    Hq, Hkv, hd, n = 16, 4, 256, 40
    kv = sum(P) * Hkv * hd * 2 * 2                     # prefix K and V once
    node_in = len(P) * n * (Hq + 2 * Hkv) * hd * 2     # q, k_new, v_new
    out = len(P) * n * (2 * Hkv + Hq) * hd * 2         # node K/V into the cache, the output
    assert bench.attn_bytes(P, n, Hq, Hkv, hd) == kv + node_in + out


def test_attention_flops_by_brute_force():
    """4 * hd flops per (query head, visible key): count the visible keys from the tree mask."""
    rng = np.random.default_rng(0)
    trees = [W.full_tree(3, 2), W.random_tree(30, rng), W.chain(7)]
    prefix = [100, 7, 0]
    Hq, hd = 4, 64
    want = 0
    for t, p in zip(trees, prefix):
        visible = p * len(t) + int(T.tree_mask(t).sum())
        want += 4 * Hq * hd * visible
    got = bench.attn_flops(prefix, [bench._depths(t) for t in trees], Hq, hd)
    assert got == want
    for t in trees:
        assert bench._depths(t) == list(T.depths(t))


def test_compaction_bytes():
    # each kept entry: K and V rows of every KV head, read once and written once
    assert bench.compact_bytes([1, 4, 3], 4, 256) == 8 * 4 * 256 * 2 * 2 * 2
