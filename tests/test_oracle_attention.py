"""Pins of the oracle's RoPE, tree attention, paged addressing and KV compaction (CPU only).

Library pins use torch's scaled_dot_product_attention in float64 (CPU) on the special cases
that reduce to it: a chain with no prefix (causal attention), a single node (decode), and
each node as its own plain sequence (the handbook chapter's brute-force check).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads as W
from oracle import attention as A
from oracle import tree as T


def _sdpa(q, k, v, causal=False):
    """q [T,H,hd], k/v [S,H,hd] float64 -> [T,H,hd] via torch's SDPA."""
    out = F.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1)[None], torch.from_numpy(k).transpose(0, 1)[None],
        torch.from_numpy(v).transpose(0, 1)[None], is_causal=causal)
    return out[0].transpose(0, 1).numpy()


def test_rope_identity_at_zero_and_norm_preserving():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 16))
    assert np.allclose(A.rope(x, np.zeros(5), 1e6), x)
    y = A.rope(x, np.array([1, 7, 100, 4096, 33000]), 1e6)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1))


def test_rope_two_dims_is_a_plane_rotation_by_position():
    x = np.array([[[0.3, -1.1]]])
    for pos in (0, 1, 5, 1000):
        c, s = np.cos(pos), np.sin(pos)
        want = np.array([0.3 * c + 1.1 * s, -1.1 * c + 0.3 * s])
        assert np.allclose(A.rope(x, np.array([pos]), 10000.0)[0, 0], want)


def test_rope_pairs_dim_i_with_dim_i_plus_half():
    x = np.zeros((1, 1, 8))
    x[0, 0, 1] = 1.0
    y = A.rope(x, np.array([3]), 100.0)[0, 0]
    assert set(np.nonzero(np.abs(y) > 1e-12)[0]) == {1, 5}
    ang = 3 * 100.0 ** (-2 * 1 / 8)
    assert np.isclose(y[1], np.cos(ang)) and np.isclose(y[5], np.sin(ang))


def test_rope_scores_depend_only_on_position_difference():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 1, 32))
    k = rng.standard_normal((1, 1, 32))
    ref = (A.rope(q, np.array([10]), 1e4) * A.rope(k, np.array([3]), 1e4)).sum()
    for shift in (1, 50, 2000):
        got = (A.rope(q, np.array([10 + shift]), 1e4) * A.rope(k, np.array([3 + shift]), 1e4)).sum()
        assert np.isclose(got, ref, rtol=1e-9)


def _f64_case(case):
    return dict(q=W.f64(case.q), k_new=W.f64(case.k_new), v_new=W.f64(case.v_new),
                k_cache=W.f64(case.k_cache), v_cache=W.f64(case.v_cache),
                block_table=case.block_table.numpy(), prefix_len=case.prefix_len.numpy(),
                parents=case.parents.numpy(), rope_theta=case.rope_theta)


def test_chain_without_prefix_is_causal_attention():
    rng = np.random.default_rng(2)
    N, H, hd = 9, 3, 16
    q, k, v = (rng.standard_normal((N, H, hd)) for _ in range(3))
    o, kr = A.attend_one(q, k, v, np.zeros((0, H, hd)), np.zeros((0, H, hd)), W.chain(N), 1e4)
    qr = A.rope(q, np.arange(N), 1e4)
    assert np.allclose(kr, A.rope(k, np.arange(N), 1e4))
    assert np.allclose(o, _sdpa(qr, kr, v, causal=True), atol=1e-12)


def test_single_node_is_decode_attention():
    rng = np.random.default_rng(3)
    P, H, hd = 37, 2, 8
    q, k, v = (rng.standard_normal((1, H, hd)) for _ in range(3))
    pk, pv = rng.standard_normal((P, H, hd)), rng.standard_normal((P, H, hd))
    o, kr = A.attend_one(q, k, v, pk, pv, [-1], 1e6)
    qr = A.rope(q, np.array([P]), 1e6)
    want = _sdpa(qr, np.concatenate([pk, kr]), np.concatenate([pv, v]))
    assert np.allclose(o, want, atol=1e-12)


def test_each_node_equals_prefix_plus_its_path_as_a_plain_sequence():
    """The handbook chapter's correctness check, at the attention level: node i's output equals
    ordinary attention of the last query over prefix + root..i at positions P..P+depth."""
    rng = np.random.default_rng(4)
    tree = [-1, 0, 0, 1, 1, 2]
    N, Hq, Hkv, hd, P = 6, 4, 2, 16, 11
    q = rng.standard_normal((N, Hq, hd))
    k = rng.standard_normal((N, Hkv, hd))
    v = rng.standard_normal((N, Hkv, hd))
    pk, pv = rng.standard_normal((P, Hkv, hd)), rng.standard_normal((P, Hkv, hd))
    o, _ = A.attend_one(q, k, v, pk, pv, tree, 1e6)
    for i in range(N):
        path = T.path_to(tree, i)
        pos = P + np.arange(len(path))
        kr = A.rope(k[path], pos, 1e6)
        qr = A.rope(q[[i]], pos[-1:], 1e6)
        K = np.concatenate([pk, kr]).repeat(Hq // Hkv, axis=1)
        V = np.concatenate([pv, v[path]]).repeat(Hq // Hkv, axis=1)
        assert np.allclose(o[i], _sdpa(qr, K, V)[0], atol=1e-12)


def test_equal_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(5)
    tree = [-1, 0, 0, 1, 2, 2, 5]
    N, H, hd, P = 7, 2, 4, 5
    q = rng.standard_normal((N, H, hd))
    k = np.zeros((N, H, hd))          # rotation of a zero key is zero
    pk = np.zeros((P, H, hd))
    v = rng.standard_normal((N, H, hd))
    pv = rng.standard_normal((P, H, hd))
    o, _ = A.attend_one(q, k, v, pk, pv, tree, 1e6)
    mask = T.tree_mask(tree)
    for i in range(N):
        vis = np.concatenate([pv, v[mask[i]]])
        assert np.allclose(o[i], vis.mean(axis=0), atol=1e-13)


def test_gqa_reads_kv_head_h_div_group():
    rng = np.random.default_rng(6)
    tree = [-1, 0, 1, 1]
    N, Hq, Hkv, hd, P = 4, 6, 2, 8, 9
    q = rng.standard_normal((N, Hq, hd))
    k, v = rng.standard_normal((N, Hkv, hd)), rng.standard_normal((N, Hkv, hd))
    pk, pv = rng.standard_normal((P, Hkv, hd)), rng.standard_normal((P, Hkv, hd))
    o, _ = A.attend_one(q, k, v, pk, pv, tree, 1e6)
    rep = lambda x: torch.from_numpy(x).repeat_interleave(Hq // Hkv, dim=1).numpy()  # noqa: E731
    o2, _ = A.attend_one(q, rep(k), rep(v), rep(pk), rep(pv), tree, 1e6)
    assert np.allclose(o, o2, atol=1e-14)


def test_paged_gather_matches_contiguous_layout():
    case = W.attn_case([W.full_tree(2, 2)] * 3, [5, 40, 16], Hq=2, Hkv=2, hd=8, seed=1)
    f = _f64_case(case)
    for b in range(3):
        P = int(f["prefix_len"][b])
        rows = A.logical_rows(f["k_cache"], f["block_table"][b], P + 7)
        for s in range(P + 7):
            blk = f["block_table"][b][s // 16]
            assert np.array_equal(rows[s], f["k_cache"][blk, :, s % 16, :])
            assert A.physical_slot(f["block_table"][b], s) == blk * 16 + s % 16


def test_paged_attention_equals_contiguous_attention():
    case = W.attn_case([W.full_tree(2, 2), [-1, 0, 1, 2, 3, 4, 5]], [20, 3], Hq=4, Hkv=2, hd=8,
                       seed=2)
    f = _f64_case(case)
    o, kr = A.tree_attention(f)
    for b in range(2):
        P = int(f["prefix_len"][b])
        pk = A.logical_rows(f["k_cache"], f["block_table"][b], P)
        pv = A.logical_rows(f["v_cache"], f["block_table"][b], P)
        ob, krb = A.attend_one(f["q"][b], f["k_new"][b], f["v_new"][b], pk, pv, f["parents"][b],
                               f["rope_theta"])
        assert np.array_equal(o[b], ob) and np.array_equal(kr[b], krb)
    kc, vc = A.cache_after_attention(f, kr)
    for b in range(2):
        P = int(f["prefix_len"][b])
        rows = A.logical_rows(kc, f["block_table"][b], P + 7)
        assert np.array_equal(rows[:P], A.logical_rows(f["k_cache"], f["block_table"][b], P))
        assert np.array_equal(rows[P:], kr[b])


def test_compaction_moves_path_slots_and_leaves_the_rest():
    tree = [-1, 0, 0, 1, 1, 2, 2]
    case = W.attn_case([tree] * 4, [16, 3, 30, 8], Hq=2, Hkv=2, hd=4, seed=3,
                       paths=[[0, 2, 6], [0, 1, 4], [0], [0, 3]])
    f = _f64_case(case)
    path, L = case.path.numpy(), case.path_len.numpy()
    kc, vc, smap, new_len = A.kv_compact(f["k_cache"], f["v_cache"], f["block_table"],
                                         f["prefix_len"], f["parents"], path, L)
    for b in range(4):
        P = int(f["prefix_len"][b])
        tab = f["block_table"][b]
        before = A.logical_rows(f["k_cache"], tab, P + 7)
        after = A.logical_rows(kc, tab, P + 7)
        if b == 3:      # 3 is not a child of 0: untouched
            assert new_len[b] == P and np.array_equal(after, before)
            assert (smap[b] == -1).all()
            continue
        assert new_len[b] == P + L[b]
        assert np.array_equal(after[:P], before[:P])
        for r in range(L[b]):
            assert np.array_equal(after[P + r], before[P + path[b][r]])
            assert smap[b, r] == A.physical_slot(tab, P + path[b][r])
        assert (smap[b, L[b]:] == -1).all()
        # compaction writes only slots P..P+L-1
        assert np.array_equal(after[P + L[b]:], before[P + L[b]:])
        assert np.array_equal(A.logical_rows(vc, tab, P + 7)[P + L[b]:],
                              A.logical_rows(f["v_cache"], tab, P + 7)[P + L[b]:])


def test_compaction_handles_overlapping_moves():
    """A chain path [0, 1, 2] is the identity; a path whose node index exceeds its rank moves
    entries down, reading every source before any write."""
    tree = [-1, 0, 1, 0, 3, 4]
    case = W.attn_case([tree], [4], Hq=1, Hkv=1, hd=4, seed=4, paths=[[0, 3, 4, 5]])
    f = _f64_case(case)
    kc, _, _, _ = A.kv_compact(f["k_cache"], f["v_cache"], f["block_table"], f["prefix_len"],
                               f["parents"], case.path.numpy(), case.path_len.numpy())
    before = A.logical_rows(f["k_cache"], f["block_table"][0], 10)
    after = A.logical_rows(kc, f["block_table"][0], 10)
    for r, node in enumerate([0, 3, 4, 5]):
        assert np.array_equal(after[4 + r], before[4 + node])


@pytest.mark.parametrize("hd", [8, 16])
def test_block_boundary_prefix_lengths(hd):
    tree = [-1, 0, 0]
    for P in (0, 1, 15, 16, 17, 31, 32):
        case = W.attn_case([tree], [P], Hq=2, Hkv=1, hd=hd, seed=P)
        f = _f64_case(case)
        o, _ = A.tree_attention(f)
        assert np.isfinite(o).all()


def test_bf16_round_is_round_to_nearest_even_at_8_significant_bits():
    # ties go to the even neighbour, anything past a tie goes up
    vals = np.array([1 + 2.0**-8, 1 + 3 * 2.0**-8, -(1 + 2.0**-8), 1 + 2.0**-8 + 2.0**-20, 3 * 2.0**-9, 255.0, 255.5])
    want = np.array([1.0, 1 + 2.0**-6, -1.0, 1 + 2.0**-7, 3 * 2.0**-9, 255.0, 256.0])
    assert np.array_equal(A.bf16_round(vals), want)
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000) * 10.0 ** rng.uniform(-6, 6, 20000)
    r = A.bf16_round(x)
    assert (np.abs(r - x) <= 2.0**-8 * np.abs(x)).all()          # at most half an ulp
    assert np.array_equal(A.bf16_round(r), r)                      # representable: a fixed point
    e = np.floor(np.log2(np.abs(r)))
    assert np.array_equal(np.ldexp(r, (7 - e).astype(int)) % 1, np.zeros_like(r))  # 8 significant bits


def test_bf16_query_is_the_plain_result_where_the_query_is_not_rotated():
    # one node and no prefix: the query sits at position 0, where the rotation is the identity,
    # and a bf16 input is already representable, so rounding the rotated query changes nothing
    f = _f64_case(W.attn_case([[-1]], [0], Hq=4, Hkv=2, hd=64, seed=3))
    o, _ = A.tree_attention(f)
    o_rq, _ = A.tree_attention(f, query_bf16=True)
    assert np.array_equal(o, o_rq)


def test_bf16_query_moves_the_output_by_a_few_hundredths_of_its_rms():
    # rotated queries off position 0 are not bf16 values: the option acts, and by no more than
    # about the half-ulp rounding of the query can move a softmax average
    rng = np.random.default_rng(4)
    f = _f64_case(W.attn_case([W.random_tree(30, rng)], [200], Hq=4, Hkv=2, hd=128, seed=4))
    o, _ = A.tree_attention(f)
    o_rq, _ = A.tree_attention(f, query_bf16=True)
    d = np.abs(o_rq - o)
    rms = np.sqrt(np.mean(o ** 2))
    assert d.max() > 0 and d.max() < 0.05 * rms
