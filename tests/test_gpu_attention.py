"""GPU vs fp64 oracle: tree-masked GQA attention over a paged prefix, its cache writes, and
KV compaction, through the C ABI."""
import numpy as np
import pytest
import torch

import _gpu
import tree_speculative_verification_gdn_gb300 as tv
import workloads as W
from oracle import attention as A

pytestmark = pytest.mark.gpu


def _check_attn(case, batch=None):
    f = _gpu.attn_f64(case)
    B = case.q.shape[0]
    seqs = list(range(B)) if batch is None else batch
    res = _gpu.run_attn(case)
    assert (res["err"] == 0).all(), res["err"]
    o_ref, kr_ref = _gpu.assert_attention_close(res["out"], f, seqs)
    # cache: node slots hold the rotated keys (bf16) and the values (exact); prefix untouched
    N = case.q.shape[1]
    kc_got, vc_got = _gpu.f32np(res["k_cache"]), _gpu.f32np(res["v_cache"])
    for b in seqs:
        P = int(f["prefix_len"][b])
        tab = f["block_table"][b]
        kg = A.logical_rows(kc_got, tab, P + N)
        vg = A.logical_rows(vc_got, tab, P + N)
        assert np.array_equal(kg[:P], A.logical_rows(f["k_cache"], tab, P))
        assert np.array_equal(vg[:P], A.logical_rows(f["v_cache"], tab, P))
        _gpu.assert_close(kg[P:], kr_ref[b], "bf16", "rotated node keys in cache", stored="bf16")
        assert np.array_equal(vg[P:], f["v_new"][b])
    return res


def test_printed_example_tree():
    case = W.attn_case([[-1, 0, 0, 1, 1, 2]], [29], Hq=4, Hkv=2, hd=64, seed=1)
    _check_attn(case)


def test_single_layer_tree_and_chain():
    _check_attn(W.single_layer_attn_case("tree"))
    _check_attn(W.single_layer_attn_case("chain"))


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_ragged_prefixes_and_sizes(hd):
    rng = np.random.default_rng(hd)
    trees = [W.random_tree(33, rng) for _ in range(4)]
    case = W.attn_case(trees, [0, 1, 17, 300], Hq=8, Hkv=2, hd=hd, seed=hd)
    _check_attn(case)


def test_single_row_tile_at_head_dim_256():
    """At most 128 query rows per KV head (20 nodes x 4 heads): the single-CTA tensor-core
    partial, at head dim 256, with prefixes that end inside a key tile."""
    rng = np.random.default_rng(7)
    trees = [W.random_tree(20, rng) for _ in range(3)]
    case = W.attn_case(trees, [0, 130, 700], Hq=8, Hkv=2, hd=256, seed=7)
    _check_attn(case)


def test_odd_row_tiles_leave_the_last_pair_a_padding_peer():
    """Three tiles of query rows per KV head (70 nodes x 4 heads = 280 rows): the second CTA
    pair's peer holds no row, and still loads its key and value halves."""
    rng = np.random.default_rng(8)
    trees = [W.random_tree(70, rng) for _ in range(2)]
    case = W.attn_case(trees, [5, 333], Hq=8, Hkv=2, hd=128, seed=8)
    _check_attn(case)


@pytest.mark.parametrize("hd", [128, 256])
@pytest.mark.parametrize("Hq,Hkv,n", [(4, 4, 200), (16, 2, 40)])
def test_group_sizes_on_cta_pairs(Hq, Hkv, n, hd):
    """Query-head groups of 1 (128 nodes per tile of query rows, two tiles) and of 8 (16 nodes per
    tile, three tiles, so the second pair's peer tile is padding) on the CTA-pair kernel."""
    rng = np.random.default_rng(Hq * 10 + hd)
    trees = [W.random_tree(n, rng) for _ in range(2)]
    case = W.attn_case(trees, [37, 290], Hq=Hq, Hkv=Hkv, hd=hd, seed=Hq + hd)
    _check_attn(case)


@pytest.mark.parametrize("n", [1, 2, 3])
def test_tiny_trees(n):
    case = W.attn_case([W.chain(n), [-1] * n], [5, 16], Hq=2, Hkv=1, hd=64, seed=n)
    _check_attn(case)


def test_wide_tree_many_words():
    rng = np.random.default_rng(5)
    case = W.attn_case([W.random_tree(256, rng), W.chain(256)], [40, 3], Hq=4, Hkv=4, hd=64, seed=3)
    _check_attn(case)


def test_paged_b32_full_size_sampled():
    """Paged attention at full size: B=32, 16q/4kv, hd 256, P ~ U[2048, 32768] paged, 40-node trees."""
    case = W.paged_attn_b32_case()
    res = _check_attn(case, batch=[0, int(np.argmax(case.prefix_len.numpy())), 31])
    # compaction of the same cache, every sequence, bit-exact
    f = _gpu.attn_f64(case)
    kc_after = _gpu.f32np(res["k_cache"])
    vc_after = _gpu.f32np(res["v_cache"])
    comp = _gpu.run_compact(case, res["k_cache"], res["v_cache"])
    assert (comp["err"] == 0).all()
    kc2, vc2, smap, new_len = A.kv_compact(kc_after, vc_after, f["block_table"], f["prefix_len"],
                                           f["parents"], case.path.numpy(), case.path_len.numpy())
    assert np.array_equal(comp["slot_map"], smap)
    assert np.array_equal(comp["new_len"], new_len)
    kc_comp, vc_comp = _gpu.f32np(comp["k_cache"]), _gpu.f32np(comp["v_cache"])
    for b in range(32):
        n = int(new_len[b])
        tab = f["block_table"][b]
        assert np.array_equal(A.logical_rows(kc_comp, tab, n), A.logical_rows(kc2, tab, n))
        assert np.array_equal(A.logical_rows(vc_comp, tab, n), A.logical_rows(vc2, tab, n))


@pytest.mark.parametrize("N,B", [(40, 4), (128, 2), (256, 2), (40, 128)])
def test_wide_tree_attention_layer_sampled(N, B):
    """Attention layers of the wide-tree sweep (16q/4kv, hd 128, prefix 8192), up to N=256 and
    B=128; the first and last sequences against the oracle."""
    case = W.sweep_attn_layer(N, B)
    _check_attn(case, batch=[0, B - 1])


def test_errors_are_per_sequence():
    tree = [-1, 0, 0, 1]
    case = W.attn_case([tree] * 4, [20, 20, 20, 20], Hq=2, Hkv=1, hd=64, seed=2)
    case.parents[1, 2] = 3                         # malformed tree
    case.prefix_len[2] = case.block_table.shape[1] * 16 - 3   # no room for 4 node slots
    case.block_table[3, 1] = case.k_cache.shape[0] + 5        # block outside the cache
    f = _gpu.attn_f64(case)
    res = _gpu.run_attn(case)
    assert res["err"].tolist() == [0, tv.TV_ERR_BAD_TREE, tv.TV_ERR_CAPACITY, tv.TV_ERR_BAD_BLOCK]
    _gpu.assert_attention_close(res["out"], f, [0], "healthy sequence")
    assert torch.isnan(res["out"][1:].float()).all()


def test_workspace_too_small_is_rejected():
    case = W.attn_case([[-1, 0]], [3], Hq=2, Hkv=1, hd=64, seed=0)
    x = {k: _gpu.to_dev(getattr(case, k)) for k in ("q", "k_new", "v_new", "k_cache", "v_cache",
                                                    "block_table", "prefix_len", "parents")}
    out = torch.empty_like(x["q"])
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(tv.TVError) as e:
        tv.tv_tree_attn(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["block_table"],
                        x["prefix_len"], x["parents"], out, ws, err, rope_theta=1e6)
    assert e.value.status == tv.TV_ERR_INVALID_ARG


def test_compaction_overlaps_and_errors():
    tree = [-1, 0, 1, 0, 3, 4, 5, 2]
    paths = [[0, 3, 4, 5], [0, 1, 2, 7], [0], [0, 2], [0, 3, 4, 5]]
    case = W.attn_case([tree] * 5, [4, 15, 16, 8, 33], Hq=2, Hkv=2, hd=128, seed=4, paths=paths)
    L = case.path_len.clone()
    L[4] = 5                                        # longer than the buffer
    f = _gpu.attn_f64(case)
    comp = _gpu.run_compact(case, case.k_cache, case.v_cache, path_len=L)
    assert comp["err"].tolist() == [0, 0, 0, tv.TV_ERR_BAD_PATH, tv.TV_ERR_BAD_PATH]
    kc2, vc2, smap, new_len = A.kv_compact(f["k_cache"], f["v_cache"], f["block_table"], f["prefix_len"],
                                           f["parents"], case.path.numpy(), L.numpy())
    assert np.array_equal(comp["slot_map"], smap)
    assert np.array_equal(comp["new_len"], new_len)
    assert np.array_equal(_gpu.f32np(comp["k_cache"]), kc2)
    assert np.array_equal(_gpu.f32np(comp["v_cache"]), vc2)


@pytest.mark.parametrize("form", ["move", "remap"])
def test_compaction_rejects_a_window_with_a_repeated_block(form):
    # Logical blocks 1 and 2 of sequence 1 (its tree's slots 20 .. 35) name one physical block:
    # a store could overwrite a source before it is read, so the sequence is refused and its
    # cache left as it was; sequence 0 is compacted as usual.
    tree = [-1, 0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14]
    paths = [[0, 1, 2, 3], [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15]]
    case = W.attn_case([tree] * 2, [20, 20], Hq=2, Hkv=2, hd=64, seed=6, paths=paths)
    case.block_table[1, 2] = case.block_table[1, 1]
    f = _gpu.attn_f64(case)
    if form == "move":
        comp = _gpu.run_compact(case, case.k_cache, case.v_cache)
        kc, vc = _gpu.f32np(comp["k_cache"]), _gpu.f32np(comp["v_cache"])
    else:
        comp = _gpu.run_compact_remap(case.k_cache, case.v_cache, case.block_table, case.prefix_len, case.parents,
                                      case.path, case.path_len)
        kc, vc = _gpu.f32np(comp["k_cache"].cpu()), _gpu.f32np(comp["v_cache"].cpu())
        assert np.array_equal(comp["table"][1], case.block_table.numpy()[1])
        assert int(comp["remapped"][1]) == 0
    assert comp["err"].tolist() == [0, tv.TV_ERR_BAD_BLOCK]
    assert comp["new_len"][1] == 20 and (comp["slot_map"][1] == -1).all()
    for blk in set(case.block_table.numpy()[1]):
        assert np.array_equal(kc[blk], f["k_cache"][blk]) and np.array_equal(vc[blk], f["v_cache"][blk])
    kc2, vc2, smap, new_len = A.kv_compact(f["k_cache"], f["v_cache"], f["block_table"][:1], f["prefix_len"][:1],
                                           f["parents"][:1], case.path.numpy()[:1], case.path_len.numpy()[:1])
    assert np.array_equal(comp["slot_map"][0], smap[0]) and comp["new_len"][0] == new_len[0]
    tab = f["block_table"][0]
    n = int(new_len[0])
    assert np.array_equal(A.logical_rows(kc, tab, n), A.logical_rows(kc2, tab, n))

