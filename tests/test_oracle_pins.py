"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against brute force on tiny inputs written in a
different form (explicit masks and Python loops over ``math.exp``), closed
forms, special cases the pages state, or invariants; a dropped term, wrong
sign, wrong index or transposed operand in the oracle fails one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import hs2_oracle as O
from top_hs2_fa_gb300 import workloads as W
from top_hs2_fa_gb300 import counting as C

GOLD = os.path.join(os.path.dirname(__file__), "golden", "counting_examples.json")


# ----------------------------------------------------------------------------- brute-force helpers
def dense_masked_bruteforce(Q, K, V, scale):
    """Causal attention of rows Q[i] (row i sees keys 0..i) with an explicit boolean
    n x n mask and a per-row softmax written with Python loops and math.exp."""
    n, d = Q.shape
    mask = [[s <= i for s in range(n)] for i in range(n)]
    out = np.zeros((n, V.shape[1]))
    lse = np.zeros(n)
    for i in range(n):
        logits = [float(Q[i] @ K[s]) * scale if mask[i][s] else -math.inf for s in range(n)]
        m = max(logits)
        ex = [math.exp(x - m) if x != -math.inf else 0.0 for x in logits]
        z = sum(ex)
        lse[i] = m + math.log(z)
        for s in range(n):
            out[i] += (ex[s] / z) * V[s]
    return out, lse


def prob_table(Q, K, scale):
    """p[h][s] = exp(x) / sum exp(x) with Python loops (ratio form, no lse)."""
    H = Q.shape[0]
    t = K.shape[0]
    p = np.zeros((H, t))
    for h in range(H):
        ex = [math.exp(float(Q[h] @ K[s]) * scale) for s in range(t)]
        z = sum(ex)
        for s in range(t):
            p[h, s] = ex[s] / z
    return p


def contiguous_rows(kv, b, g, t):
    return O.gather_rows(kv.k, kv.block_table[b], g, np.arange(t), kv.page, kv.dtype), \
        O.gather_rows(kv.v, kv.block_table[b], g, np.arange(t), kv.page, kv.dtype)


# ----------------------------------------------------------------------------- FA output
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (2, 1), (3, 3)])
def test_fa_prefill_matches_masked_dense(Hq, Hkv):
    n, d = 37, 8
    grp = W.prefill_group(n, Hq, Hkv, d, w=4, k=5, dtype="f32", seed=11, n_sa=0, page=8, permute=True)
    kv = grp.kv
    o, lse, _, _ = O.fa_prefill_rows(grp.q_fa, kv, np.arange(n), grp.w, grp.k, grp.scale)
    Q = O.to_f64(grp.q_fa, "f32")
    G = Hq // Hkv
    for g in range(Hkv):
        K, V = contiguous_rows(kv, 0, g, n)
        for h in range(g * G, (g + 1) * G):
            ref, ref_lse = dense_masked_bruteforce(Q[:, h], K, V, grp.scale)
            np.testing.assert_allclose(o[:, h], ref, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[:, h], ref_lse, rtol=0, atol=1e-12)


def test_fa_closed_forms():
    # identical keys -> uniform attention: o = mean of visible V, lse = x0 + log t
    d, t = 8, 20
    rng = np.random.default_rng(0)
    q = rng.standard_normal((3, d))
    k0 = rng.standard_normal(d)
    K = np.repeat(k0[None], t, 0)
    V = rng.standard_normal((t, d))
    x, lse, o = O.full_attention(q, K, V, 0.5)
    np.testing.assert_allclose(o, np.repeat(V.mean(0)[None], 3, 0), atol=1e-13)
    np.testing.assert_allclose(lse, 0.5 * (q @ k0) + math.log(t), atol=1e-13)
    # identical values -> output is that value whatever the logits
    V2 = np.repeat(V[:1], t, 0)
    _, _, o2 = O.full_attention(q, rng.standard_normal((t, d)), V2, 0.5)
    np.testing.assert_allclose(o2, V2[:3], atol=1e-13)


def test_gather_rows_follows_block_table():
    kv = W.random_paged_kv([150, 70], Hkv=2, d=4, dtype="f32", seed=5, page=16)
    for b, t in enumerate([150, 70]):
        for s in (0, 15, 16, t - 1):
            page = kv.block_table[b][s // 16]
            row = O.gather_rows(kv.k, kv.block_table[b], 1, np.array([s]), 16, "f32")[0]
            np.testing.assert_array_equal(row, kv.k[page, 1, s % 16].astype(np.float64))


# ----------------------------------------------------------------------------- selection
def test_window_and_far_range_match_one_based_statement():
    # window [t-w+1, t] in 1-based positions == [t-w, t-1] 0-based; far count min(k, t-w)
    for t, w in [(10, 3), (3, 3), (2, 5), (1, 1)]:
        win = O.window(t, w)
        assert list(win + 1) == list(range(max(1, t - w + 1), t + 1))
        assert O.far_count(t, w) == max(0, t - w)


def test_selection_scores_against_ratio_form():
    rng = np.random.default_rng(3)
    t, d, G, w = 12, 5, 3, 4
    Q = rng.standard_normal((G, d)) * np.array([[3.0], [0.3], [1.0]])  # very different lse per head
    K = rng.standard_normal((t, d))
    x, lse, _ = O.full_attention(Q, K, K, 0.7)
    sc = O.selection_scores(x, lse, t - w)
    p = prob_table(Q, K, 0.7)
    np.testing.assert_allclose(sc, p[:, :t - w].sum(0), atol=1e-14)
    # over all positions each head's probabilities sum to one
    np.testing.assert_allclose(O.selection_scores(x, lse, t).sum(), G, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_topk_is_best_subset_bruteforce(seed):
    rng = np.random.default_rng(100 + seed)
    t, w, d, G = int(rng.integers(5, 12)), int(rng.integers(0, 4)), 4, 2
    k = int(rng.integers(1, 4))
    Q = rng.standard_normal((G, d))
    K = rng.standard_normal((t, d)) * 1.5
    x, lse, _ = O.full_attention(Q, K, K, 1.0)
    nf = O.far_count(t, w)
    sc = O.selection_scores(x, lse, nf)
    sel = O.topk_lower_index(sc, k)
    p = prob_table(Q, K, 1.0)
    best, best_sum = None, -1.0
    for sub in itertools.combinations(range(nf), min(k, nf)):
        s = sum(p[h, j] for h in range(G) for j in sub)
        if s > best_sum:
            best, best_sum = sub, s
    assert tuple(sel) == tuple(best)


def test_selection_invariants_and_short_context():
    grp = W.decode_group([5, 20, 130, 131, 700], Hq=4, Hkv=2, d=16, w=8, k=100, dtype="f32",
                         seed=7, n_sa=0, needles=0, page=16)
    o, lse, idx, cnt = O.fa_decode(grp.q_fa, grp.kv, 8, 100, grp.scale)
    for b, t in enumerate([5, 20, 130, 131, 700]):
        for g in range(2):
            sel = idx[b, g, :cnt[b, g]]
            assert cnt[b, g] == min(100, max(0, t - 8))
            assert np.all(idx[b, g, cnt[b, g]:] == -1)
            assert np.all(np.diff(sel) > 0)
            assert sel.size == 0 or (sel.min() >= 0 and sel.max() < t - 8)
            assert not set(sel) & set(O.window(t, 8))
            if t - 8 <= 100:  # k covers the far range: S = F
                assert list(sel) == list(range(max(0, t - 8)))


def test_ties_go_to_lower_position():
    # identical keys -> every far position has the same score -> the first k win
    d, t, w, k = 8, 50, 5, 7
    rng = np.random.default_rng(1)
    K = np.repeat(rng.standard_normal(d)[None], t, 0)
    q = rng.standard_normal((2, d))
    x, lse, _ = O.full_attention(q, K, K, 0.3)
    sel = O.topk_lower_index(O.selection_scores(x, lse, t - w), k)
    assert list(sel) == list(range(k))
    assert list(O.topk_lower_index(np.array([1.0, 2.0, 2.0, 1.0, 2.0]), 2)) == [1, 2]


def test_mqa_order_equals_logit_order():
    rng = np.random.default_rng(9)
    t, d, w, k = 300, 16, 10, 40
    q = rng.standard_normal((1, d))
    K = rng.standard_normal((t, d))
    x, lse, _ = O.full_attention(q, K, K, 0.25)
    sel = O.topk_lower_index(O.selection_scores(x, lse, t - w), k)
    ref = np.sort(np.argsort(-x[0, :t - w], kind="stable")[:k])
    assert list(sel) == list(ref)


def test_needles_are_selected():
    tg = W.tiny_group(n=600, Hq=4, Hkv=1, d=64, w=16, k=64, needles=8, seed=0)
    dec = tg.decode
    _, _, idx, cnt = O.fa_decode(dec.q_fa, dec.kv, dec.w, dec.k, dec.scale)
    assert set(dec.needles[0].tolist()) <= set(idx[0, 0, :cnt[0, 0]].tolist())


# ----------------------------------------------------------------------------- SA
def test_sa_equals_dense_when_k_covers_far_range():
    grp = W.decode_group([40, 64, 65, 129], Hq=4, Hkv=2, d=8, w=6, k=200, dtype="f32", seed=2,
                         n_sa=1, needles=0, page=16)
    kv = grp.kv
    _, _, idx, cnt = O.fa_decode(grp.q_fa, kv, grp.w, grp.k, grp.scale)
    o_sa = O.sa_decode(grp.q_sa[0], kv, grp.w, idx, cnt, grp.scale)
    Qs = O.to_f64(grp.q_sa[0], "f32")
    for b, t in enumerate([40, 64, 65, 129]):
        for h in range(4):
            K, V = contiguous_rows(kv, b, h // 2, t)
            # dense attention of the SA query over all t keys = last row of a causal pass
            Qfull = np.zeros((t, 8))
            Qfull[t - 1] = Qs[b, h]
            ref, _ = dense_masked_bruteforce(Qfull, K, V, grp.scale)
            np.testing.assert_allclose(o_sa[b, h], ref[t - 1], atol=1e-12)


def test_sa_window_zero_with_everything_selected_is_dense():
    rng = np.random.default_rng(4)
    t, d = 33, 8
    kv = W.random_paged_kv([t], Hkv=1, d=d, dtype="f32", seed=8, page=8)
    q = rng.standard_normal((1, 2, d)).astype(np.float32)
    idx = np.arange(t, dtype=np.int32).reshape(1, 1, t)
    o = O.sa_decode(q, kv, 0, idx, np.array([[t]], np.int32), 0.4)
    K, V = contiguous_rows(kv, 0, 0, t)
    p = prob_table(q[0].astype(np.float64), K, 0.4)
    np.testing.assert_allclose(o[0], p @ V, atol=1e-12)


def test_sa_renormalisation_error_bound():
    grp = W.decode_group([300] * 3, Hq=8, Hkv=2, d=16, w=8, k=20, dtype="f32", seed=12, n_sa=1,
                         needles=4, page=16)
    kv = grp.kv
    _, _, idx, cnt = O.fa_decode(grp.q_fa, kv, grp.w, grp.k, grp.scale)
    o_sa = O.sa_decode(grp.q_sa[0], kv, grp.w, idx, cnt, grp.scale)
    Qs = O.to_f64(grp.q_sa[0], "f32")
    for b in range(3):
        for h in range(8):
            g = h // 4
            K, V = contiguous_rows(kv, b, g, 300)
            _, _, o_dense = O.full_attention(Qs[b, h:h + 1], K, V, grp.scale)
            p = prob_table(Qs[b, h:h + 1], K, grp.scale)[0]
            keep = np.concatenate([O.window(300, grp.w), idx[b, g, :cnt[b, g]]])
            err = np.sqrt(((o_sa[b, h] - o_dense[0]) ** 2).sum())
            assert err <= O.renormalisation_bound(p, keep, V) + 1e-12


def test_paging_is_invisible():
    grp = W.decode_group([100, 37], Hq=2, Hkv=1, d=8, w=4, k=9, dtype="bf16", seed=21, n_sa=1,
                         needles=2, page=16, permute=True)
    kv = grp.kv
    res1 = O.fa_decode(grp.q_fa, kv, 4, 9, grp.scale)
    # move every page to a new physical slot and rewrite the table
    perm = np.random.default_rng(0).permutation(kv.num_pages)
    inv = np.argsort(perm)
    kv2 = W.PagedKV(k=kv.k[perm], v=kv.v[perm], block_table=np.where(kv.block_table >= 0, inv[np.maximum(kv.block_table, 0)], -1).astype(np.int32),
                    seq_len=kv.seq_len, dtype=kv.dtype, page=kv.page)
    res2 = O.fa_decode(grp.q_fa, kv2, 4, 9, grp.scale)
    for a, b in zip(res1, res2):
        np.testing.assert_array_equal(a, b)
    s1 = O.sa_decode(grp.q_sa[0], kv, 4, res1[2], res1[3], grp.scale)
    s2 = O.sa_decode(grp.q_sa[0], kv2, 4, res1[2], res1[3], grp.scale)
    np.testing.assert_array_equal(s1, s2)


def test_sa_rejects_overlapping_sets():
    kv = W.random_paged_kv([20], Hkv=1, d=4, dtype="f32", seed=1, page=8)
    q = np.zeros((1, 1, 4), np.float32)
    with pytest.raises(ValueError):
        O.sa_decode(q, kv, 4, np.array([[[17, -1]]], np.int32), np.array([[1]], np.int32), 1.0)


def test_decode_equals_last_prefill_row():
    tg = W.tiny_group(n=200, Hq=4, Hkv=1, d=16, w=8, k=12, needles=3, seed=4)
    dec, pre = tg.decode, tg.prefill
    kv_full = W.PagedKV(k=pre.kv.k, v=pre.kv.v, block_table=pre.kv.block_table,
                        seq_len=np.array([201], np.int32), dtype="f32", page=pre.kv.page)
    q_all = np.concatenate([pre.q_fa, dec.q_fa], 0)
    r = O.fa_prefill_rows(q_all, kv_full, [200], 8, 12, dec.scale)
    d_ = O.fa_decode(dec.q_fa, dec.kv, 8, 12, dec.scale)
    for a, b in zip(r, d_):
        np.testing.assert_allclose(a, b, atol=1e-13)


# ----------------------------------------------------------------------------- CSA2
def _csa2_small(seed=0, t=(333, 100, 8), pool_blocks=20, k_top=30):
    grp = W.csa2_group(list(t), Hq=4, d=16, Hi=6, di=16, k_top=k_top, blk=8, max_blocks=pool_blocks,
                       n_reuse=1, needles=5, dtype="bf16", seed=seed, page=16)
    return grp


def test_lightning_score_special_cases():
    rng = np.random.default_rng(0)
    K = rng.standard_normal((50, 6))
    q = rng.standard_normal((4, 6))
    wv = rng.uniform(0, 1, 4)
    I = O.lightning_scores(q, wv, K)
    # single head, unit weight: relu of the dot product
    np.testing.assert_allclose(O.lightning_scores(q[:1], np.ones(1), K), np.maximum(K @ q[0], 0), atol=1e-14)
    # linear in w, zero when every dot product is negative, never negative
    np.testing.assert_allclose(O.lightning_scores(q, 3 * wv, K), 3 * I, atol=1e-12)
    Kneg = -np.sign(q[0])[None, :] * np.abs(K)
    qpos = np.abs(q[:1]) * np.sign(q[0])
    assert np.all(O.lightning_scores(qpos, np.ones(1), Kneg) == 0)
    assert np.all(I >= 0)
    # loop form
    for s in (0, 17, 49):
        ref = sum(wv[j] * max(0.0, float(q[j] @ K[s])) for j in range(4))
        assert abs(I[s] - ref) < 1e-12


def test_block_max_bruteforce_and_tail():
    I = np.random.default_rng(2).standard_normal(37)
    bm = O.block_max(I, 37, 8)
    assert len(bm) == 5
    for b in range(5):
        assert bm[b] == max(I[s] for s in range(8 * b, min(37, 8 * b + 8)))


def test_reindex_over_all_blocks_is_flat_indexer():
    grp = _csa2_small(seed=1, pool_blocks=2048)  # pool = every block
    idx, cnt, pool, pcnt = O.indexer_full(grp.q_idx[0], grp.w_idx[0], grp.kidx, grp.k_top, 8, 2048)
    for b, t in enumerate(grp.kidx.seq_len):
        assert pcnt[b] == (int(t) + 7) // 8
    # Reindex with its own query over the full pool == flat top-k of that query
    ridx, rcnt = O.indexer_reindex(grp.q_idx[1], grp.w_idx[1], grp.kidx, grp.k_top, 8, pool, pcnt)
    fidx, fcnt, _, _ = O.indexer_full(grp.q_idx[1], grp.w_idx[1], grp.kidx, grp.k_top, 8, 2048)
    np.testing.assert_array_equal(ridx, fidx)
    np.testing.assert_array_equal(rcnt, fcnt)


def test_reindex_with_full_query_reproduces_full_topk():
    # pool_blocks >= k_top, pool smaller than the 42 blocks of t=333: a block holding a
    # top-k position has a maximum >= the k-th score, and at most k_top blocks do
    grp = _csa2_small(seed=3, pool_blocks=24, k_top=20)
    idx, cnt, pool, pcnt = O.indexer_full(grp.q_idx[0], grp.w_idx[0], grp.kidx, 20, 8, 24)
    assert pcnt[0] == 24
    ridx, rcnt = O.indexer_reindex(grp.q_idx[0], grp.w_idx[0], grp.kidx, 20, 8, pool, pcnt)
    for b, t in enumerate(grp.kidx.seq_len):
        sel = set(idx[b, :cnt[b]].tolist())
        pos = set(O.pool_positions(pool[b, :pcnt[b]], int(t), 8).tolist())
        assert sel <= pos  # a block holding a top-k position has max >= the k-th score
        assert list(ridx[b, :rcnt[b]]) == list(idx[b, :cnt[b]])


def test_csa2_attention_over_whole_pool_is_dense_over_pool():
    grp = _csa2_small(seed=5, pool_blocks=6, k_top=10_000)
    idx, cnt, pool, pcnt = O.indexer_full(grp.q_idx[0], grp.w_idx[0], grp.kidx, 10_000, 8, 6)
    ridx, rcnt = O.indexer_reindex(grp.q_idx[1], grp.w_idx[1], grp.kidx, 10_000, 8, pool, pcnt)
    kv = grp.kv
    o = O.sa_decode(grp.q_main[1], kv, 0, ridx.reshape(len(rcnt), 1, -1), rcnt.reshape(-1, 1), grp.scale)
    Q = O.to_f64(grp.q_main[1], "bf16")
    for b, t in enumerate(kv.seq_len):
        pos = O.pool_positions(pool[b, :pcnt[b]], int(t), 8)
        assert list(ridx[b, :rcnt[b]]) == list(pos)  # k >= pool size: everything in the pool
        K = O.gather_rows(kv.k, kv.block_table[b], 0, pos, kv.page, "bf16")
        V = O.gather_rows(kv.v, kv.block_table[b], 0, pos, kv.page, "bf16")
        p = prob_table(Q[b], K, grp.scale)
        np.testing.assert_allclose(o[b], p @ V, atol=1e-12)


def test_csa2_needles_in_full_topk():
    grp = _csa2_small(seed=6)
    idx, cnt, _, _ = O.indexer_full(grp.q_idx[0], grp.w_idx[0], grp.kidx, grp.k_top, 8, 20)
    for b in range(len(cnt)):
        assert set(grp.needles[b].tolist()) <= set(idx[b, :cnt[b]].tolist())


# ----------------------------------------------------------------------------- counting model
def test_counting_examples_from_pages():
    gold = json.load(open(GOLD))
    g = gold["csa2_group_nc32768"]
    flat, hier = C.selector_comparisons(g["n_c"], g["pool"], g["n_full"], g["n_reindex"], g["n_reuse"])
    assert (flat, hier) == (g["flat"], g["hierarchical"])
    assert hier / flat == g["ratio"]
    g = gold["csa2_group_1m"]
    assert g["n"] // g["m"] == g["n_c"]
    flat, hier = C.selector_comparisons(g["n_c"], g["pool"], g["n_full"], g["n_reindex"], g["n_reuse"])
    assert (flat, hier) == (g["flat"], g["hierarchical"])
    assert round(100 * hier / flat, 2) == g["ratio_percent_2dp"]
    assert (g["n_full"] + g["n_reindex"] + g["n_reuse"]) * g["k_top"] == g["attention_entry_reads"]
    g = gold["dsa_decode_crossover"]
    assert C.dsa_crossover(g["latent_bytes"], g["index_key_bytes"], g["k"]) == g["crossover_L"]
    dense, dsa = C.dsa_decode_bytes(g["crossover_L"] + 1, g["latent_bytes"], g["index_key_bytes"], g["k"])
    assert dsa < dense
    dense, dsa = C.dsa_decode_bytes(g["crossover_L"] - 1, g["latent_bytes"], g["index_key_bytes"], g["k"])
    assert dsa > dense
    g = gold["dsa_prefill_speedup"]
    assert round(g["dense_pflop"] / (g["main_pflop"] + g["indexer_pflop_fp8_equiv"]), 1) == g["speedup_1dp"]


def test_prefill_flops_model():
    f = C.prefill_flops(32768, 32, 128, 128, 1024)
    assert abs(f["fa"] - 8.796e12) / 8.796e12 < 1e-3  # 4*d*Hq*n(n+1)/2
    # SA row cost saturates at w + k keys
    small = C.prefill_flops(10, 1, 1, 2, 3)
    assert small["sa_per_layer"] == 4 * sum(min(2, t) + min(3, max(0, t - 2)) for t in range(1, 11))


def test_decode_bytes_model():
    m = C.decode_group_bytes([100, 2000], Hq=8, Hkv=2, d=16, w=8, k=64, elem=2, n_sa=5)
    assert m["fa"] == (100 + 2000) * 2 * 16 * 2 * 2
    assert m["sa_per_layer"] == 2 * ((8 + 64) + (8 + 64)) * 16 * 2 * 2


# ----------------------------------------------------------------------------- sink bias and gate
def test_sa_sink_limits_and_closed_form():
    """The per-head sink bias ([HS2] §17.1) as a zero-value key: a sink at -inf changes
    nothing, a sink far above every logit takes all the mass, and with identical keys and
    values the output is v / (1 + e^(b - x0) / n) in closed form."""
    rng = np.random.default_rng(11)
    q, K, V = rng.standard_normal((3, 8)), rng.standard_normal((5, 8)), rng.standard_normal((5, 8))
    base = O.sparse_attention(q, K, V, 0.3)
    assert np.allclose(O.sparse_attention(q, K, V, 0.3, sink=np.full(3, -np.inf)), base, atol=1e-15)
    assert np.abs(O.sparse_attention(q, K, V, 0.3, sink=np.full(3, 80.0))).max() < 1e-25
    k0, v0, n = rng.standard_normal(8), rng.standard_normal(8), 7
    b = np.array([-1.0, 0.5, 2.0])
    x0 = (q @ k0) * 0.3
    expect = v0[None, :] / (1.0 + np.exp(b - x0) / n)[:, None]
    got = O.sparse_attention(q, np.tile(k0, (n, 1)), np.tile(v0, (n, 1)), 0.3, sink=b)
    assert np.allclose(got, expect, rtol=1e-12, atol=1e-13)


def test_output_gate_limits():
    """The output sigmoid gate: logit 0 halves the output, large logits pass it or zero it."""
    o = np.random.default_rng(12).standard_normal((2, 4, 8))
    assert np.allclose(O.output_gate(o, np.zeros_like(o)), 0.5 * o)
    assert np.allclose(O.output_gate(o, np.full_like(o, 60.0)), o)
    assert np.abs(O.output_gate(o, np.full_like(o, -80.0))).max() < 1e-30
    assert O.output_gate(o, None) is o


def test_sa_decode_sink_and_gate_reach_their_heads():
    """sa_decode applies sink b_h to query head h (not to its KV head) and the gate element by
    element: a huge sink on one head zeroes that head only; a zero gate halves one query."""
    grp = W.decode_group([40, 70], Hq=4, Hkv=2, d=16, w=4, k=8, dtype="f32", seed=13, n_sa=1, needles=0)
    _, _, idx, cnt = O.fa_decode(grp.q_fa, grp.kv, grp.w, grp.k, grp.scale)
    base = O.sa_decode(grp.q_sa[0], grp.kv, grp.w, idx, cnt, grp.scale)
    sink = np.full(4, -np.inf)
    sink[1] = 90.0
    o = O.sa_decode(grp.q_sa[0], grp.kv, grp.w, idx, cnt, grp.scale, sink=sink)
    assert np.abs(o[:, 1]).max() < 1e-25
    keep = [0, 2, 3]
    assert np.allclose(o[:, keep], base[:, keep], atol=1e-15)
    gate = np.full(base.shape, 60.0, dtype=np.float32)
    gate[1] = 0.0
    og = O.sa_decode(grp.q_sa[0], grp.kv, grp.w, idx, cnt, grp.scale, gate=gate)
    assert np.allclose(og[1], 0.5 * base[1]) and np.allclose(og[0], base[0])


# ----------------------------------------------------------------------------- block-level selection
def test_block_topk_with_unit_blocks_is_token_topk():
    sc = np.random.default_rng(21).random(300)
    for k in (0, 1, 17, 299, 400):
        assert np.array_equal(O.block_topk(sc, k, 1), O.topk_lower_index(sc, k))


def test_block_topk_bruteforce_and_invariants():
    """Against enumeration of every block subset of the budget's size on small inputs: the
    chosen blocks maximise the sorted vector of block maxima (ties to lower block ids);
    the output is whole blocks (a partial last block included), ascending, within F."""
    import itertools

    for seed in range(6):
        rng = np.random.default_rng(30 + seed)
        n, blk = int(rng.integers(20, 60)), int(rng.integers(2, 9))
        sc = rng.random(n)
        if seed % 2:
            sc = np.round(sc * 4) / 4  # many ties
        k = blk * int(rng.integers(1, 5))
        sel = O.block_topk(sc, k, blk)
        nb = (n + blk - 1) // blk
        kb = min(k // blk, nb)
        maxes = [sc[b * blk:min(n, b * blk + blk)].max() for b in range(nb)]
        best = max(itertools.combinations(range(nb), kb), key=lambda c: (sorted((maxes[b] for b in c), reverse=True),
                                                                         [-b for b in c]))
        expect = np.concatenate([np.arange(b * blk, min(n, b * blk + blk)) for b in best]) if kb else np.zeros(0)
        assert np.array_equal(sel, expect), (seed, sel, expect)
        assert np.all(np.diff(sel) > 0) and (len(sel) == 0 or (sel.min() >= 0 and sel.max() < n))


def test_block_decode_selection_respects_window_and_budget():
    grp = W.decode_group([1500, 777], Hq=4, Hkv=1, d=32, w=64, k=256, dtype="f32", seed=22, n_sa=0, needles=4)
    _, _, idx, cnt, _ = O.fa_decode(grp.q_fa, grp.kv, grp.w, grp.k, grp.scale, return_scores=True, blk=64)
    for b, t in enumerate([1500, 777]):
        s = idx[b, 0, :cnt[b, 0]]
        assert cnt[b, 0] <= 256 and (s < t - 64).all()
        assert set(grp.needles[b].tolist()) <= set(s.tolist())  # needles' blocks are chosen
        blocks = np.unique(s // 64)
        assert len(blocks) <= 4
        for bl in blocks:  # whole blocks (clipped to the far range)
            lo, hi = bl * 64, min(t - 64, bl * 64 + 64)
            assert set(range(lo, hi)) <= set(s.tolist())


# ----------------------------------------------------------------------------- FP8 KV
def test_fp8_e4m3_values_from_the_format():
    """E4M3 facts: 0x00 = 0, 0x01 = 2^-9 (smallest subnormal), 0x08 = 2^-6 (smallest normal),
    0x38 = 1, 0x7E = 448 (largest), 0xB8 = -1, 0x7F = NaN (no infinity)."""
    v = O.fp8_e4m3_to_f64(np.array([0x00, 0x01, 0x08, 0x38, 0x7E, 0xB8, 0x7F], dtype=np.uint8))
    assert v[0] == 0.0 and v[1] == 2.0 ** -9 and v[2] == 2.0 ** -6 and v[3] == 1.0 and v[4] == 448.0
    assert v[5] == -1.0 and np.isnan(v[6])
    every = O.fp8_e4m3_to_f64(np.arange(256, dtype=np.uint8))
    finite = every[np.isfinite(every)]
    assert len(finite) == 254 and np.all(np.diff(np.sort(np.unique(np.abs(finite)))) > 0)


def test_fp8_encoder_rounds_to_nearest_even():
    """The input encoder: decode(encode(x)) is a nearest finite E4M3 value (ties to the even
    code), by enumeration of all 254 finite values; every finite code round-trips."""
    table = O.fp8_e4m3_to_f64(np.arange(256, dtype=np.uint8))
    fin = np.isfinite(table)
    x = np.concatenate([np.random.default_rng(40).standard_normal(3000) * 30, table[fin][:126] + 1e-12,
                        (table[1:126] + table[2:127]) / 2])  # includes exact midpoints
    c = W.f32_to_fp8_e4m3(x)
    got = O.fp8_e4m3_to_f64(c)
    err = np.abs(table[fin][None, :] - np.clip(x, -448, 448)[:, None])
    assert np.allclose(np.abs(got - np.clip(x, -448, 448)), err.min(axis=1), atol=0, rtol=0)
    mids = slice(3000 + 126, None)
    assert np.all((c[mids] & 1) == 0)  # ties went to the even code
    codes = np.arange(127, dtype=np.uint8)
    assert np.array_equal(W.f32_to_fp8_e4m3(table[:127]), codes)


def test_oracle_on_fp8_pool_equals_oracle_on_its_dequantised_values():
    """FA + selection + SA on an FP8 pool equal the same on a float32 pool holding code *
    scale, dequantised independently here."""
    grp = W.decode_group_fp8([300, 170], Hq=4, Hkv=2, d=32, w=8, k=16, seed=41, n_sa=1, needles=0)
    kv = grp.kv
    table = O.fp8_e4m3_to_f64(np.arange(256, dtype=np.uint8))
    deq = lambda codes, sc: (table[codes] * sc[:, :, None, None]).astype(np.float32)
    kv32 = W.PagedKV(k=deq(kv.k, kv.k_scale), v=deq(kv.v, kv.v_scale), block_table=kv.block_table,
                     seq_len=kv.seq_len, dtype="f32")
    q32 = O.to_f64(grp.q_fa, "bf16").astype(np.float32)
    qs32 = O.to_f64(grp.q_sa[0], "bf16").astype(np.float32)
    a = O.fa_decode(grp.q_fa, kv, grp.w, grp.k, grp.scale)
    b = O.fa_decode(q32, kv32, grp.w, grp.k, grp.scale)
    assert np.allclose(a[0], b[0], atol=1e-12) and np.array_equal(a[2], b[2])
    sa = O.sa_decode(grp.q_sa[0], kv, grp.w, a[2], a[3], grp.scale)
    sb = O.sa_decode(qs32, kv32, grp.w, a[2], a[3], grp.scale)
    assert np.allclose(sa, sb, atol=1e-12)


def test_fp4_e2m1_values_from_the_format():
    """E2M1 facts (1 sign, 2 exponent bits with bias 1, 1 mantissa bit, no inf/NaN): the eight
    magnitudes are 0, 0.5 (the one subnormal), 1, 1.5, 2, 3, 4, 6; bit 3 is the sign."""
    v = O.fp4_e2m1_to_f64(np.arange(16, dtype=np.uint8))
    assert list(v[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(v[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_fp4_unpack_channel_order():
    """Channel 2i is the low nibble of byte i, channel 2i+1 the high nibble."""
    packed = np.array([[0x21, 0xF7]], dtype=np.uint8)
    np.testing.assert_array_equal(O.fp4_unpack(packed), [[1, 2, 7, 15]])
    np.testing.assert_array_equal(O.fp4_e2m1_to_f64(O.fp4_unpack(packed)), [[0.5, 1.0, 6.0, -6.0]])


def test_fp4_encoder_rounds_to_nearest_even():
    """The input encoder: decode(encode(x)) is a nearest E2M1 value (ties to the even code)
    among all 15 distinct values, saturating at 6; every code round-trips."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    vals = np.concatenate([-mags[:0:-1], mags])
    x = np.concatenate([np.random.default_rng(42).standard_normal(2000) * 3, (mags[:-1] + mags[1:]) / 2,
                        -(mags[:-1] + mags[1:]) / 2])
    c = W.f32_to_fp4_e2m1(x)
    got = O.fp4_e2m1_to_f64(c)
    xc = np.clip(x, -6, 6)
    best = np.abs(vals[None, :] - xc[:, None]).min(axis=1)
    assert np.array_equal(np.abs(got - xc), best)
    assert np.all((c[2000:] & 1) == 0)  # midpoints went to the even code
    assert np.array_equal(W.f32_to_fp4_e2m1(mags), np.arange(8))


def test_oracle_on_fp4_pool_equals_oracle_on_its_dequantised_values():
    """FA + selection + SA on an FP4 pool (E2M1 codes, E4M3 scales per 16 channels, a slab
    scale) equal the same on a float32 pool dequantised here with a table written out."""
    grp = W.decode_group_fp4([300, 170], Hq=4, Hkv=2, d=32, w=8, k=16, seed=41, n_sa=1, needles=0)
    kv = grp.kv
    e2m1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
    e4m3 = O.fp8_e4m3_to_f64(np.arange(256, dtype=np.uint8))  # pinned by its own tests above

    def deq(packed, sf, slab):
        P, Hh, S, half = packed.shape
        out = np.empty((P, Hh, S, 2 * half))
        for c in range(2 * half):
            nib = (packed[..., c // 2] >> (4 * (c % 2))) & 0xF
            out[..., c] = e2m1[nib] * e4m3[sf[..., c // 16]]
        return (out * slab[:, :, None, None]).astype(np.float32)

    kv32 = W.PagedKV(k=deq(kv.k, kv.k_sf, kv.k_scale), v=deq(kv.v, kv.v_sf, kv.v_scale),
                     block_table=kv.block_table, seq_len=kv.seq_len, dtype="f32")
    assert np.all(np.abs(kv32.k) < 1e30)  # dequantised in float32 without overflow
    q32 = O.to_f64(grp.q_fa, "bf16").astype(np.float32)
    qs32 = O.to_f64(grp.q_sa[0], "bf16").astype(np.float32)
    a = O.fa_decode(grp.q_fa, kv, grp.w, grp.k, grp.scale)
    b = O.fa_decode(q32, kv32, grp.w, grp.k, grp.scale)
    assert np.allclose(a[0], b[0], atol=1e-6) and np.array_equal(a[2], b[2])
    sa = O.sa_decode(grp.q_sa[0], kv, grp.w, a[2], a[3], grp.scale)
    sb = O.sa_decode(qs32, kv32, grp.w, a[2], a[3], grp.scale)
    assert np.allclose(sa, sb, atol=1e-6)


# ----------------------------------------------------------------------------- decode KV append
def logical_view(pool, bt_row, npages):
    """[Hkv][npages * page][d] rows of one sequence, by concatenating its pages in table
    order (a route independent of the oracle's position arithmetic)."""
    return np.concatenate([pool[int(p)] for p in bt_row[:npages]], axis=1)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kv_append_writes_exactly_the_current_token_row(dtype):
    # current tokens on the first, the last and a middle slot of a page
    lens = [17, 16, 1, 40]
    grp = W.decode_group(lens, Hq=4, Hkv=2, d=8, w=4, k=6, dtype=dtype, seed=41, n_sa=0, needles=0, page=16)
    kv = grp.kv
    rng = np.random.default_rng(5)
    shape = (len(lens), kv.Hkv, 8)
    k_new = W.store(rng.standard_normal(shape).astype(np.float32), dtype)
    v_new = W.store(rng.standard_normal(shape).astype(np.float32), dtype)
    out = O.kv_append(kv, k_new, v_new)
    owned = set()
    for b, t in enumerate(lens):
        npg = (t + kv.page - 1) // kv.page
        owned.update(int(p) for p in kv.block_table[b][:npg])
        for pool0, pool1, new in ((kv.k, out.k, k_new), (kv.v, out.v, v_new)):
            before = logical_view(pool0, kv.block_table[b], npg)
            after = logical_view(pool1, kv.block_table[b], npg)
            np.testing.assert_array_equal(after[:, t - 1], new[b])
            keep = np.ones(npg * kv.page, dtype=bool)
            keep[t - 1] = False
            np.testing.assert_array_equal(after[:, keep], before[:, keep])
    for p in range(kv.num_pages):  # pages of no sequence are untouched
        if p not in owned:
            np.testing.assert_array_equal(out.k[p], kv.k[p])
            np.testing.assert_array_equal(out.v[p], kv.v[p])


def test_fa_after_append_is_dense_over_sequence_ending_in_new_row():
    lens = [23, 9]
    grp = W.decode_group(lens, Hq=2, Hkv=1, d=8, w=4, k=5, dtype="f32", seed=43, n_sa=0, needles=0, page=8)
    kv = grp.kv
    rng = np.random.default_rng(6)
    k_new = rng.standard_normal((2, 1, 8)).astype(np.float32)
    v_new = rng.standard_normal((2, 1, 8)).astype(np.float32)
    o, lse, _, _ = O.fa_decode(grp.q_fa, O.kv_append(kv, k_new, v_new), 4, 5, grp.scale)
    Q = O.to_f64(grp.q_fa, "f32")
    for b, t in enumerate(lens):
        npg = (t + kv.page - 1) // kv.page
        K = logical_view(kv.k, kv.block_table[b], npg)[0, :t].astype(np.float64)
        V = logical_view(kv.v, kv.block_table[b], npg)[0, :t].astype(np.float64)
        K[t - 1], V[t - 1] = k_new[b, 0], v_new[b, 0]
        for h in range(2):
            x = [float(Q[b, h] @ K[s]) * grp.scale for s in range(t)]
            m = max(x)
            ex = [math.exp(v - m) for v in x]
            z = sum(ex)
            ref = sum((e / z) * V[s] for s, e in enumerate(ex))
            np.testing.assert_allclose(o[b, h], ref, rtol=0, atol=1e-12)
            assert abs(lse[b, h] - (m + math.log(z))) < 1e-12


# ----------------------------------------------------------------------------- SA prefill rows
def sa_rows_bruteforce(Q, K, V, scale, rows, allowed, sink=None, gate=None):
    """SA of query rows ``rows`` written with an explicit mask: ``allowed(i, s)`` says whether
    row i may attend to key position s; one softmax over the allowed keys with Python loops and
    math.exp, a sink logit b adding exp(b) to the denominator, and a gate g multiplying each
    output element by 1 / (1 + exp(-g)). Q [n][d], K, V [n][d]; returns [len(rows)][d]."""
    n, d = K.shape[0], V.shape[1]
    out = np.zeros((len(rows), d))
    for r, i in enumerate(rows):
        logits = [float(Q[i] @ K[s]) * scale for s in range(n) if allowed(i, s)]
        pos = [s for s in range(n) if allowed(i, s)]
        m = max(logits + ([sink] if sink is not None else []))
        ex = [math.exp(x - m) for x in logits]
        z = sum(ex) + (math.exp(sink - m) if sink is not None else 0.0)
        for e, s in zip(ex, pos):
            out[r] += (e / z) * V[s]
        if gate is not None:
            out[r] = [out[r][c] / (1.0 + math.exp(-float(gate[i][c]))) for c in range(d)]
    return out


def _random_far_sets(n, Hkv, w, k, seed):
    """Independent of the FA: row i's set is a random subset of F(i + 1) = [0, i - w] of size
    min(k, |F|), ascending and -1 padded, so every row's set differs from its neighbours'."""
    rng = np.random.default_rng(seed)
    idx = np.full((n, Hkv, k), -1, np.int32)
    cnt = np.zeros((n, Hkv), np.int32)
    for i in range(n):
        nf = max(0, i + 1 - w)
        for g in range(Hkv):
            c = min(k, nf)
            idx[i, g, :c] = np.sort(rng.choice(nf, size=c, replace=False)) if c else []
            cnt[i, g] = c
    return idx, cnt


_SA_ROWS = [44, 3, 20, 0, 5, 4, 31]  # unsorted, not 0..R-1: row i and sample r differ


@pytest.mark.parametrize("sink_gate", [False, True])
def test_sa_prefill_rows_dense_when_k_covers_far_range(sink_gate):
    """k >= |F| for every row => SA prefill row i is dense causal attention of the SA query of
    row i over keys 0..i ([CSA2] §5.1 degeneration check; [HS2] §7.2 window + far set under one
    normaliser), through a permuted block table, with and without sink bias and output gate."""
    n, Hq, Hkv, d, w, k = 45, 4, 2, 8, 5, 60
    grp = W.prefill_group(n, Hq, Hkv, d, w=w, k=k, dtype="f32", seed=31, n_sa=1, page=8, permute=True)
    kv = grp.kv
    idx = np.full((n, Hkv, k), -1, np.int32)
    cnt = np.zeros((n, Hkv), np.int32)
    for i in range(n):
        f = max(0, i + 1 - w)
        idx[i, :, :f] = np.arange(f)
        cnt[i, :] = f
    rng = np.random.default_rng(5)
    sink = rng.standard_normal(Hq) if sink_gate else None
    gate = rng.standard_normal((n, Hq, d)).astype(np.float32) if sink_gate else None
    o = O.sa_prefill_rows(grp.q_sa[0], kv, _SA_ROWS, w, idx, cnt, grp.scale, sink=sink, gate=gate)
    Q = O.to_f64(grp.q_sa[0], "f32")
    G = Hq // Hkv
    for g in range(Hkv):
        K, V = contiguous_rows(kv, 0, g, n)
        for h in range(g * G, (g + 1) * G):
            ref = sa_rows_bruteforce(Q[:, h], K, V, grp.scale, _SA_ROWS, lambda i, s: s <= i,
                                     sink=None if sink is None else float(sink[h]),
                                     gate=None if gate is None else gate[:, h].astype(np.float64))
            np.testing.assert_allclose(o[:, h], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("sink_gate", [False, True])
def test_sa_prefill_rows_partial_sets_bruteforce(sink_gate):
    """Each row attends exactly to its own window W(i + 1) = [i - w + 1, i] and its own far set
    idx[i] (a random subset of [0, i - w]), under one softmax: an explicit per-row mask."""
    n, Hq, Hkv, d, w, k = 40, 4, 2, 8, 4, 3
    grp = W.prefill_group(n, Hq, Hkv, d, w=w, k=k, dtype="f32", seed=32, n_sa=1, page=8, permute=True)
    kv = grp.kv
    idx, cnt = _random_far_sets(n, Hkv, w, k, seed=9)
    rng = np.random.default_rng(6)
    sink = rng.standard_normal(Hq) if sink_gate else None
    gate = rng.standard_normal((n, Hq, d)).astype(np.float32) if sink_gate else None
    rows = [39, 2, 17, 0, 8, 4, 3, 25]
    o = O.sa_prefill_rows(grp.q_sa[0], kv, rows, w, idx, cnt, grp.scale, sink=sink, gate=gate)
    Q = O.to_f64(grp.q_sa[0], "f32")
    G = Hq // Hkv
    for g in range(Hkv):
        K, V = contiguous_rows(kv, 0, g, n)
        sets = [set(idx[i, g, :cnt[i, g]].tolist()) for i in range(n)]
        allowed = (lambda i, s, sets=sets: (i - w < s <= i) or s in sets[i])
        for h in range(g * G, (g + 1) * G):
            ref = sa_rows_bruteforce(Q[:, h], K, V, grp.scale, rows, allowed,
                                     sink=None if sink is None else float(sink[h]),
                                     gate=None if gate is None else gate[:, h].astype(np.float64))
            np.testing.assert_allclose(o[:, h], ref, rtol=0, atol=1e-12)


def test_sa_prefill_last_row_equals_decode():
    """SA prefill row n-1 (t = n) and an SA decode query with seq_len n over the same cache,
    query and indices give the same output (both are [HS2] §7.2 at one query)."""
    n, Hq, Hkv, d, w, k = 70, 4, 2, 8, 6, 9
    grp = W.prefill_group(n, Hq, Hkv, d, w=w, k=k, dtype="bf16", seed=33, n_sa=1, page=16, permute=True)
    kv = grp.kv
    idx, cnt = _random_far_sets(n, Hkv, w, k, seed=10)
    pre = O.sa_prefill_rows(grp.q_sa[0], kv, [n - 1], w, idx, cnt, grp.scale)
    dec = O.sa_decode(grp.q_sa[0][n - 1:n], kv, w, idx[n - 1:n], cnt[n - 1:n], grp.scale)
    np.testing.assert_allclose(pre, dec, rtol=0, atol=1e-13)


def test_bf16_widening_known_bit_patterns():
    """bfloat16 is the top half of an IEEE binary32 word: 1 sign, 8 exponent bits (bias 127),
    7 mantissa bits; values written out from the format, not from a conversion routine."""
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x8000, 0x7F7F, 0x3F81, 0x0080, 0x4049], np.uint16)
    want = [1.0, -2.0, 2.0 ** -133, 0.0, (2.0 - 2.0 ** -7) * 2.0 ** 127, 1.0 + 2.0 ** -7, 2.0 ** -126,
            3.140625]
    got = O.to_f64(bits, "bf16")
    assert got.dtype == np.float64
    assert list(got) == want
    assert math.copysign(1.0, got[3]) == -1.0  # 0x8000 is negative zero
