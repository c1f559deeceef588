"""GPU parity of the CSA2 hierarchical indexer (Full / Reindex) and its MQA sparse attention.

Through the C ABI; the oracle gets the same seeded arrays. Index sets follow the same rule
as the FA selection: equal counts, differences only within 1e-3 relative of the k-th score.
"""
import numpy as np
import pytest

from oracle import hs2_oracle as O
from top_hs2_fa_gb300 import workloads as W

from hs2_testutil import check_index_sets, kv_to_device, max_abs, to_torch, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def H():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_hs2_fa_gb300 import build
    build.build()
    from top_hs2_fa_gb300 import hs2
    hs2.load()
    return hs2


def run_group(H, grp, max_blocks, k_top):
    import torch

    kidx = kv_to_device(grp.kidx)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q0, q1 = (to_torch(q, "bf16") for q in grp.q_idx)
    w0, w1 = (to_torch(w, "f32") for w in grp.w_idx)
    max_t = int(grp.kidx.seq_len.max())
    idx_f, cnt_f, pool, pcnt = H.hs2_hier_reindex(H.FULL, q0, w0, kidx, k_top, 8, max_blocks, max_t=max_t,
                                                  dev_err=err)
    idx_r, cnt_r, _, _ = H.hs2_hier_reindex(H.REINDEX, q1, w1, kidx, k_top, 8, max_blocks, pool_blocks=pool,
                                            pool_cnt=pcnt, max_t=max_t, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    return [x.cpu().numpy() for x in (idx_f, cnt_f, pool, pcnt, idx_r, cnt_r)]


def check_indexer(H, grp, max_blocks, k_top, batches=None):
    idx_f, cnt_f, pool, pcnt, idx_r, cnt_r = run_group(H, grp, max_blocks, k_top)
    kx = grp.kidx
    sel = list(range(kx.B)) if batches is None else list(batches)
    sub = W.PagedKV(k=kx.k, v=None, block_table=kx.block_table[sel], seq_len=kx.seq_len[sel], dtype=kx.dtype,
                    page=kx.page)
    o_idx, o_cnt, o_pool, o_pcnt, sc = O.indexer_full(grp.q_idx[0][sel], grp.w_idx[0][sel], sub, k_top, 8,
                                                      max_blocks, return_scores=True)
    check_index_sets(idx_f[sel], cnt_f[sel], o_idx, o_cnt, {(i,): sc[i][0] for i in range(len(sel))}, "full ")
    check_index_sets(pool[sel], pcnt[sel], o_pool, o_pcnt, {(i,): sc[i][1] for i in range(len(sel))}, "pool ")
    # Reindex on the GPU's own pool, against the oracle's Reindex on that pool
    r_idx, r_cnt, rsc = O.indexer_reindex(grp.q_idx[1][sel], grp.w_idx[1][sel], sub, k_top, 8, pool[sel],
                                          pcnt[sel], return_scores=True)
    # express the band rule in candidate space (scores indexed by pool candidate order)
    for i in range(len(sel)):
        pos, I = rsc[i]
        rank = {int(p): j for j, p in enumerate(pos)}
        g_c = np.array([rank[int(p)] for p in idx_r[sel[i]][:cnt_r[sel[i]]]], dtype=np.int64)
        o_c = np.array([rank[int(p)] for p in r_idx[i][:r_cnt[i]]], dtype=np.int64)
        gpad = np.full(k_top, -1, np.int64)
        gpad[:len(g_c)] = np.sort(g_c)
        opad = np.full(k_top, -1, np.int64)
        opad[:len(o_c)] = np.sort(o_c)
        check_index_sets(gpad[None], np.array([cnt_r[sel[i]]]), opad[None], np.array([r_cnt[i]]), {(0,): I},
                         "reindex ")
        assert np.all(np.diff(idx_r[sel[i]][:cnt_r[sel[i]]]) > 0)
    return idx_f, cnt_f, pool, pcnt, idx_r, cnt_r


def test_indexer_small_ragged(H):
    grp = W.csa2_group([333, 1000, 5000, 8, 129], Hq=8, d=128, Hi=64, di=128, k_top=64, blk=8, max_blocks=100,
                       n_reuse=1, needles=6, seed=11)
    idx_f, cnt_f, pool, pcnt, _, _ = check_indexer(H, grp, 100, 64)
    for b in range(5):
        assert set(grp.needles[b].tolist()) <= set(idx_f[b, :cnt_f[b]].tolist())


def test_indexer_pool_covers_everything(H):
    # pool = every block: Reindex with the Full layer's own query equals the flat top-k
    grp = W.csa2_group([700, 2000], Hq=8, d=128, Hi=64, di=128, k_top=50, blk=8, max_blocks=4096, n_reuse=1,
                       needles=3, seed=12)
    grp.q_idx[1] = grp.q_idx[0]
    grp.w_idx[1] = grp.w_idx[0]
    idx_f, cnt_f, pool, pcnt, idx_r, cnt_r = check_indexer(H, grp, 4096, 50)
    assert np.array_equal(pcnt, (grp.kidx.seq_len + 7) // 8)
    assert np.array_equal(idx_f, idx_r) and np.array_equal(cnt_f, cnt_r)


def test_csa2_attention_full_reindex_reuse(H):
    """Full -> SA, Reindex -> SA, Reuse -> SA with the Reindex indices (w = 0, MQA)."""
    import torch

    grp = W.csa2_group([3000, 4500], Hq=32, d=128, Hi=64, di=128, k_top=128, blk=8, max_blocks=64, n_reuse=2,
                       needles=8, seed=13)
    idx_f, cnt_f, pool, pcnt, idx_r, cnt_r = run_group(H, grp, 64, 128)
    dkv = kv_to_device(grp.kv)
    outs = []
    for layer, (ii, cc) in enumerate([(idx_f, cnt_f), (idx_r, cnt_r), (idx_r, cnt_r), (idx_r, cnt_r)]):
        q = to_torch(grp.q_main[layer], "bf16")
        o = H.hs2_sa_reuse(q, dkv, 0, to_torch(ii[:, None, :], "i32"), to_torch(cc[:, None], "i32"), 128,
                           grp.scale)
        outs.append(o.cpu().numpy())
        ref = O.sa_decode(grp.q_main[layer], grp.kv, 0, ii[:, None, :], cc[:, None], grp.scale)
        assert max_abs(outs[-1], ref) <= tol("bf16")


def test_indexer_rejects_unsupported(H):
    import torch

    grp = W.csa2_group([100], Hq=8, d=128, Hi=64, di=128, k_top=8, blk=8, max_blocks=4, n_reuse=1, needles=0,
                       seed=14)
    kidx = kv_to_device(grp.kidx)
    q = to_torch(grp.q_idx[0], "bf16")
    with pytest.raises(H.HS2Error):
        H.hs2_hier_reindex(H.FULL, q[:, :32].contiguous(), to_torch(grp.w_idx[0][:, :32].copy(), "f32"), kidx, 8, 8, 4)
    with pytest.raises(H.HS2Error):
        H.hs2_hier_reindex(H.FULL, q, to_torch(grp.w_idx[0], "f32"), kidx, 8, 16, 4)


@pytest.mark.parametrize("distinct", [7, 300])
def test_indexer_cluster_selection_with_ties(H, distinct):
    """Few long rows (the multi-CTA cluster selection) whose indexer keys repeat `distinct`
    rows, so scores tie exactly: the GPU's top-k (positions) and block pool must equal the
    oracle's element by element (ties to the lower position / block). 7 distinct rows put
    thousands of candidates on the k-th key's digit (the single-CTA fallback passes); 300
    keep them within the candidate buffer (the cluster path)."""
    grp = W.csa2_group([40000, 29000], Hq=8, d=128, Hi=64, di=128, k_top=256, blk=8, max_blocks=512,
                       n_reuse=1, needles=0, seed=13)
    kx = grp.kidx
    rng = np.random.default_rng(14)
    P, _, S, d = kx.k.shape
    src = kx.k.reshape(P * S, d)
    pick = rng.integers(0, distinct, size=P * S)
    kx.k = np.ascontiguousarray(src[:distinct][pick].reshape(P, 1, S, d))
    idx_f, cnt_f, pool, pcnt, _, _ = run_group(H, grp, 512, 256)
    o_idx, o_cnt, o_pool, o_pcnt = O.indexer_full(grp.q_idx[0], grp.w_idx[0], kx, 256, 8, 512)
    np.testing.assert_array_equal(cnt_f, o_cnt)
    np.testing.assert_array_equal(idx_f, o_idx)
    np.testing.assert_array_equal(pcnt, o_pcnt)
    np.testing.assert_array_equal(pool, o_pool)


@pytest.mark.slow
def test_csa2_full_size_sampled(H):
    """CSA2 decode at full size (B=8, t=131072, 64 indexer heads, top-512, 2048-block pool):
    two sampled rows against the oracle, invariants on all rows; then the five attention
    layers (Full -> SA with its own top-512, Reindex -> SA, three Reuse -> SA with the
    Reindex indices; w = 0, MQA) on the sampled rows against the oracle."""
    import torch

    grp = W.csa2_group([131072] * 8, Hq=32, d=128, Hi=64, di=128, k_top=512, blk=8, max_blocks=2048,
                       n_reuse=3, needles=32, seed=0)
    sample = [0, 5]
    idx_f, cnt_f, pool, pcnt, idx_r, cnt_r = check_indexer(H, grp, 2048, 512, batches=sample)
    assert (cnt_f == 512).all() and (pcnt == 2048).all() and (cnt_r == 512).all()
    for b in range(8):
        assert set(grp.needles[b].tolist()) <= set(idx_f[b].tolist())
        pos = set(O.pool_positions(pool[b], 131072, 8).tolist())
        assert set(idx_f[b].tolist()) <= pos and set(idx_r[b].tolist()) <= pos
    kv = grp.kv
    dkv = kv_to_device(kv)
    sub = W.PagedKV(k=kv.k, v=kv.v, block_table=kv.block_table[sample], seq_len=kv.seq_len[sample], dtype=kv.dtype,
                    page=kv.page)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    layers = [(idx_f, cnt_f), (idx_r, cnt_r)] + [(idx_r, cnt_r)] * 3
    assert len(grp.q_main) == len(layers)
    for layer, (ii, cc) in enumerate(layers):
        o = H.hs2_sa_reuse(to_torch(grp.q_main[layer], "bf16"), dkv, 0, to_torch(ii[:, None, :], "i32"),
                           to_torch(cc[:, None], "i32"), 512, grp.scale, dev_err=err).cpu().numpy()
        ref = O.sa_decode(grp.q_main[layer][sample], sub, 0, ii[sample][:, None, :], cc[sample][:, None], grp.scale)
        assert max_abs(o[sample], ref) <= tol("bf16"), (layer, max_abs(o[sample], ref))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
