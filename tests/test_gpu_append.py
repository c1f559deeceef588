"""GPU parity of the decode KV append against the oracle's ``kv_append``, through the C ABI:
several caches in one call (bf16 and f32, a key-only cache), and the append fused into the
decode FA call (the bf16 tensor-core scan writes the row itself; other paths append first).
Pools are compared bit for bit; FA / SA outputs and index sets as in the decode tests.
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


def to_host(t, dtype):
    import torch

    x = t.detach().cpu()
    return x.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else x.numpy()


def rows(rng, B, Hkv, d, dtype):
    return W.store(rng.standard_normal((B, Hkv, d)).astype(np.float32), dtype)


def poison_current(kv, value=1000.0):
    """A copy of the cache whose current-token rows hold `value` (the append must replace them)."""
    import copy

    out = copy.copy(kv)
    out.k, out.v = np.array(kv.k, copy=True), np.array(kv.v, copy=True)
    bad = W.store(np.full(kv.k.shape[-1], value, dtype=np.float32), kv.dtype)
    for b, t in enumerate(kv.seq_len):
        pg = kv.block_table[b][(int(t) - 1) // kv.page]
        out.k[pg, :, (int(t) - 1) % kv.page, :] = bad
        out.v[pg, :, (int(t) - 1) % kv.page, :] = bad
    return out


def test_kv_append_several_caches_one_call(H):
    import torch

    rng = np.random.default_rng(71)
    # current tokens on slots 16, 63, 0, 0, 43 / 0, 7, 1 / 32, 6
    ga = W.decode_group([17, 64, 1, 129, 300], 8, 4, 128, 4, 8, "bf16", seed=72, n_sa=0, needles=0)
    gb = W.decode_group([65, 5000, 2], 4, 2, 64, 4, 8, "bf16", seed=73, n_sa=0, needles=0)
    gc = W.decode_group([33, 7], 2, 1, 64, 4, 8, "f32", seed=74, n_sa=0, needles=0)
    gd = W.decode_group([130, 64], 2, 1, 128, 4, 8, "bf16", seed=75, n_sa=0, needles=0)
    kd = W.PagedKV(k=gd.kv.k, v=None, block_table=gd.kv.block_table, seq_len=gd.kv.seq_len, dtype="bf16",
                   page=gd.kv.page)  # key-only cache (an indexer-key cache has no V)
    kvs = [ga.kv, gb.kv, gc.kv, kd]
    k_new = [rows(rng, len(kv.seq_len), kv.Hkv, kv.k.shape[-1], kv.dtype) for kv in kvs]
    v_new = [rows(rng, len(kv.seq_len), kv.Hkv, kv.k.shape[-1], kv.dtype) for kv in kvs[:3]] + [None]
    dev = [kv_to_device(kv) for kv in kvs]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    H.hs2_kv_append(dev, [to_torch(x, kv.dtype) for x, kv in zip(k_new, kvs)],
                    [None if x is None else to_torch(x, kv.dtype) for x, kv in zip(v_new, kvs)], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for kv, d, kn, vn in zip(kvs, dev, k_new, v_new):
        ref = O.kv_append(kv, kn, vn)
        np.testing.assert_array_equal(to_host(d.k, kv.dtype), ref.k)
        if kv.v is not None:
            np.testing.assert_array_equal(to_host(d.v, kv.dtype), ref.v)


def test_kv_append_bad_entries_flagged_not_written(H):
    import torch

    rng = np.random.default_rng(81)
    g = W.decode_group([100, 70, 20], 4, 2, 64, 4, 8, "bf16", seed=82, n_sa=0, needles=0)
    kv = g.kv
    bt, sl = kv.block_table.copy(), kv.seq_len.copy()
    bt[1][(int(sl[1]) - 1) // kv.page] = -1  # sequence 1: its current page is unmapped
    sl[2] = kv.block_table.shape[1] * kv.page + 1  # sequence 2: longer than its table
    bad = W.PagedKV(k=kv.k, v=kv.v, block_table=bt, seq_len=sl, dtype=kv.dtype, page=kv.page)
    kn, vn = rows(rng, 3, 2, 64, "bf16"), rows(rng, 3, 2, 64, "bf16")
    d = kv_to_device(bad)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    H.hs2_kv_append([d], [to_torch(kn, "bf16")], [to_torch(vn, "bf16")], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == H.DEV_BAD_PAGE | H.DEV_BAD_LENGTH
    only0 = W.PagedKV(k=kv.k, v=kv.v, block_table=kv.block_table[:1], seq_len=kv.seq_len[:1], dtype=kv.dtype,
                      page=kv.page)
    ref = O.kv_append(only0, kn[:1], vn[:1])  # sequence 0 alone is written
    np.testing.assert_array_equal(to_host(d.k, "bf16"), ref.k)
    np.testing.assert_array_equal(to_host(d.v, "bf16"), ref.v)


@pytest.mark.parametrize("dtype,Hq,Hkv,d", [("bf16", 32, 4, 128), ("bf16", 16, 2, 64), ("bf16", 32, 1, 128),
                                            ("f32", 8, 2, 64)])
def test_fa_select_with_fused_append(H, dtype, Hq, Hkv, d):
    """The current token's K/V come with the FA call. bf16 takes the tensor-core scan, which
    writes the rows itself (8 and 32 query heads per KV head); f32 appends first. The pool's
    current rows are poisoned beforehand."""
    import torch

    lens = [3000, 64, 129, 1000, 17]
    grp = W.decode_group(lens, Hq, Hkv, d, 64, 256, dtype, seed=91, n_sa=1, needles=4)
    rng = np.random.default_rng(92)
    kn, vn = rows(rng, len(lens), Hkv, d, dtype), rows(rng, len(lens), Hkv, d, dtype)
    kvp = poison_current(grp.kv)
    dkv = kv_to_device(kvp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse, idx, cnt = H.hs2_fa_select(to_torch(grp.q_fa, dtype), dkv, grp.w, grp.k, grp.scale, max_t=max(lens),
                                       dev_err=err, k_new=to_torch(kn, dtype), v_new=to_torch(vn, dtype))
    sa = H.hs2_sa_reuse(to_torch(grp.q_sa[0], dtype), dkv, grp.w, idx, cnt, grp.k, grp.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.kv_append(kvp, kn, vn)
    np.testing.assert_array_equal(to_host(dkv.k, dtype), ref.k)
    np.testing.assert_array_equal(to_host(dkv.v, dtype), ref.v)
    o_r, lse_r, idx_r, cnt_r, scores = O.fa_decode(grp.q_fa, ref, grp.w, grp.k, grp.scale, return_scores=True)
    t_ = tol(dtype)
    assert max_abs(o.cpu().numpy(), o_r) <= t_
    assert max_abs(lse.cpu().numpy(), lse_r) <= t_
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    check_index_sets(gi, gc, idx_r, cnt_r, scores, "append ")
    sa_r = O.sa_decode(grp.q_sa[0], ref, grp.w, gi, gc, grp.scale)
    assert max_abs(sa.cpu().numpy(), sa_r) <= t_


def test_append_refuses_fp8_pool(H):
    import torch

    grp = W.decode_group_fp8([300, 100], 8, 1, 128, 16, 32, seed=95, n_sa=0, needles=0)
    dkv = kv_to_device(grp.kv)
    kn = torch.zeros((2, 1, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(H.HS2Error):
        H.hs2_kv_append([dkv], [kn], [kn])
    with pytest.raises(H.HS2Error):
        H.hs2_fa_select(to_torch(grp.q_fa, "bf16"), dkv, 16, 32, grp.scale, k_new=kn, v_new=kn)
    torch.cuda.synchronize()
