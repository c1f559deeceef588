"""GPU parity of the decode path (FA + selection, SA reuse) against the CPU oracle.

Every call goes through the C ABI (ctypes binding). Oracle inputs are the same
seeded arrays the GPU receives; no expected value comes from the GPU.
"""
import dataclasses

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


def qdt(kv):
    """Storage dtype of the queries: bf16 for an FP8 cache, else the cache's dtype."""
    return "bf16" if kv.dtype in ("fp8", "fp4") else kv.dtype


def run_decode_group(H, grp, sa_layers=None):
    import torch

    kv = grp.kv
    dkv = kv_to_device(kv)
    q = to_torch(grp.q_fa, qdt(kv))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse, idx, cnt = H.hs2_fa_select(q, dkv, grp.w, grp.k, grp.scale, max_t=int(kv.seq_len.max()), dev_err=err)
    sa = []
    outs = []
    Hq = grp.q_fa.shape[1]
    ws = torch.empty(H.hs2_sa_reuse_workspace(kv.B, Hq, dkv, grp.w, grp.k), dtype=torch.uint8, device="cuda")
    for j in range(len(grp.q_sa) if sa_layers is None else sa_layers):
        qs = to_torch(grp.q_sa[j], qdt(kv))
        # layers after the first run back to back on one workspace with HS2_SA_OVERLAP, as a
        # group step does
        outs.append(H.hs2_sa_reuse(qs, dkv, grp.w, idx, cnt, grp.k, grp.scale, workspace=ws, dev_err=err,
                                   overlap=j > 0))
    sa = [x.cpu().numpy() for x in outs]
    torch.cuda.synchronize()
    return o.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy(), sa, int(err.item())


def check_group(H, grp, batches=None, sa_layers=None):
    kv = grp.kv
    o, lse, idx, cnt, sa, err = run_decode_group(H, grp, sa_layers)
    assert err == 0, f"device error flags {err}"
    sel = list(range(kv.B)) if batches is None else list(batches)
    sub = dataclasses.replace(kv, block_table=kv.block_table[sel], seq_len=kv.seq_len[sel])
    o_r, lse_r, idx_r, cnt_r, scores = O.fa_decode(grp.q_fa[sel], sub, grp.w, grp.k, grp.scale,
                                                   return_scores=True)
    t_ = tol(qdt(kv))
    assert max_abs(o[sel], o_r) <= t_, f"FA output error {max_abs(o[sel], o_r)}"
    assert max_abs(lse[sel], lse_r) <= t_, f"lse error {max_abs(lse[sel], lse_r)}"
    check_index_sets(idx[sel], cnt[sel], idx_r, cnt_r, scores, "decode ")
    for j, osa in enumerate(sa):
        # SA parity with the GPU's own index sets (near-tie swaps are not output errors) ...
        ref = O.sa_decode(grp.q_sa[j][sel], sub, grp.w, idx[sel], cnt[sel], grp.scale)
        assert max_abs(osa[sel], ref) <= t_, f"SA{j} error {max_abs(osa[sel], ref)}"
    if sa:
        # ... and with the oracle's index sets fed to both
        import torch
        dkv = kv_to_device(sub)
        o2 = H.hs2_sa_reuse(to_torch(grp.q_sa[0][sel], qdt(kv)), dkv, grp.w, to_torch(idx_r, "i32"),
                            to_torch(cnt_r, "i32"), grp.k, grp.scale).cpu().numpy()
        ref2 = O.sa_decode(grp.q_sa[0][sel], sub, grp.w, idx_r, cnt_r, grp.scale)
        assert max_abs(o2, ref2) <= t_
    return o, idx, cnt


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_ragged_small(H, dtype):
    # lengths around page and window boundaries, a multi-split sequence, G=4 (padded MMA columns)
    lens = [1, 15, 16, 17, 63, 64, 65, 100, 129, 1000, 3001, 4097]
    grp = W.decode_group(lens, Hq=8, Hkv=2, d=128, w=16, k=64, dtype=dtype, seed=1, n_sa=2, needles=4)
    check_group(H, grp)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_gqa8(H, d):
    grp = W.decode_group([2000, 5000, 777, 4096], Hq=32, Hkv=4, d=d, w=128, k=256, dtype="bf16", seed=2,
                         n_sa=1, needles=16)
    check_group(H, grp)


@pytest.mark.parametrize("Hq,Hkv", [(16, 1), (32, 1), (4, 4), (8, 4)])
def test_decode_other_head_ratios(H, Hq, Hkv):
    grp = W.decode_group([300, 1500], Hq=Hq, Hkv=Hkv, d=128, w=32, k=100, dtype="bf16", seed=3, n_sa=1,
                         needles=8)
    check_group(H, grp)


def test_decode_sharp_logits(H):
    # Q, K ~ N(0,1) without the 1/sqrt(d) damping: concentrated attention makes the set check bite
    grp = W.decode_group([2500, 3300], Hq=8, Hkv=1, d=128, w=16, k=64, dtype="f32", seed=4, n_sa=1, needles=0)
    o, idx, cnt = check_group(H, grp)
    assert (cnt == 64).all()


def test_decode_degenerate(H):
    # k = 0; w = 0; w >= t; k >= far range
    for w, k, lens in [(16, 0, [50, 200]), (0, 10, [50, 200]), (500, 10, [50, 200]), (8, 1000, [50, 200])]:
        grp = W.decode_group(lens, Hq=4, Hkv=1, d=64, w=w, k=k, dtype="bf16", seed=5, n_sa=1, needles=0)
        check_group(H, grp)


@pytest.mark.parametrize("lens", [[3000, 2100], [9000, 6000]])
def test_decode_all_far_scores_tied(H, lens):
    # identical keys: every far score is equal, so each (query, KV head) takes its first k
    # positions; 3000 tied keys fit the one-pass select's candidate list, 9000 overflow it and
    # take the radix passes over all keys
    grp = W.decode_group(lens, Hq=8, Hkv=2, d=128, w=32, k=100, dtype="bf16", seed=8, n_sa=1, needles=0)
    grp.kv.k[:] = grp.kv.k[0:1, :, 0:1, :]
    o, idx, cnt = check_group(H, grp)
    for b in range(len(lens)):
        for g in range(2):
            assert cnt[b, g] == 100 and (idx[b, g] == np.arange(100)).all()


def test_tiny_fp32_decode(H):
    tg = W.tiny_group(seed=0)
    o, idx, cnt = check_group(H, tg.decode)
    assert set(tg.decode.needles[0].tolist()) <= set(idx[0, 0, :cnt[0, 0]].tolist())


def test_bad_block_table_entry_is_flagged(H):
    import torch

    grp = W.decode_group([300, 300], Hq=8, Hkv=1, d=128, w=16, k=32, dtype="bf16", seed=6, n_sa=0, needles=0)
    kv = grp.kv
    bt = kv.block_table.copy()
    bt[1, 2] = kv.num_pages + 5  # out of range: the kernels must skip and flag it
    dkv = kv_to_device(W.PagedKV(k=kv.k, v=kv.v, block_table=bt, seq_len=kv.seq_len, dtype=kv.dtype))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    H.hs2_fa_select(to_torch(grp.q_fa, "bf16"), dkv, 16, 32, grp.scale, max_t=300, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & H.DEV_BAD_PAGE


@pytest.mark.slow
def test_decode_bf16_full_size_sampled(H):
    """Decode workload at full size (B=64, t ~ U[16K, 32K], Hq=32, Hkv=4, d=128, w=128, k=1024,
    five SA layers): every sequence checked for set invariants, 6 sampled sequences against the
    oracle element by element."""
    grp = W.decode_bf16_workload(seed=0)
    rng = np.random.default_rng(123)
    sample = sorted(rng.choice(64, size=6, replace=False).tolist())
    o, idx, cnt = check_group(H, grp, batches=sample)
    t = grp.kv.seq_len
    assert np.array_equal(cnt, np.repeat(np.minimum(1024, t - 128)[:, None], 4, 1))
    for b in range(64):
        for g in range(4):
            s = idx[b, g, :cnt[b, g]]
            assert s.min() >= 0 and s.max() < t[b] - 128 and np.all(np.diff(s) > 0)
            assert set(grp.needles[b].tolist()) <= set(s.tolist())


def fused_lengths(B, seed):
    """B ragged lengths around the window and budget edges (w = 16, k = 64) and a few long
    ones, so every branch of the fused selection runs: t < w, t - w <= k, t - w = k + 1, and
    thousands of far keys."""
    edge = [1, 15, 16, 17, 63, 64, 80, 81, 100, 129, 1000, 3001, 4097, 7000]
    rng = np.random.default_rng(seed)
    return [edge[i] if i < len(edge) else int(rng.integers(200, 6000)) for i in range(B)]


def test_decode_fused_selection_ragged(H):
    """The fused merge + score + top-k kernel (taken when a call has at least 152 (query, KV
    head) pairs: here 40 sequences x 4 KV heads) on ragged lengths at the window and budget
    edges, every sequence against the oracle."""
    lens = fused_lengths(40, 52)
    grp = W.decode_group(lens, Hq=32, Hkv=4, d=128, w=16, k=64, dtype="bf16", seed=53, n_sa=1, needles=4)
    check_group(H, grp)


@pytest.mark.parametrize("n_tied", [3000, 9000])
def test_decode_fused_selection_ties(H, n_tied):
    """The fused kernel on rows whose far scores are all equal (identical keys): each takes its
    first k positions; 3000 tied keys fit the candidate list, 9000 overflow it and take the
    radix passes over all keys. 38 sequences x 4 KV heads = 152 pairs."""
    lens = [n_tied] * 38
    grp = W.decode_group(lens, Hq=16, Hkv=4, d=128, w=32, k=100, dtype="bf16", seed=54, n_sa=1, needles=0)
    grp.kv.k[:] = grp.kv.k[0:1, :, 0:1, :]
    o, idx, cnt = check_group(H, grp, batches=[0, 17, 37])
    assert (cnt == 100).all() and (idx == np.arange(100)).all()


@pytest.mark.parametrize("lens,Hkv", [([60000, 33000, 20000], 2), ([17000, 12000], 1)])
def test_decode_cluster_selection_long_rows(H, lens, Hkv):
    """Few long rows: the window-excluding top-k of each (query, KV head) is shared by a
    thread-block cluster (one CTA per 8192 keys of the longest row: 8 CTAs for the first
    case, 3 for the second), each CTA filtering its slice and rank 0 refining the candidates
    from the others' shared memory. Unit-variance keys and queries: no ties, so the cluster
    filter completes without the all-keys fallback. Every sequence against the oracle."""
    grp = W.decode_group(lens, Hq=8, Hkv=Hkv, d=128, w=128, k=1024, dtype="bf16", seed=51, n_sa=1, needles=16)
    o, idx, cnt = check_group(H, grp)
    for b, t in enumerate(lens):
        assert (cnt[b] == 1024).all()
        for g in range(Hkv):
            assert set(grp.needles[b].tolist()) <= set(idx[b, g, :1024].tolist())


def long_decode_cache(gi: int, seed: int = 0):
    """Cache ``gi`` of the long-context decode workload, drawn exactly as the benchmark draws
    it: B=16, t=131072, Hq=32, Hkv=4, d=128, w=128, k=1024, 64 needles, five SA layers."""
    s_len, s_grp = np.random.SeedSequence([seed, gi]).spawn(2)
    lens = W.uniform_lengths(16, 131072, 131072, s_len)
    return W.decode_group(lens, 32, 4, 128, 128, 1024, "bf16", s_grp, n_sa=5, needles=64, qproj=False)


@pytest.mark.slow
@pytest.mark.parametrize("gi", range(4))
def test_long_decode_full_size_sampled(H, gi):
    """Long-context decode at full size, one of the four independent Cross-group caches per
    case (each runs the same calls and launch shapes as in the timed step, including the
    4-CTA cluster selection over 130,944 far keys per row): two sampled sequences against the
    oracle element by element (FA output, lse, index sets, all five SA layers), and on every
    sequence the set invariants and the needles."""
    grp = long_decode_cache(gi)
    sample = sorted(np.random.default_rng(100 + gi).choice(16, size=2, replace=False).tolist())
    o, idx, cnt = check_group(H, grp, batches=sample)
    t = grp.kv.seq_len
    assert (cnt == 1024).all()
    for b in range(16):
        for g in range(4):
            s = idx[b, g]
            assert s.min() >= 0 and s.max() < t[b] - 128 and np.all(np.diff(s) > 0)
            assert set(grp.needles[b].tolist()) <= set(s.tolist())


@pytest.mark.parametrize("dtype,Hq,Hkv", [("bf16", 32, 4), ("bf16", 32, 1), ("f32", 8, 2)])
def test_sa_sink_bias_and_output_gate(H, dtype, Hq, Hkv):
    """hs2_sa_reuse_ex: per-head sink logits (one -inf, one dominant) and elementwise gate
    logits against the oracle, on the decode stream (bf16, 8 and 32 heads per KV head) and
    the fp32 path."""
    import torch

    lens = [900, 2500, 130, 4000]
    grp = W.decode_group(lens, Hq=Hq, Hkv=Hkv, d=128, w=32, k=100, dtype=dtype, seed=17, n_sa=1, needles=4)
    kv = grp.kv
    dkv = kv_to_device(kv)
    _, _, idx, cnt = H.hs2_fa_select(to_torch(grp.q_fa, dtype), dkv, grp.w, grp.k, grp.scale,
                                     max_t=int(kv.seq_len.max()))
    rng = np.random.default_rng(3)
    sink = rng.normal(0.0, 2.0, Hq).astype(np.float32)
    sink[0], sink[1] = -np.inf, 30.0
    gate = rng.normal(0.0, 2.0, (len(lens), Hq, 128)).astype(np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    osa = H.hs2_sa_reuse(to_torch(grp.q_sa[0], dtype), dkv, grp.w, idx, cnt, grp.k, grp.scale, dev_err=err,
                         sink=torch.from_numpy(sink).cuda(), gate=torch.from_numpy(gate).cuda()).cpu().numpy()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.sa_decode(grp.q_sa[0], kv, grp.w, idx.cpu().numpy(), cnt.cpu().numpy(), grp.scale, sink=sink, gate=gate)
    assert max_abs(osa, ref) <= tol(dtype), max_abs(osa, ref)
    assert np.abs(osa[:, 1]).max() < 1e-6  # the dominant sink takes the head's mass


@pytest.mark.parametrize("dtype,lens,k,blk", [("bf16", [3000, 1500, 700, 5000], 256, 64),
                                              ("f32", [900, 2222], 128, 32),
                                              ("bf16", [520, 610], 1024, 64)])
def test_block_level_selection(H, dtype, lens, k, blk):
    """hs2_fa_select_ex with sel_block > 1 against the oracle's block-level selection: whole
    blocks by block maximum (ties to lower blocks), including a partial last far block and a
    budget that covers every block; SA over the chosen positions."""
    import torch

    grp = W.decode_group(lens, Hq=8, Hkv=2, d=128, w=32, k=k, dtype=dtype, seed=19, n_sa=1, needles=4)
    kv = grp.kv
    dkv = kv_to_device(kv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse, idx, cnt = H.hs2_fa_select(to_torch(grp.q_fa, dtype), dkv, grp.w, k, grp.scale,
                                       max_t=int(kv.seq_len.max()), dev_err=err, sel_block=blk)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_r, _, idx_r, cnt_r, sc = O.fa_decode(grp.q_fa, kv, grp.w, k, grp.scale, return_scores=True, blk=blk)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    assert max_abs(o.cpu().numpy(), o_r) <= tol(dtype)
    for b in range(len(lens)):
        for g in range(2):
            got, ref = idx[b, g, :cnt[b, g]], idx_r[b, g, :cnt_r[b, g]]
            if not np.array_equal(got, ref):
                # near ties between block maxima may swap whole blocks: compare block maxima
                s = sc[(b, g)]
                gb, rb = set(got // blk), set(ref // blk)
                kth = sorted((s[bl * blk:min(len(s), bl * blk + blk)].max() for bl in rb))[0]
                for bl in gb ^ rb:
                    m = s[bl * blk:min(len(s), bl * blk + blk)].max()
                    assert abs(m - kth) <= 1e-3 * kth, (b, g, bl, m, kth)
            assert (idx[b, g, cnt[b, g]:] == -1).all()
    osa = H.hs2_sa_reuse(to_torch(grp.q_sa[0], dtype), dkv, grp.w, to_torch(idx, "i32"), to_torch(cnt, "i32"), k,
                         grp.scale).cpu().numpy()
    ref = O.sa_decode(grp.q_sa[0], kv, grp.w, idx, cnt, grp.scale)
    assert max_abs(osa, ref) <= tol(dtype)


def test_block_level_selection_rejects_bad_sizes(H):
    import torch

    grp = W.decode_group([300], Hq=8, Hkv=1, d=128, w=16, k=96, dtype="bf16", seed=20, n_sa=0, needles=0)
    dkv = kv_to_device(grp.kv)
    q = to_torch(grp.q_fa, "bf16")
    with pytest.raises(H.HS2Error):
        H.hs2_fa_select(q, dkv, 16, 96, grp.scale, max_t=300, sel_block=64)  # k not a multiple
    with pytest.raises(H.HS2Error):
        H.hs2_fa_select(q, dkv, 16, 96, grp.scale, max_t=300, sel_block=6)  # not a multiple of 4


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 4, 128), (8, 8, 64), (32, 1, 128)])
def test_fp8_kv_decode(H, Hq, Hkv, d):
    """FP8 E4M3 cache (one scale per page and KV head): FA output, lse and index sets against
    the oracle on the same codes and scales, and the SA layers over them."""
    grp = W.decode_group_fp8([3000, 1700, 130, 5000], Hq, Hkv, d, 64, 256, seed=23, n_sa=2, needles=8)
    check_group(H, grp)


def test_fp8_kv_small_wide_values(H):
    """FP8 cache whose V slabs are tiny and span four decades (V scales ~1e-9..1e-5): the FA
    and SA outputs keep their accuracy relative to their own magnitude."""
    grp = W.decode_group([2600, 900, 4100], 16, 2, 128, 64, 128, "bf16", seed=29, n_sa=1, needles=4)
    kv = grp.kv
    rng = np.random.default_rng(31)
    fac = 1e-4 * 10.0 ** rng.uniform(-2.0, 2.0, size=kv.v.shape[:2])
    vf = (W.values(kv.v, "bf16") * fac[:, :, None, None]).astype(np.float32)
    f32 = W.PagedKV(k=W.values(kv.k, "bf16"), v=vf, block_table=kv.block_table, seq_len=kv.seq_len, dtype="f32",
                    page=kv.page)
    grp.kv = W.quantize_kv_fp8(f32)
    o, lse, idx, cnt, sa, err = run_decode_group(H, grp)
    assert err == 0
    o_r, lse_r, idx_r, cnt_r, scores = O.fa_decode(grp.q_fa, grp.kv, grp.w, grp.k, grp.scale, return_scores=True)
    assert max_abs(o, o_r) <= 1e-2 * np.abs(o_r).max(), f"FA relative error {max_abs(o, o_r) / np.abs(o_r).max()}"
    assert max_abs(lse, lse_r) <= 2e-2
    check_index_sets(idx, cnt, idx_r, cnt_r, scores, "decode ")
    ref = O.sa_decode(grp.q_sa[0], grp.kv, grp.w, idx, cnt, grp.scale)
    assert max_abs(sa[0], ref) <= 1e-2 * np.abs(ref).max(), f"SA relative error {max_abs(sa[0], ref) / np.abs(ref).max()}"


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 4, 128), (8, 8, 64), (32, 1, 128), (16, 2, 64)])
def test_fp4_kv_decode(H, Hq, Hkv, d):
    """FP4 cache (E2M1 codes, an E4M3 scale per 16 channels, a slab scale per page and KV
    head): FA output, lse and index sets against the oracle on the same codes and scales,
    and the SA layers over them."""
    grp = W.decode_group_fp4([3000, 1700, 130, 5000], Hq, Hkv, d, 64, 256, seed=25, n_sa=2, needles=8)
    check_group(H, grp)


def test_fp4_kv_small_wide_values(H):
    """FP4 cache whose V slabs are tiny and span four decades: outputs keep their accuracy
    relative to their own magnitude."""
    grp = W.decode_group([2600, 900, 4100], 16, 2, 128, 64, 128, "bf16", seed=29, n_sa=1, needles=4)
    kv = grp.kv
    rng = np.random.default_rng(33)
    fac = 1e-4 * 10.0 ** rng.uniform(-2.0, 2.0, size=kv.v.shape[:2])
    vf = (W.values(kv.v, "bf16") * fac[:, :, None, None]).astype(np.float32)
    f32 = W.PagedKV(k=W.values(kv.k, "bf16"), v=vf, block_table=kv.block_table, seq_len=kv.seq_len, dtype="f32",
                    page=kv.page)
    grp.kv = W.quantize_kv_fp4(f32)
    o, lse, idx, cnt, sa, err = run_decode_group(H, grp)
    assert err == 0
    o_r, lse_r, idx_r, cnt_r, scores = O.fa_decode(grp.q_fa, grp.kv, grp.w, grp.k, grp.scale, return_scores=True)
    assert max_abs(o, o_r) <= 1e-2 * np.abs(o_r).max(), f"FA relative error {max_abs(o, o_r) / np.abs(o_r).max()}"
    assert max_abs(lse, lse_r) <= 2e-2
    check_index_sets(idx, cnt, idx_r, cnt_r, scores, "decode ")
    ref = O.sa_decode(grp.q_sa[0], grp.kv, grp.w, idx, cnt, grp.scale)
    assert max_abs(sa[0], ref) <= 1e-2 * np.abs(ref).max(), f"SA relative error {max_abs(sa[0], ref) / np.abs(ref).max()}"


def test_fp4_kv_rejects_prefill(H):
    import torch

    grp = W.prefill_group(300, 8, 1, 128, w=16, k=32, dtype="bf16", seed=26, n_sa=0)
    kv = W.quantize_kv_fp4(grp.kv)
    with pytest.raises(H.HS2Error):
        H.hs2_fa_select(to_torch(grp.q_fa, "bf16"), kv_to_device(kv), 16, 32, grp.scale, prefill=True)
    torch.cuda.synchronize()


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_low_precision_kv_sink_and_gate(H, fmt):
    """The FP8 / FP4 SA stream with the sink bias and the output gate (its richer epilogue
    variant), against the oracle on the same codes and scales."""
    import torch

    lens = [900, 2500, 130, 4000]
    make = W.decode_group_fp8 if fmt == "fp8" else W.decode_group_fp4
    grp = make(lens, 32, 4, 128, 32, 100, seed=19, n_sa=1, needles=4)
    kv = grp.kv
    dkv = kv_to_device(kv)
    _, _, idx, cnt = H.hs2_fa_select(to_torch(grp.q_fa, "bf16"), dkv, grp.w, grp.k, grp.scale,
                                     max_t=int(kv.seq_len.max()))
    rng = np.random.default_rng(4)
    sink = rng.normal(0.0, 2.0, 32).astype(np.float32)
    sink[0], sink[1] = -np.inf, 30.0
    gate = rng.normal(0.0, 2.0, (len(lens), 32, 128)).astype(np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    osa = H.hs2_sa_reuse(to_torch(grp.q_sa[0], "bf16"), dkv, grp.w, idx, cnt, grp.k, grp.scale, dev_err=err,
                         sink=torch.from_numpy(sink).cuda(), gate=torch.from_numpy(gate).cuda()).cpu().numpy()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.sa_decode(grp.q_sa[0], kv, grp.w, idx.cpu().numpy(), cnt.cpu().numpy(), grp.scale, sink=sink, gate=gate)
    assert max_abs(osa, ref) <= tol("bf16"), max_abs(osa, ref)
    assert np.abs(osa[:, 1]).max() < 1e-6  # the dominant sink takes the head's mass


def test_fp8_kv_rejects_prefill(H):
    import torch

    grp = W.prefill_group(300, 8, 1, 128, w=16, k=32, dtype="bf16", seed=24, n_sa=0)
    kv = W.quantize_kv_fp8(grp.kv)
    with pytest.raises(H.HS2Error):
        H.hs2_fa_select(to_torch(grp.q_fa, "bf16"), kv_to_device(kv), 16, 32, grp.scale, prefill=True)
    torch.cuda.synchronize()


def test_sa_layers_share_a_workspace_with_overlap(H):
    """Three decode SA layers back to back on one workspace that starts as random bytes: the
    first call clears the pair counters, the next two (HS2_SA_OVERLAP) take them as the call
    before left them; twice over, against the oracle."""
    import torch

    grp = W.decode_group([3000, 9000, 20000, 5000], Hq=32, Hkv=4, d=128, w=128, k=512, dtype="bf16", seed=31,
                         n_sa=3, needles=8)
    kv = grp.kv
    dkv = kv_to_device(kv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = to_torch(grp.q_fa, "bf16")
    _, _, idx, cnt = H.hs2_fa_select(q, dkv, grp.w, grp.k, grp.scale, max_t=int(kv.seq_len.max()), dev_err=err)
    nb = H.hs2_sa_reuse_workspace(kv.B, 32, dkv, grp.w, grp.k)
    ws = torch.randint(0, 256, (nb,), dtype=torch.uint8, device="cuda")
    idx_h, cnt_h = idx.cpu().numpy(), cnt.cpu().numpy()
    for rep in range(2):
        outs = [H.hs2_sa_reuse(to_torch(grp.q_sa[j], "bf16"), dkv, grp.w, idx, cnt, grp.k, grp.scale, workspace=ws,
                               dev_err=err, overlap=j > 0) for j in range(3)]
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for j, o in enumerate(outs):
            ref = O.sa_decode(grp.q_sa[j], kv, grp.w, idx_h, cnt_h, grp.scale)
            assert max_abs(o.cpu().numpy(), ref) <= tol("bf16"), (rep, j)


def test_group_step_in_a_cuda_graph_matches_eager(H):
    """The decode group step as bench.py runs it, captured in a CUDA graph: the FA call, then
    three SA layers on one workspace (the second and third with HS2_SA_OVERLAP, so their
    kernels overlap the previous one through programmatic dependent launch). Two replays give
    the eager run's outputs bit for bit (the merges sum partials in a fixed order) and those
    match the oracle."""
    import torch

    grp = W.decode_group([3000, 9000, 20000, 5000, 12000, 7000], Hq=32, Hkv=4, d=128, w=128, k=512, dtype="bf16",
                         seed=41, n_sa=3, needles=8)
    kv = grp.kv
    dkv = kv_to_device(kv)
    B, Hq, d = grp.q_fa.shape
    max_t = int(kv.seq_len.max())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = to_torch(grp.q_fa, "bf16")
    qs = [to_torch(x, "bf16") for x in grp.q_sa]
    ws_fa = torch.empty(H.hs2_fa_select_workspace(B, Hq, dkv, max_t, grp.k), dtype=torch.uint8, device="cuda")
    ws_sa = torch.empty(H.hs2_sa_reuse_workspace(B, Hq, dkv, grp.w, grp.k), dtype=torch.uint8, device="cuda")
    o = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    idx = torch.empty((B, 4, grp.k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, 4), dtype=torch.int32, device="cuda")
    osa = [torch.empty((B, Hq, d), dtype=torch.float32, device="cuda") for _ in range(3)]

    def step(stream):
        H.hs2_fa_select(q, dkv, grp.w, grp.k, grp.scale, max_t=max_t, out=(o, lse, idx, cnt), workspace=ws_fa,
                        dev_err=err, stream=stream)
        for j in range(3):
            H.hs2_sa_reuse(qs[j], dkv, grp.w, idx, cnt, grp.k, grp.scale, out=osa[j], workspace=ws_sa, dev_err=err,
                           stream=stream, overlap=j > 0)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    eager = [x.clone() for x in (o, lse, idx, cnt, *osa)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for rep in range(2):
        for x in (o, lse, *osa):
            x.fill_(float("nan"))
        idx.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, (o, lse, idx, cnt, *osa)):
            assert torch.equal(a, b), rep
    assert int(err.item()) == 0
    idx_h, cnt_h = idx.cpu().numpy(), cnt.cpu().numpy()
    for j in range(3):
        ref = O.sa_decode(grp.q_sa[j], kv, grp.w, idx_h, cnt_h, grp.scale)
        assert max_abs(osa[j].cpu().numpy(), ref) <= tol("bf16"), j
