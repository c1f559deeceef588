"""GPU parity of the prefill path (causal FA rows, their selection, SA over every row).

Through the C ABI against the oracle on the same seeded arrays. Small cases are checked on
every row; the full-size prefill workload on sampled rows.
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


def run_fa(H, grp, k=None, w=None):
    import torch

    kv = grp.kv
    dkv = kv_to_device(kv)
    q = to_torch(grp.q_fa, kv.dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = grp.k if k is None else k
    w = grp.w if w is None else w
    o, lse, idx, cnt = H.hs2_fa_select(q, dkv, w, k, grp.scale, prefill=True, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    return o.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy()


@pytest.mark.parametrize("n,Hq,Hkv,permute", [(1000, 8, 2, True), (384, 4, 4, False), (2048, 32, 4, True)])
def test_prefill_fa_rows_outputs(H, n, Hq, Hkv, permute):
    grp = W.prefill_group(n, Hq, Hkv, 128, w=16, k=0, dtype="bf16", seed=21, n_sa=0, rho=0.99, permute=permute)
    o, lse, idx, cnt = run_fa(H, grp, k=0)
    rows = np.arange(n) if n <= 1024 else np.unique(np.concatenate([
        np.random.default_rng(0).choice(n, 200, replace=False), [0, 1, 127, 128, 129, n - 1]]))
    o_r, lse_r, _, _ = O.fa_prefill_rows(grp.q_fa, grp.kv, rows, grp.w, 0, grp.scale)
    assert max_abs(o[rows], o_r) <= tol("bf16"), max_abs(o[rows], o_r)
    assert max_abs(lse[rows], lse_r) <= tol("bf16")
    assert (cnt == 0).all()


@pytest.mark.parametrize("n", [1, 50, 64, 65, 130, 200])
def test_prefill_short_sequences(H, n):
    """Sequences shorter than a key tile or ending inside one: the tile's second page lies
    past the pool, and must read as zeros (not as whatever the slot held). FA output, lse and
    the selection (k covers every far range here) on every row."""
    grp = W.prefill_group(n, 8, 1, 128, w=16, k=300, dtype="bf16", seed=27, n_sa=1, rho=0.99, permute=True)
    o, lse, idx, cnt = run_fa(H, grp)
    rows = np.arange(n)
    o_r, lse_r, idx_r, cnt_r = O.fa_prefill_rows(grp.q_fa, grp.kv, rows, grp.w, grp.k, grp.scale)
    assert np.isfinite(o).all() and max_abs(o, o_r) <= tol("bf16"), max_abs(o, o_r)
    assert max_abs(lse, lse_r) <= tol("bf16")
    assert np.array_equal(cnt, cnt_r) and np.array_equal(idx, idx_r)


def test_prefill_fa_sharp_needles(H):
    # unit-variance q and k: concentrated rows, needles aligned with the last row
    grp = W.prefill_group(700, 8, 1, 128, w=16, k=0, dtype="bf16", seed=22, n_sa=0, needles=8)
    o, lse, _, _ = run_fa(H, grp, k=0)
    rows = np.arange(700)
    o_r, lse_r, _, _ = O.fa_prefill_rows(grp.q_fa, grp.kv, rows, grp.w, 0, grp.scale)
    assert max_abs(o, o_r) <= tol("bf16")
    assert max_abs(lse, lse_r) <= tol("bf16")


def test_prefill_trivial_selection_rows(H):
    # every row's far range fits the budget (n - w <= k): each row takes all of F
    grp = W.prefill_group(300, 8, 2, 128, w=16, k=400, dtype="bf16", seed=23, n_sa=0)
    _, _, idx, cnt = run_fa(H, grp)
    for i in range(300):
        nf = max(0, i + 1 - 16)
        assert (cnt[i] == nf).all()
        assert (idx[i, :, :nf] == np.arange(nf)).all() and (idx[i, :, nf:] == -1).all()


def check_selection(H, grp, rows=None):
    o, lse, idx, cnt = run_fa(H, grp)
    n = grp.q_fa.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    o_r, lse_r, idx_r, cnt_r, sc = O.fa_prefill_rows(grp.q_fa, grp.kv, rows, grp.w, grp.k, grp.scale,
                                                     return_scores=True)
    assert max_abs(o[rows], o_r) <= tol("bf16")
    differ = check_index_sets(idx[rows], cnt[rows], idx_r, cnt_r, sc, "prefill ")
    return idx, cnt, differ


def test_prefill_selection_small_all_rows(H):
    grp = W.prefill_group(1000, 8, 2, 128, w=16, k=64, dtype="bf16", seed=31, n_sa=0, rho=0.99, permute=True)
    check_selection(H, grp)


def test_prefill_selection_gqa8_sampled(H):
    grp = W.prefill_group(2048, 32, 4, 128, w=128, k=256, dtype="bf16", seed=32, n_sa=0, rho=0.999)
    rows = np.unique(np.concatenate([np.random.default_rng(1).choice(2048, 150, replace=False),
                                     [0, 127, 128, 383, 384, 385, 1023, 2047]]))
    check_selection(H, grp, rows)


def test_prefill_selection_ties_take_lowest_positions(H):
    # identical keys: every far score is equal, so each row takes its first k positions
    grp = W.prefill_group(1500, 8, 1, 128, w=16, k=100, dtype="bf16", seed=33, n_sa=0)
    kv = grp.kv
    kv.k[:] = kv.k[0:1, :, 0:1, :]
    o, lse, idx, cnt = run_fa(H, grp)
    for i in (200, 700, 1499):
        assert cnt[i, 0] == 100 and (idx[i, 0] == np.arange(100)).all()


def sample_hiding_keys(n, Hq, Hkv, w, k, seed):
    """Prefill inputs on which the streamed candidates cannot prove many rows' top-k: keys
    at multiples of 4 (a superset of the positions the sampled sweep sees, multiples of 8)
    score low and all others high, so the sampled threshold lets about 3/4 of every far
    range through, long rows overflow
    their candidate buffers (capacity max(256, 4k)) with high keys, and the largest dropped
    key beats the k-th kept one (tests/test_selection_proof.py restates the mechanism)."""
    d = 128
    grp = W.prefill_group(n, Hq, Hkv, d, w=w, k=k, dtype="bf16", seed=seed, n_sa=0)
    rng = np.random.default_rng(seed + 1)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = 3.0 * u + 0.3 * rng.standard_normal((n, Hq, d))
    sign = np.where(np.arange(n) % 4 == 0, -1.0, 1.0)
    kv = grp.kv
    for g in range(Hkv):
        keys = sign[:, None] * 3.0 * u + 0.3 * rng.standard_normal((n, d))
        for p in range(n):
            kv.k[kv.block_table[0][p // kv.page], g, p % kv.page, :] = W.store(keys[p].astype(np.float32), "bf16")
    grp.q_fa = W.store(q.astype(np.float32), "bf16")
    return grp


@pytest.mark.parametrize("n,Hq,Hkv,all_rows", [(1500, 8, 1, True), (2600, 32, 2, False), (2100, 32, 1, False)])
def test_prefill_selection_unprovable_rows_are_completed(H, n, Hq, Hkv, all_rows):
    """Rows whose streamed candidates cannot prove their top-k are recomputed exactly over
    their whole far range within the same call: no row comes back without an answer, no
    device flag is raised, and every checked row equals the oracle (1e-3 band), for 8, 16
    and 32 query heads per KV head."""
    w, k = 16, 64
    grp = sample_hiding_keys(n, Hq, Hkv, w, k, seed=35)
    o, lse, idx, cnt = run_fa(H, grp)  # asserts dev_err == 0
    nF = np.maximum(0, np.arange(n) + 1 - w)
    assert np.array_equal(cnt, np.repeat(np.minimum(k, nF)[:, None], Hkv, 1))
    rows = np.arange(n) if all_rows else np.unique(np.concatenate([
        np.random.default_rng(2).choice(n, 160, replace=False), [w + k, w + k + 1, n - 2, n - 1]]))
    _, _, idx_r, cnt_r, sc = O.fa_prefill_rows(grp.q_fa, grp.kv, rows, w, k, grp.scale, return_scores=True)
    check_index_sets(idx[rows], cnt[rows], idx_r, cnt_r, sc, "completed ")


def test_prefill_selection_needles(H):
    grp = W.prefill_group(3000, 8, 1, 128, w=32, k=128, dtype="bf16", seed=34, n_sa=0, needles=16)
    idx, cnt, _ = check_selection(H, grp, rows=[2999, 2500, 1200, 160, 161])


@pytest.mark.slow
def test_prefill_full_size_sampled_rows(H):
    """Prefill workload at full size (n=32768, Hq=32, Hkv=4, d=128, w=128, k=1024, AR(1) keys,
    five SA layers): 256 seeded random rows plus {0, w-1, w, w+k-1, w+k, n-1}, each exact
    against all its keys: FA output, lse and index sets; then every SA layer at those rows with
    the GPU's index sets, and the first SA layer again with the oracle's sets at those rows."""
    import torch

    n, w, k = 32768, 128, 1024
    grp = W.prefill_group(n, 32, 4, 128, w=w, k=k, dtype="bf16", seed=0, n_sa=5, rho=0.999)
    rows = np.unique(np.concatenate([np.random.default_rng(7).choice(n, 256, replace=False),
                                     [0, w - 1, w, w + k - 1, w + k, n - 1]]))
    o, lse, idx, cnt = run_fa(H, grp)
    o_r, lse_r, idx_r, cnt_r, sc = O.fa_prefill_rows(grp.q_fa, grp.kv, rows, w, k, grp.scale, return_scores=True)
    assert max_abs(o[rows], o_r) <= tol("bf16"), max_abs(o[rows], o_r)
    assert max_abs(lse[rows], lse_r) <= tol("bf16"), max_abs(lse[rows], lse_r)
    check_index_sets(idx[rows], cnt[rows], idx_r, cnt_r, sc, "prefill ")
    assert (cnt >= 0).all()
    dkv = kv_to_device(grp.kv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_idx, d_cnt = to_torch(idx, "i32"), to_torch(cnt, "i32")
    for j in range(5):
        osa = H.hs2_sa_reuse(to_torch(grp.q_sa[j], "bf16"), dkv, w, d_idx, d_cnt, k, grp.scale, prefill=True,
                             dev_err=err)[torch.from_numpy(rows).cuda()].cpu().numpy()
        ref = O.sa_prefill_rows(grp.q_sa[j], grp.kv, rows, w, idx, cnt, grp.scale)
        assert max_abs(osa, ref) <= tol("bf16"), (j, max_abs(osa, ref))
    mix_idx, mix_cnt = idx.copy(), cnt.copy()
    mix_idx[rows], mix_cnt[rows] = idx_r, cnt_r
    osa = H.hs2_sa_reuse(to_torch(grp.q_sa[0], "bf16"), dkv, w, to_torch(mix_idx, "i32"), to_torch(mix_cnt, "i32"),
                         k, grp.scale, prefill=True, dev_err=err)[torch.from_numpy(rows).cuda()].cpu().numpy()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.sa_prefill_rows(grp.q_sa[0], grp.kv, rows, w, mix_idx, mix_cnt, grp.scale)
    assert max_abs(osa, ref) <= tol("bf16"), max_abs(osa, ref)


def test_tiny_fp32_prefill_all_rows(H):
    """Tiny fp32 group, prefill half: all 2048 rows of the FA (output, lse, index sets) and
    the SA layer over every row, at the fp32 tolerance; the SA layer also with the oracle's
    index sets fed to both."""
    import torch

    tg = W.tiny_group(seed=0)
    pre = tg.prefill
    n = pre.q_fa.shape[0]
    o, lse, idx, cnt = run_fa(H, pre)
    rows = np.arange(n)
    o_r, lse_r, idx_r, cnt_r, sc = O.fa_prefill_rows(pre.q_fa, pre.kv, rows, pre.w, pre.k, pre.scale,
                                                     return_scores=True)
    assert max_abs(o, o_r) <= tol("f32"), max_abs(o, o_r)
    assert max_abs(lse, lse_r) <= tol("f32"), max_abs(lse, lse_r)
    check_index_sets(idx, cnt, idx_r, cnt_r, sc, "tiny prefill ")
    dkv = kv_to_device(pre.kv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = to_torch(pre.q_sa[0], "f32")
    osa = H.hs2_sa_reuse(q, dkv, pre.w, to_torch(idx, "i32"), to_torch(cnt, "i32"), pre.k, pre.scale, prefill=True,
                         dev_err=err).cpu().numpy()
    ref = O.sa_prefill_rows(pre.q_sa[0], pre.kv, rows, pre.w, idx, cnt, pre.scale)
    assert max_abs(osa, ref) <= tol("f32"), max_abs(osa, ref)
    osa = H.hs2_sa_reuse(q, dkv, pre.w, to_torch(idx_r, "i32"), to_torch(cnt_r, "i32"), pre.k, pre.scale,
                         prefill=True, dev_err=err).cpu().numpy()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.sa_prefill_rows(pre.q_sa[0], pre.kv, rows, pre.w, idx_r, cnt_r, pre.scale)
    assert max_abs(osa, ref) <= tol("f32"), max_abs(osa, ref)


@pytest.mark.parametrize("n,Hq,Hkv,w,k", [(1000, 8, 2, 16, 64), (777, 32, 4, 128, 256), (600, 16, 1, 32, 100)])
def test_prefill_sa_rows(H, n, Hq, Hkv, w, k):
    """SA prefill (tensor-core gather) on every row, with the GPU's own index sets, and with
    the oracle's index sets fed to both."""
    import torch

    grp = W.prefill_group(n, Hq, Hkv, 128, w=w, k=k, dtype="bf16", seed=41, n_sa=2, rho=0.99, permute=True)
    o, lse, idx, cnt = run_fa(H, grp)
    dkv = kv_to_device(grp.kv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = np.arange(n)
    for j in range(2):
        qs = to_torch(grp.q_sa[j], "bf16")
        osa = H.hs2_sa_reuse(qs, dkv, w, to_torch(idx, "i32"), to_torch(cnt, "i32"), k, grp.scale, prefill=True,
                             dev_err=err).cpu().numpy()
        ref = O.sa_prefill_rows(grp.q_sa[j], grp.kv, rows, w, idx, cnt, grp.scale)
        assert max_abs(osa, ref) <= tol("bf16"), max_abs(osa, ref)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _, _, idx_r, cnt_r = O.fa_prefill_rows(grp.q_fa, grp.kv, rows, w, k, grp.scale)
    osa = H.hs2_sa_reuse(to_torch(grp.q_sa[0], "bf16"), dkv, w, to_torch(idx_r, "i32"), to_torch(cnt_r, "i32"), k,
                         grp.scale, prefill=True).cpu().numpy()
    ref = O.sa_prefill_rows(grp.q_sa[0], grp.kv, rows, w, idx_r, cnt_r, grp.scale)
    assert max_abs(osa, ref) <= tol("bf16")


@pytest.mark.parametrize("n,Hq,Hkv", [(1000, 8, 2), (600, 16, 1)])
def test_prefill_sa_sink_bias_and_output_gate(H, n, Hq, Hkv):
    """SA prefill (tensor-core gather) with per-head sink logits and elementwise gate logits."""
    import torch

    grp = W.prefill_group(n, Hq, Hkv, 128, w=16, k=64, dtype="bf16", seed=43, n_sa=1, rho=0.99, permute=True)
    _, _, idx, cnt = run_fa(H, grp)
    rng = np.random.default_rng(5)
    sink = rng.normal(0.0, 2.0, Hq).astype(np.float32)
    sink[0] = -np.inf
    gate = rng.normal(0.0, 2.0, (n, Hq, 128)).astype(np.float32)
    osa = H.hs2_sa_reuse(to_torch(grp.q_sa[0], "bf16"), kv_to_device(grp.kv), 16, to_torch(idx, "i32"),
                         to_torch(cnt, "i32"), 64, grp.scale, prefill=True, sink=torch.from_numpy(sink).cuda(),
                         gate=torch.from_numpy(gate).cuda()).cpu().numpy()
    ref = O.sa_prefill_rows(grp.q_sa[0], grp.kv, np.arange(n), 16, idx, cnt, grp.scale, sink=sink, gate=gate)
    assert max_abs(osa, ref) <= tol("bf16"), max_abs(osa, ref)
