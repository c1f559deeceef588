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
