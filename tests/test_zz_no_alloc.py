"""hs2_fa_select_noalloc: the FA scan + top-k for callers that cannot allocate device memory.

Such callers (an engine that has reserved nearly all HBM for its KV pool, or a latency-
critical thread that must not call cudaMalloc/cudaFree because they can synchronise the
device) get the library's own static scratch instead of a workspace argument. This test
calls the entry point through the C ABI twice in a row, on two different problems, and
checks each result against hs2_fa_select with a caller workspace on the same inputs. It
also checks that a problem larger than the static scratch is rejected without a launch.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from top_hs2_fa_gb300 import workloads as W

from hs2_testutil import kv_to_device, max_abs, to_torch, tol

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


def _outputs(torch, B, Hq, Hkv, d, k):
    return (torch.empty((B, Hq, d), dtype=torch.float32, device="cuda"),
            torch.empty((B, Hq), dtype=torch.float32, device="cuda"),
            torch.full((B, Hkv, k), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, Hkv), -7, dtype=torch.int32, device="cuda"))


def test_noalloc_matches_workspace_entry_point_twice(H):
    import torch

    cases = [
        W.decode_group([3000, 1234, 4096, 77], Hq=32, Hkv=4, d=128, w=128, k=256, dtype="bf16", seed=31,
                       n_sa=0, needles=8),
        W.decode_group([5000, 129, 2500], Hq=8, Hkv=2, d=64, w=16, k=100, dtype="bf16", seed=32, n_sa=0,
                       needles=4),
    ]
    for grp in cases:  # two calls in a row; the second must not see the first call's scratch
        kv = grp.kv
        dkv = kv_to_device(kv)
        q = to_torch(grp.q_fa, kv.dtype)
        max_t = int(kv.seq_len.max())
        B, Hq, d = grp.q_fa.shape
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = H.hs2_fa_select(q, dkv, grp.w, grp.k, grp.scale, max_t=max_t, dev_err=err)
        got = H.hs2_fa_select_noalloc(q, dkv, grp.w, grp.k, grp.scale, max_t=max_t,
                                      out=_outputs(torch, B, Hq, kv.Hkv, d, grp.k), dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref = [x.cpu().numpy() for x in ref]
        got = [x.cpu().numpy() for x in got]
        assert max_abs(got[0], ref[0]) <= tol(kv.dtype)
        assert max_abs(got[1], ref[1]) <= tol(kv.dtype)
        assert np.array_equal(got[2], ref[2])
        assert np.array_equal(got[3], ref[3])


def test_noalloc_rejects_problems_beyond_its_scratch(H):
    import torch

    lib = H.load()
    cap = int(lib.hs2_fa_select_noalloc_capacity())
    assert cap == 64 << 20
    small = torch.zeros((1, 4, 64, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((64, 512), dtype=torch.int32, device="cuda")
    sl = torch.ones(64, dtype=torch.int32, device="cuda")
    kv = H.KV(k=small, v=small, block_table=bt, seq_len=sl)
    c = kv.c()
    need = lib.hs2_fa_select_workspace(64, 32, ctypes.byref(c), 32768, 1024, 0)
    assert need > cap
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = _outputs(torch, 64, 32, 4, 128, 1024)
    st = lib.hs2_fa_select_noalloc(q.data_ptr(), 64, 32, ctypes.byref(c), 32768, 128, 1024, 0.088, 0,
                                   out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), out[3].data_ptr(),
                                   None, torch.cuda.current_stream().cuda_stream)
    assert st == -5
    assert b"scratch" in lib.hs2_strerror(st)
    torch.cuda.synchronize()
    assert int(out[3].min().item()) == -7  # nothing was launched
