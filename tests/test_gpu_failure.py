"""Device-side failure detection without a fault: a bounded wait that runs out.

The library's mbarrier waits read %globaltimer and give up after a limit. The self-test entry
point waits on a barrier nothing arrives on; the test checks that the kernel returns, that the
timeout flag is set, and that the context still runs real work afterwards.
"""
import time

import pytest

from top_hs2_fa_gb300 import workloads as W

from hs2_testutil import kv_to_device, to_torch

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


def test_bounded_wait_gives_up_and_flags_timeout(H):
    import torch

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    H.hs2_selftest_wait_timeout(20000, err)  # 20 ms limit
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) & H.DEV_TIMEOUT
    assert elapsed < 5.0
    # the context is still usable: a normal call runs and flags nothing
    grp = W.decode_group([300, 500], Hq=8, Hkv=1, d=128, w=16, k=32, dtype="bf16", seed=9, n_sa=0, needles=0)
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    H.hs2_fa_select(to_torch(grp.q_fa, "bf16"), kv_to_device(grp.kv), 16, 32, grp.scale, max_t=500, dev_err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0


def test_selftest_rejects_bad_limits(H):
    import torch

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, 3_000_000):
        with pytest.raises(H.HS2Error):
            H.hs2_selftest_wait_timeout(bad, err)
