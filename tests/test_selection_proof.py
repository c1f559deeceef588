"""The prefill selection's exactness argument, checked on the host.

The GPU selection streams each row's scores once: a sampled sweep (every 8th far position)
fills a log histogram (bins of 1/8 octave over the fp32 bit pattern) and sets a threshold
tau whose estimated count is 1.35 times the budget; the exact sweep keeps, in ascending
position, every key >= tau up to a capacity and remembers only the largest dropped key. A
row's top-k is taken from its kept candidates when (a) at least k of them are >= tau and (b)
no dropped key exceeds the k-th largest kept key; otherwise the row is recomputed over its
whole far range (here: None), never approximated. Neither the stride nor the target enters
the argument, only which rows are provable.
This test restates that procedure in numpy and checks, on random, tied and adversarial rows,
that whenever (a) and (b) hold the result equals the exact top-k (score descending, lower
position first on ties). It tests the method, not the kernel: the GPU path is compared with
the oracle in tests/test_gpu_prefill.py.
"""
import numpy as np
import pytest

BINS = 256
BIN_BASE = 0x410 - (BINS - 1)  # bin 255 holds keys >> 20 == 0x410 (score 8.0)
STRIDE = 8
TARGET = 1.35


def exact_topk(keys, k):
    order = np.lexsort((np.arange(len(keys)), -keys.astype(np.int64)))
    return np.sort(order[: min(k, len(keys))])


def streamed_topk(keys, k, cap):
    """The GPU procedure on one row of uint32 keys; None when the row goes to the completion pass."""
    nF = len(keys)
    samp = keys[::STRIDE]
    bins = np.clip((samp >> 20).astype(np.int64) - BIN_BASE, 0, BINS - 1)
    hist = np.bincount(bins, minlength=BINS)
    scale = nF / len(samp)
    tau, cum = 0, 0.0
    for b in range(BINS - 1, -1, -1):
        cum += scale * hist[b]
        if cum >= TARGET * k:
            tau = 0 if b == 0 else (BIN_BASE + b) << 20
            break
    cand = np.flatnonzero(keys >= tau)  # ascending positions
    kept, dropped = cand[:cap], cand[cap:]
    if len(kept) < k:
        return None
    kth = np.sort(keys[kept])[::-1][k - 1]
    if len(dropped) and keys[dropped].max() > kth:
        return None
    sub = exact_topk(keys[kept], k)
    return np.sort(kept[sub])


def as_keys(scores):
    return np.asarray(scores, dtype=np.float32).view(np.uint32)


def rows(rng):
    for _ in range(60):
        nF = int(rng.integers(70, 6000))
        yield "lognormal", as_keys(rng.lognormal(-8, 2, nF))
    for _ in range(20):
        nF = int(rng.integers(70, 3000))
        yield "few values", as_keys(rng.choice([1e-4, 2e-4, 3e-4], nF))
    for _ in range(10):
        nF = int(rng.integers(300, 3000))
        s = np.where(np.arange(nF) % STRIDE == 0, 1e-6, 1e-3) * rng.uniform(0.9, 1.1, nF)
        yield "hidden from the sample", as_keys(s)
    for _ in range(10):
        nF = int(rng.integers(300, 3000))
        s = rng.lognormal(-8, 1, nF)
        s[-rng.integers(1, 50):] *= 1e3  # the largest scores all come last
        yield "late maxima", as_keys(s)
    yield "all equal", as_keys(np.full(2500, 3e-4))


@pytest.mark.parametrize("k,cap", [(64, 256), (100, 400), (256, 1024)])
def test_streamed_selection_is_exact_whenever_it_proves_itself(k, cap):
    rng = np.random.default_rng(k)
    proven = flagged = 0
    for kind, keys in rows(rng):
        got = streamed_topk(keys, k, cap)
        if got is None:
            flagged += 1
            continue
        proven += 1
        np.testing.assert_array_equal(got, exact_topk(keys, k), err_msg=kind)
    assert proven > 0 and flagged > 0  # both branches are exercised


def test_dropping_an_equal_key_keeps_the_proof():
    # every key equal: only the first `cap` positions are kept, the dropped keys tie the k-th
    # kept one and lose the tie (higher position), so the row is proven and takes 0..k-1
    keys = as_keys(np.full(1000, 5e-4))
    np.testing.assert_array_equal(streamed_topk(keys, 50, 200), np.arange(50))


def test_a_larger_dropped_key_flags_the_row():
    s = np.full(1000, 1e-4)
    s[900] = 1e-2  # past the capacity and larger than everything kept
    assert streamed_topk(as_keys(s), 10, 256) is None
