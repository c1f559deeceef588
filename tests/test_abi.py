"""The C-ABI library builds, loads on a machine without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from top_hs2_fa_gb300 import build
from top_hs2_fa_gb300 import hs2 as H

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "hs2.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return H.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hs2_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("hs2_fa_select", "hs2_sa_reuse", "hs2_hier_reindex"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(H.EXPORTS) <= set(declared_functions())


def test_binding_constants_match_the_header():
    """The binding's device-error bits and dtype codes are the header's."""
    text = open(HEADER).read()
    bits = {m: int(v) for m, v in re.findall(r"#define HS2_DEV_([A-Z_]+)\s+(\d+)", text)}
    assert bits == {"BAD_PAGE": H.DEV_BAD_PAGE, "BAD_INDEX": H.DEV_BAD_INDEX, "TIMEOUT": H.DEV_TIMEOUT,
                    "BAD_LENGTH": H.DEV_BAD_LENGTH, "SELECT": H.DEV_SELECT}
    dt = dict(re.findall(r"HS2_(F32|BF16|FP8_E4M3|FP4_E2M1) = (\d+)", text))
    assert {k: int(v) for k, v in dt.items()} == {"F32": H.F32, "BF16": H.BF16, "FP8_E4M3": H.FP8_E4M3,
                                                  "FP4_E2M1": H.FP4_E2M1}


def test_version_and_strings(lib):
    assert lib.hs2_abi_version() == H.ABI_VERSION == 6
    for st, word in [(0, "ok"), (-1, "invalid"), (-2, "unsupported"), (-3, "CUDA"), (-4, "device")]:
        assert word in lib.hs2_strerror(st).decode()


def _kv(**over):
    base = dict(k=16, v=32, block_table=48, seq_len=64, batch=2, num_pages=10, max_pages=5, page_size=64,
                Hkv=2, d=128, dtype=1)
    base.update(over)
    return H.hs2_kv(**base)


def _fa(lib, kv, B=2, Hq=8, max_t=100, w=16, k=8, prefill=0, q=256, ws=4096, wsb=1 << 30, o=512, idx=768, cnt=1024):
    return lib.hs2_fa_select(q, B, Hq, ctypes.byref(kv), max_t, w, k, 0.1, prefill, o, None, idx, cnt, ws, wsb,
                             None, None)


def test_host_validation_rejects_before_launch(lib):
    assert _fa(lib, _kv(page_size=32)) == -1
    assert _fa(lib, _kv(d=96)) == -1
    assert _fa(lib, _kv(), Hq=7) == -1            # Hq % Hkv != 0
    assert _fa(lib, _kv(), Hq=6) == -2            # 3 query heads per KV head
    assert _fa(lib, _kv(), B=3) == -1             # batch mismatch in decode
    assert _fa(lib, _kv(), prefill=1) == -1       # prefill needs batch == 1
    assert _fa(lib, _kv(), w=-1) == -1
    assert _fa(lib, _kv(), k=-2) == -1
    assert _fa(lib, _kv(), max_t=5 * 64 + 1) == -1  # beyond the table's capacity
    assert _fa(lib, _kv(k=17)) == -1              # misaligned K pool
    assert _fa(lib, _kv(), q=0) == -1
    assert _fa(lib, _kv(), ws=0) == -1
    assert _fa(lib, _kv(), wsb=16) == -1          # workspace too small
    assert _fa(lib, _kv(), ws=4096 + 16) == -1    # workspace not 256-byte aligned
    kv0 = _kv(batch=0)
    assert _fa(lib, kv0, B=0) == -1


def test_sa_validation(lib):
    kv = _kv()
    st = lib.hs2_sa_reuse(256, 2, 8, ctypes.byref(kv), -1, 512, 768, 8, 0.1, 0, 1024, 4096, 1 << 30, None, None)
    assert st == -1
    st = lib.hs2_sa_reuse(256, 2, 8, ctypes.byref(kv), 16, 512, 0, 8, 0.1, 0, 1024, 4096, 1 << 30, None, None)
    assert st == -1


def test_sa_flags_validation(lib):
    """hs2_sa_reuse_ex takes 0 or HS2_SA_OVERLAP; any other bit is refused before any launch."""
    kv = _kv()
    for bad in (2, 4, -1):
        st = lib.hs2_sa_reuse_ex(256, 2, 8, ctypes.byref(kv), 16, 512, 768, 8, 0.1, 0, None, None,
                                 H.SA_OVERLAP | bad, 1024, 4096, 1 << 30, None, None)
        assert st == -1


def test_workspace_sizes_grow_with_problem(lib):
    kv = _kv()
    a = lib.hs2_fa_select_workspace(2, 8, ctypes.byref(kv), 100, 8, 0)
    b = lib.hs2_fa_select_workspace(2, 8, ctypes.byref(kv), 300, 8, 0)
    assert 0 < a < b and a % 256 == 0
    assert lib.hs2_sa_reuse_workspace(2, 8, ctypes.byref(kv), 16, 64, 0) > 0
