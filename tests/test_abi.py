"""CPU-only checks of the C ABI: the library builds, loads, exports every
symbol include/twell.h declares, and its host-side logic (sizes, argument
checks, status strings) answers without touching a GPU."""
import ctypes
import os
import re

import pytest

from activation_sparse_transformer_tcgen05_gb300 import build as tbuild
from activation_sparse_transformer_tcgen05_gb300 import twell as tw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    tbuild.build()
    return tw.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "twell.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(twell_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in twell.h but not exported"
    assert set(names) == set(tw.EXPORTED_SYMBOLS)


def test_status_strings(lib):
    assert tw.twell_status_string(0) == "ok"
    assert "capacity" in tw.twell_status_string(4)
    assert tw.twell_status_string(99) == "unknown status"


def test_slot_bound_and_workspace_sizes(lib):
    assert tw.twell_buf_slots_bound(4096, 8192, 128) == 4096 * 8192
    assert tw.twell_buf_slots_bound(0, 8, 1) == -1
    fwd = tw.twell_workspace_bytes(tw.OP_FFN_FWD, 4096, 2048, 8192, 128)
    # staging: one 32-bit entry per (row, column) plus a count per (row, 256-column block)
    assert fwd >= 4096 * 8192 * 4 + 4096 * 32 * 4
    assert tw.twell_workspace_bytes(tw.OP_PACK, 64, 128, 512, 16) == 0
    bwd_small = tw.twell_workspace_bytes(tw.OP_FFN_BWD, 4096, 2048, 8192, 128, 10_000)
    bwd_big = tw.twell_workspace_bytes(tw.OP_FFN_BWD, 4096, 2048, 8192, 128, 1_000_000)
    assert bwd_big - bwd_small >= 3 * 4 * 990_000 - 3 * 256  # dpre, row and slot per stored entry
    assert tw.twell_workspace_bytes(tw.OP_FFN_FWD, 0, 2048, 8192, 128) == 0
    # union down-projection: per group a list of F unit ids, plus one word per stored entry
    u_small = tw.twell_spmm_down_tc_workspace_bytes(4096, 8192, 10_000)
    u_big = tw.twell_spmm_down_tc_workspace_bytes(4096, 8192, 1_000_000)
    assert u_small >= 32 * 8192 * 4 and u_big - u_small >= 4 * 990_000 - 256
    assert tw.twell_spmm_down_tc_workspace_bytes(4096, 65544, 10) == 0
    assert tw.twell_spmm_down_tc_workspace_bytes(4096, 100, 10) == 0  # F % 8 != 0


def test_host_argument_errors_need_no_gpu(lib):
    buf = tw._TwellBuf(64, 512, 16, 4, 0, None, None, None, None, None)
    rc = lib.twell_ffn_fwd(None, None, None, None, None, 64, 128, 512, 16, ctypes.byref(buf),
                           None, None, 0, None, None)
    assert rc == 1  # TWELL_ERR_INVALID_ARG
    rc = lib.twell_pack(None, 64, 512, 512, 16, ctypes.byref(buf), None, None)
    assert rc == 1
    rc = lib.twell_spmm_down(None, None, 128, None, None, None)
    assert rc == 1
    rc = lib.twell_ffn_bwd(None, None, None, None, None, 128, 0.0, None, None, None, None, None, 0, None, None)
    assert rc == 1
    rc = lib.twell_check(None, None, None)
    assert rc == 1
    rc = lib.twell_dense_ffn_fwd(None, None, None, None, 64, 128, 512, None, None, None, None)
    assert rc == 1
    rc = lib.twell_dense_ffn_bwd(None, None, None, None, None, 64, 128, 512, 0.0, None, None, None, None, None, 0,
                                 None, None)
    assert rc == 1
    fake = ctypes.c_void_p(256)  # never dereferenced: d % 8 != 0 is rejected first
    rc = lib.twell_dense_ffn_bwd(fake, fake, fake, fake, fake, 64, 124, 512, 0.0, fake, fake, fake, fake, fake,
                                 1 << 20, fake, None)
    assert rc == 1
    assert lib.twell_dense_bwd_workspace_bytes(64, 124, 512) == 0
    assert lib.twell_dense_bwd_workspace_bytes(256, 128, 512) == 256 * 512 * 2 + 2 * 512 * 4
    assert lib.twell_set_kernel_timer(11, None, None) == 1  # no such call site
    rc = lib.twell_spmm_down_tc(None, None, 128, None, None, 0, None, None)
    assert rc == 1
    big = tw._TwellBuf(64, 65544, 16, 4, 0, fake, fake, fake, None, None)  # F above the union kernel's limit
    rc = lib.twell_spmm_down_tc(ctypes.byref(big), fake, 128, fake, fake, 1 << 20, fake, None)
    assert rc == 2  # TWELL_ERR_UNSUPPORTED
    assert lib.twell_wait_selftest(2, fake, fake, None) == 1  # no such wait
    assert lib.twell_wait_selftest(0, None, None, None) == 1


def test_ops_fail_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        tw.load_library(str(tmp_path / "missing.so"))
