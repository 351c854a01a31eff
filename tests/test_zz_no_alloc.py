"""The allocation-free forward, twell_ffn_fwd_static_ws, against twell_ffn_fwd.

Some callers of this library cannot allocate device memory: a plugin inside a
host framework that owns all GPU memory has no allocator to call, and a
latency-critical decode loop must not call cudaMalloc/cudaFree because they
synchronise the device. twell_ffn_fwd_static_ws serves them by running the
forward on a workspace array the library owns. These tests call it through the
C ABI and check that it gives what the regular entry point (with a
caller-allocated workspace) gives, on two calls in a row with different inputs,
since the shared array keeps the previous call's contents.

This file sorts last so that a run stopping at its first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import (assert_close_rms, assert_twell_identical, bf16_f64, dev_bf16, dev_f32, host_bf16_bits,
                     status_tensor, twell_to_host)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from activation_sparse_transformer_tcgen05_gb300 import build as _build
    _build.build()
import activation_sparse_transformer_tcgen05_gb300 as tw  # noqa: E402
from activation_sparse_transformer_tcgen05_gb300 import twell as tw_binding  # noqa: E402


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _regular(inp, cap):
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf = tw.TwellBuffers(M, F, T, cap)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    op = tw.OP_GATED_FWD if inp.W_gate is not None else tw.OP_FFN_FWD
    ws = torch.empty(tw.twell_workspace_bytes(op, M, d, F, T, cap), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), None if inp.W_gate is None else dev_bf16(inp.W_gate),
                     dev_f32(inp.b), dev_bf16(inp.W_down), T, buf, y, ws, st)
    assert tw.twell_check(st) == 0
    return twell_to_host(buf), bf16_f64(host_bf16_bits(y))


def _static(inp, cap):
    """One call of twell_ffn_fwd_static_ws straight through the C ABI (ctypes)."""
    lib = tw.load_library()
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf = tw.TwellBuffers(M, F, T, cap)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    x, Wu, Wd, b = dev_bf16(inp.x), dev_bf16(inp.W_up), dev_bf16(inp.W_down), dev_f32(inp.b)
    Wg = None if inp.W_gate is None else dev_bf16(inp.W_gate)
    rc = lib.twell_ffn_fwd_static_ws(_vp(x), _vp(Wu), _vp(Wg), _vp(b), _vp(Wd), M, d, F, T, buf.ref, _vp(y),
                                     _vp(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, tw.twell_status_string(rc)
    assert tw.twell_check(st) == 0
    return twell_to_host(buf), bf16_f64(host_bf16_bits(y))


@pytest.mark.parametrize("gated", [False, True])
def test_static_workspace_forward_matches_regular_twice(gated):
    shape = (8, 512, 2048, 8) if gated else (64, 256, 1024, 16)
    M, d, F, T = shape
    for seed in (11, 12):  # two calls in a row, different inputs
        inp = syn.ffn_inputs(M, d, F, T, -1.0, seed=seed, gated=gated)
        cap = M * F
        ref_tw, ref_y = _regular(inp, cap)
        got_tw, got_y = _static(inp, cap)
        assert_twell_identical(got_tw, ref_tw)
        assert_close_rms(got_y, ref_y, what="y", bf16_out=True)


def test_static_workspace_rejects_too_large_problem():
    lib = tw.load_library()
    M, d, F, T = 4096, 2048, 8192, 128  # needs ~134 MB of staging, more than the array
    assert tw.twell_workspace_bytes(tw.OP_FFN_FWD, M, d, F, T, M * F) > tw.STATIC_WS_BYTES
    buf = tw_binding._TwellBuf(M, F, T, (M + T - 1) // T, M * F, None, None, None, None, None)
    rc = lib.twell_ffn_fwd_static_ws(None, None, None, None, None, M, d, F, T, ctypes.byref(buf), None, None, None)
    assert rc == 3  # TWELL_ERR_WORKSPACE, nothing enqueued
