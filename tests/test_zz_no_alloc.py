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


def _static_call(lib, inp, buf, y, st, dev):
    """One call of twell_ffn_fwd_static_ws straight through the C ABI (ctypes)."""
    x, Wu, Wg, b, Wd = dev
    return lib.twell_ffn_fwd_static_ws(_vp(x), _vp(Wu), _vp(Wg), _vp(b), _vp(Wd), inp.M, inp.d, inp.F, inp.T,
                                       buf.ref, _vp(y), _vp(st),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _static(inp, cap):
    lib = tw.load_library()
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf = tw.TwellBuffers(M, F, T, cap)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    dev = (dev_bf16(inp.x), dev_bf16(inp.W_up), None if inp.W_gate is None else dev_bf16(inp.W_gate),
           dev_f32(inp.b), dev_bf16(inp.W_down))
    rc = _static_call(lib, inp, buf, y, st, dev)
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


def test_static_workspace_inference_layer_with_small_staging():
    # 4096 x 2048 x 8192 at ~99 % sparsity: only the 32-entry staging (~17 MB)
    # fits the array; the regular call gets the full 256-entry staging
    inp = syn.config_inputs("inference")
    cap = inp.M * 256
    ref_tw, ref_y = _regular(inp, cap)
    got_tw, got_y = _static(inp, cap)
    assert_twell_identical(got_tw, ref_tw)
    assert_close_rms(got_y, ref_y, what="y", bf16_out=True)


def test_static_workspace_allocates_nothing():
    lib = tw.load_library()
    inp = syn.ffn_inputs(64, 256, 1024, 16, -1.0, seed=13)
    buf = tw.TwellBuffers(inp.M, inp.F, inp.T, inp.M * inp.F)
    y = torch.empty(inp.M, inp.d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    dev = (dev_bf16(inp.x), dev_bf16(inp.W_up), None, dev_f32(inp.b), dev_bf16(inp.W_down))
    assert _static_call(lib, inp, buf, y, st, dev) == 0  # warm-up: first call on this device
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    launches0 = tw.twell_kernel_launches()
    for _ in range(3):
        assert _static_call(lib, inp, buf, y, st, dev) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert tw.twell_check(st) == 0
    assert tw.twell_kernel_launches() > launches0, "the forward's kernels did not run"
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"


def test_static_workspace_rejects_too_large_problem():
    lib = tw.load_library()
    M, d, F, T = 16384, 4096, 16384, 128  # even the 32-entry staging needs ~134 MB
    assert tw.twell_fwd_workspace_bytes(M, d, F, T, M * F, 32) > tw.STATIC_WS_BYTES
    buf = tw_binding._TwellBuf(M, F, T, (M + T - 1) // T, M * F, None, None, None, None, None)
    rc = lib.twell_ffn_fwd_static_ws(None, None, None, None, None, M, d, F, T, ctypes.byref(buf), None, None, None)
    assert rc == 3  # TWELL_ERR_WORKSPACE, nothing enqueued
