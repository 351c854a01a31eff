"""Guard canaries around every buffer an entry point writes (compute-sanitizer
is not available here): each output is a slice of a larger tensor whose guard
regions before and after are filled with a pattern, and the pattern must
survive the call. Ragged sizes, so that partial tiles and tails are exercised."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from helpers import dev_bf16, dev_f32, status_tensor

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from activation_sparse_transformer_tcgen05_gb300 import build as _build
    _build.build()
import activation_sparse_transformer_tcgen05_gb300 as tw  # noqa: E402
from activation_sparse_transformer_tcgen05_gb300 import twell as twb  # noqa: E402

GUARD = 4096  # bytes on each side


class Guarded:
    """A device tensor of `n` elements of `dtype` inside a byte buffer with guard bytes on both sides."""

    def __init__(self, n, dtype):
        esz = torch.empty(0, dtype=dtype).element_size()
        self.raw = torch.full((2 * GUARD + max(n, 1) * esz,), 0xA5, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n * esz].view(dtype)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return bool((self.raw[:GUARD] == 0xA5).all()) and bool((self.raw[-GUARD:] == 0xA5).all())


class GuardedTwell:
    """TwELL buffers whose every array is guarded (same C struct as TwellBuffers)."""

    def __init__(self, M, F, T, cap):
        self.M, self.F, self.T = M, F, T
        self.n_tiles = (M + T - 1) // T
        self.cap_slots = cap
        self.parts = [Guarded(M, torch.int32), Guarded(self.n_tiles, torch.int32),
                      Guarded(self.n_tiles + 1, torch.int64), Guarded(cap, torch.int32), Guarded(cap, torch.int16)]
        self.nnz, self.K, self.off, self.idx, self.val = (p.t for p in self.parts)
        self.struct = twb._TwellBuf(M, F, T, self.n_tiles, cap, *(p.t.data_ptr() for p in self.parts))

    @property
    def ref(self):
        return ctypes.byref(self.struct)

    def intact(self):
        return all(p.intact() for p in self.parts)


def _guarded_like(shape, dtype):
    return Guarded(int(np.prod(shape)), dtype)


@pytest.mark.parametrize("gated", [False, True])
def test_forward_and_backward_stay_inside_their_buffers(gated):
    M, d, F, T = (200, 136, 520, 48) if not gated else (24, 136, 520, 24)
    inp = syn.ffn_inputs(M, d, F, T, -1.0, seed=7, gated=gated, with_dy=True)
    cap = M * F
    buf = GuardedTwell(M, F, T, cap)
    y = _guarded_like((M, d), torch.int16)
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_GATED_FWD if gated else tw.OP_FFN_FWD, M, d, F, T, cap),
                     dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), dev_bf16(inp.W_gate) if gated else None, dev_f32(inp.b),
                     dev_bf16(inp.W_down), T, buf, y.t.view(M, d), ws, st)
    assert tw.twell_check(st) == 0
    assert buf.intact() and y.intact()
    if gated:
        return
    dx = _guarded_like((M, d), torch.int16)
    dWu, dWd = _guarded_like((F, d), torch.float32), _guarded_like((F, d), torch.float32)
    db = Guarded(F, torch.float32)
    wsb = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_BWD, M, d, F, T, cap), dtype=torch.uint8, device="cuda")
    tw.twell_ffn_bwd(dev_bf16(inp.x), dev_bf16(inp.W_up), dev_bf16(inp.W_down), buf, dev_bf16(inp.dy), 1e-3,
                     dx.t.view(M, d), dWu.t.view(F, d), dWd.t.view(F, d), db.t, wsb, st)
    assert tw.twell_check(st) == 0
    assert dx.intact() and dWu.intact() and dWd.intact() and db.intact() and buf.intact()


def test_pack_stays_inside_its_buffers():
    M, F, T = 130, 264, 7
    h = syn.sparse_hidden(M, F, 0.05, seed=9)
    buf = GuardedTwell(M, F, T, M * F)
    st = status_tensor()
    tw.twell_pack(dev_bf16(h).view(M, F), T, buf, st)
    assert tw.twell_check(st) == 0 and buf.intact()
    y = _guarded_like((M, 136), torch.int16)
    W = syn.ffn_inputs(M, 136, F, T, -1.0, seed=9).W_down
    tw.twell_spmm_down(buf, dev_bf16(W), y.t.view(M, 136), st)
    assert tw.twell_check(st) == 0 and y.intact()


def test_hybrid_stays_inside_its_buffers():
    M, d, F, T, C = 150, 136, 520, 16, 40
    inp = syn.ffn_inputs(M, d, F, T, -1.2816, seed=8, row_skew_sigma=1.0, with_dy=True)
    buf = GuardedTwell(M, F, T, M * C)
    cap_rows = M
    n_rows, rows, dense = Guarded(1, torch.int32), Guarded(cap_rows, torch.int32), Guarded(cap_rows * F, torch.int16)
    ov = tw.TwellOverflow(F, C, cap_rows)  # for its struct type; arrays replaced by guarded ones
    ov.struct = twb._TwellOverflow(C, cap_rows, n_rows.t.data_ptr(), rows.t.data_ptr(), dense.t.data_ptr())
    y = _guarded_like((M, d), torch.int16)
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_HYBRID_FWD, M, d, F, T, 0), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_hybrid_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), dev_f32(inp.b), dev_bf16(inp.W_down),
                            dev_bf16(np.ascontiguousarray(inp.W_down.T)), T, buf, ov, y.t.view(M, d), ws, st)
    assert tw.twell_check(st) == 0
    assert int(n_rows.t.item()) > 0
    assert buf.intact() and y.intact() and n_rows.intact() and rows.intact() and dense.intact()
    dx = _guarded_like((M, d), torch.int16)
    dWu, dWd = _guarded_like((F, d), torch.float32), _guarded_like((F, d), torch.float32)
    db = Guarded(F, torch.float32)
    wsb = torch.empty(tw.twell_hybrid_bwd_workspace_bytes(M, d, F, T, M * C, cap_rows), dtype=torch.uint8,
                      device="cuda")
    tw.twell_hybrid_ffn_bwd(dev_bf16(inp.x), dev_bf16(inp.W_up), dev_bf16(inp.W_down),
                            dev_bf16(np.ascontiguousarray(inp.W_up.T)), buf, ov, dev_bf16(inp.dy), 1e-3,
                            dx.t.view(M, d), dWu.t.view(F, d), dWd.t.view(F, d), db.t, wsb, st)
    assert tw.twell_check(st) == 0
    assert dx.intact() and dWu.intact() and dWd.intact() and db.intact() and dense.intact() and buf.intact()
