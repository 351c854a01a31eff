"""The library's bounded waits, made to run out on purpose: a wait that
nothing will complete (an mbarrier no thread arrives on; the decode tail's grid
barrier with a target the grid cannot reach) gives up after its limit and
reports TWELL_ERR_TIMEOUT through the status word, and the CUDA context stays
usable for the next call. No fault, trap or endless loop is involved."""
import time

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from helpers import assert_twell_identical, dev_bf16, dev_f32, status_tensor, twell_to_host

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from activation_sparse_transformer_tcgen05_gb300 import build as _build
    _build.build()
import activation_sparse_transformer_tcgen05_gb300 as tw  # noqa: E402


@pytest.mark.parametrize("which", [0, 1])
def test_wait_runs_out_and_reports_timeout(which):
    st = status_tensor()
    scratch = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    tw.twell_wait_selftest(which, scratch, st)
    code = tw.twell_check(st)
    waited = time.time() - t0
    assert code == 5, tw.twell_status_string(code)  # TWELL_ERR_TIMEOUT
    assert 0.5 < waited < 30.0
    # the context is intact: a forward right after it gives the oracle's TwELL
    inp = syn.integer_ffn_inputs(64, 128, 512, 16, seed=1, lo=-2, hi=2, bias=-9)
    buf = tw.TwellBuffers(inp.M, inp.F, inp.T, inp.M * inp.F)
    y = torch.empty(inp.M, inp.d, dtype=torch.int16, device="cuda")
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_FWD, inp.M, inp.d, inp.F, inp.T, inp.M * inp.F),
                     dtype=torch.uint8, device="cuda")
    st2 = status_tensor()
    tw.twell_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), None, dev_f32(inp.b), dev_bf16(inp.W_down), inp.T, buf, y,
                     ws, st2)
    assert tw.twell_check(st2) == 0
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, inp.M, inp.d, inp.F)
    assert_twell_identical(twell_to_host(buf), oracle.twell_pack(ref["h"], inp.T))
