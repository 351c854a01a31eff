"""GPU parity of twell_spmm_down_tc, the tensor-core down-projection over
128-token group unions, against the CPU oracle's y = h W_down (2e-2 * rms(ref),
bf16 output). Shapes cover: d below and above one 256-column block, ragged
groups, F not a multiple of the 64-deep k-block, T not dividing the group,
buckets larger than the staged part (global fallback), empty and full h, and
the largest d_ff the kernel takes."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from helpers import assert_close_rms, bf16_f64, dev_bf16, host_bf16_bits, status_tensor, twell_to_device

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from activation_sparse_transformer_tcgen05_gb300 import build as _build
    _build.build()
import activation_sparse_transformer_tcgen05_gb300 as tw  # noqa: E402
from test_gpu_canaries import Guarded  # noqa: E402


def _weights(F, d, seed):
    return syn.to_bf16_bits((syn.normal(seed, 9, F * d).reshape(F, d) / np.sqrt(F)).astype(np.float32))


def _run_tc(buf, W, M, d, guard=False):
    ws = torch.empty(tw.twell_spmm_down_tc_workspace_bytes(M, buf.F, buf.cap_slots), dtype=torch.uint8,
                     device="cuda")
    g = Guarded(M * d, torch.int16) if guard else None
    y = g.t.view(M, d) if guard else torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    tw.twell_spmm_down_tc(buf, dev_bf16(W), y, ws, st)
    code = tw.twell_check(st)
    assert code == 0, f"device status {code}: {tw.twell_status_string(code)}"
    if guard:
        assert g.intact(), "twell_spmm_down_tc wrote outside y"
    return host_bf16_bits(y)


@pytest.mark.parametrize("M,F,d,T,density,seed", [
    (64, 512, 128, 16, 0.01, 0),      # tiny workload shape; 128-column tile
    (77, 264, 200, 8, 0.1, 1),        # one ragged group; F % 64 != 0; d < 256
    (300, 1024, 512, 128, 0.02, 2),   # three groups, ragged last
    (5, 64, 64, 1, 0.5, 3),           # T = 1
    (260, 520, 264, 100, 0.3, 4),     # T does not divide 128; buckets beyond the staged 1024 words
    (200, 4096, 256, 128, 0.9, 5),    # nearly dense: U = F, large buckets
    (40, 256, 128, 16, 0.0, 6),       # nothing active: y = 0
    (33, 64, 72, 8, 1.0, 7),          # everything active
    (130, 65536, 128, 64, 0.002, 8),  # the largest d_ff (shared memory of both tile shapes at their limit)
    (130, 65536, 264, 64, 0.002, 9),
])
def test_spmm_down_tc_matches_oracle(M, F, d, T, density, seed):
    h = syn.sparse_hidden(M, F, density, seed=seed)
    W = _weights(F, d, seed)
    ref_tw = oracle.twell_pack(h, T)
    y_ref = oracle.twell_spmm(ref_tw, W)
    buf = twell_to_device(ref_tw)
    y = _run_tc(buf, W, M, d, guard=True)
    if density == 0.0:
        assert not y.any()
    assert_close_rms(bf16_f64(y), y_ref, what="y", bf16_out=True)


def test_spmm_down_tc_skewed_rows():
    M, F, d, T = 384, 2048, 384, 128
    h = syn.sparse_hidden(M, F, 0.03, seed=12, row_skew_sigma=1.0)
    W = _weights(F, d, 12)
    ref_tw = oracle.twell_pack(h, T)
    y = _run_tc(twell_to_device(ref_tw), W, M, d)
    assert_close_rms(bf16_f64(y), oracle.twell_spmm(ref_tw, W), what="y", bf16_out=True)


def test_spmm_down_tc_full_inference_size_sampled_rows():
    M, F, d, T = 4096, 8192, 2048, 128
    h = syn.sparse_hidden(M, F, 0.0099, seed=11)
    W = _weights(F, d, 11)
    ref_tw = oracle.twell_pack(h, T)
    y = _run_tc(twell_to_device(ref_tw), W, M, d)
    rows = np.r_[0:3, 127:130, M - 3:M, np.random.default_rng(0).integers(0, M, 40)]
    from test_gpu_parity import _rows_twell
    sub = oracle.Twell(len(rows), F, 1, *_rows_twell(ref_tw, rows))
    assert_close_rms(bf16_f64(y)[rows], oracle.twell_spmm(sub, W), what="y rows", bf16_out=True)


def test_spmm_down_tc_is_deterministic_and_agrees_with_row_gather():
    M, F, d, T = 520, 2048, 512, 64
    h = syn.sparse_hidden(M, F, 0.02, seed=13)
    W = _weights(F, d, 13)
    buf = twell_to_device(oracle.twell_pack(h, T))
    y1 = _run_tc(buf, W, M, d)
    y2 = _run_tc(buf, W, M, d)
    np.testing.assert_array_equal(y1, y2)
    y_rows = torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    tw.twell_spmm_down(buf, dev_bf16(W), y_rows, st)
    assert tw.twell_check(st) == 0
    # both sum the same fp32 products; only the order differs
    assert_close_rms(bf16_f64(y1), bf16_f64(host_bf16_bits(y_rows)), what="tc vs rows", bf16_out=True)


def test_spmm_down_tc_rejects_small_workspace_on_host():
    M, F, d, T = 64, 512, 128, 16
    h = syn.sparse_hidden(M, F, 0.05, seed=14)
    buf = twell_to_device(oracle.twell_pack(h, T))
    need = tw.twell_spmm_down_tc_workspace_bytes(M, F, buf.cap_slots)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    with pytest.raises(tw.TwellError) as e:
        tw.twell_spmm_down_tc(buf, dev_bf16(_weights(F, d, 14)), y, ws, st)
    assert e.value.status == 3  # TWELL_ERR_WORKSPACE
