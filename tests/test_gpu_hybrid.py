"""GPU parity of the hybrid ELL + dense-overflow format ("Sparser, Faster,
Lighter Transformer Language Models", Resumo Técnico §2, "Formato Híbrido para
Treinamento"): rows with more than C nonzeros leave the TwELL for a dense block
and their down-projection runs on the tensor cores. Checked through the C ABI
against the oracle's split (oracle.hybrid_pack) and dense forward."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from helpers import (assert_close_rms, assert_twell_identical, bf16_f64, compare_hidden, dev_bf16, dev_f32,
                     host_bf16_bits, preact_tau, status_tensor, twell_to_host)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from activation_sparse_transformer_tcgen05_gb300 import build as _build
    _build.build()
import activation_sparse_transformer_tcgen05_gb300 as tw  # noqa: E402


def _hybrid(inp, C, cap_rows, cap=None):
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf = tw.TwellBuffers(M, F, T, cap if cap is not None else M * F)
    ov = tw.TwellOverflow(F, C, cap_rows)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_HYBRID_FWD, M, d, F, T, 0), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_hybrid_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), dev_f32(inp.b), dev_bf16(inp.W_down),
                            dev_bf16(np.ascontiguousarray(inp.W_down.T)), T, buf, ov, y, ws, st)
    return buf, ov, y, st


def _overflow_to_host(ov, F):
    torch.cuda.synchronize()
    n = int(ov.n_rows.item())
    rows = ov.rows[:n].cpu().numpy().astype(np.int32)
    dense = ov.dense[:n * F].cpu().numpy().view(np.uint16).reshape(n, F)
    return rows, dense


def test_hybrid_integer_inputs_bit_exact():
    # integer-valued inputs: every fp32 sum is exact, so the split, both parts
    # and y (the TwELL rows by the gather, the overflow rows by the dense GEMM)
    # must match the oracle bit for bit
    inp = syn.integer_ffn_inputs(200, 128, 520, 16, seed=1, lo=-2, hi=2, bias=-9)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, inp.M, inp.d, inp.F)
    counts = ((ref["h"] & 0x7FFF) != 0).sum(1)
    C = int(np.median(counts))
    buf, ov, y, st = _hybrid(inp, C, cap_rows=inp.M)
    assert tw.twell_check(st) == 0
    tw_ref, rows_ref, dense_ref = oracle.hybrid_pack(ref["h"], inp.T, C)
    assert 0 < len(rows_ref) < inp.M
    assert_twell_identical(twell_to_host(buf), tw_ref)
    rows, dense = _overflow_to_host(ov, inp.F)
    np.testing.assert_array_equal(rows, rows_ref)
    np.testing.assert_array_equal(dense, dense_ref)
    np.testing.assert_array_equal(host_bf16_bits(y), oracle.round_bf16(ref["y"].astype(np.float32)))


@pytest.mark.parametrize("M,d,F,T,C,seed", [
    (300, 256, 1024, 32, 60, 2),     # several pair tiles of overflow rows, ragged
    (90, 136, 264, 7, 12, 3),        # fewer overflow rows than one GEMM tile, odd T, ragged K
])
def test_hybrid_skewed_rows_match_oracle(M, d, F, T, C, seed):
    inp = syn.ffn_inputs(M, d, F, T, -1.2816, seed=seed, row_skew_sigma=1.0)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F)
    buf, ov, y, st = _hybrid(inp, C, cap_rows=M)
    assert tw.twell_check(st) == 0
    got = twell_to_host(buf)
    code, h_gpu = oracle.twell_unpack(got)
    assert code == 0
    rows, dense = _overflow_to_host(ov, F)
    assert len(rows) > 0
    # the split is the one the format defines, on the GPU's own h
    assert (np.diff(rows) > 0).all()
    assert (got.nnz[rows] == 0).all() and (got.K <= C).all()
    h_gpu[rows] = dense
    counts = ((h_gpu & 0x7FFF) != 0).sum(1)
    np.testing.assert_array_equal(np.flatnonzero(counts > C), rows)
    # and its h agrees with the oracle's up to the fp32 band
    tau = preact_tau(inp.x, inp.W_up, ref["pre"])
    compare_hidden(h_gpu, ref["h"], h_gpu != 0, ref["active"] != 0, ref["pre"], tau)
    assert_close_rms(bf16_f64(host_bf16_bits(y)), ref["y"], what="y", bf16_out=True)


def test_hybrid_overflow_capacity_reported():
    inp = syn.ffn_inputs(120, 128, 512, 16, -1.0, seed=4, row_skew_sigma=1.0)
    buf, ov, y, st = _hybrid(inp, 5, cap_rows=3)
    assert tw.twell_check(st) == 4  # TWELL_ERR_CAPACITY
    assert int(ov.n_rows.item()) == 3


def test_hybrid_without_overflow_is_the_twell_forward():
    inp = syn.ffn_inputs(200, 256, 1024, 128, -1.0, seed=5)
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf, ov, y, st = _hybrid(inp, F, cap_rows=0)
    assert tw.twell_check(st) == 0 and int(ov.n_rows.item()) == 0
    buf2 = tw.TwellBuffers(M, F, T, M * F)
    y2 = torch.empty(M, d, dtype=torch.int16, device="cuda")
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_FWD, M, d, F, T, M * F), dtype=torch.uint8, device="cuda")
    st2 = status_tensor()
    tw.twell_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), None, dev_f32(inp.b), dev_bf16(inp.W_down), T, buf2, y2,
                     ws, st2)
    assert tw.twell_check(st2) == 0
    assert_twell_identical(twell_to_host(buf), twell_to_host(buf2))
    np.testing.assert_array_equal(host_bf16_bits(y), host_bf16_bits(y2))


@pytest.mark.parametrize("name", ["sweep90", "sweep90s", "sweep99s", "sweep999s"])
def test_hybrid_sweep_full_size_sampled_rows(name):
    """The skewed sweep workloads at full size (8192 x 4096 x 16384; nominal
    90 % and the skew-corrected 90 / 99 / 99.9 % biases) in the configuration
    the benchmark times (C = 1.25 % of d_ff, room for every row): y and h on
    sampled overflow and TwELL rows against the oracle."""
    inp = syn.config_inputs(name)
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    C = round(0.0125 * F)
    buf, ov, y, st = _hybrid(inp, C, cap_rows=M, cap=M * C)
    assert tw.twell_check(st) == 0
    got = twell_to_host(buf)
    rows_ov, dense = _overflow_to_host(ov, F)
    assert 0 < len(rows_ov) < M
    in_ell = np.setdiff1d(np.arange(M), rows_ov)
    rng = np.random.default_rng(7)
    pick = np.r_[rng.choice(rows_ov, 5, replace=False), rng.choice(in_ell, 5, replace=False)].astype(np.int32)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, rows=pick)
    pos = {int(r): i for i, r in enumerate(rows_ov)}
    h_rows = np.zeros((len(pick), F), np.uint16)
    for i, r in enumerate(pick):
        if int(r) in pos:
            h_rows[i] = dense[pos[int(r)]]
        else:
            t, ii = divmod(int(r), T)
            base = got.off[t] + ii * got.K[t]
            n = got.nnz[r]
            h_rows[i, got.idx[base:base + n]] = got.val[base:base + n]
    tau = preact_tau(inp.x[pick], inp.W_up, ref["pre"])
    compare_hidden(h_rows, ref["h"], h_rows != 0, ref["active"] != 0, ref["pre"], tau)
    y_rows = host_bf16_bits(y)[pick]
    assert_close_rms(bf16_f64(y_rows), ref["y"], what="y", bf16_out=True)


# ------------------------------------------------------------------ backward --

def _hybrid_bwd(inp, h_bits, C, cap_rows, l1):
    """The hybrid backward on the oracle's own split of h (uploaded), through the C ABI."""
    from helpers import twell_to_device
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    tw_ref, rows, dense = oracle.hybrid_pack(h_bits, T, C)
    buf = twell_to_device(tw_ref)
    ov = tw.TwellOverflow(F, C, cap_rows)
    n = len(rows)
    ov.n_rows.fill_(n)
    if n:
        ov.rows[:n].copy_(torch.from_numpy(rows.astype(np.int32)))
        ov.dense[:n * F].copy_(torch.from_numpy(np.ascontiguousarray(dense).view(np.int16).reshape(-1)))
    dx = torch.empty(M, d, dtype=torch.int16, device="cuda")
    dWu = torch.empty(F, d, dtype=torch.float32, device="cuda")
    dWd = torch.empty(F, d, dtype=torch.float32, device="cuda")
    db = torch.empty(F, dtype=torch.float32, device="cuda")
    ws = torch.empty(tw.twell_hybrid_bwd_workspace_bytes(M, d, F, T, buf.cap_slots, cap_rows), dtype=torch.uint8,
                     device="cuda")
    st = status_tensor()
    tw.twell_hybrid_ffn_bwd(dev_bf16(inp.x), dev_bf16(inp.W_up), dev_bf16(inp.W_down),
                            dev_bf16(np.ascontiguousarray(inp.W_up.T)), buf, ov, dev_bf16(inp.dy), l1, dx, dWu, dWd,
                            db, ws, st)
    assert tw.twell_check(st) == 0
    return n, bf16_f64(host_bf16_bits(dx)), dWu.cpu().numpy(), dWd.cpu().numpy(), db.cpu().numpy()


@pytest.mark.parametrize("M,d,F,T,C,cap_extra,l1,seed,bias", [
    (300, 256, 1024, 32, 60, 0, 1e-3, 2, -1.2816),   # several pair tiles of overflow rows; skewed 14 % density
    (90, 136, 264, 7, 12, 40, 0.0, 3, -1.2816),      # ragged d and F, room for more rows than overflow
    (200, 128, 520, 16, 300, 8, 5e-2, 4, -1.2816),   # nothing overflows: the sparse backward alone
    (300, 256, 1024, 32, 30, 0, 1e-3, 5, -7.8373),   # skew-corrected 99 %: few dense rows, most empty
    (600, 256, 1024, 64, 12, 0, 1e-3, 6, -20.2430),  # skew-corrected 99.9 %
])
def test_hybrid_backward_matches_oracle(M, d, F, T, C, cap_extra, l1, seed, bias):
    # the hybrid format is another storage of the same h: the gradients are
    # the plain backward's, compared with the oracle's on the full h
    inp = syn.ffn_inputs(M, d, F, T, bias, seed=seed, with_dy=True, row_skew_sigma=1.0)
    fw = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, want_y=False)
    counts = ((fw["h"] & 0x7FFF) != 0).sum(1)
    cap_rows = int((counts > C).sum()) + cap_extra
    n, dx, dWu, dWd, db = _hybrid_bwd(inp, fw["h"], C, cap_rows, l1)
    assert (n > 0) == (C < counts.max())
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, fw["h"], inp.dy))
    _, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1)
    assert_close_rms(dx, dx_ref, what="dx", bf16_out=True)
    assert_close_rms(dWu, gu, what="dW_up")
    assert_close_rms(dWd, gd, what="dW_down")
    assert_close_rms(db, gb, what="db")


def test_hybrid_backward_is_deterministic():
    inp = syn.ffn_inputs(160, 128, 512, 32, -1.2816, seed=6, with_dy=True, row_skew_sigma=1.0)
    fw = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, inp.M, inp.d, inp.F, want_y=False)
    a = _hybrid_bwd(inp, fw["h"], 40, inp.M, 1e-3)
    b = _hybrid_bwd(inp, fw["h"], 40, inp.M, 1e-3)
    assert a[0] > 0
    for u, v in zip(a[1:], b[1:]):
        np.testing.assert_array_equal(u, v)


@pytest.mark.parametrize("density", [0.0103, 0.0012])
def test_hybrid_backward_full_size_sampled(density):
    """The hybrid backward at the sweep workloads' full size (8192 x 4096 x
    16384) in the configuration the benchmark times (C = 1.25 % of d_ff, room
    for every row), on a synthetic h whose row densities are 1.03 % or 0.12 %
    scaled by LogNormal(0, 1) (3471 and 89 overflow rows): dx on sampled rows
    (overflow and TwELL rows) and dW_up, dW_down, db on sampled columns against
    the oracle on the full h."""
    M, d, F, T, l1 = 8192, 4096, 16384, 128, 1e-4
    C = round(0.0125 * F)
    h = syn.sparse_hidden(M, F, density, seed=41, row_skew_sigma=1.0)
    inp = syn.ffn_inputs(M, d, F, T, -2.33, seed=41, with_dy=True)
    n, dx, dWu, dWd, db = _hybrid_bwd(inp, h, C, M, l1)
    counts = ((h & 0x7FFF) != 0).sum(1)
    rows_ov = np.flatnonzero(counts > C)
    assert n == len(rows_ov) and 0 < n < M
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, h, inp.dy))
    rng = np.random.default_rng(9)
    in_ell = np.setdiff1d(np.arange(M), rows_ov)
    rows = np.r_[rng.choice(rows_ov, min(4, n), replace=False), rng.choice(in_ell, 6, replace=False)].astype(np.int32)
    cols = np.r_[0, F - 1, rng.integers(0, F, 10)].astype(np.int32)
    _, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1, rows=rows)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1, cols=cols)
    assert_close_rms(dx[rows], dx_ref, what="dx rows", bf16_out=True)
    assert_close_rms(dWu[cols], gu, what="dW_up cols")
    assert_close_rms(dWd[cols], gd, what="dW_down cols")
    assert_close_rms(db[cols], gb, what="db cols")
