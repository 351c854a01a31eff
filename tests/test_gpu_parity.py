"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs. Bit-exact for the TwELL layout, 2e-2 * rms(ref) for
floating-point outputs; see tests/helpers.py for the rules."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from helpers import (assert_close_rms, assert_close_rms_plus, assert_twell_identical, bf16_f64, compare_hidden,
                     dev_bf16, dev_f32, host_bf16_bits, preact_tau, status_tensor, twell_to_device, twell_to_host)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from activation_sparse_transformer_tcgen05_gb300 import build as _build
    _build.build()
import activation_sparse_transformer_tcgen05_gb300 as tw  # noqa: E402


def _status_ok(st):
    code = tw.twell_check(st)
    assert code == 0, f"device status {code}: {tw.twell_status_string(code)}"


# ------------------------------------------------------------- twell_pack ---

@pytest.mark.parametrize("M,F,T,density,skew,seed", [
    (64, 512, 16, 0.01, 0.0, 0),       # tiny workload shape
    (129, 264, 16, 0.05, 0.0, 1),      # ragged last tile, F not a multiple of 256
    (37, 96, 1, 0.2, 0.0, 2),          # T = 1: per-row ELL
    (50, 128, 200, 0.1, 0.0, 3),       # T >= M: classic ELL
    (33, 64, 8, 1.0, 0.0, 4),          # everything active: K = F
    (40, 256, 16, 0.0, 0.0, 5),        # nothing active: K = 0, no slots
    (300, 1024, 128, 0.01, 1.0, 6),    # skewed row densities
])
def test_pack_bit_exact(M, F, T, density, skew, seed):
    h = syn.sparse_hidden(M, F, density, seed=seed, row_skew_sigma=skew)
    h[::5, ::7] = np.where(h[::5, ::7] == 0, np.uint16(0x8000), h[::5, ::7])  # -0.0 counts as zero
    ref = oracle.twell_pack(h, T)
    buf = tw.TwellBuffers(M, F, T, max(ref.slots, 1))
    st = status_tensor()
    tw.twell_pack(dev_bf16(h), T, buf, st)
    _status_ok(st)
    assert_twell_identical(twell_to_host(buf), ref)


def test_pack_full_inference_size():
    M, F, T = 4096, 8192, 128
    h = syn.sparse_hidden(M, F, 0.0099, seed=7)
    ref = oracle.twell_pack(h, T)
    buf = tw.TwellBuffers(M, F, T, ref.slots)
    st = status_tensor()
    tw.twell_pack(dev_bf16(h), T, buf, st)
    _status_ok(st)
    assert_twell_identical(twell_to_host(buf), ref)


def test_pack_capacity_overflow_reports_and_keeps_layout():
    M, F, T = 64, 512, 16
    h = syn.sparse_hidden(M, F, 0.05, seed=8)
    ref = oracle.twell_pack(h, T)
    buf = tw.TwellBuffers(M, F, T, ref.slots - 1)
    st = status_tensor()
    tw.twell_pack(dev_bf16(h), T, buf, st)
    assert tw.twell_check(st) == 4  # TWELL_ERR_CAPACITY
    np.testing.assert_array_equal(buf.nnz.cpu().numpy(), ref.nnz)
    np.testing.assert_array_equal(buf.K.cpu().numpy(), ref.K)
    np.testing.assert_array_equal(buf.off.cpu().numpy(), ref.off)


# ------------------------------------------------------------- spmm down ----

@pytest.mark.parametrize("M,F,d,T,density,seed", [
    (64, 512, 128, 16, 0.01, 0),
    (77, 264, 200, 8, 0.1, 1),     # ragged rows, d not a multiple of 256
    (300, 1024, 512, 128, 0.02, 2),
    (5, 64, 64, 1, 0.5, 3),
])
def test_spmm_down(M, F, d, T, density, seed):
    h = syn.sparse_hidden(M, F, density, seed=seed)
    W = syn.to_bf16_bits((syn.normal(seed, 9, F * d).reshape(F, d) / np.sqrt(F)).astype(np.float32))
    ref_tw = oracle.twell_pack(h, T)
    y_ref = oracle.twell_spmm(ref_tw, W)
    buf = twell_to_device(ref_tw)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    tw.twell_spmm_down(buf, dev_bf16(W), y, st)
    _status_ok(st)
    assert_close_rms(bf16_f64(host_bf16_bits(y)), y_ref, what="y", bf16_out=True)


def test_spmm_down_full_inference_size_sampled_rows():
    M, F, d, T = 4096, 8192, 2048, 128
    h = syn.sparse_hidden(M, F, 0.0099, seed=11)
    W = syn.to_bf16_bits((syn.normal(11, 9, F * d).reshape(F, d) / np.sqrt(F)).astype(np.float32))
    ref_tw = oracle.twell_pack(h, T)
    buf = twell_to_device(ref_tw)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    tw.twell_spmm_down(buf, dev_bf16(W), y, st)
    _status_ok(st)
    rows = np.r_[0:3, 127:130, M - 3:M, np.random.default_rng(0).integers(0, M, 40)]
    sub = oracle.Twell(len(rows), F, 1, *_rows_twell(ref_tw, rows))
    y_ref = oracle.twell_spmm(sub, W)
    assert_close_rms(bf16_f64(host_bf16_bits(y))[rows], y_ref, what="y rows", bf16_out=True)


def _rows_twell(tw_, rows):
    """Per-row (T = 1) TwELL of selected rows of a TwELL, for the oracle."""
    nnz, K, off, idx, val = [], [], [0], [], []
    for r in rows:
        t, i = divmod(int(r), tw_.T)
        base = tw_.off[t] + i * tw_.K[t]
        n = int(tw_.nnz[r])
        nnz.append(n)
        K.append(n)
        idx.extend(tw_.idx[base:base + n])
        val.extend(tw_.val[base:base + n])
        off.append(off[-1] + n)
    return (np.array(nnz, np.int32), np.array(K, np.int32), np.array(off, np.int64),
            np.array(idx, np.int32), np.array(val, np.uint16))


# ------------------------------------------------------- fused forward ------

def _fwd(inp: syn.FFNInputs, cap=None):
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    cap = cap if cap is not None else M * F
    buf = tw.TwellBuffers(M, F, T, cap)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    gated = inp.W_gate is not None
    op = tw.OP_GATED_FWD if gated else tw.OP_FFN_FWD
    ws = torch.empty(tw.twell_workspace_bytes(op, M, d, F, T, cap), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), None if not gated else dev_bf16(inp.W_gate),
                     dev_f32(inp.b), dev_bf16(inp.W_down), T, buf, y, ws, st)
    return buf, y, st


def test_fwd_integer_inputs_bit_exact():
    # integer-valued bf16 inputs: every fp32 partial sum is exact, so the TwELL
    # and y (one rounding of an exact integer) must match the oracle bit for bit
    inp = syn.integer_ffn_inputs(200, 128, 520, 16, seed=1, lo=-2, hi=2, bias=-9)
    buf, y, st = _fwd(inp)
    _status_ok(st)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, inp.M, inp.d, inp.F)
    assert ref["active"].mean() > 0.005
    assert_twell_identical(twell_to_host(buf), oracle.twell_pack(ref["h"], inp.T))
    np.testing.assert_array_equal(host_bf16_bits(y), oracle.round_bf16(ref["y"].astype(np.float32)))


@pytest.mark.parametrize("M,d,F,T,bias,seed", [
    (64, 128, 512, 16, -2.33, 0),      # the tiny workload
    (200, 256, 1024, 128, -1.0, 1),    # several tiles, ragged last row tile
    (130, 136, 264, 7, -0.5, 2),       # ragged K (d % 64 != 0), F % 256 != 0, odd T
    (712, 200, 800, 64, -1.2, 3),      # several 256 x 256 pair tiles each way, ragged in M, N and K
    (1100, 64, 2304, 16, -1.5, 4),     # more rows than the small-batch fill: one-launch layout and fill
    (2100, 64, 256, 1, -1.0, 5),       # more tiles than that launch holds: separate layout and fill
])
def test_fwd_relu_matches_oracle(M, d, F, T, bias, seed):
    inp = syn.ffn_inputs(M, d, F, T, bias, seed=seed)
    buf, y, st = _fwd(inp)
    _status_ok(st)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F)
    got = twell_to_host(buf)
    code, h_gpu = oracle.twell_unpack(got)
    assert code == 0, f"GPU TwELL violates the layout (code {code})"
    tau = preact_tau(inp.x, inp.W_up, ref["pre"])
    compare_hidden(h_gpu, ref["h"], h_gpu != 0, ref["active"] != 0, ref["pre"], tau)
    assert_close_rms(bf16_f64(host_bf16_bits(y)), ref["y"], what="y", bf16_out=True)


def test_fwd_inference_full_size_sampled():
    inp = syn.config_inputs("inference")
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf, y, st = _fwd(inp)
    _status_ok(st)
    got = twell_to_host(buf)
    code, h_gpu = oracle.twell_unpack(got)
    assert code == 0
    rows = np.r_[0:2, 127:129, M - 2:M, np.random.default_rng(1).integers(0, M, 26)].astype(np.int32)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, rows=rows)
    tau = preact_tau(inp.x[rows], inp.W_up, ref["pre"])
    compare_hidden(h_gpu[rows], ref["h"], h_gpu[rows] != 0, ref["active"] != 0, ref["pre"], tau)
    assert_close_rms(bf16_f64(host_bf16_bits(y))[rows], ref["y"], what="y rows", bf16_out=True)
    dens = got.nnz.sum() / (M * F)
    assert 0.007 < dens < 0.013  # ~99 % sparse


@pytest.mark.parametrize("name", ["decode1", "decode8", "decode64"])
def test_fwd_gated_decode(name):
    _check_gated(syn.config_inputs(name))


@pytest.mark.parametrize("M,d,F,T,seed", [
    (100, 256, 1024, 32, 4),     # two token chunks of the gate GEMM; layout+fill and slot-parallel up products
    (300, 264, 1032, 64, 5),     # more than 256 rows: row-parallel up products; ragged d, F and tiles
    (40, 136, 520, 40, 6),       # a decode batch with ragged d and F (one cooperative tail)
    (300, 4360, 520, 64, 7),     # d_model past 4096 with more than 256 rows: slot-parallel up products
    (1, 4360, 1040, 1, 8),       # ... and as a one-token decode (the tail loops over the columns)
])
def test_fwd_gated_beyond_decode(M, d, F, T, seed):
    _check_gated(syn.ffn_inputs(M, d, F, T, -1.5, seed=seed, gated=True))


def _check_gated(inp):
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf, y, st = _fwd(inp)
    _status_ok(st)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, inp.W_gate, inp.b, inp.W_down, M, d, F)
    got = twell_to_host(buf)
    # the stored set is the gate's support; values are h = bf16(relu(g) * u)
    act_gpu = np.zeros((M, F), bool)
    h_gpu = np.zeros((M, F), np.uint16)
    for r in range(M):
        t, i = divmod(r, T)
        base = got.off[t] + i * got.K[t]
        cols = got.idx[base:base + got.nnz[r]]
        assert np.all(np.diff(cols) > 0)
        act_gpu[r, cols] = True
        h_gpu[r, cols] = got.val[base:base + got.nnz[r]]
    tau = preact_tau(inp.x, inp.W_gate, ref["pre"])
    diff = act_gpu != (ref["active"] != 0)
    assert not (diff & (np.abs(ref["pre"]) > tau)).any()
    both = act_gpu & (ref["active"] != 0)
    assert_close_rms(bf16_f64(h_gpu)[both], bf16_f64(ref["h"])[both], what="gated h", bf16_out=True)
    assert_close_rms(bf16_f64(host_bf16_bits(y)), ref["y"], what="y", bf16_out=True)


def test_fwd_capacity_overflow():
    inp = syn.ffn_inputs(64, 128, 512, 16, -1.0, seed=3)
    buf, y, st = _fwd(inp, cap=8)
    assert tw.twell_check(st) == 4
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, 64, 128, 512)
    nnz = buf.nnz.cpu().numpy()
    assert abs(int(nnz.sum()) - int((ref["active"] != 0).sum())) <= 4


def test_fwd_workspace_too_small_is_rejected_on_host():
    inp = syn.ffn_inputs(64, 128, 512, 16, -2.33, seed=0)
    buf = tw.TwellBuffers(64, 512, 16, 64 * 512)
    y = torch.empty(64, 128, dtype=torch.int16, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(tw.TwellError) as e:
        tw.twell_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), None, dev_f32(inp.b), dev_bf16(inp.W_down), 16,
                         buf, y, ws, status_tensor())
    assert e.value.status == 3


# ------------------------------------------------------------- backward -----

def _bwd(x, W_up, W_down, ref_tw, dy, l1):
    M, d = x.shape
    F = W_up.shape[0]
    buf = twell_to_device(ref_tw)
    dx = torch.empty(M, d, dtype=torch.int16, device="cuda")
    dWu = torch.empty(F, d, dtype=torch.float32, device="cuda")
    dWd = torch.empty(F, d, dtype=torch.float32, device="cuda")
    db = torch.empty(F, dtype=torch.float32, device="cuda")
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_BWD, M, d, F, ref_tw.T, buf.cap_slots),
                     dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_ffn_bwd(dev_bf16(x), dev_bf16(W_up), dev_bf16(W_down), buf, dev_bf16(dy), l1, dx, dWu, dWd, db, ws, st)
    _status_ok(st)
    return bf16_f64(host_bf16_bits(dx)), dWu.cpu().numpy(), dWd.cpu().numpy(), db.cpu().numpy()


@pytest.mark.parametrize("M,d,F,T,bias,l1,seed", [
    (64, 128, 512, 16, -2.33, 1e-4, 0),
    (150, 264, 520, 32, -1.5, 0.0, 1),
    (90, 64, 1024, 128, -1.0, 5e-2, 2),
    (70, 8200, 264, 16, -1.5, 1e-3, 3),   # d_model past 8192: nine SDDMM slices, the last one ragged
])
def test_bwd_matches_oracle(M, d, F, T, bias, l1, seed):
    inp = syn.ffn_inputs(M, d, F, T, bias, seed=seed, with_dy=True)
    fw = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, want_y=False)
    ref_tw = oracle.twell_pack(fw["h"], T)
    dx, dWu, dWd, db = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, l1)
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, fw["h"], inp.dy))
    _, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1)
    assert_close_rms(dx, dx_ref, what="dx", bf16_out=True)
    assert_close_rms(dWu, gu, what="dW_up")
    assert_close_rms(dWd, gd, what="dW_down")
    assert_close_rms(db, gb, what="db")
    unused = np.flatnonzero((fw["h"] != 0).sum(0) == 0)
    assert np.all(dWu[unused] == 0) and np.all(dWd[unused] == 0) and np.all(db[unused] == 0)


def test_bwd_inference_size_sampled():
    M, d, F, T, l1 = 4096, 2048, 8192, 128, 1e-4
    h = syn.sparse_hidden(M, F, 0.0099, seed=21)
    inp = syn.ffn_inputs(M, d, F, T, -2.33, seed=21, with_dy=True)
    ref_tw = oracle.twell_pack(h, T)
    dx, dWu, dWd, db = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, l1)
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, h, inp.dy))
    rng = np.random.default_rng(5)
    rows = np.r_[0, M - 1, rng.integers(0, M, 14)].astype(np.int32)
    cols = np.r_[0, F - 1, rng.integers(0, F, 14)].astype(np.int32)
    _, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1, rows=rows)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1, cols=cols)
    assert_close_rms(dx[rows], dx_ref, what="dx rows", bf16_out=True)
    assert_close_rms(dWu[cols], gu, what="dW_up cols")
    assert_close_rms(dWd[cols], gd, what="dW_down cols")
    assert_close_rms(db[cols], gb, what="db cols")


def test_bwd_is_deterministic():
    inp = syn.ffn_inputs(128, 256, 512, 32, -1.5, seed=4, with_dy=True)
    fw = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, 128, 256, 512, want_y=False)
    ref_tw = oracle.twell_pack(fw["h"], 32)
    a = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, 1e-3)
    b = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, 1e-3)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_bwd_ragged_slices_groups_and_row_blocks():
    """d = 1288: two SDDMM slices of 1024 columns, the second ending 8 columns
    into its second 256-column chunk, and a last 512-column gather group of 264
    columns; M = 300: four 64-row column-list blocks and a ragged fifth;
    F = 776; tiles of 64 rows with a ragged last tile. Every output element
    against the oracle."""
    M, d, F, T, l1 = 300, 1288, 776, 64, 1e-3
    h = syn.sparse_hidden(M, F, 0.03, seed=31)
    inp = syn.ffn_inputs(M, d, F, T, -2.0, seed=31, with_dy=True)
    ref_tw = oracle.twell_pack(h, T)
    dx, dWu, dWd, db = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, l1)
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, h, inp.dy))
    _, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1)
    assert_close_rms(dx, dx_ref, what="dx", bf16_out=True)
    assert_close_rms(dWu, gu, what="dW_up")
    assert_close_rms(dWd, gd, what="dW_down")
    assert_close_rms(db, gb, what="db")


def test_bwd_of_an_empty_hidden_matrix_is_zero():
    """No active unit anywhere (K = 0 in every tile, no slots): dx, dW_up,
    dW_down and db are exactly zero, as the oracle's definition gives."""
    M, d, F, T = 130, 256, 512, 32
    h = syn.sparse_hidden(M, F, 0.0, seed=32)
    inp = syn.ffn_inputs(M, d, F, T, -2.0, seed=32, with_dy=True)
    ref_tw = oracle.twell_pack(h, T)
    assert ref_tw.slots == 0
    dx, dWu, dWd, db = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, 1e-2)
    for a in (dx, dWu, dWd, db):
        assert np.all(a == 0)


# ------------------------------------------------------ dense baseline ------

@pytest.mark.parametrize("M,d,F", [(64, 128, 512), (200, 264, 520), (520, 1032, 776)])
def test_dense_baseline_matches_oracle(M, d, F):
    inp = syn.ffn_inputs(M, d, F, 16, -1.0, seed=6)
    h = torch.empty(M, F, dtype=torch.int16, device="cuda")
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    tw.twell_dense_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), dev_f32(inp.b), dev_bf16(inp.W_down), h, y, st)
    _status_ok(st)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F)
    hg = host_bf16_bits(h)
    tau = preact_tau(inp.x, inp.W_up, ref["pre"])
    compare_hidden(hg, ref["h"], hg != 0, ref["active"] != 0, ref["pre"], tau)
    assert_close_rms(bf16_f64(host_bf16_bits(y)), ref["y"], what="dense y", bf16_out=True)


def test_dense_fwd_training_full_size_sampled():
    """The dense baseline's forward at the training workload's size (16384 x
    4096 x 16384, the shape the benchmark times it on): h and y on sampled
    rows against the oracle."""
    inp = syn.config_inputs("training")
    M, d, F = inp.M, inp.d, inp.F
    h = torch.empty(M, F, dtype=torch.int16, device="cuda")
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    st = status_tensor()
    tw.twell_dense_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), dev_f32(inp.b), dev_bf16(inp.W_down), h, y, st)
    _status_ok(st)
    rows = np.r_[0, 255, 256, M - 1, np.random.default_rng(4).integers(0, M, 8)].astype(np.int32)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, rows=rows)
    hg = host_bf16_bits(h)[rows]
    tau = preact_tau(inp.x[rows], inp.W_up, ref["pre"])
    compare_hidden(hg, ref["h"], hg != 0, ref["active"] != 0, ref["pre"], tau)
    assert_close_rms(bf16_f64(host_bf16_bits(y))[rows], ref["y"], what="dense y rows", bf16_out=True)


def _dense_bwd(x, W_up, W_down, h, dy, l1):
    M, d = x.shape
    F = W_up.shape[0]
    dx = torch.empty(M, d, dtype=torch.int16, device="cuda")
    dWu = torch.empty(F, d, dtype=torch.float32, device="cuda")
    dWd = torch.empty(F, d, dtype=torch.float32, device="cuda")
    db = torch.empty(F, dtype=torch.float32, device="cuda")
    ws = torch.empty(tw.twell_dense_bwd_workspace_bytes(M, d, F), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_dense_ffn_bwd(dev_bf16(x), dev_bf16(W_up), dev_bf16(W_down), dev_bf16(h), dev_bf16(dy), l1, dx, dWu,
                           dWd, db, ws, st)
    _status_ok(st)
    return bf16_f64(host_bf16_bits(dx)), dWu.cpu().numpy(), dWd.cpu().numpy(), db.cpu().numpy()


# The dense baseline keeps dpre in bf16 as a GEMM operand, as a bf16 training
# step does: each product dpre_rj * v then carries a relative error of at most
# 2^-9 (the bf16 rounding of dpre), so dx and dW_up may differ from the fp64
# oracle by up to 2^-9 * sum |dpre| |v| beyond the usual 2e-2 * rms (twice that
# is allowed). dW_down (h and dy are exact bf16 inputs) and db (summed from the
# fp32 values) take the plain bound.
DPRE_BF16 = 2.0 ** -8


@pytest.mark.parametrize("M,d,F,bias,l1,seed", [
    (64, 128, 512, -2.33, 1e-4, 0),    # tiny: one CTA pair, partial tiles
    (200, 264, 520, -1.0, 0.0, 1),     # ragged M, d, F (MN-major boxes past the edge)
    (520, 1032, 776, -1.5, 5e-2, 2),   # several 256-wide tiles each way, large l1
])
def test_dense_bwd_matches_oracle(M, d, F, bias, l1, seed):
    """The dense baseline's backward: same loss and gradients as the TwELL
    backward, with the oracle's h as the mask (no oracle input from the GPU)."""
    inp = syn.ffn_inputs(M, d, F, 16, bias, seed=seed, with_dy=True)
    fw = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, want_y=False)
    dx, dWu, dWd, db = _dense_bwd(inp.x, inp.W_up, inp.W_down, fw["h"], inp.dy, l1)
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, fw["h"], inp.dy))
    dpre, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1)
    assert_close_rms_plus(dx, dx_ref, DPRE_BF16 * (np.abs(dpre) @ np.abs(Wu)), what="dense dx", bf16_out=True)
    assert_close_rms_plus(dWu, gu, DPRE_BF16 * (np.abs(dpre).T @ np.abs(X)), what="dense dW_up")
    assert_close_rms(dWd, gd, what="dense dW_down")
    assert_close_rms(db, gb, what="dense db")
    unused = np.flatnonzero((fw["h"] != 0).sum(0) == 0)
    assert np.all(dWu[unused] == 0) and np.all(dWd[unused] == 0) and np.all(db[unused] == 0)


def test_dense_bwd_integer_inputs_exact():
    """Integer-valued dy, W_down, x, W_up and h with l1 = 0 and d_model = 16:
    |dpre| <= 16 * 4 * 4 = 256 is an integer bf16 holds exactly, and every sum
    of the four GEMMs is an integer below 2^24, so the fp32 results are exact
    and dx is exactly the bf16 rounding of the exact value."""
    M, d, F = 300, 16, 264
    inp = syn.integer_ffn_inputs(M, d, F, 16, seed=3, lo=-4, hi=4)
    dyi = syn.integer_ffn_inputs(M, d, F, 16, seed=4, lo=-4, hi=4).x
    h = syn.integer_ffn_inputs(M, F, F, 16, seed=5, lo=-2, hi=3).x  # [M, F] integers
    h = np.where(oracle.bf16_to_f64(h) > 0, h, 0).astype(np.uint16)
    dx, dWu, dWd, db = _dense_bwd(inp.x, inp.W_up, inp.W_down, h, dyi, 0.0)
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, h, dyi))
    dpre = (DY @ Wd.T) * (H != 0)
    assert np.abs(dpre).max() <= 256
    dx_exact = dpre @ Wu
    np.testing.assert_array_equal(dx, bf16_f64(oracle.round_bf16(dx_exact.astype(np.float32))))
    np.testing.assert_array_equal(dWu, dpre.T @ X)
    np.testing.assert_array_equal(dWd, H.T @ DY)
    np.testing.assert_array_equal(db, dpre.sum(0))


def test_dense_bwd_training_full_size_sampled():
    """The dense backward at the training workload's size (M=16384, d=4096,
    F=16384) on a 99 %-sparse h, sampled rows and columns against the oracle."""
    M, d, F, l1 = 16384, 4096, 16384, 1e-4
    h = syn.sparse_hidden(M, F, 0.0099, seed=31)
    inp = syn.ffn_inputs(M, d, F, 128, -2.33, seed=31, with_dy=True)
    dx, dWu, dWd, db = _dense_bwd(inp.x, inp.W_up, inp.W_down, h, inp.dy, l1)
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, h, inp.dy))
    rng = np.random.default_rng(7)
    rows = np.r_[0, M - 1, rng.integers(0, M, 10)].astype(np.int32)
    cols = np.r_[0, F - 1, rng.integers(0, F, 10)].astype(np.int32)
    dpre_rows, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1, rows=rows)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1, cols=cols)
    dpre_cols = (DY @ Wd[cols].T + l1) * (H[:, cols] != 0)  # [M, len(cols)], the bound's |dpre| only
    assert_close_rms_plus(dx[rows], dx_ref, DPRE_BF16 * (np.abs(dpre_rows) @ np.abs(Wu)), what="dense dx rows",
                          bf16_out=True)
    assert_close_rms_plus(dWu[cols], gu, DPRE_BF16 * (np.abs(dpre_cols).T @ np.abs(X)), what="dense dW_up cols")
    assert_close_rms(dWd[cols], gd, what="dense dW_down cols")
    assert_close_rms(db[cols], gb, what="dense db cols")


# ------------------------------------------- training and skewed workloads ---

def test_fwd_training_full_size_sampled():
    """The training workload's forward at full size (M=16384, d=4096, F=16384)."""
    inp = syn.config_inputs("training")
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf, y, st = _fwd(inp)
    _status_ok(st)
    got = twell_to_host(buf)
    rows = np.r_[0, 127, 128, M - 1, np.random.default_rng(2).integers(0, M, 12)].astype(np.int32)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, rows=rows)
    h_rows = np.zeros((len(rows), F), np.uint16)
    for i, r in enumerate(rows):
        t, ii = divmod(int(r), T)
        base = got.off[t] + ii * got.K[t]
        n = got.nnz[r]
        h_rows[i, got.idx[base:base + n]] = got.val[base:base + n]
        assert np.all(got.idx[base + n:base + got.K[t]] == -1)
    tau = preact_tau(inp.x[rows], inp.W_up, ref["pre"])
    compare_hidden(h_rows, ref["h"], h_rows != 0, ref["active"] != 0, ref["pre"], tau)
    assert_close_rms(bf16_f64(host_bf16_bits(y))[rows], ref["y"], what="y rows", bf16_out=True)
    assert got.K.tolist() == [int(got.nnz[t * T:(t + 1) * T].max()) for t in range(M // T)]
    assert 0.007 < got.nnz.sum() / (M * F) < 0.013


def test_bwd_training_full_size_sampled():
    """The training workload's backward at full size on a synthetic 99 %-sparse h."""
    M, d, F, T, l1 = 16384, 4096, 16384, 128, 1e-4
    h = syn.sparse_hidden(M, F, 0.0099, seed=31)
    inp = syn.ffn_inputs(M, d, F, T, -2.33, seed=31, with_dy=True)
    ref_tw = oracle.twell_pack(h, T)
    dx, dWu, dWd, db = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, l1)
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, h, inp.dy))
    rng = np.random.default_rng(6)
    rows = np.r_[0, M - 1, rng.integers(0, M, 10)].astype(np.int32)
    cols = np.r_[0, F - 1, rng.integers(0, F, 10)].astype(np.int32)
    _, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1, rows=rows)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1, cols=cols)
    assert_close_rms(dx[rows], dx_ref, what="dx rows", bf16_out=True)
    assert_close_rms(dWu[cols], gu, what="dW_up cols")
    assert_close_rms(dWd[cols], gd, what="dW_down cols")
    assert_close_rms(db[cols], gb, what="db cols")


@pytest.mark.parametrize("name", ["sweep90", "sweep99", "sweep999", "sweep90s", "sweep99s", "sweep999s"])
def test_fwd_skewed_rows(name):
    """Sweep workloads (d_model 4096, d_ff 16384, lognormal row scales on x) on
    1024 of their 8192 token rows: uneven rows stretch the tile widths."""
    c = syn.CONFIGS[name]
    M, d, F, T = 1024, c["d"], c["F"], c["T"]
    inp = syn.ffn_inputs(M, d, F, T, c["bias"], seed=0, row_skew_sigma=c["skew"])
    buf, y, st = _fwd(inp)
    _status_ok(st)
    got = twell_to_host(buf)
    code, _ = oracle.twell_unpack(oracle.Twell(M, F, T, got.nnz, got.K, got.off, got.idx, got.val))
    assert code == 0
    order = np.argsort(got.nnz)
    rows = np.r_[order[:2], order[-3:], np.random.default_rng(3).integers(0, M, 5)].astype(np.int32)
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, rows=rows)
    h_rows = np.zeros((len(rows), F), np.uint16)
    for i, r in enumerate(rows):
        t, ii = divmod(int(r), T)
        base = got.off[t] + ii * got.K[t]
        n = got.nnz[r]
        h_rows[i, got.idx[base:base + n]] = got.val[base:base + n]
    tau = preact_tau(inp.x[rows], inp.W_up, ref["pre"])
    compare_hidden(h_rows, ref["h"], h_rows != 0, ref["active"] != 0, ref["pre"], tau)
    assert_close_rms(bf16_f64(host_bf16_bits(y))[rows], ref["y"], what="y rows", bf16_out=True)
    # skew makes the widest row of a tile several times its mean
    assert got.K.max() > 2 * got.nnz.mean()


@pytest.mark.parametrize("name", ["sweep90s", "sweep99s", "sweep999s"])
def test_bwd_skewed_rows(name):
    """The backward on skewed rows at the sweep's skew-corrected biases (10 /
    1 / 0.1 % density; lognormal row scales), on 512 tokens, d_model 1024,
    d_ff 4096: some rows dense, most nearly empty, wide padded tiles."""
    c = syn.CONFIGS[name]
    M, d, F, T, l1 = 512, 1024, 4096, 128, 1e-4
    inp = syn.ffn_inputs(M, d, F, T, c["bias"], seed=8, with_dy=True, row_skew_sigma=c["skew"])
    fw = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, want_y=False)
    ref_tw = oracle.twell_pack(fw["h"], T)
    assert ref_tw.K.max() > 4 * max(ref_tw.nnz.mean(), 1.0)
    dx, dWu, dWd, db = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, l1)
    X, Wu, Wd, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, fw["h"], inp.dy))
    _, dx_ref = oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, l1)
    gu, gd, gb = oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, l1)
    assert_close_rms(dx, dx_ref, what="dx", bf16_out=True)
    assert_close_rms(dWu, gu, what="dW_up")
    assert_close_rms(dWd, gd, what="dW_down")
    assert_close_rms(db, gb, what="db")


def _fwd_with_stage_cap(inp, stage_cap):
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf = tw.TwellBuffers(M, F, T, M * F)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    ws = torch.empty(tw.twell_fwd_workspace_bytes(M, d, F, T, M * F, stage_cap), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_ffn_fwd(dev_bf16(inp.x), dev_bf16(inp.W_up), None, dev_f32(inp.b), dev_bf16(inp.W_down), T, buf, y,
                     ws, st)
    return buf, y, st


@pytest.mark.parametrize("M", [520, 100])  # CTA-pair GEMM; single-CTA GEMM
def test_fwd_small_staging_gives_the_same_twell(M):
    # ~1 % active: at most a handful of nonzeros per (row, 256-column block), so
    # a 32- or 64-entry staging segment never fills and the result is the full one's
    inp = syn.ffn_inputs(M, 256, 2056, 64, -2.33, seed=8)
    b256, y256, st256 = _fwd_with_stage_cap(inp, 256)
    _status_ok(st256)
    for cap in (64, 32):
        b, y, st = _fwd_with_stage_cap(inp, cap)
        _status_ok(st)
        assert_twell_identical(twell_to_host(b), twell_to_host(b256))
        np.testing.assert_array_equal(host_bf16_bits(y), host_bf16_bits(y256))


def test_fwd_staging_overflow_is_reported():
    # half the units active: ~128 per block, more than a 32-entry segment holds
    inp = syn.ffn_inputs(300, 128, 1024, 32, 0.0, seed=9)
    _, _, st = _fwd_with_stage_cap(inp, 32)
    assert tw.twell_check(st) == 4  # TWELL_ERR_CAPACITY


def _up_pack_then_down(inp):
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    buf = tw.TwellBuffers(M, F, T, M * F)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_FWD, M, d, F, T, M * F), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    tw.twell_up_pack(dev_bf16(inp.x), dev_bf16(inp.W_up), None, dev_f32(inp.b), T, buf, ws, st)
    tw.twell_spmm_down(buf, dev_bf16(inp.W_down), y, st)
    return buf, y, st


@pytest.mark.parametrize("M,d,F,T,bias,seed", [
    (520, 264, 776, 64, -1.5, 11),     # ragged rows, columns and blocks
    (260, 136, 2048, 32, 0.5, 12),     # ~70 % active: blocks of ~180 staged entries
    (1100, 64, 2304, 16, -2.33, 13),   # the one-launch layout and fill
])
def test_fwd_matches_up_pack_then_spmm_down(M, d, F, T, bias, seed):
    """The one-call forward and the two calls it is made of (up-projection
    with TwELL packing, then the TwELL down-projection) give the same TwELL
    and y, bit for bit."""
    inp = syn.ffn_inputs(M, d, F, T, bias, seed=seed)
    buf1, y1, st1 = _fwd(inp)
    _status_ok(st1)
    buf2, y2, st2 = _up_pack_then_down(inp)
    _status_ok(st2)
    assert_twell_identical(twell_to_host(buf1), twell_to_host(buf2))
    np.testing.assert_array_equal(host_bf16_bits(y1), host_bf16_bits(y2))
    ref = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F)
    assert_close_rms(bf16_f64(host_bf16_bits(y1)), ref["y"], what="y", bf16_out=True)


def test_fwd_replayed_from_a_cuda_graph_matches_eager():
    """The forward recorded in a CUDA graph (how a serving loop would issue
    it): replays give the eager TwELL and y bit for bit."""
    M, d, F, T = 300, 264, 520, 32
    inp = syn.ffn_inputs(M, d, F, T, -1.5, seed=14)
    buf_e, y_e, st_e = _fwd(inp)  # eager, also creates the side stream
    _status_ok(st_e)
    ref_tw, ref_y = twell_to_host(buf_e), host_bf16_bits(y_e)
    x, Wu, Wd, b = dev_bf16(inp.x), dev_bf16(inp.W_up), dev_bf16(inp.W_down), dev_f32(inp.b)
    buf = tw.TwellBuffers(M, F, T, M * F)
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_FWD, M, d, F, T, M * F), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tw.twell_ffn_fwd(x, Wu, None, b, Wd, T, buf, y, ws, st)
    for _ in range(2):
        y.zero_(), buf.idx.zero_(), buf.val.zero_()
        g.replay()
        _status_ok(st)
        assert_twell_identical(twell_to_host(buf), ref_tw)
        np.testing.assert_array_equal(host_bf16_bits(y), ref_y)


def test_fwd_and_bwd_from_two_threads_on_two_streams():
    """Two host threads, each on its own stream with its own buffers, run the
    forward and the backward (whose column-list kernels go to a side stream
    of the calling thread) at the same time: each gets what it gets alone."""
    import threading
    cases = [syn.ffn_inputs(300, 264, 520, 32, -1.5, seed=s, with_dy=True) for s in (21, 22)]

    def run(inp, stream):
        M, d, F, T = inp.M, inp.d, inp.F, inp.T
        with torch.cuda.stream(stream):
            buf = tw.TwellBuffers(M, F, T, M * F)
            y = torch.empty(M, d, dtype=torch.int16, device="cuda")
            wsf = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_FWD, M, d, F, T, M * F), dtype=torch.uint8,
                              device="cuda")
            wsb = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_BWD, M, d, F, T, M * F), dtype=torch.uint8,
                              device="cuda")
            dx = torch.empty(M, d, dtype=torch.int16, device="cuda")
            dWu = torch.empty(F, d, dtype=torch.float32, device="cuda")
            dWd = torch.empty(F, d, dtype=torch.float32, device="cuda")
            db = torch.empty(F, dtype=torch.float32, device="cuda")
            st = status_tensor()
            x, Wu, Wd, dy = dev_bf16(inp.x), dev_bf16(inp.W_up), dev_bf16(inp.W_down), dev_bf16(inp.dy)
            b = dev_f32(inp.b)
            for _ in range(3):
                tw.twell_ffn_fwd(x, Wu, None, b, Wd, T, buf, y, wsf, st)
                tw.twell_ffn_bwd(x, Wu, Wd, buf, dy, 1e-3, dx, dWu, dWd, db, wsb, st)
            stream.synchronize()
            return (tw.twell_check(st), host_bf16_bits(y), host_bf16_bits(dx), dWu.cpu().numpy(), dWd.cpu().numpy(),
                    db.cpu().numpy())

    alone = [run(c, torch.cuda.Stream()) for c in cases]
    out = [None, None]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    def worker(i):
        out[i] = run(cases[i], streams[i])

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for got, ref in zip(out, alone):
        assert got[0] == 0 and ref[0] == 0
        for u, v in zip(got[1:], ref[1:]):
            np.testing.assert_array_equal(u, v)


def test_bwd_replayed_from_a_cuda_graph_matches_eager():
    """The backward forks its index-only column-list kernels onto a side stream
    and joins them back by events; captured in a CUDA graph and replayed it must
    give the eager result bit for bit (and the oracle's within tolerance)."""
    M, d, F, T = 200, 264, 520, 32
    inp = syn.ffn_inputs(M, d, F, T, -1.5, seed=9, with_dy=True)
    fw = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, M, d, F, want_y=False)
    ref_tw = oracle.twell_pack(fw["h"], T)
    eager = _bwd(inp.x, inp.W_up, inp.W_down, ref_tw, inp.dy, 1e-3)  # also creates the side stream
    buf = twell_to_device(ref_tw)
    x, Wu, Wd, dy = dev_bf16(inp.x), dev_bf16(inp.W_up), dev_bf16(inp.W_down), dev_bf16(inp.dy)
    dx = torch.empty(M, d, dtype=torch.int16, device="cuda")
    dWu = torch.empty(F, d, dtype=torch.float32, device="cuda")
    dWd = torch.empty(F, d, dtype=torch.float32, device="cuda")
    db = torch.empty(F, dtype=torch.float32, device="cuda")
    ws = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_BWD, M, d, F, T, buf.cap_slots), dtype=torch.uint8,
                     device="cuda")
    st = status_tensor()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tw.twell_ffn_bwd(x, Wu, Wd, buf, dy, 1e-3, dx, dWu, dWd, db, ws, st)
    for _ in range(2):
        dx.zero_(), dWu.zero_(), dWd.zero_(), db.zero_()
        g.replay()
        _status_ok(st)
        got = (bf16_f64(host_bf16_bits(dx)), dWu.cpu().numpy(), dWd.cpu().numpy(), db.cpu().numpy())
        for u, v in zip(got, eager):
            np.testing.assert_array_equal(u, v)
    X, WU, WD, H, DY = (bf16_f64(a) for a in (inp.x, inp.W_up, inp.W_down, fw["h"], inp.dy))
    _, dx_ref = oracle.ffn_bwd_rows(X, WU, WD, H, DY, 1e-3)
    gu, gd, gb = oracle.ffn_bwd_cols(X, WU, WD, H, DY, 1e-3)
    assert_close_rms(got[0], dx_ref, what="dx", bf16_out=True)
    assert_close_rms(got[1], gu, what="dW_up")
    assert_close_rms(got[2], gd, what="dW_down")
    assert_close_rms(got[3], gb, what="db")
