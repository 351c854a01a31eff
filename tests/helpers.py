"""Shared helpers of the GPU parity tests: moving seeded inputs to the device,
reading a device TwELL back, and the comparison rules.

Comparison rules:
  * integer and layout work (TwELL nnz, K, offsets, idx, val of twell_pack):
    bit-exact;
  * floating-point outputs (y, dx, dW_up, dW_down, db, gated h values):
    max |gpu - ref| <= 2e-2 * rms(ref), bf16 inputs with fp32 accumulation
    against the fp64 oracle. Outputs stored in bf16 (y, dx, gated h) are
    compared with the oracle value rounded to bf16, and each element may also
    differ by one bf16 ulp of itself: the fp32 and fp64 sums can round to
    neighbouring bf16 values, and on heavy-tailed rows that single rounding
    step exceeds 2e-2 * rms;
  * the hidden active set of the fused forward, where fp32 accumulation order
    decides a ReLU sign: an entry may differ from the oracle only where
    |pre_oracle| <= tau, tau = 2 * (gamma_d * sum_k |x_k w_k| + ulp32(pre)),
    gamma_d = d u / (1 - d u), u = 2^-24 (the forward error bound of a
    d-term fp32 dot product, doubled); where both are active the bf16 values
    differ by at most one bf16 ulp plus tau.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

RMS_TOL = 2e-2

# Every floating-point comparison's margins, for the summary the test session
# prints at its end (tests/conftest.py): (test, output, plain max|err| / rms,
# max|err| beyond the allowance / rms, tolerance).
MARGINS: list[tuple[str, str, float, float, float]] = []


def _record(what: str, plain: float, beyond: float, rms: float, tol: float):
    import os
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    if rms > 0:
        MARGINS.append((test, what, plain / rms, beyond / rms, tol))


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint16)


def bf16_f64(bits: np.ndarray) -> np.ndarray:
    return oracle.bf16_to_f64(bits)


def status_tensor() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def twell_to_host(buf) -> oracle.Twell:
    """Reads a device TwELL (TwellBuffers) into the oracle's container."""
    torch.cuda.synchronize()
    off = buf.off.cpu().numpy().astype(np.int64)
    n = int(off[-1])
    return oracle.Twell(buf.M, buf.F, buf.T, buf.nnz.cpu().numpy().astype(np.int32),
                        buf.K.cpu().numpy().astype(np.int32), off,
                        buf.idx[:n].cpu().numpy().astype(np.int32),
                        buf.val[:n].cpu().numpy().view(np.uint16).copy())


def twell_to_device(tw: oracle.Twell, cap: int | None = None):
    """Uploads an oracle TwELL into fresh TwellBuffers (capacity >= its slots)."""
    from activation_sparse_transformer_tcgen05_gb300 import TwellBuffers
    cap = tw.slots if cap is None else cap
    b = TwellBuffers(tw.M, tw.F, tw.T, max(cap, 1))
    b.nnz.copy_(torch.from_numpy(tw.nnz.astype(np.int32)))
    b.K.copy_(torch.from_numpy(tw.K.astype(np.int32)))
    b.off.copy_(torch.from_numpy(tw.off.astype(np.int64)))
    if tw.slots:
        b.idx[:tw.slots].copy_(torch.from_numpy(tw.idx.astype(np.int32)))
        b.val[:tw.slots].copy_(torch.from_numpy(tw.val.view(np.int16)))
    return b


def assert_twell_identical(got: oracle.Twell, ref: oracle.Twell):
    np.testing.assert_array_equal(got.nnz, ref.nnz, err_msg="nnz")
    np.testing.assert_array_equal(got.K, ref.K, err_msg="K")
    np.testing.assert_array_equal(got.off, ref.off, err_msg="off")
    np.testing.assert_array_equal(got.idx, ref.idx, err_msg="idx")
    np.testing.assert_array_equal(got.val, ref.val, err_msg="val")


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (np.maximum(e, -126) - 7), 2.0 ** -133)


def assert_close_rms(got: np.ndarray, ref: np.ndarray, tol: float = RMS_TOL, what: str = "",
                     bf16_out: bool = False):
    """max|got - ref| <= tol * rms(ref); for bf16-stored outputs ref is rounded
    to bf16 and one bf16 ulp of the element is allowed on top."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if not ref.size:
        return 0.0, 0.0
    plain = float(np.max(np.abs(got - ref)))
    if bf16_out:
        ref_q = oracle.bf16_to_f64(oracle.round_bf16(ref.astype(np.float32)))
        excess = np.abs(got - ref_q) - bf16_ulp(ref_q)
        err = float(np.max(excess))
    else:
        err = plain
    _record(what, plain, err, rms, tol)
    assert err <= tol * rms + 1e-30, f"{what}: max|err| {err:.3e} > {tol} * rms {rms:.3e}"
    return err, rms


def assert_close_rms_plus(got: np.ndarray, ref: np.ndarray, bound: np.ndarray, tol: float = RMS_TOL,
                          what: str = "", bf16_out: bool = False):
    """assert_close_rms with a per-element allowance `bound` on top: used where
    an operand is rounded to bf16 by design (the dense baseline's dpre), with
    bound = that rounding's worst-case effect on the element."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if not ref.size:
        return 0.0, 0.0
    plain = float(np.max(np.abs(got - ref)))
    if bf16_out:
        ref_q = oracle.bf16_to_f64(oracle.round_bf16(ref.astype(np.float32)))
        err = float(np.max(np.abs(got - ref_q) - bf16_ulp(ref_q) - bound))
    else:
        err = float(np.max(np.abs(got - ref) - bound))
    _record(what, plain, err, rms, tol)
    assert err <= tol * rms + 1e-30, f"{what}: max|err| - bound {err:.3e} > {tol} * rms {rms:.3e}"
    return err, rms


def preact_tau(x_bits: np.ndarray, W_bits: np.ndarray, pre: np.ndarray) -> np.ndarray:
    """Per-entry bound tau on |fp32 pre-activation - oracle| (see module doc)."""
    d = x_bits.shape[1]
    u = 2.0 ** -24
    gamma = d * u / (1 - d * u)
    mag = np.abs(bf16_f64(x_bits)) @ np.abs(bf16_f64(W_bits)).T
    ulp = np.spacing(np.abs(pre).astype(np.float32)).astype(np.float64)
    return 2.0 * (gamma * mag + ulp)


def compare_hidden(h_gpu_bits: np.ndarray, h_ref_bits: np.ndarray, active_gpu: np.ndarray,
                   active_ref: np.ndarray, pre_ref: np.ndarray, tau: np.ndarray):
    """Active-set and value agreement of a fused forward; returns mismatch count."""
    diff = active_gpu != active_ref
    bad = diff & (np.abs(pre_ref) > tau)
    assert not bad.any(), (f"{int(bad.sum())} active-set mismatches outside the fp32 error band, "
                           f"first at {np.argwhere(bad)[0].tolist()}")
    both = active_gpu & active_ref
    hg = bf16_f64(h_gpu_bits)[both]
    hr = bf16_f64(h_ref_bits)[both]
    assert np.all(np.abs(hg - hr) <= 2.0 ** -7 * np.abs(hr) + tau[both]), "hidden values beyond 1 bf16 ulp"
    return int(diff.sum())
