"""ctypes binding of libtwell.so (see include/twell.h for the contract).

Argument marshalling only: torch tensors are checked for device, dtype,
contiguity and size, their device pointers and the current CUDA stream are
passed to the C entry point of the same name, and a nonzero return code
raises TwellError. Every step of the computation runs in the library's CUDA
kernels; if the library is missing this module raises instead of computing
anything itself.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libtwell.so")

OP_PACK, OP_SPMM_DOWN, OP_FFN_FWD, OP_FFN_BWD, OP_GATED_FWD, OP_HYBRID_FWD = 0, 1, 2, 3, 4, 5

# Every symbol include/twell.h declares.
EXPORTED_SYMBOLS = (
    "twell_status_string", "twell_buf_slots_bound", "twell_workspace_bytes", "twell_device_sm_count",
    "twell_pack", "twell_up_pack", "twell_spmm_down", "twell_ffn_fwd", "twell_ffn_bwd",
    "twell_dense_ffn_fwd", "twell_dense_ffn_bwd", "twell_dense_bwd_workspace_bytes", "twell_kernel_launches", "twell_check", "twell_ffn_fwd_static_ws",
    "twell_set_kernel_timer", "twell_hybrid_up_pack", "twell_hybrid_spmm_down",
    "twell_hybrid_ffn_fwd", "twell_fwd_workspace_bytes", "twell_hybrid_bwd_workspace_bytes", "twell_hybrid_ffn_bwd",
    "twell_wait_selftest", "twell_spmm_down_tc_workspace_bytes", "twell_spmm_down_tc",
)

# Call sites of twell_set_kernel_timer.
(SITE_NONE, SITE_UP_GEMM, SITE_SPMM_DOWN, SITE_SDDMM, SITE_DX, SITE_CSC, SITE_WGRAD, SITE_DECODE_TAIL,
 SITE_OVERFLOW_GEMM, SITE_SPMM_UNION, SITE_UNION_BUILD) = range(11)

# Size of the library-owned workspace behind twell_ffn_fwd_static_ws.
STATIC_WS_BYTES = 32 * 1024 * 1024


class TwellError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {twell_status_string(status)} (status {status})")


class _TwellBuf(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int32), ("F", ctypes.c_int32), ("T", ctypes.c_int32),
                ("n_tiles", ctypes.c_int32), ("cap_slots", ctypes.c_int64),
                ("nnz_row", ctypes.c_void_p), ("K_tile", ctypes.c_void_p), ("tile_off", ctypes.c_void_p),
                ("idx", ctypes.c_void_p), ("val", ctypes.c_void_p)]


class _TwellOverflow(ctypes.Structure):
    _fields_ = [("C", ctypes.c_int32), ("cap_rows", ctypes.c_int32), ("n_rows", ctypes.c_void_p),
                ("rows", ctypes.c_void_p), ("dense", ctypes.c_void_p)]


_lib = None
P, I32, I64, SZ, F32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
BUFP = ctypes.POINTER(_TwellBuf)
OVP = ctypes.POINTER(_TwellOverflow)


def load_library(path: str | None = None):
    """Loads libtwell.so once. Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libtwell.so not found at {path}: build it first "
                           "(python -m activation_sparse_transformer_tcgen05_gb300.build)")
    lib = ctypes.CDLL(path)
    lib.twell_status_string.restype = ctypes.c_char_p
    lib.twell_status_string.argtypes = [I32]
    lib.twell_buf_slots_bound.restype = I64
    lib.twell_buf_slots_bound.argtypes = [I32, I32, I32]
    lib.twell_workspace_bytes.restype = SZ
    lib.twell_workspace_bytes.argtypes = [I32, I32, I32, I32, I32, I64]
    lib.twell_fwd_workspace_bytes.restype = SZ
    lib.twell_fwd_workspace_bytes.argtypes = [I32, I32, I32, I32, I64, I32]
    lib.twell_device_sm_count.restype = I32
    lib.twell_pack.restype = I32
    lib.twell_pack.argtypes = [P, I32, I32, I32, I32, BUFP, P, P]
    lib.twell_up_pack.restype = I32
    lib.twell_up_pack.argtypes = [P, P, P, P, I32, I32, I32, I32, BUFP, P, SZ, P, P]
    lib.twell_kernel_launches.restype = I64
    lib.twell_set_kernel_timer.restype = I32
    lib.twell_set_kernel_timer.argtypes = [I32, P, P]
    lib.twell_spmm_down.restype = I32
    lib.twell_spmm_down.argtypes = [BUFP, P, I32, P, P, P]
    lib.twell_spmm_down_tc_workspace_bytes.restype = SZ
    lib.twell_spmm_down_tc_workspace_bytes.argtypes = [I32, I32, I64]
    lib.twell_spmm_down_tc.restype = I32
    lib.twell_spmm_down_tc.argtypes = [BUFP, P, I32, P, P, SZ, P, P]
    lib.twell_ffn_fwd.restype = I32
    lib.twell_ffn_fwd.argtypes = [P, P, P, P, P, I32, I32, I32, I32, BUFP, P, P, SZ, P, P]
    lib.twell_ffn_bwd.restype = I32
    lib.twell_ffn_bwd.argtypes = [P, P, P, BUFP, P, I32, F32, P, P, P, P, P, SZ, P, P]
    lib.twell_dense_ffn_fwd.restype = I32
    lib.twell_dense_ffn_fwd.argtypes = [P, P, P, P, I32, I32, I32, P, P, P, P]
    lib.twell_dense_bwd_workspace_bytes.restype = SZ
    lib.twell_dense_bwd_workspace_bytes.argtypes = [I32, I32, I32]
    lib.twell_dense_ffn_bwd.restype = I32
    lib.twell_dense_ffn_bwd.argtypes = [P, P, P, P, P, I32, I32, I32, F32, P, P, P, P, P, SZ, P, P]
    lib.twell_ffn_fwd_static_ws.restype = I32
    lib.twell_ffn_fwd_static_ws.argtypes = [P, P, P, P, P, I32, I32, I32, I32, BUFP, P, P, P]
    lib.twell_hybrid_up_pack.restype = I32
    lib.twell_hybrid_up_pack.argtypes = [P, P, P, I32, I32, I32, I32, BUFP, OVP, P, SZ, P, P]
    lib.twell_hybrid_spmm_down.restype = I32
    lib.twell_hybrid_spmm_down.argtypes = [BUFP, OVP, P, P, I32, P, P, P]
    lib.twell_hybrid_ffn_fwd.restype = I32
    lib.twell_hybrid_ffn_fwd.argtypes = [P, P, P, P, P, I32, I32, I32, I32, BUFP, OVP, P, P, SZ, P, P]
    lib.twell_hybrid_bwd_workspace_bytes.restype = SZ
    lib.twell_hybrid_bwd_workspace_bytes.argtypes = [I32, I32, I32, I32, I64, I32]
    lib.twell_hybrid_ffn_bwd.restype = I32
    lib.twell_hybrid_ffn_bwd.argtypes = [P, P, P, P, BUFP, OVP, P, I32, F32, P, P, P, P, P, SZ, P, P]
    lib.twell_wait_selftest.restype = I32
    lib.twell_wait_selftest.argtypes = [I32, P, P, P]
    lib.twell_check.restype = I32
    lib.twell_check.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    _lib = lib
    return lib


def twell_status_string(status: int) -> str:
    return load_library().twell_status_string(int(status)).decode()


def twell_buf_slots_bound(M: int, F: int, T: int) -> int:
    return int(load_library().twell_buf_slots_bound(M, F, T))


def twell_workspace_bytes(op: int, M: int, d: int, F: int, T: int, cap_slots: int = 0) -> int:
    return int(load_library().twell_workspace_bytes(op, M, d, F, T, cap_slots))


def twell_fwd_workspace_bytes(M: int, d: int, F: int, T: int, cap_slots: int, stage_cap: int) -> int:
    """ReLU-forward workspace whose epilogue staging holds stage_cap entries per (row, 256-column block)."""
    return int(load_library().twell_fwd_workspace_bytes(M, d, F, T, cap_slots, stage_cap))


def twell_device_sm_count() -> int:
    return int(load_library().twell_device_sm_count())


# ------------------------------------------------------------- marshalling --

def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None, name: str, *, bytes_per_elem: int | None = None, numel: int | None = None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if bytes_per_elem is not None and t.element_size() != bytes_per_elem:
        raise ValueError(f"{name} must have {bytes_per_elem}-byte elements, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


def _check(status: int, where: str):
    if status != 0:
        raise TwellError(status, where)


class TwellBuffers:
    """Device arrays of one TwELL (allocated by torch) and the C struct describing them."""

    def __init__(self, M: int, F: int, T: int, cap_slots: int, device="cuda"):
        self.M, self.F, self.T = M, F, T
        self.n_tiles = (M + T - 1) // T
        self.cap_slots = int(cap_slots)
        self.nnz = torch.empty(M, dtype=torch.int32, device=device)
        self.K = torch.empty(self.n_tiles, dtype=torch.int32, device=device)
        self.off = torch.empty(self.n_tiles + 1, dtype=torch.int64, device=device)
        n = max(self.cap_slots, 1)
        self.idx = torch.empty(n, dtype=torch.int32, device=device)
        self.val = torch.empty(n, dtype=torch.int16, device=device)  # bf16 bit patterns
        self.struct = _TwellBuf(M, F, T, self.n_tiles, self.cap_slots, self.nnz.data_ptr(),
                                self.K.data_ptr(), self.off.data_ptr(), self.idx.data_ptr(),
                                self.val.data_ptr())

    @property
    def ref(self):
        return ctypes.byref(self.struct)

    def slots(self) -> int:
        """Total slot count (reads tile_off[n_tiles] back; synchronises)."""
        return int(self.off[-1].item())


class TwellOverflow:
    """Dense overflow block of the hybrid format (allocated by torch) and its C struct:
    rows with more than C nonzeros, at most cap_rows of them, each as a full hidden row."""

    def __init__(self, F: int, C: int, cap_rows: int, device="cuda"):
        self.F, self.C, self.cap_rows = F, int(C), int(cap_rows)
        self.n_rows = torch.zeros(1, dtype=torch.int32, device=device)
        self.rows = torch.empty(max(self.cap_rows, 1), dtype=torch.int32, device=device)
        self.dense = torch.empty(max(self.cap_rows, 1) * F, dtype=torch.int16, device=device)  # bf16 bits
        self.struct = _TwellOverflow(self.C, self.cap_rows, self.n_rows.data_ptr(), self.rows.data_ptr(),
                                     self.dense.data_ptr())

    @property
    def ref(self):
        return ctypes.byref(self.struct)


def twell_pack(h: torch.Tensor, T: int, out: TwellBuffers, status: torch.Tensor, stream=None):
    M, F = h.shape
    if not h.is_cuda or h.element_size() != 2 or h.stride(1) != 1:
        raise ValueError("h must be a CUDA bf16/int16 matrix with unit column stride")
    _check(load_library().twell_pack(ctypes.c_void_p(h.data_ptr()), M, F, h.stride(0), T, out.ref,
                                     _ptr(status, "status", bytes_per_elem=4), _stream(stream)),
           "twell_pack")


def twell_kernel_launches() -> int:
    return int(load_library().twell_kernel_launches())


def twell_set_kernel_timer(site: int, ev_begin=None, ev_end=None):
    """Record the torch.cuda.Events ev_begin / ev_end around the kernel at `site`
    (SITE_*) on every launch until reset with site = SITE_NONE. The events must
    have been recorded once before (torch creates them lazily)."""
    b = ctypes.c_void_p(ev_begin.cuda_event) if ev_begin is not None else None
    e = ctypes.c_void_p(ev_end.cuda_event) if ev_end is not None else None
    _check(load_library().twell_set_kernel_timer(int(site), b, e), "twell_set_kernel_timer")


def twell_wait_selftest(which: int, scratch, status, stream=None):
    """A bounded wait that runs out (about 1 s) and reports TWELL_ERR_TIMEOUT in status."""
    _check(load_library().twell_wait_selftest(int(which), _ptr(scratch, "scratch", bytes_per_elem=4, numel=1),
                                              _ptr(status, "status", bytes_per_elem=4), _stream(stream)),
           "twell_wait_selftest")


def twell_up_pack(x, W_up, W_gate, b, T: int, h_out: TwellBuffers, ws, status, stream=None):
    M, d = x.shape
    F = W_up.shape[0]
    _check(load_library().twell_up_pack(
        _ptr(x, "x", bytes_per_elem=2), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(W_gate, "W_gate", bytes_per_elem=2, numel=F * d), _ptr(b, "b", bytes_per_elem=4, numel=F),
        M, d, F, T, h_out.ref, _ptr(ws, "ws"), ws.numel() * ws.element_size(),
        _ptr(status, "status", bytes_per_elem=4), _stream(stream)), "twell_up_pack")


def twell_spmm_down(h: TwellBuffers, W_down: torch.Tensor, y: torch.Tensor, status: torch.Tensor, stream=None):
    d = W_down.shape[1]
    _check(load_library().twell_spmm_down(h.ref, _ptr(W_down, "W_down", bytes_per_elem=2, numel=h.F * d), d,
                                          _ptr(y, "y", bytes_per_elem=2, numel=h.M * d),
                                          _ptr(status, "status", bytes_per_elem=4), _stream(stream)),
           "twell_spmm_down")


def twell_spmm_down_tc_workspace_bytes(M: int, F: int, cap_slots: int) -> int:
    return int(load_library().twell_spmm_down_tc_workspace_bytes(M, F, cap_slots))


def twell_spmm_down_tc(h: TwellBuffers, W_down: torch.Tensor, y: torch.Tensor, ws: torch.Tensor,
                       status: torch.Tensor, stream=None):
    """y = h W_down on the tensor cores over each 128-token group's union of active units."""
    d = W_down.shape[1]
    _check(load_library().twell_spmm_down_tc(h.ref, _ptr(W_down, "W_down", bytes_per_elem=2, numel=h.F * d), d,
                                             _ptr(y, "y", bytes_per_elem=2, numel=h.M * d), _ptr(ws, "ws"),
                                             ws.numel() * ws.element_size(),
                                             _ptr(status, "status", bytes_per_elem=4), _stream(stream)),
           "twell_spmm_down_tc")


def twell_ffn_fwd(x, W_up, W_gate, b, W_down, T: int, h_out: TwellBuffers, y, ws, status, stream=None):
    M, d = x.shape
    F = W_up.shape[0]
    _check(load_library().twell_ffn_fwd(
        _ptr(x, "x", bytes_per_elem=2), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(W_gate, "W_gate", bytes_per_elem=2, numel=F * d), _ptr(b, "b", bytes_per_elem=4, numel=F),
        _ptr(W_down, "W_down", bytes_per_elem=2, numel=F * d), M, d, F, T, h_out.ref,
        _ptr(y, "y", bytes_per_elem=2, numel=M * d), _ptr(ws, "ws"), ws.numel() * ws.element_size(),
        _ptr(status, "status", bytes_per_elem=4), _stream(stream)), "twell_ffn_fwd")


def twell_hybrid_up_pack(x, W_up, b, T: int, h_out: TwellBuffers, ov: TwellOverflow, ws, status, stream=None):
    M, d = x.shape
    F = W_up.shape[0]
    _check(load_library().twell_hybrid_up_pack(
        _ptr(x, "x", bytes_per_elem=2), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(b, "b", bytes_per_elem=4, numel=F), M, d, F, T, h_out.ref, ov.ref, _ptr(ws, "ws"),
        ws.numel() * ws.element_size(), _ptr(status, "status", bytes_per_elem=4), _stream(stream)),
        "twell_hybrid_up_pack")


def twell_hybrid_spmm_down(h: TwellBuffers, ov: TwellOverflow, W_down, W_downT, y, status, stream=None):
    d = W_down.shape[1]
    _check(load_library().twell_hybrid_spmm_down(
        h.ref, ov.ref, _ptr(W_down, "W_down", bytes_per_elem=2, numel=h.F * d),
        _ptr(W_downT, "W_downT", bytes_per_elem=2, numel=h.F * d), d,
        _ptr(y, "y", bytes_per_elem=2, numel=h.M * d), _ptr(status, "status", bytes_per_elem=4), _stream(stream)),
        "twell_hybrid_spmm_down")


def twell_hybrid_ffn_fwd(x, W_up, b, W_down, W_downT, T: int, h_out: TwellBuffers, ov: TwellOverflow, y, ws,
                         status, stream=None):
    M, d = x.shape
    F = W_up.shape[0]
    _check(load_library().twell_hybrid_ffn_fwd(
        _ptr(x, "x", bytes_per_elem=2), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(b, "b", bytes_per_elem=4, numel=F), _ptr(W_down, "W_down", bytes_per_elem=2, numel=F * d),
        _ptr(W_downT, "W_downT", bytes_per_elem=2, numel=F * d), M, d, F, T, h_out.ref, ov.ref,
        _ptr(y, "y", bytes_per_elem=2, numel=M * d), _ptr(ws, "ws"), ws.numel() * ws.element_size(),
        _ptr(status, "status", bytes_per_elem=4), _stream(stream)), "twell_hybrid_ffn_fwd")


def twell_hybrid_bwd_workspace_bytes(M: int, d: int, F: int, T: int, cap_slots: int, cap_rows: int) -> int:
    return int(load_library().twell_hybrid_bwd_workspace_bytes(M, d, F, T, cap_slots, cap_rows))


def twell_hybrid_ffn_bwd(x, W_up, W_down, W_upT, h: TwellBuffers, ov: TwellOverflow, dy, l1: float, dx, dW_up,
                         dW_down, db, ws, status, stream=None):
    M, d = x.shape
    F = h.F
    _check(load_library().twell_hybrid_ffn_bwd(
        _ptr(x, "x", bytes_per_elem=2, numel=M * d), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(W_down, "W_down", bytes_per_elem=2, numel=F * d), _ptr(W_upT, "W_upT", bytes_per_elem=2, numel=F * d),
        h.ref, ov.ref, _ptr(dy, "dy", bytes_per_elem=2, numel=M * d), d, float(l1),
        _ptr(dx, "dx", bytes_per_elem=2, numel=M * d), _ptr(dW_up, "dW_up", bytes_per_elem=4, numel=F * d),
        _ptr(dW_down, "dW_down", bytes_per_elem=4, numel=F * d), _ptr(db, "db", bytes_per_elem=4, numel=F),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _ptr(status, "status", bytes_per_elem=4), _stream(stream)),
        "twell_hybrid_ffn_bwd")


def twell_ffn_fwd_static_ws(x, W_up, W_gate, b, W_down, T: int, h_out: TwellBuffers, y, status, stream=None):
    """twell_ffn_fwd on the library-owned static workspace (no allocation)."""
    M, d = x.shape
    F = W_up.shape[0]
    _check(load_library().twell_ffn_fwd_static_ws(
        _ptr(x, "x", bytes_per_elem=2), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(W_gate, "W_gate", bytes_per_elem=2, numel=F * d), _ptr(b, "b", bytes_per_elem=4, numel=F),
        _ptr(W_down, "W_down", bytes_per_elem=2, numel=F * d), M, d, F, T, h_out.ref,
        _ptr(y, "y", bytes_per_elem=2, numel=M * d), _ptr(status, "status", bytes_per_elem=4),
        _stream(stream)), "twell_ffn_fwd_static_ws")


def twell_ffn_bwd(x, W_up, W_down, h: TwellBuffers, dy, l1: float, dx, dW_up, dW_down, db, ws, status,
                  stream=None):
    M, d = x.shape
    F = W_up.shape[0]
    _check(load_library().twell_ffn_bwd(
        _ptr(x, "x", bytes_per_elem=2, numel=M * d), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(W_down, "W_down", bytes_per_elem=2, numel=F * d), h.ref,
        _ptr(dy, "dy", bytes_per_elem=2, numel=M * d), d, float(l1),
        _ptr(dx, "dx", bytes_per_elem=2, numel=M * d), _ptr(dW_up, "dW_up", bytes_per_elem=4, numel=F * d),
        _ptr(dW_down, "dW_down", bytes_per_elem=4, numel=F * d), _ptr(db, "db", bytes_per_elem=4, numel=F),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _ptr(status, "status", bytes_per_elem=4),
        _stream(stream)), "twell_ffn_bwd")


def twell_dense_ffn_fwd(x, W_up, b, W_down, h_dense, y, status, stream=None):
    """The dense baseline layer: h_dense = bf16(relu(x W_up^T + b)), y = h_dense W_down."""
    M, d = x.shape
    F = W_up.shape[0]
    _check(load_library().twell_dense_ffn_fwd(
        _ptr(x, "x", bytes_per_elem=2), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(b, "b", bytes_per_elem=4, numel=F), _ptr(W_down, "W_down", bytes_per_elem=2, numel=F * d),
        M, d, F, _ptr(h_dense, "h_dense", bytes_per_elem=2, numel=M * F),
        _ptr(y, "y", bytes_per_elem=2, numel=M * d), _ptr(status, "status", bytes_per_elem=4),
        _stream(stream)), "twell_dense_ffn_fwd")


def twell_dense_bwd_workspace_bytes(M: int, d: int, F: int) -> int:
    return int(load_library().twell_dense_bwd_workspace_bytes(M, d, F))


def twell_dense_ffn_bwd(x, W_up, W_down, h_dense, dy, l1: float, dx, dW_up, dW_down, db, ws, status, stream=None):
    """Backward of the dense baseline layer (same loss and gradients as twell_ffn_bwd)."""
    M, d = x.shape
    F = W_up.shape[0]
    _check(load_library().twell_dense_ffn_bwd(
        _ptr(x, "x", bytes_per_elem=2, numel=M * d), _ptr(W_up, "W_up", bytes_per_elem=2, numel=F * d),
        _ptr(W_down, "W_down", bytes_per_elem=2, numel=F * d),
        _ptr(h_dense, "h_dense", bytes_per_elem=2, numel=M * F), _ptr(dy, "dy", bytes_per_elem=2, numel=M * d),
        M, d, F, float(l1), _ptr(dx, "dx", bytes_per_elem=2, numel=M * d),
        _ptr(dW_up, "dW_up", bytes_per_elem=4, numel=F * d), _ptr(dW_down, "dW_down", bytes_per_elem=4, numel=F * d),
        _ptr(db, "db", bytes_per_elem=4, numel=F), _ptr(ws, "ws"), ws.numel() * ws.element_size(),
        _ptr(status, "status", bytes_per_elem=4), _stream(stream)), "twell_dense_ffn_bwd")


def twell_check(status: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the device status word."""
    out = ctypes.c_int32(0)
    _check(load_library().twell_check(_ptr(status, "status", bytes_per_elem=4), _stream(stream),
                                      ctypes.byref(out)), "twell_check")
    return int(out.value)
