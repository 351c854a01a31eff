"""CPU oracle for the TwELL activation-sparse feed-forward layer.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product path (the CUDA
library and its binding) never imports this package.

A thin ctypes wrapper over ``twell_oracle.c`` (plain C loops, fp64
accumulation). The C library is compiled with gcc on first use, into
``oracle/_build/``. Functions take and return numpy arrays; bf16 tensors are
uint16 bit arrays.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "twell_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP). Returns the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (force or not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


P = ctypes.c_void_p
I32 = ctypes.c_int
I64 = ctypes.c_int64
DBL = ctypes.c_double


def _declare(lib):
    lib.oracle_num_threads.restype = I32
    lib.oracle_round_bf16.argtypes = [P, P, I64]
    lib.oracle_ffn_fwd_rows.argtypes = [P, P, P, P, P, I32, I32, I32, P, I32, P, P, P, P, P]
    lib.oracle_twell_layout.argtypes = [P, P, I32, I32, I32, I32, P, P, P]
    lib.oracle_twell_layout.restype = I64
    lib.oracle_twell_fill.argtypes = [P, P, I32, I32, I32, I32, P, P, P, P]
    lib.oracle_twell_unpack.argtypes = [I32, I32, I32, P, P, P, P, P, P]
    lib.oracle_twell_unpack.restype = I32
    lib.oracle_twell_spmm.argtypes = [I32, I32, I32, P, P, P, P, P, P, I32, P]
    lib.oracle_ffn_bwd_rows.argtypes = [P, P, P, P, P, DBL, I32, I32, I32, P, I32, P, P]
    lib.oracle_ffn_bwd_cols.argtypes = [P, P, P, P, P, DBL, I32, I32, I32, P, I32, P, P, P]
    lib.oracle_ffn_loss_f64.argtypes = [P, P, P, P, P, DBL, I32, I32, I32, P]
    lib.oracle_ffn_loss_f64.restype = DBL


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def round_bf16(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, nearest-even (the oracle's own rounding)."""
    a = _c(a, np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_round_bf16(_p(a), _p(out), a.size)
    return out


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclasses.dataclass
class Twell:
    """A TwELL as numpy arrays (layout in the oracle's C comments)."""
    M: int
    F: int
    T: int
    nnz: np.ndarray   # int32 [M]
    K: np.ndarray     # int32 [n_tiles]
    off: np.ndarray   # int64 [n_tiles + 1]
    idx: np.ndarray   # int32 [off[-1]]
    val: np.ndarray   # uint16 [off[-1]] (bf16 bits)

    @property
    def n_tiles(self) -> int:
        return (self.M + self.T - 1) // self.T

    @property
    def slots(self) -> int:
        return int(self.off[-1])


def ffn_fwd_rows(x, W_up, W_gate, b, W_down, M, d, F, rows=None, want_y=True):
    """Dense forward of the listed rows: returns dict(pre, u, h, active, y)."""
    rows = np.arange(M, dtype=np.int32) if rows is None else _c(rows, np.int32)
    n = len(rows)
    x, W_up, W_down = _c(x, np.uint16), _c(W_up, np.uint16), _c(W_down, np.uint16)
    W_gate = None if W_gate is None else _c(W_gate, np.uint16)
    b = _c(b, np.float32)
    pre = np.empty((n, F), np.float32)
    u = np.empty((n, F), np.float32) if W_gate is not None else None
    h = np.empty((n, F), np.uint16)
    act = np.empty((n, F), np.uint8)
    y = np.empty((n, d), np.float64) if want_y else None
    _load().oracle_ffn_fwd_rows(_p(x), _p(W_up), _p(W_gate), _p(b), _p(W_down), M, d, F,
                                _p(rows), n, _p(pre), _p(u), _p(h), _p(act), _p(y))
    return dict(pre=pre, u=u, h=h, active=act, y=y)


def twell_pack(h: np.ndarray, T: int, active: np.ndarray | None = None) -> Twell:
    """TwELL of a dense [M, F] bf16 matrix (active set h != 0, or `active`)."""
    h = _c(h, np.uint16)
    M, F = h.shape
    act = None if active is None else _c(active, np.uint8)
    n_tiles = (M + T - 1) // T
    nnz = np.empty(M, np.int32)
    K = np.empty(n_tiles, np.int32)
    off = np.empty(n_tiles + 1, np.int64)
    lib = _load()
    total = lib.oracle_twell_layout(_p(h), _p(act), M, F, F, T, _p(nnz), _p(K), _p(off))
    idx = np.empty(max(total, 1), np.int32)
    val = np.empty(max(total, 1), np.uint16)
    lib.oracle_twell_fill(_p(h), _p(act), M, F, F, T, _p(K), _p(off), _p(idx), _p(val))
    return Twell(M, F, T, nnz, K, off, idx[:total].copy(), val[:total].copy())


def hybrid_pack(h: np.ndarray, T: int, C: int) -> tuple[Twell, np.ndarray, np.ndarray]:
    """Hybrid format of a dense [M, F] bf16 matrix ("Sparser, Faster, Lighter
    Transformer Language Models", Resumo Técnico §2, "Formato Híbrido para
    Treinamento"): a row with more than C nonzeros (+-0 are zeros) overflows.
    Returns (TwELL of h with the overflow rows emptied, overflow row ids
    ascending, their dense rows [n, F])."""
    h = _c(h, np.uint16)
    counts = ((h & 0x7FFF) != 0).sum(axis=1)
    rows = np.nonzero(counts > C)[0].astype(np.int32)
    h_ell = h.copy()
    h_ell[rows] = 0
    return twell_pack(h_ell, T), rows, h[rows].copy()


def twell_unpack(tw: Twell) -> tuple[int, np.ndarray]:
    """(status, dense h). status 0 = valid TwELL; see the C comment for codes."""
    h = np.empty((tw.M, tw.F), np.uint16)
    idx = _c(tw.idx, np.int32) if tw.slots else np.zeros(1, np.int32)
    val = _c(tw.val, np.uint16) if tw.slots else np.zeros(1, np.uint16)
    code = _load().oracle_twell_unpack(tw.M, tw.F, tw.T, _p(_c(tw.nnz, np.int32)),
                                       _p(_c(tw.K, np.int32)), _p(_c(tw.off, np.int64)),
                                       _p(idx), _p(val), _p(h))
    return int(code), h


def twell_spmm(tw: Twell, W: np.ndarray) -> np.ndarray:
    """y = TwELL @ W (fp64), W [F, d] bf16 bits."""
    W = _c(W, np.uint16)
    d = W.shape[1]
    y = np.empty((tw.M, d), np.float64)
    idx = _c(tw.idx, np.int32) if tw.slots else np.zeros(1, np.int32)
    val = _c(tw.val, np.uint16) if tw.slots else np.zeros(1, np.uint16)
    _load().oracle_twell_spmm(tw.M, tw.F, tw.T, _p(_c(tw.nnz, np.int32)), _p(_c(tw.K, np.int32)),
                              _p(_c(tw.off, np.int64)), _p(idx), _p(val), _p(W), d, _p(y))
    return y


def ffn_bwd_rows(x, W_up, W_down, h, dy, l1, rows=None):
    """dpre [n, F] and dx [n, d] (fp64) for the listed token rows.

    All array arguments are fp64 (widen bf16 with bf16_to_f64)."""
    x, W_up, W_down, h, dy = (_c(a, np.float64) for a in (x, W_up, W_down, h, dy))
    M, d = x.shape
    F = W_up.shape[0]
    rows = np.arange(M, dtype=np.int32) if rows is None else _c(rows, np.int32)
    n = len(rows)
    dpre = np.empty((n, F), np.float64)
    dx = np.empty((n, d), np.float64)
    _load().oracle_ffn_bwd_rows(_p(x), _p(W_up), _p(W_down), _p(h), _p(dy), float(l1),
                                M, d, F, _p(rows), n, _p(dpre), _p(dx))
    return dpre, dx


def ffn_bwd_cols(x, W_up, W_down, h, dy, l1, cols=None):
    """dW_up [n, d], dW_down [n, d], db [n] (fp64) for the listed hidden units."""
    x, W_up, W_down, h, dy = (_c(a, np.float64) for a in (x, W_up, W_down, h, dy))
    M, d = x.shape
    F = W_up.shape[0]
    cols = np.arange(F, dtype=np.int32) if cols is None else _c(cols, np.int32)
    n = len(cols)
    gu = np.empty((n, d), np.float64)
    gd = np.empty((n, d), np.float64)
    gb = np.empty(n, np.float64)
    _load().oracle_ffn_bwd_cols(_p(x), _p(W_up), _p(W_down), _p(h), _p(dy), float(l1),
                                M, d, F, _p(cols), n, _p(gu), _p(gd), _p(gb))
    return gu, gd, gb


def ffn_loss_f64(x, W_up, b, W_down, dy, l1, want_h=False):
    """Unrounded fp64 loss <dy, relu(x W_up^T + b) W_down> + l1 * sum(h)."""
    x, W_up, b, W_down, dy = (_c(a, np.float64) for a in (x, W_up, b, W_down, dy))
    M, d = x.shape
    F = W_up.shape[0]
    h = np.empty((M, F), np.float64) if want_h else None
    L = _load().oracle_ffn_loss_f64(_p(x), _p(W_up), _p(b), _p(W_down), _p(dy), float(l1),
                                    M, d, F, _p(h))
    return (float(L), h) if want_h else float(L)
