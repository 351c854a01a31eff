"""Seeded synthetic inputs for the TwELL feed-forward layer.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path's tests and benchmark. It draws random numbers and rounds them to the
storage dtype; it holds none of the layer's arithmetic (no products, no
activation, no packing).

Generator: a counter-based splitmix64 stream (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014: the splitmix64
finaliser applied to ``seed + (i+1) * golden_gamma``), uniform doubles from the
top 53 bits, and normals by the Box–Muller transform (Box and Muller, 1958).
Element ``i`` of stream ``s`` depends only on ``(seed, s, i)``, so any slice of
a tensor can be regenerated independently.

Workload recipes follow the synthetic configurations of the layer:
x ~ N(0,1), W_up and W_gate ~ N(0, 1/d_model), W_down ~ N(0, 1/d_ff),
dy ~ N(0,1), a scalar bias broadcast to every hidden unit, and optionally a
per-token row scale s_r ~ LogNormal(0, 1) on x for skewed sparsity.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids: one independent stream per tensor of a workload.
STREAM_X = 1
STREAM_W_UP = 2
STREAM_W_GATE = 3
STREAM_W_DOWN = 4
STREAM_DY = 5
STREAM_ROW_SCALE = 6
STREAM_MASK = 7
STREAM_VALUES = 8


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: int) -> np.uint64:
    s = np.array([(seed & 0xFFFFFFFF) | ((stream & 0xFFFFFFFF) << 32)], dtype=np.uint64)
    return _mix(s + _GAMMA)[0]


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Elements ``start .. start+count-1`` of stream ``stream`` as uint64."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(_stream_base(seed, stream) + i * _GAMMA)


def uniform(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Doubles in (0, 1]: ``((z >> 11) + 1) * 2**-53``."""
    z = raw_u64(seed, stream, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def _normal_range(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    u = uniform(seed, stream, 2 * count, start=2 * start)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


_CHUNK = 1 << 21


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """Standard normals by Box–Muller; element i uses uniforms 2i and 2i+1.

    Large draws are computed in chunks on a thread pool (numpy releases the
    interpreter lock inside its array loops); every element still depends only
    on (seed, stream, i), so the result is the same as one sequential draw."""
    if count <= 2 * _CHUNK:
        return _normal_range(seed, stream, 0, count)
    import concurrent.futures as cf
    import os
    out = np.empty(count, dtype=np.float64)
    starts = list(range(0, count, _CHUNK))

    def one(s0: int) -> None:
        n = min(_CHUNK, count - s0)
        out[s0:s0 + n] = _normal_range(seed, stream, s0, n)

    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        list(ex.map(one, starts))
    return out


def normal_at(seed: int, stream: int, index: np.ndarray) -> np.ndarray:
    """Elements `index` of the stream normal(seed, stream, .) without drawing the rest."""
    i = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        base = _stream_base(seed, stream)
        z1 = _mix(base + (np.uint64(2) * i + np.uint64(1)) * _GAMMA)
        z2 = _mix(base + (np.uint64(2) * i + np.uint64(2)) * _GAMMA)
    u1 = ((z1 >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    u2 = ((z2 >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits.

    NaN maps to a quiet NaN of the same sign. Inputs here are finite draws, so
    that branch exists only for completeness.
    """
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    hi = u >> np.uint64(16)
    lo = u & np.uint64(0xFFFF)
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & np.uint64(1)) == 1))
    out = (hi + up.astype(np.uint64)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class FFNInputs:
    """One synthetic layer instance. bf16 tensors are uint16 bit arrays."""
    M: int
    d: int
    F: int
    T: int
    x: np.ndarray            # [M, d] bf16 bits
    W_up: np.ndarray         # [F, d] bf16 bits
    W_gate: np.ndarray | None  # [F, d] bf16 bits (gated layer) or None
    W_down: np.ndarray       # [F, d] bf16 bits
    b: np.ndarray            # [F] float32
    dy: np.ndarray | None    # [M, d] bf16 bits
    l1: float = 0.0
    seed: int = 0


def ffn_inputs(M: int, d: int, F: int, T: int, bias: float, *, seed: int = 0,
               gated: bool = False, with_dy: bool = False, l1: float = 0.0,
               row_skew_sigma: float = 0.0) -> FFNInputs:
    """Draw x, W_up (, W_gate), W_down, b (, dy) for one configuration.

    Weights are stored [F, d] row-major (out x in for the up/gate projections,
    one row per hidden unit for the down projection). ``row_skew_sigma > 0``
    multiplies token row r of x by exp(sigma * z_r), z_r ~ N(0,1), before the
    bf16 rounding.
    """
    x = normal(seed, STREAM_X, M * d).reshape(M, d)
    if row_skew_sigma > 0.0:
        s = np.exp(row_skew_sigma * normal(seed, STREAM_ROW_SCALE, M))
        x = x * s[:, None]
    w_up = normal(seed, STREAM_W_UP, F * d).reshape(F, d) * (1.0 / math.sqrt(d))
    w_gate = (normal(seed, STREAM_W_GATE, F * d).reshape(F, d) * (1.0 / math.sqrt(d))
              if gated else None)
    w_down = normal(seed, STREAM_W_DOWN, F * d).reshape(F, d) * (1.0 / math.sqrt(F))
    dy = normal(seed, STREAM_DY, M * d).reshape(M, d) if with_dy else None
    return FFNInputs(
        M=M, d=d, F=F, T=T,
        x=to_bf16_bits(x.astype(np.float32)),
        W_up=to_bf16_bits(w_up.astype(np.float32)),
        W_gate=None if w_gate is None else to_bf16_bits(w_gate.astype(np.float32)),
        W_down=to_bf16_bits(w_down.astype(np.float32)),
        b=np.full(F, bias, dtype=np.float32),
        dy=None if dy is None else to_bf16_bits(dy.astype(np.float32)),
        l1=l1, seed=seed)


def integer_ffn_inputs(M: int, d: int, F: int, T: int, *, seed: int = 0,
                       lo: int = -4, hi: int = 4, bias: int = -8) -> FFNInputs:
    """Integer-valued bf16 inputs in [lo, hi] and an integer bias.

    Every product and partial sum of the up projection is an integer far below
    2**24, so any fp32 summation order gives the same pre-activation, and the
    layer's TwELL is fixed exactly, independent of the accumulation order.
    """
    def ints(stream: int, n: int) -> np.ndarray:
        u = uniform(seed, stream, n)
        return np.floor(lo + u * (hi - lo + 1) - 1e-12).clip(lo, hi)
    x = ints(STREAM_X, M * d).reshape(M, d)
    w_up = ints(STREAM_W_UP, F * d).reshape(F, d)
    w_down = ints(STREAM_W_DOWN, F * d).reshape(F, d)
    return FFNInputs(
        M=M, d=d, F=F, T=T,
        x=to_bf16_bits(x.astype(np.float32)),
        W_up=to_bf16_bits(w_up.astype(np.float32)),
        W_gate=None,
        W_down=to_bf16_bits(w_down.astype(np.float32)),
        b=np.full(F, float(bias), dtype=np.float32),
        dy=None, seed=seed)


def sparse_hidden(M: int, F: int, density: float, *, seed: int = 0,
                  row_skew_sigma: float = 0.0) -> np.ndarray:
    """A random nonnegative hidden matrix h [M, F] (bf16 bits) with given density.

    Entry (r, j) is active when uniform draw r*F + j is below ``density`` (scaled
    by the row's skew factor when ``row_skew_sigma > 0``, clipped to 1); an
    active value is |z| + 2**-8 with z normal draw r*F + j, so none rounds to
    zero. Generated in row chunks; only active entries draw their normal.
    """
    h = np.zeros((M, F), dtype=np.uint16)
    if row_skew_sigma > 0.0:
        p_row = np.clip(density * np.exp(row_skew_sigma * normal(seed, STREAM_ROW_SCALE, M)), 0.0, 1.0)
    else:
        p_row = np.full(M, density)
    rows_per_chunk = max(1, (1 << 22) // max(F, 1))
    for r0 in range(0, M, rows_per_chunk):
        r1 = min(M, r0 + rows_per_chunk)
        u = uniform(seed, STREAM_MASK, (r1 - r0) * F, start=r0 * F).reshape(r1 - r0, F)
        rr, jj = np.nonzero(u <= p_row[r0:r1, None])
        flat = (rr + r0).astype(np.uint64) * np.uint64(F) + jj.astype(np.uint64)
        vals = np.abs(normal_at(seed, STREAM_VALUES, flat)) + 2.0 ** -8
        h[rr + r0, jj] = to_bf16_bits(vals.astype(np.float32))
    return h


# The synthetic configurations of the layer, by name. Sizes, biases and tile
# heights are those of the workloads the method is measured on; seed 0 for all.
CONFIGS = {
    "tiny": dict(M=64, d=128, F=512, T=16, bias=-2.33, gated=False),
    "inference": dict(M=4096, d=2048, F=8192, T=128, bias=-2.33, gated=False),
    "decode1": dict(M=1, d=4096, F=14336, T=1, bias=-2.58, gated=True),
    "decode8": dict(M=8, d=4096, F=14336, T=8, bias=-2.58, gated=True),
    "decode64": dict(M=64, d=4096, F=14336, T=64, bias=-2.58, gated=True),
    "training": dict(M=16384, d=4096, F=16384, T=128, bias=-2.33, gated=False, l1=1e-4),
    # sparsity/skew sweep, nominal biases: Phi^-1 of the target density, the
    # bias that gives it without skew (with the row scales the realised
    # density is higher: about 14 / 7.4 / 5.1 %)
    "sweep90": dict(M=8192, d=4096, F=16384, T=128, bias=-1.2816, gated=False, skew=1.0),
    "sweep99": dict(M=8192, d=4096, F=16384, T=128, bias=-2.3263, gated=False, skew=1.0),
    "sweep999": dict(M=8192, d=4096, F=16384, T=128, bias=-3.0902, gated=False, skew=1.0),
    # the same with skew-corrected biases: b solves E_s[Phi(b / s)] = 10 / 1 / 0.1 %
    # for s ~ LogNormal(0, 1), the density of ReLU(s z + b) with z ~ N(0, 1)
    # (x . w is ~N(0, 1) for x ~ N(0, I), w ~ N(0, I / d_model))
    "sweep90s": dict(M=8192, d=4096, F=16384, T=128, bias=-1.8108, gated=False, skew=1.0),
    "sweep99s": dict(M=8192, d=4096, F=16384, T=128, bias=-7.8373, gated=False, skew=1.0),
    "sweep999s": dict(M=8192, d=4096, F=16384, T=128, bias=-20.2430, gated=False, skew=1.0),
}

# Target hidden density of each sweep workload (fraction of active units).
SWEEP_TARGETS = {"sweep90": 0.10, "sweep99": 0.01, "sweep999": 0.001,
                 "sweep90s": 0.10, "sweep99s": 0.01, "sweep999s": 0.001}


def config_inputs(name: str, *, seed: int = 0, with_dy: bool = False) -> FFNInputs:
    c = CONFIGS[name]
    return ffn_inputs(c["M"], c["d"], c["F"], c["T"], c["bias"], seed=seed,
                      gated=c["gated"], with_dy=with_dy, l1=c.get("l1", 0.0),
                      row_skew_sigma=c.get("skew", 0.0))
