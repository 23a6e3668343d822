"""CPU oracle for the normalize-then-quantize path: TEST INFRASTRUCTURE ONLY.

Python view of ``fp8norm_oracle.c`` (loaded through ctypes).  Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import this
package; the product library (``rmsnorm_fp8_activation_gb300``) never does.

Arrays: bf16 tensors are ``numpy.uint16`` bit patterns, e4m3 and E8M0 tensors
are ``numpy.uint8`` codes, scales and descales are ``numpy.float32``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

ACT_SIGMOID = 0
ACT_SILU = 1

_lib = None


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        _lib = load_library(_build.build())
    return _lib


def use_library(L) -> None:
    """Route every function of this module through the library ``L`` (a
    ``load_library`` result).  The mutation tests use it to run the pins
    against a copy of the oracle with a planted mistake."""
    global _lib
    _lib = L


def load_library(path: str) -> ctypes.CDLL:
    """Open an oracle shared library and declare its signatures."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_double.restype = ctypes.c_double
    L.oracle_bf16_from_double.argtypes = [ctypes.c_double]
    L.oracle_bf16_from_double.restype = ctypes.c_uint16
    L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_double.restype = ctypes.c_double
    L.oracle_e4m3_from_float.argtypes = [f32]
    L.oracle_e4m3_from_float.restype = ctypes.c_uint8
    L.oracle_act_bf16.argtypes = [ctypes.c_uint16, ctypes.c_int]
    L.oracle_act_bf16.restype = ctypes.c_uint16
    L.oracle_bf16_from_float_n.argtypes = [P, i64, P]
    L.oracle_bf16_from_float_n.restype = None
    L.oracle_e4m3_from_float_n.argtypes = [P, i64, P]
    L.oracle_e4m3_from_float_n.restype = None
    L.oracle_act_bf16_n.argtypes = [P, i64, ctypes.c_int, P]
    L.oracle_act_bf16_n.restype = None
    L.oracle_mean_square_bf16.argtypes = [P, i64]
    L.oracle_mean_square_bf16.restype = f32
    L.oracle_rms_factor.argtypes = [f32, f32]
    L.oracle_rms_factor.restype = f32
    L.oracle_e8m0_code.argtypes = [ctypes.c_uint16]
    L.oracle_e8m0_code.restype = ctypes.c_uint8
    L.oracle_gated_rmsnorm_quant_token.argtypes = [
        P, i64, P, i64, P, i64, i32, i32, f32, ctypes.c_int, P, i64, P]
    L.oracle_gated_rmsnorm_quant_token.restype = None
    L.oracle_gated_rmsnorm_quant_one.argtypes = [
        P, P, P, i32, i32, f32, ctypes.c_int, P, P, P]
    L.oracle_gated_rmsnorm_quant_one.restype = None
    L.oracle_gated_rmsnorm_quant_one_ms.argtypes = [
        P, P, P, i32, i32, f32, ctypes.c_int, P, P, P, P]
    L.oracle_gated_rmsnorm_quant_one_ms.restype = None
    L.oracle_inv_rope_row.argtypes = [P, i32, i32, i32, i32, ctypes.c_int, P, P]
    L.oracle_inv_rope_row.restype = None
    L.oracle_inv_rope_quant_mx.argtypes = [P, i64, i64, i32, i32, P, P, i32, i32, ctypes.c_int,
                                           P, i64, P, i64]
    L.oracle_inv_rope_quant_mx.restype = None
    L.oracle_rmsnorm_quant_mx.argtypes = [
        P, i64, P, i32, P, i64, P, i32, i64, f32, P, i64, P, i64, P, i64]
    L.oracle_rmsnorm_quant_mx.restype = None
    L.oracle_static_head_quant.argtypes = [P, i64, i64, i64, i32, i32, P, P]
    L.oracle_static_head_quant.restype = None
    L.oracle_quant_row.argtypes = [P, i64, P, P]
    L.oracle_quant_row.restype = None
    L.oracle_gated_rmsnorm_row.argtypes = [P, P, P, i32, i32, f32, ctypes.c_int, P]
    L.oracle_gated_rmsnorm_row.restype = None
    L.oracle_gated_quant_row.argtypes = [P, P, i64, ctypes.c_int, P, P, P]
    L.oracle_gated_quant_row.restype = None
    L.oracle_rmsnorm_row.argtypes = [P, P, i32, f32, P]
    L.oracle_rmsnorm_row.restype = None
    L.oracle_quant_mx_row.argtypes = [P, i32, P, P]
    L.oracle_quant_mx_row.restype = None
    L.oracle_head_amax.argtypes = [P, i64, i64, i64, i32, i32, P]
    L.oracle_head_amax.restype = None
    L.oracle_dynamic_head_quant.argtypes = [P, i64, i64, i64, i32, i32, P, P]
    L.oracle_dynamic_head_quant.restype = None
    return L


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def host_threads() -> int:
    """Host threads available to this process."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # not on Linux
        return max(1, os.cpu_count() or 1)


def sliced(fn, n: int, threads: int | None = None, min_slice: int = 1):
    """Run ``fn(start, stop)`` over [0, n) cut into contiguous slices, on a
    pool of host threads (the oracle's functions are called through ctypes,
    which releases the interpreter lock, so the slices run in parallel; each
    call is the same single-threaded function on its own rows).  Returns the
    results in slice order.  threads=1 runs the slices in order on the calling
    thread."""
    from concurrent.futures import ThreadPoolExecutor
    threads = host_threads() if threads is None else max(1, int(threads))
    lib()  # load once, before the pool
    parts = min(max(1, n // max(1, min_slice)), 4 * threads) if n > 0 else 0
    bounds = [(n * i // parts, n * (i + 1) // parts) for i in range(parts)]
    if threads == 1 or parts <= 1:
        return [fn(a, b) for a, b in bounds]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda ab: fn(*ab), bounds))


# ---- codecs ---------------------------------------------------------------

def bf16_to_float(bits) -> np.ndarray:
    """Exact float32 values of bf16 bit patterns (vectorised bit shift)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_from_double(v: float) -> int:
    return int(lib().oracle_bf16_from_double(float(v)))


def e4m3_to_double(code: int) -> float:
    return float(lib().oracle_e4m3_to_double(int(code)))


def e4m3_from_float(v: float) -> int:
    return int(lib().oracle_e4m3_from_float(float(v)))


def act_bf16(g: int, act: int) -> int:
    return int(lib().oracle_act_bf16(int(g), int(act)))


def bf16_from_float_n(v) -> np.ndarray:
    """bf16 bits of binary32 values, nearest-even."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_bf16_from_float_n(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_from_float_n(v) -> np.ndarray:
    """Saturating nearest-even E4M3 codes of binary32 values."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().oracle_e4m3_from_float_n(_ptr(v), v.size, _ptr(out))
    return out


def act_bf16_n(g, act: int) -> np.ndarray:
    g = _c(g, np.uint16)
    out = np.empty(g.shape, dtype=np.uint16)
    lib().oracle_act_bf16_n(_ptr(g), g.size, int(act), _ptr(out))
    return out


def act_table(act: int) -> np.ndarray:
    """bf16(act(g)) for all 65536 gate bit patterns."""
    return act_bf16_n(np.arange(65536, dtype=np.uint16), act)


def mean_square(x_bits) -> float:
    x = _c(x_bits, np.uint16)
    return float(lib().oracle_mean_square_bf16(_ptr(x), x.size))


def rms_factor(ms: float, eps: float) -> float:
    return float(lib().oracle_rms_factor(ms, eps))


def e8m0_code(amax_bits: int) -> int:
    return int(lib().oracle_e8m0_code(int(amax_bits)))


# ---- operations -----------------------------------------------------------

def gated_rmsnorm_quant_token(x, gate, weight, eps: float, act: int):
    """Operation (A).  x, gate: uint16 [T, H, D]; weight: uint16 [D].

    Returns (codes uint8 [T, H*D], scale float32 [T]).
    """
    x = _c(x, np.uint16)
    gate = _c(gate, np.uint16)
    weight = _c(weight, np.uint16)
    T, H, D = x.shape
    out = np.zeros((T, H * D), dtype=np.uint8)
    scale = np.zeros((T,), dtype=np.float32)
    lib().oracle_gated_rmsnorm_quant_token(
        _ptr(x), H * D, _ptr(gate), H * D, _ptr(weight), T, H, D, float(eps), int(act),
        _ptr(out), H * D, _ptr(scale))
    return out, scale


def gated_rmsnorm_quant_one(x_tok, gate_tok, weight, eps: float, act: int):
    """Operation (A) on one token.  x_tok, gate_tok: uint16 [H, D].

    Returns (y bf16 bits [H*D], codes uint8 [H*D], scale float).
    """
    x_tok = _c(x_tok, np.uint16)
    gate_tok = _c(gate_tok, np.uint16)
    weight = _c(weight, np.uint16)
    H, D = x_tok.shape
    y = np.zeros((H * D,), dtype=np.uint16)
    out = np.zeros((H * D,), dtype=np.uint8)
    scale = np.zeros((1,), dtype=np.float32)
    lib().oracle_gated_rmsnorm_quant_one(
        _ptr(x_tok), _ptr(gate_tok), _ptr(weight), H, D, float(eps), int(act),
        _ptr(y), _ptr(out), _ptr(scale))
    return y, out, float(scale[0])


def gated_rmsnorm_quant_one_ms(x_tok, gate_tok, weight, eps: float, act: int, ms):
    """Operation (A) on one token with each head's mean square given (float32
    [H]) instead of computed: a diagnostic that the parity checks use to tell
    whether a differing token is explained by one head's summation order.

    Returns (y bf16 bits [H*D], codes uint8 [H*D], scale float).
    """
    x_tok = _c(x_tok, np.uint16)
    gate_tok = _c(gate_tok, np.uint16)
    weight = _c(weight, np.uint16)
    ms = _c(ms, np.float32)
    H, D = x_tok.shape
    assert ms.shape == (H,)
    y = np.zeros((H * D,), dtype=np.uint16)
    out = np.zeros((H * D,), dtype=np.uint8)
    scale = np.zeros((1,), dtype=np.float32)
    lib().oracle_gated_rmsnorm_quant_one_ms(
        _ptr(x_tok), _ptr(gate_tok), _ptr(weight), H, D, float(eps), int(act), _ptr(ms),
        _ptr(y), _ptr(out), _ptr(scale))
    return y, out, float(scale[0])


def rmsnorm_quant_mx(q, q_weight, kv, kv_weight, eps: float):
    """Operation (B).  q: uint16 [M, Nq]; kv: uint16 [M, Nkv].

    Returns (q codes uint8 [M, Nq], q scales uint8 [M, Nq/32], kv bf16 bits [M, Nkv]).
    """
    q = _c(q, np.uint16)
    kv = _c(kv, np.uint16)
    q_weight = _c(q_weight, np.uint16)
    kv_weight = _c(kv_weight, np.uint16)
    M, Nq = q.shape
    M2, Nkv = kv.shape
    assert M == M2 and Nq % 32 == 0
    q_out = np.zeros((M, Nq), dtype=np.uint8)
    q_scale = np.zeros((M, Nq // 32), dtype=np.uint8)
    kv_out = np.zeros((M, Nkv), dtype=np.uint16)
    lib().oracle_rmsnorm_quant_mx(
        _ptr(q), Nq, _ptr(q_weight), Nq, _ptr(kv), Nkv, _ptr(kv_weight), Nkv, M, float(eps),
        _ptr(q_out), Nq, _ptr(q_scale), Nq // 32, _ptr(kv_out), Nkv)
    return q_out, q_scale, kv_out


def inv_rope_bf16(o, positions, cos_sin, rope_off: int, rope_dim: int, interleaved: bool):
    """The inverse-RoPE step alone: o uint16 [T, H, D] -> bf16 bits [T, H*D]."""
    o = _c(o, np.uint16)
    positions = _c(positions, np.int32)
    cos_sin = _c(cos_sin, np.float32)
    T, H, D = o.shape
    assert cos_sin.shape[1] == rope_dim and positions.shape == (T,)
    assert positions.min(initial=0) >= 0 and positions.max(initial=0) < cos_sin.shape[0]
    y = np.zeros((T, H * D), dtype=np.uint16)
    for t in range(T):
        lib().oracle_inv_rope_row(_ptr(o[t]), H, D, int(rope_off), int(rope_dim),
                                  int(bool(interleaved)), _ptr(cos_sin[positions[t]]), _ptr(y[t]))
    return y


def inv_rope_quant_mx(o, positions, cos_sin, rope_off: int, rope_dim: int, interleaved: bool):
    """Inverse RoPE then MXFP8.  o: uint16 [T, H, D]; positions int32 [T];
    cos_sin float32 [P, rope_dim].  Returns (codes uint8 [T, H*D], E8M0 uint8
    [T, H*D/32])."""
    o = _c(o, np.uint16)
    positions = _c(positions, np.int32)
    cos_sin = _c(cos_sin, np.float32)
    T, H, D = o.shape
    assert D % 32 == 0 and cos_sin.shape[1] == rope_dim and positions.shape == (T,)
    assert positions.min(initial=0) >= 0 and positions.max(initial=0) < cos_sin.shape[0]
    out = np.zeros((T, H * D), dtype=np.uint8)
    scale = np.zeros((T, H * D // 32), dtype=np.uint8)
    lib().oracle_inv_rope_quant_mx(_ptr(o), H * D, T, H, D, _ptr(positions), _ptr(cos_sin),
                                   int(rope_off), int(rope_dim), int(bool(interleaved)),
                                   _ptr(out), H * D, _ptr(scale), H * D // 32)
    return out, scale


def static_head_quant(x, descale):
    """Operation (C) on one tensor.  x: uint16 [T, H, Dh]; descale: float32 [H].

    Returns codes uint8 [T, H, Dh].
    """
    x = _c(x, np.uint16)
    descale = _c(descale, np.float32)
    T, H, Dh = x.shape
    out = np.zeros((T, H, Dh), dtype=np.uint8)
    lib().oracle_static_head_quant(_ptr(x), H * Dh, Dh, T, H, Dh, _ptr(descale), _ptr(out))
    return out


# ---- the steps of (A) and (B) on their own, and the dynamic per-head quant ----

def quant_token(y):
    """Per-token FP8 of bf16 rows y [T, N]: (codes uint8 [T, N], scale float32 [T])."""
    y = _c(y, np.uint16)
    T, N = y.shape
    out = np.zeros((T, N), dtype=np.uint8)
    scale = np.zeros((T,), dtype=np.float32)
    for t in range(T):
        lib().oracle_quant_row(_ptr(y[t]), N, _ptr(out[t]), scale[t:].ctypes.data)
    return out, scale


def gated_rmsnorm_bf16(x, gate, weight, eps: float, act: int):
    """(A) without the quantisation: y bf16 bits [T, H*D]."""
    x = _c(x, np.uint16)
    gate = _c(gate, np.uint16)
    weight = _c(weight, np.uint16)
    T, H, D = x.shape
    y = np.zeros((T, H * D), dtype=np.uint16)
    for t in range(T):
        lib().oracle_gated_rmsnorm_row(_ptr(x[t]), _ptr(gate[t]), _ptr(weight), H, D, float(eps),
                                       int(act), _ptr(y[t]))
    return y


def gated_quant_token(x, gate, act: int):
    """y = bf16(x * bf16(act(gate))) per element of [T, N], then per-token FP8.
    Returns (y bf16 bits, codes, scale)."""
    x = _c(x, np.uint16)
    gate = _c(gate, np.uint16)
    T, N = x.shape
    y = np.zeros((T, N), dtype=np.uint16)
    out = np.zeros((T, N), dtype=np.uint8)
    scale = np.zeros((T,), dtype=np.float32)
    for t in range(T):
        lib().oracle_gated_quant_row(_ptr(x[t]), _ptr(gate[t]), N, int(act), _ptr(y[t]),
                                     _ptr(out[t]), scale[t:].ctypes.data)
    return y, out, scale


def rmsnorm_bf16(x, weight, eps: float):
    """Row RMSNorm of bf16 rows x [M, N] with weight [N]: bf16 bits [M, N]."""
    x = _c(x, np.uint16)
    weight = _c(weight, np.uint16)
    M, N = x.shape
    y = np.zeros((M, N), dtype=np.uint16)
    for m in range(M):
        lib().oracle_rmsnorm_row(_ptr(x[m]), _ptr(weight), N, float(eps), _ptr(y[m]))
    return y


def quant_mx(yq):
    """MX quantisation of bf16 rows yq [M, N] (N % 32 == 0): (codes [M, N], E8M0 [M, N/32])."""
    yq = _c(yq, np.uint16)
    M, N = yq.shape
    assert N % 32 == 0
    codes = np.zeros((M, N), dtype=np.uint8)
    scales = np.zeros((M, N // 32), dtype=np.uint8)
    for m in range(M):
        lib().oracle_quant_mx_row(_ptr(yq[m]), N, _ptr(codes[m]), _ptr(scales[m]))
    return codes, scales


def head_amax(x, amax=None):
    """Running per-head max of |x| for x [T, H, Dh]; returns the updated float32 [H]."""
    x = _c(x, np.uint16)
    T, H, Dh = x.shape
    a = np.zeros((H,), dtype=np.float32) if amax is None else np.array(amax, dtype=np.float32)
    lib().oracle_head_amax(_ptr(x), H * Dh, Dh, T, H, Dh, _ptr(a))
    return a


def dynamic_head_quant(x):
    """Per-head descales from the tensor's own maxima, then codes: (descale [H], codes)."""
    x = _c(x, np.uint16)
    T, H, Dh = x.shape
    d = np.zeros((H,), dtype=np.float32)
    out = np.zeros((T, H, Dh), dtype=np.uint8)
    lib().oracle_dynamic_head_quant(_ptr(x), H * Dh, Dh, T, H, Dh, _ptr(d), _ptr(out))
    return d, out
