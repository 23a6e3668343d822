"""Python binding of libfp8norm (argument marshalling only).

Each function has the name of the C entry point it calls and passes torch CUDA
tensors to it as raw device pointers with the current CUDA stream; every step
of the computation runs in the library's kernels.  PyTorch is used only for
device memory and streams.  The shared library must have been built
(``rmsnorm_fp8_activation_gb300.build.build()``); there is no fallback.

Tensor conventions: bf16 tensors are ``torch.bfloat16`` (or 16-bit integer
views of the same bits); e4m3 outputs are ``torch.uint8`` codes (view them as
``torch.float8_e4m3fn`` if wanted); E8M0 scales are ``torch.uint8``.
"""
from __future__ import annotations

import ctypes
import os

import torch

ACT_SIGMOID = 0
ACT_SILU = 1

STATUS_BAD_DESCALE = 0x1
STATUS_PIPELINE_TIMEOUT = 0x2
STATUS_BAD_SEQLENS = 0x4
STATUS_BAD_POSITION = 0x8
ROPE_HALF = 0
ROPE_INTERLEAVED = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8norm.so")
_lib = None


class Fp8NormError(RuntimeError):
    """A libfp8norm call returned a nonzero fp8n_status."""

    def __init__(self, fn: str, code: int, msg: str):
        super().__init__("%s: %s (status %d)" % (fn, msg, code))
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libfp8norm.so is missing (%s): build it with "
                "rmsnorm_fp8_activation_gb300.build.build(); there is no fallback path" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        L.fp8n_status_string.argtypes = [ctypes.c_int]
        L.fp8n_status_string.restype = ctypes.c_char_p
        L.fp8n_last_cuda_error.argtypes = []
        L.fp8n_last_cuda_error.restype = ctypes.c_int
        L.fp8n_version.argtypes = []
        L.fp8n_version.restype = ctypes.c_uint32
        L.fp8n_gated_rmsnorm_quant_token.argtypes = [
            P, i64, P, i64, P, i64, i32, i32, f32, ctypes.c_int, P, i64, P, P, P]
        L.fp8n_gated_rmsnorm_quant_token.restype = ctypes.c_int
        L.fp8n_rmsnorm_quant_mx.argtypes = [
            P, i64, P, i32, P, i64, P, i32, i64, f32, P, i64, P, i64, P, i64, P, P]
        L.fp8n_rmsnorm_quant_mx.restype = ctypes.c_int
        L.fp8n_static_head_quant.argtypes = [
            P, P, P, i64, i64, i64, i64, i64, i32, i32, i32, P, P, P, P, i32, P, P, P, P, P]
        L.fp8n_static_head_quant.restype = ctypes.c_int
        L.fp8n_gate_act_bf16.argtypes = [P, i64, ctypes.c_int, P, P]
        L.fp8n_gate_act_bf16.restype = ctypes.c_int
        L.fp8n_convert_f32.argtypes = [P, i64, ctypes.c_int, P, P]
        L.fp8n_convert_f32.restype = ctypes.c_int
        L.fp8n_check_descales.argtypes = [P, i32, P]
        L.fp8n_check_descales.restype = ctypes.c_int
        L.fp8n_gated_rmsnorm_bf16.argtypes = [
            P, i64, P, i64, P, i64, i32, i32, f32, ctypes.c_int, P, i64, P, P]
        L.fp8n_quant_token.argtypes = [P, i64, i64, i32, P, i64, P, P, P]
        L.fp8n_gated_quant_token.argtypes = [P, i64, P, i64, i64, i32, ctypes.c_int, P, i64, P, P, P]
        L.fp8n_rmsnorm_bf16.argtypes = [P, i64, P, i64, i32, f32, P, i64, P, P]
        L.fp8n_quant_mx.argtypes = [P, i64, i64, i32, P, i64, P, i64, P, P]
        L.fp8n_dynamic_head_quant.argtypes = [
            P, P, P, i64, i64, i64, i64, i64, i32, i32, i32, P, P, P, P, P, P, P, P]
        L.fp8n_head_amax.argtypes = [P, i64, i64, i64, i32, i32, P, P]
        L.fp8n_dynamic_head_quant_noalloc.argtypes = [
            P, P, P, i64, i64, i64, i64, i64, i32, i32, i32, P, P, P, P, P, P, P]
        L.fp8n_dynamic_head_quant_noalloc.restype = ctypes.c_int
        L.fp8n_inv_rope_quant_mx.argtypes = [
            P, i64, i64, i32, i32, P, P, i32, i32, i32, ctypes.c_int, P, i64, P, i64, P, P]
        L.fp8n_inv_rope_bf16.argtypes = [
            P, i64, i64, i32, i32, P, P, i32, i32, i32, ctypes.c_int, P, i64, P, P]
        for name in ("fp8n_gated_rmsnorm_bf16", "fp8n_quant_token", "fp8n_gated_quant_token",
                     "fp8n_rmsnorm_bf16", "fp8n_quant_mx", "fp8n_dynamic_head_quant",
                     "fp8n_head_amax", "fp8n_inv_rope_quant_mx", "fp8n_inv_rope_bf16"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(fn: str, code: int) -> None:
    if code != 0:
        msg = lib().fp8n_status_string(code).decode()
        if code == 6:
            msg += " (cudaError %d)" % lib().fp8n_last_cuda_error()
        raise Fp8NormError(fn, code, msg)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtypes, ndim: int) -> None:
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise ValueError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if t.dim() != ndim:
        raise ValueError("%s must have %d dimensions" % (name, ndim))
    if t.stride(-1) != 1:
        raise ValueError("%s must be contiguous in its last dimension" % name)


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_U8 = (torch.uint8, torch.float8_e4m3fn)


def version() -> int:
    return int(lib().fp8n_version())


def fp8n_gated_rmsnorm_quant_token(x, gate, weight, eps: float = 1e-6, act: int = ACT_SIGMOID,
                                   out=None, scale=None, status=None, stream=None):
    """(A) gated RMSNorm + per-token FP8.  x, gate: [T, H, D] bf16 (heads
    contiguous inside a token); weight: [D].  Returns (out uint8 [T, H*D],
    scale float32 [T])."""
    _need(x, "x", _BF16, 3)
    _need(gate, "gate", _BF16, 3)
    _need(weight, "weight", _BF16, 1)
    T, H, D = x.shape
    if gate.shape != x.shape or weight.shape[0] != D:
        raise ValueError("shape mismatch between x, gate and weight")
    for t, n in ((x, "x"), (gate, "gate")):
        if t.stride(1) != D:
            raise ValueError("%s: heads must be contiguous inside a token" % n)
    if out is None:
        out = torch.empty((T, H * D), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((T,), dtype=torch.float32, device=x.device)
    _need(out, "out", _U8, 2)
    _check("fp8n_gated_rmsnorm_quant_token", lib().fp8n_gated_rmsnorm_quant_token(
        _ptr(x), x.stride(0), _ptr(gate), gate.stride(0), _ptr(weight), T, H, D, eps, act,
        _ptr(out), out.stride(0), _ptr(scale), _ptr(status), _stream(stream)))
    return out, scale


def fp8n_rmsnorm_quant_mx(q, q_weight, kv=None, kv_weight=None, eps: float = 1e-6,
                          q_out=None, q_scale=None, kv_out=None, status=None, stream=None):
    """(B) fused q/kv RMSNorm.  q: [M, Nq] bf16, kv: [M, Nkv] bf16.  Returns
    (q_out uint8 [M, Nq], q_scale uint8 E8M0 [M, Nq/32], kv_out bf16 [M, Nkv])."""
    _need(q, "q", _BF16, 2)
    _need(q_weight, "q_weight", _BF16, 1)
    M, Nq = q.shape
    Nkv = 0
    if kv is not None:
        _need(kv, "kv", _BF16, 2)
        _need(kv_weight, "kv_weight", _BF16, 1)
        Nkv = kv.shape[1]
        if kv.shape[0] != M:
            raise ValueError("q and kv must have the same number of rows")
    if q_out is None:
        q_out = torch.empty((M, Nq), dtype=torch.uint8, device=q.device)
    if q_scale is None:
        q_scale = torch.empty((M, Nq // 32), dtype=torch.uint8, device=q.device)
    if kv is not None and kv_out is None:
        kv_out = torch.empty((M, Nkv), dtype=torch.bfloat16, device=q.device)
    _check("fp8n_rmsnorm_quant_mx", lib().fp8n_rmsnorm_quant_mx(
        _ptr(q), q.stride(0), _ptr(q_weight), Nq, _ptr(kv), kv.stride(0) if kv is not None else 0,
        _ptr(kv_weight), Nkv, M, eps, _ptr(q_out), q_out.stride(0), _ptr(q_scale),
        q_scale.stride(0), _ptr(kv_out), kv_out.stride(0) if kv_out is not None else 0,
        _ptr(status), _stream(stream)))
    return q_out, q_scale, kv_out


def fp8n_static_head_quant(q, k, v, q_descale, k_descale, v_descale, cu_seqlens=None,
                           q_out=None, k_out=None, v_out=None, status=None, stream=None):
    """(C) static per-head FP8 of packed Q [T,H,Dqk], K [T,H,Dqk], V [T,H,Dv]
    (bf16) with fp32 descales [H].  Returns (q_out, k_out, v_out) uint8."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, _BF16, 3)
    for t, n in ((q_descale, "q_descale"), (k_descale, "k_descale"), (v_descale, "v_descale")):
        _need(t, n, (torch.float32,), 1)
    T, H, Dqk = q.shape
    Dv = v.shape[2]
    if k.shape != q.shape or v.shape[:2] != (T, H) or k.stride() != q.stride():
        raise ValueError("q and k must share shape and strides; v must match [T, H]")
    outs = []
    for o, d in ((q_out, Dqk), (k_out, Dqk), (v_out, Dv)):
        outs.append(o if o is not None else torch.empty((T, H, d), dtype=torch.uint8, device=q.device))
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", (torch.int32,), 1)
    nseq = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("fp8n_static_head_quant", lib().fp8n_static_head_quant(
        _ptr(q), _ptr(k), _ptr(v), q.stride(0), q.stride(1), v.stride(0), v.stride(1), T, H, Dqk,
        Dv, _ptr(q_descale), _ptr(k_descale), _ptr(v_descale), _ptr(cu_seqlens), nseq,
        _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(status), _stream(stream)))
    return tuple(outs)


def _rope_args(o, positions, cos_sin, rope_dim):
    _need(o, "o", _BF16, 3)
    T, H, D = o.shape
    if o.stride(1) != D:
        raise ValueError("o: heads must be contiguous inside a token")
    if rope_dim > 0:
        _need(positions, "positions", (torch.int32,), 1)
        _need(cos_sin, "cos_sin", (torch.float32,), 2)
        if positions.shape[0] != T or cos_sin.shape[1] != rope_dim or not cos_sin.is_contiguous():
            raise ValueError("positions must be [T] and cos_sin a contiguous [P, rope_dim]")
    P = 0 if cos_sin is None else cos_sin.shape[0]
    return T, H, D, P


def fp8n_inv_rope_quant_mx(o, positions, cos_sin, rope_off: int, rope_dim: int,
                           style: int = ROPE_HALF, out=None, scale=None, status=None, stream=None):
    """Inverse RoPE then MXFP8.  o: [T, H, D] bf16; positions int32 [T];
    cos_sin fp32 [P, rope_dim].  Returns (out uint8 [T, H*D], scale uint8 E8M0
    [T, H*D/32])."""
    T, H, D, P = _rope_args(o, positions, cos_sin, rope_dim)
    if out is None:
        out = torch.empty((T, H * D), dtype=torch.uint8, device=o.device)
    if scale is None:
        scale = torch.empty((T, H * D // 32), dtype=torch.uint8, device=o.device)
    _need(out, "out", _U8, 2)
    _check("fp8n_inv_rope_quant_mx", lib().fp8n_inv_rope_quant_mx(
        _ptr(o), o.stride(0), T, H, D, _ptr(positions), _ptr(cos_sin), P, rope_off, rope_dim,
        style, _ptr(out), out.stride(0), _ptr(scale), scale.stride(0), _ptr(status),
        _stream(stream)))
    return out, scale


def fp8n_inv_rope_bf16(o, positions, cos_sin, rope_off: int, rope_dim: int,
                       style: int = ROPE_HALF, y=None, status=None, stream=None):
    """The inverse-RoPE step alone: bf16 [T, H*D]."""
    T, H, D, P = _rope_args(o, positions, cos_sin, rope_dim)
    if y is None:
        y = torch.empty((T, H * D), dtype=torch.bfloat16, device=o.device)
    _need(y, "y", _BF16, 2)
    _check("fp8n_inv_rope_bf16", lib().fp8n_inv_rope_bf16(
        _ptr(o), o.stride(0), T, H, D, _ptr(positions), _ptr(cos_sin), P, rope_off, rope_dim,
        style, _ptr(y), y.stride(0), _ptr(status), _stream(stream)))
    return y


def fp8n_gate_act_bf16(g, act: int = ACT_SIGMOID, out=None, stream=None):
    """bf16(act(g)) elementwise, correctly rounded.  g: bf16 tensor (any shape,
    contiguous).  Returns a bf16 tensor of the same shape."""
    if not g.is_cuda or g.dtype not in _BF16 or not g.is_contiguous():
        raise ValueError("g must be a contiguous bf16 CUDA tensor")
    if out is None:
        out = torch.empty(g.shape, dtype=torch.bfloat16, device=g.device)
    _check("fp8n_gate_act_bf16", lib().fp8n_gate_act_bf16(
        _ptr(g), g.numel(), act, _ptr(out), _stream(stream)))
    return out


CVT_BF16 = 0
CVT_E4M3 = 1


def fp8n_convert_f32(x, to: int, out=None, stream=None):
    """bf16 (to=CVT_BF16) or E4M3 codes (to=CVT_E4M3, uint8) of each value of a
    contiguous fp32 CUDA tensor, by the kernels' own conversions."""
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16 if to == CVT_BF16 else torch.uint8,
                          device=x.device)
    _check("fp8n_convert_f32", lib().fp8n_convert_f32(_ptr(x), x.numel(), to, _ptr(out),
                                                      _stream(stream)))
    return out


def fp8n_check_descales(descale, stream=None) -> bool:
    """True when every descale is finite and positive (synchronous)."""
    _need(descale, "descale", (torch.float32,), 1)
    code = lib().fp8n_check_descales(_ptr(descale), descale.numel(), _stream(stream))
    if code == 5:
        return False
    _check("fp8n_check_descales", code)
    return True


# ---- the steps of (A) and (B) on their own, dynamic per-head quantisation ----

def fp8n_gated_rmsnorm_bf16(x, gate, weight, eps: float = 1e-6, act: int = ACT_SIGMOID, y=None,
                            status=None, stream=None):
    """(A) without the quantisation.  x, gate: [T, H, D] bf16; returns y bf16 [T, H*D]."""
    _need(x, "x", _BF16, 3)
    _need(gate, "gate", _BF16, 3)
    _need(weight, "weight", _BF16, 1)
    T, H, D = x.shape
    if gate.shape != x.shape or weight.shape[0] != D:
        raise ValueError("shape mismatch between x, gate and weight")
    for t, n in ((x, "x"), (gate, "gate")):
        if t.stride(1) != D:
            raise ValueError("%s: heads must be contiguous inside a token" % n)
    if y is None:
        y = torch.empty((T, H * D), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", _BF16, 2)
    _check("fp8n_gated_rmsnorm_bf16", lib().fp8n_gated_rmsnorm_bf16(
        _ptr(x), x.stride(0), _ptr(gate), gate.stride(0), _ptr(weight), T, H, D, eps, act,
        _ptr(y), y.stride(0), _ptr(status), _stream(stream)))
    return y


def fp8n_quant_token(y, out=None, scale=None, status=None, stream=None):
    """Per-token FP8 of bf16 rows y [T, N].  Returns (out uint8 [T, N], scale float32 [T])."""
    _need(y, "y", _BF16, 2)
    T, N = y.shape
    if out is None:
        out = torch.empty((T, N), dtype=torch.uint8, device=y.device)
    if scale is None:
        scale = torch.empty((T,), dtype=torch.float32, device=y.device)
    _need(out, "out", _U8, 2)
    _check("fp8n_quant_token", lib().fp8n_quant_token(
        _ptr(y), y.stride(0), T, N, _ptr(out), out.stride(0), _ptr(scale), _ptr(status),
        _stream(stream)))
    return out, scale


def fp8n_gated_quant_token(x, gate, act: int = ACT_SIGMOID, out=None, scale=None, status=None,
                           stream=None):
    """y = bf16(x * bf16(act(gate))) on rows [T, N], then per-token FP8.
    Returns (out uint8 [T, N], scale float32 [T])."""
    _need(x, "x", _BF16, 2)
    _need(gate, "gate", _BF16, 2)
    if gate.shape != x.shape:
        raise ValueError("x and gate must have the same shape")
    T, N = x.shape
    if out is None:
        out = torch.empty((T, N), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((T,), dtype=torch.float32, device=x.device)
    _need(out, "out", _U8, 2)
    _check("fp8n_gated_quant_token", lib().fp8n_gated_quant_token(
        _ptr(x), x.stride(0), _ptr(gate), gate.stride(0), T, N, act, _ptr(out), out.stride(0),
        _ptr(scale), _ptr(status), _stream(stream)))
    return out, scale


def fp8n_rmsnorm_bf16(x, weight, eps: float = 1e-6, y=None, status=None, stream=None):
    """Row RMSNorm of bf16 rows x [M, N] with weight [N]: y bf16 [M, N]."""
    _need(x, "x", _BF16, 2)
    _need(weight, "weight", _BF16, 1)
    M, N = x.shape
    if weight.shape[0] != N:
        raise ValueError("weight must have one entry per column")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", _BF16, 2)
    _check("fp8n_rmsnorm_bf16", lib().fp8n_rmsnorm_bf16(
        _ptr(x), x.stride(0), _ptr(weight), M, N, eps, _ptr(y), y.stride(0), _ptr(status),
        _stream(stream)))
    return y


def fp8n_quant_mx(y, out=None, scale=None, status=None, stream=None):
    """MXFP8 of bf16 rows y [M, N] (N % 32 == 0).
    Returns (out uint8 [M, N], scale uint8 E8M0 [M, N/32])."""
    _need(y, "y", _BF16, 2)
    M, N = y.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.uint8, device=y.device)
    if scale is None:
        scale = torch.empty((M, N // 32), dtype=torch.uint8, device=y.device)
    _check("fp8n_quant_mx", lib().fp8n_quant_mx(
        _ptr(y), y.stride(0), M, N, _ptr(out), out.stride(0), _ptr(scale), scale.stride(0),
        _ptr(status), _stream(stream)))
    return out, scale


def fp8n_dynamic_head_quant(q, k, v, workspace=None, descales=None, q_out=None, k_out=None,
                            v_out=None, stream=None):
    """Dynamic per-head FP8 of packed Q [T,H,Dqk], K [T,H,Dqk], V [T,H,Dv] (bf16).
    Returns ((q_descale, k_descale, v_descale) float32 [H] each, (q_out, k_out, v_out))."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, _BF16, 3)
    T, H, Dqk = q.shape
    Dv = v.shape[2]
    if k.shape != q.shape or v.shape[:2] != (T, H) or k.stride() != q.stride():
        raise ValueError("q and k must share shape and strides; v must match [T, H]")
    dev = q.device
    if workspace is None:
        workspace = torch.empty((3 * H,), dtype=torch.int32, device=dev)
    if descales is None:
        descales = tuple(torch.empty((H,), dtype=torch.float32, device=dev) for _ in range(3))
    outs = []
    for o, d in ((q_out, Dqk), (k_out, Dqk), (v_out, Dv)):
        outs.append(o if o is not None else torch.empty((T, H, d), dtype=torch.uint8, device=dev))
    _check("fp8n_dynamic_head_quant", lib().fp8n_dynamic_head_quant(
        _ptr(q), _ptr(k), _ptr(v), q.stride(0), q.stride(1), v.stride(0), v.stride(1), T, H, Dqk,
        Dv, _ptr(workspace), _ptr(descales[0]), _ptr(descales[1]), _ptr(descales[2]),
        _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _stream(stream)))
    return tuple(descales), tuple(outs)


def fp8n_head_amax(x, amax=None, stream=None):
    """Running per-head max |x| of x [T, H, Dh] (bf16) folded into amax float32 [H]
    (zeros when not given).  Returns amax."""
    _need(x, "x", _BF16, 3)
    T, H, Dh = x.shape
    if amax is None:
        amax = torch.zeros((H,), dtype=torch.float32, device=x.device)
    _need(amax, "amax", (torch.float32,), 1)
    _check("fp8n_head_amax", lib().fp8n_head_amax(
        _ptr(x), x.stride(0), x.stride(1), T, H, Dh, _ptr(amax), _stream(stream)))
    return amax


def fp8n_dynamic_head_quant_noalloc(q, k, v, descales=None, q_out=None, k_out=None, v_out=None,
                                    stream=None):
    """fp8n_dynamic_head_quant with the library's static scratch instead of a
    workspace (for callers that cannot allocate device memory; the outputs
    must still be passed or are allocated here by torch).  Calls whose work
    overlaps on the GPU race on the shared scratch."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, _BF16, 3)
    T, H, Dqk = q.shape
    Dv = v.shape[2]
    if k.shape != q.shape or v.shape[:2] != (T, H) or k.stride() != q.stride():
        raise ValueError("q and k must share shape and strides; v must match [T, H]")
    dev = q.device
    if descales is None:
        descales = tuple(torch.empty((H,), dtype=torch.float32, device=dev) for _ in range(3))
    outs = []
    for o, d in ((q_out, Dqk), (k_out, Dqk), (v_out, Dv)):
        outs.append(o if o is not None else torch.empty((T, H, d), dtype=torch.uint8, device=dev))
    _check("fp8n_dynamic_head_quant_noalloc", lib().fp8n_dynamic_head_quant_noalloc(
        _ptr(q), _ptr(k), _ptr(v), q.stride(0), q.stride(1), v.stride(0), v.stride(1), T, H, Dqk,
        Dv, _ptr(descales[0]), _ptr(descales[1]), _ptr(descales[2]), _ptr(outs[0]), _ptr(outs[1]),
        _ptr(outs[2]), _stream(stream)))
    return tuple(descales), tuple(outs)
