"""Seeded synthetic inputs of the workloads (no method arithmetic here).

Every tensor is drawn from a counter-based Philox4x32-10 generator (Salmon,
Moraes, Dror, Shaw: "Parallel random numbers: as easy as 1, 2, 3", SC'11), with
key (seed, stream id) and counter = block index, so any slice of any tensor can
be regenerated on its own.  Normals come from the Box-Muller transform in
double precision and are rounded to bf16 (through binary32, round-to-nearest-
even at both steps).  The same arrays feed the CUDA library and the oracle.

The generator runs in ``gen.c`` (built into ``libsynth.so``), called from a
thread pool; ``philox4x32_10`` below is a numpy restatement of the same block
function, kept to cross-check the C words.

Workloads (sizes and distributions of the normalize-then-quantize path):
  gated_small   x, gate [56, 12, 128] ~ N(0,1); weight 1 + 0.1 N; eps 1e-6; sigmoid
  gated_silu    x, gate [4096, 32, 128] ~ N(0,1), each element independently x50
                with probability 0.005; weight 1 + 0.1 N; eps 1e-6; silu
  qkv_mx        q [8192, 1536], kv [8192, 512] ~ N(0, 2) (variance 2);
                weights 1 + 0.1 N; eps 1e-6
  static_head   16 sequence lengths uniform in [1024, 16384]; Q, K [T, 12, 192],
                V [T, 12, 128] ~ N(0,1); descale[h] = amax_h / 448 * U(1, 1.2)
  gated_large   x, gate [65536, 64, 128] ~ N(0,1), each element x100 with
                probability 0.01; weight 1 + 0.1 N; eps 1e-6; sigmoid
  inv_rope_mx   o [4096, 16, 576] ~ N(0,1), RoPE on the last 64 dims of each head
                (rotate-half), positions uniform in [0, 4096), the FP32 cos/sin
                cache [4096, 64] of base 10000
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_MASK = np.uint64(0xFFFFFFFF)
_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85


def philox4x32_10(ctr: np.ndarray, key0: int, key1: int) -> np.ndarray:
    """Philox4x32 with 10 rounds.  ctr: uint64 [n, 4] holding 32-bit words.

    Returns uint64 [n, 4] of 32-bit outputs.
    """
    c0, c1, c2, c3 = (ctr[:, i].astype(np.uint64) for i in range(4))
    k0, k1 = key0 & 0xFFFFFFFF, key1 & 0xFFFFFFFF
    for _ in range(10):
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0
        k0 = (k0 + _W0) & 0xFFFFFFFF
        k1 = (k1 + _W1) & 0xFFFFFFFF
    return np.stack([c0, c1, c2, c3], axis=1)


_lib = None


def _L():
    global _lib
    if _lib is None:
        import ctypes
        from . import build as _build
        L = ctypes.CDLL(_build.build())
        u32, i64, u64, f64, P = (ctypes.c_uint32, ctypes.c_int64, ctypes.c_uint64,
                                 ctypes.c_double, ctypes.c_void_p)
        L.synth_philox_words.argtypes = [u32, u32, u64, i64, P]
        L.synth_uniform.argtypes = [u32, u32, i64, i64, P]
        L.synth_bf16_normal.argtypes = [u32, u32, i64, i64, f64, f64, f64, f64, P]
        for f in (L.synth_philox_words, L.synth_uniform, L.synth_bf16_normal):
            f.restype = None
        _lib = L
    return _lib


def philox_words(key0: int, key1: int, block0: int, nblocks: int) -> np.ndarray:
    """uint32 [nblocks, 4] words of blocks block0.. from the C generator."""
    out = np.empty((nblocks, 4), dtype=np.uint32)
    _L().synth_philox_words(key0, key1, block0, nblocks, out.ctypes.data)
    return out


def uniform(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Elements [start, start+n) of a uniform (0,1) stream, float64."""
    out = np.empty((max(n, 0),), dtype=np.float64)
    if n > 0:
        _L().synth_uniform(seed, stream, start, n, out.ctypes.data)
    return out


_CHUNK = 1 << 22


def _pool_map(fn, n: int):
    chunks = [(s, min(_CHUNK, n - s)) for s in range(0, n, _CHUNK)]
    if len(chunks) <= 1:
        return [fn(s, c) for s, c in chunks]
    workers = min(len(chunks), os.cpu_count() or 1, 64)
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(lambda sc: fn(*sc), chunks))


def bf16_normal(seed: int, stream: int, n: int, sigma: float = 1.0, mean: float = 0.0,
                outlier_p: float = 0.0, outlier_scale: float = 1.0,
                start: int = 0) -> np.ndarray:
    """bf16 bits of mean + sigma * N(0,1), optionally with outliers.

    An element is multiplied by outlier_scale when an independent uniform
    (stream + 0x10000) is below outlier_p."""
    out = np.empty((n,), dtype=np.uint16)
    L = _L()
    base = out.ctypes.data

    def fill(s, c):  # ctypes drops the GIL for the call
        L.synth_bf16_normal(seed, stream, start + s, c, mean, sigma, outlier_p,
                            outlier_scale, base + 2 * s)

    _pool_map(fill, n)
    return out


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

ACT_SIGMOID = 0
ACT_SILU = 1


@dataclass
class GatedWorkload:
    name: str
    T: int
    H: int
    D: int
    act: int
    eps: float = 1e-6
    outlier_p: float = 0.0
    outlier_scale: float = 1.0
    seed: int = 0
    stream_base: int = 0

    @property
    def elements(self) -> int:
        return self.T * self.H * self.D

    def x(self, start_token: int = 0, n_tokens: int | None = None) -> np.ndarray:
        return self._tensor(1, start_token, n_tokens)

    def gate(self, start_token: int = 0, n_tokens: int | None = None) -> np.ndarray:
        return self._tensor(2, start_token, n_tokens)

    def weight(self) -> np.ndarray:
        return bf16_normal(self.seed, self.stream_base + 3, self.D, sigma=0.1, mean=1.0)

    def _tensor(self, tid: int, start_token: int, n_tokens: int | None) -> np.ndarray:
        if n_tokens is None:
            n_tokens = self.T - start_token
        row = self.H * self.D
        v = bf16_normal(self.seed, self.stream_base + tid, n_tokens * row,
                        outlier_p=self.outlier_p, outlier_scale=self.outlier_scale,
                        start=start_token * row)
        return v.reshape(n_tokens, self.H, self.D)

    def algorithmic_bytes(self) -> int:
        # read x and gate (2 B each), write e4m3 (1 B) per element; weight; scales
        return 5 * self.elements + 2 * self.D + 4 * self.T


@dataclass
class MxWorkload:
    name: str
    M: int
    Nq: int
    Nkv: int
    eps: float = 1e-6
    sigma: float = float(np.sqrt(2.0))
    seed: int = 0
    stream_base: int = 0

    def q(self, start_row: int = 0, n_rows: int | None = None) -> np.ndarray:
        return self._rows(1, self.Nq, start_row, n_rows)

    def kv(self, start_row: int = 0, n_rows: int | None = None) -> np.ndarray:
        return self._rows(2, self.Nkv, start_row, n_rows)

    def q_weight(self) -> np.ndarray:
        return bf16_normal(self.seed, self.stream_base + 3, self.Nq, sigma=0.1, mean=1.0)

    def kv_weight(self) -> np.ndarray:
        return bf16_normal(self.seed, self.stream_base + 4, self.Nkv, sigma=0.1, mean=1.0)

    def _rows(self, tid: int, n: int, start_row: int, n_rows: int | None) -> np.ndarray:
        if n_rows is None:
            n_rows = self.M - start_row
        v = bf16_normal(self.seed, self.stream_base + tid, n_rows * n, sigma=self.sigma,
                        start=start_row * n)
        return v.reshape(n_rows, n)

    def algorithmic_bytes(self) -> int:
        q = self.M * self.Nq * (2 + 1) + self.M * (self.Nq // 32)
        kv = self.M * self.Nkv * (2 + 2)
        return q + kv + 2 * (self.Nq + self.Nkv)


@dataclass
class StaticHeadWorkload:
    name: str
    num_seqs: int = 16
    len_lo: int = 1024
    len_hi: int = 16384
    H: int = 12
    Dqk: int = 192
    Dv: int = 128
    seed: int = 0
    stream_base: int = 0
    lengths: np.ndarray = field(default=None)  # type: ignore[assignment]

    def __post_init__(self):
        if self.lengths is None:
            u = uniform(self.seed, self.stream_base + 9, 0, self.num_seqs)
            span = self.len_hi - self.len_lo + 1
            self.lengths = (self.len_lo + np.floor(u * span)).astype(np.int64)
        self.lengths = np.asarray(self.lengths, dtype=np.int64)

    @property
    def T(self) -> int:
        return int(self.lengths.sum())

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    def tensor(self, which: str, start_token: int = 0, n_tokens: int | None = None) -> np.ndarray:
        tid = {"q": 1, "k": 2, "v": 3}[which]
        d = self.Dv if which == "v" else self.Dqk
        if n_tokens is None:
            n_tokens = self.T - start_token
        row = self.H * d
        v = bf16_normal(self.seed, self.stream_base + tid, n_tokens * row, start=start_token * row)
        return v.reshape(n_tokens, self.H, d)

    def descales(self, tensors: dict[str, np.ndarray]) -> dict[str, np.ndarray]:
        """descale[h] = fp32(amax over the data of head h / 448 * U(1, 1.2))."""
        out = {}
        for i, which in enumerate(("q", "k", "v")):
            x = tensors[which]
            f = (x.astype(np.uint32) << 16).view(np.float32)
            amax = np.abs(f).max(axis=(0, 2)).astype(np.float64)
            u = uniform(self.seed, self.stream_base + 10 + i, 0, self.H)
            out[which] = (amax / 448.0 * (1.0 + 0.2 * u)).astype(np.float32)
        return out

    def algorithmic_bytes(self) -> int:
        per_tok = self.H * (2 * self.Dqk + self.Dv) * 3
        return self.T * per_tok + 3 * 4 * self.H


@dataclass
class InvRopeWorkload:
    """The o-projection input: attention output o [T, H, D] ~ N(0, 1) whose
    span [rope_off, rope_off + rope_dim) of every head carries RoPE, token
    positions uniform in [0, P), and the FP32 cos/sin cache [P, rope_dim] of
    the angles p * base^(-2i / rope_dim) (cos of the rope_dim/2 angles, then
    their sin), computed in double and rounded to binary32.  The cache is an
    input of the operation, as a layer holds it."""
    name: str
    T: int = 4096
    H: int = 16
    D: int = 576
    rope_off: int = 512
    rope_dim: int = 64
    interleaved: bool = False
    P: int = 4096
    base: float = 10000.0
    seed: int = 0
    stream_base: int = 0

    def o(self, start_token: int = 0, n_tokens: int | None = None) -> np.ndarray:
        if n_tokens is None:
            n_tokens = self.T - start_token
        row = self.H * self.D
        v = bf16_normal(self.seed, self.stream_base + 1, n_tokens * row, start=start_token * row)
        return v.reshape(n_tokens, self.H, self.D)

    def positions(self) -> np.ndarray:
        u = uniform(self.seed, self.stream_base + 2, 0, self.T)
        return np.minimum(np.floor(u * self.P), self.P - 1).astype(np.int32)

    def cos_sin(self) -> np.ndarray:
        half = self.rope_dim // 2
        theta = self.base ** (-2.0 * np.arange(half, dtype=np.float64) / self.rope_dim)
        ang = np.arange(self.P, dtype=np.float64)[:, None] * theta[None, :]
        return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)

    def algorithmic_bytes(self) -> int:
        # read o (2 B), write e4m3 (1 B) per element and one E8M0 byte per 32;
        # positions and the cos/sin cache once
        n = self.T * self.H * self.D
        return 3 * n + n // 32 + 4 * self.T + 4 * self.P * self.rope_dim


def workloads(seed: int = 0) -> dict:
    """The five workloads, keyed by name, with independent stream ranges."""
    return {
        "gated_small": GatedWorkload("gated_small", 56, 12, 128, ACT_SIGMOID, seed=seed,
                                     stream_base=0x100),
        "gated_silu": GatedWorkload("gated_silu", 4096, 32, 128, ACT_SILU, outlier_p=0.005,
                                    outlier_scale=50.0, seed=seed, stream_base=0x200),
        "qkv_mx": MxWorkload("qkv_mx", 8192, 1536, 512, seed=seed, stream_base=0x300),
        "static_head": StaticHeadWorkload("static_head", seed=seed, stream_base=0x400),
        "gated_large": GatedWorkload("gated_large", 65536, 64, 128, ACT_SIGMOID,
                                     outlier_p=0.01, outlier_scale=100.0, seed=seed,
                                     stream_base=0x500),
        "inv_rope_mx": InvRopeWorkload("inv_rope_mx", seed=seed, stream_base=0x600),
    }
