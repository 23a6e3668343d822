"""The C ABI on a CPU-only machine: the library builds, loads and exports every
entry point declared in include/fp8norm.h, and argument validation returns
its status codes before any CUDA call is made (no compute without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8norm.h")


@pytest.fixture(scope="module")
def L():
    from rmsnorm_fp8_activation_gb300 import build
    path = build.build()
    import rmsnorm_fp8_activation_gb300 as B
    assert path == B.LIB_PATH
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8n_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("fp8n_gated_rmsnorm_quant_token", "fp8n_rmsnorm_quant_mx",
              "fp8n_static_head_quant", "fp8n_check_descales", "fp8n_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(7):
        s = L.fp8n_status_string(code).decode()
        assert s.startswith("FP8N_")
    assert L.fp8n_version() == 0x000200


# Validation paths return before touching the device.
OK, NULL, SHAPE, MISALIGNED, UNSUPPORTED = 0, 1, 2, 3, 4
P16 = 0x10000  # a 16-byte aligned fake address, never dereferenced


def gated(L, **kw):
    a = dict(x=P16, xs=4096, g=P16, gs=4096, w=P16, T=4, H=32, D=128, eps=1e-6, act=0,
             out=P16, os=4096, sc=P16, st=None)
    a.update(kw)
    return L.fp8n_gated_rmsnorm_quant_token(a["x"], a["xs"], a["g"], a["gs"], a["w"], a["T"],
                                            a["H"], a["D"], a["eps"], a["act"], a["out"],
                                            a["os"], a["sc"], a["st"], None)


def test_gated_validation(L):
    assert gated(L, T=0) == OK                      # empty: no launch
    assert gated(L, T=-1) == SHAPE
    assert gated(L, D=12) == UNSUPPORTED            # D not a multiple of 8
    assert gated(L, D=16384, H=1) == UNSUPPORTED    # D > 8192
    assert gated(L, H=256, D=128) == UNSUPPORTED    # H*D > 16384
    assert gated(L, act=7) == UNSUPPORTED
    assert gated(L, eps=float("nan")) == UNSUPPORTED
    assert gated(L, eps=-1.0) == UNSUPPORTED
    assert gated(L, xs=100) == SHAPE                # stride below the row
    assert gated(L, x=None) == NULL
    assert gated(L, sc=None) == NULL
    assert gated(L, x=P16 + 8) == MISALIGNED
    assert gated(L, xs=4100) == MISALIGNED
    assert gated(L, os=4100) == MISALIGNED


def mx(L, **kw):
    a = dict(q=P16, qs=1536, qw=P16, Nq=1536, kv=P16, ks=512, kw=P16, Nkv=512, M=8, eps=1e-6,
             qo=P16, qos=1536, qsc=P16, qscs=48, ko=P16, kos=512)
    a.update(kw)
    return L.fp8n_rmsnorm_quant_mx(a["q"], a["qs"], a["qw"], a["Nq"], a["kv"], a["ks"], a["kw"],
                                   a["Nkv"], a["M"], a["eps"], a["qo"], a["qos"], a["qsc"],
                                   a["qscs"], a["ko"], a["kos"], None, None)


def test_mx_validation(L):
    assert mx(L, M=0) == OK
    assert mx(L, Nq=48) == UNSUPPORTED               # not a multiple of 32
    assert mx(L, Nkv=12) == UNSUPPORTED
    assert mx(L, qscs=10) == SHAPE
    assert mx(L, q=None) == NULL
    assert mx(L, kv=None) == NULL
    assert mx(L, kv=None, kw=None, ko=None, Nkv=0, M=0) == OK
    assert mx(L, qo=P16 + 4) == MISALIGNED


def static(L, **kw):
    a = dict(q=P16, k=P16, v=P16, qts=2304, qhs=192, vts=1536, vhs=128, T=10, H=12, Dqk=192,
             Dv=128, qd=P16, kd=P16, vd=P16, qo=P16, ko=P16, vo=P16)
    a.update(kw)
    return L.fp8n_static_head_quant(a["q"], a["k"], a["v"], a["qts"], a["qhs"], a["vts"],
                                    a["vhs"], a["T"], a["H"], a["Dqk"], a["Dv"], a["qd"],
                                    a["kd"], a["vd"], None, 0, a["qo"], a["ko"], a["vo"], None,
                                    None)


def test_static_validation(L):
    assert static(L, T=0) == OK
    assert static(L, H=300) == UNSUPPORTED
    assert static(L, Dqk=100) == UNSUPPORTED
    assert static(L, T=1 << 30) == UNSUPPORTED       # beyond 2^31 chunks
    assert static(L, qhs=64) == SHAPE
    assert static(L, vd=None) == NULL
    assert static(L, qd=P16 + 2) == MISALIGNED
    assert static(L, qhs=196) == MISALIGNED


def test_gate_act_and_check_validation(L):
    assert L.fp8n_gate_act_bf16(P16, 0, 0, P16, None) == OK
    assert L.fp8n_gate_act_bf16(P16, -1, 0, P16, None) == SHAPE
    assert L.fp8n_gate_act_bf16(None, 4, 0, P16, None) == NULL
    assert L.fp8n_gate_act_bf16(P16 + 1, 4, 0, P16, None) == MISALIGNED
    assert L.fp8n_check_descales(P16, 0, None) == SHAPE
    assert L.fp8n_check_descales(None, 4, None) == NULL


def test_convert_validation(L):
    assert L.fp8n_convert_f32(P16, 0, 0, P16, None) == OK
    assert L.fp8n_convert_f32(P16, -1, 0, P16, None) == SHAPE
    assert L.fp8n_convert_f32(P16, 4, 2, P16, None) == UNSUPPORTED
    assert L.fp8n_convert_f32(None, 4, 1, P16, None) == NULL
    assert L.fp8n_convert_f32(P16, 4, 1, None, None) == NULL
    assert L.fp8n_convert_f32(P16 + 2, 4, 1, P16, None) == MISALIGNED
    assert L.fp8n_convert_f32(P16, 4, 0, P16 + 1, None) == MISALIGNED


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import rmsnorm_fp8_activation_gb300 as B
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        B.lib()


def test_step_entry_points_validation(L):
    # per-token quantisation of bf16 rows
    assert L.fp8n_quant_token(P16, 4096, 0, 4096, P16, 4096, P16, None, None) == OK
    assert L.fp8n_quant_token(P16, 4096, 3, 12, P16, 4096, P16, None, None) == UNSUPPORTED
    assert L.fp8n_quant_token(P16, 4096, 3, 16392, P16, 16392, P16, None, None) == UNSUPPORTED
    assert L.fp8n_quant_token(P16, 132, 3, 128, P16, 128, P16, None, None) == MISALIGNED
    assert L.fp8n_quant_token(P16, 64, 3, 128, P16, 128, P16, None, None) == SHAPE
    assert L.fp8n_quant_token(None, 128, 3, 128, P16, 128, P16, None, None) == NULL
    assert L.fp8n_quant_token(P16, 128, 3, 128, P16, 128, None, None, None) == NULL
    assert L.fp8n_quant_token(P16, 128, 3, 128, P16, 132, P16, None, None) == MISALIGNED
    # gate product + quantisation
    g = L.fp8n_gated_quant_token
    assert g(P16, 128, P16, 128, 3, 128, 2, P16, 128, P16, None, None) == UNSUPPORTED
    assert g(P16, 128, None, 128, 3, 128, 0, P16, 128, P16, None, None) == NULL
    assert g(P16, 128, P16 + 8, 128, 3, 128, 1, P16, 128, P16, None, None) == MISALIGNED
    assert g(P16, 128, P16, 120, 3, 128, 1, P16, 128, P16, None, None) == SHAPE
    # gated norm to bf16
    n = L.fp8n_gated_rmsnorm_bf16
    assert n(P16, 512, P16, 512, P16, 0, 4, 128, 1e-6, 0, P16, 512, None, None) == OK
    assert n(P16, 512, P16, 512, P16, 2, 4, 128, 1e-6, 0, P16, 500, None, None) == SHAPE
    assert n(P16, 512, P16, 512, P16, 2, 4, 128, 1e-6, 0, None, 512, None, None) == NULL
    assert n(P16, 512, P16, 512, P16, 2, 4, 128, float("inf"), 0, P16, 512, None, None) == UNSUPPORTED
    assert n(P16, 512, P16, 512, P16, 2, 4, 12, 1e-6, 0, P16, 512, None, None) == UNSUPPORTED
    # row RMSNorm to bf16 and MX quantisation
    assert L.fp8n_rmsnorm_bf16(P16, 512, P16, 0, 512, 1e-6, P16, 512, None, None) == OK
    assert L.fp8n_rmsnorm_bf16(P16, 512, P16, 4, 500, 1e-6, P16, 512, None, None) == UNSUPPORTED
    assert L.fp8n_rmsnorm_bf16(P16, 512, None, 4, 512, 1e-6, P16, 512, None, None) == NULL
    assert L.fp8n_rmsnorm_bf16(P16, 512, P16, 4, 512, 1e-6, P16 + 4, 512, None, None) == MISALIGNED
    assert L.fp8n_quant_mx(P16, 512, 0, 512, P16, 512, P16, 16, None, None) == OK
    assert L.fp8n_quant_mx(P16, 512, 4, 520, P16, 520, P16, 17, None, None) == UNSUPPORTED
    assert L.fp8n_quant_mx(P16, 512, 4, 512, P16, 512, P16, 15, None, None) == SHAPE
    assert L.fp8n_quant_mx(P16, 512, 4, 512, P16, 512, None, 16, None, None) == NULL


def test_dynamic_and_amax_validation(L):
    def dyn(**kw):
        a = dict(q=P16, k=P16, v=P16, qts=2304, qhs=192, vts=1536, vhs=128, T=10, H=12, Dqk=192,
                 Dv=128, ws=P16, qd=P16, kd=P16, vd=P16, qo=P16, ko=P16, vo=P16)
        a.update(kw)
        return L.fp8n_dynamic_head_quant(a["q"], a["k"], a["v"], a["qts"], a["qhs"], a["vts"],
                                         a["vhs"], a["T"], a["H"], a["Dqk"], a["Dv"], a["ws"],
                                         a["qd"], a["kd"], a["vd"], a["qo"], a["ko"], a["vo"], None)
    assert dyn(T=0) == OK
    assert dyn(H=257) == UNSUPPORTED
    assert dyn(ws=None) == NULL
    assert dyn(kd=None) == NULL
    assert dyn(ws=P16 + 2) == MISALIGNED
    assert dyn(vhs=120) == SHAPE
    assert L.fp8n_head_amax(P16, 2304, 192, 0, 12, 192, P16, None) == OK
    assert L.fp8n_head_amax(P16, 2304, 192, 10, 12, 196, P16, None) == UNSUPPORTED
    assert L.fp8n_head_amax(P16, 2304, 100, 10, 12, 192, P16, None) == SHAPE
    assert L.fp8n_head_amax(P16, 2304, 192, 10, 12, 192, None, None) == NULL
    assert L.fp8n_head_amax(P16 + 8, 2304, 192, 10, 12, 192, P16, None) == MISALIGNED


def test_inv_rope_validation(L):
    def rope(fn="q", **kw):
        a = dict(o=P16, os=9216, T=10, H=16, D=576, pos=P16, cs=P16, P=4096, off=512, R=64,
                 style=0, out=P16, ost=9216, sc=P16, sst=288, st=None)
        a.update(kw)
        if fn == "q":
            return L.fp8n_inv_rope_quant_mx(a["o"], a["os"], a["T"], a["H"], a["D"], a["pos"],
                                            a["cs"], a["P"], a["off"], a["R"], a["style"],
                                            a["out"], a["ost"], a["sc"], a["sst"], a["st"], None)
        return L.fp8n_inv_rope_bf16(a["o"], a["os"], a["T"], a["H"], a["D"], a["pos"], a["cs"],
                                    a["P"], a["off"], a["R"], a["style"], a["out"], a["ost"],
                                    a["st"], None)
    assert rope(T=0) == OK and rope("y", T=0) == OK
    assert rope(D=560) == UNSUPPORTED                  # D not a multiple of 32
    assert rope(off=516) == UNSUPPORTED                # span start not on a chunk
    assert rope(R=56) == UNSUPPORTED                   # span not whole chunk pairs
    assert rope(off=544, R=64) == UNSUPPORTED          # span past the head
    assert rope(style=2) == UNSUPPORTED
    assert rope(T=1 << 30) == UNSUPPORTED              # beyond 2^31 MX blocks
    assert rope(os=9000) == SHAPE
    assert rope(sst=287) == SHAPE
    assert rope(P=0) == SHAPE
    assert rope(pos=None) == NULL and rope(cs=None) == NULL and rope(sc=None) == NULL
    assert rope(cs=P16 + 4) == MISALIGNED
    assert rope(ost=9224) == MISALIGNED                # code rows of 16-byte multiples
    assert rope(os=9220) == MISALIGNED
    assert rope("y", out=P16 + 8) == MISALIGNED
    assert rope("y", ost=9000) == SHAPE
