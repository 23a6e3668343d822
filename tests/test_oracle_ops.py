"""Pins for the oracle's three operations (CPU only).

* hand-worked rows (tests/golden/*.json, each with its citation and derivation);
* brute force on 1-4-row inputs against the independent exact-rational
  checker (tests/exact_ref.py);
* invariants and special cases that reduce to a library routine.
"""
import json
import math
import os
import random
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact_ref as X
import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def h(s):
    return int(s, 16)


def f32_from_bits(u):
    return struct.unpack("<f", struct.pack("<I", u))[0]


def f32_to_bits(f):
    return struct.unpack("<I", struct.pack("<f", f))[0]


ACTS = {"sigmoid": O.ACT_SIGMOID, "silu": O.ACT_SILU}


# ---------------------------------------------------------------------------
# hand-worked rows
# ---------------------------------------------------------------------------

def test_golden_gated_unit_rows():
    g = load("gated_unit_rows.json")
    H, D = g["H"], g["D"]
    x = np.full((1, H, D), 0x3F80, np.uint16)
    gate = np.zeros((1, H, D), np.uint16)
    w = np.array([h(v) for v in g["weight"]], np.uint16)
    codes, scale = O.gated_rmsnorm_quant_token(x, gate, w, g["eps"], ACTS[g["act"]])
    assert f32_to_bits(float(scale[0])) == h(g["scale_bits"][0])
    # the stated bits are also the IEEE quotient 1.5/448 (numpy's binary32 division)
    assert f32_to_bits(float(np.float32(1.5) / np.float32(448))) == h(g["scale_bits"][0])
    want = [h(c) for c in g["codes_per_head"]] * H
    assert codes[0].tolist() == want


def test_golden_gated_constant_rows():
    g = load("gated_constant_rows.json")
    for c in g["cases"]:
        T, H, D = c["T"], c["H"], c["D"]
        x = np.stack([np.full((H, D), h(v), np.uint16) for v in c["x"]])
        gate = np.full((T, H, D), h(c["gate"]), np.uint16)
        w = np.full((D,), h(c["weight"]), np.uint16)
        codes, scale = O.gated_rmsnorm_quant_token(x, gate, w, c["eps"], ACTS[c["act"]])
        for t in range(T):
            assert f32_to_bits(float(scale[t])) == h(c["scale_bits"][t])
            assert (codes[t] == h(c["codes"][t])).all()


def test_golden_mx_unit_rows():
    g = load("mx_unit_rows.json")
    M, Nq, Nkv = g["M"], g["Nq"], g["Nkv"]
    q = np.stack([np.full((Nq,), h(v), np.uint16) for v in g["q_rows"]])
    kv = np.stack([np.full((Nkv,), h(v), np.uint16) for v in g["kv_rows"]])
    wq = np.zeros((Nq,), np.uint16)
    blocks = g["q_weight_blocks"]
    for b, blk in enumerate(blocks):
        if isinstance(blk, str):
            wq[32 * b:32 * b + 32] = h(blk.split()[-1])
        else:
            wq[32 * b:32 * b + len(blk)] = [h(v) for v in blk]
    wkv = np.full((Nkv,), h(g["kv_weight"]), np.uint16)
    codes, scales, kv_out = O.rmsnorm_quant_mx(q, wq, kv, wkv, g["eps"])
    e0 = g["expected_row0"]
    assert scales[0].tolist() == [h(v) for v in e0["scales"]]
    assert codes[0, 0:6].tolist() == [h(v) for v in e0["codes_block0"]]
    assert (codes[0, 6:32] == 0).all()
    assert codes[0, 32:36].tolist() == [h(v) for v in e0["codes_block1"]]
    assert (codes[0, 36:64] == 0).all()
    assert (codes[0, 64:96] == 0x78).all()
    assert (kv_out[0] == 0x3FC0).all()
    # row 1: zeros
    assert scales[1].tolist() == [0, 0, 0]
    neg = (wq & 0x8000) != 0
    assert (codes[1][neg] == 0x80).all() and (codes[1][~neg] == 0x00).all()
    assert (kv_out[1] == 0).all()


def test_golden_static_unit_rows():
    g = load("static_unit_rows.json")
    H, Dh = g["H"], g["Dh"]
    x = np.zeros((1, H, Dh), np.uint16)
    for hh, head in enumerate(g["heads"]):
        x[0, hh, :len(head["x"])] = [h(v) for v in head["x"]]
    d = np.array([f32_from_bits(h(b)) for b in g["descale_bits"]], np.float32)
    codes = O.static_head_quant(x, d)
    for hh, head in enumerate(g["heads"]):
        n = len(head["codes"])
        assert codes[0, hh, :n].tolist() == [h(c) for c in head["codes"]]
        assert (codes[0, hh, n:] == 0).all()


# ---------------------------------------------------------------------------
# brute force against the exact-rational checker
# ---------------------------------------------------------------------------

def _rand_bf16(rng, n, scale=1.0, p_out=0.0, out_scale=1.0):
    v = []
    for _ in range(n):
        a = rng.gauss(0.0, scale)
        if rng.random() < p_out:
            a *= out_scale
        v.append(X.bf16_bits(Fraction(a)))
    return v


@pytest.fixture(scope="module")
def act_tabs():
    return {"sigmoid": X.act_table_exact("sigmoid"), "silu": X.act_table_exact("silu")}


@pytest.mark.parametrize("T,H,D,act", [
    (1, 1, 8, "sigmoid"), (2, 3, 8, "silu"), (3, 2, 32, "sigmoid"),
    (4, 1, 32, "silu"), (1, 2, 128, "sigmoid"), (2, 1, 128, "silu"), (2, 2, 40, "sigmoid"),
])
def test_gated_matches_exact_checker(T, H, D, act, act_tabs):
    rng = random.Random(T * 1000 + H * 100 + D + (act == "silu"))
    for trial in range(3):
        xs = [_rand_bf16(rng, H * D, 1.0, 0.05, 30.0) for _ in range(T)]
        gs = [_rand_bf16(rng, H * D, 2.0, 0.05, 40.0) for _ in range(T)]
        w = _rand_bf16(rng, D, 0.3)
        w = [X.bf16_bits(X.bf16_to_frac(b) + 1) for b in w]
        x = np.array(xs, np.uint16).reshape(T, H, D)
        g = np.array(gs, np.uint16).reshape(T, H, D)
        codes, scale = O.gated_rmsnorm_quant_token(x, g, np.array(w, np.uint16), 1e-6, ACTS[act])
        for t in range(T):
            y, c, s = X.gated_token(xs[t], gs[t], w, H, D, 1e-6, act, act_tabs[act])
            assert Fraction(float(scale[t])) == s
            assert codes[t].tolist() == c, (t, trial)


@pytest.mark.parametrize("H,D,act", [(2, 32, "sigmoid"), (3, 16, "silu"), (1, 128, "sigmoid")])
def test_gated_given_ms_matches_exact_checker(H, D, act, act_tabs):
    """The diagnostic entry that takes each head's mean square as an input:
    with every ms moved by -2..+2 units in the last place (one head at a
    time, and all at once), the oracle's y, codes and scale equal the exact
    checker's with the same ms; with the exact ms it is operation (A)."""
    rng = random.Random(H * 31 + D + (act == "silu"))
    xs = _rand_bf16(rng, H * D, 1.0, 0.05, 30.0)
    gs = _rand_bf16(rng, H * D, 2.0, 0.05, 40.0)
    w = [X.bf16_bits(X.bf16_to_frac(b) + 1) for b in _rand_bf16(rng, D, 0.3)]
    x = np.array(xs, np.uint16).reshape(H, D)
    g = np.array(gs, np.uint16).reshape(H, D)
    wa = np.array(w, np.uint16)
    ms0 = np.array([O.mean_square(x[h]) for h in range(H)], np.float32)
    y0, c0, s0 = O.gated_rmsnorm_quant_one(x, g, wa, 1e-6, ACTS[act])
    y1, c1, s1 = O.gated_rmsnorm_quant_one_ms(x, g, wa, 1e-6, ACTS[act], ms0)
    assert np.array_equal(y0, y1) and np.array_equal(c0, c1) and s0 == s1
    nudges = [(h, k) for h in range(H) for k in (-2, -1, 1, 2)] + [(None, 1)]
    for h, k in nudges:
        ms = ms0.copy()
        sel = slice(None) if h is None else slice(h, h + 1)
        ms[sel] = (ms0[sel].view(np.uint32) + np.uint32(k & 0xFFFFFFFF)).view(np.float32)
        y, c, s = O.gated_rmsnorm_quant_one_ms(x, g, wa, 1e-6, ACTS[act], ms)
        yx, cx, sx = X.gated_token(xs, gs, w, H, D, 1e-6, act, act_tabs[act], ms_given=ms)
        assert y.tolist() == yx and c.tolist() == cx and Fraction(s) == sx, (h, k)


@pytest.mark.parametrize("M,Nq,Nkv", [(1, 32, 8), (2, 64, 40), (3, 96, 64), (4, 32, 0)])
def test_mx_matches_exact_checker(M, Nq, Nkv):
    rng = random.Random(M * 7 + Nq + Nkv)
    for trial in range(3):
        q = [_rand_bf16(rng, Nq, 1.4, 0.05, 50.0) for _ in range(M)]
        kv = [_rand_bf16(rng, Nkv, 1.4) for _ in range(M)]
        wq = [X.bf16_bits(1 + X.bf16_to_frac(b)) for b in _rand_bf16(rng, Nq, 0.1)]
        wkv = [X.bf16_bits(1 + X.bf16_to_frac(b)) for b in _rand_bf16(rng, Nkv, 0.1)]
        codes, scales, kv_out = O.rmsnorm_quant_mx(
            np.array(q, np.uint16).reshape(M, Nq), np.array(wq, np.uint16),
            np.array(kv, np.uint16).reshape(M, Nkv), np.array(wkv, np.uint16), 1e-6)
        for m in range(M):
            yq = X.rmsnorm_row(q[m], wq, 1e-6)
            for b in range(Nq // 32):
                sc, cs = X.mx_block(yq[32 * b:32 * b + 32])
                assert scales[m, b] == sc
                assert codes[m, 32 * b:32 * b + 32].tolist() == cs
            if Nkv:
                assert kv_out[m].tolist() == X.rmsnorm_row(kv[m], wkv, 1e-6)


@pytest.mark.parametrize("T,H,Dh", [(1, 1, 8), (3, 2, 24), (4, 3, 16)])
def test_static_matches_exact_checker(T, H, Dh):
    rng = random.Random(T + H + Dh)
    x = _rand_bf16(rng, T * H * Dh, 1.0, 0.05, 100.0)
    d = np.array([rng.uniform(0.001, 0.01) for _ in range(H)], np.float32)
    codes = O.static_head_quant(np.array(x, np.uint16).reshape(T, H, Dh), d)
    for t in range(T):
        for hh in range(H):
            seg = x[(t * H + hh) * Dh:(t * H + hh + 1) * Dh]
            assert codes[t, hh].tolist() == X.static_quant(seg, float(d[hh]))


# ---------------------------------------------------------------------------
# invariants on workload-shaped inputs
# ---------------------------------------------------------------------------

def _small_gated(T=48):
    w = synth.workloads()["gated_silu"]
    return w, w.x(0, T), w.gate(0, T), w.weight()


def test_gated_invariants():
    w, x, g, wt = _small_gated()
    for act in (O.ACT_SIGMOID, O.ACT_SILU):
        codes, scale = O.gated_rmsnorm_quant_token(x, g, wt, w.eps, act)
        mag = codes & 0x7F
        assert (mag <= 0x7E).all()                           # |q| <= 448, no NaN code
        for t in range(x.shape[0]):
            y, c1, s1 = O.gated_rmsnorm_quant_one(x[t], g[t], wt, w.eps, act)
            assert c1.tolist() == codes[t].tolist() and s1 == scale[t]
            yf = O.bf16_to_float(y).astype(np.float64)
            amax = np.abs(yf).max()
            assert scale[t] == np.float32(amax) / np.float32(448)
            # the token's largest |y| maps to exactly +-448
            assert set((codes[t][np.abs(yf) == amax] & 0x7F).tolist()) == {0x7E}
            # sign(q) = sign(y) wherever q is not zero
            nz = mag[t] != 0
            assert ((codes[t][nz] & 0x80) != 0).tolist() == (yf[nz] < 0).tolist()
            # dequantised value within half an E4M3 step of y
            deq = np.array([O.e4m3_to_double(c) for c in codes[t]]) * float(scale[t])
            tol = np.maximum(np.abs(yf) * 2.0 ** -4, float(scale[t]) * 2.0 ** -10) * 1.0001
            assert (np.abs(deq - yf) <= tol).all()


def test_gated_norm_matches_torch_rms_norm():
    """With sigmoid(gate) = 1 (gate = 100) y is the RMSNorm of x times the
    weight; torch.nn.functional.rms_norm in fp32 agrees within the bf16
    roundings (two of 2^-8 relative)."""
    w, x, _, wt = _small_gated(8)
    gate = np.full_like(x, 0x42C8)                              # 100.0
    xt = torch.from_numpy(O.bf16_to_float(x).copy())
    wtt = torch.from_numpy(O.bf16_to_float(wt).copy())
    ref = torch.nn.functional.rms_norm(xt, (x.shape[2],), wtt, eps=w.eps).numpy()
    for t in range(x.shape[0]):
        y, _, _ = O.gated_rmsnorm_quant_one(x[t], gate[t], wt, w.eps, O.ACT_SIGMOID)
        yf = O.bf16_to_float(y).reshape(ref[t].shape)
        assert np.allclose(yf, ref[t], rtol=2.0 ** -7, atol=1e-30)


def test_constant_head_closed_form():
    """A head with x = c everywhere has ms = c^2 exactly and r =
    RN32(1/RN32(sqrt(RN32(c^2 + eps))))."""
    for c in (0x3F80, 0x4040, 0x3E4D, 0xC2C8, 0x0081):
        cf = float(X.bf16_to_frac(c))
        ms = O.mean_square(np.full(128, c, np.uint16))
        assert ms == np.float32(cf * cf) == cf * cf
        v = np.float32(ms) + np.float32(1e-6)
        r = np.float32(1.0) / np.sqrt(v)
        assert O.rms_factor(ms, 1e-6) == r


def test_mx_invariants():
    mw = synth.workloads()["qkv_mx"]
    q, kv = mw.q(0, 16), mw.kv(0, 16)
    codes, scales, kv_out = O.rmsnorm_quant_mx(q, mw.q_weight(), kv, mw.kv_weight(), mw.eps)
    assert ((codes & 0x7F) <= 0x7E).all()
    for m in range(q.shape[0]):
        for b in range(q.shape[1] // 32):
            blk = codes[m, 32 * b:32 * b + 32]
            mx = max(O.e4m3_to_double(c & 0x7F) for c in blk)
            assert 256.0 <= mx <= 448.0                         # the block max sits in the top binade


def test_static_invariants():
    sw = synth.StaticHeadWorkload("t", lengths=np.array([3, 5]))
    xs = {k: sw.tensor(k) for k in ("q", "k", "v")}
    d = sw.descales(xs)
    for k in ("q", "k", "v"):
        codes = O.static_head_quant(xs[k], d[k])
        xf = O.bf16_to_float(xs[k]).astype(np.float32)
        q = (xf / d[k][None, :, None]).astype(np.float32)
        assert (np.abs(q) <= 448.0).all()                       # descale >= amax/448: no clipping
        ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes, ref)                       # in range: torch's cast agrees
