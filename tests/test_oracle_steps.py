"""Pins for the oracle's step functions (the unfused pieces of (A) and (B), the
standalone per-token and gated quantisers, the per-head maxima and the dynamic
per-head quant): hand-worked rows, brute force against the exact-rational
checker, and compositions that must reproduce the fused operations."""
import json
import os
import random
from fractions import Fraction

import numpy as np
import pytest

import exact_ref as X
import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def h(s):
    return int(s, 16)


def _rand(rng, n, sigma=1.0, p_out=0.0, scale=1.0):
    out = []
    for _ in range(n):
        a = rng.gauss(0.0, sigma)
        if rng.random() < p_out:
            a *= scale
        out.append(X.bf16_bits(Fraction(a)))
    return out


def test_golden_quant_token_rows():
    g = json.load(open(os.path.join(GOLDEN, "quant_token_rows.json")))
    for case in g["cases"]:
        y = np.array([[h(v) for v in case["y"]]], np.uint16)
        codes, scale = O.quant_token(y)
        assert scale[0].view(np.uint32) == h(case["scale_bits"])
        assert codes[0].tolist() == [h(c) for c in case["codes"]]


@pytest.mark.parametrize("n", [8, 40, 128, 1024])
def test_quant_row_matches_exact(n):
    rng = random.Random(n)
    for _ in range(4):
        y = _rand(rng, n, 1.0, 0.05, 80.0)
        codes, scale = O.quant_token(np.array([y], np.uint16))
        c, s = X.quant_row(y)
        assert codes[0].tolist() == c and Fraction(float(scale[0])) == s


@pytest.mark.parametrize("act,name", [(O.ACT_SIGMOID, "sigmoid"), (O.ACT_SILU, "silu")])
def test_gated_quant_row_matches_exact(act, name):
    rng = random.Random(11 + act)
    for _ in range(3):
        x = _rand(rng, 96, 1.0, 0.05, 30.0)
        gt = _rand(rng, 96, 2.0, 0.05, 40.0)
        y, codes, scale = O.gated_quant_token(np.array([x], np.uint16), np.array([gt], np.uint16), act)
        ye, ce, se = X.gated_quant_row(x, gt, name)
        assert y[0].tolist() == ye and codes[0].tolist() == ce and Fraction(float(scale[0])) == se


def test_fused_gated_equals_its_steps():
    """(A) = per-token quant of the gated RMSNorm output (the sequential path
    the pages check the fused kernel against)."""
    w = synth.workloads()["gated_silu"]
    x, g, wt = w.x(0, 16), w.gate(0, 16), w.weight()
    for act in (O.ACT_SIGMOID, O.ACT_SILU):
        codes, scale = O.gated_rmsnorm_quant_token(x, g, wt, w.eps, act)
        y = O.gated_rmsnorm_bf16(x, g, wt, w.eps, act)
        c2, s2 = O.quant_token(y)
        assert np.array_equal(codes, c2) and np.array_equal(scale, s2)


def test_fused_mx_equals_its_steps():
    """(B) = MX quant of the row RMSNorm of q, and kv = the row RMSNorm of kv."""
    w = synth.workloads()["qkv_mx"]
    q, kv = w.q(0, 12), w.kv(0, 12)
    codes, scales, kv_out = O.rmsnorm_quant_mx(q, w.q_weight(), kv, w.kv_weight(), w.eps)
    yq = O.rmsnorm_bf16(q, w.q_weight(), w.eps)
    c2, s2 = O.quant_mx(yq)
    assert np.array_equal(codes, c2) and np.array_equal(scales, s2)
    assert np.array_equal(kv_out, O.rmsnorm_bf16(kv, w.kv_weight(), w.eps))


def test_rmsnorm_row_matches_exact():
    rng = random.Random(5)
    for n in (8, 40, 512):
        x = _rand(rng, n, 1.4, 0.05, 50.0)
        wt = [X.bf16_bits(1 + X.bf16_to_frac(b)) for b in _rand(rng, n, 0.1)]
        y = O.rmsnorm_bf16(np.array([x], np.uint16), np.array(wt, np.uint16), 1e-6)
        assert y[0].tolist() == X.rmsnorm_row(x, wt, 1e-6)


def test_head_amax_and_dynamic_quant_match_exact():
    rng = random.Random(17)
    T, H, Dh = 5, 3, 16
    x = np.array(_rand(rng, T * H * Dh, 1.0, 0.05, 100.0), np.uint16).reshape(T, H, Dh)
    x[:, 2, :] = x[:, 2, :] & 0x8000                 # head 2: signed zeros only
    amax = O.head_amax(x)
    d, codes = O.dynamic_head_quant(x)
    for hh in range(H):
        vals = x[:, hh, :].reshape(-1).tolist()
        assert Fraction(float(amax[hh])) == X.head_amax(vals)
        de, ce = X.dynamic_quant(vals)
        assert Fraction(float(d[hh])) == de
        assert codes[:, hh, :].reshape(-1).tolist() == ce
    assert d[2] == 0 and set(codes[:, 2, :].reshape(-1).tolist()) <= {0x00, 0x80}


def test_head_amax_is_a_running_max():
    w = synth.StaticHeadWorkload("t", lengths=np.array([4, 6]))
    x = w.tensor("q")
    a1 = O.head_amax(x[:4])
    a2 = O.head_amax(x[4:], a1)
    assert np.array_equal(a2, O.head_amax(x))
    assert np.array_equal(a2, np.abs(O.bf16_to_float(x)).max(axis=(0, 2)))   # numpy's max


def test_dynamic_equals_static_with_its_own_descales():
    w = synth.StaticHeadWorkload("t", lengths=np.array([9]))
    x = w.tensor("k")
    d, codes = O.dynamic_head_quant(x)
    assert np.array_equal(d, (O.head_amax(x) / np.float32(448)).astype(np.float32))
    assert np.array_equal(codes, O.static_head_quant(x, d))
