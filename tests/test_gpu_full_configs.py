"""Whole-workload parity: every output of each of the five workloads.

Each workload runs through the C ABI in one launch, exactly as the benchmark
launches it, and EVERY output element is compared with the oracle on the same
seeded inputs (the oracle runs on row slices over the host's threads; each
slice is the same single-threaded function).  Tolerances are those of
tests/parity.py:
  * E8M0 scale codes, kv bf16 and the static per-head codes: bit-exact;
  * per-token E4M3 codes: one-step differences on at most 1e-4 of the codes;
  * per-token fp32 scales: relative difference <= 1e-6;
  * dequantised values within atol = rtol = 1e-3 outside the one-step set.
The per-token bar comes from "[ROCm][Kimi-K3] Fuse gated RMSNorm with
per-token FP8 for KDA o_proj" (vLLM PR 54254), Tests: the fused kernel is
checked against the sequential steps with the scale exact and the
dequantised values at 1e-3.

The fused gated kernel sums the squares of a head with a compensated sum
instead of the exact one, so in rare heads its mean square is one binary32
unit off.  Every token on which its codes or scale differ from the oracle is
re-run through the oracle with one head's mean square moved by one or two
units in the last place; the test requires each such token to match the GPU
exactly under one of those moves (a difference of summation order and
nothing else).  The counts are printed and, when FP8N_PARITY_RECORD names a
file, appended to it as JSON lines.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import parity as P
import synth

pytestmark = pytest.mark.gpu

B = None
W = synth.workloads()


@pytest.fixture(scope="module", autouse=True)
def lib():
    global B
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from rmsnorm_fp8_activation_gb300 import build
    build.build()
    import rmsnorm_fp8_activation_gb300 as mod
    B = mod
    mod.lib()
    yield


def dev16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def host16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def record(entry: dict) -> None:
    print("parity", json.dumps(entry))
    path = os.environ.get("FP8N_PARITY_RECORD")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(entry) + "\n")


def dequant_chunks(got_c, got_s, want_c, want_s, rows=4096):
    for a in range(0, got_c.shape[0], rows):
        P.compare_dequant(got_c[a:a + rows], got_s[a:a + rows], want_c[a:a + rows],
                          want_s[a:a + rows])


def nudge(v: np.float32, k: int) -> np.float32:
    """v moved by k units in the last place (v > 0)."""
    u = np.array([v], np.float32).view(np.int32)
    return (u + np.int32(k)).view(np.float32)[0]


def explain_token(x_t, g_t, wt, eps, act, got_c, got_s):
    """Whether moving the mean square of one head (or of every head whose
    codes differ, together) by one or two units reproduces the GPU's codes
    and scale exactly.  Returns the moved heads, or None."""
    H, D = x_t.shape
    ms0 = np.array([O.mean_square(x_t[h]) for h in range(H)], np.float32)
    want_c = O.gated_rmsnorm_quant_one(x_t, g_t, wt, eps, act)[1]
    diff_heads = sorted(set((np.nonzero(got_c != want_c)[0] // D).tolist()))
    order = diff_heads + [h for h in range(H) if h not in diff_heads]

    def same(ms):
        _, c, s = O.gated_rmsnorm_quant_one_ms(x_t, g_t, wt, eps, act, ms)
        return np.array_equal(c, got_c) and np.float32(s).view(np.uint32) == got_s.view(np.uint32)

    for h in order:
        for k in (-1, 1, -2, 2):
            ms = ms0.copy()
            if ms[h] > 0:
                ms[h] = nudge(ms0[h], k)
            if same(ms):
                return [(h, k)]
    if 1 < len(diff_heads) <= 4:  # two to four heads off at once: each by one unit
        import itertools
        for ks in itertools.product((-1, 1), repeat=len(diff_heads)):
            ms = ms0.copy()
            for h, k in zip(diff_heads, ks):
                ms[h] = nudge(ms0[h], k)
            if same(ms):
                return list(zip(diff_heads, ks))
    return None


def check_gated_workload(name):
    w = W[name]
    x, g, wt = w.x(), w.gate(), w.weight()
    codes, scale = B.fp8n_gated_rmsnorm_quant_token(dev16(x), dev16(g), dev16(wt), w.eps, w.act)
    torch.cuda.synchronize()
    got_c, got_s = codes.cpu().numpy(), scale.cpu().numpy()
    del codes, scale
    want_c = np.empty_like(got_c)
    want_s = np.empty_like(got_s)

    def run(a, b):
        c, s = O.gated_rmsnorm_quant_token(x[a:b], g[a:b], wt, w.eps, w.act)
        want_c[a:b] = c
        want_s[a:b] = s

    O.sliced(run, w.T, min_slice=64)
    scale_exact = got_s.view(np.uint32) == want_s.view(np.uint32)
    tok_diff = ~scale_exact | (got_c != want_c).any(axis=1)
    bad = np.nonzero(tok_diff)[0]
    explained = 0
    for t in bad:
        if explain_token(x[t], g[t], wt, w.eps, w.act, got_c[t], got_s[t]) is not None:
            explained += 1
    entry = {"workload": name, "tokens": int(w.T), "codes": int(got_c.size),
             "code_diffs": int((got_c != want_c).sum()),
             "tokens_differing": int(bad.size),
             "scales_not_bit_exact": int((~scale_exact).sum()),
             "explained_by_one_ulp_mean_square": explained}
    record(entry)
    assert explained == bad.size, entry
    P.compare_scales(got_s, want_s)
    P.compare_codes(got_c, want_c)
    dequant_chunks(got_c, got_s, want_c, want_s)
    # the amax element of every nonzero token maps to +-448
    assert ((got_c & 0x7F) == 0x7E).any(axis=1)[got_s > 0].all()
    return entry


def test_full_gated_small():
    """56 x 12 x 128, sigmoid (the decode-sized batch)."""
    e = check_gated_workload("gated_small")
    assert e["code_diffs"] == 0 and e["scales_not_bit_exact"] == 0


def test_full_gated_silu():
    """4096 x 32 x 128, silu, 0.5 % outliers x50."""
    check_gated_workload("gated_silu")


def test_full_gated_large():
    """65536 x 64 x 128, sigmoid, 1 % outliers x100 (the benchmark's (A))."""
    check_gated_workload("gated_large")


def test_full_qkv_mx():
    """q [8192, 1536] -> MXFP8, kv [8192, 512] -> bf16, every element."""
    w = W["qkv_mx"]
    q, kv, wq, wkv = w.q(), w.kv(), w.q_weight(), w.kv_weight()
    qo, qs, ko = B.fp8n_rmsnorm_quant_mx(dev16(q), dev16(wq), dev16(kv), dev16(wkv), w.eps)
    torch.cuda.synchronize()
    got_q, got_s, got_k = qo.cpu().numpy(), qs.cpu().numpy(), host16(ko)
    want_q = np.empty_like(got_q)
    want_s = np.empty_like(got_s)
    want_k = np.empty_like(got_k)

    def run(a, b):
        want_q[a:b], want_s[a:b], want_k[a:b] = O.rmsnorm_quant_mx(q[a:b], wq, kv[a:b], wkv, w.eps)

    O.sliced(run, w.M, min_slice=64)
    entry = {"workload": "qkv_mx", "rows": int(w.M),
             "q_code_diffs": int((got_q != want_q).sum()),
             "e8m0_diffs": int((got_s != want_s).sum()),
             "kv_diffs": int((got_k != want_k).sum())}
    record(entry)
    assert np.array_equal(got_s, want_s)        # E8M0: bit-exact
    assert np.array_equal(got_k, want_k)        # kv bf16: bit-exact
    P.compare_codes(got_q, want_q)
    # the exact mean square makes the q codes exact as well
    assert entry["q_code_diffs"] == 0


def test_full_static_head():
    """Q, K [151153, 12, 192], V [151153, 12, 128] with calibrated descales;
    cu_seqlens passed as the benchmark passes it."""
    sw = W["static_head"]
    xs = {k: sw.tensor(k) for k in ("q", "k", "v")}
    ds = sw.descales(xs)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = B.fp8n_static_head_quant(dev16(xs["q"]), dev16(xs["k"]), dev16(xs["v"]),
                                    *(torch.from_numpy(ds[k]).cuda() for k in ("q", "k", "v")),
                                    cu_seqlens=torch.from_numpy(sw.cu_seqlens()).cuda(),
                                    status=status)
    torch.cuda.synchronize()
    entry = {"workload": "static_head", "tokens": int(sw.T)}
    for i, k in enumerate(("q", "k", "v")):
        got = outs[i].cpu().numpy()
        want = np.empty_like(got)

        def run(a, b, k=k, want=want):
            want[a:b] = O.static_head_quant(xs[k][a:b], ds[k])

        O.sliced(run, sw.T, min_slice=256)
        entry[k + "_code_diffs"] = int((got != want).sum())
    entry["status"] = int(status.item())
    record(entry)
    assert entry["q_code_diffs"] == entry["k_code_diffs"] == entry["v_code_diffs"] == 0
    assert entry["status"] == 0
