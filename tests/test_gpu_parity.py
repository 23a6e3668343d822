"""GPU parity: the CUDA kernels (through the C ABI) against the oracle on the
same seeded inputs, element by element.  Sizes span several CTAs and a ragged
tail; the full-size workloads are checked on sampled tokens/rows in the launch
configuration the benchmark times."""
import numpy as np
import pytest
import torch

import oracle as O
import parity as P
import synth

pytestmark = pytest.mark.gpu

B = None


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
    """uint16 bf16 bits -> CUDA bfloat16 tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def host16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_gated(x, g, w, eps, act, x_pad=0):
    T, H, D = x.shape
    if x_pad:
        xb = np.zeros((T, H * D + x_pad), np.uint16)
        xb[:, :H * D] = x.reshape(T, -1)
        gb = np.zeros((T, H * D + x_pad), np.uint16)
        gb[:, :H * D] = g.reshape(T, -1)
        xt = dev16(xb)[:, :H * D].view(T, H, D)
        gt = dev16(gb)[:, :H * D].view(T, H, D)
    else:
        xt, gt = dev16(x), dev16(g)
    codes, scale = B.fp8n_gated_rmsnorm_quant_token(xt, gt, dev16(w), eps, act)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scale.cpu().numpy()


def check_gated(x, g, w, eps, act, **kw):
    got_c, got_s = run_gated(x, g, w, eps, act, **kw)
    want_c, want_s = O.gated_rmsnorm_quant_token(x, g, w, eps, act)
    r = P.compare_scales(got_s, want_s)
    r.update(P.compare_codes(got_c, want_c))
    P.compare_dequant(got_c, got_s, want_c, want_s)
    return r


# ---------------------------------------------------------------------------
# activation: every bf16 gate
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("act", [O.ACT_SIGMOID, O.ACT_SILU])
def test_gate_activation_exhaustive(act):
    g = np.arange(65536, dtype=np.uint16)
    got = host16(B.fp8n_gate_act_bf16(dev16(g), act))
    want = O.act_table(act)
    nan_g = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    nan_got = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert nan_got[nan_g].all()
    bad = np.where((got != want) & ~nan_g)[0]
    assert bad.size == 0, [(hex(int(b)), hex(int(got[b])), hex(int(want[b]))) for b in bad[:10]]


# ---------------------------------------------------------------------------
# (A)
# ---------------------------------------------------------------------------

W = synth.workloads()


def test_gated_small_full():
    w = W["gated_small"]
    r = check_gated(w.x(), w.gate(), w.weight(), w.eps, w.act)
    assert r["code_diffs"] == 0


@pytest.mark.parametrize("name,T", [("gated_silu", 611), ("gated_large", 203)])
def test_gated_workload_prefix(name, T):
    w = W[name]
    check_gated(w.x(0, T), w.gate(0, T), w.weight(), w.eps, w.act)


@pytest.mark.parametrize("T,H,D", [
    (1, 1, 8), (3, 5, 8), (5, 2, 16), (7, 3, 32), (9, 4, 64), (5, 2, 256), (3, 2, 1024),
    (2, 16, 1024), (4, 3, 40), (3, 2, 96), (2, 1, 8192), (3, 7, 120), (2, 128, 128),
])
@pytest.mark.parametrize("act", [O.ACT_SIGMOID, O.ACT_SILU])
def test_gated_shapes(T, H, D, act):
    rng = np.random.default_rng(T * 131 + H * 7 + D + act)
    x = synth.bf16_normal(5, 11 + D, T * H * D, outlier_p=0.02, outlier_scale=60.0).reshape(T, H, D)
    g = synth.bf16_normal(5, 12 + D, T * H * D, sigma=3.0, outlier_p=0.02,
                          outlier_scale=40.0).reshape(T, H, D)
    wt = synth.bf16_normal(5, 13 + D, D, sigma=0.1, mean=1.0)
    check_gated(x, g, wt, 1e-6, act)
    del rng


def test_gated_strided_rows():
    w = W["gated_silu"]
    check_gated(w.x(100, 77), w.gate(100, 77), w.weight(), w.eps, w.act, x_pad=24)


def test_gated_special_tokens():
    """zero tokens (scale 0, signed zero codes), a token that is all -x, and
    tokens whose gates sit in the subnormal / saturated regions."""
    T, H, D = 6, 4, 128
    x = W["gated_small"].x(0, T)[:, :H].copy()
    g = W["gated_small"].gate(0, T)[:, :H].copy()
    x[0] = 0                                     # all-zero token
    x[1] = x[2] ^ 0x8000                         # sign-flipped copy of token 2
    g[3] = 0xC2B4                                # gate -90: subnormal sigmoid
    g[4] = 0x42C8                                # gate 100: sigmoid 1, silu = g
    g[5, :, ::2] = 0x0001                        # smallest subnormal gate
    wt = W["gated_small"].weight()
    for act in (O.ACT_SIGMOID, O.ACT_SILU):
        got_c, got_s = run_gated(x, g, wt, 1e-6, act)
        want_c, want_s = O.gated_rmsnorm_quant_token(x, g, wt, 1e-6, act)
        assert got_s[0] == 0 and want_s[0] == 0
        assert np.array_equal(got_c, want_c)
        assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32))


@pytest.mark.parametrize("name", ["gated_silu", "gated_large"])
def test_gated_full_size_sampled(name):
    """The whole workload in one launch (the benchmark's configuration);
    48 tokens (first, last, spread) checked against the oracle one by one."""
    w = W[name]
    x, g, wt = w.x(), w.gate(), w.weight()
    codes, scale = B.fp8n_gated_rmsnorm_quant_token(dev16(x), dev16(g), dev16(wt), w.eps, w.act)
    torch.cuda.synchronize()
    rng = np.random.default_rng(17)
    toks = np.unique(np.concatenate([[0, 1, w.T - 1], rng.integers(0, w.T, 45)]))
    codes_s = codes[torch.from_numpy(toks).cuda()].cpu().numpy()
    scale_s = scale[torch.from_numpy(toks).cuda()].cpu().numpy()
    want_c = np.zeros_like(codes_s)
    want_s = np.zeros_like(scale_s)
    for i, t in enumerate(toks):
        _, want_c[i], want_s[i] = O.gated_rmsnorm_quant_one(x[t], g[t], wt, w.eps, w.act)
    P.compare_scales(scale_s, want_s)
    P.compare_codes(codes_s, want_c)
    # the row amax element maps to +-448 in every token
    assert ((codes_s & 0x7F) == 0x7E).any(axis=1).all()


# ---------------------------------------------------------------------------
# (B)
# ---------------------------------------------------------------------------

def run_mx(q, wq, kv, wkv, eps):
    kvt = dev16(kv) if kv is not None and kv.shape[1] else None
    wkvt = dev16(wkv) if kvt is not None else None
    qo, qs, ko = B.fp8n_rmsnorm_quant_mx(dev16(q), dev16(wq), kvt, wkvt, eps)
    torch.cuda.synchronize()
    return qo.cpu().numpy(), qs.cpu().numpy(), (host16(ko) if ko is not None else None)


def check_mx(q, wq, kv, wkv, eps):
    got = run_mx(q, wq, kv, wkv, eps)
    kv_ = kv if kv is not None else np.zeros((q.shape[0], 0), np.uint16)
    wkv_ = wkv if wkv is not None else np.zeros((0,), np.uint16)
    want = O.rmsnorm_quant_mx(q, wq, kv_, wkv_, eps)
    assert np.array_equal(got[1], want[1])                  # E8M0: bit-exact
    P.compare_codes(got[0], want[0])
    if kv_.shape[1]:
        assert np.array_equal(got[2], want[2])              # kv bf16: bit-exact
    return got, want


def test_mx_workload_prefix():
    w = W["qkv_mx"]
    got, want = check_mx(w.q(0, 777), w.q_weight(), w.kv(0, 777), w.kv_weight(), w.eps)
    assert np.array_equal(got[0], want[0])


@pytest.mark.parametrize("M,Nq,Nkv", [
    (1, 32, 0), (3, 32, 8), (5, 96, 40), (7, 1536, 512), (3, 2048, 2048), (2, 4096, 64),
    (2, 16384, 16384), (9, 224, 8), (33, 64, 24),
    # the row kernel's q/kv register layouts: 2 and 4 q chunks of 512, 3 and 4 kv chunks of 256
    (5, 1024, 256), (4, 2048, 1024), (6, 544, 768), (3, 1536, 0),
    # more rows than warps on the grid, so that each warp's two slots are refilled
    (9000, 544, 40), (4257, 32, 8),
])
def test_mx_shapes(M, Nq, Nkv):
    q = synth.bf16_normal(7, 21 + Nq, M * Nq, sigma=1.4, outlier_p=0.01,
                          outlier_scale=80.0).reshape(M, Nq)
    kv = synth.bf16_normal(7, 22 + Nkv, M * Nkv, sigma=1.4).reshape(M, Nkv)
    wq = synth.bf16_normal(7, 23, Nq, sigma=0.1, mean=1.0)
    wkv = synth.bf16_normal(7, 24, Nkv, sigma=0.1, mean=1.0)
    check_mx(q, wq, kv if Nkv else None, wkv if Nkv else None, 1e-6)


def test_mx_zero_and_tiny_rows():
    M, Nq, Nkv = 4, 128, 16
    q = W["qkv_mx"].q(0, M)[:, :Nq].copy()
    kv = W["qkv_mx"].kv(0, M)[:, :Nkv].copy()
    q[0] = 0
    kv[0] = 0
    q[1, 32:64] = 0                                   # one zero block in a normal row
    q[2] = 0x0001                                     # subnormal row
    wq = W["qkv_mx"].q_weight()[:Nq]
    wkv = W["qkv_mx"].kv_weight()[:Nkv]
    got, want = check_mx(q, wq, kv, wkv, 1e-6)
    assert np.array_equal(got[0], want[0])


def test_mx_full_size_sampled():
    w = W["qkv_mx"]
    q, kv = w.q(), w.kv()
    qo, qs, ko = B.fp8n_rmsnorm_quant_mx(dev16(q), dev16(w.q_weight()), dev16(kv),
                                         dev16(w.kv_weight()), w.eps)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, w.M - 1], np.random.default_rng(3).integers(0, w.M, 62)]))
    idx = torch.from_numpy(rows).cuda()
    want = O.rmsnorm_quant_mx(q[rows], w.q_weight(), kv[rows], w.kv_weight(), w.eps)
    assert np.array_equal(qs[idx].cpu().numpy(), want[1])
    P.compare_codes(qo[idx].cpu().numpy(), want[0])
    assert np.array_equal(host16(ko[idx]), want[2])


# ---------------------------------------------------------------------------
# (C)
# ---------------------------------------------------------------------------

def run_static(xs, ds, pad_tok=0, cu=None):
    def put(a):
        if not pad_tok:
            return dev16(a)
        T, H, D = a.shape
        buf = np.zeros((T, H * D + pad_tok), np.uint16)
        buf[:, :H * D] = a.reshape(T, -1)
        return dev16(buf)[:, :H * D].view(T, H, D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cut = None if cu is None else torch.tensor(np.asarray(cu, np.int32), device="cuda")
    outs = B.fp8n_static_head_quant(put(xs["q"]), put(xs["k"]), put(xs["v"]),
                                    *(torch.from_numpy(ds[k]).cuda() for k in ("q", "k", "v")),
                                    cu_seqlens=cut, status=status)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs], int(status.item())


def check_static(xs, ds, **kw):
    got, st = run_static(xs, ds, **kw)
    for i, k in enumerate(("q", "k", "v")):
        want = O.static_head_quant(xs[k], ds[k])
        assert np.array_equal(got[i], want), k
    return st


def test_static_small_varlen():
    sw = synth.StaticHeadWorkload("t", lengths=np.array([3, 130, 1, 77]))
    xs = {k: sw.tensor(k) for k in ("q", "k", "v")}
    assert check_static(xs, sw.descales(xs)) == 0
    assert check_static(xs, sw.descales(xs), pad_tok=64) == 0


def test_static_cu_seqlens_checked_on_device():
    """cu_seqlens is validated by the kernel (no host synchronisation): a
    first sum that is not 0, a decreasing sum or a last sum other than T sets
    FP8N_STATUS_BAD_SEQLENS; the codes do not depend on it."""
    sw = synth.StaticHeadWorkload("t", lengths=np.array([5, 9, 300]))
    xs = {k: sw.tensor(k) for k in ("q", "k", "v")}
    ds = sw.descales(xs)
    good = sw.cu_seqlens()
    assert good.tolist() == [0, 5, 14, 314]
    cases = {"good": (good, 0), "none": (None, 0),
             "first_not_zero": ([1, 5, 14, 314], B.STATUS_BAD_SEQLENS),
             "decreasing": ([0, 14, 5, 314], B.STATUS_BAD_SEQLENS),
             "last_not_T": ([0, 5, 14, 313], B.STATUS_BAD_SEQLENS),
             "one_seq": ([0, 314], 0), "one_seq_short": ([0, 200], B.STATUS_BAD_SEQLENS)}
    for name, (cu, want_bits) in cases.items():
        got, st = run_static(xs, ds, cu=cu)
        assert st == want_bits, name
        for i, k in enumerate(("q", "k", "v")):
            assert np.array_equal(got[i], O.static_head_quant(xs[k], ds[k])), (name, k)


def test_static_division_all_bf16_numerators():
    """every bf16 value divided by 36 descales (random, ones such as 3 and 7
    whose reciprocal is inexact, and the extremes of the binary32 range),
    against the oracle's IEEE quotient."""
    x = np.arange(65536, dtype=np.uint16)
    x = np.where((x & 0x7F80) == 0x7F80, 0x3F80, x).astype(np.uint16)   # finite only
    H, D = 12, 128
    T = 65536 // D
    q = np.broadcast_to(x.reshape(T, 1, D), (T, H, D)).copy()
    rng = np.random.default_rng(9)
    ds = {k: (10.0 ** rng.uniform(-6, 3, H)).astype(np.float32) for k in ("q", "k", "v")}
    ds["k"][:6] = np.array([3, 7, 1.0 / 3, 11, 0.1, 1e-5], np.float32)
    # both ends of the reciprocal path (2^-92 .. 2^126) and beyond it
    ds["v"][:8] = np.array([2.0 ** -100, 2.0 ** -92, 1.5 * 2.0 ** -93, 2.0 ** 125, 2.0 ** 126,
                            1.5 * 2.0 ** 126, 1e-40, np.finfo(np.float32).max], np.float32)
    xs = {"q": q, "k": q, "v": q}
    assert check_static(xs, ds) == 0


def test_static_bad_descales_flagged():
    sw = synth.StaticHeadWorkload("t", lengths=np.array([5, 9]))
    xs = {k: sw.tensor(k) for k in ("q", "k", "v")}
    ds = sw.descales(xs)
    ds["k"][2] = 0.0
    ds["v"][1] = -1.0
    ds["q"][4] = np.nan
    ds["q"][5] = np.inf
    assert check_static(xs, ds) & B.STATUS_BAD_DESCALE
    assert not B.fp8n_check_descales(torch.from_numpy(ds["q"]).cuda())
    assert B.fp8n_check_descales(torch.ones(12, device="cuda"))


def test_static_full_size_sampled():
    sw = W["static_head"]
    xs = {k: sw.tensor(k) for k in ("q", "k", "v")}
    ds = sw.descales(xs)
    dev = {k: dev16(xs[k]) for k in xs}
    outs = B.fp8n_static_head_quant(dev["q"], dev["k"], dev["v"],
                                    *(torch.from_numpy(ds[k]).cuda() for k in ("q", "k", "v")),
                                    cu_seqlens=torch.from_numpy(sw.cu_seqlens()).cuda())
    torch.cuda.synchronize()
    toks = np.unique(np.concatenate([[0, sw.T - 1], sw.cu_seqlens()[1:-1],
                                     np.random.default_rng(5).integers(0, sw.T, 200)]))
    idx = torch.from_numpy(toks).cuda()
    for i, k in enumerate(("q", "k", "v")):
        want = O.static_head_quant(xs[k][toks], ds[k])
        assert np.array_equal(outs[i][idx].cpu().numpy(), want), k


def test_zero_sizes_launch_nothing():
    e = torch.empty((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    c, s = B.fp8n_gated_rmsnorm_quant_token(e, e, torch.ones(128, dtype=torch.bfloat16,
                                                                 device="cuda"))
    assert c.shape == (0, 512) and s.shape == (0,)
