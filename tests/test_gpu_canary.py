"""Out-of-bounds accesses, checked without a sanitizer.

Writes: every output of a call is a view inside a larger buffer filled with a
sentinel byte (guard rows before and after it and, where the call takes an
output row stride, padding past the end of every row).  After the call each
byte outside the outputs must still be the sentinel.

Reads: every input is a view inside a larger buffer filled with NaN (bf16
0x7FC1, binary32 0x7FC00001): guard rows around it and padding past every row
where the call takes an input row stride.  A kernel that used a value from
outside its inputs would turn a scale, an E8M0 code or a code into NaN's.

Either way the outputs must equal those of the same call on plain tensors.
Small and odd shapes (T = 1, 3, 5; D = 8, 40; ragged row tails), the shapes
that select each kernel variant, and the workloads' row lengths.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

SENT = 0xA5
G = 3          # guard rows above and below a 2-D output
G1 = 256       # guard bytes on each side of a 1-D output
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


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


class Guarded2D:
    """[rows, cols] of dtype with a row stride of round_up(cols bytes, 16) + 32
    bytes, inside a sentinel-filled buffer with G guard rows on each side."""

    def __init__(self, rows, cols, dtype):
        es = torch.empty((), dtype=dtype).element_size()
        row_bytes = (cols * es + 15) // 16 * 16 + 32
        self.rows, self.cols, self.es, self.rb = rows, cols, es, row_bytes
        self.buf = torch.full(((rows + 2 * G) * row_bytes,), SENT, dtype=torch.uint8, device="cuda")
        full = self.buf.view(dtype).view(rows + 2 * G, row_bytes // es)
        self.view = full[G:G + rows, :cols]

    def untouched(self) -> bool:
        b = self.buf.view(self.rows + 2 * G, self.rb).cpu().numpy()
        mask = np.ones(b.shape, bool)
        mask[G:G + self.rows, :self.cols * self.es] = False
        return bool((b[mask] == SENT).all())


class Guarded1D:
    """n elements of dtype with G1 sentinel bytes on each side."""

    def __init__(self, n, dtype, shape=None):
        es = torch.empty((), dtype=dtype).element_size()
        self.n, self.es = n, es
        self.buf = torch.full((2 * G1 + n * es,), SENT, dtype=torch.uint8, device="cuda")
        self.view = self.buf[G1:G1 + n * es].view(dtype)
        if shape is not None:
            self.view = self.view.view(*shape)

    def untouched(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool((b[:G1] == SENT).all() and (b[G1 + self.n * self.es:] == SENT).all())


def nan_input(a: np.ndarray, heads_dim: int = 0) -> torch.Tensor:
    """bf16 bits a ([rows, cols] or [T, H, D]) copied into a view of a buffer
    filled with bf16 NaN: G guard rows on each side, 32 bytes past each row
    (the row is the last axis, or H * D for a [T, H, D] input)."""
    shape = a.shape
    rows_, cols = shape[0], int(np.prod(shape[1:]))
    g = Guarded2D(rows_, cols, torch.bfloat16)
    g.buf.view(torch.int16).fill_(0x7FC1)
    g.view.copy_(dev16(a.reshape(rows_, cols)))
    if len(shape) == 3:
        return g.view.as_strided(shape, (g.view.stride(0), shape[2], 1))
    return g.view


def nan_input_f32(t: torch.Tensor) -> torch.Tensor:
    """a float32 CUDA tensor copied into the middle of a NaN-filled buffer."""
    g = Guarded1D(t.numel(), torch.float32, tuple(t.shape))
    g.buf.view(torch.int32).fill_(0x7FC00001)
    g.view.copy_(t)
    return g.view


def nan_input_i32(t: torch.Tensor) -> torch.Tensor:
    """an int32 CUDA tensor copied into the middle of a buffer of -1s."""
    g = Guarded1D(t.numel(), torch.int32, tuple(t.shape))
    g.buf.view(torch.int32).fill_(-1)
    g.view.copy_(t)
    return g.view


def same(a, b):
    torch.cuda.synchronize()
    return torch.equal(a.contiguous().view(-1).view(torch.uint8), b.contiguous().view(-1).view(torch.uint8))


def rows(seed, *shape, sigma=1.0, mean=0.0):
    n = int(np.prod(shape))
    return synth.bf16_normal(31, seed, n, sigma=sigma, mean=mean, outlier_p=0.02 if mean == 0 else 0.0,
                             outlier_scale=40.0).reshape(shape)


@pytest.mark.parametrize("T,H,D,act", [
    (1, 1, 8, 0), (3, 5, 8, 1), (5, 3, 40, 0), (3, 2, 128, 1), (2, 64, 128, 0), (5, 3, 96, 0),
    (1300, 64, 128, 0),   # enough tokens per CTA for the gate table
])
def test_gated_quant_token(T, H, D, act):
    xa, ga, wa = rows(1, T, H, D), rows(2, T, H, D, sigma=2.0), rows(3, D, sigma=0.1, mean=1.0)
    x, g, w = dev16(xa), dev16(ga), dev16(wa)
    xn, gn = nan_input(xa), nan_input(ga)
    wn = nan_input(wa.reshape(1, D)).reshape(D)
    out, sc = Guarded2D(T, H * D, torch.uint8), Guarded1D(T, torch.float32)
    B.fp8n_gated_rmsnorm_quant_token(xn, gn, wn, 1e-6, act, out=out.view, scale=sc.view)
    c, s = B.fp8n_gated_rmsnorm_quant_token(x, g, w, 1e-6, act)
    assert same(out.view, c) and same(sc.view, s)
    assert out.untouched() and sc.untouched()
    # the steps on their own
    y = Guarded2D(T, H * D, torch.bfloat16)
    B.fp8n_gated_rmsnorm_bf16(xn, gn, wn, 1e-6, act, y=y.view)
    assert same(y.view, B.fp8n_gated_rmsnorm_bf16(x, g, w, 1e-6, act)) and y.untouched()
    yq = B.fp8n_gated_rmsnorm_bf16(x, g, w, 1e-6, act)
    yqn = nan_input(yq.view(torch.int16).cpu().numpy().view(np.uint16))
    out2, sc2 = Guarded2D(T, H * D, torch.uint8), Guarded1D(T, torch.float32)
    B.fp8n_quant_token(yqn, out=out2.view, scale=sc2.view)
    c2, s2 = B.fp8n_quant_token(yq)
    assert same(out2.view, c2) and same(sc2.view, s2) and out2.untouched() and sc2.untouched()
    xf, gf = x.view(T, H * D), g.view(T, H * D)
    xfn, gfn = nan_input(xa.reshape(T, H * D)), nan_input(ga.reshape(T, H * D))
    out3, sc3 = Guarded2D(T, H * D, torch.uint8), Guarded1D(T, torch.float32)
    B.fp8n_gated_quant_token(xfn, gfn, act, out=out3.view, scale=sc3.view)
    c3, s3 = B.fp8n_gated_quant_token(xf, gf, act)
    assert same(out3.view, c3) and same(sc3.view, s3) and out3.untouched() and sc3.untouched()


@pytest.mark.parametrize("M,Nq,Nkv", [
    (1, 32, 0), (3, 96, 40), (5, 1536, 512), (4, 2048, 1024), (6, 544, 768), (7, 4096, 64),
    (2, 16384, 16384), (9000, 1536, 512),
])
def test_rmsnorm_quant_mx(M, Nq, Nkv):
    qa, wqa = rows(4, M, Nq, sigma=1.4), rows(5, Nq, sigma=0.1, mean=1.0)
    q, wq = dev16(qa), dev16(wqa)
    kva = rows(6, M, Nkv, sigma=1.4) if Nkv else None
    wka = rows(7, Nkv, sigma=0.1, mean=1.0) if Nkv else None
    kv = dev16(kva) if Nkv else None
    wk = dev16(wka) if Nkv else None
    qn, wqn = nan_input(qa), nan_input(wqa.reshape(1, Nq)).reshape(Nq)
    kvn = nan_input(kva) if Nkv else None
    wkn = nan_input(wka.reshape(1, Nkv)).reshape(Nkv) if Nkv else None
    qo, qs = Guarded2D(M, Nq, torch.uint8), Guarded2D(M, Nq // 32, torch.uint8)
    ko = Guarded2D(M, Nkv, torch.bfloat16) if Nkv else None
    B.fp8n_rmsnorm_quant_mx(qn, wqn, kvn, wkn, 1e-6, q_out=qo.view, q_scale=qs.view,
                            kv_out=ko.view if Nkv else None)
    rq, rs, rk = B.fp8n_rmsnorm_quant_mx(q, wq, kv, wk, 1e-6)
    assert same(qo.view, rq) and same(qs.view, rs) and qo.untouched() and qs.untouched()
    if Nkv:
        assert same(ko.view, rk) and ko.untouched()
    # the steps: row RMSNorm to bf16, MX quantisation of a bf16 row
    y = Guarded2D(M, Nq, torch.bfloat16)
    B.fp8n_rmsnorm_bf16(qn, wqn, 1e-6, y=y.view)
    assert same(y.view, B.fp8n_rmsnorm_bf16(q, wq, 1e-6)) and y.untouched()
    mo, ms = Guarded2D(M, Nq, torch.uint8), Guarded2D(M, Nq // 32, torch.uint8)
    B.fp8n_quant_mx(qn, out=mo.view, scale=ms.view)
    c, s = B.fp8n_quant_mx(q)
    assert same(mo.view, c) and same(ms.view, s) and mo.untouched() and ms.untouched()


@pytest.mark.parametrize("lengths,H,Dqk,Dv", [
    ([1], 1, 8, 8), ([3, 5], 3, 40, 24), ([7, 13], 12, 192, 128), ([1000, 3], 12, 192, 128),
])
def test_static_and_dynamic_head_quant(lengths, H, Dqk, Dv):
    T = int(sum(lengths))
    arrs = [rows(8 + i, T, H, d) for i, d in enumerate((Dqk, Dqk, Dv))]
    q, k, v = (dev16(a) for a in arrs)
    # q and k must share strides: both get the same padding
    qn, kn, vn = (nan_input(a) for a in arrs)
    ds = [torch.rand(H, device="cuda") * 0.05 + 0.01 for _ in range(3)]
    dsn = [nan_input_f32(d) for d in ds]
    outs = [Guarded1D(T * H * d, torch.uint8, (T, H, d)) for d in (Dqk, Dqk, Dv)]
    B.fp8n_static_head_quant(qn, kn, vn, *dsn, q_out=outs[0].view, k_out=outs[1].view,
                             v_out=outs[2].view)
    ref = B.fp8n_static_head_quant(q, k, v, *ds)
    for o, r in zip(outs, ref):
        assert same(o.view, r) and o.untouched()
    # dynamic per-head: workspace, descales and codes all guarded
    ws = Guarded1D(3 * H, torch.int32)
    dsc = [Guarded1D(H, torch.float32) for _ in range(3)]
    douts = [Guarded1D(T * H * d, torch.uint8, (T, H, d)) for d in (Dqk, Dqk, Dv)]
    B.fp8n_dynamic_head_quant(qn, kn, vn, workspace=ws.view, descales=tuple(d.view for d in dsc),
                              q_out=douts[0].view, k_out=douts[1].view, v_out=douts[2].view)
    rd, ro = B.fp8n_dynamic_head_quant(q, k, v)
    for g, r in zip(dsc, rd):
        assert same(g.view, r) and g.untouched()
    for g, r in zip(douts, ro):
        assert same(g.view, r) and g.untouched()
    assert ws.untouched()
    am = Guarded1D(H, torch.float32)
    am.view.zero_()
    B.fp8n_head_amax(qn, amax=am.view)
    assert same(am.view, B.fp8n_head_amax(q)) and am.untouched()


@pytest.mark.parametrize("T,H,D,off,R,inter", [
    (1, 1, 32, 0, 32, False), (3, 2, 64, 32, 32, True), (5, 3, 96, 16, 64, False),
    (4, 16, 576, 512, 64, False), (2, 8, 8192, 8064, 128, False),
])
def test_inv_rope(T, H, D, off, R, inter):
    oa = rows(20, T, H, D)
    o, on = dev16(oa), nan_input(oa)
    P = 17
    ang = np.random.default_rng(T + D).uniform(-3, 3, size=(P, R // 2))
    cs = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)).cuda()
    pos = torch.from_numpy(np.arange(T, dtype=np.int32) % P).cuda()
    csn, posn = nan_input_f32(cs), nan_input_i32(pos)
    style = B.ROPE_INTERLEAVED if inter else B.ROPE_HALF
    out, sc = Guarded2D(T, H * D, torch.uint8), Guarded2D(T, H * D // 32, torch.uint8)
    B.fp8n_inv_rope_quant_mx(on, posn, csn, off, R, style, out=out.view, scale=sc.view)
    c, s = B.fp8n_inv_rope_quant_mx(o, pos, cs, off, R, style)
    assert same(out.view, c) and same(sc.view, s) and out.untouched() and sc.untouched()
    y = Guarded2D(T, H * D, torch.bfloat16)
    B.fp8n_inv_rope_bf16(on, posn, csn, off, R, style, y=y.view)
    assert same(y.view, B.fp8n_inv_rope_bf16(o, pos, cs, off, R, style)) and y.untouched()


@pytest.mark.parametrize("n", [1, 3, 65536, 100001])
def test_elementwise_helpers(n):
    gbits = rows(30, n, sigma=4.0)
    g, gn = dev16(gbits), nan_input(gbits.reshape(1, n)).reshape(n)
    ga = Guarded1D(n, torch.bfloat16)
    B.fp8n_gate_act_bf16(gn, 0, out=ga.view)
    assert same(ga.view, B.fp8n_gate_act_bf16(g, 0)) and ga.untouched()
    x = torch.randn(n, device="cuda") * 100
    xn = nan_input_f32(x)
    for to, dt in ((B.CVT_BF16, torch.bfloat16), (B.CVT_E4M3, torch.uint8)):
        cv = Guarded1D(n, dt)
        B.fp8n_convert_f32(xn, to, out=cv.view)
        assert same(cv.view, B.fp8n_convert_f32(x, to)) and cv.untouched()


def test_the_read_guard_is_visible():
    """The harness itself: a call that does read the NaN padding (here handed
    a view eight elements wider than the data) shows it in its outputs."""
    T, N = 4, 64
    ya = rows(40, T, N)
    yn = nan_input(ya)
    wide = yn.as_strided((T, N + 8), yn.stride())   # the data and 8 elements of padding
    _, sc = B.fp8n_quant_token(wide)
    _, sc_plain = B.fp8n_quant_token(dev16(ya))
    torch.cuda.synchronize()
    assert torch.isnan(sc).all() and not torch.isnan(sc_plain).any()
