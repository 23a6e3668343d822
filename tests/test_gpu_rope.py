"""GPU parity of the inverse-RoPE + MXFP8 producer against the oracle.

The map has no reduction whose order could matter (each rotated value is two
products and one sum in binary32, the block maximum is exact), so codes, E8M0
scales and the bf16 step are compared bit for bit, on every element of the
o-projection workload in one launch and on small shapes that cover both pair
layouts, spans at offsets, ragged batches, strided rows, the hand-worked rows
and positions outside the cache.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu

B = None
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


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


def run(o, pos, cs, off, R, inter, o_pad=0, status=None):
    T, H, D = o.shape
    if o_pad:
        buf = np.zeros((T, H * D + o_pad), np.uint16)
        buf[:, :H * D] = o.reshape(T, -1)
        ot = dev16(buf)[:, :H * D].view(T, H, D)
    else:
        ot = dev16(o)
    pt = torch.from_numpy(np.ascontiguousarray(pos, np.int32)).cuda()
    ct = torch.from_numpy(np.ascontiguousarray(cs, np.float32)).cuda()
    style = B.ROPE_INTERLEAVED if inter else B.ROPE_HALF
    codes, scale = B.fp8n_inv_rope_quant_mx(ot, pt, ct, off, R, style, status=status)
    y = B.fp8n_inv_rope_bf16(ot, pt, ct, off, R, style, status=status)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scale.cpu().numpy(), host16(y), (y, codes, scale)


def test_inv_rope_full_workload():
    """o [4096, 16, 576], rope on the last 64 dims, every code and scale."""
    w = synth.workloads()["inv_rope_mx"]
    o, pos, cs = w.o(), w.positions(), w.cos_sin()
    got_c, got_s, got_y, _ = run(o, pos, cs, w.rope_off, w.rope_dim, w.interleaved)
    want_c = np.empty_like(got_c)
    want_s = np.empty_like(got_s)

    def ref(a, b):
        want_c[a:b], want_s[a:b] = O.inv_rope_quant_mx(o[a:b], pos[a:b], cs, w.rope_off,
                                                       w.rope_dim, w.interleaved)

    O.sliced(ref, w.T, min_slice=64)
    print("parity", json.dumps({"workload": "inv_rope_mx", "tokens": w.T, "codes": int(got_c.size),
                                "code_diffs": int((got_c != want_c).sum()),
                                "e8m0_diffs": int((got_s != want_s).sum())}))
    for t, j in zip(*np.nonzero(got_c != want_c)):  # context of any difference, for the log
        h, d = divmod(int(j), w.D)
        print("diff", json.dumps({"t": int(t), "h": h, "d": d, "pos": int(pos[t]),
                                  "x": int(o[t, h, d]), "got": int(got_c[t, j]),
                                  "want": int(want_c[t, j]), "scale": int(got_s[t, j // 32]),
                                  "y_gpu": int(got_y[t, j]),
                                  "y_oracle": int(O.inv_rope_bf16(o[t:t + 1], pos[t:t + 1], cs,
                                                                  w.rope_off, w.rope_dim,
                                                                  w.interleaved)[0, j])}))
    assert np.array_equal(got_s, want_s)
    assert np.array_equal(got_c, want_c)
    rows = np.arange(0, w.T, 97)
    assert np.array_equal(got_y[rows], O.inv_rope_bf16(o[rows], pos[rows], cs, w.rope_off,
                                                       w.rope_dim, w.interleaved))


@pytest.mark.parametrize("T,H,D,off,R,inter", [
    (1, 1, 32, 0, 32, False), (3, 1, 32, 0, 32, True), (5, 2, 64, 32, 32, False),
    (7, 3, 96, 16, 64, True), (9, 2, 128, 64, 64, False), (4, 4, 576, 512, 64, False),
    (6, 2, 576, 512, 64, True), (2, 1, 8192, 8064, 128, False), (11, 3, 64, 8, 16, True),
    (13, 2, 64, 0, 0, False), (33, 1, 256, 0, 256, False),
    # long rows (8 and 9 heads of 8192), the span at the start, the end and absent
    (3, 8, 8192, 8064, 128, False), (2, 8, 8192, 0, 64, True), (2, 9, 8192, 4096, 0, False),
    # more tokens than one pass of the grid's warps covers
    (300, 3, 192, 128, 64, False), (257, 5, 96, 32, 32, True),
])
def test_inv_rope_shapes(T, H, D, off, R, inter):
    rng = np.random.default_rng(T * 7 + D + R)
    P = 50
    o = synth.bf16_normal(8, 31 + D + R, T * H * D, outlier_p=0.03, outlier_scale=40.0).reshape(T, H, D)
    ang = rng.uniform(-30.0, 30.0, size=(P, max(R, 2) // 2))
    cs = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)[:, :R]
    if R == 0:
        cs = np.zeros((P, 0), np.float32)
    pos = rng.integers(0, P, size=T).astype(np.int32)
    got_c, got_s, got_y, _ = run(o, pos, cs, off, R, inter)
    want_c, want_s = O.inv_rope_quant_mx(o, pos, cs if R else np.zeros((P, 0), np.float32), off, R, inter)
    assert np.array_equal(got_s, want_s)
    assert np.array_equal(got_c, want_c)
    assert np.array_equal(got_y, O.inv_rope_bf16(o, pos, cs, off, R, inter))


def test_inv_rope_strided_rows_and_fused_equals_steps():
    w = synth.InvRopeWorkload("t", T=300, H=4, D=576, P=512)
    o, pos, cs = w.o(), w.positions(), w.cos_sin()
    got_c, got_s, _, (y, codes, scale) = run(o, pos, cs, w.rope_off, w.rope_dim, False, o_pad=64)
    want_c, want_s = O.inv_rope_quant_mx(o, pos, cs, w.rope_off, w.rope_dim, False)
    assert np.array_equal(got_c, want_c) and np.array_equal(got_s, want_s)
    # the two steps on the GPU: the MX quantiser of the bf16 step, bit for bit
    c2, s2 = B.fp8n_quant_mx(y)
    torch.cuda.synchronize()
    assert torch.equal(c2, codes) and torch.equal(s2, scale)


def test_inv_rope_golden_rows():
    with open(os.path.join(GOLDEN, "inv_rope_rows.json")) as f:
        g = json.load(f)
    import struct
    for row in g["rows"]:
        H, D, R = row["H"], row["D"], row["R"]
        bits = [0x8000 if v == "-0" else struct.unpack("<I", struct.pack("<f", float(v)))[0] >> 16
                for v in row["x"]]
        o = np.array(bits, np.uint16).reshape(1, H, D)
        cs = np.array([[row["cos"]] * (R // 2) + [row["sin"]] * (R // 2)], np.float32)
        got_c, got_s, _, _ = run(o, np.zeros(1, np.int32), cs, row["rope_off"], R,
                                 row["interleaved"])
        assert got_c[0].tolist() == [int(c, 16) for c in row["codes"]], row["name"]
        assert got_s[0].tolist() == [int(c, 16) for c in row["scale"]], row["name"]


def test_inv_rope_no_fused_multiply_add():
    """Two rotations where one rounding of x1*c + x2*s (a contracted
    multiply-add) lands on the other bf16 neighbour: the kernel rounds the
    product and the sum apart, as the oracle does."""
    import test_oracle_rope as R
    o, cs = R.contraction_row()
    _, _, got_y, _ = run(o, np.zeros(1, np.int32), cs, 0, 32, False)
    assert np.array_equal(got_y, O.inv_rope_bf16(o, np.zeros(1, np.int32), cs, 0, 32, False))
    for i, (_, _, _, _, apart, _) in enumerate(R.CONTRACTION_CASES):
        assert got_y[0, i] == apart


def test_inv_rope_positions_outside_the_cache_are_flagged():
    w = synth.InvRopeWorkload("t", T=40, H=2, D=576, P=64)
    o, pos, cs = w.o(), w.positions(), w.cos_sin()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run(o, pos, cs, w.rope_off, w.rope_dim, False, status=status)
    assert int(status.item()) == 0
    bad = pos.copy()
    bad[3], bad[17] = -5, 64
    got_c, got_s, _, _ = run(o, bad, cs, w.rope_off, w.rope_dim, False, status=status)
    assert int(status.item()) & B.STATUS_BAD_POSITION
    clamped = np.clip(bad, 0, 63).astype(np.int32)
    want_c, want_s = O.inv_rope_quant_mx(o, clamped, cs, w.rope_off, w.rope_dim, False)
    assert np.array_equal(got_c, want_c) and np.array_equal(got_s, want_s)
