"""Ordering of back-to-back calls launched with programmatic dependent launch.

The staged gated kernels and the q/kv producer may begin while the previous
kernel of their stream still runs, and touch global memory only after it has
completed.  This chain on one stream has each call read what the call before
it wrote (read after write), and overwrite a buffer that the call before it
reads (write after read); both results must be the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from rmsnorm_fp8_activation_gb300 import build
    build.build()
    import rmsnorm_fp8_activation_gb300 as mod
    mod.lib()
    return mod


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def test_dependent_chain_read_after_write_and_write_after_read(B):
    T, H, D = 200, 8, 128
    xs = [synth.bf16_normal(21, 300 + i, T * H * D).reshape(T, H, D) for i in range(2)]
    gs = [synth.bf16_normal(21, 310 + i, T * H * D, sigma=2.0).reshape(T, H, D) for i in range(2)]
    w = synth.bf16_normal(21, 320, D, sigma=0.1, mean=1.0)
    x = [dev16(a) for a in xs]
    g = [dev16(a) for a in gs]
    wt = dev16(w)
    y = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")   # shared by both halves
    codes = [torch.empty((T, H * D), dtype=torch.uint8, device="cuda") for _ in range(2)]
    scales = [torch.empty((T,), dtype=torch.float32, device="cuda") for _ in range(2)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(25):
            for i in range(2):
                # writes y (after the previous quantisation has read it), then reads it
                B.fp8n_gated_rmsnorm_bf16(x[i], g[i], wt, 1e-6, 0, y=y, stream=s)
                B.fp8n_quant_token(y, out=codes[i], scale=scales[i], stream=s)
    s.synchronize()
    for i in range(2):
        want_c, want_s = O.gated_rmsnorm_quant_token(xs[i], gs[i], w, 1e-6, 0)
        assert np.array_equal(codes[i].cpu().numpy(), want_c), i
        assert np.array_equal(scales[i].cpu().numpy().view(np.uint32), want_s.view(np.uint32)), i


def test_dependent_chain_qkv(B):
    """The q/kv producer after a gated call on the same stream, reading what
    it wrote (the gated bf16 output taken as q rows)."""
    T, H, D = 64, 12, 128
    x = synth.bf16_normal(22, 330, T * H * D).reshape(T, H, D)
    g = synth.bf16_normal(22, 331, T * H * D).reshape(T, H, D)
    w = synth.bf16_normal(22, 332, D, sigma=0.1, mean=1.0)
    wq = synth.bf16_normal(22, 333, H * D, sigma=0.1, mean=1.0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = B.fp8n_gated_rmsnorm_bf16(dev16(x), dev16(g), dev16(w), 1e-6, 1, stream=s)
        qo, qs, _ = B.fp8n_rmsnorm_quant_mx(y, dev16(wq), None, None, 1e-6, stream=s)
    s.synchronize()
    y_want = O.gated_rmsnorm_bf16(x, g, w, 1e-6, 1)
    want = O.rmsnorm_quant_mx(y_want, wq, np.zeros((T, 0), np.uint16), np.zeros((0,), np.uint16), 1e-6)
    assert np.array_equal(qs.cpu().numpy(), want[1])
    assert np.array_equal(qo.cpu().numpy(), want[0])
