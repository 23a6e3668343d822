"""The allocation-free variant of the dynamic per-head quantisation.

fp8n_dynamic_head_quant_noalloc serves callers that cannot allocate device
memory (a host application that owns all device memory through its own
pool, or a latency-critical path where cudaMalloc would synchronise the
device): it keeps its per-head maxima in a static device array of the
library instead of a caller workspace.  This test calls it through the C ABI
with raw pointers and checks its descales and codes against those of the
workspace entry point and against the oracle, bit for bit (the tolerance of
the per-head path), on two calls in a row: the second call's tensors have
much smaller maxima than the first's, so maxima left in the shared array by
the first call would show.

The file is named to be collected last, so that a run stopping at the first
failure has run every other test before it; it also passes on its own in a
fresh process (its first call performs the per-device set-up).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from rmsnorm_fp8_activation_gb300 import build
    build.build()
    import rmsnorm_fp8_activation_gb300 as B
    return B.lib()


def dev16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def call(L, fn, xs, workspace=None):
    """One call of `fn` through the C ABI; returns (descales, codes) on the host."""
    q, k, v = (dev16(xs[n]) for n in ("q", "k", "v"))
    T, H, Dqk = xs["q"].shape
    Dv = xs["v"].shape[2]
    ds = [torch.full((H,), -1.0, dtype=torch.float32, device="cuda") for _ in range(3)]
    outs = [torch.full((T, H, d), 0x55, dtype=torch.uint8, device="cuda") for d in (Dqk, Dqk, Dv)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    args = [ptr(q), ptr(k), ptr(v), H * Dqk, Dqk, H * Dv, Dv, T, H, Dqk, Dv]
    if workspace is not None:
        args.append(ptr(workspace))
    args += [ptr(d) for d in ds] + [ptr(o) for o in outs] + [stream]
    assert fn(*args) == 0
    torch.cuda.synchronize()
    return [d.cpu().numpy() for d in ds], [o.cpu().numpy() for o in outs]


def test_noalloc_matches_workspace_entry_point_twice(L):
    sw = synth.StaticHeadWorkload("t", lengths=np.array([37, 300, 5]))
    first = {n: sw.tensor(n) for n in ("q", "k", "v")}
    # second call: the same shapes, values 2^-10 times smaller
    second = {n: synth.bf16_normal(3, 40 + i, first[n].size, sigma=2.0 ** -10).reshape(first[n].shape)
              for i, n in enumerate(("q", "k", "v"))}
    H = first["q"].shape[1]
    ws = torch.zeros(3 * H, dtype=torch.int32, device="cuda")
    for xs in (first, second):
        want_d, want_c = call(L, L.fp8n_dynamic_head_quant, xs, workspace=ws)
        got_d, got_c = call(L, L.fp8n_dynamic_head_quant_noalloc, xs)
        for i, n in enumerate(("q", "k", "v")):
            assert np.array_equal(got_d[i].view(np.uint32), want_d[i].view(np.uint32))
            assert np.array_equal(got_c[i], want_c[i])
            ora_d, ora_c = O.dynamic_head_quant(xs[n])
            assert np.array_equal(got_d[i].view(np.uint32), ora_d.view(np.uint32)), n
            assert np.array_equal(got_c[i], ora_c), n
    assert float(got_d[0].max()) < 2.0 ** -8       # the second call's own maxima


def test_noalloc_rejects_heads_beyond_its_scratch(L):
    P16 = 0x10000
    rc = L.fp8n_dynamic_head_quant_noalloc(P16, P16, P16, 257 * 8, 8, 257 * 8, 8, 4, 257, 8, 8,
                                           P16, P16, P16, P16, P16, P16, None)
    assert rc == 4  # FP8N_ERR_UNSUPPORTED
