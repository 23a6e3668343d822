"""Every binary32 bit pattern through the device roundings that the kernels
end with (fp8n_convert_f32: to bf16 nearest-even, to OCP E4M3 saturating
nearest-even), against the oracle's encoders, bit for bit.  NaN inputs
(exponent all ones, nonzero fraction) must give a NaN of the target format;
their payload is not compared.  The 2^32 patterns go in chunks of 2^28: the
GPU generates each chunk itself and the oracle runs over row slices on the
host's threads.
"""
import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from rmsnorm_fp8_activation_gb300 import build
    build.build()
    import rmsnorm_fp8_activation_gb300 as mod
    mod.lib()
    return mod


def device_patterns(start: int) -> torch.Tensor:
    """float32 tensor of the bit patterns start .. start + CHUNK - 1."""
    a = torch.arange(start, start + CHUNK, dtype=torch.int64, device="cuda")
    a = torch.where(a >= 1 << 31, a - (1 << 32), a).to(torch.int32)
    return a.view(torch.float32)


def nan_span(start: int) -> tuple[int, int]:
    """Offsets [lo, hi) of the NaN patterns inside the chunk at start (one
    span per sign; none in most chunks)."""
    for base in (0x7F800001, 0xFF800001):
        end = base - 1 + (1 << 23)
        lo, hi = max(base, start), min(end, start + CHUNK)
        if lo < hi:
            return lo - start, hi - start
    return 0, 0


@pytest.mark.parametrize("to", ["bf16", "e4m3"])
def test_every_binary32_pattern(B, to):
    kind = B.CVT_BF16 if to == "bf16" else B.CVT_E4M3
    enc = O.bf16_from_float_n if to == "bf16" else O.e4m3_from_float_n
    odt = np.uint16 if to == "bf16" else np.uint8
    checked = 0
    for start in range(0, 1 << 32, CHUNK):
        out = B.fp8n_convert_f32(device_patterns(start), kind)
        v = np.arange(start, start + CHUNK, dtype=np.uint32).view(np.float32)
        want = np.empty(CHUNK, odt)

        def ref(a, b):
            want[a:b] = enc(v[a:b])

        O.sliced(ref, CHUNK, min_slice=1 << 22)
        got = out.view(torch.int16 if to == "bf16" else torch.uint8).cpu().numpy().view(odt)
        lo, hi = nan_span(start)
        ok = np.array_equal(got[:lo], want[:lo]) and np.array_equal(got[hi:], want[hi:])
        if not ok:
            bad = np.nonzero(np.concatenate([got[:lo] != want[:lo], got[hi:] != want[hi:]]))[0][:8]
            idx = [int(i) if i < lo else int(i) - lo + hi for i in bad]
            pytest.fail("%s: patterns %s: got %s want %s" % (
                to, [hex(start + i) for i in idx], [hex(int(got[i])) for i in idx],
                [hex(int(want[i])) for i in idx]))
        if hi > lo:
            g = got[lo:hi].astype(np.uint32)
            if to == "bf16":
                assert (((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)).all()
            else:
                assert ((g & 0x7F) == 0x7F).all()
        checked += CHUNK
    assert checked == 1 << 32
