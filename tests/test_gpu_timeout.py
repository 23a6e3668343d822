"""The pipeline-timeout path of the staged kernels, run without a hang.

The staged kernels of (A) and (B) wait on mbarriers for their bulk copies
with an iteration limit; a wait that runs out sets
FP8N_STATUS_PIPELINE_TIMEOUT in the status word, stops the CTA, lets the
copies already issued land (with the normal limit) and returns.  A test-only
build sets the main-loop limit to zero iterations (FP8N_WAIT_LIMIT_MAIN=0),
so every main-loop wait gives up at once while the copies themselves are
real, valid and complete: the test checks that each call returns, that the
status bit is set, and that the context still works afterwards.  The copy
runs in a child process that loads only that build.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import synth
from rmsnorm_fp8_activation_gb300 import build
path = build.build(variant="wait0", defines=("FP8N_WAIT_LIMIT_MAIN=0",))
L = ctypes.CDLL(path)
P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
L.fp8n_gated_rmsnorm_quant_token.argtypes = [P, i64, P, i64, P, i64, i32, i32, f32, ctypes.c_int,
                                             P, i64, P, P, P]
L.fp8n_rmsnorm_quant_mx.argtypes = [P, i64, P, i32, P, i64, P, i32, i64, f32, P, i64, P, i64,
                                    P, i64, P, P]
dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
ptr = lambda t: ctypes.c_void_p(t.data_ptr())
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
out = {}
# (A): 1000 tokens of 8 heads x 128 (the staged kernel, several tokens per CTA)
T, H, D = 1000, 8, 128
x = dev(synth.bf16_normal(0, 901, T * H * D))
g = dev(synth.bf16_normal(0, 902, T * H * D))
w = dev(synth.bf16_normal(0, 903, D, sigma=0.1, mean=1.0))
codes = torch.zeros((T, H * D), dtype=torch.uint8, device="cuda")
scale = torch.zeros((T,), dtype=torch.float32, device="cuda")
st = torch.zeros(1, dtype=torch.int32, device="cuda")
out["gated_rc"] = L.fp8n_gated_rmsnorm_quant_token(ptr(x), H * D, ptr(g), H * D, ptr(w), T, H, D,
                                                   1e-6, 0, ptr(codes), H * D, ptr(scale), ptr(st),
                                                   stream)
torch.cuda.synchronize()
out["gated_status"] = int(st.item())
# (B): 1000 rows of q 1536 + kv 512 (the staged kernel)
M, Nq, Nkv = 1000, 1536, 512
q = dev(synth.bf16_normal(0, 911, M * Nq))
kv = dev(synth.bf16_normal(0, 912, M * Nkv))
wq = dev(synth.bf16_normal(0, 913, Nq, sigma=0.1, mean=1.0))
wk = dev(synth.bf16_normal(0, 914, Nkv, sigma=0.1, mean=1.0))
qo = torch.zeros((M, Nq), dtype=torch.uint8, device="cuda")
qs = torch.zeros((M, Nq // 32), dtype=torch.uint8, device="cuda")
ko = torch.zeros((M, Nkv), dtype=torch.int16, device="cuda")
st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
out["mx_rc"] = L.fp8n_rmsnorm_quant_mx(ptr(q), Nq, ptr(wq), Nq, ptr(kv), Nkv, ptr(wk), Nkv, M,
                                       1e-6, ptr(qo), Nq, ptr(qs), Nq // 32, ptr(ko), Nkv,
                                       ptr(st2), stream)
torch.cuda.synchronize()
out["mx_status"] = int(st2.item())
# the context still works
out["after"] = float(torch.arange(10, device="cuda", dtype=torch.float32).sum().item())
print("RESULT " + json.dumps(out))
"""


def test_zero_wait_limit_sets_timeout_and_returns():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    assert res["gated_rc"] == 0 and res["mx_rc"] == 0
    assert res["gated_status"] & 0x2, res
    assert res["mx_status"] & 0x2, res
    assert res["after"] == 45.0


def test_normal_build_reports_no_timeout():
    """The same two calls through the library as built: no status bit."""
    from rmsnorm_fp8_activation_gb300 import build
    build.build()
    import rmsnorm_fp8_activation_gb300 as B
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    T, H, D = 1000, 8, 128
    x = dev(synth.bf16_normal(0, 901, T * H * D)).view(T, H, D)
    g = dev(synth.bf16_normal(0, 902, T * H * D)).view(T, H, D)
    w = dev(synth.bf16_normal(0, 903, D, sigma=0.1, mean=1.0))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp8n_gated_rmsnorm_quant_token(x, g, w, 1e-6, 0, status=st)
    M, Nq, Nkv = 1000, 1536, 512
    q = dev(synth.bf16_normal(0, 911, M * Nq)).view(M, Nq)
    kv = dev(synth.bf16_normal(0, 912, M * Nkv)).view(M, Nkv)
    wq = dev(synth.bf16_normal(0, 913, Nq, sigma=0.1, mean=1.0))
    wk = dev(synth.bf16_normal(0, 914, Nkv, sigma=0.1, mean=1.0))
    B.fp8n_rmsnorm_quant_mx(q, wq, kv, wk, 1e-6, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
