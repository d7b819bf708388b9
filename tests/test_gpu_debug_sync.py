"""LF_DEBUG_SYNC: with the variable set in the environment, every call
synchronises its stream and reads the device error word, so a device-side wait
that ran out is returned by the call itself (LF_ERR_DEVICE_TIMEOUT) instead of
by a later lf_check_device_error.  The switch is read once per process, so the
check runs in a child process.  The stall is the library's test hook (bounded
wait, no fault)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import math, sys
sys.path.insert(0, %r)
import torch
import layout_folding_gb300 as lf
from layout_folding_gb300 import synthetic
torch.cuda.set_device(0)
M, N, K = 256, 1024, 512
x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
xd, wd = x.cuda(), w.cuda()
out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
lab = synthetic.labels_uniform(M, N).cuda()
loss = torch.empty(M, dtype=torch.float32, device="cuda")
L = lf.lib()
s = torch.cuda.current_stream().cuda_stream
assert L.gemm_nt(xd.data_ptr(), wd.data_ptr(), out.data_ptr(), M, N, K, s) == 0
lf.set_test_hooks(True, 200_000_000)
try:
    st_gemm = L.gemm_nt(xd.data_ptr(), wd.data_ptr(), out.data_ptr(), M, N, K, s)
    st_xent = L.gemm_nt_xent(xd.data_ptr(), wd.data_ptr(), lab.data_ptr(), loss.data_ptr(), None, M, N, K, s)
finally:
    lf.set_test_hooks(False, 0)
assert (st_gemm, st_xent) == (6, 6), (st_gemm, st_xent)
assert L.gemm_nt(xd.data_ptr(), wd.data_ptr(), out.data_ptr(), M, N, K, s) == 0
torch.cuda.synchronize()
print("debug-sync ok")
''' % ROOT


def test_debug_sync_returns_device_timeouts_from_the_call():
    env = dict(os.environ, LF_DEBUG_SYNC="1")
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "debug-sync ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
