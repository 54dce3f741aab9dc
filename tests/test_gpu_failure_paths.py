"""Failure handling on the GPU, without faulting it.

* The give-up path of the bounded waits: iq_selftest_wait_timeout runs the
  fused GEMM kernel with its TMA loads left out, so the barriers that its MMA
  issuer and epilogue wait on are never completed by anything (nothing
  asynchronous is in flight); the waits must give up after the short limit,
  record their bits in the status word, take the teardown path and leave the
  context usable.
* A failed per-device set-up is not cached: the next call tries again.

Each case runs in a fresh Python process so that its first call is the
device's first set-up and so that nothing it does can disturb the other tests.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_PRELUDE = f"""
import ctypes, sys
sys.path.insert(0, {ROOT!r})
import numpy as np, torch
from fp4_fp8_quant_gb300 import iq, workloads as W
from oracle import iq_oracle as O
from tests.parity import check_fp4
L = iq.lib()

def check_prepare(M, seed):
    x, wq, wsf, pos = W.chain_workload(M, seed=seed, outlier_p=0.001, outlier_scale=50.0)
    lat = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    w, ws, p = torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda()
    q = torch.empty((M, 4096), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, 256), dtype=torch.uint8, device="cuda")
    work = torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    rc = L.iq_prepare_q(lat.data_ptr(), M, w.data_ptr(), ws.data_ptr(), p.data_ptr(), q.data_ptr(),
                        s.data_ptr(), work.data_ptr(), work.numel(), st)
    if rc != 0:
        return rc
    torch.cuda.synchronize()
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    check_fp4(q.cpu().numpy(), s.cpu().numpy(), oq, osf, oz)
    return 0
"""


def _run(body: str):
    r = subprocess.run([sys.executable, "-c", _PRELUDE + body], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, f"child failed:\n{r.stdout}\n{r.stderr}"
    return r.stdout


def test_bounded_waits_give_up_and_leave_the_context_usable(cuda_device):
    out = _run("""
ws = torch.empty(L.iq_selftest_workspace(), dtype=torch.uint8, device="cuda")
flags = ctypes.c_uint32(0)
st = torch.cuda.current_stream().cuda_stream
rc = L.iq_selftest_wait_timeout(ws.data_ptr(), ws.numel(), 2_000_000, ctypes.byref(flags), st)
print("selftest", rc, flags.value)
assert rc == -7, rc                                  # IQ_ERR_TIMEOUT
assert flags.value & 0x7 == 0x7, hex(flags.value)    # producer, MMA issuer and epilogue waits gave up
assert flags.value & 0x8 == 0, hex(flags.value)      # the teardown completed within its limit
assert iq.device_status() == 0                       # the self-test reset the word
# the context is usable: the real path runs and matches the oracle on both routes
assert check_prepare(300, 71) == 0
assert check_prepare(9, 72) == 0
assert iq.device_status() == 0
# and the self-test is repeatable
rc = L.iq_selftest_wait_timeout(ws.data_ptr(), ws.numel(), 1_000_000, ctypes.byref(flags), st)
assert rc == -7 and flags.value & 0x7 == 0x7, (rc, hex(flags.value))
assert check_prepare(130, 73) == 0
print("ok")
""")
    assert "ok" in out


def test_selftest_argument_errors(cuda_device):
    out = _run("""
n = L.iq_selftest_workspace()
ws = torch.empty(n + 256, dtype=torch.uint8, device="cuda")
st = torch.cuda.current_stream().cuda_stream
assert L.iq_selftest_wait_timeout(None, n, 1000000, None, st) == -1
assert L.iq_selftest_wait_timeout(ws.data_ptr(), n, 0, None, st) == -1
assert L.iq_selftest_wait_timeout(ws.data_ptr() + 16, n, 1000000, None, st) == -2
assert L.iq_selftest_wait_timeout(ws.data_ptr(), n - 1, 1000000, None, st) == -6
print("ok")
""")
    assert "ok" in out


def test_failed_device_setup_is_retried(cuda_device):
    out = _run("""
L.iq_debug_fail_next_setups(1)
assert check_prepare(40, 81) == -5     # IQ_ERR_CUDA: the first set-up failed
assert check_prepare(40, 81) == 0      # the next call set the device up and ran
assert check_prepare(500, 82) == 0
L.iq_debug_fail_next_setups(3)         # no effect once the device is set up
assert check_prepare(7, 83) == 0
L.iq_debug_fail_next_setups(0)
print("ok")
""")
    assert "ok" in out
