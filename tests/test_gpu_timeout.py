"""The device-timeout path, exercised without faulting or hanging the GPU.

Every kernel of the library waits on its mbarriers with a bounded wait; when
one gives up, the kernel sets bit 1 of the device error word in the workspace
and unwinds, and kda_device_status reports KDA_ERR_DEVICE_TIMEOUT. The
self-test entry point runs that same wait on a barrier nothing arrives at, with
a short limit and no copy or MMA in flight. The test checks that the status is
reported, and that the next ordinary call on the same workspace clears the word
and still matches the FP64 oracle.
"""

import ctypes
import time

import pytest
import torch

from tests.test_gpu_parity import TOL, compare_full, packed_np
from workloads import make_case

pytestmark = pytest.mark.gpu

KDA_ERR_DEVICE_TIMEOUT = 5


def _selftest(lib, p, ws, limit_us):
    f = lib.kda_selftest_device_timeout
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint, ctypes.c_void_p]
    f.restype = ctypes.c_int
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(ctypes.addressof(p.c), ctypes.c_void_p(ws.data_ptr()), ws.numel(), limit_us, stream)


@pytest.mark.parametrize("limit_us", [20, 2000])
def test_a_wait_that_runs_out_is_reported_and_the_device_stays_usable(limit_us):
    import chunkwise_delta_rule_gb300 as kda
    from chunkwise_delta_rule_gb300 import _lib
    from oracle.cases import run_oracle
    lib = _lib.load()
    case = make_case(io="bf16", gate="channel", B=2, T=200, H=2, K=128, V=128, seed=61)
    c = case.to("cuda")
    p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate="channel", initial_state=c.h0)
    ws = torch.empty(kda.kda_workspace_size(p, True), dtype=torch.uint8, device="cuda")
    # an ordinary call leaves the word clear
    kda.kda_chunk_fwd(p, workspace=ws)
    assert kda.kda_device_status(p, ws) == (0, 0)
    # the self-test's wait gives up after limit_us and reports it
    t0 = time.perf_counter()
    assert _selftest(lib, p, ws, limit_us) == 0, _lib.last_error()
    st, word = kda.kda_device_status(p, ws)
    elapsed = time.perf_counter() - t0
    assert st == KDA_ERR_DEVICE_TIMEOUT and word & 2, (st, word)
    assert "bounded device wait" in _lib.last_error()
    assert elapsed < 5.0
    # the next forward + backward on the same workspace clears the word and matches the oracle
    o, ht, _ = kda.kda_chunk_fwd(p, workspace=ws)
    assert kda.kda_device_status(p, ws) == (0, 0)
    grads = kda.kda_chunk_bwd(p, c.do, c.dht, workspace=ws)
    assert kda.kda_device_status(p, ws) == (0, 0)
    torch.cuda.synchronize()
    got = packed_np(case, dict(o=o, ht=ht, dq=grads[0], dk=grads[1], dv=grads[2], dg=grads[3],
                               dbeta=grads[4], dh0=grads[5]))
    compare_full(case, got, run_oracle(case), TOL["bf16"])


def test_selftest_validates_its_arguments():
    import chunkwise_delta_rule_gb300 as kda
    from chunkwise_delta_rule_gb300 import _lib
    lib = _lib.load()
    c = make_case(io="bf16", gate="channel", B=1, T=64, H=1, K=128, V=128, seed=62).to("cuda")
    p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate="channel")
    ws = torch.empty(kda.kda_workspace_size(p, False), dtype=torch.uint8, device="cuda")
    assert _selftest(lib, p, ws, 0) == 1            # limit below 1 us
    assert _selftest(lib, p, ws, 2000000) == 1      # limit above 1 s
    small = ws[:64]
    assert _selftest(lib, p, small, 20) == 3        # workspace below the chunk table
