"""The no-allocation forward entry point, kda_chunk_fwd_noalloc.

It serves callers that cannot allocate device memory (allocator hooks, fully
reserved arenas, paths that cannot afford an allocation's synchronisation):
its workspace is a static device array owned by the library. The test calls it
through the C ABI twice in a row and compares each result with the ordinary
allocating entry point, kda_chunk_fwd, within the tolerance of the parity
tests. This file is collected last so that a failing run that stops at the
first failure has already run every other test; it also passes alone.
"""

import ctypes

import pytest
import torch

from tests.helpers import check_close, np64
from workloads import make_case

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}


def _noalloc(lib, p, o, ht):
    f = lib.kda_chunk_fwd_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(ctypes.addressof(p.c), ctypes.c_void_p(o.data_ptr()),
             ctypes.c_void_p(ht.data_ptr()), stream)


@pytest.mark.parametrize("kw", [
    dict(io="bf16", gate="channel", B=2, T=300, H=2, K=128, V=128),
    dict(io="fp32", gate="scalar", B=1, T=130, H=3, K=64, V=64),
    dict(io="bf16", gate="channel", B=1, T=130, H=2, K=48, V=64),     # padded to 128
    dict(io="bf16", gate="scalar", B=1, T=100, H=2, K=192, V=160),    # padded to 256
])
def test_noalloc_forward_matches_allocating_forward_twice(kw):
    import chunkwise_delta_rule_gb300 as kda
    from chunkwise_delta_rule_gb300 import _lib
    lib = _lib.load()
    for call, seed in enumerate((71, 72)):
        case = make_case(seed=seed, **kw).to("cuda")
        p = kda.make_problem(case.q, case.k, case.v, case.g, case.beta, gate=case.gate,
                             initial_state=case.h0)
        o_ref, ht_ref, _ = kda.kda_chunk_fwd(p)
        o = torch.full_like(o_ref, float("nan"))
        ht = torch.full_like(ht_ref, float("nan"))
        st = _noalloc(lib, p, o, ht)
        assert st == 0, _lib.last_error()
        torch.cuda.synchronize()
        check_close(f"o (call {call})", np64(o), np64(o_ref), TOL[kw["io"]])
        check_close(f"ht (call {call})", np64(ht), np64(ht_ref), TOL[kw["io"]])


def _noalloc_status(lib, p):
    f = lib.kda_noalloc_device_status
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    f.restype = ctypes.c_int
    word = ctypes.c_int32(-1)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = f(ctypes.addressof(p.c), stream, ctypes.byref(word))
    return st, word.value


@pytest.mark.parametrize("variant", ["value_blocks", "prologue"])
def test_noalloc_wider_layouts_match_allocating_forward(variant):
    """The no-allocation call carves the same sub-layouts as the allocating one: value widths
    above 128 run as value blocks (split buffers after the core workspace), and the gate
    activation and q/k normalisation write their buffers after it. Each is compared with
    kda_chunk_fwd, and the error word read back from the static array is clear."""
    import chunkwise_delta_rule_gb300 as kda
    from chunkwise_delta_rule_gb300 import _lib
    lib = _lib.load()
    for call, seed in enumerate((81, 82)):
        if variant == "value_blocks":
            case = make_case(io="bf16", gate="channel", B=1, T=150, H=2, K=128, V=256, seed=seed).to("cuda")
            p = kda.make_problem(case.q, case.k, case.v, case.g, case.beta, gate="channel", initial_state=case.h0)
        else:
            case = make_case(io="bf16", gate="channel", B=2, T=100, H=2, K=128, V=128, seed=seed).to("cuda")
            gen = torch.Generator().manual_seed(seed)
            a_log = torch.log(torch.rand(2, generator=gen) * 3 + 1).cuda()
            raw_g = torch.randn(case.g.shape, generator=gen).cuda()
            p = kda.make_problem(case.q * 1.7, case.k * 0.6, case.v, raw_g, case.beta, gate="channel",
                                 initial_state=case.h0, A_log=a_log, qk_l2norm=True)
        o_ref, ht_ref, _ = kda.kda_chunk_fwd(p)
        o = torch.full_like(o_ref, float("nan"))
        ht = torch.full_like(ht_ref, float("nan"))
        st = _noalloc(lib, p, o, ht)
        assert st == 0, _lib.last_error()
        assert _noalloc_status(lib, p) == (0, 0)
        torch.cuda.synchronize()
        check_close(f"o (call {call})", np64(o), np64(o_ref), TOL["bf16"])
        check_close(f"ht (call {call})", np64(ht), np64(ht_ref), TOL["bf16"])


def test_noalloc_rejects_problems_beyond_its_scratch():
    from chunkwise_delta_rule_gb300 import _lib
    lib = _lib.load()
    p = _lib.KdaProblem()
    p.B, p.T, p.H, p.K, p.V = 2, 8192, 32, 128, 128
    p.io, p.gate, p.scale = 0, 2, 0.0
    p.q = p.k = p.v = p.beta = p.g = 0x1000   # never dereferenced: rejected before launch
    f = lib.kda_chunk_fwd_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    st = f(ctypes.addressof(p), ctypes.c_void_p(0x2000), None, None)
    assert st == 3
    assert "exceeds the no-allocation scratch" in _lib.last_error()
