"""GPU parity of the token-by-token forward (kda_recurrent_fwd) against the
FP64 oracle, plus its serving properties: in-place state update, decoding one
token per call, agreement with the chunked forward, and the error word for
inconsistent cu_seqlens.

Tolerances as for the chunked path: normwise relative error <= 1e-4 (fp32
I/O) or 2e-2 (bf16 I/O) for o and ht.
"""

import numpy as np
import pytest
import torch

from tests.helpers import check_close, np64, run_oracle
from workloads import make_case

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}


def rec_run(case, ht=None, err=None):
    import chunkwise_delta_rule_gb300 as kda
    c = case.to("cuda")
    p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate=case.gate, scale=case.scale,
                         initial_state=c.h0, cu_seqlens=c.cu_seqlens)
    o, ht = kda.kda_recurrent_fwd(p, ht=ht, err=err)
    torch.cuda.synchronize()
    return o, ht


def check_fwd(case, o, ht, tol):
    ref = run_oracle(case, backward=False)
    BT = case.B * case.T
    check_close("o", np64(o).reshape(BT, case.H, case.V), ref["o"], tol)
    check_close("ht", np64(ht), ref["ht"], tol)


CASES = [
    dict(io="fp32", gate="channel", B=2, T=70, H=3, K=64, V=64),
    dict(io="fp32", gate="scalar", B=2, T=7, H=2, K=128, V=128),
    dict(io="fp32", gate="none", B=1, T=1, H=2, K=64, V=64),
    dict(io="bf16", gate="channel", B=3, T=1, H=4, K=128, V=128),
    dict(io="bf16", gate="channel", B=2, T=64, H=2, K=128, V=128),
    dict(io="bf16", gate="scalar", B=1, T=33, H=2, K=64, V=64),
    dict(io="bf16", gate="none", B=2, T=5, H=2, K=128, V=128, h0=False),
    # value widths other than K (any multiple of 32): Gated DeltaNet's V = 2K heads among them
    dict(io="bf16", gate="scalar", B=2, T=9, H=2, K=128, V=256),
    dict(io="fp32", gate="channel", B=1, T=20, H=3, K=64, V=96),
    dict(io="bf16", gate="channel", B=2, T=3, H=2, K=128, V=32),
    # key widths above 128 (the token-by-token kernel only): 192/160, 256, 160
    dict(io="bf16", gate="channel", B=2, T=12, H=2, K=192, V=160),
    dict(io="fp32", gate="scalar", B=1, T=9, H=2, K=256, V=256),
    dict(io="fp32", gate="channel", B=2, T=5, H=1, K=160, V=64),
]


@pytest.mark.parametrize("kw", CASES, ids=lambda kw: "{io}-{gate}-B{B}T{T}H{H}K{K}V{V}".format(**kw))
def test_recurrent_matches_oracle(kw):
    case = make_case(seed=61, **kw)
    o, ht = rec_run(case)
    check_fwd(case, o, ht, TOL[case.io])


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_recurrent_packed_sequences(io):
    case = make_case(io=io, gate="channel", B=1, H=2, K=128, V=128, seed=62, lengths=[1, 5, 64, 3, 70])
    o, ht = rec_run(case)
    check_fwd(case, o, ht, TOL[io])


def test_recurrent_updates_the_state_in_place():
    case = make_case(io="bf16", gate="channel", B=2, T=9, H=2, K=128, V=128, seed=63)
    o1, ht1 = rec_run(case)
    c = case.to("cuda")
    import chunkwise_delta_rule_gb300 as kda
    state = c.h0.clone()
    p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate=case.gate, scale=case.scale, initial_state=state)
    o2, ht2 = kda.kda_recurrent_fwd(p, ht=state)
    torch.cuda.synchronize()
    assert ht2.data_ptr() == state.data_ptr()
    assert torch.equal(o1, o2)
    assert torch.equal(ht1, state)


def test_decoding_one_token_per_call_equals_one_call():
    """A state carried through T calls of one token each gives bitwise the same
    outputs and final state as one call over the T tokens."""
    import chunkwise_delta_rule_gb300 as kda
    case = make_case(io="bf16", gate="channel", B=3, T=6, H=2, K=128, V=128, seed=64)
    o_all, ht_all = rec_run(case)
    c = case.to("cuda")
    state = c.h0.clone()
    outs = []
    for t in range(case.T):
        sl = lambda x: x[:, t:t + 1].contiguous()  # noqa: E731
        p = kda.make_problem(sl(c.q), sl(c.k), sl(c.v), sl(c.g), sl(c.beta), gate=case.gate,
                             scale=case.scale, initial_state=state)
        o, _ = kda.kda_recurrent_fwd(p, ht=state)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, 1), o_all)
    assert torch.equal(state, ht_all)


@pytest.mark.parametrize("io,D", [("fp32", 64), ("bf16", 128)])
def test_recurrent_agrees_with_the_chunked_forward(io, D):
    import chunkwise_delta_rule_gb300 as kda
    case = make_case(io=io, gate="channel", B=2, T=150, H=2, K=D, V=D, seed=65)
    o_r, ht_r = rec_run(case)
    c = case.to("cuda")
    p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate=case.gate, scale=case.scale, initial_state=c.h0)
    o_c, ht_c, _ = kda.kda_chunk_fwd(p)
    torch.cuda.synchronize()
    check_close("o", np64(o_r), np64(o_c), TOL[io])
    check_close("ht", np64(ht_r), np64(ht_c), TOL[io])


def test_recurrent_flags_inconsistent_cu_seqlens():
    """Offsets past the token count: the sequence is treated as empty (its
    state passes through) and bit 0 of the error word is set."""
    import chunkwise_delta_rule_gb300 as kda
    case = make_case(io="fp32", gate="channel", B=1, H=2, K=64, V=64, seed=66, lengths=[4, 4]).to("cuda")
    bad = torch.tensor([0, 4, 99], dtype=torch.int32, device="cuda")
    p = kda.make_problem(case.q, case.k, case.v, case.g, case.beta, gate="channel", scale=case.scale,
                         initial_state=case.h0, cu_seqlens=bad)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, ht = kda.kda_recurrent_fwd(p, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    assert torch.equal(ht[1], case.h0[1])
    assert np.all(np.isfinite(np64(ht)))
