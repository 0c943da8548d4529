"""GPU parity with grouped value heads: HV = G * H value heads share H key
heads, value head j reading q and k of key head j / G. The oracle is the
definition written out: q and k repeated per value head, the recurrence, and
dq, dk summed over each group."""

import numpy as np
import pytest
import torch

from oracle.cases import packed, run_oracle
from tests.helpers import check_close, np64
from workloads import make_case

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}


def gva_case(io, gate, B, T, Hk, G, K, seed, lengths=None):
    case = make_case(io=io, gate=gate, B=B, T=T, H=Hk * G, K=K, V=K, seed=seed, lengths=lengths)
    qk = case.q[:, :, ::G].contiguous(), case.k[:, :, ::G].contiguous()   # one q, k per key head
    case.q = qk[0].repeat_interleave(G, dim=2)                            # the oracle's expanded view
    case.k = qk[1].repeat_interleave(G, dim=2)
    return case, qk[0], qk[1]


def oracle(case, G, backward=True):
    ref = run_oracle(case, backward=backward)
    if backward:
        BT, HV = case.B * case.T, case.H
        for name in ("dq", "dk"):
            ref[name] = ref[name].reshape(BT, HV // G, G, -1).sum(axis=2)
    return ref


def gpu(case, q, k, policy=0):
    import chunkwise_delta_rule_gb300 as kda
    c = case.to("cuda")
    p = kda.make_problem(q.cuda(), k.cuda(), c.v, c.g, c.beta, gate=case.gate, scale=case.scale, initial_state=c.h0,
                         cu_seqlens=c.cu_seqlens, save_policy=policy)
    o, ht, sv = kda.kda_chunk_fwd(p)
    r = kda.kda_chunk_bwd(p, c.do, c.dht, saved=sv)
    torch.cuda.synchronize()
    return dict(o=o, ht=ht, dq=r[0], dk=r[1], dv=r[2], dg=r[3], dbeta=r[4], dh0=r[5])


def compare(case, got, ref, G, tol):
    BT, HV = case.B * case.T, case.H
    for name, x in got.items():
        if x is None:
            continue
        a = np64(x)
        if name in ("o", "dv"):
            a = a.reshape(BT, HV, -1)
        elif name in ("dq", "dk"):
            a = a.reshape(BT, HV // G, -1)
        elif name == "dbeta":
            a = a.reshape(BT, HV)
        elif name == "dg":
            a = a.reshape(ref["dg"].shape)
        check_close(name, a, ref[name], tol)


@pytest.mark.parametrize("io,gate,K,G", [("bf16", "channel", 128, 2), ("fp32", "channel", 64, 4),
                                         ("bf16", "scalar", 128, 3)])
def test_grouped_heads_match_oracle(io, gate, K, G):
    case, q, k = gva_case(io, gate, 2, 130, 2, G, K, 91)
    compare(case, gpu(case, q, k), oracle(case, G), G, TOL[io])


def test_grouped_heads_packed_and_saved():
    case, q, k = gva_case("bf16", "channel", 1, None, 2, 2, 128, 92, lengths=[5, 64, 70])
    r0 = gpu(case, q, k, policy=0)
    ra = gpu(case, q, k, policy=1)
    compare(case, r0, oracle(case, 2), 2, TOL["bf16"])
    for name in r0:
        if r0[name] is not None:
            assert torch.equal(r0[name], ra[name]), name


@pytest.mark.parametrize("io,K", [("fp32", 64), ("bf16", 128)])
def test_grouped_heads_recurrent(io, K):
    import chunkwise_delta_rule_gb300 as kda
    case, q, k = gva_case(io, "channel", 2, 20, 2, 2, K, 93)
    c = case.to("cuda")
    p = kda.make_problem(q.cuda(), k.cuda(), c.v, c.g, c.beta, gate="channel", scale=case.scale, initial_state=c.h0)
    o, ht = kda.kda_recurrent_fwd(p)
    torch.cuda.synchronize()
    ref = oracle(case, 2, backward=False)
    check_close("o", np64(o).reshape(case.B * case.T, case.H, -1), ref["o"], TOL[io])
    check_close("ht", np64(ht), ref["ht"], TOL[io])
