"""GPU parity of the GatedDeltaNet-2 rule (erase vector b on the key axis,
write vector w on the value axis; "GatedDeltaNet-2 (NVlabs) — official spec
transcription", §3) against the FP64 recurrence oracle: o, ht and every
gradient, derase and dwrite included, on the chunked path (both policies, all
gate kinds, both I/O types, packed sequences, with the prologue) and the
forward of the token-by-token path. Inputs: the workload recipe for q, k, v,
g, h0, do, dht; b = 2 sigmoid(N(0, 1)) in (0, 2), w = sigmoid(N(0, 1)) in
(0, 1) per element (the spec's typical ranges)."""

import numpy as np
import pytest
import torch

from oracle.cases import packed, run_oracle_prologue_arrays
from tests.helpers import check_close, np64
from workloads import make_case

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}


def gdn2_case(io, gate, B, T, H, K, seed, lengths=None, V=None):
    case = make_case(io=io, gate=gate, B=B, T=T, H=H, K=K, V=V or K, seed=seed, lengths=lengths)
    gen = torch.Generator().manual_seed(seed + 2000)
    dt = case.q.dtype
    b = (2.0 * torch.sigmoid(torch.randn(case.k.shape, generator=gen))).to(dt)
    w = torch.sigmoid(torch.randn(case.v.shape, generator=gen)).to(dt)
    return case, b, w


def oracle(case, b, w, backward=True, prologue=None):
    p = packed(case)
    BT = case.B * case.T
    kw = dict(A_log=None, dt_bias=None, lower_bound=0.0, eps=1e-6, qk_norm=False)
    if prologue:
        kw.update(prologue)
    return run_oracle_prologue_arrays(p["q"], p["k"], p["v"], None, p["g"], scale=case.scale, gate=case.gate,
                                      seq_starts=case.seq_starts, h0=p["h0"], do=p["do"], dht=p["dht"],
                                      backward=backward, erase=np64(b).reshape(BT, case.H, -1),
                                      write=np64(w).reshape(BT, case.H, -1), **kw)


def gpu(case, b, w, policy=0, prologue=None):
    import chunkwise_delta_rule_gb300 as kda
    c = case.to("cuda")
    extra = {}
    if prologue:
        extra = dict(A_log=torch.tensor(prologue["A_log"], dtype=torch.float32, device="cuda"),
                     dt_bias=torch.tensor(prologue["dt_bias"], dtype=torch.float32, device="cuda"),
                     qk_l2norm=prologue["qk_norm"])
    p = kda.make_problem(c.q, c.k, c.v, c.g, None, gate=case.gate, scale=case.scale, initial_state=c.h0,
                         cu_seqlens=c.cu_seqlens, save_policy=policy, erase=b.cuda(), write=w.cuda(), **extra)
    o, ht, sv = kda.kda_chunk_fwd(p)
    r = kda.kda_chunk_bwd(p, c.do, c.dht, saved=sv)
    torch.cuda.synchronize()
    assert r[4] is None
    out = dict(o=o, ht=ht, dq=r[0], dk=r[1], dv=r[2], dg=r[3], dh0=r[5], derase=r[-2], dwrite=r[-1])
    if prologue:
        out.update(dA_log=r[6], ddt_bias=r[7])
    return out


def compare(case, got, ref, tol):
    BT, H = case.B * case.T, case.H
    for name, x in got.items():
        if x is None:
            assert ref.get(name) is None, name
            continue
        a = np64(x)
        if name in ("o", "dq", "dk", "dv", "derase", "dwrite"):
            a = a.reshape(BT, H, -1)
        elif name == "dg":
            a = a.reshape(ref["dg"].shape)
        check_close(name, a, ref[name], tol)


@pytest.mark.parametrize("io,gate,K", [("fp32", "channel", 64), ("bf16", "channel", 128), ("fp32", "scalar", 128),
                                       ("bf16", "none", 64)])
def test_gdn2_matches_oracle(io, gate, K):
    case, b, w = gdn2_case(io, gate, 2, 150, 2, K, 81)
    compare(case, gpu(case, b, w), oracle(case, b, w), TOL[io])


def test_gdn2_packed_sequences_and_policies():
    case, b, w = gdn2_case("bf16", "channel", 1, None, 2, 128, 82, lengths=[1, 64, 65, 3, 90])
    ref = oracle(case, b, w)
    r0 = gpu(case, b, w, policy=0)
    ra = gpu(case, b, w, policy=1)
    compare(case, r0, ref, TOL["bf16"])
    for name in r0:
        if r0[name] is not None:
            assert torch.equal(r0[name], ra[name]), name


def test_gdn2_with_the_prologue():
    case, b, w = gdn2_case("fp32", "channel", 1, 100, 2, 64, 83)
    rng = np.random.default_rng(84)
    case.q = case.q * torch.tensor(rng.uniform(0.5, 3.0, (1, 100, 2, 1)), dtype=case.q.dtype)
    case.k = case.k * torch.tensor(rng.uniform(0.5, 3.0, (1, 100, 2, 1)), dtype=case.k.dtype)
    case.g = torch.tensor(rng.standard_normal(case.g.shape), dtype=torch.float32)
    pro = dict(A_log=np.log(rng.uniform(1, 4, 2)), dt_bias=rng.normal(-4.0, 1.0, (2, 64)), qk_norm=True)
    compare(case, gpu(case, b, w, prologue=pro), oracle(case, b, w, prologue=pro), TOL["fp32"])


@pytest.mark.parametrize("io,K,V", [("fp32", 64, 64), ("bf16", 128, 128), ("bf16", 128, 256)])
def test_gdn2_recurrent_matches_oracle(io, K, V):
    import chunkwise_delta_rule_gb300 as kda
    case, b, w = gdn2_case(io, "channel", 2, 30, 2, K, 85, V=V)
    c = case.to("cuda")
    p = kda.make_problem(c.q, c.k, c.v, c.g, None, gate="channel", scale=case.scale, initial_state=c.h0,
                         erase=b.cuda(), write=w.cuda())
    o, ht = kda.kda_recurrent_fwd(p)
    torch.cuda.synchronize()
    ref = oracle(case, b, w, backward=False)
    check_close("o", np64(o).reshape(case.B * case.T, case.H, -1), ref["o"], TOL[io])
    check_close("ht", np64(ht), ref["ht"], TOL[io])
