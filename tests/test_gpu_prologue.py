"""GPU parity of the operator with its prologue on (gate activation with A_log
and dt_bias, q/k L2 normalisation) against the FP64 oracle composition
(``oracle.prologue`` + the recurrence): o, ht and every gradient, including
dA_log and dt_bias's, for the chunked path (both policies) and the forward of
the token-by-token path.

Raw inputs: q, k are the workload's unit vectors times a per-(token, head)
norm drawn in [0.5, 3]; the raw gate ~ N(0, 1); A_log = log U(1, 4) per head;
dt_bias = the softplus inverse of dt ~ logU(1e-3, 1e-1) ("GatedDeltaNet-2
(NVlabs) — official spec transcription", §4.4 init), so the activated decay
stays inside the library's bound. Tolerances as for the plain operator.
"""

import math

import numpy as np
import pytest
import torch

from oracle.cases import packed, run_oracle_prologue_arrays
from tests.helpers import check_close, np64
from workloads import make_case

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}


def prologue_case(io, gate, B, T, H, K, seed, lb, norm=True, act=True):
    """Raw inputs: q, k rescaled only when the operator normalises them (unit
    keys keep the delta rule contractive otherwise); the gate raw only when the
    operator activates it."""
    case = make_case(io=io, gate=gate, B=B, T=T, H=H, K=K, V=K, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1000)
    dt = torch.exp(torch.rand((H, K) if gate == "channel" else (H,), generator=gen)
                   * (math.log(0.1) - math.log(1e-3)) + math.log(1e-3))
    extra = dict(
        qn=torch.rand(B, T, H, 1, generator=gen) * 2.5 + 0.5,
        kn=torch.rand(B, T, H, 1, generator=gen) * 2.5 + 0.5,
        g_raw=torch.randn(case.g.shape, generator=gen),
        A_log=torch.log(torch.rand(H, generator=gen) * 3 + 1),
        dt_bias=dt + torch.log(-torch.expm1(-dt)),
    )
    if norm:
        case.q = (case.q.float() * extra["qn"]).to(case.q.dtype)
        case.k = (case.k.float() * extra["kn"]).to(case.k.dtype)
    if act:
        case.g = extra["g_raw"].float()
    return case, extra["A_log"].float(), extra["dt_bias"].float(), lb


def oracle(case, A_log, dt_bias, lb, norm, act, backward=True):
    p = packed(case)
    return run_oracle_prologue_arrays(p["q"], p["k"], p["v"], p["beta"], p["g"],
                                      A_log=np64(A_log) if act else None, dt_bias=np64(dt_bias) if act else None,
                                      lower_bound=lb, eps=1e-6, scale=case.scale, gate=case.gate,
                                      seq_starts=case.seq_starts, h0=p["h0"], do=p["do"], dht=p["dht"],
                                      backward=backward, qk_norm=norm)


def gpu(case, A_log, dt_bias, lb, norm, act, policy=0):
    import chunkwise_delta_rule_gb300 as kda
    c = case.to("cuda")
    p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate=case.gate, scale=case.scale, initial_state=c.h0,
                         save_policy=policy, A_log=A_log.cuda() if act else None,
                         dt_bias=dt_bias.cuda() if act else None, lower_bound=lb, qk_l2norm=norm)
    o, ht, sv = kda.kda_chunk_fwd(p)
    r = kda.kda_chunk_bwd(p, c.do, c.dht, saved=sv)
    torch.cuda.synchronize()
    out = dict(o=o, ht=ht, dq=r[0], dk=r[1], dv=r[2], dg=r[3], dbeta=r[4], dh0=r[5])
    if act:
        out.update(dA_log=r[6], ddt_bias=r[7])
    return out


def compare(case, got, ref, tol):
    BT, H = case.B * case.T, case.H
    for name, x in got.items():
        a = np64(x)
        if name in ("o", "dq", "dk", "dv"):
            a = a.reshape(BT, H, -1)
        elif name == "dbeta":
            a = a.reshape(BT, H)
        elif name == "dg":
            a = a.reshape(ref["dg"].shape)
        check_close(name, a, ref[name], tol)


CASES = [
    ("fp32", "channel", 64, 0.0, True, True),
    ("bf16", "channel", 128, 0.0, True, True),
    ("bf16", "channel", 128, -5.0, True, True),
    ("bf16", "scalar", 128, 0.0, True, True),
    ("fp32", "scalar", 64, -3.0, False, True),
    ("bf16", "channel", 128, 0.0, True, False),
]


@pytest.mark.parametrize("io,gate,K,lb,norm,act", CASES,
                         ids=lambda v: str(v))
def test_prologue_matches_oracle(io, gate, K, lb, norm, act):
    case, A, dt, lb = prologue_case(io, gate, 2, 150, 2, K, 71, lb, norm, act)
    got = gpu(case, A, dt, lb, norm, act)
    ref = oracle(case, A, dt, lb, norm, act)
    compare(case, got, ref, TOL[io])


def test_prologue_policies_agree_and_are_deterministic():
    case, A, dt, lb = prologue_case("bf16", "channel", 2, 200, 2, 128, 72, 0.0)
    r1 = gpu(case, A, dt, lb, True, True, policy=0)
    r2 = gpu(case, A, dt, lb, True, True, policy=0)
    ra = gpu(case, A, dt, lb, True, True, policy=1)
    for name in r1:
        assert torch.equal(r1[name], r2[name]), name
        check_close(name, np64(ra[name]), np64(r1[name]), TOL["bf16"])


@pytest.mark.parametrize("io,gate,K,lb", [("fp32", "channel", 64, 0.0), ("bf16", "channel", 128, -5.0),
                                          ("bf16", "scalar", 128, 0.0), ("fp32", "channel", 192, 0.0)])
def test_recurrent_prologue_matches_oracle(io, gate, K, lb):
    import chunkwise_delta_rule_gb300 as kda
    case, A, dt, lb = prologue_case(io, gate, 2, 40, 2, K, 73, lb)
    c = case.to("cuda")
    p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate=gate, scale=case.scale, initial_state=c.h0,
                         A_log=A.cuda(), dt_bias=dt.cuda(), lower_bound=lb, qk_l2norm=True)
    o, ht = kda.kda_recurrent_fwd(p)
    torch.cuda.synchronize()
    ref = oracle(case, A, dt, lb, True, True, backward=False)
    check_close("o", np64(o).reshape(case.B * case.T, case.H, -1), ref["o"], TOL[io])
    check_close("ht", np64(ht), ref["ht"], TOL[io])


def test_autograd_wrapper_returns_parameter_gradients():
    import chunkwise_delta_rule_gb300 as kda
    case, A, dt, lb = prologue_case("bf16", "channel", 1, 100, 2, 128, 74, 0.0)
    c = case.to("cuda")
    q, k, v, g, beta = [x.clone().requires_grad_(True) for x in (c.q, c.k, c.v, c.g, c.beta)]
    Ag, dtg = A.cuda().requires_grad_(True), dt.cuda().requires_grad_(True)
    o, ht = kda.chunk_kda(q, k, v, g, beta, gate="channel", scale=case.scale, initial_state=c.h0,
                          A_log=Ag, dt_bias=dtg, use_qk_l2norm_in_kernel=True)
    torch.autograd.backward([o, ht], [c.do, c.dht])
    ref = gpu(case, A, dt, 0.0, True, True)
    assert torch.equal(Ag.grad, ref["dA_log"]) and torch.equal(dtg.grad, ref["ddt_bias"])
    assert torch.equal(q.grad, ref["dq"]) and torch.equal(g.grad, ref["dg"])
