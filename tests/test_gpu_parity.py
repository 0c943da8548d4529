"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Tolerances (normwise relative error per tensor, all values finite):
1e-4 for fp32 I/O and 2e-2 for bf16 I/O, for o, ht, dq, dk, dv, dg, dbeta
and dh0; a reference with near-zero norm uses max-abs <= 1e-6 instead.
"""

import numpy as np
import pytest
import torch

from tests.helpers import check_close, np64, record_errors, run_oracle, run_oracle_pairs
from workloads import CONFIGS, make_case, make_config_case

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}
NAMES = ("o", "ht", "dq", "dk", "dv", "dg", "dbeta", "dh0")


def gpu_run(case, policy=0, need_bwd=True, schedule=0):
    import chunkwise_delta_rule_gb300 as kda
    c = case.to("cuda")
    p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate=case.gate, scale=case.scale,
                         initial_state=c.h0, cu_seqlens=c.cu_seqlens, save_policy=policy, schedule=schedule)
    wsf = torch.empty(max(kda.kda_workspace_size(p, False), 1), dtype=torch.uint8, device="cuda")
    o, ht, sv = kda.kda_chunk_fwd(p, workspace=wsf)
    assert kda.kda_device_status(p, wsf) == (0, 0), "device error word set by the forward"
    out = dict(o=o, ht=ht)
    if need_bwd:
        wsb = torch.empty(max(kda.kda_workspace_size(p, True), 1), dtype=torch.uint8, device="cuda")
        dq, dk, dv, dg, dbeta, dh0 = kda.kda_chunk_bwd(p, c.do, c.dht, saved=sv, workspace=wsb)
        assert kda.kda_device_status(p, wsb) == (0, 0), "device error word set by the backward"
        out.update(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dh0=dh0)
    torch.cuda.synchronize()
    return out


def packed_np(case, out):
    """GPU outputs as float64 arrays on the packed token axis."""
    BT = case.B * case.T
    res = {}
    for k, x in out.items():
        if x is None:
            res[k] = None
            continue
        a = np64(x)
        if k in ("ht", "dh0"):
            res[k] = a
        elif k in ("dbeta",):
            res[k] = a.reshape(BT, case.H)
        elif k == "dg":
            res[k] = a.reshape((BT, case.H) + tuple(a.shape[3:]))
        else:
            res[k] = a.reshape(BT, case.H, -1)
    return res


def compare_full(case, got, ref, tol):
    errs = {}
    for name in NAMES:
        if name not in got:
            continue
        if name == "dg" and case.gate == "none":
            assert got["dg"] is None
            continue
        errs[name] = check_close(name, got[name], ref[name], tol)
    return errs


SMALL = [
    dict(io="fp32", gate="channel", B=2, T=200, H=2, K=64, V=64),
    dict(io="fp32", gate="scalar", B=2, T=130, H=2, K=64, V=64),
    dict(io="fp32", gate="none", B=1, T=129, H=3, K=64, V=64),
    dict(io="fp32", gate="channel", B=1, T=192, H=2, K=128, V=128),
    dict(io="bf16", gate="channel", B=2, T=150, H=2, K=128, V=128),
    dict(io="bf16", gate="scalar", B=1, T=257, H=2, K=128, V=128),
    dict(io="bf16", gate="none", B=2, T=100, H=2, K=128, V=128, h0=False, dht=False),
    dict(io="bf16", gate="channel", B=1, T=64, H=1, K=64, V=64),
    dict(io="fp32", gate="channel", B=3, T=1, H=2, K=64, V=64),
]


@pytest.mark.parametrize("kw", SMALL, ids=lambda kw: "{io}-{gate}-B{B}T{T}H{H}K{K}".format(**kw))
def test_small_cases_match_oracle(kw):
    case = make_case(seed=17, **kw)
    got = packed_np(case, gpu_run(case))
    ref = run_oracle(case)
    compare_full(case, got, ref, TOL[case.io])


@pytest.mark.parametrize("io,K", [("fp32", 64), ("bf16", 64), ("bf16", 48)])
def test_packed_sequences(io, K):
    # one-token, exactly-one-chunk, one-past-a-chunk, two-chunk and ragged sequences (bf16 at
    # widths below 128 runs zero-padded on the tensor-core path)
    case = make_case(io=io, gate="channel", B=1, H=2, K=K, V=64, seed=31,
                     lengths=[1, 64, 65, 130, 3, 200])
    got = packed_np(case, gpu_run(case))
    compare_full(case, got, run_oracle(case), TOL[io])


@pytest.mark.parametrize("io,D", [("fp32", 64), ("bf16", 128), ("bf16", 64)])
@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_strong_decay_takes_the_subchunk_path(gate, io, D):
    """g around -4: the in-chunk gate range exceeds the single-anchor and
    centering thresholds, so the 16-token anchored paths run (the CUDA-core
    prep of wide chunks on the tensor-core path, which bf16 at 64 reaches
    zero-padded to 128); they must stay within the I/O dtype's tolerance."""
    case = make_case(io=io, gate=gate, B=1, T=200, H=2, K=D, V=D, seed=5, g_shift=-4.0,
                     g_min=-8.0)
    g = case.g if gate == "channel" else case.g[..., None]
    G = torch.cumsum(g.double(), dim=1) / np.log(2.0)
    assert float((G[:, :64].max(dim=1).values - G[:, :64].min(dim=1).values).max()) > 80
    got = packed_np(case, gpu_run(case))
    compare_full(case, got, run_oracle(case), TOL[io])


def test_mixed_wide_and_narrow_chunks():
    """Packed sequences where some chunks have strong decay and others mild:
    the tensor-core prep and the wide-chunk prep share one launch sequence."""
    case = make_case(io="bf16", gate="channel", B=1, H=2, K=128, V=128, seed=8,
                     lengths=[64, 150, 70])
    g = case.g.clone()
    g[0, 64:214] = torch.clamp(g[0, 64:214] - 4.0, min=-8.0)   # the middle sequence decays strongly
    case.g = g
    got = packed_np(case, gpu_run(case))
    compare_full(case, got, run_oracle(case), TOL["bf16"])


@pytest.mark.parametrize("mode", ["zero_every3", "tiny"])
def test_zero_and_tiny_beta(mode):
    case = make_case(io="fp32", gate="channel", B=1, T=130, H=2, K=64, V=64, seed=9, beta_mode=mode)
    got = packed_np(case, gpu_run(case))
    compare_full(case, got, run_oracle(case), TOL["fp32"])


@pytest.mark.parametrize("policy", [0, 1], ids=["recompute", "save"])
@pytest.mark.parametrize("gate", ["channel", "scalar"])
@pytest.mark.parametrize("mode", ["zero_every3", "tiny"])
def test_zero_and_tiny_beta_tensor_core(mode, gate, policy):
    """beta = 0 on every third token, or 1e-8 everywhere, on the tensor-core path (bf16, K = V = 128)
    under both policies; the save policy's backward runs in time pieces (6 chunks, the last ragged).
    dbeta is formed undivided (<k_i gamma_i, E_bar_i> + <v_i, P_i>), so it stays finite and exact
    at beta = 0 ("ReWY" paper, numerical coverage: zero and tiny beta)."""
    case = make_case(io="bf16", gate=gate, B=2, T=330, H=2, K=128, V=128, seed=10, beta_mode=mode)
    got = packed_np(case, gpu_run(case, policy=policy))
    errs = compare_full(case, got, run_oracle(case), TOL["bf16"])
    record_errors(f"beta_{mode}:{gate}:{'save' if policy else 'recompute'}", errs, tol=TOL["bf16"])


@pytest.mark.parametrize("io,D,H", [("fp32", 64, 2), ("bf16", 128, 2), ("bf16", 128, 48)])
def test_policies_agree_and_runs_are_deterministic(io, D, H):
    """Repeated runs are bitwise identical (no atomics); the save-intermediates
    policy agrees with the recompute policy within the I/O tolerance. With 96
    (sequence, head) pairs the saved states come from the combined output scan
    rather than from a second scan beside it."""
    case = make_case(io=io, gate="channel", B=2, T=300, H=H, K=D, V=D, seed=41)
    r1 = gpu_run(case, policy=0)
    r2 = gpu_run(case, policy=0)
    ra = gpu_run(case, policy=1)
    for name in NAMES:
        assert torch.equal(r1[name], r2[name]), name
        check_close(name, np64(ra[name]), np64(r1[name]), TOL[io])


@pytest.mark.parametrize("gate,policy", [("channel", 1), ("scalar", 0), ("none", 1)])
def test_backward_schedules_agree_bitwise(gate, policy):
    """One reverse-scan pass, 2, 3 or 4 time pieces (the scan of a piece running beside the consumer of
    the one before, the state adjoint handed on in fp32) and the joint schedule (scans and consumer in
    one launch, the consumer waiting for each chunk's ready flag; one pass under the recompute policy)
    give bitwise identical results, which match the oracle. 10 chunks per sequence, the last one
    ragged."""
    case = make_case(io="bf16", gate=gate, B=2, T=610, H=3, K=128, V=128, seed=44)
    ref = gpu_run(case, policy=policy, schedule=1)
    for sch in (0, 2, 3, 4, 9):
        r = gpu_run(case, policy=policy, schedule=sch)
        for name in NAMES:
            if ref[name] is not None:
                assert torch.equal(r[name], ref[name]), (sch, name)
    compare_full(case, packed_np(case, ref), run_oracle(case), TOL["bf16"])


def test_split_call_chains_through_the_state():
    import chunkwise_delta_rule_gb300 as kda
    case = make_case(io="fp32", gate="channel", B=1, T=200, H=2, K=64, V=64, seed=43).to("cuda")
    full = gpu_run(case)
    cut = 70

    def part(a, b, h0, dht):
        sl = lambda x: x[:, a:b].contiguous()  # noqa: E731
        p = kda.make_problem(sl(case.q), sl(case.k), sl(case.v), sl(case.g), sl(case.beta),
                             gate="channel", initial_state=h0)
        o, ht, _ = kda.kda_chunk_fwd(p)
        return p, o, ht

    pa, oa, hta = part(0, cut, case.h0, None)
    pb, ob, htb = part(cut, 200, hta, None)
    gb = kda.kda_chunk_bwd(pb, case.do[:, cut:].contiguous(), case.dht)
    ga = kda.kda_chunk_bwd(pa, case.do[:, :cut].contiguous(), gb[5])
    torch.cuda.synchronize()
    tol = 1e-5
    assert float((torch.cat([oa, ob], 1) - full["o"]).norm() / full["o"].norm()) < tol
    assert float((htb - full["ht"]).norm() / full["ht"].norm()) < tol
    for i, name in enumerate(("dq", "dk", "dv", "dg", "dbeta")):
        cat = torch.cat([ga[i], gb[i]], 1)
        assert float((cat - full[name]).norm() / full[name].norm()) < tol, name
    assert float((ga[5] - full["dh0"]).norm() / full["dh0"].norm()) < tol


def test_empty_sequence_passes_states_through():
    import chunkwise_delta_rule_gb300 as kda
    case = make_case(io="bf16", gate="channel", B=2, T=0, H=2, K=64, V=64, seed=1).to("cuda")
    p = kda.make_problem(case.q, case.k, case.v, case.g, case.beta, gate="channel",
                         initial_state=case.h0)
    o, ht, _ = kda.kda_chunk_fwd(p)
    dq, dk, dv, dg, dbeta, dh0 = kda.kda_chunk_bwd(p, case.do, case.dht)
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.equal(ht, case.h0) and torch.equal(dh0, case.dht)


def test_autograd_wrapper_matches_direct_calls():
    import chunkwise_delta_rule_gb300 as kda
    case = make_case(io="bf16", gate="scalar", B=1, T=140, H=2, K=128, V=128, seed=47).to("cuda")
    ref = gpu_run(case)
    q, k, v, g, beta, h0 = (x.clone().requires_grad_(True) for x in
                            (case.q, case.k, case.v, case.g, case.beta, case.h0))
    o, ht = kda.chunk_kda(q, k, v, g, beta, gate="scalar", initial_state=h0)
    loss = (o.float() * case.do.float()).sum() + (ht * case.dht).sum()
    loss.backward()
    assert torch.equal(o, ref["o"]) and torch.equal(ht, ref["ht"])
    for t, name in ((q, "dq"), (k, "dk"), (v, "dv"), (g, "dg"), (beta, "dbeta"), (h0, "dh0")):
        assert torch.equal(t.grad, ref[name]), name


def test_cuda_graph_replay_with_new_inputs():
    """Capture forward + backward once, replay with different inputs copied
    into the captured buffers; results equal eager calls on those inputs."""
    import chunkwise_delta_rule_gb300 as kda
    a = make_case(io="bf16", gate="channel", B=1, T=200, H=2, K=128, V=128, seed=51).to("cuda")
    b = make_case(io="bf16", gate="channel", B=1, T=200, H=2, K=128, V=128, seed=52).to("cuda")
    st = a.to("cuda")
    p = kda.make_problem(st.q, st.k, st.v, st.g, st.beta, gate="channel", initial_state=st.h0)
    wf = torch.empty(kda.kda_workspace_size(p, False), dtype=torch.uint8, device="cuda")
    wb = torch.empty(kda.kda_workspace_size(p, True), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kda.kda_chunk_fwd(p, workspace=wf)
        kda.kda_chunk_bwd(p, st.do, st.dht, workspace=wb)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = kda.kda_chunk_fwd(p, workspace=wf)
        grads = kda.kda_chunk_bwd(p, st.do, st.dht, workspace=wb)
    for name in ("q", "k", "v", "g", "beta", "h0", "do", "dht"):
        getattr(st, name).copy_(getattr(b, name))
    g.replay()
    torch.cuda.synchronize()
    ref = gpu_run(b)
    assert torch.equal(outs[0], ref["o"]) and torch.equal(outs[1], ref["ht"])
    for i, name in enumerate(("dq", "dk", "dv", "dg", "dbeta", "dh0")):
        assert torch.equal(grads[i], ref[name]), name


def _sample_pairs(case, idx):
    """(sequence, head) pairs the oracle recomputes at full size: every pair of the tiny workload;
    otherwise every sequence with heads spread over the head range (16 pairs for the equal-length
    batches, two heads of each packed sequence, whose lengths all end in a ragged chunk). Each pair
    spans all of its sequence's chunks, so every time piece of the backward is covered."""
    N, H = case.N, case.H
    if idx == 1:
        return [(n, h) for n in range(N) for h in range(H)]
    per_seq = max(2, 16 // N)
    out = []
    for n in range(N):
        for j in range(per_seq):
            h = (n * 5 + j * (H // per_seq) + (H - 1) * (j == per_seq - 1)) % H
            if (n, h) not in out:
                out.append((n, h))
    return out


# The benchmark times the save policy with the library's default backward schedule (the joint
# launch when the sequence x head pairs fill at most half of the SMs, else one pass); the recompute
# policy runs beside it.
FULL_SIZE_RUNS = [dict(policy=1, schedule=0), dict(policy=0, schedule=0)]


@pytest.mark.parametrize("run", FULL_SIZE_RUNS, ids=["save-default-schedule", "recompute"])
@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_full_size_configs_on_sampled_heads(idx, run):
    """The benchmark workloads at full size. The save-policy run is the launch configuration the
    benchmark times (its forward keeps the intermediates, its backward runs in the library's default
    schedule); the oracle recomputes sampled (sequence, head) pairs one by one, and every output
    must be finite everywhere."""
    case = make_config_case(idx)
    out = gpu_run(case, policy=run["policy"], schedule=run["schedule"])
    for name, x in out.items():
        if x is not None:
            assert bool(torch.isfinite(x.float()).all()), name
    got = packed_np(case, out)
    del out
    pairs = _sample_pairs(case, idx)
    ref = run_oracle_pairs(case, pairs)
    ss = case.seq_starts
    tol = TOL[CONFIGS[idx]["io"]]
    errs = {}
    for name in NAMES:
        if name == "dg" and case.gate == "none":
            continue
        g_parts, r_parts = [], []
        for i, (n, h) in enumerate(pairs):
            if name in ("ht", "dh0"):
                g_parts.append(got[name][n, h])
            else:
                g_parts.append(got[name][ss[n]:ss[n + 1], h])
            r_parts.append(ref[name][i])
        errs[name] = check_close(f"config{idx}:{name}", np.concatenate([x.ravel() for x in g_parts]),
                                 np.concatenate([x.ravel() for x in r_parts]), tol)
    record_errors(f"{CONFIGS[idx]['name']}:{'save' if run['policy'] else 'recompute'}", errs,
                  pairs=len(pairs), tol=tol)
