"""GPU parity at key and value widths other than K = V = 64 or 128 (served
zero-padded to the working width, 64, 128 or 256, and cropped back; value
widths above the value-block width, 128 or 256 when K > 128, as value blocks,
each a value head of its own), alone and together with grouped value heads,
the GatedDeltaNet-2 vectors and the prologue, against the FP64 oracle at the
true widths."""

import numpy as np
import pytest
import torch

from oracle.cases import packed, run_oracle_prologue_arrays
from tests.helpers import check_close, np64
from workloads import make_case

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}


def width_case(io, gate, B, T, H, K, V, seed):
    return make_case(io=io, gate=gate, B=B, T=T, H=H, K=K, V=V, seed=seed)


def run_both(case, G=1, gdn2=False, prologue=False):
    import chunkwise_delta_rule_gb300 as kda
    gen = torch.Generator().manual_seed(777)
    BT, HV = case.B * case.T, case.H
    qk = (case.q[:, :, ::G].contiguous(), case.k[:, :, ::G].contiguous())
    if prologue:   # raw q, k and gate
        qk = tuple((x.float() * (torch.rand(x.shape[:3] + (1,), generator=gen) * 2 + 0.5)).to(x.dtype) for x in qk)
        case.g = torch.randn(case.g.shape, generator=gen) * 0.5
        A = torch.log(torch.rand(HV, generator=gen) * 3 + 1)
        dtb = torch.randn((HV, case.K), generator=gen) * 0.3 - 4.0
    b = w = None
    if gdn2:
        b = (2 * torch.sigmoid(torch.randn(case.k.shape, generator=gen))).to(case.q.dtype)
        w = torch.sigmoid(torch.randn(case.v.shape, generator=gen)).to(case.q.dtype)
    # oracle at the true widths, q and k repeated per value head
    case.q, case.k = qk[0].repeat_interleave(G, 2), qk[1].repeat_interleave(G, 2)
    p = packed(case)
    ref = run_oracle_prologue_arrays(p["q"], p["k"], p["v"], None if gdn2 else p["beta"], p["g"],
                                     A_log=np64(A) if prologue else None, dt_bias=np64(dtb) if prologue else None,
                                     lower_bound=0.0, eps=1e-6, scale=case.scale, gate=case.gate,
                                     seq_starts=case.seq_starts, h0=p["h0"], do=p["do"], dht=p["dht"],
                                     qk_norm=prologue, erase=None if b is None else np64(b).reshape(BT, HV, -1),
                                     write=None if w is None else np64(w).reshape(BT, HV, -1))
    for name in ("dq", "dk"):
        ref[name] = ref[name].reshape(BT, HV // G, G, -1).sum(axis=2)
    c = case.to("cuda")
    extra = dict(A_log=A.cuda(), dt_bias=dtb.cuda(), qk_l2norm=True) if prologue else {}
    if gdn2:
        extra.update(erase=b.cuda(), write=w.cuda())
    prob = kda.make_problem(qk[0].cuda(), qk[1].cuda(), c.v, c.g, None if gdn2 else c.beta, gate=case.gate,
                            scale=case.scale, initial_state=c.h0, cu_seqlens=c.cu_seqlens, **extra)
    o, ht, sv = kda.kda_chunk_fwd(prob)
    r = kda.kda_chunk_bwd(prob, c.do, c.dht, saved=sv)
    torch.cuda.synchronize()
    got = dict(o=o, ht=ht, dq=r[0], dk=r[1], dv=r[2], dg=r[3], dbeta=r[4], dh0=r[5])
    if prologue:
        got.update(dA_log=r[6], ddt_bias=r[7])
    if gdn2:
        got.update(derase=r[-2], dwrite=r[-1])
    return got, ref


def compare(case, got, ref, G, tol):
    BT, HV = case.B * case.T, case.H
    for name, x in got.items():
        if x is None:
            continue
        a = np64(x)
        if name in ("o", "dv", "derase", "dwrite"):
            a = a.reshape(BT, HV, -1)
        elif name in ("dq", "dk"):
            a = a.reshape(BT, HV // G, -1)
        elif name == "dbeta":
            a = a.reshape(BT, HV)
        elif name == "dg":
            a = a.reshape(ref["dg"].shape)
        check_close(name, a, ref[name], tol)


@pytest.mark.parametrize("io,gate,K,V", [("bf16", "channel", 80, 112), ("fp32", "channel", 32, 48),
                                         ("bf16", "scalar", 128, 64), ("fp32", "none", 96, 128)])
def test_unequal_widths_match_oracle(io, gate, K, V):
    case = width_case(io, gate, 2, 100, 2, K, V, 101)
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL[io])


def test_widths_with_grouped_heads_gdn2_and_prologue():
    case = width_case("bf16", "channel", 1, 90, 4, 96, 80, 102)
    got, ref = run_both(case, G=2, gdn2=True, prologue=True)
    compare(case, got, ref, 2, TOL["bf16"])


# value widths above 128: NB = ceil(V / 128) blocks of ceil(V / NB) columns; 256 runs as two
# 128-wide blocks on the tensor-core path, 201 as two blocks of 101 with the value rows padded
@pytest.mark.parametrize("io,gate,K,V", [("bf16", "channel", 128, 256), ("fp32", "scalar", 64, 201),
                                         ("bf16", "none", 96, 160), ("fp32", "channel", 128, 384)])
def test_wide_values_match_oracle(io, gate, K, V):
    case = width_case(io, gate, 2, 100, 2, K, V, 103)
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL[io])


def test_wide_values_with_grouped_heads_gdn2_and_prologue():
    case = width_case("bf16", "channel", 1, 90, 4, 128, 192, 104)
    got, ref = run_both(case, G=2, gdn2=True, prologue=True)
    compare(case, got, ref, 2, TOL["bf16"])


def test_wide_values_saved_equals_recomputed():
    import chunkwise_delta_rule_gb300 as kda
    case = width_case("bf16", "channel", 1, 150, 2, 128, 256, 105)
    c = case.to("cuda")
    out = []
    for policy in (0, 1):
        p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate="channel", scale=case.scale, initial_state=c.h0,
                             save_policy=policy)
        o, ht, sv = kda.kda_chunk_fwd(p)
        out.append((o, ht) + tuple(kda.kda_chunk_bwd(p, c.do, c.dht, saved=sv)))
    torch.cuda.synchronize()
    for a, b in zip(*out):
        if a is not None:
            assert torch.equal(a, b)


# key widths above 128: every key- and value-side tensor runs zero-padded to 256 (K = V = 256 as
# is) on the fp32 CUDA-core kernels, which take the features in blocks of 128
@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
@pytest.mark.parametrize("K,V", [(192, 160), (256, 256), (160, 64)])
def test_wide_keys_match_oracle(gate, K, V):
    case = width_case("bf16", gate, 2, 100, 2, K, V, 106)
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL["bf16"])


@pytest.mark.parametrize("gate,K,V", [("channel", 256, 256), ("scalar", 200, 136)])
def test_wide_keys_fp32_packed(gate, K, V):
    case = make_case(io="fp32", gate=gate, B=1, H=2, K=K, V=V, seed=107, lengths=[1, 64, 130, 3, 70])
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL["fp32"])


def test_wide_keys_strong_decay():
    """g around -4 at K = 256: the in-chunk gate range passes the centering
    threshold, so the consumer's 16-token anchored path runs in both feature
    blocks."""
    case = make_case(io="bf16", gate="channel", B=1, T=200, H=2, K=256, V=256, seed=108, g_shift=-4.0,
                     g_min=-8.0)
    G = torch.cumsum(case.g.double(), dim=1) / np.log(2.0)
    assert float((G[:, :64].max(dim=1).values - G[:, :64].min(dim=1).values).max()) > 80
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL["bf16"])


def test_wide_keys_with_value_blocks_grouped_heads_gdn2_and_prologue():
    # K = 192, V = 512: two value blocks of 256
    case = width_case("bf16", "channel", 1, 90, 2, 192, 512, 109)
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL["bf16"])
    case = width_case("bf16", "channel", 1, 90, 4, 192, 160, 110)
    got, ref = run_both(case, G=2, gdn2=True, prologue=True)
    compare(case, got, ref, 2, TOL["bf16"])


def test_wide_keys_saved_equals_recomputed():
    import chunkwise_delta_rule_gb300 as kda
    case = width_case("bf16", "scalar", 1, 150, 2, 256, 256, 111)
    c = case.to("cuda")
    out = []
    for policy in (0, 1):
        p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate="scalar", scale=case.scale, initial_state=c.h0,
                             save_policy=policy)
        o, ht, sv = kda.kda_chunk_fwd(p)
        out.append((o, ht) + tuple(kda.kda_chunk_bwd(p, c.do, c.dht, saved=sv)))
    torch.cuda.synchronize()
    for a, b in zip(*out):
        if a is not None:
            assert torch.equal(a, b)


# bf16 widths that are multiples of 8 run on the tensor cores at their own widths (the tensor maps
# read the missing columns as zeros; the state, tail outputs, gradients and GatedDeltaNet-2 vectors
# are read and written at K and V); other bf16 widths are padded to 128
@pytest.mark.parametrize("gate,K,V", [("channel", 96, 48), ("scalar", 40, 120), ("channel", 36, 44)])
def test_native_and_padded_bf16_widths(gate, K, V):
    case = width_case("bf16", gate, 2, 150, 2, K, V, 112)
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL["bf16"])


def test_native_widths_gdn2_and_strong_decay():
    case = width_case("bf16", "channel", 1, 150, 2, 80, 112, 113)
    got, ref = run_both(case, gdn2=True)
    compare(case, got, ref, 1, TOL["bf16"])
    case = make_case(io="bf16", gate="channel", B=1, T=200, H=2, K=80, V=48, seed=114, g_shift=-4.0, g_min=-8.0)
    G = torch.cumsum(case.g.double(), dim=1) / np.log(2.0)
    assert float((G[:, :64].max(dim=1).values - G[:, :64].min(dim=1).values).max()) > 80
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL["bf16"])


def test_native_widths_backward_schedules_agree_bitwise():
    """Joint, time pieces and one pass hand the state adjoint over at [K][V] (80 x 112 here)."""
    import chunkwise_delta_rule_gb300 as kda
    case = width_case("bf16", "channel", 2, 640, 2, 80, 112, 115)
    c = case.to("cuda")
    outs = []
    for sched in (1, 3, 9):
        p = kda.make_problem(c.q, c.k, c.v, c.g, c.beta, gate="channel", scale=case.scale, initial_state=c.h0,
                             save_policy=1, schedule=sched)
        o, ht, sv = kda.kda_chunk_fwd(p)
        outs.append((o, ht) + tuple(kda.kda_chunk_bwd(p, c.do, c.dht, saved=sv)))
    torch.cuda.synchronize()
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            if a is not None:
                assert torch.equal(a, b)
    got = dict(o=outs[0][0], ht=outs[0][1], dq=outs[0][2], dk=outs[0][3], dv=outs[0][4], dg=outs[0][5],
               dbeta=outs[0][6], dh0=outs[0][7])
    p = packed(case)
    ref = run_oracle_prologue_arrays(p["q"], p["k"], p["v"], p["beta"], p["g"], A_log=None, dt_bias=None,
                                     lower_bound=0.0, eps=1e-6, scale=case.scale, gate=case.gate,
                                     seq_starts=case.seq_starts, h0=p["h0"], do=p["do"], dht=p["dht"],
                                     qk_norm=False, erase=None, write=None)
    compare(case, got, ref, 1, TOL["bf16"])


# Grouped heads and value blocks on the tensor-core path without the prologue read q, k (value
# head j: key head j / G, times the block count) and g, beta, erase (head j / NB for value
# blocks) in place; the cases meet every input the divisors touch: both gate kinds, the
# GatedDeltaNet-2 erase rows, widths below 128 and value blocks together with grouped heads.
@pytest.mark.parametrize("gate,K,V,G,gdn2", [("channel", 128, 256, 2, False), ("channel", 128, 256, 1, True),
                                              ("scalar", 128, 384, 2, False), ("channel", 80, 112, 2, True),
                                              ("none", 96, 160, 2, False)])
def test_grouped_inputs_read_in_place(gate, K, V, G, gdn2):
    case = width_case("bf16", gate, 2, 100, 4, K, V, 116)
    got, ref = run_both(case, G=G, gdn2=gdn2)
    compare(case, got, ref, G, TOL["bf16"])


def test_grouped_inputs_read_in_place_strong_decay():
    """Chunks whose gate range exceeds the tensor-core prep's limit go to the CUDA-core kernels,
    which read q, k, g and erase through the same head divisors."""
    case = make_case(io="bf16", gate="channel", B=1, T=200, H=4, K=128, V=256, seed=117, g_shift=-4.0, g_min=-8.0)
    G = torch.cumsum(case.g.double(), dim=1) / np.log(2.0)
    assert float((G[:, :64].max(dim=1).values - G[:, :64].min(dim=1).values).max()) > 80
    got, ref = run_both(case, G=2, gdn2=True)
    compare(case, got, ref, 2, TOL["bf16"])


def test_grouped_heads_in_place_equal_expanded_inputs():
    """Value head j reading key head j / 2 in place gives, bit for bit, what the caller gets by
    repeating q and k per value head (dq, dk as the sums over each pair, rounded once)."""
    import chunkwise_delta_rule_gb300 as kda
    case = width_case("bf16", "channel", 2, 150, 4, 128, 128, 118)
    c = case.to("cuda")
    qk = c.q[:, :, ::2].contiguous(), c.k[:, :, ::2].contiguous()
    runs = []
    for q, k in (qk, (qk[0].repeat_interleave(2, 2), qk[1].repeat_interleave(2, 2))):
        p = kda.make_problem(q, k, c.v, c.g, c.beta, gate="channel", scale=case.scale, initial_state=c.h0,
                             save_policy=1)
        o, ht, sv = kda.kda_chunk_fwd(p)
        runs.append((o, ht) + tuple(kda.kda_chunk_bwd(p, c.do, c.dht, saved=sv)))
    torch.cuda.synchronize()
    for name, a, b in zip(("o", "ht", "dq", "dk", "dv", "dg", "dbeta", "dh0"), *runs):
        if name in ("dq", "dk"):
            x = b.float().reshape(b.shape[0], b.shape[1], b.shape[2] // 2, 2, b.shape[3])
            b = (x[..., 0, :] + x[..., 1, :]).to(b.dtype)
        assert torch.equal(a, b), name


def test_value_blocks_share_the_prep_under_strong_decay():
    """The value blocks of a head prepared by one CTA (beta rule) when some chunks are too wide for the
    tensor-core prep: every block's unit is listed for the CUDA-core kernels."""
    case = make_case(io="bf16", gate="channel", B=1, T=200, H=2, K=128, V=384, seed=119, g_shift=-4.0, g_min=-8.0)
    G = torch.cumsum(case.g.double(), dim=1) / np.log(2.0)
    assert float((G[:, :64].max(dim=1).values - G[:, :64].min(dim=1).values).max()) > 80
    got, ref = run_both(case)
    compare(case, got, ref, 1, TOL["bf16"])
