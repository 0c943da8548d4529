"""Host checks of the seeded workload generators (CPU only)."""

import torch

from workloads import CONFIGS, make_case, varlen_lengths


def test_small_case_shapes_and_determinism():
    a = make_case(io="bf16", gate="channel", B=2, T=70, H=3, K=16, V=8, seed=5)
    b = make_case(io="bf16", gate="channel", B=2, T=70, H=3, K=16, V=8, seed=5)
    for x in ("q", "k", "v", "beta", "g", "h0", "do", "dht"):
        assert torch.equal(getattr(a, x), getattr(b, x)), x
    assert a.q.dtype == torch.bfloat16 and a.g.dtype == torch.float32
    assert a.q.shape == (2, 70, 3, 16) and a.v.shape == (2, 70, 3, 8)
    assert a.g.shape == (2, 70, 3, 16) and a.h0.shape == (2, 3, 16, 8)
    assert float(a.g.min()) >= -5.0 and float(a.g.max()) < 0.0
    n = a.k.float().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-2)


def test_varlen_lengths_recipe():
    gen = torch.Generator().manual_seed(4)
    lens = varlen_lengths(gen, 32768)
    assert sum(lens) == 32768
    assert all(64 <= x <= 8192 for x in lens[:-1]) and 1 <= lens[-1] <= 8192
    c = make_case(io="bf16", gate="channel", B=1, T=32768, H=1, K=8, V=8, seed=4, lengths="draw")
    assert c.cu_seqlens[0] == 0 and int(c.cu_seqlens[-1]) == 32768
    assert [int(x) for x in (c.cu_seqlens[1:] - c.cu_seqlens[:-1])] == lens


def test_config_table():
    assert CONFIGS[1]["io"] == "fp32" and CONFIGS[1]["K"] == 64
    assert CONFIGS[2]["gate"] == "none" and not CONFIGS[2]["h0"] and not CONFIGS[2]["dht"]
    assert CONFIGS[3]["gate"] == "scalar"
    assert CONFIGS[4]["B"] * CONFIGS[4]["T"] == 16384 and CONFIGS[4]["H"] == 32
    assert CONFIGS[5]["lengths"] == "draw" and CONFIGS[5]["T"] == 32768
