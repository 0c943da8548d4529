"""The five benchmark workloads and a generic seeded case builder.

Input recipe (the same for every consumer of these tensors):

* draws come from one CPU ``torch.Generator`` seeded per case, in the fixed
  order: (sequence lengths for packed cases), q, k, v, beta-logits,
  gate-logits (gated cases only), h0 (when present), do, dht (when present);
* q and k are standard normal, L2-normalised per (token, head) in fp32 and
  then rounded to the I/O dtype; v and do are standard normal; beta is the
  sigmoid of a standard normal; all four are rounded to the I/O dtype;
* per-channel log-decay: g = max(logsigmoid(x + 3), -5), shape [B, T, H, K];
  scalar log-decay: g = logsigmoid(x + 4), shape [B, T, H]; both fp32;
* h0 ~ N(0, 0.1^2) and dht ~ N(0, 1) in fp32, shape [N, H, K, V];
* packed (varlen) cases: B = 1, lengths uniform in [64, 8192] drawn until the
  running sum reaches the total, the last one trimmed to fit.

Every value the GPU path sees is exactly the value the oracle sees (the oracle
upcasts the rounded tensors to float64).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

# The five workloads. ``kind`` names the operator family: "kda" has a
# per-channel log-decay, "gdn" a scalar per-head log-decay, "deltanet" none.
CONFIGS = {
    1: dict(name="kda_tiny_fp32", io="fp32", B=1, T=256, H=2, K=64, V=64,
            gate="channel", h0=True, dht=True, seed=0, lengths=None),
    2: dict(name="deltanet_bf16", io="bf16", B=4, T=4096, H=16, K=128, V=128,
            gate="none", h0=False, dht=False, seed=1, lengths=None),
    3: dict(name="gdn_bf16", io="bf16", B=8, T=4096, H=16, K=128, V=128,
            gate="scalar", h0=True, dht=True, seed=2, lengths=None),
    4: dict(name="kda_bf16", io="bf16", B=2, T=8192, H=32, K=128, V=128,
            gate="channel", h0=True, dht=True, seed=3, lengths=None),
    5: dict(name="kda_varlen_bf16", io="bf16", B=1, T=32768, H=32, K=128, V=128,
            gate="channel", h0=True, dht=True, seed=4, lengths="draw"),
}

_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


@dataclass
class Case:
    """One seeded problem instance (CPU tensors)."""

    io: str
    gate: str
    B: int
    T: int
    H: int
    K: int
    V: int
    scale: float
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    beta: torch.Tensor
    g: Optional[torch.Tensor]
    h0: Optional[torch.Tensor]
    do: torch.Tensor
    dht: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return self.B if self.cu_seqlens is None else int(self.cu_seqlens.numel() - 1)

    @property
    def seq_starts(self) -> list:
        """Token offsets of every sequence in the packed [B*T] token axis."""
        if self.cu_seqlens is None:
            return [b * self.T for b in range(self.B + 1)]
        return [int(x) for x in self.cu_seqlens.tolist()]

    def to(self, device) -> "Case":
        def mv(x):
            return None if x is None else x.to(device)
        return Case(self.io, self.gate, self.B, self.T, self.H, self.K, self.V, self.scale,
                    mv(self.q), mv(self.k), mv(self.v), mv(self.beta), mv(self.g), mv(self.h0),
                    mv(self.do), mv(self.dht), mv(self.cu_seqlens), self.name, dict(self.meta))


def varlen_lengths(gen: torch.Generator, total: int, lo: int = 64, hi: int = 8192) -> list:
    """Lengths uniform in [lo, hi] drawn until they cover ``total``; last one trimmed."""
    lens = []
    s = 0
    while s < total:
        x = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
        x = min(x, total - s)
        lens.append(x)
        s += x
    return lens


def _l2n(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make_case(*, io="bf16", gate="channel", B=1, T=256, H=2, K=64, V=64, seed=0,
              lengths=None, h0=True, dht=True, scale=None,
              g_shift=None, g_min=-5.0, beta_mode="sigmoid", name="",
              zero_g=False) -> Case:
    """Build a seeded case.

    ``lengths``: None for B equal sequences of length T; a list of lengths for
    a packed case (then B must be 1 and T is their sum); or "draw" to draw
    them from the case generator with the varlen recipe (T is the total).
    ``g_shift``/``g_min`` change the gate recipe (strong-decay tests).
    ``beta_mode``: "sigmoid" (recipe), "zero_every3" (every third beta is 0),
    "tiny" (all beta 1e-8), "one" (all beta 1).
    ``zero_g``: keep the gate tensor but make it all zeros (family checks).
    """
    gen = torch.Generator().manual_seed(int(seed))
    cu = None
    if lengths is not None:
        if B != 1:
            raise ValueError("packed cases have B == 1")
        if isinstance(lengths, str):
            lengths = varlen_lengths(gen, T)
        lengths = [int(x) for x in lengths]
        T = sum(lengths)
        cu = torch.tensor([0] + list(torch.tensor(lengths).cumsum(0).tolist()), dtype=torch.int32)
    N = B if cu is None else len(lengths)
    dt = _DT[io]
    q = _l2n(torch.randn(B, T, H, K, generator=gen)).to(dt)
    k = _l2n(torch.randn(B, T, H, K, generator=gen)).to(dt)
    v = torch.randn(B, T, H, V, generator=gen).to(dt)
    bl = torch.randn(B, T, H, generator=gen)
    if beta_mode == "sigmoid":
        beta = torch.sigmoid(bl)
    elif beta_mode == "zero_every3":
        beta = torch.sigmoid(bl)
        beta.view(-1)[::3] = 0.0
    elif beta_mode == "tiny":
        beta = torch.full_like(bl, 1e-8)
    elif beta_mode == "one":
        beta = torch.ones_like(bl)
    else:
        raise ValueError(beta_mode)
    beta = beta.to(dt)
    g = None
    if gate == "channel":
        x = torch.randn(B, T, H, K, generator=gen)
        shift = 3.0 if g_shift is None else g_shift
        g = torch.nn.functional.logsigmoid(x + shift).clamp_min(g_min)
    elif gate == "scalar":
        x = torch.randn(B, T, H, generator=gen)
        shift = 4.0 if g_shift is None else g_shift
        g = torch.nn.functional.logsigmoid(x + shift)
        if g_shift is not None:
            g = g.clamp_min(g_min)
    elif gate != "none":
        raise ValueError(gate)
    if g is not None:
        g = g.float().contiguous()
        if zero_g:
            g.zero_()
    h0t = (torch.randn(N, H, K, V, generator=gen) * 0.1).float() if h0 else None
    do = torch.randn(B, T, H, V, generator=gen).to(dt)
    dhtt = torch.randn(N, H, K, V, generator=gen).float() if dht else None
    sc = float(K) ** -0.5 if scale is None else float(scale)
    return Case(io, gate, B, T, H, K, V, sc, q.contiguous(), k.contiguous(), v.contiguous(),
                beta.contiguous(), g, h0t, do.contiguous(), dhtt, cu, name=name,
                meta=dict(seed=seed, lengths=lengths))


def make_config_case(idx: int) -> Case:
    """The full-size workload ``idx`` (1..5)."""
    c = CONFIGS[idx]
    return make_case(io=c["io"], gate=c["gate"], B=c["B"], T=c["T"], H=c["H"], K=c["K"],
                     V=c["V"], seed=c["seed"], lengths=c["lengths"], h0=c["h0"],
                     dht=c["dht"], name=c["name"])
