"""PyTorch-facing binding of the C ABI (same names as include/kda.h).

PyTorch provides device memory and the current stream; every step of the
operator runs in libkda.so's CUDA kernels. Tensors use the layouts of the C
ABI: q, k [B, T, H, K]; v [B, T, H, V]; beta [B, T, H]; g [B, T, H, K]
(per-channel) or [B, T, H] (scalar) in fp32; states [N, H, K, V] in fp32.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib

_IO = {torch.bfloat16: "bf16", torch.float32: "fp32"}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class Problem:
    """A validated problem description plus the tensors it points to."""

    c: _lib.KdaProblem
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    beta: torch.Tensor
    g: Optional[torch.Tensor]
    h0: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    N: int
    A_log: Optional[torch.Tensor] = None
    dt_bias: Optional[torch.Tensor] = None
    erase: Optional[torch.Tensor] = None
    write: Optional[torch.Tensor] = None

    @property
    def state_shape(self):
        return (self.N, self.c.HV or self.c.H, self.c.K, self.c.V)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def make_problem(q, k, v, g, beta, *, gate: str, scale: Optional[float] = None,
                 initial_state: Optional[torch.Tensor] = None,
                 cu_seqlens: Optional[torch.Tensor] = None, save_policy: int = 0,
                 A_log: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
                 lower_bound: float = 0.0, qk_l2norm: bool = False, l2norm_eps: float = 1e-6,
                 erase: Optional[torch.Tensor] = None, write: Optional[torch.Tensor] = None,
                 schedule: int = 0) -> Problem:
    """Describe one call. With ``A_log`` (fp32 [H]) ``g`` is the raw gate and the
    decay is activated inside the operator (softplus form, or the lower-bound
    form when ``lower_bound`` < 0), with the optional ``dt_bias`` (fp32, [H, K]
    for a per-channel gate, [H] for a scalar one); ``qk_l2norm`` normalises q
    and k per (token, head) first. GatedDeltaNet-2: ``erase`` [B, T, H, K] and
    ``write`` [B, T, H, V] (the I/O dtype) replace ``beta``, which may be None.
    ``schedule``: 0 the library's choice, 1 one reverse-scan pass before the
    consumer, P >= 2 that many time pieces (equal-length batches; see kda.h).
    Grouped value heads: v may carry HV = G * H heads (q, k keep H); then every
    per-head tensor but q and k has HV heads (read H as HV above)."""
    _need(q.dim() == 4 and k.shape == q.shape, "q and k must be [B, T, H, K]")
    B, T, Hk, K = q.shape
    _need(v.dim() == 4 and v.shape[:2] == q.shape[:2], "v must be [B, T, HV, V]")
    H = v.shape[2]   # value heads: the head count of every other tensor
    _need(H % Hk == 0, "the value heads must be a multiple of the key heads")
    V = v.shape[3]
    _need((erase is None) == (write is None), "erase and write come together")
    if erase is not None:
        _need(erase.dtype == q.dtype and tuple(erase.shape) == (B, T, H, K), "erase must be [B, T, H, K], q's dtype")
        _need(write.dtype == q.dtype and tuple(write.shape) == (B, T, H, V), "write must be [B, T, H, V], q's dtype")
    else:
        _need(beta is not None, "beta is required without erase/write")
    _need(q.dtype in _IO and k.dtype == q.dtype and v.dtype == q.dtype and (beta is None or beta.dtype == q.dtype),
          "q, k, v, beta must share one dtype (bf16 or fp32)")
    _need(beta is None or tuple(beta.shape) == (B, T, H), "beta must be [B, T, H]")
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("erase", erase), ("write", write)):
        if t is None:
            continue
        _need(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    if gate == "none":
        _need(g is None, "g must be None without a gate")
    else:
        _need(g is not None and g.dtype == torch.float32 and g.is_cuda and g.is_contiguous(),
              "g must be a contiguous fp32 CUDA tensor")
        want = (B, T, H, K) if gate == "channel" else (B, T, H)
        _need(tuple(g.shape) == want, f"g must be {list(want)}")
    N = B
    if cu_seqlens is not None:
        _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda and cu_seqlens.dim() == 1,
              "cu_seqlens must be an int32 CUDA vector")
        N = cu_seqlens.numel() - 1
    if initial_state is not None:
        _need(initial_state.dtype == torch.float32 and initial_state.is_contiguous()
              and tuple(initial_state.shape) == (N, H, K, V), "initial_state must be fp32 [N, H, K, V]")
    c = _lib.KdaProblem()
    c.B, c.T, c.H, c.K, c.V = B, T, Hk, K, V
    c.HV = H if H != Hk else 0
    c.N = N if cu_seqlens is not None else 0
    c.cu_seqlens = None if cu_seqlens is None else cu_seqlens.data_ptr()
    c.io = _lib.DTYPES[_IO[q.dtype]]
    c.gate = _lib.GATES[gate]
    c.scale = float(scale) if scale is not None else 0.0
    c.q, c.k, c.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    c.beta = None if beta is None else beta.data_ptr()
    c.erase = None if erase is None else erase.data_ptr()
    c.write = None if write is None else write.data_ptr()
    c.g = None if g is None else g.data_ptr()
    c.h0 = None if initial_state is None else initial_state.data_ptr()
    c.save_policy = int(save_policy)
    c.schedule = int(schedule)
    if A_log is not None:
        _need(gate != "none", "A_log needs a gate")
        _need(A_log.dtype == torch.float32 and A_log.is_cuda and A_log.is_contiguous()
              and tuple(A_log.shape) == (H,), "A_log must be a contiguous fp32 CUDA tensor [H]")
    if dt_bias is not None:
        _need(A_log is not None, "dt_bias needs A_log")
        want = (H, K) if gate == "channel" else (H,)
        _need(dt_bias.dtype == torch.float32 and dt_bias.is_cuda and dt_bias.is_contiguous()
              and tuple(dt_bias.shape) == want, f"dt_bias must be a contiguous fp32 CUDA tensor {list(want)}")
    c.A_log = None if A_log is None else A_log.data_ptr()
    c.dt_bias = None if dt_bias is None else dt_bias.data_ptr()
    c.lower_bound = float(lower_bound)
    c.qk_l2norm = 1 if qk_l2norm else 0
    c.l2norm_eps = float(l2norm_eps)
    return Problem(c, q, k, v, beta, g, initial_state, cu_seqlens, N, A_log, dt_bias, erase, write)


def kda_workspace_size(p: Problem, for_backward: bool) -> int:
    return int(_lib.load().kda_workspace_size(ctypes.byref(p.c), 1 if for_backward else 0))


def kda_saved_size(p: Problem) -> int:
    return int(_lib.load().kda_saved_size(ctypes.byref(p.c)))


def kda_last_error() -> str:
    return _lib.last_error()


def _buffer(nbytes: int, device, given: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return given
    if given is not None and given.numel() * given.element_size() >= nbytes:
        return given
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def kda_device_status(p: Problem, workspace: torch.Tensor, stream=None):
    """Synchronise and read the device error word a call left in `workspace`.
    Returns (status, word); status 0 = OK."""
    word = ctypes.c_int32(0)
    nbytes = workspace.numel() * workspace.element_size()
    st = _lib.load().kda_device_status(ctypes.byref(p.c), _ptr(workspace), nbytes, _stream(stream),
                                       ctypes.byref(word))
    return int(st), int(word.value)


def kda_chunk_fwd(p: Problem, *, output_final_state: bool = True, workspace=None, saved=None,
                  stream=None):
    """Forward pass. Returns (o, ht or None, saved or None)."""
    lib = _lib.load()
    dev = p.q.device
    o = torch.empty_like(p.v)
    ht = torch.empty(p.state_shape, dtype=torch.float32, device=dev) if output_final_state else None
    ws = _buffer(kda_workspace_size(p, False), dev, workspace)
    sv = None
    if p.c.save_policy:
        sv = _buffer(kda_saved_size(p), dev, saved)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = lib.kda_chunk_fwd(ctypes.byref(p.c), _ptr(o), _ptr(ht), _ptr(sv), _ptr(ws), nbytes,
                           _stream(stream))
    _lib.check(st, "kda_chunk_fwd")
    return o, ht, sv


def kda_recurrent_fwd(p: Problem, *, output_final_state: bool = True, ht: Optional[torch.Tensor] = None,
                      err: Optional[torch.Tensor] = None, stream=None):
    """Token-by-token forward (decoding, short prompts). Returns (o, ht or None).
    ``ht`` may be given (fp32 [N, H, K, V], for example the initial state itself
    for an in-place update); ``err`` is an optional int32 device word."""
    _need(p.c.save_policy == 0, "the recurrent forward has no saved buffer: use save_policy 0")
    dev = p.q.device
    o = torch.empty_like(p.v)
    if ht is None and output_final_state:
        ht = torch.empty(p.state_shape, dtype=torch.float32, device=dev)
    if ht is not None:
        _need(ht.dtype == torch.float32 and ht.is_contiguous() and tuple(ht.shape) == p.state_shape,
              "ht must be fp32 [N, H, K, V]")
    if err is not None:
        _need(err.dtype == torch.int32 and err.is_cuda and err.numel() >= 1, "err must be an int32 CUDA tensor")
    st = _lib.load().kda_recurrent_fwd(ctypes.byref(p.c), _ptr(o), _ptr(ht), _ptr(err), _stream(stream))
    _lib.check(st, "kda_recurrent_fwd")
    return o, ht


def kda_chunk_bwd(p: Problem, do: torch.Tensor, dht: Optional[torch.Tensor] = None, *,
                  saved=None, workspace=None, stream=None, need_dh0: bool = True):
    """Backward pass of <do, o> + <dht, ht>. Returns dq, dk, dv, dg, dbeta, dh0,
    then, when the problem activates its gate (A_log given), dA_log and
    ddt_bias (None without dt_bias), then, with erase/write (GatedDeltaNet-2;
    dbeta is None), derase and dwrite."""
    lib = _lib.load()
    dev = p.q.device
    _need(do.shape == p.v.shape and do.dtype == p.v.dtype and do.is_contiguous(), "do must match v")
    if dht is not None:
        _need(dht.dtype == torch.float32 and dht.is_contiguous() and tuple(dht.shape) == p.state_shape,
              "dht must be fp32 [N, H, K, V]")
    dq = torch.empty_like(p.q)
    dk = torch.empty_like(p.k)
    dv = torch.empty_like(p.v)
    dbeta = None if p.erase is not None else torch.empty_like(p.beta)
    der = None if p.erase is None else torch.empty_like(p.erase)
    dwr = None if p.write is None else torch.empty_like(p.write)
    dg = None if p.g is None else torch.empty_like(p.g)
    dh0 = torch.empty(p.state_shape, dtype=torch.float32, device=dev) if need_dh0 else None
    dA = None if p.A_log is None else torch.empty_like(p.A_log)
    ddt = None if p.dt_bias is None else torch.empty_like(p.dt_bias)
    ws = _buffer(kda_workspace_size(p, True), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = lib.kda_chunk_bwd(ctypes.byref(p.c), _ptr(do), _ptr(dht), _ptr(saved), _ptr(dq), _ptr(dk),
                           _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(der), _ptr(dwr), _ptr(dh0), _ptr(dA), _ptr(ddt),
                           _ptr(ws), nbytes,
                           _stream(stream))
    _lib.check(st, "kda_chunk_bwd")
    out = (dq, dk, dv, dg, dbeta, dh0)
    if p.A_log is not None:
        out += (dA, ddt)
    if p.erase is not None:
        out += (der, dwr)
    return out


class ChunkKDAFunction(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run the CUDA library."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, A_log, dt_bias, gate, scale, cu_seqlens, save_policy,
                lower_bound, qk_l2norm, l2norm_eps):
        kw = dict(gate=gate, scale=scale, save_policy=save_policy, lower_bound=lower_bound,
                  qk_l2norm=qk_l2norm, l2norm_eps=l2norm_eps)
        p = make_problem(q, k, v, g, beta, initial_state=initial_state, cu_seqlens=cu_seqlens,
                         A_log=A_log, dt_bias=dt_bias, **kw)
        o, ht, sv = kda_chunk_fwd(p)
        e = torch.empty(0)
        ctx.save_for_backward(q, k, v, g if g is not None else e, beta,
                              initial_state if initial_state is not None else e,
                              cu_seqlens if cu_seqlens is not None else e, sv if sv is not None else e,
                              A_log if A_log is not None else e, dt_bias if dt_bias is not None else e)
        ctx.meta = (kw, g is not None, initial_state is not None, cu_seqlens is not None, A_log is not None,
                    dt_bias is not None)
        return o, ht

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g, beta, h0, cu, sv, A_log, dt_bias = ctx.saved_tensors
        kw, has_g, has_h0, has_cu, has_A, has_dt = ctx.meta
        p = make_problem(q, k, v, g if has_g else None, beta, initial_state=h0 if has_h0 else None,
                         cu_seqlens=cu if has_cu else None, A_log=A_log if has_A else None,
                         dt_bias=dt_bias if has_dt else None, **kw)
        do = do.contiguous()
        dht = None if dht is None else dht.contiguous()
        r = kda_chunk_bwd(p, do, dht, saved=sv if kw["save_policy"] else None, need_dh0=has_h0)
        dq, dk, dv, dg, dbeta, dh0 = r[:6]
        dA, ddt = (r[6], r[7]) if has_A else (None, None)
        return dq, dk, dv, dg, dbeta, dh0, dA, ddt, None, None, None, None, None, None, None


def chunk_kda(q, k, v, g, beta, *, gate: str = "channel", scale: Optional[float] = None,
              initial_state: Optional[torch.Tensor] = None,
              cu_seqlens: Optional[torch.Tensor] = None, save_policy: int = 0,
              A_log: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
              lower_bound: float = 0.0, use_qk_l2norm_in_kernel: bool = False, l2norm_eps: float = 1e-6):
    """Differentiable chunkwise gated delta rule. Returns (o, final_state).
    With ``A_log`` the gate ``g`` is raw and activated inside the operator;
    ``use_qk_l2norm_in_kernel`` normalises q and k per (token, head)."""
    return ChunkKDAFunction.apply(q, k, v, g, beta, initial_state, A_log, dt_bias, gate, scale, cu_seqlens,
                                  save_policy, lower_bound, use_qk_l2norm_in_kernel, l2norm_eps)
