"""Host-side checks of the C ABI (no GPU needed: no call here reaches CUDA)."""

import ctypes
import os
import re

import pytest

from chunkwise_delta_rule_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "kda.h")


def declared_functions():
    text = open(HDR).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    names = declared_functions()
    assert "kda_chunk_fwd" in names and "kda_chunk_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    assert lib.kda_abi_version() == 4


def _prob(**kw):
    p = _lib.KdaProblem()
    p.B, p.T, p.H, p.K, p.V = kw.get("B", 2), kw.get("T", 130), kw.get("H", 3), kw.get("K", 128), kw.get("V", 128)
    p.N = kw.get("N", 0)
    p.cu_seqlens = kw.get("cu", None)
    p.io = kw.get("io", 0)
    p.gate = kw.get("gate", 2)
    p.scale = 0.0
    fake = 0x1000
    p.q = p.k = p.v = p.beta = fake
    p.g = fake if p.gate != 0 else None
    p.h0 = None
    p.save_policy = kw.get("save", 0)
    p.schedule = kw.get("schedule", 0)
    return p


def _ws(p, bwd):
    return _lib.load().kda_workspace_size(ctypes.byref(p), bwd)


def test_workspace_size_arithmetic():
    # B=2, T=130 -> 3 chunks per sequence, 6 chunk slots, H=3, D=128; fp32 I/O
    # runs the CUDA-core kernels, bf16 I/O at D = 128 the tensor-core forward
    p = _prob(io=1)
    NC, H, D, BT = 6, 3, 128, 64

    def up(x):
        return (x + 255) // 256 * 256

    table = up(4 * NC) * 2 + up(4 * 3) + up(4 * 2) * 3 + up(4)
    chd = NC * H
    fcore = up(4 * chd * BT * D) * 4 + up(4 * chd * BT * BT) * 2 + up(4 * chd * D)
    fextra = up(4 * chd * BT * D) + up(4 * chd * D * D)
    bwd = up(4 * chd * BT * D) * 4 + up(4 * chd * D * D) + up(4 * chd * BT * BT) * 2 + up(4 * chd * D) + up(4 * chd * BT)
    assert _ws(p, 0) == table + fcore
    assert _ws(p, 1) == table + fcore + fextra + bwd
    ptc = _prob(io=0)
    # bf16 W, F, Q_g, U tiles, C_q; fp32 gate at the chunk end; wide flags and list
    ftc = up(2 * chd * BT * D) * 4 + up(2 * chd * BT * BT) + up(4 * chd * D) + up(4 * chd) + up(4 * (chd + 1))
    assert _ws(ptc, 0) == table + ftc
    # saved for the backward: A, S, R and, with a per-channel gate, alpha and two rows of 128 per unit
    ftc_b = up(2 * chd * BT * BT) + up(2 * chd * D * D) + up(2 * chd * BT * D) + up(4 * chd * (BT * D + 2 * D))
    btc = up(2 * chd * D * D) + up(2 * chd * BT * D)
    wscr = up(4 * chd * BT * D) * 3 + up(4 * chd * BT * BT) * 2 + up(4 * chd * D) + up(4 * chd * BT)
    # equal-length batches: two fp32 state adjoints and eight claim counters for a backward in time
    # pieces, and a ready flag per chunk x head for the joint schedule
    piece = 2 * up(4 * 2 * H * D * D) + up(4 * 8) + up(4 * chd)
    assert _ws(ptc, 1) == table + ftc + ftc_b + btc + wscr + piece
    ptca = _prob(io=0, save=1)
    assert _ws(ptca, 0) == table
    assert _ws(ptca, 1) == table + btc + wscr + piece
    assert _lib.load().kda_saved_size(ctypes.byref(ptca)) == ftc + ftc_b
    # a scalar gate saves one alpha per token and its two constants (80 floats per unit), no gate none
    alk = up(4 * chd * (BT * D + 2 * D))
    assert _lib.load().kda_saved_size(ctypes.byref(_prob(io=0, save=1, gate=1))) == ftc + ftc_b - alk + up(4 * chd * 80)
    assert _lib.load().kda_saved_size(ctypes.byref(_prob(io=0, save=1, gate=0))) == ftc + ftc_b - alk
    pa = _prob(save=1, io=1)
    assert _ws(pa, 0) == table
    assert _ws(pa, 1) == table + bwd
    assert _lib.load().kda_saved_size(ctypes.byref(pa)) == fcore + fextra
    assert _lib.load().kda_saved_size(ctypes.byref(p)) == 0
    # packed: chunk slots = ceil(T/64) + N
    pv = _prob(B=1, T=300, N=4, cu=0x2000, io=1)
    NCv = 5 + 4
    tablev = up(4 * NCv) * 2 + up(4 * 5) + up(4 * 4) * 3 + up(4)
    chv = NCv * 3
    assert _ws(pv, 0) == tablev + up(4 * chv * BT * D) * 4 + up(4 * chv * BT * BT) * 2 + up(4 * chv * D)


@pytest.mark.parametrize("kw,status", [
    (dict(K=257, V=192), 2),
    (dict(K=320, V=128), 2),
    (dict(B=0), 1),
    (dict(gate=7), 1),
    (dict(io=5), 1),
    (dict(B=2, cu=0x2000, N=3), 1),
    (dict(save=3), 1),
    (dict(schedule=10), 1),
    (dict(schedule=-1), 1),
])
def test_invalid_problems_are_rejected_before_launch(kw, status):
    lib = _lib.load()
    p = _prob(**kw)
    st = lib.kda_chunk_fwd(ctypes.byref(p), ctypes.c_void_p(0x3000), None, None, None, 0, None)
    assert st == status, _lib.last_error()
    assert _lib.last_error()
    assert _ws(p, 0) == 0


def test_missing_pointers_and_workspace():
    lib = _lib.load()
    p = _prob()
    p.q = None
    assert lib.kda_chunk_fwd(ctypes.byref(p), ctypes.c_void_p(0x3000), None, None, None, 0, None) == 1
    p = _prob(gate=0)
    p.g = 0x1000
    assert lib.kda_chunk_fwd(ctypes.byref(p), ctypes.c_void_p(0x3000), None, None, None, 0, None) == 1
    p = _prob()
    # workspace missing, misaligned, too small
    assert lib.kda_chunk_fwd(ctypes.byref(p), ctypes.c_void_p(0x3000), None, None, None, 0, None) == 3
    assert lib.kda_chunk_fwd(ctypes.byref(p), ctypes.c_void_p(0x3000), None, None,
                             ctypes.c_void_p(0x10010), 1 << 40, None) == 3
    assert lib.kda_chunk_fwd(ctypes.byref(p), ctypes.c_void_p(0x3000), None, None,
                             ctypes.c_void_p(0x10000), 100, None) == 3
    # backward: dg required with a gate
    z = ctypes.c_void_p(0x3000)
    st = lib.kda_chunk_bwd(ctypes.byref(p), z, None, None, z, z, z, None, z, None, None, None, None, None, None, 0, None)
    assert st == 1 and "dg" in _lib.last_error()


def test_recurrent_forward_validates_before_launch():
    lib = _lib.load()
    z = ctypes.c_void_p(0x3000)
    p = _prob(save=1)
    assert lib.kda_recurrent_fwd(ctypes.byref(p), z, None, None, None) == 1
    assert "saved" in _lib.last_error()
    p = _prob()
    assert lib.kda_recurrent_fwd(ctypes.byref(p), None, None, None, None) == 1   # tokens but no o
    p = _prob(K=96, V=96)
    assert lib.kda_recurrent_fwd(ctypes.byref(p), z, None, None, None) == 2
    p = _prob()
    p.beta = None
    assert lib.kda_recurrent_fwd(ctypes.byref(p), z, None, None, None) == 1


def test_prologue_fields_are_validated_and_sized():
    lib = _lib.load()
    z = ctypes.c_void_p(0x3000)
    base = _prob()
    core_f, core_b = _ws(base, 0), _ws(base, 1)
    # A_log without a gate, dt_bias without A_log, lower_bound out of range, qk_l2norm not 0/1
    for kw, fld in ((dict(gate=0), ("A_log", 0x5000)), (dict(), ("dt_bias", 0x5000)), (dict(), ("qk_l2norm", 2))):
        p = _prob(**kw)
        setattr(p, *fld)
        assert lib.kda_chunk_fwd(ctypes.byref(p), z, None, None, None, 0, None) == 1
        assert _ws(p, 0) == 0
    p = _prob()
    p.A_log = 0x5000
    p.lower_bound = -6.0
    assert lib.kda_chunk_fwd(ctypes.byref(p), z, None, None, None, 0, None) == 1
    def up(x):
        return (x + 255) // 256 * 256

    # workspace: the pipeline's, then normalised q, k (io dtype), the activated gate and,
    # in the backward, per-64-token-block partial sums
    p = _prob()   # bf16, channel gate, B=2, T=130, H=3, K=128
    p.A_log, p.dt_bias, p.qk_l2norm = 0x5000, 0x6000, 1
    tok = 2 * 130 * 3 * 128
    nb = (2 * 130 + 63) // 64
    extra_f = 2 * up(2 * tok) + up(4 * tok)
    assert _ws(p, 0) == core_f + extra_f
    assert _ws(p, 1) == core_b + extra_f + up(4 * nb * 3 * 128) + up(4 * nb * 3)


def test_grouped_value_heads_are_validated_and_sized():
    lib = _lib.load()
    p = _prob(H=3)
    p.HV = 4   # not a multiple of H
    assert lib.kda_chunk_fwd(ctypes.byref(p), ctypes.c_void_p(0x3000), None, None, None, 0, None) == 1
    assert _ws(p, 0) == 0

    def up(x):
        return (x + 255) // 256 * 256

    g = _prob(H=2)
    g.HV = 6
    flat = _prob(H=6)   # the same problem with one key head per value head
    copy = up(2 * 2 * 130 * 6 * 128)   # bf16 q (or k, dq, dk) per value head
    # tensor-core path: q, k read in place by key head; the backward's dq, dk per value head
    assert _ws(g, 0) == _ws(flat, 0)
    assert _ws(g, 1) == _ws(flat, 1) + 2 * copy
    # with the prologue (q, k normalised first) or fp32 I/O, q and k are copied per value head
    for kw, es in ((dict(), 2), (dict(io=1), 4)):
        gp, fp = _prob(H=2, **kw), _prob(H=6, **kw)
        gp.HV = 6
        if not kw:
            gp.qk_l2norm = fp.qk_l2norm = 1
        one = up(es * 2 * 130 * 6 * 128)
        assert _ws(gp, 0) == _ws(fp, 0) + 2 * one
        assert _ws(gp, 1) == _ws(fp, 1) + 4 * one


def test_unequal_widths_pad_to_the_working_width():
    def up(x):
        return (x + 255) // 256 * 256

    lib = _lib.load()
    # bf16 widths that are multiples of 8 run on the tensor cores as they are: the 128-wide path's
    # workspace and no padded copies
    assert _ws(_prob(K=80, V=112), 0) == _ws(_prob(K=128, V=128), 0)
    # backward: the two state-adjoint hand-over buffers of the time pieces hold [K][V] states
    assert _ws(_prob(K=80, V=112), 1) == _ws(_prob(K=128, V=128), 1) - 2 * (up(4 * 2 * 3 * 128 * 128) - up(4 * 2 * 3 * 80 * 112))
    p = _prob(K=84, V=116)              # bf16, channel gate, B=2, T=130, H=3: padded to 128
    work = _prob(K=128, V=128)
    T, H, D = 2 * 130, 3, 128
    # q, k, v, g (fp32), o, ht (fp32) at the working width
    pad_f = 3 * up(2 * T * H * D) + up(4 * T * H * D) + up(2 * T * H * D) + up(4 * 2 * H * D * D)
    assert _ws(p, 0) == _ws(work, 0) + pad_f
    # backward adds dout, dht, dq, dk, dv, dg, dh0
    pad_b = pad_f + up(2 * T * H * D) + up(4 * 2 * H * D * D) + 3 * up(2 * T * H * D) + up(4 * T * H * D) \
        + up(4 * 2 * H * D * D)
    assert _ws(p, 1) == _ws(work, 1) + pad_b
    # bf16 widths up to 128 all run at 128 (the tensor-core width; 32/48 and 64/64 unpadded, 36/44
    # padded), fp32 ones within 64 at 64
    assert _ws(_prob(K=32, V=48), 0) == _ws(work, 0)
    assert _ws(_prob(K=64, V=64), 0) == _ws(work, 0)
    assert _ws(_prob(K=36, V=44), 0) == _ws(p, 0)
    D = 64
    pad64 = 3 * up(4 * T * H * D) + up(4 * T * H * D) + up(4 * T * H * D) + up(4 * 2 * H * D * D)
    assert _ws(_prob(K=32, V=48, io=1), 0) == _ws(_prob(K=64, V=64, io=1), 0) + pad64
    D = 128
    z = ctypes.c_void_p(0x3000)
    assert lib.kda_recurrent_fwd(ctypes.byref(p), z, None, None, None) == 2
    # key widths above 128 run at 256 (the value side too)
    wide = _prob(K=192, V=160)
    work = _prob(K=256, V=256)
    D = 256
    pad_f = 3 * up(2 * T * H * D) + up(4 * T * H * D) + up(2 * T * H * D) + up(4 * 2 * H * D * D)
    assert _ws(wide, 0) == _ws(work, 0) + pad_f
    pad_b = pad_f + up(2 * T * H * D) + up(4 * 2 * H * D * D) + 3 * up(2 * T * H * D) + up(4 * T * H * D) \
        + up(4 * 2 * H * D * D)
    assert _ws(wide, 1) == _ws(work, 1) + pad_b
    # K = V = 256 is a working width itself: its workspace is the chunk pipeline's (fp32 intermediates)
    NC, chd = 2 * 3, 2 * 3 * 3
    table = 2 * up(4 * NC) + up(4 * 3) + 3 * up(4 * 2) + up(4)
    fcore = 4 * up(4 * chd * 64 * D) + 2 * up(4 * chd * 64 * 64) + up(4 * chd * D)
    assert _ws(work, 0) == table + fcore


def test_wide_values_run_as_value_blocks():
    def up(x):
        return (x + 255) // 256 * 256

    lib = _lib.load()
    z = ctypes.c_void_p(0x3000)
    # K = 128, V = 256: two value blocks of 128, each a value head of its own (HV = 2 H)
    p = _prob(V=256)                    # bf16, channel gate, B=2, T=130, H=3, no h0
    inner = _prob(V=128)
    inner.HV = 6
    T, Hv, K, NB = 2 * 130, 3, 128, 2
    # tensor-core blocks at their own width read beta and g in place (block value head j reads
    # head j / NB): the blocks' final states only
    split_f = up(4 * 2 * Hv * K * 256)
    assert _ws(p, 0) == _ws(inner, 0) + split_f
    # backward adds the blocks' dbeta, dg, dht and dh0
    split_b = split_f + up(2 * T * Hv * NB) + up(4 * T * Hv * NB * K) + 2 * up(4 * 2 * Hv * K * 256)
    assert _ws(p, 1) == _ws(inner, 1) + split_b
    # with the prologue, beta and g repeat per block
    pp, ip = _prob(V=256), _set(_prob(V=128), HV=6)
    pp.qk_l2norm = ip.qk_l2norm = 1
    split_f = up(2 * T * Hv * NB) + up(4 * T * Hv * NB * K) + up(4 * 2 * Hv * K * 256)
    assert _ws(pp, 0) == _ws(ip, 0) + split_f
    assert lib.kda_saved_size(ctypes.byref(_prob(V=256, save=1))) == \
        lib.kda_saved_size(ctypes.byref(_set(_prob(V=128, save=1), HV=6)))
    # V = 201: two blocks of 101, value rows padded to 202 (v and o in the forward)
    odd = _prob(V=201, gate=1)
    inner = _set(_prob(V=101, gate=1), HV=6)
    rows = up(2 * T * Hv * 202)
    split_f = 2 * rows + up(2 * T * Hv * NB) + up(4 * T * Hv * NB) + up(4 * 2 * Hv * K * 202)
    assert _ws(odd, 0) == _ws(inner, 0) + split_f
    # above K = 128 the value blocks are 256 wide: K = 192, V = 512 is two blocks of 256
    kb = _prob(K=192, V=512)
    inner = _set(_prob(K=192, V=256), HV=6)
    split_f = up(2 * T * Hv * NB) + up(4 * T * Hv * NB * 192) + up(4 * 2 * Hv * 192 * 512)
    assert _ws(kb, 0) == _ws(inner, 0) + split_f
    # limits: key width above 256; value width above 4096; value heads x blocks above 65535
    for kw, fld in ((dict(K=257), None), (dict(V=4097), None), (dict(H=30000, V=384), None)):
        q = _prob(**kw)
        assert lib.kda_chunk_fwd(ctypes.byref(q), z, None, None, None, 0, None) == 2
        assert _ws(q, 0) == 0
    # the token-by-token forward takes K = 64 or 128 and V a multiple of 32 (its CTAs own 32 columns)
    assert lib.kda_recurrent_fwd(ctypes.byref(_prob(V=200)), z, None, None, None) == 2
    assert lib.kda_recurrent_fwd(ctypes.byref(_prob(K=96, V=256)), z, None, None, None) == 2
    # the backward's argument checks come before any launch
    p = _prob(V=256)
    assert lib.kda_chunk_bwd(ctypes.byref(p), z, None, None, z, z, z, z, None, None, None, None, None, None,
                             z, 1 << 40, None) == 1
    assert "dbeta" in _lib.last_error()


def _set(p, **kw):
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_in_place_grouped_reads_follow_the_tensor_core_path():
    """Grouped heads and value blocks read q, k (and g, beta) in place exactly when the problem runs on
    the tensor-core path at its own widths without the prologue; the workspace shows which."""
    def up(x):
        return (x + 255) // 256 * 256

    T = 2 * 130
    # bf16 80/112 with two value heads per key head: in place (no q, k copies in the forward)
    g, flat = _set(_prob(H=2, K=80, V=112), HV=4), _prob(H=4, K=80, V=112)
    assert _ws(g, 0) == _ws(flat, 0)
    # fp32 I/O at 64: the CUDA-core path, q and k copied per value head
    g, flat = _set(_prob(H=2, K=64, V=64, io=1), HV=4), _prob(H=4, K=64, V=64, io=1)
    assert _ws(g, 0) == _ws(flat, 0) + 2 * up(4 * T * 4 * 64)
    # bf16 96/160: two 80-wide value blocks, native widths, in place (the blocks' final states only)
    p, inner = _prob(K=96, V=160), _set(_prob(K=96, V=80), HV=6)
    assert _ws(p, 0) == _ws(inner, 0) + up(4 * 2 * 3 * 96 * 160)
    # bf16 128/200: two blocks of 100, padded to 128 inside, so beta and g repeat per block and the
    # value rows are padded to 200 (no copy: NB * Vb = V)
    p, inner = _prob(V=200), _set(_prob(V=100), HV=6)
    assert _ws(p, 0) == _ws(inner, 0) + up(2 * T * 3 * 2) + up(4 * T * 3 * 2 * 128) + up(4 * 2 * 3 * 128 * 200)
