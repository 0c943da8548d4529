// C ABI of libkda.so: argument validation, workspace layout, launch order.
// Declarations and the contract of every entry point are in include/kda.h.
#include <cstring>
#include <string>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace {

thread_local std::string g_err;

kda_status fail(kda_status st, const std::string& msg) {
    g_err = msg;
    return st;
}

constexpr size_t ALIGN = 256;
size_t up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

struct Dims {
    int N = 0, NC = 0, Ttot = 0, H = 0;
    int D = 0, V = 0;   // key and value widths of the problem
    int WD = 0;         // working width of the chunk intermediates (the tile width of the path)
    int alk = 0;        // floats per chunk x head of the alpha the tensor-core prep saves for the backward
    int per = 0;        // chunks per sequence of an equal-length batch (0: packed sequences)
};

// Value widths above the block width (128; 256 when K > 128) run as value blocks.
int vblock_max(const kda_problem* p) { return p->K > 128 ? 256 : 128; }

// Checks the size fields; fills d. Returns KDA_OK or an error (message set). Key widths up to
// 256 (the token-by-token call checks its own list on top).
kda_status check_dims(const kda_problem* p, Dims& d) {
    if (!p) return fail(KDA_ERR_INVALID_ARG, "problem is NULL");
    if (p->B < 1 || p->T < 0 || p->H < 1 || p->K < 1 || p->V < 1)
        return fail(KDA_ERR_INVALID_ARG, "B, H, K, V must be >= 1 and T >= 0");
    if (p->K > 256) return fail(KDA_ERR_UNSUPPORTED, "key width above 256");
    if (p->V > 4096) return fail(KDA_ERR_UNSUPPORTED, "value width above 4096");
    if (p->H > 65535) return fail(KDA_ERR_UNSUPPORTED, "H > 65535");
    if (p->io != KDA_BF16 && p->io != KDA_FP32) return fail(KDA_ERR_INVALID_ARG, "unknown io dtype");
    if (p->gate != KDA_GATE_NONE && p->gate != KDA_GATE_SCALAR && p->gate != KDA_GATE_CHANNEL)
        return fail(KDA_ERR_INVALID_ARG, "unknown gate kind");
    if (p->save_policy != 0 && p->save_policy != 1)
        return fail(KDA_ERR_INVALID_ARG, "save_policy must be 0 or 1");
    if (p->schedule < 0 || (p->schedule > kda::MAX_PIECES && p->schedule != kda::SCHEDULE_JOINT))
        return fail(KDA_ERR_INVALID_ARG,
                    "schedule must be 0 (default), 1 (one pass), a piece count up to 8, or 9 (joint)");
    if (p->qk_l2norm != 0 && p->qk_l2norm != 1) return fail(KDA_ERR_INVALID_ARG, "qk_l2norm must be 0 or 1");
    if (p->HV != 0 && p->HV != p->H && (p->HV < p->H || p->HV % p->H != 0 || p->HV > 65535))
        return fail(KDA_ERR_INVALID_ARG, "HV must be 0 or a multiple of H (at most 65535)");
    if ((long long)(p->HV ? p->HV : p->H) * ((p->V + vblock_max(p) - 1) / vblock_max(p)) > 65535)
        return fail(KDA_ERR_UNSUPPORTED, "value heads times value blocks above 65535");
    if ((p->erase == nullptr) != (p->write == nullptr))
        return fail(KDA_ERR_INVALID_ARG, "erase and write come together (GatedDeltaNet-2)");
    if (p->A_log && p->gate == KDA_GATE_NONE) return fail(KDA_ERR_INVALID_ARG, "A_log needs a gate");
    if (p->dt_bias && !p->A_log) return fail(KDA_ERR_INVALID_ARG, "dt_bias needs A_log");
    if (p->A_log && !(p->lower_bound == 0.f || (p->lower_bound >= -5.f && p->lower_bound < 0.f)))
        return fail(KDA_ERR_INVALID_ARG, "lower_bound must be 0 or in [-5, 0)");
    const long long tok = (long long)p->B * p->T;
    if (tok > 0x7fffffffLL / 2) return fail(KDA_ERR_UNSUPPORTED, "too many tokens");
    d.Ttot = (int)tok;
    d.D = p->K;
    d.V = p->V;
    // bf16 up to 128 wide runs on the tensor cores at 128; otherwise the width itself (the
    // CUDA-core path's problems are padded to K = V = 64, 128 or 256 before they get here)
    d.WD = (p->io == KDA_BF16 && p->K <= 128 && p->V <= 128) ? 128 : p->K;
    d.H = p->H;
    d.alk = p->gate == KDA_GATE_CHANNEL ? kda::ALK_UNIT : p->gate == KDA_GATE_SCALAR ? kda::ALK_SCALAR : 0;
    const long long per = (p->T + kda::BT - 1) / kda::BT;
    if (p->cu_seqlens) {
        if (p->B != 1) return fail(KDA_ERR_INVALID_ARG, "packed sequences need B == 1");
        if (p->N < 1) return fail(KDA_ERR_INVALID_ARG, "packed sequences need N >= 1");
        d.N = p->N;
        const long long nc = per + p->N;
        if (nc > 0x7fffffffLL) return fail(KDA_ERR_UNSUPPORTED, "too many chunks");
        d.NC = (int)nc;
    } else {
        d.N = p->B;
        d.NC = (int)(per * p->B);
        d.per = (int)per;
    }
    return KDA_OK;
}

struct Layout {
    size_t table = 0, fcore = 0, fextra = 0, bwd = 0;   // CUDA-core path
    size_t ftc = 0, ftc_b = 0, btc = 0, wscr = 0;       // tensor-core path
    size_t piece = 0;   // time pieces of the tensor-core backward: two state adjoints, the claim counters
};

// The tensor-core path serves bf16 I/O with K, V <= 128 (at 128, its tile width: widths that are
// multiples of 8 are read and written as they are, others arrive padded to 128); everything else
// runs the fp32 CUDA-core kernels.
bool use_tc(const kda_problem* p) { return p->io == KDA_BF16 && p->K <= 128 && p->V <= 128; }

Layout layout(const Dims& d) {
    Layout L;
    const size_t NC = (size_t)d.NC, H = (size_t)d.H, D = (size_t)d.WD, BT = kda::BT;
    const size_t N = (size_t)d.N;
    L.table = up(sizeof(int32_t) * NC) * 2 + up(sizeof(int32_t) * (N + 1)) + up(sizeof(int32_t) * N) * 3 +
              up(sizeof(int32_t));   // the error word last (kda_device_status reads it there)
    const size_t chd = NC * H;
    L.fcore = up(4 * chd * BT * D) * 4 + up(4 * chd * BT * BT) * 2 + up(4 * chd * D);
    L.fextra = up(4 * chd * BT * D) + up(4 * chd * D * D);
    L.bwd = up(4 * chd * BT * D) * 4 + up(4 * chd * D * D) + up(4 * chd * BT * BT) * 2 +
            up(4 * chd * D) + up(4 * chd * BT);
    L.ftc = up(2 * chd * BT * D) * 4 + up(2 * chd * BT * BT) + up(4 * chd * D) + up(4 * chd) + up(4 * (chd + 1));
    L.ftc_b = up(2 * chd * BT * BT) + up(2 * chd * D * D) + up(2 * chd * BT * D) +
              (d.alk ? up(4 * chd * (size_t)d.alk) : 0);
    L.btc = up(2 * chd * D * D) + up(2 * chd * BT * D);
    L.wscr = up(4 * chd * BT * D) * 3 + up(4 * chd * BT * BT) * 2 + up(4 * chd * D) + up(4 * chd * BT);
    if (d.per) L.piece = 2 * up(4 * N * H * (size_t)d.D * d.V) + up(4 * kda::MAX_PIECES) + up(4 * chd);
    return L;
}

struct Carver {
    char* p;
    template <class T>
    T* take(size_t bytes) {
        T* r = reinterpret_cast<T*>(p);
        p += up(bytes);
        return r;
    }
};

kda::Table carve_table(Carver& c, const Dims& d) {
    kda::Table t;
    t.chunk_tok0 = c.take<int32_t>(sizeof(int32_t) * d.NC);
    t.chunk_len = c.take<int32_t>(sizeof(int32_t) * d.NC);
    t.seq_chunk0 = c.take<int32_t>(sizeof(int32_t) * (d.N + 1));
    t.seq_tok0 = c.take<int32_t>(sizeof(int32_t) * d.N);
    t.seq_len = c.take<int32_t>(sizeof(int32_t) * d.N);
    t.seq_order = c.take<int32_t>(sizeof(int32_t) * d.N);
    t.err = c.take<int32_t>(sizeof(int32_t));
    return t;
}

void carve_fwd(Carver& c, const Dims& d, kda::Fwd& f, bool extra) {
    const size_t chd = (size_t)d.NC * d.H, D = d.WD, BT = kda::BT;
    f.W = c.take<float>(4 * chd * BT * D);
    f.U = c.take<float>(4 * chd * BT * D);
    f.KG = c.take<float>(4 * chd * BT * D);
    f.QG = c.take<float>(4 * chd * BT * D);
    f.AQK = c.take<float>(4 * chd * BT * BT);
    f.AINV = c.take<float>(4 * chd * BT * BT);
    f.GL = c.take<float>(4 * chd * D);
    if (extra) {
        f.R = c.take<float>(4 * chd * BT * D);
        f.SIN = c.take<float>(4 * chd * D * D);
    } else {
        f.R = nullptr;
        f.SIN = nullptr;
    }
}

void carve_bwd(Carver& c, const Dims& d, kda::Bwd& b) {
    const size_t chd = (size_t)d.NC * d.H, D = d.WD, BT = kda::BT;
    b.P = c.take<float>(4 * chd * BT * D);
    b.QS = c.take<float>(4 * chd * BT * D);
    b.PS = c.take<float>(4 * chd * BT * D);
    b.FB = c.take<float>(4 * chd * BT * D);
    b.SBP = c.take<float>(4 * chd * D * D);
    b.DM = c.take<float>(4 * chd * BT * BT);
    b.HQ = c.take<float>(4 * chd * BT * BT);
    b.LAMB = c.take<float>(4 * chd * D);
    b.DBW = c.take<float>(4 * chd * BT);
}

void carve_fwd_tc(Carver& c, const Dims& d, kda::FwdTC& f, bool bwd_arrays) {
    const size_t chd = (size_t)d.NC * d.H, D = d.WD, BT = kda::BT;
    std::memset(&f, 0, sizeof(f));
    f.W = c.take<__nv_bfloat16>(2 * chd * BT * D);
    f.KG = c.take<__nv_bfloat16>(2 * chd * BT * D);
    f.QG = c.take<__nv_bfloat16>(2 * chd * BT * D);
    f.AQK = c.take<__nv_bfloat16>(2 * chd * BT * BT);
    f.U = c.take<__nv_bfloat16>(2 * chd * BT * D);
    f.GL = c.take<float>(4 * chd * D);
    f.WIDE = c.take<int32_t>(4 * chd);
    f.WLIST = c.take<int32_t>(4 * (chd + 1));
    if (bwd_arrays) {
        f.AI = c.take<__nv_bfloat16>(2 * chd * BT * BT);
        f.HS = c.take<__nv_bfloat16>(2 * chd * D * D);
        f.R = c.take<__nv_bfloat16>(2 * chd * BT * D);
        if (d.alk) f.ALK = c.take<float>(4 * chd * (size_t)d.alk);
    }
}

void carve_bwd_tc(Carver& c, const Dims& d, kda::BwdTC& b, kda::Bwd& scr) {
    const size_t chd = (size_t)d.NC * d.H, D = d.WD, BT = kda::BT;
    b.SBP = c.take<__nv_bfloat16>(2 * chd * D * D);
    b.P = c.take<__nv_bfloat16>(2 * chd * BT * D);
    std::memset(&scr, 0, sizeof(scr));
    scr.QS = c.take<float>(4 * chd * BT * D);
    scr.PS = c.take<float>(4 * chd * BT * D);
    scr.FB = c.take<float>(4 * chd * BT * D);
    scr.DM = c.take<float>(4 * chd * BT * BT);
    scr.HQ = c.take<float>(4 * chd * BT * BT);
    scr.LAMB = c.take<float>(4 * chd * D);
    scr.DBW = c.take<float>(4 * chd * BT);
}

kda::Shape shape_of(const kda_problem* p, const Dims& d) {
    kda::Shape s;
    s.H = p->H;
    s.K = p->K;
    s.V = p->V;
    s.N = d.N;
    s.NC = d.NC;
    s.Ttot = d.Ttot;
    s.scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->K);
    s.Hq = s.Hg = p->H;   // one q, k and one g, beta, erase head per value head
    return s;
}

// The width every key- and value-side tensor is zero-padded to (0: no padding). bf16 I/O with
// K, V <= 128 runs on the tensor cores at their own widths when both are multiples of 8 (the
// tensor maps read the missing columns as zeros) and the in-operator prologue, built for
// K = 64, 128 and 256, is off or fits; otherwise bf16 pads to 128. fp32 I/O runs K = V = 64 or
// 128 as they are and pads to 64 when both fit, else 128. K > 128 pads to 256 (K = V = 256 as is).
int pad_width(const kda_problem* p) {
    const bool bf16 = p->io == KDA_BF16;
    if (p->K == p->V && (p->K == 128 || p->K == 256 || (p->K == 64 && !bf16))) return 0;
    if (p->K > 128) return 256;
    if (bf16) {
        const bool prologue = p->A_log || p->qk_l2norm;
        if (p->V <= 128 && p->K % 8 == 0 && p->V % 8 == 0 && (!prologue || p->K == 64 || p->K == 128)) return 0;
        return 128;
    }
    return (p->K <= 64 && p->V <= 64) ? 64 : 128;
}
// The padded buffers, in a fixed order after the inner problem's workspace (base NULL: size only).
struct PadBufs {
    void *q = nullptr, *k = nullptr, *v = nullptr, *erase = nullptr, *write = nullptr, *o = nullptr, *dout = nullptr;
    void *dq = nullptr, *dk = nullptr, *dv = nullptr, *derase = nullptr, *dwrite = nullptr;
    float *g = nullptr, *h0 = nullptr, *dtb = nullptr, *ht = nullptr, *dht = nullptr, *dg = nullptr, *dh0 = nullptr,
          *ddtb = nullptr;
};
size_t pad_layout(const kda_problem* p, const Dims& d, bool bwd, char* base, PadBufs& b) {
    const size_t D = (size_t)pad_width(p), es = p->io == KDA_BF16 ? 2 : 4;
    const size_t Hv = (size_t)(p->HV ? p->HV : p->H), Hk = (size_t)p->H, T = (size_t)d.Ttot, N = (size_t)d.N;
    const bool ch = p->gate == KDA_GATE_CHANNEL;
    size_t n = 0;
    auto take = [&](size_t bytes) -> char* {
        char* r = base ? base + n : nullptr;
        n += up(bytes);
        return r;
    };
    b.q = take(es * T * Hk * D);
    b.k = take(es * T * Hk * D);
    b.v = take(es * T * Hv * D);
    if (ch) b.g = reinterpret_cast<float*>(take(4 * T * Hv * D));
    if (p->erase) {
        b.erase = take(es * T * Hv * D);
        b.write = take(es * T * Hv * D);
    }
    if (p->h0) b.h0 = reinterpret_cast<float*>(take(4 * N * Hv * D * D));
    if (p->dt_bias && ch) b.dtb = reinterpret_cast<float*>(take(4 * Hv * D));
    b.o = take(es * T * Hv * D);
    b.ht = reinterpret_cast<float*>(take(4 * N * Hv * D * D));
    if (bwd) {
        b.dout = take(es * T * Hv * D);
        b.dht = reinterpret_cast<float*>(take(4 * N * Hv * D * D));
        b.dq = take(es * T * Hk * D);
        b.dk = take(es * T * Hk * D);
        b.dv = take(es * T * Hv * D);
        if (ch) b.dg = reinterpret_cast<float*>(take(4 * T * Hv * D));
        if (p->erase) {
            b.derase = take(es * T * Hv * D);
            b.dwrite = take(es * T * Hv * D);
        }
        b.dh0 = reinterpret_cast<float*>(take(4 * N * Hv * D * D));
        if (p->dt_bias && ch) b.ddtb = reinterpret_cast<float*>(take(4 * Hv * D));
    }
    return n;
}
// The padded problem (sizes only, or pointed at the padded buffers).
kda_problem pad_inner(const kda_problem* p, const PadBufs* b) {
    kda_problem c = *p;
    c.K = c.V = pad_width(p);
    if (b) {
        c.q = b->q;
        c.k = b->k;
        c.v = b->v;
        if (b->g) c.g = b->g;
        if (p->erase) {
            c.erase = b->erase;
            c.write = b->write;
        }
        c.h0 = b->h0;
        if (b->dtb) c.dt_bias = b->dtb;
    }
    return c;
}

// Grouped value heads: the problem the rest of the library sees has one key head per value
// head. On the tensor-core path without the prologue its kernels read q, k of key head j / G
// for value head j in place; otherwise q, k are first copied per value head into the workspace.
bool gva(const kda_problem* p) { return p->HV != 0 && p->HV != p->H; }
bool has_prologue(const kda_problem* p);
bool gva_in_place(const kda_problem* p) { return use_tc(p) && !has_prologue(p); }
kda_problem gva_inner(const kda_problem* p, const void* qx, const void* kx) {
    kda_problem c = *p;
    c.H = p->HV;
    c.HV = 0;
    c.q = qx;
    c.k = kx;
    return c;
}
size_t gva_bytes(const kda_problem* p, const Dims& d, bool bwd) {
    const size_t one = up((size_t)(p->io == KDA_BF16 ? 2 : 4) * d.Ttot * p->HV * d.D);
    // q, k copies unless read in place; backward, their gradients per value head
    return one * ((gva_in_place(p) ? 0 : 2) + (bwd ? 2 : 0));
}

// Value widths above the block width M (128, or 256 when K > 128): NB = ceil(V / M) value blocks
// of width Vb = ceil(V / NB), each run as a value head of its own (the state's value columns
// evolve independently). Value rows are viewed as [tokens][value heads * NB][Vb] in place when
// NB * Vb == V, else padded first; per-head inputs repeat per block and their gradients sum over
// the blocks.
int vblocks(const kda_problem* p) {
    const int M = vblock_max(p);
    return p->V > M ? (p->V + M - 1) / M : 1;
}
int vblock_width(const kda_problem* p) { return (p->V + vblocks(p) - 1) / vblocks(p); }
bool vsplit(const kda_problem* p) { return vblocks(p) > 1; }
long long heads_v(const kda_problem* p) { return p->HV ? p->HV : p->H; }
struct SplitBufs;
kda_problem split_inner(const kda_problem* p, const SplitBufs* b);
// The blocks read g, beta and erase in place (block value head j reads head j / NB) when they run on
// the tensor-core path at their own width without the prologue; otherwise those repeat per block.
bool split_in_place(const kda_problem* p) {
    const kda_problem in = split_inner(p, nullptr);
    return use_tc(&in) && !has_prologue(p) && pad_width(&in) == 0;
}
// channels of g (and dt_bias) per token and head
int gate_width(const kda_problem* p) { return p->gate == KDA_GATE_NONE ? 0 : (p->gate == KDA_GATE_CHANNEL ? p->K : 1); }
struct SplitBufs {
    void *v = nullptr, *write = nullptr, *o = nullptr, *dout = nullptr, *dv = nullptr, *dwrite = nullptr;   // padded
    void *beta = nullptr, *erase = nullptr, *dbeta = nullptr, *derase = nullptr;   // per block
    float *g = nullptr, *A_log = nullptr, *dtb = nullptr, *dg = nullptr, *dA = nullptr, *ddtb = nullptr;
    float *h0 = nullptr, *ht = nullptr, *dht = nullptr, *dh0 = nullptr;   // [N][value heads * NB][K][Vb]
};
size_t split_layout(const kda_problem* p, const Dims& d, bool bwd, char* base, SplitBufs& b) {
    const size_t NB = vblocks(p), Vp = NB * vblock_width(p), es = p->io == KDA_BF16 ? 2 : 4;
    const size_t Hv = heads_v(p), T = d.Ttot, N = d.N, K = p->K, gw = gate_width(p);
    const bool padv = Vp != (size_t)p->V, gd2 = p->erase != nullptr, inpl = split_in_place(p);
    size_t n = 0;
    auto take = [&](size_t bytes) -> char* {
        char* r = base ? base + n : nullptr;
        n += up(bytes);
        return r;
    };
    if (padv) {
        b.v = take(es * T * Hv * Vp);
        if (gd2) b.write = take(es * T * Hv * Vp);
        b.o = take(es * T * Hv * Vp);
    }
    if (!inpl) {
        if (!gd2) b.beta = take(es * T * Hv * NB);
        if (gd2) b.erase = take(es * T * Hv * NB * K);
        if (gw) b.g = reinterpret_cast<float*>(take(4 * T * Hv * NB * gw));
    }
    if (p->A_log) b.A_log = reinterpret_cast<float*>(take(4 * Hv * NB));
    if (p->dt_bias) b.dtb = reinterpret_cast<float*>(take(4 * Hv * NB * gw));
    if (p->h0) b.h0 = reinterpret_cast<float*>(take(4 * N * Hv * K * Vp));
    b.ht = reinterpret_cast<float*>(take(4 * N * Hv * K * Vp));
    if (bwd) {
        if (padv) {
            b.dout = take(es * T * Hv * Vp);
            b.dv = take(es * T * Hv * Vp);
            if (gd2) b.dwrite = take(es * T * Hv * Vp);
        }
        if (!gd2) b.dbeta = take(es * T * Hv * NB);
        if (gd2) b.derase = take(es * T * Hv * NB * K);
        if (gw) b.dg = reinterpret_cast<float*>(take(4 * T * Hv * NB * gw));
        if (p->A_log) b.dA = reinterpret_cast<float*>(take(4 * Hv * NB));
        if (p->dt_bias) b.ddtb = reinterpret_cast<float*>(take(4 * Hv * NB * gw));
        b.dht = reinterpret_cast<float*>(take(4 * N * Hv * K * Vp));
        b.dh0 = reinterpret_cast<float*>(take(4 * N * Hv * K * Vp));
    }
    return n;
}
// The value-block problem (sizes only, or pointed at the split buffers).
kda_problem split_inner(const kda_problem* p, const SplitBufs* b) {
    kda_problem c = *p;
    c.V = vblock_width(p);
    c.HV = (int)(heads_v(p) * vblocks(p));
    if (b) {
        if (b->v) c.v = b->v;
        if (b->write) c.write = b->write;
        if (b->beta) c.beta = b->beta;
        if (b->erase) c.erase = b->erase;
        if (b->g) c.g = b->g;
        if (b->A_log) c.A_log = b->A_log;
        if (b->dtb) c.dt_bias = b->dtb;
        c.h0 = b->h0;
    }
    return c;
}

// The optional prologue (normalised q, k; activated decay) and what it needs.
bool has_prologue(const kda_problem* p) { return p->A_log || p->qk_l2norm; }
float l2eps(const kda_problem* p) { return p->l2norm_eps > 0.f ? p->l2norm_eps : 1e-6f; }
// The problem the chunk pipeline sees once the prologue has run.
kda_problem core_problem(const kda_problem* p) {
    kda_problem c = *p;
    c.A_log = nullptr;
    c.dt_bias = nullptr;
    c.lower_bound = 0.f;
    c.qk_l2norm = 0;
    return c;
}
size_t gate_elems(const kda_problem* p, const Dims& d) {
    return (size_t)d.Ttot * d.H * (p->gate == KDA_GATE_CHANNEL ? d.D : 1);
}
// Workspace after the pipeline's own: normalised q, k; activated decay; (backward) per-block partials.
size_t prologue_bytes(const kda_problem* p, const Dims& d, bool bwd) {
    if (!has_prologue(p) || d.Ttot == 0) return 0;
    const size_t es = p->io == KDA_BF16 ? 2 : 4, tok = (size_t)d.Ttot * d.H * d.D;
    size_t n = 0;
    if (p->qk_l2norm) n += 2 * up(es * tok);
    if (p->A_log) {
        n += up(4 * gate_elems(p, d));
        if (bwd) {
            const size_t nb = (size_t)kda::prologue_blocks(d.Ttot);
            n += up(4 * nb * d.H * (p->gate == KDA_GATE_CHANNEL ? d.D : 1)) + up(4 * nb * d.H);
        }
    }
    return n;
}

kda_status check_inputs(const kda_problem* p, const Dims& d) {
    if (d.Ttot > 0 && (!p->q || !p->k || !p->v || (!p->beta && !p->erase)))
        return fail(KDA_ERR_INVALID_ARG, "q, k, v and beta (or erase and write) must be non-NULL");
    if (p->gate == KDA_GATE_NONE && p->g) return fail(KDA_ERR_INVALID_ARG, "g must be NULL without a gate");
    if (p->gate != KDA_GATE_NONE && !p->g && d.Ttot > 0)
        return fail(KDA_ERR_INVALID_ARG, "g must be non-NULL with a gate");
    return KDA_OK;
}

kda_status check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (need == 0) return KDA_OK;
    if (!ws) return fail(KDA_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) % ALIGN) return fail(KDA_ERR_WORKSPACE, "workspace not 256-byte aligned");
    if (ws_bytes < need)
        return fail(KDA_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes");
    return KDA_OK;
}

kda_status cuda_fail(cudaError_t e, const char* where) {
    return fail(KDA_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

size_t state_bytes(const Dims& d) { return sizeof(float) * (size_t)d.N * d.H * d.D * d.V; }

// ------------------------------------------------------------------ tracing
struct Prof {
    bool on = false;
    struct Rec {
        const char* name;
        cudaEvent_t a, b;
    };
    std::vector<Rec> recs;
    std::vector<cudaEvent_t> pool;
    size_t used = 0;
    cudaEvent_t ev() {
        if (used == pool.size()) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
            pool.push_back(e);
        }
        return pool[used++];
    }
};
Prof g_prof;

// Runs one launch, bracketed by events when tracing is on.
template <class F>
cudaError_t traced(const char* name, cudaStream_t cs, F&& launch) {
    if (!g_prof.on) return launch();
    cudaEvent_t a = g_prof.ev(), b = g_prof.ev();
    if (a) cudaEventRecord(a, cs);
    cudaError_t e = launch();
    if (b) cudaEventRecord(b, cs);
    if (a && b) g_prof.recs.push_back({name, a, b});
    return e;
}

// A second stream for kernels that can run beside the caller's stream: two
// scans of one (sequence, head) each occupy a whole SM, so when the pairs fill
// at most half the GPU, two independent scans side by side cost one. One side
// stream and its fork/join events per host thread and device (so threads that
// call concurrently never share an event); created on first use and kept.
struct Side {
    cudaStream_t st = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool tried = false;
};
thread_local Side t_side[64];

// The side stream of the current device, or nullptr (then everything stays on
// the caller's stream).
Side* side_stream() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    Side& sd = t_side[dev];
    if (!sd.tried) {
        sd.tried = true;
        if (cudaStreamCreateWithFlags(&sd.st, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            sd.st = nullptr;
        }
    }
    return sd.st ? &sd : nullptr;
}

// Work enqueued on `side` after fork() follows everything already on `main`;
// work enqueued on `main` after join() follows everything enqueued on `side`.
cudaError_t side_fork(Side* sd, cudaStream_t main) {
    cudaError_t e = cudaEventRecord(sd->fork, main);
    return e != cudaSuccess ? e : cudaStreamWaitEvent(sd->st, sd->fork, 0);
}
cudaError_t side_join(Side* sd, cudaStream_t main) {
    cudaError_t e = cudaEventRecord(sd->join, sd->st);
    return e != cudaSuccess ? e : cudaStreamWaitEvent(main, sd->join, 0);
}

// Two concurrent scans fit when both grids (one CTA per (sequence, head) pair,
// one CTA per SM) are resident together.
bool scans_fit_together(const kda::Shape& s) { return 2L * s.N * s.H <= (long)kda::sm_count(); }

// Time pieces of the tensor-core backward (equal-length batches only): the reverse scan runs piece by
// piece, latest first, and each piece's units are consumed on the side stream while the scan goes on
// with the next piece, on the SMs it leaves idle. schedule 1 = one pass, P >= 2 = P pieces; the
// library's choice is the joint schedule where it applies and one pass elsewhere (under recompute
// the side stream already carries the recomputed scan ahead of the consumers, and one pass measured
// faster than pieces). At least two chunks per piece.
// The joint schedule: equal-length batches under the save policy whose scans fit beside the
// consumer (one (sequence, head) pair per SM at most). Asked for with schedule 9; the library's
// choice (schedule 0) when the scans leave at least half of the SMs to the consumer (measured:
// backward 0.855 ms against 0.950 in three pieces and 1.026 in one pass at the KDA workload, 0.408
// against 0.445 / 0.459 at the DeltaNet one; with 128 pairs on 152 SMs one pass was faster, 0.939
// against 0.971).
bool bwd_joint(const kda_problem* p, const Dims& d) {
    if (!d.per || !p->save_policy) return false;
    const long pairs = (long)d.N * d.H, sms = kda::sm_count();
    return p->schedule == kda::SCHEDULE_JOINT ? pairs <= sms : (p->schedule == 0 && 2 * pairs <= sms);
}

int bwd_pieces(const kda_problem* p, const Dims& d) {
    if (!d.per || p->schedule == kda::SCHEDULE_JOINT) return 1;
    int P = p->schedule >= 2 ? p->schedule : 1;
    while (P > 1 && d.per < 2 * P) --P;
    return P;
}

}  // namespace

namespace kda {
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace kda

extern "C" {

int kda_abi_version(void) { return 4; }

const char* kda_last_error(void) { return g_err.c_str(); }

static size_t core_workspace(const kda_problem* p, const Dims& d, int for_backward) {
    const Layout L = layout(d);
    if (use_tc(p)) {
        if (!for_backward) return L.table + (p->save_policy ? 0 : L.ftc);
        return L.table + (p->save_policy ? 0 : L.ftc + L.ftc_b) + L.btc + L.wscr + L.piece;
    }
    if (!for_backward) return L.table + (p->save_policy ? 0 : L.fcore);
    return L.table + (p->save_policy ? 0 : L.fcore + L.fextra) + L.bwd;
}

size_t kda_workspace_size(const kda_problem* p, int for_backward) {
    Dims d;
    if (check_dims(p, d) != KDA_OK) return 0;
    if (d.Ttot == 0) return 0;
    if (vsplit(p)) {
        SplitBufs b;
        const kda_problem in = split_inner(p, nullptr);
        return kda_workspace_size(&in, for_backward) + split_layout(p, d, for_backward != 0, nullptr, b);
    }
    if (pad_width(p)) {
        PadBufs b;
        const kda_problem in = pad_inner(p, nullptr);
        return kda_workspace_size(&in, for_backward) + pad_layout(p, d, for_backward != 0, nullptr, b);
    }
    if (gva(p)) {
        const kda_problem in = gva_inner(p, p->q, p->k);
        return kda_workspace_size(&in, for_backward) + gva_bytes(p, d, for_backward != 0);
    }
    const kda_problem c = core_problem(p);
    return core_workspace(&c, d, for_backward) + prologue_bytes(p, d, for_backward != 0);
}

size_t kda_saved_size(const kda_problem* p) {
    Dims d;
    if (check_dims(p, d) != KDA_OK) return 0;
    if (vsplit(p) && d.Ttot > 0) {
        const kda_problem in = split_inner(p, nullptr);
        return kda_saved_size(&in);
    }
    if (pad_width(p)) {
        const kda_problem in = pad_inner(p, nullptr);
        return kda_saved_size(&in);
    }
    if (gva(p)) {
        const kda_problem in = gva_inner(p, p->q, p->k);
        return kda_saved_size(&in);
    }
    if (!p->save_policy || d.Ttot == 0) return 0;
    const Layout L = layout(d);
    return use_tc(p) ? L.ftc + L.ftc_b : L.fcore + L.fextra;
}

// Value heads per head of q, k (Gq) and of g, beta, erase (Gg) for the tensor-core kernels' in-place
// reads of grouped heads and value blocks (1, 1: every input has one head per value head).
struct HeadGroups {
    int Gq = 1, Gg = 1;
};

// The chunk pipeline proper (the prologue, if any, has already run).
static kda_status chunk_fwd_core(const kda_problem* p, void* o, float* ht, void* saved, void* ws,
                                 size_t ws_bytes, kda_stream_t stream, HeadGroups hgr = {}) {
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    if (d.Ttot > 0 && !o) return fail(KDA_ERR_INVALID_ARG, "o must be non-NULL");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (d.Ttot == 0) {  // no tokens: the final state is the initial state
        if (ht) {
            cudaError_t e = p->h0 ? cudaMemcpyAsync(ht, p->h0, state_bytes(d), cudaMemcpyDeviceToDevice, cs)
                                  : cudaMemsetAsync(ht, 0, state_bytes(d), cs);
            if (e != cudaSuccess) return cuda_fail(e, "copy h0");
        }
        return KDA_OK;
    }
    if ((st = check_ws(ws, ws_bytes, kda_workspace_size(p, 0))) != KDA_OK) return st;
    if (p->save_policy && (st = check_ws(saved, kda_saved_size(p), kda_saved_size(p))) != KDA_OK)
        return fail(KDA_ERR_WORKSPACE, "saved buffer: " + g_err);
    if ((hgr.Gq != 1 || hgr.Gg != 1) && !use_tc(p))
        return fail(KDA_ERR_INVALID_ARG, "grouped inputs read in place need the tensor-core path");
    kda::Shape s = shape_of(p, d);
    s.Gq = hgr.Gq;
    s.Gg = hgr.Gg;
    s.Hq = s.H / hgr.Gq;
    s.Hg = s.H / hgr.Gg;
    Carver cw{static_cast<char*>(ws)};
    kda::Table t = carve_table(cw, d);
    const int bf16 = p->io == KDA_BF16;
    cudaError_t e;
    if (use_tc(p)) {
        kda::FwdTC f;
        const bool save = p->save_policy != 0;
        if (save) {
            Carver cs2{static_cast<char*>(saved)};
            carve_fwd_tc(cs2, d, f, true);
        } else {
            carve_fwd_tc(cw, d, f, false);
        }
        kda::TableZeros z;   // the prep's list of wide chunks starts empty
        z.p[0] = f.WLIST;
        z.n[0] = 1;
        e = traced("k_table", cs, [&] { return kda::launch_table(s, p->B, p->T, p->cu_seqlens, t, cs, z); });
        if (e != cudaSuccess) return cuda_fail(e, "chunk table");
        e = traced("k_prep_tc", cs, [&] { return kda::launch_prep_tc(s, (int)p->gate, save ? 1 : 0, p->q, p->k, p->v, p->beta, p->g, t, f, cs, kda::Gdn2{p->erase, p->write}); });
        if (e != cudaSuccess) return cuda_fail(e, "prep");
        e = traced("k_prep_wide", cs, [&] { return kda::launch_prep_wide(s, (int)p->gate, p->q, p->k, p->v, p->beta, p->g, t, f, cs, kda::Gdn2{p->erase, p->write}); });
        if (e != cudaSuccess) return cuda_fail(e, "prep (wide chunks)");
        // policy A: outputs and saved S, R from one scan, or (when the SMs allow) the output
        // scan and the S, R scan side by side
        Side* sd = (save && scans_fit_together(s)) ? side_stream() : nullptr;
        if (sd) {
            if ((e = side_fork(sd, cs)) != cudaSuccess) return cuda_fail(e, "side stream");
            e = traced("k_fwd_scan_tc_save", sd->st, [&] { return kda::launch_fwd_scan_tc(s, 2, p->h0, t, f, nullptr, nullptr, sd->st); });
            if (e != cudaSuccess) return cuda_fail(e, "forward scan (saved states)");
        }
        e = traced("k_fwd_scan_tc", cs, [&] { return kda::launch_fwd_scan_tc(s, (save && !sd) ? 3 : 1, p->h0, t, f, o, ht, cs); });
        if (e != cudaSuccess) return cuda_fail(e, "forward scan");
        if (sd && (e = side_join(sd, cs)) != cudaSuccess) return cuda_fail(e, "side stream");
        return KDA_OK;
    }
    e = traced("k_table", cs, [&] { return kda::launch_table(s, p->B, p->T, p->cu_seqlens, t, cs); });
    if (e != cudaSuccess) return cuda_fail(e, "chunk table");
    kda::Fwd f;
    if (p->save_policy) {
        Carver cs2{static_cast<char*>(saved)};
        carve_fwd(cs2, d, f, true);
    } else {
        carve_fwd(cw, d, f, false);
    }
    e = traced("k_prep", cs, [&] { return kda::launch_prep(s, bf16, (int)p->gate, p->q, p->k, p->v, p->beta, p->g, t, f, cs,
                                                                                  kda::Gdn2{p->erase, p->write}); });
    if (e != cudaSuccess) return cuda_fail(e, "prep");
    e = traced("k_fwd_scan", cs, [&] { return kda::launch_fwd_scan(s, bf16, p->save_policy ? 3 : 1, p->h0, t, f, o, ht, cs); });
    if (e != cudaSuccess) return cuda_fail(e, "forward scan");
    return KDA_OK;
}

static kda_status chunk_bwd_core(const kda_problem* p, const void* dout, const float* dht, const void* saved,
                                 void* dq, void* dk, void* dv, float* dg, void* dbeta, void* derase, void* dwrite,
                                 float* dh0, void* ws, size_t ws_bytes, kda_stream_t stream, HeadGroups hgr = {}) {
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    if (d.Ttot > 0 && (!dout || !dq || !dk || !dv || (!p->erase && !dbeta)))
        return fail(KDA_ERR_INVALID_ARG, "dout, dq, dk, dv and dbeta must be non-NULL");
    if (d.Ttot > 0 && p->erase && (!derase || !dwrite))
        return fail(KDA_ERR_INVALID_ARG, "derase and dwrite must be non-NULL with erase and write");
    const kda::Gdn2 gd{p->erase, p->write, derase, dwrite};
    if (p->gate == KDA_GATE_NONE && dg) return fail(KDA_ERR_INVALID_ARG, "dg must be NULL without a gate");
    if (p->gate != KDA_GATE_NONE && !dg && d.Ttot > 0)
        return fail(KDA_ERR_INVALID_ARG, "dg must be non-NULL with a gate");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (d.Ttot == 0) {  // no tokens: dh0 = dht
        if (dh0) {
            cudaError_t e = dht ? cudaMemcpyAsync(dh0, dht, state_bytes(d), cudaMemcpyDeviceToDevice, cs)
                                : cudaMemsetAsync(dh0, 0, state_bytes(d), cs);
            if (e != cudaSuccess) return cuda_fail(e, "copy dht");
        }
        return KDA_OK;
    }
    if ((st = check_ws(ws, ws_bytes, kda_workspace_size(p, 1))) != KDA_OK) return st;
    if (p->save_policy) {
        if (!saved) return fail(KDA_ERR_WORKSPACE, "policy A needs the saved buffer");
        if (reinterpret_cast<uintptr_t>(saved) % ALIGN)
            return fail(KDA_ERR_WORKSPACE, "saved buffer not 256-byte aligned");
    }
    if ((hgr.Gq != 1 || hgr.Gg != 1) && !use_tc(p))
        return fail(KDA_ERR_INVALID_ARG, "grouped inputs read in place need the tensor-core path");
    kda::Shape s = shape_of(p, d);
    s.Gq = hgr.Gq;
    s.Gg = hgr.Gg;
    s.Hq = s.H / hgr.Gq;
    s.Hg = s.H / hgr.Gg;
    Carver cw{static_cast<char*>(ws)};
    kda::Table t = carve_table(cw, d);
    if (use_tc(p)) {
        const bool save = p->save_policy != 0;
        kda::FwdTC f;
        if (save) {
            Carver cs2{static_cast<char*>(const_cast<void*>(saved))};
            carve_fwd_tc(cs2, d, f, true);
        } else {
            carve_fwd_tc(cw, d, f, true);
        }
        kda::BwdTC b;
        kda::Bwd scr;
        carve_bwd_tc(cw, d, b, scr);
        const int gate = (int)p->gate;
        // zeroed by the table's launch: the recompute prep's list of wide chunks and, for equal
        // lengths, the claim counters and ready flags after the two state adjoints of the piece area
        kda::TableZeros z;
        if (!save) {
            z.p[0] = f.WLIST;
            z.n[0] = 1;
        }
        if (d.per) {
            char* pz = cw.p + 2 * up(state_bytes(d));
            z.p[1] = reinterpret_cast<int32_t*>(pz);
            z.n[1] = kda::MAX_PIECES;
            z.p[2] = reinterpret_cast<int32_t*>(pz + up(4 * kda::MAX_PIECES));
            z.n[2] = d.NC * d.H;
        }
        cudaError_t e = traced("k_table", cs, [&] { return kda::launch_table(s, p->B, p->T, p->cu_seqlens, t, cs, z); });
        if (e != cudaSuccess) return cuda_fail(e, "chunk table");
        Side* sd = nullptr;
        if (!save) {
            e = traced("k_prep_tc", cs, [&] { return kda::launch_prep_tc(s, gate, 1, p->q, p->k, p->v, p->beta, p->g, t, f, cs, kda::Gdn2{p->erase, p->write}); });
            if (e != cudaSuccess) return cuda_fail(e, "prep (recompute)");
            e = traced("k_prep_wide", cs, [&] { return kda::launch_prep_wide(s, gate, p->q, p->k, p->v, p->beta, p->g, t, f, cs, kda::Gdn2{p->erase, p->write}); });
            if (e != cudaSuccess) return cuda_fail(e, "prep (recompute, wide chunks)");
            // the S, R recompute and the reverse scan need only the prep: side by side
            sd = side_stream();
            cudaStream_t rs = cs;
            if (sd) {
                if ((e = side_fork(sd, cs)) != cudaSuccess) return cuda_fail(e, "side stream");
                rs = sd->st;
            }
            e = traced("k_fwd_scan_tc_recompute", rs, [&] { return kda::launch_fwd_scan_tc(s, 2, p->h0, t, f, nullptr, nullptr, rs); });
            if (e != cudaSuccess) return cuda_fail(e, "forward scan (recompute)");
        }
        if (bwd_joint(p, d)) {
            // the joint schedule: scans and consumer in one cooperative launch; the ready flags and the
            // unit counter start at zero (the table's launch zeroed them)
            cw.take<float>(state_bytes(d));
            cw.take<float>(state_bytes(d));
            int* ctr = cw.take<int>(4 * kda::MAX_PIECES);
            int* flags = cw.take<int>(sizeof(int) * (size_t)d.NC * d.H);
            kda::ConsPiece pc;
            pc.per = d.per;
            pc.ctr = ctr;
            pc.flags = flags;
            e = traced("k_bwd_joint_tc", cs, [&] { return kda::launch_bwd_joint_tc(s, gate, p->q, p->k, p->v, p->beta, dout, dht, dh0, t, f, b, dq, dk, dv, dbeta, dg, cs, gd, pc); });
            if (e != cudaSuccess) return cuda_fail(e, "joint scan and consumer");
            e = traced("k_bwd_wide", cs, [&] { return gate == KDA_GATE_NONE ? cudaSuccess : kda::launch_bwd_wide(s, gate, p->q, p->k, p->v, p->beta, p->g, dout, t, f, b, scr, dq, dk, dv, dbeta, dg, cs, gd); });
            if (e != cudaSuccess) return cuda_fail(e, "consumer (wide chunks)");
            return KDA_OK;
        }
        int P = bwd_pieces(p, d);
        if (P > 1 && !sd) {
            sd = side_stream();
            if (!sd) P = 1;
            else if ((e = side_fork(sd, cs)) != cudaSuccess) return cuda_fail(e, "side stream");
        }
        if (P <= 1) {
            e = traced("k_bwd_scan_tc", cs, [&] { return kda::launch_bwd_scan_tc(s, dout, dht, t, f, b, dh0, cs); });
            if (e != cudaSuccess) return cuda_fail(e, "reverse scan");
            if (sd && (e = side_join(sd, cs)) != cudaSuccess) return cuda_fail(e, "side stream");
            e = traced("k_bwd_consumer_tc", cs, [&] { return kda::launch_bwd_consumer_tc(s, gate, p->q, p->k, p->v, p->beta, dout, t, f, b, dq, dk, dv, dbeta, dg, cs, gd); });
            if (e != cudaSuccess) return cuda_fail(e, "consumer");
        } else {
            // time pieces: the scan of piece q+1 (main stream) runs beside the consumer of piece q (side
            // stream, which also holds the recompute scan under policy R); the state adjoint entering a
            // piece goes to the next through one of two fp32 buffers
            float* hb[2] = {cw.take<float>(state_bytes(d)), cw.take<float>(state_bytes(d))};
            int* ctr = cw.take<int>(4 * kda::MAX_PIECES);   // zeroed by the table's launch
            for (int q = 0; q < P; ++q) {
                kda::ConsPiece pc;
                pc.per = d.per;
                pc.lo = (int)((long)d.per * (P - 1 - q) / P);
                pc.L = (int)((long)d.per * (P - q) / P) - pc.lo;
                pc.ctr = ctr + q;
                const float* din = q == 0 ? dht : hb[(q - 1) & 1];
                float* dnext = q == P - 1 ? dh0 : hb[q & 1];
                e = traced("k_bwd_scan_tc", cs, [&] { return kda::launch_bwd_scan_tc(s, dout, din, t, f, b, dnext, cs, pc); });
                if (e != cudaSuccess) return cuda_fail(e, "reverse scan");
                if ((e = side_fork(sd, cs)) != cudaSuccess) return cuda_fail(e, "side stream");
                e = traced("k_bwd_consumer_tc", sd->st, [&] { return kda::launch_bwd_consumer_tc(s, gate, p->q, p->k, p->v, p->beta, dout, t, f, b, dq, dk, dv, dbeta, dg, sd->st, gd, pc); });
                if (e != cudaSuccess) return cuda_fail(e, "consumer");
            }
            if ((e = side_join(sd, cs)) != cudaSuccess) return cuda_fail(e, "side stream");
        }
        if (gate != KDA_GATE_NONE) {
            e = traced("k_bwd_wide", cs, [&] { return kda::launch_bwd_wide(s, gate, p->q, p->k, p->v, p->beta, p->g, dout, t, f, b, scr, dq, dk, dv, dbeta, dg, cs, gd); });
            if (e != cudaSuccess) return cuda_fail(e, "consumer (wide chunks)");
        }
        return KDA_OK;
    }
    kda::Fwd f;
    if (p->save_policy) {
        Carver cs2{static_cast<char*>(const_cast<void*>(saved))};
        carve_fwd(cs2, d, f, true);
    } else {
        carve_fwd(cw, d, f, true);
    }
    kda::Bwd b;
    carve_bwd(cw, d, b);
    const int bf16 = p->io == KDA_BF16;
    cudaError_t e = traced("k_table", cs, [&] { return kda::launch_table(s, p->B, p->T, p->cu_seqlens, t, cs); });
    if (e != cudaSuccess) return cuda_fail(e, "chunk table");
    if (!p->save_policy) {
        e = traced("k_prep", cs, [&] { return kda::launch_prep(s, bf16, (int)p->gate, p->q, p->k, p->v, p->beta, p->g, t, f, cs,
                                                                                  kda::Gdn2{p->erase, p->write}); });
        if (e != cudaSuccess) return cuda_fail(e, "prep (recompute)");
        e = traced("k_fwd_scan_recompute", cs, [&] { return kda::launch_fwd_scan(s, bf16, 2, p->h0, t, f, nullptr, nullptr, cs); });
        if (e != cudaSuccess) return cuda_fail(e, "forward scan (recompute)");
    }
    e = traced("k_bwd_scan", cs, [&] { return kda::launch_bwd_scan(s, bf16, dout, dht, t, f, b, dh0, cs); });
    if (e != cudaSuccess) return cuda_fail(e, "reverse scan");
    e = traced("k_bwd_dstate", cs, [&] { return kda::launch_bwd_dstate(s, bf16, dout, p->v, p->beta, t, f, b, dv, cs, gd); });
    if (e != cudaSuccess) return cuda_fail(e, "state-gradient consumer");
    e = traced("k_bwd_intra", cs, [&] { return kda::launch_bwd_intra(s, bf16, (int)p->gate, p->q, p->k, p->beta, p->g, t, f, b, dq, dk, dbeta, dg, cs, gd); });
    if (e != cudaSuccess) return cuda_fail(e, "intra consumer");
    return KDA_OK;
}

// Runs the prologue into the workspace past the pipeline's part (at `core` bytes) and
// points a copy of the problem at its outputs.
static kda_status run_prologue(const kda_problem* p, const Dims& d, char* w, kda_problem& c, cudaStream_t cs) {
    Carver cv{w};
    const size_t es = p->io == KDA_BF16 ? 2 : 4, tok = (size_t)d.Ttot * d.H * d.D;
    kda::PrologueArgs a{};
    a.q = p->q;
    a.k = p->k;
    a.g = p->g;
    a.A_log = p->A_log;
    a.dt_bias = p->dt_bias;
    a.lower_bound = p->lower_bound;
    a.eps = l2eps(p);
    a.qk_norm = p->qk_l2norm;
    if (p->qk_l2norm) {
        a.qh = cv.take<char>(es * tok);
        a.kh = cv.take<char>(es * tok);
        c.q = a.qh;
        c.k = a.kh;
    }
    if (p->A_log) {
        a.ga = cv.take<float>(4 * gate_elems(p, d));
        c.g = a.ga;
    }
    const kda::Shape s = shape_of(p, d);
    cudaError_t e = traced("k_prologue", cs, [&] { return kda::launch_prologue(s, p->io == KDA_BF16, (int)p->gate, a, cs); });
    return e == cudaSuccess ? KDA_OK : cuda_fail(e, "prologue");
}

static kda_status chunk_fwd_pro(const kda_problem* p, void* o, float* ht, void* saved, void* ws, size_t ws_bytes,
                                kda_stream_t stream) {
    if (!p || !has_prologue(p)) return chunk_fwd_core(p, o, ht, saved, ws, ws_bytes, stream);
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    kda_problem c = core_problem(p);
    if (d.Ttot == 0) return chunk_fwd_core(&c, o, ht, saved, ws, ws_bytes, stream);
    const size_t core = core_workspace(&c, d, 0);
    if ((st = check_ws(ws, ws_bytes, core + prologue_bytes(p, d, false))) != KDA_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = run_prologue(p, d, static_cast<char*>(ws) + core, c, cs)) != KDA_OK) return st;
    return chunk_fwd_core(&c, o, ht, saved, ws, core, stream);
}

static kda_status chunk_bwd_pro(const kda_problem* p, const void* dout, const float* dht, const void* saved, void* dq,
                                void* dk, void* dv, float* dg, void* dbeta, void* derase, void* dwrite, float* dh0,
                                float* dA_log, float* ddt_bias, void* ws, size_t ws_bytes, kda_stream_t stream) {
    if (!p || !has_prologue(p))
        return chunk_bwd_core(p, dout, dht, saved, dq, dk, dv, dg, dbeta, derase, dwrite, dh0, ws, ws_bytes, stream);
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    kda_problem c = core_problem(p);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (!p->A_log) dA_log = nullptr;
    if (!p->dt_bias) ddt_bias = nullptr;
    if (d.Ttot == 0) {   // no tokens: the parameters get zero gradients
        cudaError_t e = cudaSuccess;
        if (dA_log) e = cudaMemsetAsync(dA_log, 0, sizeof(float) * d.H, cs);
        if (e == cudaSuccess && ddt_bias)
            e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * d.H * (p->gate == KDA_GATE_CHANNEL ? d.D : 1), cs);
        if (e != cudaSuccess) return cuda_fail(e, "zero parameter gradients");
        return chunk_bwd_core(&c, dout, dht, saved, dq, dk, dv, dg, dbeta, derase, dwrite, dh0, ws, ws_bytes, stream);
    }
    const size_t core = core_workspace(&c, d, 1);
    if ((st = check_ws(ws, ws_bytes, core + prologue_bytes(p, d, true))) != KDA_OK) return st;
    char* w = static_cast<char*>(ws) + core;
    if ((st = run_prologue(p, d, w, c, cs)) != KDA_OK) return st;
    st = chunk_bwd_core(&c, dout, dht, saved, dq, dk, dv, dg, dbeta, derase, dwrite, dh0, ws, core, stream);
    if (st != KDA_OK) return st;
    // the prologue's buffers, then the partial sums
    const size_t es = p->io == KDA_BF16 ? 2 : 4, tok = (size_t)d.Ttot * d.H * d.D;
    Carver cv{w};
    if (p->qk_l2norm) {
        cv.take<char>(es * tok);
        cv.take<char>(es * tok);
    }
    kda::EpilogueArgs a{};
    a.q = p->q;
    a.k = p->k;
    a.g = p->g;
    a.A_log = p->A_log;
    a.dt_bias = p->dt_bias;
    a.lower_bound = p->lower_bound;
    a.eps = l2eps(p);
    a.qk_norm = p->qk_l2norm;
    a.dq = dq;
    a.dk = dk;
    a.dg = dg;
    if (p->A_log) {
        cv.take<float>(4 * gate_elems(p, d));
        const size_t nb = (size_t)kda::prologue_blocks(d.Ttot);
        a.pz = cv.take<float>(4 * nb * d.H * (p->gate == KDA_GATE_CHANNEL ? d.D : 1));
        a.pA = cv.take<float>(4 * nb * d.H);
    }
    a.ddt_bias = ddt_bias;
    a.dA_log = dA_log;
    const kda::Shape s = shape_of(p, d);
    cudaError_t e = traced("k_epilogue", cs, [&] { return kda::launch_epilogue(s, p->io == KDA_BF16, (int)p->gate, a, cs); });
    if (e == cudaSuccess && p->A_log)
        e = traced("k_prologue_sum", cs, [&] { return kda::launch_prologue_sum(s, (int)p->gate, a, cs); });
    return e == cudaSuccess ? KDA_OK : cuda_fail(e, "epilogue");
}

// Grouped value heads: q, k copied per value head after the pipeline's workspace, then the
// one-key-head-per-value-head problem.
static kda_status gva_expand(const kda_problem* p, const Dims& d, char* w, kda_problem& in, cudaStream_t cs) {
    const size_t one = up((size_t)(p->io == KDA_BF16 ? 2 : 4) * d.Ttot * p->HV * d.D);
    in = gva_inner(p, w, w + one);
    cudaError_t e = traced("k_gva_expand", cs, [&] {
        return kda::launch_gva_expand(d.Ttot, p->HV, p->HV / p->H, d.D, p->io == KDA_BF16, p->q, p->k,
                                      const_cast<void*>(in.q), const_cast<void*>(in.k), cs);
    });
    return e == cudaSuccess ? KDA_OK : cuda_fail(e, "grouped heads: expand q, k");
}

// Gg > 1: the value-block caller's g, beta and erase, read in place (value head j reads head j / Gg).
static kda_status chunk_fwd_gva(const kda_problem* p, void* o, float* ht, void* saved, void* ws, size_t ws_bytes,
                                kda_stream_t stream, int Gg = 1) {
    if (!p || !gva(p)) return chunk_fwd_pro(p, o, ht, saved, ws, ws_bytes, stream);
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    kda_problem in = gva_inner(p, p->q, p->k);
    if (d.Ttot == 0) return chunk_fwd_pro(&in, o, ht, saved, ws, ws_bytes, stream);
    const size_t core = kda_workspace_size(&in, 0);
    if ((st = check_ws(ws, ws_bytes, core + gva_bytes(p, d, false))) != KDA_OK) return st;
    if (gva_in_place(p)) return chunk_fwd_core(&in, o, ht, saved, ws, core, stream, HeadGroups{p->HV / p->H, Gg});
    if (Gg != 1) return fail(KDA_ERR_INVALID_ARG, "value blocks read in place need grouped heads read in place");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = gva_expand(p, d, static_cast<char*>(ws) + core, in, cs)) != KDA_OK) return st;
    return chunk_fwd_pro(&in, o, ht, saved, ws, core, stream);
}

static kda_status chunk_bwd_gva(const kda_problem* p, const void* dout, const float* dht, const void* saved, void* dq,
                                void* dk, void* dv, float* dg, void* dbeta, void* derase, void* dwrite, float* dh0,
                                float* dA_log, float* ddt_bias, void* ws, size_t ws_bytes, kda_stream_t stream,
                                int Gg = 1) {
    if (!p || !gva(p))
        return chunk_bwd_pro(p, dout, dht, saved, dq, dk, dv, dg, dbeta, derase, dwrite, dh0, dA_log, ddt_bias, ws,
                             ws_bytes, stream);
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    kda_problem in = gva_inner(p, p->q, p->k);
    if (d.Ttot == 0)
        return chunk_bwd_pro(&in, dout, dht, saved, dq, dk, dv, dg, dbeta, derase, dwrite, dh0, dA_log, ddt_bias, ws,
                             ws_bytes, stream);
    if (!dq || !dk) return fail(KDA_ERR_INVALID_ARG, "dq and dk must be non-NULL");
    const size_t core = kda_workspace_size(&in, 1);
    if ((st = check_ws(ws, ws_bytes, core + gva_bytes(p, d, true))) != KDA_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    char* w = static_cast<char*>(ws) + core;
    const size_t one = up((size_t)(p->io == KDA_BF16 ? 2 : 4) * d.Ttot * p->HV * d.D);
    const bool inpl = gva_in_place(p);
    if (!inpl && Gg != 1) return fail(KDA_ERR_INVALID_ARG, "value blocks read in place need grouped heads read in place");
    if (!inpl && (st = gva_expand(p, d, w, in, cs)) != KDA_OK) return st;
    void* dqx = w + (inpl ? 0 : 2) * one;   // dq, dk per value head, after the q, k copies if any
    void* dkx = w + (inpl ? 1 : 3) * one;
    if (inpl)
        st = chunk_bwd_core(&in, dout, dht, saved, dqx, dkx, dv, dg, dbeta, derase, dwrite, dh0, ws, core, stream,
                            HeadGroups{p->HV / p->H, Gg});
    else
        st = chunk_bwd_pro(&in, dout, dht, saved, dqx, dkx, dv, dg, dbeta, derase, dwrite, dh0, dA_log, ddt_bias, ws,
                           core, stream);
    if (st != KDA_OK) return st;
    cudaError_t e = traced("k_gva_reduce", cs, [&] {
        return kda::launch_gva_reduce(d.Ttot, p->H, p->HV / p->H, d.D, p->io == KDA_BF16, dqx, dkx, dq, dk, cs);
    });
    return e == cudaSuccess ? KDA_OK : cuda_fail(e, "grouped heads: reduce dq, dk");
}

// Widths pad_width pads: every key- and value-side tensor zero-padded to the working width after
// the inner problem's workspace, outputs and gradients cropped back.
struct PadIo {
    const kda_problem* p;
    const Dims& d;
    cudaStream_t cs;
    cudaError_t e = cudaSuccess;
    int D() const { return pad_width(p); }
    long long Hv() const { return p->HV ? p->HV : p->H; }
    // token rows [rows][w] <-> [rows][D]
    void rows(bool pad, int es, long long n, int w, const void* src, void* dst) {
        if (e == cudaSuccess && src && dst)
            e = traced(pad ? "k_pad" : "k_crop", cs, [&] { return kda::launch_pad(pad, es, n, 1, w, 1, D(), src, dst, cs); });
    }
    // states [N * Hv][K][V] <-> [N * Hv][D][D]
    void states(bool pad, const void* src, void* dst) {
        if (e == cudaSuccess && src && dst)
            e = traced(pad ? "k_pad" : "k_crop", cs, [&] {
                return kda::launch_pad(pad, 4, (long long)d.N * Hv(), p->K, p->V, D(), D(), src, dst, cs);
            });
    }
};

static kda_status pad_inputs(const kda_problem* p, const Dims& d, const PadBufs& b, cudaStream_t cs) {
    PadIo io{p, d, cs};
    const int es = p->io == KDA_BF16 ? 2 : 4;
    const long long T = d.Ttot, Hk = p->H, Hv = io.Hv();
    io.rows(true, es, T * Hk, p->K, p->q, b.q);
    io.rows(true, es, T * Hk, p->K, p->k, b.k);
    io.rows(true, es, T * Hv, p->V, p->v, b.v);
    io.rows(true, 4, T * Hv, p->K, p->gate == KDA_GATE_CHANNEL ? p->g : nullptr, b.g);
    io.rows(true, es, T * Hv, p->K, p->erase, b.erase);
    io.rows(true, es, T * Hv, p->V, p->write, b.write);
    io.states(true, p->h0, b.h0);
    io.rows(true, 4, Hv, p->K, b.dtb ? p->dt_bias : nullptr, b.dtb);
    return io.e == cudaSuccess ? KDA_OK : cuda_fail(io.e, "pad to the working width");
}

static kda_status chunk_fwd_pad(const kda_problem* p, void* o, float* ht, void* saved, void* ws, size_t ws_bytes,
                                kda_stream_t stream) {
    if (!p || !pad_width(p)) return chunk_fwd_gva(p, o, ht, saved, ws, ws_bytes, stream);
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    if (d.Ttot > 0 && !o) return fail(KDA_ERR_INVALID_ARG, "o must be non-NULL");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t sb = sizeof(float) * (size_t)d.N * (p->HV ? p->HV : p->H) * p->K * p->V;
    if (d.Ttot == 0) {   // no tokens: the final state is the initial state
        if (!ht) return KDA_OK;
        cudaError_t e = p->h0 ? cudaMemcpyAsync(ht, p->h0, sb, cudaMemcpyDeviceToDevice, cs) : cudaMemsetAsync(ht, 0, sb, cs);
        return e == cudaSuccess ? KDA_OK : cuda_fail(e, "copy h0");
    }
    const kda_problem in0 = pad_inner(p, nullptr);
    const size_t core = kda_workspace_size(&in0, 0);
    PadBufs b;
    if ((st = check_ws(ws, ws_bytes, core + pad_layout(p, d, false, nullptr, b))) != KDA_OK) return st;
    pad_layout(p, d, false, static_cast<char*>(ws) + core, b);
    if ((st = pad_inputs(p, d, b, cs)) != KDA_OK) return st;
    const kda_problem in = pad_inner(p, &b);
    if ((st = chunk_fwd_gva(&in, b.o, b.ht, saved, ws, core, stream)) != KDA_OK) return st;
    PadIo io{p, d, cs};
    io.rows(false, p->io == KDA_BF16 ? 2 : 4, (long long)d.Ttot * io.Hv(), p->V, b.o, o);
    io.states(false, b.ht, ht);
    return io.e == cudaSuccess ? KDA_OK : cuda_fail(io.e, "crop from the working width");
}

static kda_status chunk_bwd_pad(const kda_problem* p, const void* dout, const float* dht, const void* saved,
                                void* dq, void* dk, void* dv, float* dg, void* dbeta, void* derase, void* dwrite,
                                float* dh0, float* dA_log, float* ddt_bias, void* ws, size_t ws_bytes,
                                kda_stream_t stream) {
    if (!p || !pad_width(p))
        return chunk_bwd_gva(p, dout, dht, saved, dq, dk, dv, dg, dbeta, derase, dwrite, dh0, dA_log, ddt_bias, ws,
                             ws_bytes, stream);
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const bool ch = p->gate == KDA_GATE_CHANNEL;
    if (d.Ttot == 0) {   // no tokens: dh0 = dht, parameters get zero gradients
        const size_t sb = sizeof(float) * (size_t)d.N * (p->HV ? p->HV : p->H) * p->K * p->V;
        cudaError_t e = cudaSuccess;
        if (dh0) e = dht ? cudaMemcpyAsync(dh0, dht, sb, cudaMemcpyDeviceToDevice, cs) : cudaMemsetAsync(dh0, 0, sb, cs);
        const size_t hv = (size_t)(p->HV ? p->HV : p->H);
        if (e == cudaSuccess && dA_log && p->A_log) e = cudaMemsetAsync(dA_log, 0, 4 * hv, cs);
        if (e == cudaSuccess && ddt_bias && p->dt_bias) e = cudaMemsetAsync(ddt_bias, 0, 4 * hv * (ch ? p->K : 1), cs);
        return e == cudaSuccess ? KDA_OK : cuda_fail(e, "empty backward");
    }
    if (!dout || !dq || !dk || !dv) return fail(KDA_ERR_INVALID_ARG, "dout, dq, dk and dv must be non-NULL");
    const kda_problem in0 = pad_inner(p, nullptr);
    const size_t core = kda_workspace_size(&in0, 1);
    PadBufs b;
    if ((st = check_ws(ws, ws_bytes, core + pad_layout(p, d, true, nullptr, b))) != KDA_OK) return st;
    pad_layout(p, d, true, static_cast<char*>(ws) + core, b);
    if ((st = pad_inputs(p, d, b, cs)) != KDA_OK) return st;
    PadIo io{p, d, cs};
    const int es = p->io == KDA_BF16 ? 2 : 4;
    const long long T = d.Ttot, Hk = p->H, Hv = io.Hv();
    io.rows(true, es, T * Hv, p->V, dout, b.dout);
    io.states(true, dht, b.dht);
    if (io.e != cudaSuccess) return cuda_fail(io.e, "pad to the working width");
    const kda_problem in = pad_inner(p, &b);
    st = chunk_bwd_gva(&in, b.dout, dht ? b.dht : nullptr, saved, b.dq, b.dk, b.dv, ch ? b.dg : dg, dbeta,
                       p->erase ? b.derase : nullptr, p->erase ? b.dwrite : nullptr, b.dh0, dA_log,
                       b.ddtb ? b.ddtb : ddt_bias, ws, core, stream);
    if (st != KDA_OK) return st;
    io.rows(false, es, T * Hk, p->K, b.dq, dq);
    io.rows(false, es, T * Hk, p->K, b.dk, dk);
    io.rows(false, es, T * Hv, p->V, b.dv, dv);
    if (ch) io.rows(false, 4, T * Hv, p->K, b.dg, dg);
    io.rows(false, es, T * Hv, p->K, b.derase, derase);
    io.rows(false, es, T * Hv, p->V, b.dwrite, dwrite);
    io.states(false, b.dh0, dh0);
    if (b.ddtb) io.rows(false, 4, Hv, p->K, b.ddtb, ddt_bias);
    return io.e == cudaSuccess ? KDA_OK : cuda_fail(io.e, "crop from the working width");
}

// Value widths above 128: the value-block problem after the inner problem's workspace.
struct SplitIo {
    const kda_problem* p;
    const Dims& d;
    cudaStream_t cs;
    cudaError_t e = cudaSuccess;
    int NB() const { return vblocks(p); }
    int Vb() const { return vblock_width(p); }
    int Vp() const { return NB() * Vb(); }
    long long rows() const { return (long long)d.Ttot * heads_v(p); }
    // value rows [rows][V] <-> [rows][NB * Vb]
    void value_rows(bool pad, int es, const void* src, void* dst) {
        if (e == cudaSuccess && src && dst)
            e = traced(pad ? "k_pad" : "k_crop", cs,
                       [&] { return kda::launch_pad(pad, es, rows(), 1, p->V, 1, Vp(), src, dst, cs); });
    }
    // per-head rows [M][W] -> [M][NB][W]
    void repeat(int es, long long M, int W, const void* src, void* dst) {
        if (e == cudaSuccess && src && dst)
            e = traced("k_vblock_repeat", cs, [&] { return kda::launch_vblock_repeat(es, M, NB(), W, src, dst, cs); });
    }
    // gradients [M][NB][W] -> [M][W]
    void sum(int es, long long M, int W, const void* src, void* dst) {
        if (e == cudaSuccess && src && dst)
            e = traced("k_vblock_sum", cs, [&] { return kda::launch_vblock_sum(es, M, NB(), W, src, dst, cs); });
    }
    // states [N * Hv][K][V] <-> [N * Hv][NB][K][Vb]
    void states(bool split, const float* src, float* dst) {
        if (e == cudaSuccess && src && dst)
            e = traced("k_vblock_state", cs, [&] {
                return kda::launch_vblock_state(split, (long long)d.N * heads_v(p), p->K, p->V, NB(), Vb(), src, dst, cs);
            });
    }
};

static kda_status split_inputs(const kda_problem* p, const Dims& d, const SplitBufs& b, cudaStream_t cs) {
    SplitIo io{p, d, cs};
    const int es = p->io == KDA_BF16 ? 2 : 4, gw = gate_width(p);
    const long long Hv = heads_v(p);
    io.value_rows(true, es, p->v, b.v);
    io.value_rows(true, es, p->write, b.write);
    io.repeat(es, io.rows(), 1, p->beta, b.beta);
    io.repeat(es, io.rows(), p->K, p->erase, b.erase);
    io.repeat(4, io.rows(), gw, p->g, b.g);
    io.repeat(4, Hv, 1, p->A_log, b.A_log);
    io.repeat(4, Hv, gw, p->dt_bias, b.dtb);
    io.states(true, p->h0, b.h0);
    return io.e == cudaSuccess ? KDA_OK : cuda_fail(io.e, "split into value blocks");
}

kda_status kda_chunk_fwd(const kda_problem* p, void* o, float* ht, void* saved, void* ws, size_t ws_bytes,
                         kda_stream_t stream) {
    if (!p || !vsplit(p)) return chunk_fwd_pad(p, o, ht, saved, ws, ws_bytes, stream);
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    if (d.Ttot == 0) return chunk_fwd_pad(p, o, ht, saved, ws, ws_bytes, stream);   // ht = h0, no kernel
    if (!o) return fail(KDA_ERR_INVALID_ARG, "o must be non-NULL");
    const kda_problem in0 = split_inner(p, nullptr);
    const size_t core = kda_workspace_size(&in0, 0);
    SplitBufs b;
    if ((st = check_ws(ws, ws_bytes, core + split_layout(p, d, false, nullptr, b))) != KDA_OK) return st;
    split_layout(p, d, false, static_cast<char*>(ws) + core, b);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = split_inputs(p, d, b, cs)) != KDA_OK) return st;
    const kda_problem in = split_inner(p, &b);
    // in place: the blocks run at their own width, so the padding layer has nothing to do
    st = split_in_place(p) ? chunk_fwd_gva(&in, b.o ? b.o : o, b.ht, saved, ws, core, stream, vblocks(p))
                           : chunk_fwd_pad(&in, b.o ? b.o : o, b.ht, saved, ws, core, stream);
    if (st != KDA_OK) return st;
    SplitIo io{p, d, cs};
    io.value_rows(false, p->io == KDA_BF16 ? 2 : 4, b.o, o);
    io.states(false, b.ht, ht);
    return io.e == cudaSuccess ? KDA_OK : cuda_fail(io.e, "merge the value blocks");
}

kda_status kda_chunk_bwd(const kda_problem* p, const void* dout, const float* dht, const void* saved, void* dq,
                         void* dk, void* dv, float* dg, void* dbeta, void* derase, void* dwrite, float* dh0,
                         float* dA_log, float* ddt_bias, void* ws, size_t ws_bytes, kda_stream_t stream) {
    if (!p || !vsplit(p))
        return chunk_bwd_pad(p, dout, dht, saved, dq, dk, dv, dg, dbeta, derase, dwrite, dh0, dA_log, ddt_bias, ws,
                             ws_bytes, stream);
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    if (d.Ttot == 0)   // dh0 = dht and zero parameter gradients, no kernel
        return chunk_bwd_pad(p, dout, dht, saved, dq, dk, dv, dg, dbeta, derase, dwrite, dh0, dA_log, ddt_bias, ws,
                             ws_bytes, stream);
    if (!dout || !dq || !dk || !dv || (!p->erase && !dbeta))
        return fail(KDA_ERR_INVALID_ARG, "dout, dq, dk, dv and dbeta must be non-NULL");
    if (p->erase && (!derase || !dwrite))
        return fail(KDA_ERR_INVALID_ARG, "derase and dwrite must be non-NULL with erase and write");
    if ((p->gate == KDA_GATE_NONE) != (dg == nullptr))
        return fail(KDA_ERR_INVALID_ARG, "dg must be non-NULL exactly when there is a gate");
    const kda_problem in0 = split_inner(p, nullptr);
    const size_t core = kda_workspace_size(&in0, 1);
    SplitBufs b;
    if ((st = check_ws(ws, ws_bytes, core + split_layout(p, d, true, nullptr, b))) != KDA_OK) return st;
    split_layout(p, d, true, static_cast<char*>(ws) + core, b);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = split_inputs(p, d, b, cs)) != KDA_OK) return st;
    SplitIo io{p, d, cs};
    const int es = p->io == KDA_BF16 ? 2 : 4, gw = gate_width(p);
    io.value_rows(true, es, dout, b.dout);
    io.states(true, dht, b.dht);
    if (io.e != cudaSuccess) return cuda_fail(io.e, "split into value blocks");
    const kda_problem in = split_inner(p, &b);
    if (split_in_place(p))
        st = chunk_bwd_gva(&in, b.dout ? b.dout : dout, dht ? b.dht : nullptr, saved, dq, dk, b.dv ? b.dv : dv, b.dg,
                           b.dbeta, b.derase, b.dwrite ? b.dwrite : dwrite, b.dh0, b.dA, b.ddtb, ws, core, stream,
                           vblocks(p));
    else
        st = chunk_bwd_pad(&in, b.dout ? b.dout : dout, dht ? b.dht : nullptr, saved, dq, dk, b.dv ? b.dv : dv, b.dg,
                           b.dbeta, b.derase, b.dwrite ? b.dwrite : dwrite, b.dh0, b.dA, b.ddtb, ws, core, stream);
    if (st != KDA_OK) return st;
    const long long Hv = heads_v(p);
    io.value_rows(false, es, b.dv, dv);
    io.value_rows(false, es, b.dwrite, dwrite);
    io.sum(4, io.rows(), gw, b.dg, dg);
    io.sum(es, io.rows(), 1, b.dbeta, dbeta);
    io.sum(es, io.rows(), p->K, b.derase, derase);
    io.sum(4, Hv, 1, b.dA, dA_log);
    io.sum(4, Hv, gw, b.ddtb, ddt_bias);
    io.states(false, b.dh0, dh0);
    return io.e == cudaSuccess ? KDA_OK : cuda_fail(io.e, "merge the value blocks");
}

kda_status kda_recurrent_fwd(const kda_problem* p, void* o, float* ht, int32_t* err, kda_stream_t stream) {
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if ((st = check_inputs(p, d)) != KDA_OK) return st;
    if (p->save_policy != 0) return fail(KDA_ERR_INVALID_ARG, "the recurrent forward has no saved buffer: use save_policy 0");
    if (!kda::recurrent_key_width(p->K) || p->V % 32 != 0)
        return fail(KDA_ERR_UNSUPPORTED,
                    "the token-by-token forward needs K = 64, 128, 160, 192 or 256 and V a multiple of 32");
    if (d.Ttot > 0 && !o) return fail(KDA_ERR_INVALID_ARG, "o must be non-NULL");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const kda_problem in = gva(p) ? gva_inner(p, p->q, p->k) : *p;   // value heads; q, k read per group
    const kda::Shape s = shape_of(&in, d);
    const int group = gva(p) ? p->HV / p->H : 1;
    cudaError_t e = traced("k_recurrent", cs, [&] {
        return kda::launch_recurrent(s, p->io == KDA_BF16, (int)p->gate, p->T, p->cu_seqlens, p->q, p->k, p->v, p->beta,
                                     p->g, p->h0, o, ht, err, p->A_log, p->dt_bias, p->lower_bound, p->qk_l2norm,
                                     l2eps(p), cs, kda::Gdn2{p->erase, p->write}, group);
    });
    if (e != cudaSuccess) return cuda_fail(e, "recurrent forward");
    return KDA_OK;
}

int kda_profile_begin(void) {
    g_prof.on = true;
    g_prof.recs.clear();
    g_prof.used = 0;
    return 0;
}

int kda_profile_end(kda_kernel_time* out, int max_entries) {
    g_prof.on = false;
    std::vector<kda_kernel_time> agg;
    for (auto& r : g_prof.recs) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -1;
        size_t i = 0;
        for (; i < agg.size(); ++i)
            if (std::strncmp(agg[i].name, r.name, sizeof(agg[i].name)) == 0) break;
        if (i == agg.size()) {
            kda_kernel_time k;
            std::memset(&k, 0, sizeof(k));
            std::strncpy(k.name, r.name, sizeof(k.name) - 1);
            agg.push_back(k);
        }
        agg[i].launches += 1;
        agg[i].total_ms += ms;
    }
    g_prof.recs.clear();
    g_prof.used = 0;
    const int n = (int)agg.size() < max_entries ? (int)agg.size() : max_entries;
    for (int i = 0; i < n && out; ++i) out[i] = agg[i];
    return n;
}

kda_status kda_device_status(const kda_problem* p, const void* ws, size_t ws_bytes, kda_stream_t stream,
                             int32_t* word) {
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if (!word) return fail(KDA_ERR_INVALID_ARG, "word is NULL");
    *word = 0;
    if (d.Ttot == 0) return KDA_OK;
    const Layout L = layout(d);
    if (!ws || ws_bytes < L.table) return fail(KDA_ERR_WORKSPACE, "workspace too small");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    const size_t off = L.table - up(sizeof(int32_t));
    e = cudaMemcpy(word, static_cast<const char*>(ws) + off, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    if (*word & 2) return fail(KDA_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up; results are not valid");
    if (*word & 1) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens was inconsistent and was clamped");
    return KDA_OK;
}

kda_status kda_selftest_device_timeout(const kda_problem* p, void* ws, size_t ws_bytes, unsigned limit_us,
                                       kda_stream_t stream) {
    Dims d;
    kda_status st = check_dims(p, d);
    if (st != KDA_OK) return st;
    if (d.Ttot == 0) return fail(KDA_ERR_INVALID_ARG, "the self-test needs a problem with tokens (a chunk table)");
    if (limit_us < 1 || limit_us > 1000000) return fail(KDA_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
    const Layout L = layout(d);
    if ((st = check_ws(ws, ws_bytes, L.table)) != KDA_OK) return st;
    Carver cw{static_cast<char*>(ws)};
    kda::Table t = carve_table(cw, d);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = kda::launch_wait_selftest(t, (uint64_t)limit_us * 1000ull, cs);
    return e == cudaSuccess ? KDA_OK : cuda_fail(e, "timeout self-test");
}

}  // extern "C"
