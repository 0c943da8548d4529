// Tensor-core backward path (bf16 I/O, K = V = 128) on tcgen05.
//
// k_bwd_scan_tc (a8, a9 first product), one CTA per (sequence, head), 256
// threads, warps w and w+4 own value columns 32(w%4).. . The transposed state adjoint
// S_bar^T (V x K, fp32) stays in TMEM; chunks are visited last to first:
//     R_bar^T = S+bar^T F^T + dO^T C_q          ("State and gate composition":
//                                               both uses of R before the pullback)
//     P^T     = R_bar^T A                        (Algorithm 1, step 1: P = A^T R_bar)
//     S_bar^T = S+bar^T diag(lambda) + dO^T Q_g - R_bar^T W
// where -R_bar^T W is the residual state term -E^T P supplied once
// ("ReWY: Faster Backpropagation for Delta-Rule Attention", Algorithm 1 step 5
// and "Complete Reverse Execution and Boundaries"). S+bar and P of every chunk
// go to HBM (bf16) for the consumer. C_q, A, Q_g and W are read as MN-major
// operands from their tile images, staged by bulk copies.
//
// k_bwd_consumer_tc (a9-a12), persistent (one CTA per SM walks the (chunk slot, head)
// units, loading the next unit's tiles while it finishes the current one), 512 threads:
//     [H_q ; -D] = [dO ; P] R^T   (masked: inclusive / strict, sign of D)
//     [dO S^T ; P S^T] = [dO ; P] S^T        F_bar^T = S+bar R^T
//     [T_q ; T_e] = [H_q ; D] (K zeta)        (A operand read from TMEM)
//     T_y^T       = [E_alpha^T | Q_alpha^T] [D ; H_q]
// with alpha = 2^(G2 - c), zeta = 2^(c - G2) around the per-feature midpoint
// c ("Matrix intra for vector-gated interactions", centered factors), alpha and
// 2^c as the forward prep saved them for this pass; a scalar
// gate instead folds 2^(G2_i - G2_j) into H_q and D and uses unit factors, so
// the key-gradient contractions carry the gate reduction without a key Gram
// matrix ("Gram elimination for scalar-gate gradients"). Then the chain rule
// and the reverse in-chunk cumsum of the log-gate gradient ("Complete
// Reverse Execution and Boundaries", steps 3-4). Chunks whose gate range is
// wider than the single-anchor limit (sub-chunk anchoring for per-channel
// gates; strong scalar decay, where the log-gate gradient cancels heavily)
// are left to the fp32 CUDA-core consumers.
#include <string.h>

#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using bf16 = __nv_bfloat16;
constexpr int D = 128;

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, int32_t* err) {
    bool ok = tc::mbar_wait(bar, parity);
    ok = __syncthreads_and(ok) != 0;
    if (!ok && threadIdx.x == 0) atomicOr(err, 2);
    return ok;
}

// ====================================================== k_bwd_scan_tc
constexpr int ST = 256;            // compute warps: warps w and w+4 share lane quarter w%4, split columns
constexpr int ST_ALL = ST + 32;    // + one warp that issues the MMAs and the bulk fills
constexpr int NB_AS = 1;           // named barriers (compute warps + issuer): A operands of R_bar staged
constexpr int NB_AR = 2;           //   A operands of the state adjoint update and P staged
constexpr int NB_C = 3;            //   compute warps only
// B operands as tile images: F read K-major, the rest MN-major
constexpr int B_STAGE = 0;      // two stages of B operands
constexpr int S_KG = 0;         // F   [64][128] 16 KB
constexpr int S_AQ = 16384;     // C_q [64][64]   8 KB
constexpr int S_AI = 24576;     // A   [64][64]   8 KB
constexpr int S_QG = 32768;     // Q_g [64][128] 16 KB
constexpr int S_W = 49152;      // W   [64][128] 16 KB
constexpr int S_DO = 65536;     // dO  [64][128] 16 KB, TMA (read MN-major as the A operand dO^T)
constexpr int B_STG = 81920;
// S+bar of one chunk and P of the chunk after it as tile images, written to HBM by the issuer
// (one bulk copy each) after the next hand-over
constexpr int B_SST = B_STAGE + 2 * B_STG;     // S+bar [128][128] bf16 32 KB
constexpr int B_PST = B_SST + D * D * 2;       // P     [64][128]  bf16 16 KB
constexpr int B_LAM = B_PST + BT * D * 2;      // lambda [128] fp32
constexpr int B_TST = B_LAM + 512;             // per-warp transpose staging, 8 x 1280 B
constexpr int B_BAR = B_TST + 8 * 1280;
constexpr int BSCAN_SMEM = B_BAR + 64 + 1024;
// TMEM columns: S_bar^T fp32 [0,128), R_bar^T fp32 [128,192), P^T double buffer [192,320);
// bf16 A operands (two values per column): S+bar^T [320,384), R_bar^T [384,416),
// -R_bar^T [416,448)
constexpr int T_RB = 128, T_P = 192, T_AS = 320, T_AR = 384, T_NR = 416;

// Stages the operand tiles of one chunk (tile images by bulk copies, dO by
// TMA from the token tensor); one thread; completion arrives on `full` as
// transaction bytes. dO rows past the chunk end meet zero rows of C_q and Q_g.
__device__ __forceinline__ void bscan_fill(uint32_t stg, const FwdTC& f, size_t ch, const CUtensorMap* tmo, int h,
                                           int tok0, uint64_t* full) {
    constexpr uint32_t TILE = BT * D * 2, TQ = BT * BT * 2;
    tc::mbar_arrive_expect_tx(full, 4 * TILE + 2 * TQ);
    tc::tma_load3(stg + S_DO, tmo, 0, h, tok0, full);
    tc::tma_load3(stg + S_DO + 8192, tmo, 64, h, tok0, full);
    tc::bulk_g2s(stg + S_KG, f.KG + ch * BT * D, TILE, full);
    tc::bulk_g2s(stg + S_AQ, f.AQK + ch * BT * BT, TQ, full);
    tc::bulk_g2s(stg + S_AI, f.AI + ch * BT * BT, TQ, full);
    tc::bulk_g2s(stg + S_QG, f.QG + ch * BT * D, TILE, full);
    tc::bulk_g2s(stg + S_W, f.W + ch * BT * D, TILE, full);
}

// Compute warps: per chunk (last to first) S+bar^T -> bf16 A operand, then
// (while R_bar runs) S_bar^T <- S+bar^T diag(lambda); R_bar^T -> bf16 A operands;
// then, while the state adjoint update runs, S+bar and the previous P to HBM.
// NARROW: the states are [K][V] with K, V taken at run time (at most D); otherwise [D][D], folded into
// the addressing.
template <bool NARROW>
__device__ __forceinline__ void bscan_compute(const Shape& s, const float* __restrict__ dht, const Table& t,
                                              const FwdTC& f, const BwdTC& b, float* __restrict__ dh0,
                                              unsigned char* base, uint64_t* bar, uint32_t tb, int nseq, int h,
                                              int c0, int c1, const int* flags) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    float* sLam = reinterpret_cast<float*>(base + B_LAM);
    bf16* tst = reinterpret_cast<bf16*>(base + B_TST + warp * 1280);
    const int H = s.H;
    const int vcol = 32 * quad + lane;
    const int kb = 64 * half, ib = 32 * half;
    const uint32_t tl = tc::taddr(tb, 32 * quad, 0);
    const int K = NARROW ? s.K : D, V = NARROW ? s.V : D;   // the state's widths ([K][V] per sequence and head)
    const size_t st_off = ((size_t)nseq * H + h) * K * V;

#pragma unroll 1
    for (int cb = kb; cb < kb + 64; cb += 16) {
        float a[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
            a[jj] = (dht && cb + jj < K && vcol < V) ? dht[st_off + (size_t)(cb + jj) * V + vcol] : 0.f;
        tc::tmem_st16(tl + cb, a);
    }
    tc::tmem_wait_st();

    bool ok = true;
    auto wait_one = [&](uint64_t* bb, uint32_t parity) {
        if (ok && !tc::mbar_wait(bb, parity)) {
            ok = false;
            atomicOr(t.err, 2);
        }
        tc::fence_after_sync();
    };
    // P of a chunk (rows ib..ib+31 of this thread's value column) from its TMEM buffer to HBM
    auto store_p = [&](int cc, int buf) {
        bf16* P = b.P + ((size_t)cc * H + h) * BT * D;
        float pv[2][16];
        const uint32_t tp = tl + T_P + 64 * buf;
        tc::tmem_ld16(tp + ib, pv[0]);
        tc::tmem_ld16(tp + ib + 16, pv[1]);
        tc::tmem_wait_ld();
        tc::warp_store_t16_img(tst, pv[0], P, BT, ib, 32 * quad, lane);
        tc::warp_store_t16_img(tst, pv[1], P, BT, ib + 16, 32 * quad, lane);
    };
    float gln = 0.f;
    if (c0 < c1 && tid < D) gln = f.GL[((size_t)(c1 - 1) * H + h) * D + tid];
    for (int c = c1 - 1; c >= c0; --c) {
        const int it = c1 - 1 - c;
        const size_t ch = (size_t)c * H + h;
        if (tid < D) sLam[tid] = exp2f(gln);
        if (c - 1 >= c0 && tid < D) gln = f.GL[(ch - H) * D + tid];
        if (it > 0) wait_one(&bar[1], (it - 1) & 1);   // state adjoint update of the later chunk
        tc::named_sync(NB_C, ST);
        // 1. S+bar^T -> bf16 A operand in TMEM, handed to the issuer
        float sv[4][16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld16(tl + kb + 16 * q4, sv[q4]);
        tc::tmem_wait_ld();
        uint32_t sp[2][16];   // bf16 S+bar^T, also what goes to HBM
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                sp[hq][jj] = tc::pack_bf16(sv[2 * hq][2 * jj], sv[2 * hq][2 * jj + 1]);
                sp[hq][8 + jj] = tc::pack_bf16(sv[2 * hq + 1][2 * jj], sv[2 * hq + 1][2 * jj + 1]);
            }
            tc::tmem_st16u(tl + T_AS + kb / 2 + 16 * hq, sp[hq]);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::named_sync(NB_AS, ST_ALL);
        // 2. while R_bar runs: S_bar^T <- S+bar^T diag(lambda) (before the update MMAs accumulate)
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const int cb = kb + 16 * q4;
            float a[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) a[jj] = sv[q4][jj] * sLam[cb + jj];
            tc::tmem_st16(tl + cb, a);
        }
        tc::tmem_wait_st();
        // 3. R_bar^T -> bf16 A operands R_bar^T and -R_bar^T, handed over
        wait_one(&bar[0], it & 1);
        {
            float rv[2][16];
            tc::tmem_ld16(tl + T_RB + ib, rv[0]);
            tc::tmem_ld16(tl + T_RB + ib + 16, rv[1]);
            tc::tmem_wait_ld();
            uint32_t pw[16], nw[16];
#pragma unroll
            for (int cq = 0; cq < 2; ++cq)
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    pw[8 * cq + jj] = tc::pack_bf16(rv[cq][2 * jj], rv[cq][2 * jj + 1]);
                    nw[8 * cq + jj] = tc::pack_bf16(-rv[cq][2 * jj], -rv[cq][2 * jj + 1]);
                }
            tc::tmem_st16u(tl + T_AR + ib / 2, pw);
            tc::tmem_st16u(tl + T_NR + ib / 2, nw);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::named_sync(NB_AR, ST_ALL);
        // 4. while the update runs: S+bar of this chunk and P of the later one as tile images into
        //    the staging area (the issuer copies them to HBM after the next hand-over)
        // A lane holds bf16 pairs along keys for its value column; neighbouring lanes swap halves
        // so that each writes pairs along values (one 32-bit store per pair of rows)
        const bool odd = lane & 1;
        // the staging addresses are loop-invariant; an opaque zero keeps the compiler from holding
        // all of them in registers across the chunk loop
        int col2;
        asm volatile("mov.b32 %0, %1;" : "=r"(col2) : "r"(vcol & ~1));
        auto put2 = [&](uint16_t* img, int R, int row0, uint32_t mine) {
            const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
            const uint32_t w = odd ? __byte_perm(other, mine, 0x7632) : __byte_perm(mine, other, 0x5410);
            *reinterpret_cast<uint32_t*>(img + tile_el(R, row0 + (odd ? 1 : 0), col2)) = w;
        };
        {
            uint16_t* hs = reinterpret_cast<uint16_t*>(base + B_SST);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                for (int m = 0; m < 8; ++m) put2(hs, D, kb + 16 * q4 + 2 * m, sp[q4 >> 1][8 * (q4 & 1) + m]);
        }
        if (it > 0) {
            // P of the later chunk: one barrier per TMEM buffer, so the commit of this chunk's P
            // (already possible here) cannot be mistaken for it
            wait_one(&bar[2 + ((it - 1) & 1)], ((it - 1) >> 1) & 1);
            float pv[2][16];
            const uint32_t tp = tl + T_P + 64 * ((it - 1) & 1);
            tc::tmem_ld16(tp + ib, pv[0]);
            tc::tmem_ld16(tp + ib + 16, pv[1]);
            tc::tmem_wait_ld();
            uint16_t* ps = reinterpret_cast<uint16_t*>(base + B_PST);
#pragma unroll
            for (int m = 0; m < 16; ++m)
                put2(ps, BT, ib + 2 * m, tc::pack_bf16(pv[m >> 3][(2 * m) & 15], pv[m >> 3][(2 * m + 1) & 15]));
        }
        tc::fence_async_smem();
    }
    if (c1 > c0) {
        const int last = c1 - 1 - c0;
        wait_one(&bar[1], last & 1);
        wait_one(&bar[2 + (last & 1)], (last >> 1) & 1);
        store_p(c0, last & 1);
        if (flags) __threadfence();   // P of the first chunk, published after the CTA barrier
    }
    if (ok && dh0) {
#pragma unroll 1
        for (int cb = kb; cb < kb + 64; cb += 16) {
            float a[16];
            tc::tmem_ld16(tl + cb, a);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
                if (cb + jj < K && vcol < V) dh0[st_off + (size_t)(cb + jj) * V + vcol] = a[jj];
        }
    }
}

// Issuer warp: bulk / TMA fills (lane 0) and the three MMA groups of every
// chunk (warp-uniform descriptors, one elected lane issuing).
__device__ __forceinline__ void bscan_issue(const Shape& s, const Table& t, const FwdTC& f, const BwdTC& b,
                                            const CUtensorMap* tmo, uint32_t sb, uint64_t* bar, uint64_t* full,
                                            uint32_t tb, int h, int c0, int c1, int& filled, int& waited, int* flags) {
    const int lane = threadIdx.x & 31;
    const int H = s.H;
    const uint32_t i64 = tc::idesc_bf16(128, 64), m64 = tc::idesc_bf16_bmn(128, 64),
                   m128 = tc::idesc_bf16_bmn(128, 128), am64 = tc::idesc_bf16_abmn(128, 64),
                   am128 = tc::idesc_bf16_abmn(128, 128);
    int tok_next = (c1 - 2 >= c0) ? t.chunk_tok0[c1 - 2] : 0;   // first token of the chunk filled next
    for (int c = c1 - 1; c >= c0; --c) {
        const int it = c1 - 1 - c, stage = it & 1;
        const uint32_t stg = sb + B_STAGE + stage * B_STG;
        const uint64_t dO = tc::sdesc_mn(stg + S_DO, BT * 128, 0);
        tc::named_sync(NB_AS, ST_ALL);
        tc::fence_after_sync();
        if (!tc::mbar_wait(&full[stage], (it >> 1) & 1) && lane == 0) atomicOr(t.err, 2);
        {
            // R_bar^T = S+bar^T F^T + dO^T C_q (dO^T read MN-major from the staged dO rows)
            const uint64_t dF = tc::sdesc(stg + S_KG), dC = tc::sdesc_mn(stg + S_AQ, BT * 128, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16_ts_w(tb + T_RB, tb + T_AS + 8 * ks, tc::kstep_k(dF, BT, ks), i64, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16_w(tb + T_RB, tc::kstep_mn(dO, ks), tc::kstep_mn(dC, ks), am64, 1);
            tc::mma_commit_w(&bar[0]);
        }
        if (lane == 0) {
            ++waited;
            if (c - 1 >= c0) {
                // the other stage is free once every MMA of the later chunk has completed
                if (it > 0 && !tc::mbar_wait(&bar[2 + ((it - 1) & 1)], ((it - 1) >> 1) & 1)) atomicOr(t.err, 2);
                bscan_fill(sb + B_STAGE + (stage ^ 1) * B_STG, f, (size_t)(c - 1) * H + h, tmo, h, tok_next,
                           &full[stage ^ 1]);
                ++filled;
                tok_next = (c - 2 >= c0) ? t.chunk_tok0[c - 2] : 0;
            }
            // S+bar of the later chunk c+1 and P of chunk c+2, staged during the last iteration;
            // the staging area is rewritten after the next hand-over, so their reads must be done
            if (it >= 1) {
                tc::bulk_s2g(b.SBP + ((size_t)(c + 1) * H + h) * D * D, sb + B_SST, D * D * 2);
                if (it >= 2) tc::bulk_s2g(b.P + ((size_t)(c + 2) * H + h) * BT * D, sb + B_PST, BT * D * 2);
                tc::bulk_commit();
                tc::bulk_wait_read();
                // joint schedule: the group committed one iteration ago (S+bar of chunk c+2, P of chunk
                // c+3) is complete, so chunk c+3 (whose S+bar went out an iteration before) is ready
                if (flags && it >= 3) {
                    tc::bulk_wait_prev();
                    tc::publish_flag(flags + (size_t)(c + 3) * H + h);
                }
            }
        }
        __syncwarp();
        tc::named_sync(NB_AR, ST_ALL);
        tc::fence_after_sync();
        {
            // S_bar^T += dO^T Q_g - R_bar^T W (it gates the next chunk), then P^T = R_bar^T A
            const uint64_t dQ = tc::sdesc_mn(stg + S_QG, BT * 128, 0), dW = tc::sdesc_mn(stg + S_W, BT * 128, 0);
            const uint64_t dA = tc::sdesc_mn(stg + S_AI, BT * 128, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc::mma_bf16_w(tb, tc::kstep_mn(dO, ks), tc::kstep_mn(dQ, ks), am128, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc::mma_bf16_ts_w(tb, tb + T_NR + 8 * ks, tc::kstep_mn(dW, ks), m128, 1);
            tc::mma_commit_w(&bar[1]);
            const uint32_t tP = tb + T_P + 64 * stage;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc::mma_bf16_ts_w(tP, tb + T_AR + 8 * ks, tc::kstep_mn(dA, ks), m64, ks > 0);
            tc::mma_commit_w(&bar[2 + stage]);
        }
    }
}

// The reverse scan of one (sequence, head), or of one time piece of it (chunks plo .. plo+pl-1: dht is
// then the state adjoint leaving the piece and dh0 the one entering it), by a CTA of ST_ALL or more
// threads: warps 0..7 compute, warp 8 issues, further warps only meet the CTA barriers. tb: 512 TMEM
// columns allocated by the caller. flags (the joint schedule): a ready flag per (chunk slot, head), set
// once the chunk's S+bar and P are in HBM.
template <bool NARROW>
__device__ __forceinline__ void bscan_body(const Shape& s, const CUtensorMap* tmo, const float* __restrict__ dht,
                                           const Table& t, const FwdTC& f, const BwdTC& b, float* __restrict__ dh0,
                                           int nseq, int h, int plo, int pl, int* flags, unsigned char* base,
                                           uint32_t tb) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(base + B_BAR);   // R_bar, state adjoint update, P (x2)
    uint64_t* full = bar + 4;                                      // operand stages 0, 1
    const uint32_t sb = tc::smem_u32(base);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int c0 = t.seq_chunk0[nseq] + (pl ? plo : 0), c1 = pl ? c0 + pl : t.seq_chunk0[nseq + 1];
    const bool issuer = warp == ST / 32;
    int filled = 0, waited = 0;   // bulk fills issued / consumed (issuer lane 0)

    if (issuer && (tid & 31) == 0) {
        for (int i = 0; i < 6; ++i) tc::mbar_init(&bar[i], 1);
        tc::fence_mbar_init();
        if (c0 < c1) {
            bscan_fill(sb + B_STAGE, f, (size_t)(c1 - 1) * s.H + h, tmo, h, t.chunk_tok0[c1 - 1], &full[0]);
            filled = 1;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (issuer)
        bscan_issue(s, t, f, b, tmo, sb, bar, full, tb, h, c0, c1, filled, waited, flags);
    else if (warp < ST / 32)
        bscan_compute<NARROW>(s, dht, t, f, b, dh0, base, bar, tb, nseq, h, c0, c1, flags);
    // a bulk fill still in flight (only after a timeout) lands before the CTA moves on
    if (issuer && (tid & 31) == 0)
        for (; waited < filled; ++waited) tc::mbar_wait(&full[waited & 1], (waited >> 1) & 1);
    tc::fence_before_sync();
    __syncthreads();
    // S+bar of the first chunk and P of the one after it, staged in the last iteration; the chunks not
    // published inside the loop are published now
    if (issuer && (tid & 31) == 0 && c1 > c0) {
        tc::bulk_s2g(b.SBP + ((size_t)c0 * s.H + h) * D * D, sb + B_SST, D * D * 2);
        if (c1 - c0 >= 2) tc::bulk_s2g(b.P + ((size_t)(c0 + 1) * s.H + h) * BT * D, sb + B_PST, BT * D * 2);
        tc::bulk_commit();
        tc::bulk_wait_all();
        if (flags)
            for (int c = c0; c < c1 && c < c0 + 3; ++c) tc::publish_flag(flags + (size_t)c * s.H + h);
    }
}

__global__ void __launch_bounds__(ST_ALL, 1)
    k_bwd_scan_tc(Shape s, const __grid_constant__ CUtensorMap tmo, const float* __restrict__ dht, Table t,
                  FwdTC f, BwdTC b, float* __restrict__ dh0, int plo, int pl) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + B_BAR + 48);
    if (threadIdx.x < 32) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tb = *tslot;
    // sequences in the table's order (longest first), every head of one before the next
    const int lin = (int)(blockIdx.x + blockIdx.y * gridDim.x);
    bscan_body<true>(s, &tmo, dht, t, f, b, dh0, t.seq_order[lin / s.H], lin % s.H, plo, pl, nullptr, base, tb);
    tc::fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) tc::tmem_dealloc(tb, 512);
}

// ================================================== k_bwd_consumer_tc
// Persistent: one CTA per SM walks the (chunk slot, head) units u = c * H + h,
// u = blockIdx.x, blockIdx.x + gridDim.x, ...; the inputs of the next unit are
// loaded while this one finishes (three groups, each on its own mbarrier):
//   X1: [R ; S], S+bar tile images        } after this unit's phase-B MMAs (the phase-B
//   X2: [dO ; P], v                        }   operands are the last readers of the X region)
//   C:  k, q (SW128 rows), the prep's   after this unit's key-major epilogue
//       alpha (per-channel gate: fp32 token rows; scalar gate: one per token)
// Every accumulator the chain rule reads is key-major (TMEM lane = key k, column = token j), so
// one pass in registers forms dq, dk, dbeta and G_bar, the reverse in-chunk cumsum runs inside
// each thread over its tokens, and dq, dk, dg go from registers to HBM.
constexpr int CT = 512;   // 16 warps: warp w reads TMEM lane quarter w % 4 and token group w / 4
constexpr int LDR = CT - 32;   // the thread that finds the next unit and issues its loads
// region X: phase A operands, then phase B operands
constexpr int X_RS = 0;          // [R ; S]   bf16 [192][128]  48 KB   (X1)
constexpr int X_SB = 49152;      // S+bar     bf16 [128][128]  32 KB   (X1)
constexpr int X_OP = 81920;      // [dO ; P]  bf16 [128][128]  32 KB   (X2)
constexpr int X_V = 114688;      // v         bf16 [64][128]   16 KB   (X2, SW128 rows)
constexpr int X_EQ = 0;          // [E_a^T | Q_a^T] tf32 [128][128] 64 KB   (rows key k, K = i')
constexpr int X_DH = 65536;      // [D ; H_q]^T     tf32 [64][128]   32 KB   (rows token j, K = i')
constexpr int X_BT = 98304;      // [D ; H_q]       tf32 [128][64]   32 KB   (rows i', K = token j)
constexpr int X_END = 131072;
constexpr int X_STG = X_END;     // per-warp staging of the transposed bf16 stores, 16 x 512 B; from the
                                 // next unit's group C to its alpha pass, a scalar gate's alphas
constexpr int C_A = X_STG + 16 * 512;             // the prep's alpha = 2^(G2 - c) as fp32 token rows
                                                  // [64][128] (per-channel gate), then key-major
constexpr int C_K = C_A + 4 * BT * D;             // k bf16 [64][128], SW128 rows
constexpr int C_Q = C_K + 2 * BT * D;             // q bf16 [64][128], SW128 rows
constexpr int C_MISC = C_Q + 2 * BT * D;          // small arrays (floats)
constexpr int M_BETA = 0, M_C2 = 64, M_AL = 192, M_DBW = 320, M_ROWP = 384, M_ENDP = 640, M_ROWG = 1152,
              M_META = 1408, M_LAMP = 1416, M_SEG = 1928, M_ENDQ = 2440, M_END = 2448;
constexpr int C_BAR = C_MISC + 4 * M_END;
constexpr int CONS_SMEM = C_BAR + 64 + 1024;
// TMEM columns: [H_q ; -D] token-major, then the key-major accumulators (lane = key k, column =
// token j): S dO^T, S P^T, F_bar^T, T_e^T, T_q^T, T_y^T; (K zeta)^T is the A operand of [T_e ; T_q]^T
constexpr int T_HD = 0, T_SDO = 64, T_SP = 128, T_FB = 192, T_TE = 256, T_TQ = 320, T_Y = 384, T_KZ = 448;
static_assert(X_V + BT * D * 2 <= X_END && X_BT + 2 * BT * BT * 4 <= X_END && X_DH + BT * D * 4 <= X_BT, "X region");
static_assert(X_STG + 16 * 512 <= C_A && 4 * ALK_SCALAR <= 16 * 512, "staging region");
static_assert(X_OP % 1024 == 0 && X_V % 1024 == 0 && X_SB % 1024 == 0 && X_DH % 1024 == 0 && X_BT % 1024 == 0 &&
              C_A % 1024 == 0 && C_K % 1024 == 0 && C_Q % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(CONS_SMEM <= 232448, "consumer shared memory above the per-block limit");
// The joint kernel: the larger of the two maps; its TMEM slot lies past both roles' barriers.
constexpr int J_SLOT = B_BAR + 56;
constexpr int JOINT_SMEM = BSCAN_SMEM > CONS_SMEM ? BSCAN_SMEM : CONS_SMEM;
static_assert(J_SLOT + 4 <= JOINT_SMEM - 1024 && C_BAR + 40 <= J_SLOT, "joint kernel TMEM slot");

__device__ __forceinline__ float bfx(const bf16* p) { return __bfloat162float(*p); }

// Byte offset of element (token j, key k) in a [64][128] bf16 tile stored in SW128 rows, from the
// column part kcol = (k / 64) * 64 * 128 + (k % 8) * 2 and the chunk index kch = (k / 8) % 8.
__device__ __forceinline__ uint32_t swrow(uint32_t kcol, int kch, int j) {
    return kcol + (uint32_t)(j * 128) + ((uint32_t)(kch ^ (j & 7)) << 4);
}

// Key-major tiles the alpha pass writes over the tiles it has read (each thread writes, and later
// reads, its own key and 16 tokens): alpha fp32 [128 keys][64 tokens] over the alpha rows, k and q
// bf16 [128 keys][64 tokens] over the token-major k and q tiles. Their 16-byte chunks are XORed
// with the key, so that eight consecutive keys reach distinct bank groups.
__device__ __forceinline__ int akm4(int kr, int c4) { return kr * BT + ((c4 ^ (kr & 15)) << 2); }   // alpha, tokens 4 c4 ..
__device__ __forceinline__ int kkm8(int kr, int c8) { return kr * BT + ((c8 ^ (kr & 7)) << 3); }   // bf16, tokens 8 c8 ..
__device__ __forceinline__ void ld_alpha16(const float* sA, int kr, int grp, float (&al)[16]) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 v = *reinterpret_cast<const float4*>(sA + akm4(kr, 4 * grp + m));
        al[4 * m] = v.x;
        al[4 * m + 1] = v.y;
        al[4 * m + 2] = v.z;
        al[4 * m + 3] = v.w;
    }
}
__device__ __forceinline__ void ld_bf16x16(const bf16* t, int kr, int grp, uint32_t (&w)[8]) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const uint4 v = *reinterpret_cast<const uint4*>(t + kkm8(kr, 2 * grp + b));
        w[4 * b] = v.x;
        w[4 * b + 1] = v.y;
        w[4 * b + 2] = v.z;
        w[4 * b + 3] = v.w;
    }
}
// The low (hi = 0) or high bf16 of a packed pair, as a float.
__device__ __forceinline__ float bf_lo_hi(uint32_t w, int hi) { return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16)); }

// Units of one consumer launch, as an index space i in [0, units): all units (L == 0, i = u), or, for
// a batch of equal-length sequences of `per` chunks each, chunks lo .. lo+L-1 of every sequence
// (i runs over sequence, then chunk, then head). A CTA takes index blockIdx.x first; later indices
// come from the launch's counter (zeroed before the launch) or, without one, in strides of gridDim.
// The joint schedule (pc.flags set) runs every unit, latest chunk first (the order in which the
// reverse scans finish them): index i is chunk per-1-i/(N H) of sequence (i mod N H) / H, head i mod H;
// every index comes from the launch's counter.
__device__ __forceinline__ int piece_units(const ConsPiece& pc, int N, int H, int total) {
    return pc.flags ? total : pc.L ? N * pc.L * H : total;
}
__device__ __forceinline__ int piece_unit(const ConsPiece& pc, int i, int N, int H) {
    if (pc.flags) {
        const int NH = N * H, r = i / NH, p = i - r * NH;
        return ((p / H) * pc.per + pc.per - 1 - r) * H + p % H;
    }
    if (!pc.L) return i;
    const int LH = pc.L * H, n = i / LH, r = i - n * LH;
    return (n * pc.per + pc.lo + r / H) * H + r % H;
}
__device__ __forceinline__ int claim_next(const ConsPiece& pc, int i) {
    if (pc.flags) return atomicAdd(pc.ctr, 1);
    return pc.ctr ? (int)gridDim.x + atomicAdd(pc.ctr, 1) : i + (int)gridDim.x;
}

// The first unit at index i or after it (claiming further indices) that has tokens and a narrow
// gate range (-1 when none is left); i ends at that unit's index, n and tok0 give its chunk extent.
template <int GATE>
__device__ __forceinline__ int cons_find(int& i, int units, const ConsPiece& pc, int N, int H, const Table& t,
                                         const FwdTC& f, int& n, int& tok0) {
    for (; i < units; i = claim_next(pc, i)) {
        const int u = piece_unit(pc, i, N, H), c = u / H;
        n = t.chunk_len[c];
        if (n > 0 && (GATE == 0 || f.WIDE[u] == 0)) {
            tok0 = t.chunk_tok0[c];
            return u;
        }
    }
    n = 0;
    tok0 = 0;
    return -1;
}

// Load group C of unit ch from tok0: k, q of head hq by TMA in SW128 rows, and the prep's alpha
// as it is: per-channel gate, fp32 token rows into the alpha tile and its 2^c, 2^(G2_last - c)
// rows into theirs; scalar gate, the BT alphas and two constants into the staging region.
template <int GATE>
__device__ __forceinline__ void cons_load_c(uint32_t sb, const CUtensorMap* tmk, const CUtensorMap* tmq,
                                            const FwdTC& f, size_t ch, int hq, int tok0, uint64_t* b) {
    tc::mbar_arrive_expect_tx(b, 2 * BT * D * 2 + (GATE == 2 ? 4 * ALK_UNIT : GATE == 1 ? 4 * ALK_SCALAR : 0));
    tc::tma_load3(sb + C_K, tmk, 0, hq, tok0, b);
    tc::tma_load3(sb + C_K + 8192, tmk, 64, hq, tok0, b);
    tc::tma_load3(sb + C_Q, tmq, 0, hq, tok0, b);
    tc::tma_load3(sb + C_Q + 8192, tmq, 64, hq, tok0, b);
    if (GATE == 2) {
        const float* img = f.ALK + ch * ALK_UNIT;
        tc::bulk_g2s(sb + C_A, img, 4 * BT * D, b);
        tc::bulk_g2s(sb + C_MISC + 4 * M_C2, img + BT * D, 4 * 2 * D, b);
    } else if (GATE == 1) {
        tc::bulk_g2s(sb + X_STG, f.ALK + ch * ALK_SCALAR, 4 * ALK_SCALAR, b);
    }
}

// Load group X1 of unit ch: R in rows 0..63 and S in rows 64..191 of each atom column of the
// [R ; S] tile, S+bar as it is (tile images, one bulk copy per piece).
__device__ __forceinline__ void cons_load_x1(uint32_t sb, const FwdTC& f, const BwdTC& bw, size_t ch, uint64_t* b) {
    tc::mbar_arrive_expect_tx(b, BT * D * 2 + 2 * D * D * 2);
    const unsigned char* R0 = reinterpret_cast<const unsigned char*>(f.R + ch * BT * D);
    const unsigned char* S0 = reinterpret_cast<const unsigned char*>(f.HS + ch * D * D);
    tc::bulk_g2s(sb + X_RS, R0, 8192, b);
    tc::bulk_g2s(sb + X_RS + 24576, R0 + 8192, 8192, b);
    tc::bulk_g2s(sb + X_RS + 8192, S0, 16384, b);
    tc::bulk_g2s(sb + X_RS + 24576 + 8192, S0 + 16384, 16384, b);
    tc::bulk_g2s(sb + X_SB, bw.SBP + ch * D * D, 32768, b);
}

// Load group X2 of unit (ch, h, tok0): dO (TMA) in rows 0..63 and P (tile image) in rows
// 64..127 of each atom column of the [dO ; P] tile; v by TMA in SW128 rows. Rows past the
// chunk end hold the following tokens (or zeros past the tensor); every use masks them or
// only reaches rows that are never stored.
__device__ __forceinline__ void cons_load_x2(uint32_t sb, const CUtensorMap* tmo, const CUtensorMap* tmv,
                                             const BwdTC& bw, size_t ch, int h, int tok0, uint64_t* b) {
    tc::mbar_arrive_expect_tx(b, 3 * BT * D * 2);
    const unsigned char* P0 = reinterpret_cast<const unsigned char*>(bw.P + ch * BT * D);
    tc::bulk_g2s(sb + X_OP + 8192, P0, 8192, b);
    tc::bulk_g2s(sb + X_OP + 16384 + 8192, P0 + 8192, 8192, b);
    tc::tma_load3(sb + X_OP, tmo, 0, h, tok0, b);
    tc::tma_load3(sb + X_OP + 16384, tmo, 64, h, tok0, b);
    tc::tma_load3(sb + X_V, tmv, 0, h, tok0, b);
    tc::tma_load3(sb + X_V + 8192, tmv, 64, h, tok0, b);
}

// Waits for one load group (parity = groups already waited, counted by every thread) and
// meets the CTA; false (and the device error bit) when any thread's wait ran out.
__device__ __forceinline__ bool cons_wait(uint64_t* b, int& w, int32_t* err) {
    const bool r = tc::mbar_wait(b, w & 1);
    if (r) ++w;
    const bool ok = __syncthreads_and(r) != 0;
    if (!ok && threadIdx.x == 0) atomicOr(err, 2);
    return ok;
}

// The consumer loop of one CTA (CT threads): units from the launch's index space until none is left.
// tb: 512 TMEM columns allocated by the caller. In the joint schedule the X tiles of a unit are loaded
// once its ready flag is set.
// FX (what the addressing takes at run time, the rest folded in by the compiler): 0 = nothing, the
// token rows D wide and one head of every input per value head; 1 = value head h reads q, k of
// head h / Gq and g, beta, erase of head h / Gg; 2 = that, and token rows K and V wide (multiples
// of 8, at most D).
template <int GATE, bool GD2, int FX>
__device__ __forceinline__ void cons_body(const Shape& s, const CUtensorMap* tmq_, const CUtensorMap* tmk_,
                                          const CUtensorMap* tmo_, const CUtensorMap* tmv_,
                                          const bf16* __restrict__ beta, const Table& t,
                                          const FwdTC& f, const BwdTC& bw, bf16* __restrict__ dq,
                                          bf16* __restrict__ dk, bf16* __restrict__ dv, bf16* __restrict__ dbeta,
                                          float* __restrict__ dg, const Gdn2& gd, const ConsPiece& pc,
                                          unsigned char* base, uint32_t tb) {
    const CUtensorMap &tmq = *tmq_, &tmk = *tmk_, &tmo = *tmo_, &tmv = *tmv_;
    const int Kw = FX == 2 ? s.K : D, Vw = FX == 2 ? s.V : D;   // row widths of the key- and value-side tensors
    const int Hg = FX ? s.Hg : s.H;                               // heads of the g, beta and erase rows
    float* sA = reinterpret_cast<float*>(base + C_A);
    const unsigned char* sK = base + C_K;
    const unsigned char* sQ = base + C_Q;
    bf16* sKm = reinterpret_cast<bf16*>(base + C_K);   // the same tiles, key-major after the alpha pass
    bf16* sQm = reinterpret_cast<bf16*>(base + C_Q);
    float* sm = reinterpret_cast<float*>(base + C_MISC);
    float* sBeta = sm + M_BETA;
    float* sC2 = sm + M_C2;       // 2^c per feature
    float* sAL = sm + M_AL;       // 2^(G2_last - c) per feature
    float* sLamP = sm + M_LAMP;   // [4][128] partial rowsum(S .* S+bar) per key
    float* sDbw = sm + M_DBW;     // <v_i, P_i>
    float* sRowP = sm + M_ROWP;   // [4][64] partial <k_j, gamma E_bar_j> per lane quarter
    float* sEndP = sm + M_ENDP;   // [4][128] partial sum_j F_j . F_bar_j per token group
    float* sRowG = sm + M_ROWG;   // [4][64] scalar gate: partial row sums of G_bar per lane quarter
    float* sSeg = sm + M_SEG;     // [4][128] per-channel gate: G_bar summed over each token group
    float* sEndQ = sm + M_ENDQ;   // [4] scalar gate: endpoint terms summed per lane quarter
    int* sMeta = reinterpret_cast<int*>(sm + M_META);             // two slots {unit, n, tok0, -}
    uint64_t* bar = reinterpret_cast<uint64_t*>(base + C_BAR);    // MMA completions
    uint64_t* bldC = bar + 1;                                     // load groups C, X1, X2
    uint64_t* bldX1 = bar + 2;
    uint64_t* bldX2 = bar + 3;
    const uint32_t sb = tc::smem_u32(base);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, grp = warp >> 2;
    const int H = s.H, units = piece_units(pc, s.N, s.H, s.NC * s.H);
    const float scale = s.scale;
    int icur = (int)blockIdx.x, icand = units;   // indices of the current unit and the candidate (thread LDR)
    const int N = s.N;
    int nC = 0, nX1 = 0, nX2 = 0;   // load groups issued (thread LDR)
    int wC = 0, wX1 = 0, wX2 = 0;   // load groups waited for (every thread)
    // this thread's key (TMEM lane) and token group in the key-major passes, and the key's byte
    // offsets in the k / q tiles
    const int kr = 32 * quad + lane, jb = 16 * grp;
    const uint32_t kcol = (uint32_t)((kr >> 6) * BT * 128 + (kr & 7) * 2);
    const int kch = (kr >> 3) & 7;
    bf16* stg = reinterpret_cast<bf16*>(base + X_STG + warp * 512);

    if (tid == LDR) {
        for (int i = 0; i < 4; ++i) tc::mbar_init(&bar[i], 1);
        tc::fence_mbar_init();
        if (pc.flags) icur = atomicAdd(pc.ctr, 1);
        int n0 = 0, t0 = 0;
        const int u0 = cons_find<GATE>(icur, units, pc, N, H, t, f, n0, t0);
        sMeta[0] = u0;
        sMeta[1] = n0;
        sMeta[2] = t0;
        if (u0 >= 0) {
            const int h0 = u0 % H;
            cons_load_c<GATE>(sb, &tmk, &tmq, f, (size_t)u0, FX ? h0 / s.Gq : h0, t0, bldC);
            if (pc.flags && !tc::wait_flag(pc.flags + u0, t.err)) atomicOr(t.err, 2);
            cons_load_x1(sb, f, bw, (size_t)u0, bldX1);
            cons_load_x2(sb, &tmo, &tmv, bw, (size_t)u0, h0, t0, bldX2);
            nC = nX1 = nX2 = 1;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tl = tc::taddr(tb, 32 * quad, 0);
    bf16 beta_nx = __float2bfloat16_rn(0.f);   // beta of the next unit (threads < BT), read during this one
    int cand = 0, cn = 0, ct0 = 0, cw = 0;   // next-unit candidate and its table entries (thread LDR)

    for (int k = 0;; ++k) {
        const int* meta = sMeta + 4 * (k & 1);
        const int u = meta[0];
        if (u < 0) break;
        const int n = meta[1], tok0 = meta[2];
        const int c = u / H, h = u - c * H;
        const int* nm = sMeta + 4 * ((k + 1) & 1);   // the next unit, settled below by thread LDR
        if (tid == LDR) {   // the next candidate and its table entries
            icand = claim_next(pc, icur);
            if (icand < units) {
                cand = piece_unit(pc, icand, N, H);
                cn = __ldg(t.chunk_len + cand / H);
                ct0 = __ldg(t.chunk_tok0 + cand / H);
                cw = (GATE != 0) ? __ldg(f.WIDE + cand) : 0;
            }
        }
        const float beta_r =
            (k == 0) ? ((tid < BT && tid < n && !GD2) ? bfx(beta + (size_t)(tok0 + tid) * Hg + (FX ? h / s.Gg : h)) : 0.f)
                     : __bfloat162float(beta_nx);
        if (tid < BT) sBeta[tid] = beta_r;
        // groups X1 and X2: [R ; S], S+bar, [dO ; P], v
        {
            const bool r1 = tc::mbar_wait(bldX1, wX1 & 1);
            const bool r2 = tc::mbar_wait(bldX2, wX2 & 1);
            wX1 += r1;
            wX2 += r2;
            if (!__syncthreads_and(r1 && r2)) {
                if (tid == 0) atomicOr(t.err, 2);
                break;
            }
        }
        if (warp == 0) {
            tc::fence_after_sync();
            // phase A (warp-uniform descriptors, one elected lane issuing); it needs only the X
            // tiles, so it runs under the rowsum, dv and alpha passes:
            //   [dO ; P] R^T -> [H_q ; -D] (token rows), S [dO ; P]^T -> [S dO^T | S P^T] and
            //   S+bar R^T -> F_bar^T (key rows); S is rows 64..191 of the [R ; S] tile
            const uint32_t i64 = tc::idesc_bf16(128, 64), i128 = tc::idesc_bf16(128, 128);
            const uint64_t dOP = tc::sdesc(sb + X_OP), dRS = tc::sdesc(sb + X_RS), dSB = tc::sdesc(sb + X_SB);
            const uint64_t dS = tc::sdesc(sb + X_RS + BT * 128);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16_w(tb + T_HD, tc::kstep_k(dOP, D, ks), tc::kstep_k(dRS, BT + D, ks), i64, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16_w(tb + T_SDO, tc::kstep_k(dS, BT + D, ks), tc::kstep_k(dOP, D, ks), i128, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16_w(tb + T_FB, tc::kstep_k(dSB, D, ks), tc::kstep_k(dRS, BT + D, ks), i64, ks > 0);
            tc::mma_commit_w(bar);
        }
        // the next unit: the candidate, else a walk over the table; every thread sees it after the
        // wait for group C below
        if (tid == LDR) {
            int nxt = -1, nn = 0, nt = 0;
            if (icand < units && cn > 0 && cw == 0) {
                nxt = cand;
                nn = cn;
                nt = ct0;
                icur = icand;
            } else if (icand < units) {
                icur = claim_next(pc, icand);
                nxt = cons_find<GATE>(icur, units, pc, N, H, t, f, nn, nt);
            }
            int* wm = sMeta + 4 * ((k + 1) & 1);
            wm[0] = nxt;
            wm[1] = nn;
            wm[2] = nt;
        }
        // rowsum(S .* S+bar) (key kq, a quarter of the values per thread), <v_i, P_i> and
        // dv = beta P from the staged tiles, while group C lands
        {
            const int kq = tid & (D - 1), q4 = tid >> 7;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int cc = 4 * q4; cc < 4 * q4 + 4; ++cc) {
                const uint4 a = *reinterpret_cast<const uint4*>(base + X_RS + tc::sw128_off(BT + D, BT + kq, cc * 16));
                const uint4 bb = *reinterpret_cast<const uint4*>(base + X_SB + tc::sw128_off(D, kq, cc * 16));
                const bf16* pa = reinterpret_cast<const bf16*>(&a);
                const bf16* pb = reinterpret_cast<const bf16*>(&bb);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    a0 = fmaf(__bfloat162float(pa[e]), __bfloat162float(pb[e]), a0);
                    a1 = fmaf(__bfloat162float(pa[e + 1]), __bfloat162float(pb[e + 1]), a1);
                }
            }
            sLamP[q4 * D + kq] = a0 + a1;
        }
#pragma unroll
        for (int uu = 0; uu < BT * 16 / CT; ++uu) {   // 16 threads per row, 8 values each
            const int idx = tid + CT * uu, r = idx >> 4, cc = idx & 15;
            float acc = 0.f;
            if (r < n && cc * 8 < Vw) {
                const size_t tok = (size_t)(tok0 + r) * H + h;   // value rows of width V
                const float bt = sBeta[r];
                const uint4 pp = *reinterpret_cast<const uint4*>(base + X_OP + tc::sw128_off(2 * BT, BT + r, cc * 16));
                const uint4 vv = *reinterpret_cast<const uint4*>(base + X_V + tc::sw128_off(BT, r, cc * 16));
                const bf16* pp2 = reinterpret_cast<const bf16*>(&pp);
                const bf16* vv2 = reinterpret_cast<const bf16*>(&vv);
                uint32_t out[4], wout[4];
                if (GD2) {   // GatedDeltaNet-2: dv = w .* P, dw = v .* P
                    const uint4 ww = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(gd.write) + tok * Vw + cc * 8);
                    const bf16* ww2 = reinterpret_cast<const bf16*>(&ww);
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float p0 = __bfloat162float(pp2[e]), p1 = __bfloat162float(pp2[e + 1]);
                        out[e / 2] = tc::pack_bf16(__bfloat162float(ww2[e]) * p0, __bfloat162float(ww2[e + 1]) * p1);
                        wout[e / 2] = tc::pack_bf16(__bfloat162float(vv2[e]) * p0, __bfloat162float(vv2[e + 1]) * p1);
                    }
                    *reinterpret_cast<uint4*>(static_cast<bf16*>(gd.dwrite) + tok * Vw + cc * 8) =
                        make_uint4(wout[0], wout[1], wout[2], wout[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float p0 = __bfloat162float(pp2[e]), p1 = __bfloat162float(pp2[e + 1]);
                        acc = fmaf(__bfloat162float(vv2[e]), p0, acc);
                        acc = fmaf(__bfloat162float(vv2[e + 1]), p1, acc);
                        out[e / 2] = tc::pack_bf16(bt * p0, bt * p1);
                    }
                }
                *reinterpret_cast<uint4*>(dv + tok * Vw + cc * 8) = make_uint4(out[0], out[1], out[2], out[3]);
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, 16);
            if (cc == 0) sDbw[r] = acc;
        }
        if (!cons_wait(bldC, wC, t.err)) break;
        // the next unit's beta, kept as bf16 in a register so that the load stays in flight until
        // that unit starts; GatedDeltaNet-2: its erase and write rows (two 128-byte lines each)
        // into L2, so that its direct loads of them find them there
        if (nm[0] >= 0) {
            const int nh = nm[0] % H, nhg = FX ? nh / s.Gg : nh;
            if (tid < BT)
                beta_nx = (tid < nm[1] && !GD2) ? beta[(size_t)(nm[2] + tid) * Hg + nhg] : __float2bfloat16_rn(0.f);
            if (GD2 && (tid >> 2) < nm[1]) {
                const bool wr = (tid & 2) != 0;
                const int w = wr ? Vw : Kw;   // the row widths of the write and erase vectors
                const bf16* vec = static_cast<const bf16*>(wr ? gd.write : gd.erase);
                const size_t row = (size_t)(nm[2] + (tid >> 2)) * (wr ? H : Hg) + (wr ? nh : nhg);
                if ((tid & 1) * 64 < w) tc::prefetch_l2(vec + row * w + (tid & 1) * 64);
            }
        }
        // alpha of this thread's key kr and rows jb .. jb+15 (the same key and tokens it handles in
        // every later pass): the prep's (per-channel gate: token rows in the alpha tile; scalar gate:
        // one per token in the staging region), or 1 without a gate. alpha, k and q are then
        // rewritten key-major over their own tiles.
        {
            uint32_t kk[8], qq[8];   // k and q of this key for the 16 rows, bf16 pairs
#pragma unroll
            for (int r = 0; r < 16; r += 2) {
                const uint32_t o0 = swrow(kcol, kch, jb + r), o1 = swrow(kcol, kch, jb + r + 1);
                kk[r / 2] = (uint32_t)*reinterpret_cast<const uint16_t*>(sK + o0) |
                            ((uint32_t)*reinterpret_cast<const uint16_t*>(sK + o1) << 16);
                qq[r / 2] = (uint32_t)*reinterpret_cast<const uint16_t*>(sQ + o0) |
                            ((uint32_t)*reinterpret_cast<const uint16_t*>(sQ + o1) << 16);
            }
            const float* sAs = reinterpret_cast<const float*>(base + X_STG);   // scalar gate: [BT] alpha, 2^c, 2^(G2_last - c)
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = GATE == 2 ? sA[(jb + r) * D + kr] : GATE == 1 ? sAs[jb + r] : 1.f;
            if (GATE != 2 && grp == 0) {
                sC2[kr] = GATE == 1 ? sAs[BT] : 1.f;
                sAL[kr] = GATE == 1 ? sAs[BT + 1] : 1.f;
            }
            __syncthreads();   // (also: every alpha, k, q read before the key-major tiles overwrite them)
#pragma unroll
            for (int m = 0; m < 4; ++m)
                *reinterpret_cast<float4*>(sA + akm4(kr, 4 * grp + m)) =
                    make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) {
                *reinterpret_cast<uint4*>(sKm + kkm8(kr, 2 * grp + b2)) =
                    make_uint4(kk[4 * b2], kk[4 * b2 + 1], kk[4 * b2 + 2], kk[4 * b2 + 3]);
                *reinterpret_cast<uint4*>(sQm + kkm8(kr, 2 * grp + b2)) =
                    make_uint4(qq[4 * b2], qq[4 * b2 + 1], qq[4 * b2 + 2], qq[4 * b2 + 3]);
            }
        }
        // (K zeta)^T into TMEM (the A operand of [T_e ; T_q]^T; this thread's key and 16 tokens,
        // zero past the chunk end; zeta = 1/alpha, unit without a per-channel gate)
        {
            float al[16], kz[16];
            uint32_t kw[8];
            ld_alpha16(sA, kr, grp, al);
            ld_bf16x16(sKm, kr, grp, kw);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float kv = bf_lo_hi(kw[e >> 1], e & 1);
                kz[e] = (jb + e < n) ? ((GATE == 2) ? kv * tc::rcp_approx(al[e]) : kv) : 0.f;
            }
            tc::tmem_st16(tl + T_KZ + jb, kz);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        if (!wait_all(bar, 0, t.err)) break;   // phase A done; every key-major tile written
        tc::fence_after_sync();
        // ---- epilogue A: mask [H_q ; -D] into [H_q ; D] (scalar gate: fold the pairwise decay
        // alpha_i / alpha_j) and write it twice as tf32 operands: [D ; H_q] (rows i', K = token j,
        // the B operand of [T_e ; T_q]^T) and its transpose (the B operand of T_y^T)
        {
            const int row = 32 * quad + lane, cb0 = grp * 16;
            float a[16];
            tc::tmem_ld16(tc::taddr(tb + T_HD, 32 * quad, cb0), a);
            tc::tmem_wait_ld();
            const bool isH = row < BT;
            const int i = isH ? row : row - BT;
            const int kidx = isH ? BT + i : i;   // row of [D ; H_q]: D rows first, then H_q rows
            const float ai = (GATE == 1) ? sA[akm4(0, i >> 2) + (i & 3)] : 1.f;   // the gate is one per token
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int j = cb0 + jj;
                float x = (i < n && (isH ? j <= i : j < i)) ? (isH ? a[jj] : -a[jj]) : 0.f;
                if (GATE == 1) x *= fminf(ai * tc::rcp_approx(sA[akm4(0, j >> 2) + (j & 3)]), 1.f);
                a[jj] = x;
                *reinterpret_cast<float*>(base + X_DH + tc::sw128_off(BT, j, kidx * 4)) = x;
            }
#pragma unroll
            for (int m = 0; m < 4; ++m)
                *reinterpret_cast<float4*>(base + X_BT + tc::sw128_off(2 * BT, kidx, (cb0 + 4 * m) * 4)) =
                    make_float4(a[4 * m], a[4 * m + 1], a[4 * m + 2], a[4 * m + 3]);
        }
        // [E_alpha^T | Q_alpha^T] (rows = key kr, K = token: E part, then Q part): this thread's key
        // and 16 tokens, four at a time; rows past the chunk end are zero
        {
            float al[16];
            uint32_t kw[8], qw[8];
            ld_alpha16(sA, kr, grp, al);
            ld_bf16x16(sKm, kr, grp, kw);
            ld_bf16x16(sQm, kr, grp, qw);
#pragma unroll
            for (int uq = 0; uq < 4; ++uq) {
                float ea[4], qa[4];
                const float4 b4 = *reinterpret_cast<const float4*>(sBeta + jb + 4 * uq);
                const float bq[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int q16 = 4 * uq + e, j = jb + q16;
                    const float kv = bf_lo_hi(kw[q16 >> 1], q16 & 1);
                    const float qv = bf_lo_hi(qw[q16 >> 1], q16 & 1);
                    const float av = (GATE == 2) ? al[q16] : 1.f;
                    const bool in = j < n;
                    const float eb = GD2 ? ((in && kr < Kw) ? bfx(static_cast<const bf16*>(gd.erase) +
                                                                   ((size_t)(tok0 + j) * Hg + (FX ? h / s.Gg : h)) * Kw + kr) : 0.f)
                                         : bq[e];
                    ea[e] = in ? eb * kv * av : 0.f;
                    qa[e] = in ? scale * qv * av : 0.f;
                }
                *reinterpret_cast<float4*>(base + X_EQ + tc::sw128_off(D, kr, (jb + 4 * uq) * 4)) =
                    make_float4(ea[0], ea[1], ea[2], ea[3]);
                *reinterpret_cast<float4*>(base + X_EQ + tc::sw128_off(D, kr, (BT + jb + 4 * uq) * 4)) =
                    make_float4(qa[0], qa[1], qa[2], qa[3]);
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) {
            tc::fence_after_sync();
            // phase B (tf32): [T_e ; T_q]^T = (K zeta)^T [D ; H_q]^T (A from TMEM) and
            // T_y^T = [E_alpha^T | Q_alpha^T] [D ; H_q]
            const uint32_t i128 = tc::idesc_tf32(128, 128), i64 = tc::idesc_tf32(128, 64);
            const uint64_t dBT = tc::sdesc(sb + X_BT), dEQ = tc::sdesc(sb + X_EQ), dDH = tc::sdesc(sb + X_DH);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_tf32_ts_w(tb + T_TE, tb + T_KZ + 8 * ks, tc::kstep_k(dBT, 2 * BT, ks), i128, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 16; ++ks)
                tc::mma_tf32_w(tb + T_Y, tc::kstep_k(dEQ, D, ks), tc::kstep_k(dDH, BT, ks), i64, ks > 0);
            tc::mma_commit_w(bar);
        }
        if (!wait_all(bar, 1, t.err)) break;
        tc::fence_after_sync();
        // groups X1 and X2 of the next unit into the X region, free since the phase-B MMAs completed
        if (tid == LDR && nm[0] >= 0) {
            if (pc.flags && !tc::wait_flag(pc.flags + nm[0], t.err)) atomicOr(t.err, 2);
            cons_load_x1(sb, f, bw, (size_t)nm[0], bldX1);
            cons_load_x2(sb, &tmo, &tmv, bw, (size_t)nm[0], nm[0] % H, nm[2], bldX2);
            ++nX1;
            ++nX2;
        }
        // ---- key-major epilogue: key kr, tokens jb .. jb+15 in two halves of 8, later half first
        // (the reverse cumsum runs inside the thread). With gamma = alpha 2^c:
        //   gamma Q_g_bar = fac T_q + gamma (dO S^T),  dq = s gamma Q_g_bar
        //   gamma E_bar   = fac T_e - gamma (P S^T),   dk = beta gamma E_bar + Y_bar / gamma
        //   Y_bar / gamma = zeta T_y + (lambda / gamma) F_bar
        //   G_bar = s q gamma Q_g_bar + beta k gamma E_bar - k Y_bar / gamma
        // (fac = alpha, zeta = 1 / alpha for a per-channel gate; unit otherwise)
        const float c2k = sC2[kr], alk = sAL[kr];
        float gx[16];   // per-channel gate: in-group suffix sums of G_bar
        float run = 0.f, endp = 0.f;
#pragma unroll
        for (int h2 = 1; h2 >= 0; --h2) {
            const int j0 = jb + 8 * h2;
            const int nrow = min(max(n - j0, 0), 8);
            float kvs[8], als[8], dkv[8], gb[8];
            {
                float te[8], tq[8], tdo[8], tps[8], dqv[8], dbp[8];
                tc::tmem_ld8(tl + T_TE + j0, te);
                tc::tmem_ld8(tl + T_TQ + j0, tq);
                tc::tmem_ld8(tl + T_SDO + j0, tdo);
                tc::tmem_ld8(tl + T_SP + j0, tps);
                const uint4 k8 = *reinterpret_cast<const uint4*>(sKm + kkm8(kr, 2 * grp + h2));
                const uint4 q8 = *reinterpret_cast<const uint4*>(sQm + kkm8(kr, 2 * grp + h2));
                const float4 a0 = *reinterpret_cast<const float4*>(sA + akm4(kr, 4 * grp + 2 * h2));
                const float4 a1 = *reinterpret_cast<const float4*>(sA + akm4(kr, 4 * grp + 2 * h2 + 1));
                const float4 b0 = *reinterpret_cast<const float4*>(sBeta + j0);
                const float4 b1 = *reinterpret_cast<const float4*>(sBeta + j0 + 4);
                const uint32_t kw[4] = {k8.x, k8.y, k8.z, k8.w}, qw[4] = {q8.x, q8.y, q8.z, q8.w};
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                tc::tmem_wait_ld();
                // pairs of tokens in packed fp32x2 arithmetic
                const float2 s2 = make_float2(scale, scale), c22 = make_float2(c2k, c2k), nc22 = make_float2(-c2k, -c2k);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const int j = j0 + e;
                    const float2 kv2 = make_float2(bf_lo_hi(kw[e >> 1], 0), bf_lo_hi(kw[e >> 1], 1));
                    const float2 qv2 = make_float2(bf_lo_hi(qw[e >> 1], 0), bf_lo_hi(qw[e >> 1], 1));
                    const float2 al2 = make_float2(av[e], av[e + 1]);
                    const float2 fac2 = (GATE == 2) ? al2 : make_float2(1.f, 1.f);
                    const float2 gam2 = __fmul2_rn(al2, c22);
                    const float2 Qt2 = __ffma2_rn(fac2, make_float2(tq[e], tq[e + 1]),
                                                  __fmul2_rn(gam2, make_float2(tdo[e], tdo[e + 1])));
                    const float2 Et2 = __ffma2_rn(fac2, make_float2(te[e], te[e + 1]),
                                                  __fmul2_rn(__fmul2_rn(al2, nc22), make_float2(tps[e], tps[e + 1])));
                    float2 be2;
                    if (GD2) {
                        const bf16* er = static_cast<const bf16*>(gd.erase) + ((size_t)(tok0 + j) * Hg + (FX ? h / s.Gg : h)) * Kw + kr;
                        const bool kin = kr < Kw;   // erase rows of width K
                        be2 = make_float2((kin && j < n) ? bfx(er) : 0.f, (kin && j + 1 < n) ? bfx(er + (size_t)Hg * Kw) : 0.f);
                    } else {
                        be2 = make_float2(bv[e], bv[e + 1]);
                    }
                    const float2 dq2 = __fmul2_rn(s2, Qt2), dk2 = __fmul2_rn(be2, Et2), db2 = __fmul2_rn(kv2, Et2);
                    const float2 gb2 = __ffma2_rn(__fmul2_rn(s2, qv2), Qt2, __fmul2_rn(be2, db2));
                    dqv[e] = dq2.x;
                    dqv[e + 1] = dq2.y;
                    dkv[e] = dk2.x;
                    dkv[e + 1] = dk2.y;
                    dbp[e] = db2.x;   // <k_j, gamma E_bar_j> term; GatedDeltaNet-2: d erase
                    dbp[e + 1] = db2.y;
                    gb[e] = gb2.x;
                    gb[e + 1] = gb2.y;
                    kvs[e] = kv2.x;
                    kvs[e + 1] = kv2.y;
                    als[e] = al2.x;
                    als[e + 1] = al2.y;
                }
                // key rows of width K: this warp's 32 keys from 32 quad, wk of them present
                const size_t row0 = ((size_t)(tok0 + j0) * H + h) * Kw + 32 * quad;
                const int wk = Kw - 32 * quad;
                if (wk > 0) tc::warp_store_t8(stg, dqv, dq + row0, (size_t)H * Kw, nrow, lane, wk);
                if (GD2) {
                    if (wk > 0)
                        tc::warp_store_t8(stg, dbp, static_cast<bf16*>(gd.derase) + row0, (size_t)H * Kw, nrow, lane, wk);
                } else {
                    const float tot = tc::warp_sum8_spread(dbp, lane);
                    if ((lane & 3) == 0) sRowP[quad * BT + j0 + (lane >> 2)] = tot;
                }
            }
            {
                float ty[8], fb[8];
                tc::tmem_ld8(tl + T_Y + j0, ty);
                tc::tmem_ld8(tl + T_FB + j0, fb);
                tc::tmem_wait_ld();
                const float2 alk2 = make_float2(alk, alk);
                float2 ep2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 rinv2 = make_float2(tc::rcp_approx(als[e]), tc::rcp_approx(als[e + 1]));
                    const float2 ze2 = (GATE == 2) ? rinv2 : make_float2(1.f, 1.f);
                    const float2 dec2 = __fmul2_rn(alk2, rinv2);              // lambda / gamma_j
                    const float2 fb2 = make_float2(fb[e], fb[e + 1]);
                    const float2 Yt2 = __ffma2_rn(ze2, make_float2(ty[e], ty[e + 1]), __fmul2_rn(fb2, dec2));   // Y_bar / gamma
                    const float2 nkv2 = make_float2(-kvs[e], -kvs[e + 1]);
                    const float2 dk2 = __fadd2_rn(make_float2(dkv[e], dkv[e + 1]), Yt2);
                    const float2 gb2 = __ffma2_rn(nkv2, Yt2, make_float2(gb[e], gb[e + 1]));
                    // F_j . F_bar_j, tokens past the chunk end left out
                    const float2 fm = make_float2((j0 + e < n) ? kvs[e] : 0.f, (j0 + e + 1 < n) ? kvs[e + 1] : 0.f);
                    ep2 = __ffma2_rn(__fmul2_rn(fm, dec2), fb2, ep2);
                    dkv[e] = dk2.x;
                    dkv[e + 1] = dk2.y;
                    gb[e] = gb2.x;
                    gb[e + 1] = gb2.y;
                }
                endp += ep2.x + ep2.y;
            }
            if (Kw > 32 * quad)
                tc::warp_store_t8(stg, dkv, dk + ((size_t)(tok0 + j0) * H + h) * Kw + 32 * quad, (size_t)H * Kw, nrow,
                                  lane, Kw - 32 * quad);
            if (GATE == 2) {
#pragma unroll
                for (int e = 7; e >= 0; --e) {
                    run += (j0 + e < n) ? gb[e] : 0.f;
                    gx[8 * h2 + e] = run;
                }
            } else if (GATE == 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) gb[e] = (j0 + e < n) ? gb[e] : 0.f;
                const float tot = tc::warp_sum8_spread(gb, lane);
                if ((lane & 3) == 0) sRowG[quad * BT + j0 + (lane >> 2)] = tot;
            }
        }
        if (GATE != 0) {
            sEndP[grp * D + kr] = endp;
            if (GATE == 2) sSeg[grp * D + kr] = run;
        }
        // every read of k, q, alpha and beta is done: group C of the next unit may land
        tc::fence_async_smem();   // the key-major tiles' generic writes before the next tiles land by TMA
        tc::fence_before_sync();
        __syncthreads();
        if (tid == LDR && nm[0] >= 0) {
            const int nh = nm[0] % H;
            cons_load_c<GATE>(sb, &tmk, &tmq, f, (size_t)nm[0], FX ? nh / s.Gq : nh, nm[2], bldC);
            ++nC;
        }
        if (!GD2 && tid < BT && tid < n)
            dbeta[(size_t)(tok0 + tid) * H + h] = __float2bfloat16_rn(sRowP[tid] + sRowP[BT + tid] + sRowP[2 * BT + tid] +
                                                                      sRowP[3 * BT + tid] + sDbw[tid]);
        if (GATE == 2) {
            // the endpoint terms of the last row (lambda rowsum(S .* S+bar) + sum_j F_j . F_bar_j) reach
            // every earlier row through the reverse cumsum, as do the later token groups' totals
            float off = alk * c2k * (sLamP[kr] + sLamP[D + kr] + sLamP[2 * D + kr] + sLamP[3 * D + kr]) +
                        sEndP[kr] + sEndP[D + kr] + sEndP[2 * D + kr] + sEndP[3 * D + kr];
#pragma unroll
            for (int g2 = 1; g2 < 4; ++g2)
                if (g2 > grp) off += sSeg[g2 * D + kr];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = jb + e;
                if (j < n && kr < Kw) dg[((size_t)(tok0 + j) * H + h) * Kw + kr] = gx[e] + off;
            }
        } else if (GATE == 1) {
            // scalar gate: dg_j = sum over j' >= j of the feature sums of G_bar, plus the endpoint
            // terms summed over features
            if (warp < 4) {
                float e = alk * c2k * (sLamP[kr] + sLamP[D + kr] + sLamP[2 * D + kr] + sLamP[3 * D + kr]) +
                          sEndP[kr] + sEndP[D + kr] + sEndP[2 * D + kr] + sEndP[3 * D + kr];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
                if (lane == 0) sEndQ[quad] = e;
                tc::named_sync(1, 128);
                if (tid == 0) {
                    float acc = sEndQ[0] + sEndQ[1] + sEndQ[2] + sEndQ[3];
                    for (int r = n - 1; r >= 0; --r) {
                        acc += sRowG[r] + sRowG[BT + r] + sRowG[2 * BT + r] + sRowG[3 * BT + r];
                        dg[(size_t)(tok0 + r) * H + h] = acc;
                    }
                }
            }
        }
    }
    // a load still in flight (only after a timeout) lands before the CTA leaves
    if (tid == LDR) {
        for (; wC < nC; ++wC) tc::mbar_wait(bldC, wC & 1);
        for (; wX1 < nX1; ++wX1) tc::mbar_wait(bldX1, wX1 & 1);
        for (; wX2 < nX2; ++wX2) tc::mbar_wait(bldX2, wX2 & 1);
    }
}

template <int GATE, bool GD2, int FX>
__global__ void __launch_bounds__(CT, 1)
    k_bwd_consumer_tc(Shape s, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmo, const __grid_constant__ CUtensorMap tmv,
                      const bf16* __restrict__ beta,
                      Table t, FwdTC f, BwdTC bw, bf16* __restrict__ dq,
                      bf16* __restrict__ dk, bf16* __restrict__ dv, bf16* __restrict__ dbeta,
                      float* __restrict__ dg, Gdn2 gd, ConsPiece pc) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + C_BAR + 32);
    if (threadIdx.x < 32) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tb = *tslot;
    cons_body<GATE, GD2, FX>(s, &tmq, &tmk, &tmo, &tmv, beta, t, f, bw, dq, dk, dv, dbeta, dg, gd, pc, base, tb);
    tc::fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) tc::tmem_dealloc(tb, 512);
}

// The joint schedule in one cooperative launch of one CTA per SM: CTA n H + h (n < N) first runs the
// reverse scan of sequence n, head h, publishing each chunk as its S+bar and P reach HBM, then joins
// the other CTAs in the consumer loop, which takes the units latest chunk first and waits for each
// unit's flag before loading its scan outputs. No CTA waits for one that is not running: the launch
// is cooperative, so all of them are resident, and the scans never wait for the consumers.
template <int GATE, bool GD2, int FX>
__global__ void __launch_bounds__(CT, 1)
    k_bwd_joint_tc(Shape s, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmo, const __grid_constant__ CUtensorMap tmv,
                   const float* __restrict__ dht, float* __restrict__ dh0,
                   const bf16* __restrict__ beta, Table t, FwdTC f, BwdTC bw,
                   bf16* __restrict__ dq, bf16* __restrict__ dk, bf16* __restrict__ dv, bf16* __restrict__ dbeta,
                   float* __restrict__ dg, Gdn2 gd, ConsPiece pc) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + J_SLOT);
    if (threadIdx.x < 32) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tb = *tslot;
    if ((int)blockIdx.x < s.N * s.H) {
        bscan_body<FX == 2>(s, &tmo, dht, t, f, bw, dh0, t.seq_order[(int)blockIdx.x / s.H], (int)blockIdx.x % s.H, 0, 0,
                   pc.flags, base, tb);
        tc::fence_async_smem();   // the scan's shared-memory writes before the consumer's tile loads land
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    cons_body<GATE, GD2, FX>(s, &tmq, &tmk, &tmo, &tmv, beta, t, f, bw, dq, dk, dv, dbeta, dg, gd, pc, base, tb);
    tc::fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) tc::tmem_dealloc(tb, 512);
}

template <int GATE, bool GD2, int FX>
cudaError_t run_consumer(const Shape& s, const void* q, const void* k, const void* v, const void* beta,
                         const void* dout, Table t, FwdTC f, BwdTC b, void* dq, void* dk,
                         void* dv, void* dbeta, float* dg, cudaStream_t st, const Gdn2& gd, const ConsPiece& pc) {
    cudaError_t e = set_smem_once<k_bwd_consumer_tc<GATE, GD2, FX>>(CONS_SMEM);
    if (e != cudaSuccess) return e;
    CUtensorMap mq, mk, mo, mv;
    // the inputs at their own widths K, V (<= D): the boxes' columns past them read as zeros (q, k
    // with heads_q(s) heads; a per-channel gate reaches the consumer as the prep's alpha rows)
    if (!tmap_rows_bf16(&mq, q, s.Ttot, heads_q(s), s.K) || !tmap_rows_bf16(&mk, k, s.Ttot, heads_q(s), s.K) ||
        !tmap_rows_bf16(&mo, dout, s.Ttot, s.H, s.V) || !tmap_rows_bf16(&mv, v, s.Ttot, s.H, s.V))
        return cudaErrorInvalidValue;
    if (GATE != 0 && !f.ALK) return cudaErrorInvalidValue;
    const long units = pc.L ? (long)s.N * pc.L * s.H : (long)s.NC * s.H;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffL) return cudaErrorInvalidValue;
    const int grid = (int)(units < sm_count() ? units : sm_count());   // one CTA per SM, persistent
    k_bwd_consumer_tc<GATE, GD2, FX><<<grid, CT, CONS_SMEM, st>>>(s, mq, mk, mo, mv, (const bf16*)beta, t, f, b,
                                                         (bf16*)dq, (bf16*)dk, (bf16*)dv, (bf16*)dbeta, dg, gd, pc);
    return cudaGetLastError();
}

template <int GATE, bool GD2, int FX>
cudaError_t run_joint(const Shape& s, const void* q, const void* k, const void* v, const void* beta,
                      const void* dout, const float* dht, float* dh0, Table t, FwdTC f, BwdTC b, void* dq, void* dk,
                      void* dv, void* dbeta, float* dg, cudaStream_t st, const Gdn2& gd, const ConsPiece& pc) {
    cudaError_t e = set_smem_once<k_bwd_joint_tc<GATE, GD2, FX>>(JOINT_SMEM);
    if (e != cudaSuccess) return e;
    CUtensorMap mq, mk, mo, mv;
    // the inputs at their own widths K, V (<= D): the boxes' columns past them read as zeros (q, k
    // with heads_q(s) heads; a per-channel gate reaches the consumer as the prep's alpha rows)
    if (!tmap_rows_bf16(&mq, q, s.Ttot, heads_q(s), s.K) || !tmap_rows_bf16(&mk, k, s.Ttot, heads_q(s), s.K) ||
        !tmap_rows_bf16(&mo, dout, s.Ttot, s.H, s.V) || !tmap_rows_bf16(&mv, v, s.Ttot, s.H, s.V))
        return cudaErrorInvalidValue;
    if (GATE != 0 && !f.ALK) return cudaErrorInvalidValue;
    const int grid = sm_count();
    if (s.N * s.H > grid || !pc.flags || !pc.ctr) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CT);
    cfg.dynamicSmemBytes = JOINT_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: consumers may wait for scan CTAs
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_bwd_joint_tc<GATE, GD2, FX>, s, mq, mk, mo, mv, dht, dh0, (const bf16*)beta,
                              t, f, b, (bf16*)dq, (bf16*)dk, (bf16*)dv, (bf16*)dbeta, dg, gd, pc);
}

}  // namespace

cudaError_t launch_bwd_joint_tc(const Shape& s, int gate, const void* q, const void* k, const void* v,
                                const void* beta, const void* dout, const float* dht, float* dh0,
                                Table t, FwdTC f, BwdTC b, void* dq, void* dk, void* dv, void* dbeta, float* dg,
                                cudaStream_t st, const Gdn2& gd, const ConsPiece& pc) {
    // narrower inputs (and grouped heads with them), grouped heads at the tile width, or neither
    const int fx = (s.K != D || s.V != D) ? 2 : (s.Gq != 1 || s.Gg != 1) ? 1 : 0;
#define KDA_JOINT_FX(G, X, F) run_joint<G, X, F>(s, q, k, v, beta, dout, dht, dh0, t, f, b, dq, dk, dv, dbeta, dg, st, gd, pc)
#define KDA_JOINT(G, X) (fx == 2 ? KDA_JOINT_FX(G, X, 2) : fx == 1 ? KDA_JOINT_FX(G, X, 1) : KDA_JOINT_FX(G, X, 0))
    switch (gate) {
        case 0: return gd.erase ? KDA_JOINT(0, true) : KDA_JOINT(0, false);
        case 1: return gd.erase ? KDA_JOINT(1, true) : KDA_JOINT(1, false);
        default: return gd.erase ? KDA_JOINT(2, true) : KDA_JOINT(2, false);
    }
#undef KDA_JOINT
#undef KDA_JOINT_FX
}

cudaError_t launch_bwd_scan_tc(const Shape& s, const void* dout, const float* dht, Table t, FwdTC f, BwdTC b,
                               float* dh0, cudaStream_t st, const ConsPiece& pc) {
    cudaError_t e = set_smem_once<k_bwd_scan_tc>(BSCAN_SMEM);
    if (e != cudaSuccess) return e;
    CUtensorMap mo;
    if (!tmap_rows_bf16(&mo, dout, s.Ttot, s.H, s.V)) return cudaErrorInvalidValue;
    dim3 grid(s.N, s.H);
    k_bwd_scan_tc<<<grid, ST_ALL, BSCAN_SMEM, st>>>(s, mo, dht, t, f, b, dh0, pc.lo, pc.L);
    return cudaGetLastError();
}

cudaError_t launch_bwd_consumer_tc(const Shape& s, int gate, const void* q, const void* k, const void* v,
                                   const void* beta, const void* dout, Table t, FwdTC f,
                                   BwdTC b, void* dq, void* dk, void* dv, void* dbeta, float* dg,
                                   cudaStream_t st, const Gdn2& gd, const ConsPiece& pc) {
    // narrower inputs or grouped heads (the consumer's flexible variant keeps its registers at the
    // tile width too), or neither
    const bool flex = s.K != D || s.V != D || s.Gq != 1 || s.Gg != 1;
#define KDA_CONS(G, X)                                                                                    \
    (flex ? run_consumer<G, X, 2>(s, q, k, v, beta, dout, t, f, b, dq, dk, dv, dbeta, dg, st, gd, pc) \
          : run_consumer<G, X, 0>(s, q, k, v, beta, dout, t, f, b, dq, dk, dv, dbeta, dg, st, gd, pc))
    switch (gate) {
        case 0: return gd.erase ? KDA_CONS(0, true) : KDA_CONS(0, false);
        case 1: return gd.erase ? KDA_CONS(1, true) : KDA_CONS(1, false);
        default: return gd.erase ? KDA_CONS(2, true) : KDA_CONS(2, false);
    }
#undef KDA_CONS
}

}  // namespace kda
