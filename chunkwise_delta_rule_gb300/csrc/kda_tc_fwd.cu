// Tensor-core forward path (bf16 I/O, K = V = 128) on tcgen05.
//
// k_prep_tc, one CTA per (chunk slot, head), or per (chunk slot, head) of value blocks
// sharing everything but U (a1-a4):
//   G2 = in-chunk cumsum of g / ln 2; one anchor c per feature (the midpoint
//   of the chunk's range) so that
//       [Akk ; Aqk] = [beta K 2^(G2-c) ; s Q 2^(G2-c)] (K 2^(c-G2))^T
//   is a single M = 128, N = 64, K = 128 bf16 MMA ("Kimi Delta Attention"
//   blog, sections 6.3 and 6.5; "ReWY" paper, centered factors); strict /
//   inclusive masks on the TMEM read-back; A = (I + Akk)^-1 in fp32, 16 x 16
//   diagonal blocks by forward substitution and two levels of block merges; W^T = (E'^T A^T) diag(2^c) and
//   U^T = V^T (A diag(beta))^T as M = 128 bf16 MMAs whose A operands E' =
//   beta K alpha (already in shared memory for the first MMA) and V are read
//   MN-major. A chunk whose gate range exceeds 2^80 is left to the CUDA-core
//   prep (flag WIDE), which anchors per 16-token sub-chunk instead.
//
// k_fwd_scan_tc, one CTA per (sequence, head), 256 threads; warps w and w+4
// own value columns 32(w%4).. (TMEM lanes) and split the other axis. The
// transposed state S^T (V x K, fp32) stays in TMEM for the whole sequence.
// Per chunk (a5, a6):
//       R^T  = U^T - S^T W^T            (MMA, bf16 S^T written to TMEM as its A operand)
//       S^T <- S^T diag(lambda) + R^T F (lambda applied in TMEM, then MMA)
//       O^T  = S^T Q_g^T + R^T C_q^T    (MMAs issued after the state update,
//                                        read back during the next chunk)
// ("ReWY" paper, "The chunk system and conventional WY backward"; "Kimi Delta
// Attention" blog, section 6.4). The operand tiles of chunk c+1 (stored as
// tile images) are fetched with bulk copies while chunk c computes; F is read
// as an MN-major operand.
#include <string.h>

#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using bf16 = __nv_bfloat16;
constexpr int D = 128;

__device__ __forceinline__ float bfx(const bf16* p) { return __bfloat162float(*p); }

// All threads wait for the barrier phase; the result is made uniform and a
// timeout is recorded in the device error word (bit 1).
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, int32_t* err) {
    bool ok = tc::mbar_wait(bar, parity);
    ok = __syncthreads_and(ok) != 0;
    if (!ok && threadIdx.x == 0) atomicOr(err, 2);
    return ok;
}

// =========================================================== k_prep_tc
constexpr int PT = 256;     // 8 warps; ~100 KB of shared memory, so two CTAs share an SM
constexpr int LG = D;       // fp32 row stride of the G / alpha tile (dense rows, as TMA lands them)
constexpr int LW = D + 8;   // row stride (bf16) of the staged W tile

// A = (I + L)^-1 for the strictly lower 64 x 64 L, given as L^T (fp32, row m
// holds column m of L), into sAi (fp32, row stride LA), blockwise:
//  1. the four 16 x 16 diagonal blocks by forward substitution on row vectors,
//     A_i = e_i - sum_{m<i} L_im A_m, applied right-looking (warp b owns block
//     b; lane l holds row l % 16, half l / 16 of the columns);
//  2. the 16 x 16 blocks below them, A_10 = -A_11 (L_10 A_00) (and 3, 2);
//  3. the lower-left 32 x 32 block the same way from the 32 x 32 halves.
// Every block row/column product is a plain fp32 sum; 256 threads.
constexpr int LA = BT + 4;   // row stride of sAi (16-byte aligned rows for vector loads)
constexpr int LT1 = 18, LT2 = 36;
__device__ __forceinline__ void inverse_blocked(const float* __restrict__ sLt, float* __restrict__ sAi,
                                                float* __restrict__ sT, int tid, int warp, int lane) {
    if (warp < 4) {
        const int b0 = 16 * warp, r = lane & 15, ch = lane >> 4;
        float x[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) x[cc] = (r == 8 * ch + cc) ? 1.f : 0.f;
#pragma unroll 1
        for (int m = 0; m < 15; ++m) {
            const float l = sLt[(b0 + m) * BT + b0 + r];   // L[b0 + r][b0 + m]
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) x[cc] = fmaf(-l, __shfl_sync(0xffffffffu, x[cc], (lane & 16) | m), x[cc]);
        }
        *reinterpret_cast<float4*>(sAi + (b0 + r) * LA + b0 + 8 * ch) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(sAi + (b0 + r) * LA + b0 + 8 * ch + 4) = make_float4(x[4], x[5], x[6], x[7]);
    } else {
        // zero blocks above the diagonal
        for (int idx = tid - 128; idx < 6 * 64; idx += 128) {
            const int blk = idx >> 6, e = idx & 63;
            const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            *reinterpret_cast<float4*>(sAi + (16 * bi + (e >> 2)) * LA + 16 * bj + 4 * (e & 3)) =
                make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();
    {   // T = L_10 A_00 (pair 0) and L_32 A_22 (pair 1); two outputs per thread
        const int pr = tid >> 7, r = (tid >> 3) & 15, c = (tid & 7) * 2;
        const int bi = 32 * pr + 16, bj = 32 * pr;
        float2 t = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float l = sLt[(bj + k) * BT + bi + r];
            const float2 a = *reinterpret_cast<const float2*>(sAi + (bj + k) * LA + bj + c);
            t.x = fmaf(l, a.x, t.x);
            t.y = fmaf(l, a.y, t.y);
        }
        *reinterpret_cast<float2*>(sT + (16 * pr + r) * LT1 + c) = t;
    }
    __syncthreads();
    {   // A_10 = -A_11 T
        const int pr = tid >> 7, r = (tid >> 3) & 15, c = (tid & 7) * 2;
        const int bi = 32 * pr + 16, bj = 32 * pr;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float x = sAi[(bi + r) * LA + bi + k];
            const float2 tt = *reinterpret_cast<const float2*>(sT + (16 * pr + k) * LT1 + c);
            acc.x = fmaf(x, tt.x, acc.x);
            acc.y = fmaf(x, tt.y, acc.y);
        }
        *reinterpret_cast<float2*>(sAi + (bi + r) * LA + bj + c) = make_float2(-acc.x, -acc.y);
    }
    __syncthreads();
    {   // T = L[32:64][0:32] A[0:32][0:32]; four outputs per thread
        const int r = tid >> 3, c = (tid & 7) * 4;
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            const float l = sLt[k * BT + 32 + r];
            const float4 a = *reinterpret_cast<const float4*>(sAi + k * LA + c);
            t.x = fmaf(l, a.x, t.x);
            t.y = fmaf(l, a.y, t.y);
            t.z = fmaf(l, a.z, t.z);
            t.w = fmaf(l, a.w, t.w);
        }
        *reinterpret_cast<float4*>(sT + r * LT2 + c) = t;
    }
    __syncthreads();
    {   // A[32:64][0:32] = -A[32:64][32:64] T
        const int r = tid >> 3, c = (tid & 7) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            const float x = sAi[(32 + r) * LA + 32 + k];
            const float4 tt = *reinterpret_cast<const float4*>(sT + k * LT2 + c);
            acc.x = fmaf(x, tt.x, acc.x);
            acc.y = fmaf(x, tt.y, acc.y);
            acc.z = fmaf(x, tt.z, acc.z);
            acc.w = fmaf(x, tt.w, acc.w);
        }
        *reinterpret_cast<float4*>(sAi + (32 + r) * LA + c) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
}

// Shared-memory map of k_prep_tc (bytes from the 1024-aligned base); regions
// are reused once the MMA that reads them has completed.
constexpr int P_A1 = 0;            // [beta K alpha ; s Q alpha] bf16 [128][128], K-major    32 KB
                                   //   (rows 64..127 first hold q as loaded)
                                   //   rows 0..63 double as E' (MN-major view) for W^T
constexpr int P_W = 0;             //   after MMA 2: W staged bf16 [64][LW]
constexpr int P_B1 = 32768;        // K / alpha bf16 [64][128], K-major (first k as loaded)  16 KB
constexpr int P_LT = 32768;        //   after MMA 1: L^T fp32 [64][64]                        16 KB
constexpr int P_V = 49152;         // V bf16 [64][128] (MN-major view for U^T)              16 KB
constexpr int P_ALPHA = 65536;     // g, then alpha = 2^(G2 - c), fp32 [64][LG]              32 KB
constexpr int P_BA = 65536;        //   after MMA 1: A bf16 [64][64], K-major                 8 KB
constexpr int P_BB = 65536 + 8192; //                A diag(beta) bf16 [64][64], K-major      8 KB
constexpr int P_AIF = 65536 + 16384;  //              A fp32 [64][LA] (the blocked inverse)  16.3 KB
constexpr int P_TMP = 8192;        //   after MMA 1 (rows 64..127 of A1's first atom): products  4.2 KB
constexpr int P_MISC = P_AIF + 4 * BT * LA;    // beta [64], 2^c [128], 2^(G2_last - c) [128],
                                               // cumsum exchange: segment total [128], hi, lo [2][128]
constexpr int P_BAR = P_MISC + 4 * (BT + 2 * D + 5 * D);
constexpr size_t PREP_SMEM = P_BAR + 64 + 1024;
static_assert(P_ALPHA + 4 * BT * LG <= P_MISC, "the G tile overlaps the constants");
static_assert(P_TMP + 4 * 32 * LT2 <= 16384, "inverse scratch overlaps E'");
static_assert(BT * LW * 2 <= P_B1, "W staging overlaps L^T");

// SHARE: the value blocks of a head (s.Gg of them, beta rule) prepared by one CTA per key unit.
template <int GATE, bool BWD, bool GD2, bool SHARE>
__global__ void __launch_bounds__(PT, 2)
    k_prep_tc(Shape s, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
              const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmg,
              const bf16* __restrict__ beta, const float* __restrict__ g, Table t, FwdTC f, Gdn2 gd) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    float* sA = reinterpret_cast<float*>(base + P_ALPHA);  // g, then alpha
    float* sBeta = reinterpret_cast<float*>(base + P_MISC);
    float* sC2 = sBeta + BT;   // 2^c
    float* sAL = sC2 + D;      // 2^(G2_last - c)
    float* sLt = reinterpret_cast<float*>(base + P_LT);
    uint64_t* bar = reinterpret_cast<uint64_t*>(base + P_BAR);   // MMA completions
    uint64_t* bld = bar + 1;                                       // input tiles
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);
    const uint32_t sb = tc::smem_u32(base);

    // value blocks of one head (Gg of them, read in place) share everything but U: one CTA per key
    // unit writes the shared tiles to each block's slot and computes each block's U from its own V
    const int nbk = SHARE ? s.Gg : 1;
    const int c = blockIdx.x, h = blockIdx.y * nbk, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = t.chunk_len[c];
    if (n <= 0) return;
    const int tok0 = t.chunk_tok0[c];
    const int H = s.H;
    const int hq = h / s.Gq, hg = h / s.Gg, Hg = heads_g(s);   // heads of q, k and of g, beta, erase
    const size_t ch = (size_t)c * H + h;
    const float scale = s.scale;
    const int c8 = (tid & 15) * 8;   // the 8 feature columns of this thread in every row pass

    // ---- inputs by TMA: k -> B1, q -> rows 64..127 of A1, v -> V (SW128 rows, in place for the
    // MMAs), g -> the G tile (fp32 rows). Rows past the chunk end hold the following tokens (or
    // zeros past the tensor) and are masked out below.
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::mbar_init(bld, 1);
        tc::fence_mbar_init();
        tc::mbar_arrive_expect_tx(bld, 6 * 8192 + (GATE == 2 ? BT * D * 4 : 0));
        tc::tma_load3(sb + P_B1, &tmk, 0, hq, tok0, bld);
        tc::tma_load3(sb + P_B1 + 8192, &tmk, 64, hq, tok0, bld);
        tc::tma_load3(sb + P_A1 + 8192, &tmq, 0, hq, tok0, bld);
        tc::tma_load3(sb + P_A1 + 24576, &tmq, 64, hq, tok0, bld);
        tc::tma_load3(sb + P_V, &tmv, 0, h, tok0, bld);
        tc::tma_load3(sb + P_V + 8192, &tmv, 64, h, tok0, bld);
        if (GATE == 2) tc::tma_load3(sb + P_ALPHA, &tmg, 0, hg, tok0, bld);
    }
    const float beta_r = (tid < BT && tid < n && !GD2) ? bfx(beta + (size_t)(tok0 + tid) * Hg + hg) : 0.f;
    // GatedDeltaNet-2: this chunk's erase and write rows (two 128-byte lines each) into L2 while
    // the cumsum runs; the operand pass reads them
    if (GD2 && (tid >> 2) < n) {
        const bool wr = (tid & 2) != 0;
        const int w = wr ? s.V : s.K;   // the row widths of the write and erase vectors
        const bf16* vec = static_cast<const bf16*>(wr ? gd.write : gd.erase);
        const size_t row = (size_t)(tok0 + (tid >> 2)) * (wr ? H : Hg) + (wr ? h : hg);
        if ((tid & 1) * 64 < w) tc::prefetch_l2(vec + row * w + (tid & 1) * 64);
    }
    if (GATE != 2) {
        // scalar gate: the G tile repeats the token's log-decay; no gate: zeros (this thread's eight
        // rows loaded before any of its stores)
        constexpr int NF = BT * D / 4 / PT;
        float xr[NF];
#pragma unroll
        for (int u = 0; u < NF; ++u) {
            const int r = (tid + PT * u) >> 5;
            xr[u] = (GATE == 1 && r < n) ? __ldg(g + (size_t)(tok0 + r) * Hg + hg) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < NF; ++u) {
            const int idx = tid + PT * u, r = idx >> 5, c4 = (idx & 31) * 4;
            *reinterpret_cast<float4*>(sA + r * LG + c4) = make_float4(xr[u], xr[u], xr[u], xr[u]);
        }
    }
    if (warp == 0) {
        tc::tmem_alloc(tslot, 256);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tb = *tslot;
    bool ok = wait_all(bld, 0, t.err);
    if (!ok && tid == 0) tc::mbar_wait(bld, 0);   // let late tiles land before the CTA can leave

    // a1: cumsum, one feature per lane: warps 0-3 rows 0..31, warps 4-7 rows 32..63 (segment
    // totals and ranges exchanged through shared memory), range, midpoint anchor; alpha =
    // 2^(G2 - c) replaces G2 (one exp2 per element; every decay factor of the chunk is alpha
    // times a per-feature constant or its reciprocal)
    if (tid < BT) sBeta[tid] = beta_r;
    int wide_col = 0;
    if (ok) {
        float* sTot = sAL + D;       // [128] total of rows 0..31
        float* sHi = sTot + D;       // [2][128]
        float* sLo = sHi + 2 * D;    // [2][128]
        const int col = tid & (D - 1), seg = tid >> 7;
        float x[32];
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int row = 32 * seg + r;
            acc += (row < n) ? sA[row * LG + col] : 0.f;
            x[r] = acc;
        }
        if (seg == 0) sTot[col] = acc;
        __syncthreads();
        const float pre = seg ? sTot[col] : 0.f;
        float hi = -INFINITY, lo = INFINITY;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            x[r] = (x[r] + pre) * LOG2E;
            if (32 * seg + r < n) {
                hi = fmaxf(hi, x[r]);
                lo = fminf(lo, x[r]);
            }
        }
        sHi[seg * D + col] = hi;
        sLo[seg * D + col] = lo;
        __syncthreads();
        hi = fmaxf(sHi[col], sHi[D + col]);
        lo = fminf(sLo[col], sLo[D + col]);
        const float cc = 0.5f * (hi + lo);
        // saving for the backward: alpha, 2^c and 2^(G2_last - c) for the backward consumer, which
        // loads them in place of g (per-channel gate: token rows, coalesced over the features;
        // scalar gate: the values of feature 0, equal for every feature)
        constexpr int AU = GATE == 2 ? ALK_UNIT : ALK_SCALAR;
        float* img = (BWD && GATE != 0) ? f.ALK + ch * AU : nullptr;
        const bool put = BWD && (GATE == 2 || (GATE == 1 && col == 0));
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const float a = exp2f(x[r] - cc);
            sA[(32 * seg + r) * LG + col] = a;
            if (put)
                for (int b = 0; b < nbk; ++b) img[b * AU + (32 * seg + r) * (GATE == 2 ? D : 1) + (GATE == 2 ? col : 0)] = a;
        }
        if (seg == 1) {   // G2 at row 63 = last token
            const float c2 = exp2f(cc), al = exp2f(x[31] - cc);
            sC2[col] = c2;
            sAL[col] = al;
            for (int b = 0; b < nbk; ++b) {
                f.GL[(ch + b) * D + col] = x[31];
                if (put) {
                    img[b * AU + BT * (GATE == 2 ? D : 1) + (GATE == 2 ? col : 0)] = c2;
                    img[b * AU + BT * (GATE == 2 ? D : 1) + (GATE == 2 ? D + col : 1)] = al;
                }
            }
        }
        wide_col = (hi - lo) > PREP_RANGE_LOG2;
    }
    const bool wide = __syncthreads_or(wide_col) != 0;
    if (tid == 0 && ok) {
        // every block unit of this key unit, listed for the CUDA-core kernels when wide
        const int w0 = wide ? atomicAdd(f.WLIST, nbk) : 0;
        for (int b = 0; b < nbk; ++b) {
            f.WIDE[ch + b] = wide ? 1 : 0;
            if (wide) f.WLIST[1 + w0 + b] = (int32_t)(ch + b);
        }
    }
    if (!wide && ok) {
        // a2 operands (bf16), in place over the loaded tiles, one pass over the row chunks of this
        // thread: A1 rows 0..63 beta_i k_i alpha_i, rows 64..127 s q_i alpha_i; B1 rows j:
        // k_j / alpha_j; rows past the chunk end zero. Q_g = s q alpha 2^c and
        // F = K 2^(G2_last - G2) = k 2^(G2_last - c) / alpha go to HBM.
        float c2r[8], alr[8];
#pragma unroll
        for (int e = 0; e < 8; e += 4) {
            *reinterpret_cast<float4*>(c2r + e) = *reinterpret_cast<const float4*>(sC2 + c8 + e);
            *reinterpret_cast<float4*>(alr + e) = *reinterpret_cast<const float4*>(sAL + c8 + e);
        }
        constexpr int NU = BT * D / 8 / PT;   // 16-byte chunks per thread
        // GatedDeltaNet-2: the erase and write vectors of this thread's chunks, all read from HBM
        // before the pass's first shared-memory store so that the loads overlap one another
        uint4 er_all[GD2 ? NU : 1], wr_all[GD2 ? NU : 1];
        if (GD2) {
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const int i = (tid + PT * u) >> 4;
                er_all[u] = wr_all[u] = make_uint4(0, 0, 0, 0);
                if (i < n) {
                    const size_t row = (size_t)(tok0 + i) * H + h, rowe = (size_t)(tok0 + i) * Hg + hg;
                    // widths K and V, zero past them
                    if (c8 < s.K) er_all[u] = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(gd.erase) + rowe * s.K + c8);
                    if (c8 < s.V) wr_all[u] = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(gd.write) + row * s.V + c8);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int i = (tid + PT * u) >> 4;
            unsigned char* kp = base + P_B1 + tc::sw128_off(BT, i, c8 * 2);
            unsigned char* qp = base + P_A1 + tc::sw128_off(2 * BT, BT + i, c8 * 2);
            uint4 kr = *reinterpret_cast<const uint4*>(kp), qr = *reinterpret_cast<const uint4*>(qp);
            if (i >= n) kr = qr = make_uint4(0, 0, 0, 0);
            const bf16* kv = reinterpret_cast<const bf16*>(&kr);
            const bf16* qv = reinterpret_cast<const bf16*>(&qr);
            // GatedDeltaNet-2: the erase vector on E's key rows in place of beta, and V scaled by
            // the write vector in place (U = A (w .* V))
            const uint4 er4 = er_all[GD2 ? u : 0];
            if (GD2 && i < n) {
                const uint4 wr4 = wr_all[GD2 ? u : 0];
                uint4* vp = reinterpret_cast<uint4*>(base + P_V + tc::sw128_off(BT, i, c8 * 2));
                const uint4 v4 = *vp;
                const bf16* vv = reinterpret_cast<const bf16*>(&v4);
                const bf16* wv = reinterpret_cast<const bf16*>(&wr4);
                uint32_t pv[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2)
                    pv[e / 2] = tc::pack_bf16(__bfloat162float(wv[e]) * __bfloat162float(vv[e]),
                                              __bfloat162float(wv[e + 1]) * __bfloat162float(vv[e + 1]));
                *vp = make_uint4(pv[0], pv[1], pv[2], pv[3]);
            } else if (GD2) {
                *reinterpret_cast<uint4*>(base + P_V + tc::sw128_off(BT, i, c8 * 2)) = make_uint4(0, 0, 0, 0);
            }
            const bf16* ev = reinterpret_cast<const bf16*>(&er4);
            float al[8];
            *reinterpret_cast<float4*>(al) = *reinterpret_cast<const float4*>(sA + i * LG + c8);
            *reinterpret_cast<float4*>(al + 4) = *reinterpret_cast<const float4*>(sA + i * LG + c8 + 4);
            const float bt = sBeta[i];
            uint32_t pe[4], pq[4], pz[4], pg[4], pf[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float a0 = al[e], a1 = al[e + 1];
                const float r0 = tc::rcp_approx(a0), r1 = tc::rcp_approx(a1);
                const float k0 = __bfloat162float(kv[e]), k1 = __bfloat162float(kv[e + 1]);
                const float q0 = scale * __bfloat162float(qv[e]) * a0, q1 = scale * __bfloat162float(qv[e + 1]) * a1;
                const float z0 = k0 * r0, z1 = k1 * r1;
                const float b0 = GD2 ? __bfloat162float(ev[e]) : bt, b1 = GD2 ? __bfloat162float(ev[e + 1]) : bt;
                pe[e / 2] = tc::pack_bf16(b0 * k0 * a0, b1 * k1 * a1);
                pq[e / 2] = tc::pack_bf16(q0, q1);
                pz[e / 2] = tc::pack_bf16(z0, z1);
                pg[e / 2] = tc::pack_bf16(q0 * c2r[e], q1 * c2r[e + 1]);
                pf[e / 2] = tc::pack_bf16(z0 * alr[e], z1 * alr[e + 1]);
            }
            *reinterpret_cast<uint4*>(base + P_A1 + tc::sw128_off(2 * BT, i, c8 * 2)) = make_uint4(pe[0], pe[1], pe[2], pe[3]);
            *reinterpret_cast<uint4*>(qp) = make_uint4(pq[0], pq[1], pq[2], pq[3]);
            *reinterpret_cast<uint4*>(kp) = make_uint4(pz[0], pz[1], pz[2], pz[3]);
            for (int b = 0; b < nbk; ++b) {
                *reinterpret_cast<uint4*>(f.QG + (ch + b) * BT * D + tile_el(BT, i, c8)) = make_uint4(pg[0], pg[1], pg[2], pg[3]);
                *reinterpret_cast<uint4*>(f.KG + (ch + b) * BT * D + tile_el(BT, i, c8)) = make_uint4(pf[0], pf[1], pf[2], pf[3]);
            }
        }
        tc::fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t id = tc::idesc_bf16(128, 64);
#pragma unroll 1
            for (int st = 0; st < 8; ++st)
                tc::mma_bf16(tb, tc::sdesc_k(sb + P_A1, 2 * BT, st), tc::sdesc_k(sb + P_B1, BT, st), id, st > 0);
            tc::mma_commit(bar);
        }
        ok = wait_all(bar, 0, t.err);
    }
    if (!wide && ok) {
        tc::fence_after_sync();
        // read back [Akk ; Aqk]: warps w and w+4 share lanes 32(w%4).., 32 columns each;
        // Akk -> L^T (fp32, strict, rows < n), Aqk -> C_q (bf16, inclusive) in HBM
        {
            const int row = 32 * (warp & 3) + lane, cb = (warp >> 2) * 32;
            float a[32];
            tc::tmem_ld16(tc::taddr(tb, 32 * (warp & 3), cb), *reinterpret_cast<float(*)[16]>(a));
            tc::tmem_ld16(tc::taddr(tb, 32 * (warp & 3), cb + 16), *reinterpret_cast<float(*)[16]>(a + 16));
            tc::tmem_wait_ld();
            if (row < BT) {
                const int i = row;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = cb + jj;
                    sLt[j * BT + i] = (j < i && i < n) ? a[jj] : 0.f;
                }
            } else {
                const int i = row - BT;
                uint32_t pw[16];
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2) {
                    const int j = cb + jj;
                    pw[jj / 2] = tc::pack_bf16((j <= i && i < n) ? a[jj] : 0.f, (j + 1 <= i && i < n) ? a[jj + 1] : 0.f);
                }
                for (int b = 0; b < nbk; ++b) {
                    bf16* dst = f.AQK + (ch + b) * BT * BT;
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
                        *reinterpret_cast<uint4*>(dst + tile_el(BT, i, cb + 8 * qq)) =
                            make_uint4(pw[4 * qq], pw[4 * qq + 1], pw[4 * qq + 2], pw[4 * qq + 3]);
                }
            }
        }
        __syncthreads();
        // a3 + a4: A = (I + Akk)^-1, then the bf16 B operands A (for W^T = E'^T A^T) and
        // A diag(beta) (for U^T = V^T (A diag(beta))^T), and A itself for the backward
        float* sAi = reinterpret_cast<float*>(base + P_AIF);
        inverse_blocked(sLt, sAi, reinterpret_cast<float*>(base + P_TMP), tid, warp, lane);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int i = tid >> 2, c8 = 16 * (tid & 3) + 8 * hh;
            const float* ai = sAi + i * LA + c8;
            uint32_t a[4], bb[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                a[e] = tc::pack_bf16(ai[2 * e], ai[2 * e + 1]);
                bb[e] = tc::pack_bf16(ai[2 * e] * sBeta[c8 + 2 * e], ai[2 * e + 1] * sBeta[c8 + 2 * e + 1]);
            }
            const uint4 va = make_uint4(a[0], a[1], a[2], a[3]);
            *reinterpret_cast<uint4*>(base + P_BA + tc::sw128_off(BT, i, 2 * c8)) = va;
            *reinterpret_cast<uint4*>(base + P_BB + tc::sw128_off(BT, i, 2 * c8)) = make_uint4(bb[0], bb[1], bb[2], bb[3]);
            if (BWD)
                for (int b = 0; b < nbk; ++b) *reinterpret_cast<uint4*>(f.AI + (ch + b) * BT * BT + tile_el(BT, i, c8)) = va;
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            // W^T 2^-c = E'^T A^T and U^T = V^T (A diag(beta))^T; E' and V are read MN-major
            const uint32_t id = tc::idesc_bf16_amn(128, 64);
#pragma unroll 1
            for (int st = 0; st < 4; ++st)
                tc::mma_bf16(tb + 64, tc::sdesc_mn(sb + P_A1, 2 * BT * 128, st), tc::sdesc_k(sb + P_BA, BT, st), id, st > 0);
#pragma unroll 1
            for (int st = 0; st < 4; ++st)
                tc::mma_bf16(tb + 128, tc::sdesc_mn(sb + P_V, BT * 128, st),
                             tc::sdesc_k(sb + (GD2 ? P_BA : P_BB), BT, st), id, st > 0);
            tc::mma_commit(bar);
        }
        ok = wait_all(bar, 1, t.err);
        if (ok) {
            tc::fence_after_sync();
            bf16* sW = reinterpret_cast<bf16*>(base + P_W);   // staged W [64][LW]
            const int row = 32 * (warp & 3) + lane;
            if (warp < 4) {
                // W^T row = key `row`, scaled by 2^c -> staged W[i][row]
                const float c2 = sC2[row];
#pragma unroll
                for (int cb = 0; cb < BT; cb += 16) {
                    float a[16];
                    tc::tmem_ld16(tc::taddr(tb + 64, 32 * warp, cb), a);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) sW[(cb + jj) * LW + row] = __float2bfloat16_rn(a[jj] * c2);
                }
            } else {
                // U^T row = value `row` -> U[i][row] (bf16, coalesced over the value index)
                bf16* U = f.U + ch * BT * D + row;
#pragma unroll
                for (int cb = 0; cb < BT; cb += 16) {
                    float a[16];
                    tc::tmem_ld16(tc::taddr(tb + 128, 32 * (warp & 3), cb), a);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) U[(size_t)(cb + jj) * D] = __float2bfloat16_rn(a[jj]);
                }
            }
            __syncthreads();
            for (int idx = tid; idx < BT * 16; idx += PT) {
                const int i = idx >> 4, cc8 = (idx & 15) * 8;
                const uint4 wv = *reinterpret_cast<const uint4*>(sW + i * LW + cc8);
                for (int b = 0; b < nbk; ++b) *reinterpret_cast<uint4*>(f.W + (ch + b) * BT * D + tile_el(BT, i, cc8)) = wv;
            }
            // the further value blocks: U = A diag(beta) V of each from its own V tile, loaded into the
            // V region (free once MMA 2 has completed) on the input barrier's next phases
            for (int b = 1; b < nbk && ok; ++b) {
                tc::fence_before_sync();
                __syncthreads();   // the previous U read back from TMEM
                if (tid == 0) {
                    tc::fence_after_sync();
                    tc::mbar_arrive_expect_tx(bld, 2 * 8192);
                    tc::tma_load3(sb + P_V, &tmv, 0, h + b, tok0, bld);
                    tc::tma_load3(sb + P_V + 8192, &tmv, 64, h + b, tok0, bld);
                }
                ok = wait_all(bld, b & 1, t.err);
                if (!ok) {
                    if (tid == 0) tc::mbar_wait(bld, b & 1);   // let the late tile land before the CTA can leave
                    break;
                }
                if (tid == 0) {
                    tc::fence_after_sync();
                    const uint32_t id = tc::idesc_bf16_amn(128, 64);
#pragma unroll 1
                    for (int st = 0; st < 4; ++st)
                        tc::mma_bf16(tb + 128, tc::sdesc_mn(sb + P_V, BT * 128, st), tc::sdesc_k(sb + P_BB, BT, st), id,
                                     st > 0);
                    tc::mma_commit(bar);
                }
                ok = wait_all(bar, (1 + b) & 1, t.err);
                if (!ok) break;
                tc::fence_after_sync();
                if (warp >= 4) {
                    bf16* U = f.U + (ch + b) * BT * D + 32 * (warp & 3) + lane;
#pragma unroll
                    for (int cb = 0; cb < BT; cb += 16) {
                        float a[16];
                        tc::tmem_ld16(tc::taddr(tb + 128, 32 * (warp & 3), cb), a);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) U[(size_t)(cb + jj) * D] = __float2bfloat16_rn(a[jj]);
                    }
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 256);
}

// ======================================================= k_fwd_scan_tc
constexpr int ST = 256;            // compute warps: warps w and w+4 share TMEM lane quarter w%4
constexpr int ST_ALL = ST + 32;    // + one warp that issues the MMAs and the bulk fills
// Named barriers; compute warps and the issuer meet on each (also keeping them
// in lockstep if an MMA wait ever times out).
constexpr int NB_AS = 1;           // S^T staged for D1
constexpr int NB_AR = 2;           // R^T staged for the state update and the output
constexpr int NB_C = 3;            //                compute warps only

// Shared-memory map per mode (bytes from the 1024-aligned base): two operand stages (B operands
// only), the staging the mode stores from, then lambda [128] fp32, per-warp transpose staging
// (8 x 1280 B) and barriers. A smaller map leaves more of the SM's shared storage to the L1
// cache, which carries the U loads of every chunk.
//   mode 1 (output):        stage = [W ; Q_g] as one K-major [128][128] tile (32 KB), F [64][128]
//                           (16 KB, read MN-major), C_q [64][64] (8 KB); two [64][128] output tile
//                           images for the TMA stores
//   mode 2 (S, R):          stage = W [64][128] (16 KB), F; S and R tile images of two chunks
//   mode 3 (output, S, R):  stage and output tiles as mode 1; S and R of one chunk
// S and R go to HBM by one bulk copy each. Every mode also holds one bf16 U tile [64][128] (16 KB,
// row-major), bulk-copied by the issuer a chunk ahead.
template <int MODE>
struct ScanMap {
    static constexpr bool OUT = (MODE & 1) != 0;
    static constexpr int WROWS = OUT ? 2 * BT : BT;             // rows of the [W ; Q_g] (or W) tile
    static constexpr int KG = WROWS * D * 2;                    // F
    static constexpr int AQ = KG + BT * D * 2;                  // C_q (output modes)
    static constexpr int STG = OUT ? AQ + BT * BT * 2 : AQ;     // bytes of one stage
    static constexpr int NOST = (MODE & 1) ? 2 : 0;             // output staging tiles
    static constexpr int NSR = (MODE == 2) ? 2 : (MODE == 3) ? 1 : 0;   // S/R staging pairs
    static constexpr int OST = 2 * STG;
    static constexpr int HST = OST + NOST * BT * D * 2;         // S [128][128] bf16 each
    static constexpr int RST = HST + NSR * D * D * 2;           // R [64][128] bf16 each
    static constexpr int UST = RST + NSR * BT * D * 2;          // U [64][128] bf16
    static constexpr int LAM = UST + BT * D * 2;
    static constexpr int TST = LAM + 512;
    static constexpr int BAR = TST + 8 * 1280;
    static constexpr int SMEM = BAR + 128 + 1024;
    static_assert(SMEM <= 232448, "scan shared memory above the per-block limit");
    static_assert(OST % 1024 == 0, "swizzled TMA stores need 1024-byte aligned tiles");
};

// TMEM columns: S^T fp32 [0,128); two buffers [D1 | O^T] of 128 columns at
// [128,256) and [256,384), where one N = 128 pass S^T [W ; Q_g]^T gives D1 = S^T W^T
// and the first output term, and R^T C_q^T is added to the output half after
// the state update (read back during the next chunk); the bf16 A operands
// S^T (64 columns) at [384,448) and R^T (32 columns) at [448,480). The MMAs read
// only their B operands from shared memory.
constexpr int T_DO = 128, T_AS = 384, T_AR = 448;

// Stages the operand tiles of one chunk (stored as tile images) with bulk
// copies; one thread; completion arrives on `full` as transaction bytes.
template <int MODE>
__device__ __forceinline__ void fscan_fill(uint32_t stg, const FwdTC& f, size_t ch, uint64_t* full) {
    using M = ScanMap<MODE>;
    constexpr uint32_t TILE = BT * D * 2, TQ = BT * BT * 2;
    tc::mbar_arrive_expect_tx(full, M::OUT ? 3 * TILE + TQ : 2 * TILE);
    const unsigned char* w = reinterpret_cast<const unsigned char*>(f.W + ch * BT * D);
    if (M::OUT) {
        // W in rows 0..63 and Q_g in rows 64..127 of each 64-column atom block
        const unsigned char* qg = reinterpret_cast<const unsigned char*>(f.QG + ch * BT * D);
        tc::bulk_g2s(stg, w, TILE / 2, full);
        tc::bulk_g2s(stg + 2 * BT * 128, w + TILE / 2, TILE / 2, full);
        tc::bulk_g2s(stg + BT * 128, qg, TILE / 2, full);
        tc::bulk_g2s(stg + 3 * BT * 128, qg + TILE / 2, TILE / 2, full);
        tc::bulk_g2s(stg + M::AQ, f.AQK + ch * BT * BT, TQ, full);
    } else {
        tc::bulk_g2s(stg, w, TILE, full);   // the W tile image as it is
    }
    tc::bulk_g2s(stg + M::KG, f.KG + ch * BT * D, TILE, full);
}

// The output of a full chunk from its staging tile (a [64][128] tile image) to
// HBM: two TMA box stores, one per 64-column atom block (lane 0 of the caller).
// A box that would start past the value width V is not issued (its columns would all be dropped).
__device__ __forceinline__ void fscan_tma_out(const CUtensorMap* tmo, uint32_t ost, int tok0, int h, int V, int lane) {
    if (lane == 0) {
        tc::tma_store3(tmo, 0, h, tok0, ost);
        if (V > 64) tc::tma_store3(tmo, 64, h, tok0, ost + BT * 128);
        tc::bulk_commit();
    }
}

// Output rows [ib, ib+32) of a chunk straight from O^T in TMEM (this thread: value
// column vcol), 16 rows at a time, rows >= len skipped.
__device__ __forceinline__ void fscan_store_tail(uint32_t tl_o, int len, int tok0, int H, int V, int h, int ib,
                                                 int quad, int lane, bf16* tst, bf16* __restrict__ o) {
    const int wcols = V - 32 * quad;   // value columns of this warp's 32 that o has
    if (wcols <= 0) return;
#pragma unroll 1
    for (int cq = 0; cq < 32; cq += 16) {
        const int r0 = ib + cq;
        if (r0 < len) {
            float ov[16];
            tc::tmem_ld16(tl_o + r0, ov);
            tc::tmem_wait_ld();
            tc::warp_store_t16(tst, ov, o + ((size_t)(tok0 + r0) * H + h) * V + 32 * quad, (size_t)H * V, len - r0,
                               lane, wcols);
        }
    }
}

// A full chunk's output from O^T in TMEM into its staging tile image (rows
// [ib, ib+32) of value column vcol), then made visible to the TMA store.
__device__ __forceinline__ void fscan_stage_out(uint32_t tl_o, bf16* ost, int ib, int vcol) {
    float ov[2][16];
    tc::tmem_ld16(tl_o + ib, ov[0]);
    tc::tmem_ld16(tl_o + ib + 16, ov[1]);
    tc::tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) ost[tile_el(BT, ib + j, vcol)] = __float2bfloat16_rn(ov[j >> 4][j & 15]);
    tc::fence_async_smem();
}

// Compute warps: every per-element pass over S^T, D1, R^T and O^T. The work
// that gates the next MMA (the bf16 copies of S^T and R^T) comes first and is
// handed over on a named barrier; the rest (lambda scaling of S^T, saved
// states, the previous chunk's output) overlaps the MMA that follows.
template <int MODE>
__device__ __forceinline__ void fscan_compute(const Shape& s, const float* __restrict__ h0, const Table& t,
                                              const FwdTC& f, bf16* __restrict__ o, float* __restrict__ ht,
                                              unsigned char* base, uint64_t* bar, uint32_t tb, int nseq, int h,
                                              int c0, int c1) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    float* sLam = reinterpret_cast<float*>(base + ScanMap<MODE>::LAM);
    bf16* tst = reinterpret_cast<bf16*>(base + ScanMap<MODE>::TST + warp * 1280);
    const int H = s.H;
    const int vcol = 32 * quad + lane;  // TMEM lane and value column of this thread
    const uint32_t tl = tc::taddr(tb, 32 * quad, 0);
    const int K = s.K, V = s.V;         // the state's widths ([K][V] per sequence and head; K, V <= D)
    const size_t st_off = ((size_t)nseq * H + h) * K * V;
    uint64_t* ufull = bar + 7;          // the U tile of the current chunk has landed
    const int kb = 64 * half;   // this thread's half of the key columns of S^T
    const int ib = 32 * half;   // this thread's half of the chunk rows

    // S^T <- h0^T (thread holds row v: h0[k][v] for its keys)
#pragma unroll 1
    for (int cb = kb; cb < kb + 64; cb += 16) {
        float a[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
            a[jj] = (h0 && cb + jj < K && vcol < V) ? h0[st_off + (size_t)(cb + jj) * V + vcol] : 0.f;
        tc::tmem_st16(tl + cb, a);
    }
    tc::tmem_wait_st();

    bool ok = true;
    auto wait_one = [&](uint64_t* b, uint32_t parity) {
        if (ok && !tc::mbar_wait(b, parity)) {
            ok = false;
            atomicOr(t.err, 2);
        }
        tc::fence_after_sync();
    };
    // G at the chunk end (threads < D), loaded a chunk ahead; the previous chunk's extent
    float gln = 0.f;
    if (c0 < c1 && tid < D) gln = __ldg(f.GL + ((size_t)c0 * H + h) * D + tid);
    int lenp = 0, tok0p = 0;
    for (int c = c0; c < c1; ++c) {
        const int it = c - c0, stage = it & 1;
        const size_t ch = (size_t)c * H + h;
        if (tid < D) sLam[tid] = exp2f(gln);
        if (c + 1 < c1 && tid < D) gln = __ldg(f.GL + (ch + H) * D + tid);
        if (it > 0) wait_one(&bar[1], (it - 1) & 1);   // the state update of chunk c-1
        tc::named_sync(NB_C, ST);
        // 1. S^T -> bf16 A operand of D1 = S^T W^T (TMEM), handed to the issuer
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            float sv[2][16];
            tc::tmem_ld16(tl + kb + 32 * hq, sv[0]);
            tc::tmem_ld16(tl + kb + 32 * hq + 16, sv[1]);
            tc::tmem_wait_ld();
            uint32_t pw[16];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                pw[jj] = tc::pack_bf16(sv[0][2 * jj], sv[0][2 * jj + 1]);
                pw[8 + jj] = tc::pack_bf16(sv[1][2 * jj], sv[1][2 * jj + 1]);
            }
            tc::tmem_st16u(tl + T_AS + kb / 2 + 16 * hq, pw);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::named_sync(NB_AS, ST_ALL);
        // 2. while D1 runs: S^T <- S^T diag(lambda) (before the update MMAs accumulate)
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const int cb = kb + 16 * q4;
            float a[16];
            tc::tmem_ld16(tl + cb, a);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) a[jj] *= sLam[cb + jj];
            tc::tmem_st16(tl + cb, a);
        }
        tc::tmem_wait_st();
        // U rows of this thread's value column (staged by the issuer a chunk ahead)
        float u[32];
        wait_one(ufull, it & 1);
        {
            const bf16* sU = reinterpret_cast<const bf16*>(base + ScanMap<MODE>::UST) + ib * D + vcol;
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __bfloat162float(sU[i * D]);
        }
        // 3. R^T = U^T - D1 -> bf16 A operand (TMEM) of the state update and the output
        wait_one(&bar[0], it & 1);
        uint32_t rp[16];   // R^T rows ib.. of this value column, bf16 pairs (kept for the saved R)
        {
            float rv[2][16];
            tc::tmem_ld16(tl + T_DO + 128 * stage + ib, rv[0]);
            tc::tmem_ld16(tl + T_DO + 128 * stage + ib + 16, rv[1]);
            tc::tmem_wait_ld();
#pragma unroll
            for (int cq = 0; cq < 2; ++cq) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) rv[cq][jj] = u[16 * cq + jj] - rv[cq][jj];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) rp[8 * cq + jj] = tc::pack_bf16(rv[cq][2 * jj], rv[cq][2 * jj + 1]);
            }
            tc::tmem_st16u(tl + T_AR + ib / 2, rp);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::named_sync(NB_AR, ST_ALL);
        // 4. while the state update runs: the output of chunk c-1 (one output barrier per TMEM
        //    buffer, so the commit of this chunk's output cannot be taken for it), then the saved S
        //    and R (mode 3: once the issuer reports the single staging pair read out by the bulk
        //    copy of the previous chunk's)
        if ((MODE & 1) && it > 0) {
            // output of chunk c-1: a full chunk goes to staging tile (it-1)&1 (stored by the
            // issuer after the next hand-over), a tail chunk straight to HBM
            wait_one(&bar[2 + ((it - 1) & 1)], ((it - 1) >> 1) & 1);
            const uint32_t to = tl + T_DO + 128 * ((it - 1) & 1) + 64;
            if ((MODE & 1) && lenp == BT)
                fscan_stage_out(to, reinterpret_cast<bf16*>(base + ScanMap<MODE>::OST) + ((it - 1) & 1) * BT * D, ib, vcol);
            else
                fscan_store_tail(to, lenp, tok0p, H, s.V, h, ib, quad, lane, tst, o);
        }
        if (MODE & 2) {
            // R and S (from the bf16 S^T operand still in TMEM) as tile images into their staging
            // buffer; the issuer copies them to HBM after the next hand-over
            if (ScanMap<MODE>::NSR == 1) wait_one(bar + 8, it & 1);
            const int sbuf = (ScanMap<MODE>::NSR == 2) ? (it & 1) : 0;
            uint16_t* hs = reinterpret_cast<uint16_t*>(base + ScanMap<MODE>::HST) + sbuf * D * D;
            uint16_t* rs = reinterpret_cast<uint16_t*>(base + ScanMap<MODE>::RST) + sbuf * BT * D;
            const uint16_t* r16 = reinterpret_cast<const uint16_t*>(rp);
#pragma unroll
            for (int j = 0; j < 32; ++j) rs[tile_el(BT, ib + j, vcol)] = r16[j];
#pragma unroll 1
            for (int hq = 0; hq < 2; ++hq) {
                float pv[16];
                tc::tmem_ld16(tl + T_AS + kb / 2 + 16 * hq, pv);
                tc::tmem_wait_ld();
                const uint16_t* p16 = reinterpret_cast<const uint16_t*>(pv);
#pragma unroll
                for (int j = 0; j < 32; ++j) hs[tile_el(D, kb + 32 * hq + j, vcol)] = p16[j];
            }
            tc::fence_async_smem();
        }
        lenp = __ldg(t.chunk_len + c);
        tok0p = __ldg(t.chunk_tok0 + c);
    }
    if (c1 > c0) {
        const int last = c1 - 1 - c0;
        wait_one(&bar[1], last & 1);
        if (MODE & 1) {
            // the last output: staging tile last&1 (stored by the issuer at the end) or HBM
            wait_one(&bar[2 + (last & 1)], (last >> 1) & 1);
            const uint32_t to = tl + T_DO + 128 * (last & 1) + 64;
            if ((MODE & 1) && lenp == BT)
                fscan_stage_out(to, reinterpret_cast<bf16*>(base + ScanMap<MODE>::OST) + (last & 1) * BT * D, ib, vcol);
            else
                fscan_store_tail(to, lenp, tok0p, H, s.V, h, ib, quad, lane, tst, o);
        }
    }
    if (ok && ht) {
#pragma unroll 1
        for (int cb = kb; cb < kb + 64; cb += 16) {
            float a[16];
            tc::tmem_ld16(tl + cb, a);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
                if (cb + jj < K && vcol < V) ht[st_off + (size_t)(cb + jj) * V + vcol] = a[jj];
        }
    }
}

// Issuer warp: bulk fills of the operand stages (lane 0) and every MMA (the
// whole warp with warp-uniform descriptors, one elected lane issuing).
template <int MODE>
__device__ __forceinline__ void fscan_issue(const Shape& s, const Table& t, const FwdTC& f, const CUtensorMap* tmo,
                                            uint32_t sb, uint64_t* bar, uint64_t* full, uint32_t tb, int h, int c0,
                                            int c1, int& pl, int& pt, int& filled, int& waited) {
    const int lane = threadIdx.x & 31;
    const int H = s.H;
    const uint32_t i1 = tc::idesc_bf16(128, (MODE & 1) ? 128 : 64), i64 = tc::idesc_bf16(128, 64),
                   i128m = tc::idesc_bf16_bmn(128, 128);
    const uint32_t aS = tb + T_AS, aR = tb + T_AR;   // A operands in TMEM
    for (int c = c0; c < c1; ++c) {
        const int it = c - c0, stage = it & 1;
        const uint32_t stg = sb + stage * ScanMap<MODE>::STG;
        const uint32_t tD = tb + T_DO + 128 * stage;
        tc::named_sync(NB_AS, ST_ALL);
        tc::fence_after_sync();
        if (!tc::mbar_wait(&full[stage], (it >> 1) & 1) && lane == 0) atomicOr(t.err, 2);
        {
            // [D1 | O] = S^T [W ; Q_g]^T (D1 alone without the output)
            const uint64_t dWQ = tc::sdesc(stg);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16_ts_w(tD, aS + 8 * ks, tc::kstep_k(dWQ, ScanMap<MODE>::WROWS, ks), i1, ks > 0);
            tc::mma_commit_w(&bar[0]);
        }
        if (lane == 0) {
            ++waited;
            if (c + 1 < c1) {
                // the other stage is free once every MMA of chunk c-1 has completed (a commit
                // covers all earlier MMAs of the issuing thread)
                if (it > 0) {
                    const bool done = (MODE & 1) ? tc::mbar_wait(&bar[2 + ((it - 1) & 1)], ((it - 1) >> 1) & 1)
                                                 : tc::mbar_wait(&bar[1], (it - 1) & 1);
                    if (!done) atomicOr(t.err, 2);
                }
                fscan_fill<MODE>(sb + (stage ^ 1) * ScanMap<MODE>::STG, f, (size_t)(c + 1) * H + h,
                                 &full[stage ^ 1]);
                ++filled;
            }
        }
        // S and R of chunk c-1, staged during chunk c-1 (the older bulk group of this iteration)
        if ((MODE & 2) && it >= 1 && lane == 0) {
            const size_t cp = (size_t)(c - 1) * H + h;
            const int sbuf = (ScanMap<MODE>::NSR == 2) ? ((it - 1) & 1) : 0;
            tc::bulk_s2g(f.HS + cp * D * D, sb + ScanMap<MODE>::HST + sbuf * D * D * 2, D * D * 2);
            tc::bulk_s2g(f.R + cp * BT * D, sb + ScanMap<MODE>::RST + sbuf * BT * D * 2, BT * D * 2);
            tc::bulk_commit();
        }
        // the output of chunk c-2 (a full chunk), staged by the compute warps during chunk c-1
        const bool o_out = (MODE & 1) && it >= 2 && pl == BT;
        if (o_out) fscan_tma_out(tmo, sb + ScanMap<MODE>::OST + (it & 1) * BT * D * 2, pt, h, s.V, lane);
        if ((MODE & 1) && it >= 1) {   // extent of chunk c-1, whose output is stored next iteration
            pl = __ldg(t.chunk_len + c - 1);
            pt = __ldg(t.chunk_tok0 + c - 1);
        }
        // the staging tiles stored during chunk c-1 are rewritten after this hand-over; the output
        // tile stored just now may still be read (it is rewritten during chunk c+1), and so may a
        // double-buffered S/R pair; a single S/R pair is rewritten after this hand-over
        if (lane == 0 && ScanMap<MODE>::NSR != 1) tc::bulk_wait_read_prev();
        __syncwarp();
        tc::named_sync(NB_AR, ST_ALL);
        tc::fence_after_sync();
        // S^T += R^T F first (it gates the next chunk), then O^T += R^T C_q^T
        {
            const uint64_t dF = tc::sdesc_mn(stg + ScanMap<MODE>::KG, BT * 128, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc::mma_bf16_ts_w(tb, aR + 8 * ks, tc::kstep_mn(dF, ks), i128m, 1);
            tc::mma_commit_w(&bar[1]);
        }
        if (MODE & 1) {
            const uint64_t dA = tc::sdesc(stg + ScanMap<MODE>::AQ);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc::mma_bf16_ts_w(tD + 64, aR + 8 * ks, tc::kstep_k(dA, BT, ks), i64, 1);
            tc::mma_commit_w(&bar[2 + stage]);
        }
        // a single S/R staging pair (mode 3) is rewritten by the compute warps during this chunk:
        // report it free once the bulk copy of the previous chunk's pair has read it (waiting here,
        // after the MMAs are issued, keeps the copy off the chain)
        if (ScanMap<MODE>::NSR == 1 && lane == 0) {
            tc::bulk_wait_read();
            tc::mbar_arrive(bar + 8);
        }
        // U of chunk c+1: the compute warps read this chunk's U before the R hand-over above
        if (lane == 0 && c + 1 < c1) {
            tc::mbar_arrive_expect_tx(bar + 7, BT * D * 2);
            tc::bulk_g2s(sb + ScanMap<MODE>::UST, f.U + ((size_t)(c + 1) * H + h) * BT * D, BT * D * 2, bar + 7);
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(ST_ALL, 1)
    k_fwd_scan_tc(Shape s, const __grid_constant__ CUtensorMap tmo, const float* __restrict__ h0, Table t, FwdTC f,
                  bf16* __restrict__ o, float* __restrict__ ht) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(base + ScanMap<MODE>::BAR);   // D1, state update, output (x2)
    uint64_t* full = bar + 4;                                        // operand stages 0, 1
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 6);
    const uint32_t sb = tc::smem_u32(base);
    // (sequence, head) from the linear CTA index: sequences in the table's order, longest first,
    // every head of one before the next
    const int lin = (int)(blockIdx.x + blockIdx.y * gridDim.x);
    const int nseq = t.seq_order[lin / s.H], h = lin % s.H, tid = threadIdx.x, warp = tid >> 5;
    const int c0 = t.seq_chunk0[nseq], c1 = t.seq_chunk0[nseq + 1];
    const bool issuer = warp == ST / 32;
    int filled = 0, waited = 0;   // bulk fills issued / consumed (issuer lane 0)
    int pl = 0, pt = 0;           // extent of the chunk whose output is staged but not yet stored

    if (issuer && (tid & 31) == 0) {
        for (int i = 0; i < 6; ++i) tc::mbar_init(&bar[i], 1);
        tc::mbar_init(&bar[7], 1);   // U tile (bar + 6 holds the TMEM slot)
        tc::mbar_init(&bar[8], 1);   // mode 3: the S/R staging pair is free
        tc::fence_mbar_init();
        if (c0 < c1) {
            fscan_fill<MODE>(sb, f, (size_t)c0 * s.H + h, &full[0]);
            filled = 1;
            tc::mbar_arrive_expect_tx(&bar[7], BT * D * 2);
            tc::bulk_g2s(sb + ScanMap<MODE>::UST, f.U + ((size_t)c0 * s.H + h) * BT * D, BT * D * 2, &bar[7]);
        }
    }
    if (warp == 0) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tb = *tslot;
    if (issuer)
        fscan_issue<MODE>(s, t, f, &tmo, sb, bar, full, tb, h, c0, c1, pl, pt, filled, waited);
    else
        fscan_compute<MODE>(s, h0, t, f, o, ht, base, bar, tb, nseq, h, c0, c1);
    // a bulk fill still in flight (only after a timeout) lands before the CTA leaves; the last U
    // tile (chunk c1-1, parity of its chunk index) likewise
    if (issuer && (tid & 31) == 0) {
        for (; waited < filled; ++waited) tc::mbar_wait(&full[waited & 1], (waited >> 1) & 1);
        if (c1 > c0) tc::mbar_wait(&bar[7], (c1 - 1 - c0) & 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    // S and R of the last chunk (staged after the issuer's loop ended)
    if ((MODE & 2) && issuer && c1 > c0 && (tid & 31) == 0) {
        const int last = c1 - 1 - c0;
        const size_t cp = (size_t)(c1 - 1) * s.H + h;
        const int sbuf = (ScanMap<MODE>::NSR == 2) ? (last & 1) : 0;
        tc::bulk_s2g(f.HS + cp * D * D, sb + ScanMap<MODE>::HST + sbuf * D * D * 2, D * D * 2);
        tc::bulk_s2g(f.R + cp * BT * D, sb + ScanMap<MODE>::RST + sbuf * BT * D * 2, BT * D * 2);
        tc::bulk_commit();
        tc::bulk_wait_all();
    }
    // the last two outputs (staged after the issuer's loop ended)
    if ((MODE & 1) && issuer && c1 > c0) {
        const int last = c1 - 1 - c0, lane = tid & 31;
        constexpr int OST = ScanMap<MODE>::OST;
        if (last >= 1 && pl == BT) fscan_tma_out(&tmo, sb + OST + ((last - 1) & 1) * BT * D * 2, pt, h, s.V, lane);
        if (t.chunk_len[c1 - 1] == BT)
            fscan_tma_out(&tmo, sb + OST + (last & 1) * BT * D * 2, t.chunk_tok0[c1 - 1], h, s.V, lane);
        if (lane == 0) tc::bulk_wait_all();
    }
    if (warp == 0) tc::tmem_dealloc(tb, 512);
}

template <int GATE, bool BWD, bool GD2, bool SHARE>
cudaError_t run_prep_k(const Shape& s, const void* q, const void* k, const void* v, const void* beta,
                       const float* g, Table t, FwdTC f, cudaStream_t st, const Gdn2& gd) {
    cudaError_t e = set_smem_once<k_prep_tc<GATE, BWD, GD2, SHARE>>(PREP_SMEM);
    if (e != cudaSuccess) return e;
    CUtensorMap mq, mk, mv, mg;
    memset(&mg, 0, sizeof(mg));
    // the inputs at their own widths K, V (<= D): the boxes' columns past them read as zeros
    // (q, k with heads_q(s) heads, g with heads_g(s))
    if (!tmap_rows_bf16(&mq, q, s.Ttot, heads_q(s), s.K) || !tmap_rows_bf16(&mk, k, s.Ttot, heads_q(s), s.K) ||
        !tmap_rows_bf16(&mv, v, s.Ttot, s.H, s.V) ||
        (GATE == 2 && !tmap_rows_f32(&mg, g, s.Ttot, heads_g(s), s.K, D)))
        return cudaErrorInvalidValue;
    // value blocks read in place (beta rule): one CTA per key unit, covering its Gg blocks
    dim3 grid(s.NC, SHARE ? s.H / s.Gg : s.H);
    k_prep_tc<GATE, BWD, GD2, SHARE><<<grid, PT, PREP_SMEM, st>>>(s, mq, mk, mv, mg, (const bf16*)beta, g, t, f, gd);
    return cudaGetLastError();
}

template <int GATE, bool BWD, bool GD2>
cudaError_t run_prep(const Shape& s, const void* q, const void* k, const void* v, const void* beta,
                     const float* g, Table t, FwdTC f, cudaStream_t st, const Gdn2& gd) {
    if constexpr (!GD2) {
        if (s.Gg > 1) return run_prep_k<GATE, BWD, false, true>(s, q, k, v, beta, g, t, f, st, gd);
    }
    return run_prep_k<GATE, BWD, GD2, false>(s, q, k, v, beta, g, t, f, st, gd);
}

template <int MODE>
cudaError_t run_scan(const Shape& s, const float* h0, Table t, FwdTC f, void* o, float* ht, cudaStream_t st) {
    cudaError_t e = set_smem_once<k_fwd_scan_tc<MODE>>(ScanMap<MODE>::SMEM);
    if (e != cudaSuccess) return e;
    CUtensorMap mo;
    memset(&mo, 0, sizeof(mo));
    if ((MODE & 1) && !tmap_rows_bf16(&mo, o, s.Ttot, s.H, s.V)) return cudaErrorInvalidValue;
    dim3 grid(s.N, s.H);
    k_fwd_scan_tc<MODE><<<grid, ST_ALL, ScanMap<MODE>::SMEM, st>>>(s, mo, h0, t, f, (bf16*)o, ht);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tc(const Shape& s, int gate, int for_bwd, const void* q, const void* k,
                           const void* v, const void* beta, const float* g, Table t, FwdTC f,
                           cudaStream_t st, const Gdn2& gd) {
    if (for_bwd) {
        switch (gate) {
            case 0: return (gd.erase ? run_prep<0, true, true>(s, q, k, v, beta, g, t, f, st, gd) : run_prep<0, true, false>(s, q, k, v, beta, g, t, f, st, gd));
            case 1: return (gd.erase ? run_prep<1, true, true>(s, q, k, v, beta, g, t, f, st, gd) : run_prep<1, true, false>(s, q, k, v, beta, g, t, f, st, gd));
            default: return (gd.erase ? run_prep<2, true, true>(s, q, k, v, beta, g, t, f, st, gd) : run_prep<2, true, false>(s, q, k, v, beta, g, t, f, st, gd));
        }
    }
    switch (gate) {
        case 0: return (gd.erase ? run_prep<0, false, true>(s, q, k, v, beta, g, t, f, st, gd) : run_prep<0, false, false>(s, q, k, v, beta, g, t, f, st, gd));
        case 1: return (gd.erase ? run_prep<1, false, true>(s, q, k, v, beta, g, t, f, st, gd) : run_prep<1, false, false>(s, q, k, v, beta, g, t, f, st, gd));
        default: return (gd.erase ? run_prep<2, false, true>(s, q, k, v, beta, g, t, f, st, gd) : run_prep<2, false, false>(s, q, k, v, beta, g, t, f, st, gd));
    }
}

cudaError_t launch_fwd_scan_tc(const Shape& s, int mode, const float* h0, Table t, FwdTC f, void* o,
                               float* ht, cudaStream_t st) {
    switch (mode) {
        case 1: return run_scan<1>(s, h0, t, f, o, ht, st);
        case 2: return run_scan<2>(s, h0, t, f, o, ht, st);
        default: return run_scan<3>(s, h0, t, f, o, ht, st);
    }
}

}  // namespace kda
