// Chunk-parallel backward consumers, one CTA per (chunk slot, head).
//
// k_bwd_dstate (a9 + a10, the contractions over the value width):
//     dv = beta P ; <v_i, P_i> ; D = -L_<(P R^T) ; H_q = L_<=(dO R^T) ;
//     dO S^T ; -P S^T ; F_bar = R S+bar^T ; rowsum(S .* S+bar)
// ("ReWY" paper, Algorithm 1 steps 2-3 and "Output, state, and
// effective-input gradients").
//
// k_bwd_intra (a11 / a11' + a12, the interaction contractions and chain rule):
//     gamma*Q_g_bar = gamma*(dO S^T) + gamma*(H_q Y)
//     gamma*E_bar   = gamma*(-P S^T) + gamma*(D Y)
//     Y_bar/gamma   = (D^T E + H_q^T Q_g)/gamma + F_bar*lambda/gamma
// with the pairwise decays factored as alpha = exp(G - c), zeta = exp(c - G)
// around the per-feature midpoint c of the chunk ("Matrix intra for
// vector-gated interactions", centered factors); chunks whose gate range
// exceeds the threshold use 16-token sub-chunks anchored so every factor is
// bounded; scalar gates fold exp(G_i - G_j) into D and H_q exactly and never
// form the key Gram matrix ("Gram elimination for scalar-gate gradients").
// Then dq = scale*gamma*Q_g_bar ; dk = beta*gamma*E_bar + Y_bar/gamma ;
// dbeta = <k_i, gamma*E_bar_i> + <v_i, P_i> (undivided, valid at beta = 0) ;
// G_bar = Q_g .* Q_g_bar + E .* E_bar - Y .* Y_bar plus the two state
// endpoints at the last valid token, and dg = reverse in-chunk cumsum of
// G_bar ("Complete Reverse Execution and Boundaries", steps 3-4).
#include "kda_internal.cuh"

namespace kda {
namespace {

using bf16 = __nv_bfloat16;

constexpr int SL = 32;  // value columns of S per slice in k_bwd_dstate

// IT: element type of the P, R, S and S+bar inputs: fp32 row-major here, bf16
// tile images (tile_el) when finishing the wide chunks of the tensor-core
// path, listed in `list`. Widths are taken in blocks of at most 128 (two at
// D = 256): the contractions over the value width add up over value blocks,
// the [BT x D] outputs are formed one key block at a time.
template <typename TI, typename IT, int D>
__device__ __forceinline__ void dstate_chunk(int c, int h, const Shape& s, const TI* __restrict__ dout,
                                             const TI* __restrict__ v, const TI* __restrict__ beta, const Table& t,
                                             const IT* __restrict__ Pin, const IT* __restrict__ Rin,
                                             const IT* __restrict__ Sin, const IT* __restrict__ SBin, const Bwd& b,
                                             TI* __restrict__ dv, const Gdn2& gd) {
    constexpr int DC = D > 128 ? 128 : D;   // columns per block
    constexpr int NB = D / DC;              // blocks
    // rows of 16-byte aligned storage (both operands of every product are read four elements of
    // the contraction per load), strides 4 mod 32 words
    constexpr int LD = DC + 4, LS = SL + 4;
    extern __shared__ float smem[];
    float* sO = smem;              // [BT][LD] dO, one value block
    float* sP = sO + BT * LD;      // [BT][LD] P
    float* sR = sP + BT * LD;      // [BT][LD] R
    float* sS = sR + BT * LD;      // [DC][LS] slice of S (one key block)
    float* sT = sS + DC * LS;      // [DC][LS] slice of S+bar

    const int tid = threadIdx.x;
    const int len = t.chunk_len[c];
    if (len <= 0) return;
    const int tok0 = t.chunk_tok0[c];
    const int H = s.H;
    constexpr bool TCW = D == 128;   // the tensor-core path's wide chunks (narrower rows, grouped heads)
    const int Vw = TCW ? s.V : D;   // token rows of dO, v, write and of dv, dwrite (V = D but for the wide chunks
                          // of the tensor-core path, whose rows may be narrower)
    const size_t ch = (size_t)c * H + h;
    const int lane = tid & 31, warp = tid >> 5;

    constexpr bool IMG = sizeof(IT) == 2;
    const IT* P = Pin + ch * BT * D;
    const IT* R = Rin + ch * BT * D;
    // dO, P and R of value columns v0 .. v0+DC-1
    auto load_block = [&](int v0) {
        auto e = [&](int r, int col) { return IMG ? tile_el(BT, r, v0 + col) : r * D + v0 + col; };
        tile_copy<BT, DC>(
            [&](int r, int col) {
                return (r < len && v0 + col < Vw) ? ldg(dout + ((size_t)(tok0 + r) * H + h) * Vw + v0 + col) : 0.f;
            },
            [&](int r, int col, float x) { sO[r * LD + col] = x; });
        tile_copy<BT, DC>([&](int r, int col) { return ldg(P + e(r, col)); },
                          [&](int r, int col, float x) { sP[r * LD + col] = x; });
        tile_copy<BT, DC>([&](int r, int col) { return ldg(R + e(r, col)); },
                          [&](int r, int col, float x) { sR[r * LD + col] = x; });
    };
    // ---- value-width contractions, value block by value block:
    // dv = beta P and <v_i, P_i>, one warp per row (GatedDeltaNet-2: dv = w .* P, dw = v .* P);
    // D = -L_<(P R^T), H_q = L_<=(dO R^T)
    {
        const TI* wr = static_cast<const TI*>(gd.write);
        constexpr int RW = BT / (NTHREADS / 32);   // rows per warp
        float dbw[RW];
#pragma unroll
        for (int i = 0; i < RW; ++i) dbw[i] = 0.f;
        using TMp = TileMap<BT, BT, 8, 2>;
        float acc[8][2], acc2[8][2];
        zero(acc);
        zero(acc2);
        for (int vb = 0; vb < NB; ++vb) {
            const int v0 = vb * DC;
            if (vb > 0) __syncthreads();   // the previous block's tiles are no longer read
            load_block(v0);
            __syncthreads();
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                const int r = warp + i * (NTHREADS / 32);
                if (r < len) {
                    const size_t tok = (size_t)(tok0 + r) * H + h;
                    const float bt = wr ? 0.f : ld(beta + (size_t)(tok0 + r) * (TCW ? heads_g(s) : H) + (TCW ? h / s.Gg : h));
                    for (int cc = lane; cc < DC; cc += 32) {
                        const int col = v0 + cc;
                        if (col >= Vw) break;
                        const float p = sP[r * LD + cc], vv = ld(v + tok * Vw + col);
                        if (wr) {
                            st(dv + tok * Vw + col, ld(wr + tok * Vw + col) * p);
                            st(static_cast<TI*>(gd.dwrite) + tok * Vw + col, vv * p);
                        } else {
                            dbw[i] = fmaf(vv, p, dbw[i]);
                            st(dv + tok * Vw + col, bt * p);
                        }
                    }
                }
            }
            tile_gemm_nt<BT, BT, 8, 2>(acc, sP, LD, sR, LD, 0, DC);
            tile_gemm_nt<BT, BT, 8, 2>(acc2, sO, LD, sR, LD, 0, DC);
        }
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            float x = dbw[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (lane == 0) b.DBW[ch * BT + warp + i * (NTHREADS / 32)] = x;
        }
        float* DM = b.DM + ch * BT * BT;
        float* HQ = b.HQ + ch * BT * BT;
#pragma unroll
        for (int ii = 0; ii < 8; ++ii)
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int m = TMp::row(ii), nn = TMp::col(jj);
                DM[m * BT + nn] = (nn < m) ? -acc[ii][jj] : 0.f;
                HQ[m * BT + nn] = (nn <= m) ? acc2[ii][jj] : 0.f;
            }
    }
    // ---- dO S^T, -P S^T, R S+bar^T and rowsum(S .* S+bar), one key block at a
    // time, summed over value slices
    constexpr int TN = DC / 32;
    using TK = TileMap<BT, DC, 8, TN>;
    constexpr int TPR = NTHREADS / DC;          // threads per key row for the rowsum
    const int kr = tid / TPR, kpart = tid % TPR;
    const IT* SIN = Sin + ch * D * D;
    const IT* SBP = SBin + ch * D * D;
    float* QS = b.QS + ch * BT * D;
    float* PS = b.PS + ch * BT * D;
    float* FB = b.FB + ch * BT * D;
    for (int kb = 0; kb < NB; ++kb) {
        const int k0 = kb * DC;
        float aQ[8][TN], aP[8][TN], aF[8][TN];
        zero(aQ);
        zero(aP);
        zero(aF);
        float lam = 0.f;
        for (int vb = 0; vb < NB; ++vb) {
            const int v0 = vb * DC;
            if (NB > 1) {
                __syncthreads();
                load_block(v0);
            }
            for (int vs = 0; vs < DC; vs += SL) {
                __syncthreads();
                auto e = [&](int r, int cc) {
                    return IMG ? (size_t)tile_el(D, k0 + r, v0 + vs + cc) : (size_t)(k0 + r) * D + v0 + vs + cc;
                };
                tile_copy<DC, SL>([&](int r, int cc) { return ldg(SIN + e(r, cc)); },
                                  [&](int r, int cc, float x) { sS[r * LS + cc] = x; });
                tile_copy<DC, SL>([&](int r, int cc) { return ldg(SBP + e(r, cc)); },
                                  [&](int r, int cc, float x) { sT[r * LS + cc] = x; });
                __syncthreads();
                tile_gemm_nt<BT, DC, 8, TN>(aQ, sO + vs, LD, sS, LS, 0, SL);
                tile_gemm_nt<BT, DC, 8, TN>(aP, sP + vs, LD, sS, LS, 0, SL);
                tile_gemm_nt<BT, DC, 8, TN>(aF, sR + vs, LD, sT, LS, 0, SL);
                for (int cc = kpart; cc < SL; cc += TPR) lam = fmaf(sS[kr * LS + cc], sT[kr * LS + cc], lam);
            }
        }
#pragma unroll
        for (int ii = 0; ii < 8; ++ii)
#pragma unroll
            for (int jj = 0; jj < TN; ++jj) {
                const size_t o = (size_t)TK::row(ii) * D + k0 + TK::col(jj);
                QS[o] = aQ[ii][jj];
                PS[o] = -aP[ii][jj];
                FB[o] = aF[ii][jj];
            }
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, o);
        if (kpart == 0) b.LAMB[ch * D + k0 + kr] = lam;
    }
}

// Features are taken in column blocks of at most 128 (two passes at D = 256);
// every contraction here runs over tokens, so the blocks are independent but
// for the per-row sums (dbeta, the scalar gate's G_bar), carried across them.
// The gate-range dispatch is made per block.
template <typename TI, int D, int GATE>
__device__ __forceinline__ void intra_chunk(int c, int h, const Shape& s, const TI* __restrict__ q,
                                            const TI* __restrict__ k, const TI* __restrict__ beta,
                                            const float* __restrict__ g, const Table& t, const Bwd& b,
                                            TI* __restrict__ dq, TI* __restrict__ dk, TI* __restrict__ dbeta,
                                            float* __restrict__ dg, const Gdn2& gd) {
    constexpr int DC = D > 128 ? 128 : D;   // feature columns per pass
    constexpr int NB = D / DC;              // passes
    constexpr int LD = DC + 1, LA = BT + 4;   // D and H_q rows 16-byte aligned (read four at a time)
    extern __shared__ float smem[];
    float* sK = smem;               // [BT][LD] keys of the column block
    float* sQ = sK + BT * LD;       // [BT][LD] queries
    float* sG = sQ + BT * LD;       // [BT][LD] cumulative log2-decay
    float* sF3 = sG + BT * LD;      // [BT][LD] operand
    float* sF4 = sF3 + BT * LD;     // [BT][LD] operand / G_bar
    float* sDM = sF4 + BT * LD;     // [BT][LA] D
    float* sHQ = sDM + BT * LA;     // [BT][LA] H_q
    float* sBeta = sHQ + BT * LA;   // [BT]
    float* sC = sBeta + BT;         // [DC] center of each feature
    float* sRow = sC + DC;          // [BT] per-row reductions

    const int tid = threadIdx.x;
    const int len = t.chunk_len[c];
    if (len <= 0) return;
    const int tok0 = t.chunk_tok0[c];
    const int H = s.H;
    constexpr bool TCW = D == 128;   // the tensor-core path's wide chunks (narrower rows, grouped heads)
    const int Kw = TCW ? s.K : D;   // token rows of q, k, g, erase and of dq, dk, dg, derase (K = D but for the
                          // wide chunks of the tensor-core path, whose rows may be narrower)
    const size_t ch = (size_t)c * H + h;
    const float scale = s.scale;
    const int lane = tid & 31, warp = tid >> 5;

    {
        const float* DM = b.DM + ch * BT * BT;
        const float* HQ = b.HQ + ch * BT * BT;
        tile_copy<BT, BT>([&](int r, int cc) { return ldg(DM + r * BT + cc); },
                          [&](int r, int cc, float x) { sDM[r * LA + cc] = x; });
        tile_copy<BT, BT>([&](int r, int cc) { return ldg(HQ + r * BT + cc); },
                          [&](int r, int cc, float x) { sHQ[r * LA + cc] = x; });
    }
    // heads of q, k and of g, beta, erase (value head h reads q, k of head h / Gq, the rest of h / Gg)
    const int hq = TCW ? h / s.Gq : h, Hq = TCW ? heads_q(s) : H, hg = TCW ? h / s.Gg : h, Hg = TCW ? heads_g(s) : H;
    if (tid < BT) sBeta[tid] = (tid < len && !gd.erase) ? ldg(beta + (size_t)(tok0 + tid) * Hg + hg) : 0.f;
    // GatedDeltaNet-2: the erase vector takes beta's place on the key side (E = b .* K exp(G))
    const TI* er = static_cast<const TI*>(gd.erase);
    auto ebeta = [&](int r, int gcol) {
        return er ? ((r < len && gcol < Kw) ? ld(er + ((size_t)(tok0 + r) * Hg + hg) * Kw + gcol) : 0.f) : sBeta[r];
    };
    const float* QS = b.QS + ch * BT * D;
    const float* PS = b.PS + ch * BT * D;
    const float* FB = b.FB + ch * BT * D;
    constexpr int TN = DC / 32;
    using TK = TileMap<BT, DC, 8, TN>;
    float rowacc[8];
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) rowacc[ii] = 0.f;

    for (int cb = 0; cb < NB; ++cb) {
        const int c0 = cb * DC;
        if (cb > 0) __syncthreads();   // the previous block's tiles are no longer read
        auto offq = [&](int r, int col) { return ((size_t)(tok0 + r) * Hq + hq) * Kw + c0 + col; };
        auto offg = [&](int r, int col) { return ((size_t)(tok0 + r) * Hg + hg) * Kw + c0 + col; };
        tile_copy<BT, DC>([&](int r, int col) { return (r < len && c0 + col < Kw) ? ldg(k + offq(r, col)) : 0.f; },
                          [&](int r, int col, float x) { sK[r * LD + col] = x; });
        tile_copy<BT, DC>([&](int r, int col) { return (r < len && c0 + col < Kw) ? ldg(q + offq(r, col)) : 0.f; },
                          [&](int r, int col, float x) { sQ[r * LD + col] = x; });
        tile_copy<BT, DC>(
            [&](int r, int col) {
                if (GATE == 0 || r >= len) return 0.f;
                if (GATE == 2) return c0 + col < Kw ? ldg(g + offg(r, col)) * LOG2E : 0.f;
                return ldg(g + (size_t)(tok0 + r) * Hg + hg) * LOG2E;
            },
            [&](int r, int col, float x) { sG[r * LD + col] = x; });
        __syncthreads();
        int wide_col = 0;
        if (tid < DC) {
            float acc = 0.f;
            for (int r = 0; r < BT; ++r) {
                acc += sG[r * LD + tid];
                sG[r * LD + tid] = acc;
            }
            float hi = sG[tid], lo = sG[tid];
            for (int r = 1; r < len; ++r) {
                hi = fmaxf(hi, sG[r * LD + tid]);
                lo = fminf(lo, sG[r * LD + tid]);
            }
            sC[tid] = (GATE == 2) ? 0.5f * (hi + lo) : 0.f;   // midpoint center
            wide_col = (GATE == 2) && (hi - lo > CENTER_RANGE_LOG2);
        }
        // gate-range dispatch: one wide feature sends the block to the sub-chunk path (per-channel
        // gates only, so that the other instantiations drop that path at compile time)
        bool wide = false;
        if (GATE == 2) {
            wide = __syncthreads_or(wide_col) != 0;
        } else {
            __syncthreads();
        }
        if (GATE == 1 && cb == 0) {
            // scalar gate: fold the exact pairwise decay exp(G_i - G_j) (<= 1) into D and H_q
            for (int idx = tid; idx < BT * BT; idx += NTHREADS) {
                const int i = idx / BT, j = idx % BT;
                if (j <= i) {
                    const float e = exp2f(sG[i * LD] - sG[j * LD]);
                    sDM[i * LA + j] *= e;
                    sHQ[i * LA + j] *= e;
                }
            }
            __syncthreads();
        }

        float aQ[8][TN], aE[8][TN], aY[8][TN];
        zero(aQ);
        zero(aE);
        zero(aY);
        // factors: unit for scalar / no gate (already folded), centered otherwise
        auto alpha = [&](int i, int col) { return GATE == 2 ? exp2f(sG[i * LD + col] - sC[col]) : 1.f; };
        auto zeta = [&](int i, int col) { return GATE == 2 ? exp2f(sC[col] - sG[i * LD + col]) : 1.f; };

        if (!wide) {
            // T_q = H_q (K zeta), T_e = D (K zeta)
            for (int idx = tid; idx < BT * DC; idx += NTHREADS) {
                const int r = idx / DC, col = idx % DC;
                sF3[r * LD + col] = sK[r * LD + col] * zeta(r, col);
            }
            __syncthreads();
            tile_gemm_ar<BT, DC, 8, TN>(aQ, sHQ, LA, 0, BT, [&](int kk, int nn) { return sF3[kk * LD + nn]; });
            tile_gemm_ar<BT, DC, 8, TN>(aE, sDM, LA, 0, BT, [&](int kk, int nn) { return sF3[kk * LD + nn]; });
#pragma unroll
            for (int ii = 0; ii < 8; ++ii)
#pragma unroll
                for (int jj = 0; jj < TN; ++jj) {
                    const float a = alpha(TK::row(ii), TK::col(jj));
                    aQ[ii][jj] *= a;
                    aE[ii][jj] *= a;
                }
            __syncthreads();
            // T_y = D^T (beta K alpha) + H_q^T (scale Q alpha)
            for (int idx = tid; idx < BT * DC; idx += NTHREADS) {
                const int r = idx / DC, col = idx % DC;
                const float a = alpha(r, col);
                sF3[r * LD + col] = ebeta(r, c0 + col) * sK[r * LD + col] * a;
                sF4[r * LD + col] = scale * sQ[r * LD + col] * a;
            }
            __syncthreads();
            tile_gemm<BT, DC, 8, TN>(aY, 0, BT, [&](int m, int kk) { return sDM[kk * LA + m]; },
                                     [&](int kk, int nn) { return sF3[kk * LD + nn]; });
            tile_gemm<BT, DC, 8, TN>(aY, 0, BT, [&](int m, int kk) { return sHQ[kk * LA + m]; },
                                     [&](int kk, int nn) { return sF4[kk * LD + nn]; });
#pragma unroll
            for (int ii = 0; ii < 8; ++ii)
#pragma unroll
                for (int jj = 0; jj < TN; ++jj) aY[ii][jj] *= zeta(TK::row(ii), TK::col(jj));
        } else {
            // Strong gates: 16-token sub-chunks. Receiving rows i of sub-chunk sb
            // take earlier sub-chunks with the anchor G at the first row of sb
            // (both factors <= 1) and the diagonal block with its midpoint row.
            // A thread's rows in sub-chunk sb are TK::row(2 sb) and TK::row(2 sb + 1).
            const int tm = TK::tm(), tn = TK::tn();
            for (int sb = 0; sb < BT / BC; ++sb) {
                if (sb * BC >= len) break;
                const int ra = sb * BC, rm = sb * BC + BC / 2;
                __syncthreads();
                for (int idx = tid; idx < BT * DC; idx += NTHREADS) {
                    const int j = idx / DC, col = idx % DC;
                    float val = 0.f;
                    if (j < ra) val = sK[j * LD + col] * exp2f(sG[ra * LD + col] - sG[j * LD + col]);
                    else if (j < ra + BC) val = sK[j * LD + col] * exp2f(sG[rm * LD + col] - sG[j * LD + col]);
                    sF3[j * LD + col] = val;
                }
                __syncthreads();
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const float* Mx = which == 0 ? sHQ : sDM;
                    float off[2][TN], dia[2][TN];
                    zero(off);
                    zero(dia);
                    for (int kk = 0; kk < ra + BC; ++kk) {
                        float a[2], bv[TN];
#pragma unroll
                        for (int r = 0; r < 2; ++r) a[r] = Mx[(tm + 8 * (2 * sb + r)) * LA + kk];
#pragma unroll
                        for (int jj = 0; jj < TN; ++jj) bv[jj] = sF3[kk * LD + tn + 32 * jj];
#pragma unroll
                        for (int r = 0; r < 2; ++r)
#pragma unroll
                            for (int jj = 0; jj < TN; ++jj) {
                                if (kk < ra) off[r][jj] = fmaf(a[r], bv[jj], off[r][jj]);
                                else dia[r][jj] = fmaf(a[r], bv[jj], dia[r][jj]);
                            }
                    }
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int i = tm + 8 * (2 * sb + r);
#pragma unroll
                        for (int jj = 0; jj < TN; ++jj) {
                            const int col = tn + 32 * jj;
                            const float gi = sG[i * LD + col];
                            const float val = exp2f(gi - sG[ra * LD + col]) * off[r][jj] +
                                              exp2f(gi - sG[rm * LD + col]) * dia[r][jj];
                            if (which == 0) aQ[2 * sb + r][jj] = val;
                            else aE[2 * sb + r][jj] = val;
                        }
                    }
                }
            }
            // Transposed contractions: output rows j of sub-chunk sb; summed rows i
            // of later sub-chunks use the anchor G at the last row of sb, the
            // diagonal block its midpoint row.
            for (int sb = 0; sb < BT / BC; ++sb) {
                if (sb * BC >= len) break;
                const int ra = sb * BC, re = sb * BC + BC - 1, rm = sb * BC + BC / 2;
                __syncthreads();
                for (int idx = tid; idx < BT * DC; idx += NTHREADS) {
                    const int i = idx / DC, col = idx % DC;
                    float e = 0.f;
                    if (i >= ra + BC) e = exp2f(sG[i * LD + col] - sG[re * LD + col]);
                    else if (i >= ra) e = exp2f(sG[i * LD + col] - sG[rm * LD + col]);
                    sF3[i * LD + col] = ebeta(i, c0 + col) * sK[i * LD + col] * e;
                    sF4[i * LD + col] = scale * sQ[i * LD + col] * e;
                }
                __syncthreads();
                float off[2][TN], dia[2][TN];
                zero(off);
                zero(dia);
                for (int kk = ra; kk < BT; ++kk) {
                    float a1[2], a2[2], b1[TN], b2[TN];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int j = tm + 8 * (2 * sb + r);
                        a1[r] = sDM[kk * LA + j];
                        a2[r] = sHQ[kk * LA + j];
                    }
#pragma unroll
                    for (int jj = 0; jj < TN; ++jj) {
                        b1[jj] = sF3[kk * LD + tn + 32 * jj];
                        b2[jj] = sF4[kk * LD + tn + 32 * jj];
                    }
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int jj = 0; jj < TN; ++jj) {
                            const float x = fmaf(a1[r], b1[jj], a2[r] * b2[jj]);
                            if (kk >= ra + BC) off[r][jj] += x;
                            else dia[r][jj] += x;
                        }
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int j = tm + 8 * (2 * sb + r);
#pragma unroll
                    for (int jj = 0; jj < TN; ++jj) {
                        const int col = tn + 32 * jj;
                        const float gj = sG[j * LD + col];
                        aY[2 * sb + r][jj] = exp2f(sG[re * LD + col] - gj) * off[r][jj] +
                                             exp2f(sG[rm * LD + col] - gj) * dia[r][jj];
                    }
                }
            }
        }
        __syncthreads();  // operand buffers free from here on

        // ---- chain rule (a12) for the block's features
        const float* gl2 = sG + (len - 1) * LD;
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
            const int m = TK::row(ii);
#pragma unroll
            for (int jj = 0; jj < TN; ++jj) {
                const int col = TK::col(jj);
                const size_t o = (size_t)m * D + c0 + col;
                const float gm = sG[m * LD + col];
                const float gam = exp2f(gm);
                const float Qt = aQ[ii][jj] + gam * QS[o];                    // gamma * Q_g_bar
                const float Et = aE[ii][jj] + gam * PS[o];                    // gamma * E_bar
                const float Yt = aY[ii][jj] + FB[o] * exp2f(gl2[col] - gm);   // Y_bar / gamma
                const float kv = sK[m * LD + col], qv = sQ[m * LD + col], bt = ebeta(m, c0 + col);
                if (m < len && c0 + col < Kw) {
                    const size_t go = ((size_t)(tok0 + m) * H + h) * Kw + c0 + col;
                    st(dq + go, scale * Qt);
                    st(dk + go, bt * Et + Yt);
                    if (er) st(static_cast<TI*>(gd.derase) + go, kv * Et);   // db = K exp(G) .* E_bar
                }
                rowacc[ii] = fmaf(kv, Et, rowacc[ii]);
                sF4[m * LD + col] = scale * qv * Qt + bt * kv * Et - kv * Yt;  // G_bar
            }
        }
        if (GATE == 0) continue;
        __syncthreads();
        // state endpoints at the last valid token: lambda*rowsum(S.*S+bar) + sum_i F_i .* F_bar_i
        if (tid < DC) {
            const float glc = gl2[tid];
            float e = exp2f(glc) * b.LAMB[ch * D + c0 + tid];
            for (int i = 0; i < len; ++i)
                e = fmaf(sK[i * LD + tid] * exp2f(glc - sG[i * LD + tid]), FB[(size_t)i * D + c0 + tid], e);
            sF4[(len - 1) * LD + tid] += e;
        }
        __syncthreads();
        if (GATE == 2) {
            if (tid < DC) {
                float acc = 0.f;
                for (int r = len - 1; r >= 0; --r) {
                    acc += sF4[r * LD + tid];
                    if (c0 + tid < Kw) dg[((size_t)(tok0 + r) * H + h) * Kw + c0 + tid] = acc;
                }
            }
        } else {
            // scalar gate: G_bar summed over the features of every block, per row
            for (int r = warp; r < BT; r += NTHREADS / 32) {
                float x = 0.f;
                for (int col = lane; col < DC; col += 32) x += sF4[r * LD + col];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                if (lane == 0) sRow[r] = cb == 0 ? x : sRow[r] + x;
            }
        }
    }
    // dbeta = <k_i, gamma E_bar_i> + <v_i, P_i>; a warp owns whole rows (TNX = 32)
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
        float x = rowacc[ii];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        const int m = TK::row(ii);
        if (lane == 0 && m < len && !er)
            st(dbeta + (size_t)(tok0 + m) * H + h, x + b.DBW[ch * BT + m]);
    }
    if (GATE == 1) {
        // scalar gate: reverse cumsum of the row sums
        __syncthreads();
        if (tid == 0) {
            float acc = 0.f;
            for (int r = len - 1; r >= 0; --r) {
                acc += sRow[r];
                dg[(size_t)(tok0 + r) * H + h] = acc;
            }
        }
    }
}

// One CTA per (chunk slot, head).
template <typename TI, typename IT, int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_bwd_dstate(Shape s, const TI* __restrict__ dout, const TI* __restrict__ v,
                 const TI* __restrict__ beta, Table t, const IT* __restrict__ Pin,
                 const IT* __restrict__ Rin, const IT* __restrict__ Sin, const IT* __restrict__ SBin,
                 Bwd b, TI* __restrict__ dv, Gdn2 gd) {
    dstate_chunk<TI, IT, D>(blockIdx.x, blockIdx.y, s, dout, v, beta, t, Pin, Rin, Sin, SBin, b, dv, gd);
}

template <typename TI, int D, int GATE>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_bwd_intra(Shape s, const TI* __restrict__ q, const TI* __restrict__ k,
                const TI* __restrict__ beta, const float* __restrict__ g, Table t,
                Bwd b, TI* __restrict__ dq, TI* __restrict__ dk,
                TI* __restrict__ dbeta, float* __restrict__ dg, Gdn2 gd) {
    intra_chunk<TI, D, GATE>(blockIdx.x, blockIdx.y, s, q, k, beta, g, t, b, dq, dk, dbeta, dg, gd);
}

// The chunks the tensor-core prep listed as wide (count, then chunk slot * H + head), spread over
// a grid of one CTA per SM: for each, the state-gradient pass and then the intra pass, which reads
// what the first wrote for that chunk (made visible within the CTA by the barrier between them).
template <int GATE>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_bwd_wide(Shape s, const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
               const bf16* __restrict__ beta, const float* __restrict__ g, const bf16* __restrict__ dout, Table t,
               const bf16* __restrict__ Pin, const bf16* __restrict__ Rin, const bf16* __restrict__ Sin,
               const bf16* __restrict__ SBin, const int32_t* __restrict__ list, Bwd b, bf16* __restrict__ dq,
               bf16* __restrict__ dk, bf16* __restrict__ dv, bf16* __restrict__ dbeta, float* __restrict__ dg,
               Gdn2 gd) {
    const int cnt = list[0];
    for (int w = blockIdx.x; w < cnt; w += gridDim.x) {
        const int ch = list[1 + w];
        dstate_chunk<bf16, bf16, 128>(ch / s.H, ch % s.H, s, dout, v, beta, t, Pin, Rin, Sin, SBin, b, dv, gd);
        __syncthreads();
        intra_chunk<bf16, 128, GATE>(ch / s.H, ch % s.H, s, q, k, beta, g, t, b, dq, dk, dbeta, dg, gd);
        __syncthreads();
    }
}

// Shared memory of the two passes (floats): the state-gradient pass's tiles and the intra pass's.
template <int D>
constexpr size_t dstate_smem() {
    constexpr int DC = D > 128 ? 128 : D, LD = DC + 4, LS = SL + 4;
    return sizeof(float) * (3 * BT * LD + 2 * DC * LS);
}
template <int D>
constexpr size_t intra_smem() {
    constexpr int DC = D > 128 ? 128 : D, LD = DC + 1, LA = BT + 4;
    return sizeof(float) * (5 * BT * LD + 2 * BT * LA + 2 * BT + DC);
}

template <typename TI, typename IT, int D>
cudaError_t run_dstate(const Shape& s, const void* dout, const void* v, const void* beta, Table t,
                       const IT* P, const IT* R, const IT* S, const IT* SB, Bwd b,
                       void* dv, cudaStream_t st, const Gdn2& gd = Gdn2{}) {
    constexpr size_t smem = dstate_smem<D>();
    auto kern = k_bwd_dstate<TI, IT, D>;
    cudaError_t e = set_smem_once<k_bwd_dstate<TI, IT, D>>(smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(s.NC, s.H), NTHREADS, smem, st>>>(s, (const TI*)dout, (const TI*)v, (const TI*)beta, t, P, R, S, SB,
                                                  b, (TI*)dv, gd);
    return cudaGetLastError();
}

template <typename TI, int D, int GATE>
cudaError_t run_intra(const Shape& s, const void* q, const void* k, const void* beta, const float* g,
                      Table t, Bwd b, void* dq, void* dk, void* dbeta, float* dg,
                      cudaStream_t st, const Gdn2& gd) {
    constexpr size_t smem = intra_smem<D>();
    auto kern = k_bwd_intra<TI, D, GATE>;
    cudaError_t e = set_smem_once<k_bwd_intra<TI, D, GATE>>(smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(s.NC, s.H), NTHREADS, smem, st>>>(s, (const TI*)q, (const TI*)k, (const TI*)beta, g, t, b,
                                                  (TI*)dq, (TI*)dk, (TI*)dbeta, dg, gd);
    return cudaGetLastError();
}

template <typename TI, int D>
cudaError_t run_intra_gate(int gate, const Shape& s, const void* q, const void* k, const void* beta,
                           const float* g, Table t, Bwd b, void* dq, void* dk,
                           void* dbeta, float* dg, cudaStream_t st, const Gdn2& gd = Gdn2{}) {
    switch (gate) {
        case 0: return run_intra<TI, D, 0>(s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd);
        case 1: return run_intra<TI, D, 1>(s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd);
        default: return run_intra<TI, D, 2>(s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd);
    }
}

template <int GATE>
cudaError_t run_wide(const Shape& s, const void* q, const void* k, const void* v, const void* beta, const float* g,
                     const void* dout, Table t, FwdTC f, BwdTC bt, Bwd b, void* dq, void* dk, void* dv, void* dbeta,
                     float* dg, cudaStream_t st, const Gdn2& gd) {
    constexpr size_t smem = dstate_smem<128>() > intra_smem<128>() ? dstate_smem<128>() : intra_smem<128>();
    cudaError_t e = set_smem_once<k_bwd_wide<GATE>>(smem);
    if (e != cudaSuccess) return e;
    k_bwd_wide<GATE><<<sm_count(), NTHREADS, smem, st>>>(
        s, (const bf16*)q, (const bf16*)k, (const bf16*)v, (const bf16*)beta, g, (const bf16*)dout, t, bt.P, f.R, f.HS,
        bt.SBP, f.WLIST, b, (bf16*)dq, (bf16*)dk, (bf16*)dv, (bf16*)dbeta, dg, gd);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dstate(const Shape& s, int io_bf16, const void* dout, const void* v,
                              const void* beta, Table t, Fwd f, Bwd b, void* dv, cudaStream_t st, const Gdn2& gd) {
    if (s.K == 256)
        return io_bf16 ? run_dstate<__nv_bfloat16, float, 256>(s, dout, v, beta, t, b.P, f.R, f.SIN, b.SBP, b, dv, st, gd)
                       : run_dstate<float, float, 256>(s, dout, v, beta, t, b.P, f.R, f.SIN, b.SBP, b, dv, st, gd);
    if (s.K == 128)
        return io_bf16 ? run_dstate<__nv_bfloat16, float, 128>(s, dout, v, beta, t, b.P, f.R, f.SIN, b.SBP, b, dv, st, gd)
                       : run_dstate<float, float, 128>(s, dout, v, beta, t, b.P, f.R, f.SIN, b.SBP, b, dv, st, gd);
    return io_bf16 ? run_dstate<__nv_bfloat16, float, 64>(s, dout, v, beta, t, b.P, f.R, f.SIN, b.SBP, b, dv, st, gd)
                   : run_dstate<float, float, 64>(s, dout, v, beta, t, b.P, f.R, f.SIN, b.SBP, b, dv, st, gd);
}

cudaError_t launch_bwd_intra(const Shape& s, int io_bf16, int gate, const void* q, const void* k,
                             const void* beta, const float* g, Table t, Fwd f, Bwd b, void* dq,
                             void* dk, void* dbeta, float* dg, cudaStream_t st, const Gdn2& gd) {
    (void)f;
    if (s.K == 256)
        return io_bf16 ? run_intra_gate<__nv_bfloat16, 256>(gate, s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd)
                       : run_intra_gate<float, 256>(gate, s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd);
    if (s.K == 128)
        return io_bf16 ? run_intra_gate<__nv_bfloat16, 128>(gate, s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd)
                       : run_intra_gate<float, 128>(gate, s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd);
    return io_bf16 ? run_intra_gate<__nv_bfloat16, 64>(gate, s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd)
                   : run_intra_gate<float, 64>(gate, s, q, k, beta, g, t, b, dq, dk, dbeta, dg, st, gd);
}

cudaError_t launch_bwd_wide(const Shape& s, int gate, const void* q, const void* k, const void* v,
                            const void* beta, const float* g, const void* dout, Table t, FwdTC f,
                            BwdTC bt, Bwd scratch, void* dq, void* dk, void* dv, void* dbeta, float* dg,
                            cudaStream_t st, const Gdn2& gd) {
    switch (gate) {
        case 0: return run_wide<0>(s, q, k, v, beta, g, dout, t, f, bt, scratch, dq, dk, dv, dbeta, dg, st, gd);
        case 1: return run_wide<1>(s, q, k, v, beta, g, dout, t, f, bt, scratch, dq, dk, dv, dbeta, dg, st, gd);
        default: return run_wide<2>(s, q, k, v, beta, g, dout, t, f, bt, scratch, dq, dk, dv, dbeta, dg, st, gd);
    }
}

}  // namespace kda
