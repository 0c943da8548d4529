// Chunk-parallel forward preparation, one CTA per (chunk slot, head):
//   a1  in-chunk cumulative log2-decay G2 = cumsum(g) / ln 2 (exp2(G2) = exp(G))
//   a2  L = Akk = L_<(E Y^T) (strict) and C_q = Aqk = L_<=(Q_g Y^T) (inclusive)
//   a3  A = (I + L)^-1
//   a4  W = A E, U = A Z, F = keys decayed to the chunk end, Q_g
// ("ReWY" paper: "The chunk system and conventional WY backward"; "Kimi Delta
// Attention" blog, sections 6.3-6.6; GatedDeltaNet-2 spec transcription,
// sections 2.1-2.5 for the base-2 cumsum, the sub-chunk anchoring and the
// u/w auxiliaries).
//
// Numerics: the pairwise decay exp(G_i - G_j) is split into a row factor and
// a column factor anchored at the midpoint row of the receiving 16-token
// sub-chunk, so factors stay within exp(8 |g|max) and products never
// overflow; A is built in fp32 by column-parallel forward substitution.
#include "kda_internal.cuh"

namespace kda {
namespace {

// TCOUT: prepare only the chunks the tensor-core prep flagged as too wide for
// one anchor, and write the tensor-core path's layouts (bf16 tile images).
// Features are taken in column blocks of at most 128 (two passes at D = 256):
// the a2 contractions over the key width add up block by block, everything
// else is per feature.
template <typename TI, int D, int GATE, bool TCOUT>
__device__ __forceinline__ void prep_chunk(int c, int h, const Shape& s, const TI* __restrict__ q,
                                           const TI* __restrict__ k, const TI* __restrict__ v,
                                           const TI* __restrict__ beta, const float* __restrict__ g,
                                           const Table& t, const Fwd& f, const FwdTC& ft, const Gdn2& gd) {
    constexpr int DC = D > 128 ? 128 : D;   // feature columns per pass
    constexpr int NB = D / DC;              // passes
    // row strides of [BT x DC] and [BT x BT] tiles: 16-byte aligned rows, 4 mod 32 words, so that
    // the products read both operands four elements of the contraction per load
    constexpr int LD = DC + 4;
    constexpr int LA = BT + 4;
    extern __shared__ float smem[];
    float* sK = smem;               // [BT][LD] keys (fp32) of the column block
    float* sG = sK + BT * LD;       // [BT][LD] cumulative log2-decay
    float* sQ = sG + BT * LD;       // [BT][LD] queries, later beta*v
    float* sL = sQ + BT * LD;       // [2*BC][LD] row factors
    float* sR = sL + 2 * BC * LD;   // [BT][LD] column factors / E
    float* sAkk = sR + BT * LD;     // [BT][LA]
    float* sAi = sAkk + BT * LA;    // [BT][LA]
    float* sBeta = sAi + BT * LA;   // [BT]
    float* sAq = sBeta + BT;        // [BT][LA] C_q summed over the blocks (NB > 1 only)

    const int tid = threadIdx.x;
    const int n = t.chunk_len[c];
    if (n <= 0) return;
    const int tok0 = t.chunk_tok0[c];
    const int H = s.H;
    // heads of q, k and of g, beta, erase: grouped or per block only for the wide chunks of the
    // tensor-core path (D = 128); the CUDA-core path's inputs have one head per value head
    constexpr bool TCW = D == 128;
    const int hq = TCW ? h / s.Gq : h, Hq = TCW ? heads_q(s) : H, hg = TCW ? h / s.Gg : h, Hg = TCW ? heads_g(s) : H;
    const size_t ch = (size_t)c * H + h;

    if (tid < BT) sBeta[tid] = (tid < n && !gd.erase) ? ldg(beta + (size_t)(tok0 + tid) * Hg + hg) : 0.f;
    // GatedDeltaNet-2: the erase vector takes beta's place on the key rows of E. The token rows of
    // q, k, g and erase are K wide, those of v and write V wide (K = V = D but for the wide chunks
    // of the tensor-core path, whose inputs may be narrower than its 128 columns); columns past
    // them read as zeros.
    const int Kw = TCW ? s.K : D, Vw = TCW ? s.V : D;
    const TI* er = static_cast<const TI*>(gd.erase);
    auto ebeta = [&](int r, int gcol) {
        return er ? ((r < n && gcol < Kw) ? ld(er + ((size_t)(tok0 + r) * Hg + hg) * Kw + gcol) : 0.f) : sBeta[r];
    };
    // ---- chunk rows of features c0 .. c0+DC-1 (rows >= n are zero keys/queries
    // and zero decay), then a1: inclusive cumsum down each feature column
    // (padding rows keep G[n-1])
    auto load_block = [&](int c0) {
        auto offq = [&](int r, int col) { return ((size_t)(tok0 + r) * Hq + hq) * Kw + c0 + col; };
        auto offg = [&](int r, int col) { return ((size_t)(tok0 + r) * Hg + hg) * Kw + c0 + col; };
        tile_copy<BT, DC>([&](int r, int col) { return (r < n && c0 + col < Kw) ? ldg(k + offq(r, col)) : 0.f; },
                          [&](int r, int col, float x) { sK[r * LD + col] = x; });
        tile_copy<BT, DC>([&](int r, int col) { return (r < n && c0 + col < Kw) ? ldg(q + offq(r, col)) : 0.f; },
                          [&](int r, int col, float x) { sQ[r * LD + col] = x; });
        tile_copy<BT, DC>(
            [&](int r, int col) {
                if (GATE == 0 || r >= n) return 0.f;
                if (GATE == 2) return c0 + col < Kw ? ldg(g + offg(r, col)) * LOG2E : 0.f;
                return ldg(g + (size_t)(tok0 + r) * Hg + hg) * LOG2E;
            },
            [&](int r, int col, float x) { sG[r * LD + col] = x; });
        __syncthreads();
        if (tid < DC) {
            float acc = 0.f;
            for (int r = 0; r < BT; ++r) {
                acc += sG[r * LD + tid];
                sG[r * LD + tid] = acc;
            }
        }
        __syncthreads();
    };

    // ---- a2: Akk and Aqk, one 16-row sub-chunk of receiving rows at a time
    const float scale = s.scale;
    float* AQK = TCOUT ? nullptr : f.AQK + ch * BT * BT;
    auto put_aqk = [&](int i, int j, float x) {
        if (TCOUT) {
            ft.AQK[ch * BT * BT + tile_el(BT, i, j)] = __float2bfloat16_rn(x);
        } else {
            AQK[i * BT + j] = x;
        }
    };
    for (int cb = 0; cb < NB; ++cb) {
        const int c0 = cb * DC;
        if (cb > 0) __syncthreads();   // the previous block's tiles are no longer read
        load_block(c0);
        for (int b = 0; b < BT / BC; ++b) {
            const int ra = b * BC + BC / 2;          // anchor row (padding rows repeat G[n-1])
            const int ncol = (b + 1) * BC;           // columns j that can be <= i
            for (int idx = tid; idx < 2 * BC * DC; idx += NTHREADS) {
                const int r = idx / DC, col = idx % DC;
                const int i = b * BC + (r & (BC - 1));
                const float e = exp2f(sG[i * LD + col] - sG[ra * LD + col]);
                sL[r * LD + col] = (r < BC) ? ebeta(i, c0 + col) * sK[i * LD + col] * e : scale * sQ[i * LD + col] * e;
            }
            for (int idx = tid; idx < ncol * DC; idx += NTHREADS) {
                const int j = idx / DC, col = idx % DC;
                sR[j * LD + col] = sK[j * LD + col] * exp2f(sG[ra * LD + col] - sG[j * LD + col]);
            }
            __syncthreads();
            float acc[4][2];
            zero(acc);
            // columns j >= ncol read rows of sR this sub-chunk did not write: they lie above the
            // diagonal (j > i) and are masked out below
            tile_gemm_nt<2 * BC, BT, 4, 2>(acc, sL, LD, sR, LD, 0, DC);
            using TMp = TileMap<2 * BC, BT, 4, 2>;
            // a thread owns the same (i, j) entries in every pass, so the block sums need no barrier
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int r = TMp::row(ii), j = TMp::col(jj);
                    const int i = b * BC + (r & (BC - 1));
                    if (r < BC) {
                        const float x = (j < i && i < n) ? acc[ii][jj] : 0.f;
                        sAkk[i * LA + j] = cb == 0 ? x : sAkk[i * LA + j] + x;
                    } else {
                        const float x = (j <= i && i < n) ? acc[ii][jj] : 0.f;
                        if (NB == 1) {
                            put_aqk(i, j, x);
                        } else {
                            sAq[i * LA + j] = cb == 0 ? x : sAq[i * LA + j] + x;
                            if (cb == NB - 1) put_aqk(i, j, sAq[i * LA + j]);
                        }
                    }
                }
            }
            __syncthreads();
        }
    }

    // ---- a3: A = (I + Akk)^-1 by forward substitution; 4 lanes per column
    {
        const int col = tid >> 2, part = tid & 3;
        for (int r = part; r < BT; r += 4) sAi[r * LA + col] = (r == col) ? 1.f : 0.f;
        __syncwarp();
        for (int i = 1; i < BT; ++i) {
            float acc = 0.f;
            if (i > col) {
                for (int j = col + part; j < i; j += 4) acc = fmaf(sAkk[i * LA + j], sAi[j * LA + col], acc);
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0 && i > col) sAi[i * LA + col] = -acc;
            __syncwarp();
        }
    }
    __syncthreads();
    for (int idx = tid; idx < BT * BT; idx += NTHREADS) {
        const float a = sAi[(idx / BT) * LA + idx % BT];
        if (TCOUT) {
            if (ft.AI) ft.AI[ch * BT * BT + tile_el(BT, idx / BT, idx % BT)] = __float2bfloat16_rn(a);
        } else {
            f.AINV[ch * BT * BT + idx] = a;
        }
    }

    // ---- a4, per column block: Q_g, F (keys to chunk end), G at the last token,
    // W = A E and U = A Z
    constexpr int TN = DC / 32;
    using TM8 = TileMap<BT, DC, 8, TN>;
    for (int cb = 0; cb < NB; ++cb) {
        const int c0 = cb * DC;
        if (NB > 1) {
            __syncthreads();   // the previous block's tiles are no longer read
            load_block(c0);
        }
        const float* gl = sG + (n - 1) * LD;
        for (int idx = tid; idx < BT * DC; idx += NTHREADS) {
            const int r = idx / DC, col = idx % DC;
            const float gr = sG[r * LD + col];
            const float qg = scale * sQ[r * LD + col] * exp2f(gr);
            const float kg = sK[r * LD + col] * exp2f(gl[col] - gr);
            if (TCOUT) {
                ft.QG[ch * BT * D + tile_el(BT, r, c0 + col)] = __float2bfloat16_rn(qg);
                ft.KG[ch * BT * D + tile_el(BT, r, c0 + col)] = __float2bfloat16_rn(kg);
            } else {
                f.QG[ch * BT * D + (size_t)r * D + c0 + col] = qg;
                f.KG[ch * BT * D + (size_t)r * D + c0 + col] = kg;
            }
        }
        if (tid < DC) (TCOUT ? ft.GL : f.GL)[ch * D + c0 + tid] = gl[tid];
        // E = diag(beta) K exp(G) into sR; beta*v into sQ
        for (int idx = tid; idx < BT * DC; idx += NTHREADS) {
            const int r = idx / DC, col = idx % DC;
            sR[r * LD + col] = ebeta(r, c0 + col) * sK[r * LD + col] * exp2f(sG[r * LD + col]);
        }
        __syncthreads();  // all reads of sQ (queries) are done
        tile_copy<BT, DC>(
            [&](int r, int col) {
                if (r >= n || c0 + col >= Vw) return 0.f;
                const size_t off = ((size_t)(tok0 + r) * H + h) * Vw + c0 + col;
                const float wv = gd.write ? ldg(static_cast<const TI*>(gd.write) + off) : sBeta[r];
                return wv * ldg(v + off);
            },
            [&](int r, int col, float x) { sQ[r * LD + col] = x; });
        __syncthreads();
        {
            float acc[8][TN];
            zero(acc);
            tile_gemm_ar<BT, DC, 8, TN>(acc, sAi, LA, 0, BT, [&](int kk, int nn) { return sR[kk * LD + nn]; });
#pragma unroll
            for (int ii = 0; ii < 8; ++ii)
#pragma unroll
                for (int jj = 0; jj < TN; ++jj) {
                    const int r = TM8::row(ii), cl = c0 + TM8::col(jj);
                    if (TCOUT) {
                        ft.W[ch * BT * D + tile_el(BT, r, cl)] = __float2bfloat16_rn(acc[ii][jj]);
                    } else {
                        f.W[ch * BT * D + r * D + cl] = acc[ii][jj];
                    }
                }
        }
        {
            float acc[8][TN];
            zero(acc);
            tile_gemm_ar<BT, DC, 8, TN>(acc, sAi, LA, 0, BT, [&](int kk, int nn) { return sQ[kk * LD + nn]; });
#pragma unroll
            for (int ii = 0; ii < 8; ++ii)
#pragma unroll
                for (int jj = 0; jj < TN; ++jj) {
                    const size_t o = ch * BT * D + TM8::row(ii) * D + c0 + TM8::col(jj);
                    if (TCOUT) {
                        ft.U[o] = __float2bfloat16_rn(acc[ii][jj]);
                    } else {
                        f.U[o] = acc[ii][jj];
                    }
                }
        }
    }
}

// TCOUT: the chunks the tensor-core prep listed as wide, spread over a grid of
// one CTA per SM; otherwise one CTA per (chunk slot, head).
template <typename TI, int D, int GATE, bool TCOUT>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_prep(Shape s, const TI* __restrict__ q, const TI* __restrict__ k, const TI* __restrict__ v,
           const TI* __restrict__ beta, const float* __restrict__ g, Table t, Fwd f, FwdTC ft, Gdn2 gd) {
    if (TCOUT) {
        const int cnt = ft.WLIST[0];
        for (int w = blockIdx.x; w < cnt; w += gridDim.x) {
            const int ch = ft.WLIST[1 + w];
            prep_chunk<TI, D, GATE, TCOUT>(ch / s.H, ch % s.H, s, q, k, v, beta, g, t, f, ft, gd);
            __syncthreads();
        }
    } else {
        prep_chunk<TI, D, GATE, TCOUT>(blockIdx.x, blockIdx.y, s, q, k, v, beta, g, t, f, ft, gd);
    }
}

template <typename TI, int D, int GATE, bool TCOUT>
cudaError_t run(const Shape& s, const void* q, const void* k, const void* v, const void* beta,
                const float* g, Table t, Fwd f, FwdTC ft, cudaStream_t st, const Gdn2& gd = Gdn2{}) {
    constexpr int DC = D > 128 ? 128 : D, LD = DC + 4, LA = BT + 4;
    constexpr size_t smem = sizeof(float) * (4 * BT * LD + 2 * BC * LD + (D > DC ? 3 : 2) * BT * LA + BT);
    auto kern = k_prep<TI, D, GATE, TCOUT>;
    cudaError_t e = set_smem_once<k_prep<TI, D, GATE, TCOUT>>(smem);
    if (e != cudaSuccess) return e;
    const dim3 grid = TCOUT ? dim3(sm_count()) : dim3(s.NC, s.H);
    kern<<<grid, NTHREADS, smem, st>>>(s, (const TI*)q, (const TI*)k, (const TI*)v, (const TI*)beta, g, t, f, ft, gd);
    return cudaGetLastError();
}

template <typename TI, int D>
cudaError_t run_gate(int gate, const Shape& s, const void* q, const void* k, const void* v,
                     const void* beta, const float* g, Table t, Fwd f, cudaStream_t st, const Gdn2& gd) {
    FwdTC none{};
    switch (gate) {
        case 0: return run<TI, D, 0, false>(s, q, k, v, beta, g, t, f, none, st, gd);
        case 1: return run<TI, D, 1, false>(s, q, k, v, beta, g, t, f, none, st, gd);
        default: return run<TI, D, 2, false>(s, q, k, v, beta, g, t, f, none, st, gd);
    }
}

}  // namespace

cudaError_t launch_prep_wide(const Shape& s, int gate, const void* q, const void* k, const void* v,
                             const void* beta, const float* g, Table t, FwdTC ft, cudaStream_t st,
                             const Gdn2& gd) {
    Fwd none{};
    switch (gate) {
        case 0: return run<__nv_bfloat16, 128, 0, true>(s, q, k, v, beta, g, t, none, ft, st, gd);
        case 1: return run<__nv_bfloat16, 128, 1, true>(s, q, k, v, beta, g, t, none, ft, st, gd);
        default: return run<__nv_bfloat16, 128, 2, true>(s, q, k, v, beta, g, t, none, ft, st, gd);
    }
}

cudaError_t launch_prep(const Shape& s, int io_bf16, int gate, const void* q, const void* k,
                        const void* v, const void* beta, const float* g, Table t, Fwd f,
                        cudaStream_t st, const Gdn2& gd) {
    if (s.K == 256) {
        return io_bf16 ? run_gate<__nv_bfloat16, 256>(gate, s, q, k, v, beta, g, t, f, st, gd)
                       : run_gate<float, 256>(gate, s, q, k, v, beta, g, t, f, st, gd);
    }
    if (s.K == 128) {
        return io_bf16 ? run_gate<__nv_bfloat16, 128>(gate, s, q, k, v, beta, g, t, f, st, gd)
                       : run_gate<float, 128>(gate, s, q, k, v, beta, g, t, f, st, gd);
    }
    return io_bf16 ? run_gate<__nv_bfloat16, 64>(gate, s, q, k, v, beta, g, t, f, st, gd)
                   : run_gate<float, 64>(gate, s, q, k, v, beta, g, t, f, st, gd);
}

}  // namespace kda
