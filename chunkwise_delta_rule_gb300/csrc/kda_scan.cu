// Inter-chunk state scans, one CTA per (sequence, head, value tile), serial
// over the sequence's chunks; the state tile S[:, tile] stays in shared memory
// in fp32 for the whole sequence.
//
// Forward (a5 + a6; "ReWY" paper, "The chunk system and conventional WY
// backward"; "Kimi Delta Attention" blog, sections 6.4-6.5):
//     R = U - W S ;  O = Q_g S + C_q R ;  S <- diag(lambda) S + F^T R
// Reverse (a8; "ReWY" paper, "State and gate composition" and "Complete
// Reverse Execution and Boundaries"):
//     R_bar = C_q^T dO + F S+bar ;  P = A^T R_bar ;
//     S_bar <- diag(lambda) S+bar + Q_g^T dO - W^T R_bar
// where -W^T R_bar = -E^T P is the residual state term, supplied once here.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int VT = 32;  // value columns per CTA

// Key blocks: the [BT x D] operands (W, Q_g, F) are staged DK = min(D, 128) keys at a time in one
// [BT][DK] buffer, so that two CTAs share an SM at every width; the products over the key width
// add up block by block, the state update runs block by block over its rows. Row strides: the
// A operands of the products (W, Q_g, F, C_q, A) sit in rows of 16-byte aligned storage (DK + 4,
// BT + 4) so that they are read four elements per load; the B operands (S, U/R, dO, R_bar) in
// rows of VT + 1.
// (sequence, head, value tile) of this CTA from its linear index over the grid (N, H, D / VT):
// value tiles fastest, then heads, then sequences in the table's order (longest first).
__device__ __forceinline__ void cta_unit(const Table& t, int H, int& nseq, int& h, int& v0) {
    const int lin = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    const int nvt = (int)gridDim.z, rest = lin / nvt;
    v0 = (lin - rest * nvt) * VT;
    h = rest % H;
    nseq = t.seq_order[rest / H];
}

template <int D>
struct ScanDims {
    static constexpr int DK = D > 128 ? 128 : D;   // keys per staged block
    static constexpr int NKB = D / DK;             // key blocks
    static constexpr int LD = DK + 4, LV = VT + 1, LA = BT + 4;
};

template <typename TI, int D, int MODE>
__global__ void __launch_bounds__(NTHREADS, 2)
    k_fwd_scan(Shape s, const float* __restrict__ h0, Table t, Fwd f, TI* __restrict__ o,
               float* __restrict__ ht) {
    using SD = ScanDims<D>;
    constexpr int DK = SD::DK, NKB = SD::NKB, LD = SD::LD, LV = SD::LV, LA = SD::LA;
    extern __shared__ float smem[];
    float* sS = smem;             // [D][LV] state tile
    float* sM = sS + D * LV;      // [BT][LD] one key block of W, then Q_g, then F
    float* sR = sM + BT * LD;     // [BT][LV] U, then R
    float* sA = sR + BT * LV;     // [BT][LA] C_q
    float* sLam = sA + BT * LA;   // [D]

    const int H = s.H, tid = threadIdx.x;
    int nseq, h, v0;
    cta_unit(t, H, nseq, h, v0);
    const size_t st_off = ((size_t)nseq * H + h) * D * D;
    tile_copy<D, VT>([&](int r, int cc) { return h0 ? ldg(h0 + st_off + (size_t)r * D + v0 + cc) : 0.f; },
                     [&](int r, int cc, float x) { sS[r * LV + cc] = x; });
    const int c0 = t.seq_chunk0[nseq], c1 = t.seq_chunk0[nseq + 1];
    using TR = TileMap<BT, VT, 8, 1>;
    using TS = TileMapB<DK, VT, DK / 8, 1>;
    // one key block of a [BT][D] operand into sM
    auto stage = [&](const float* X, int kb) {
        tile_copy<BT, DK>([&](int r, int cc) { return ldg(X + r * D + kb * DK + cc); },
                          [&](int r, int cc, float x) { sM[r * LD + cc] = x; });
    };
    for (int c = c0; c < c1; ++c) {
        const size_t ch = (size_t)c * H + h;
        const int len = t.chunk_len[c], tok0 = t.chunk_tok0[c];
        const float* W = f.W + ch * BT * D;
        const float* U = f.U + ch * BT * D;
        tile_copy<BT, VT>([&](int r, int cc) { return ldg(U + (size_t)r * D + v0 + cc); },
                          [&](int r, int cc, float x) { sR[r * LV + cc] = x; });
        if (tid < D) sLam[tid] = exp2f(ldg(f.GL + ch * D + tid));
        // R = U - W S
        {
            float acc[8][1];
            zero(acc);
#pragma unroll 1
            for (int kb = 0; kb < NKB; ++kb) {
                if (kb > 0) __syncthreads();   // the previous block is read
                stage(W, kb);
                __syncthreads();
                tile_gemm_ar<BT, VT, 8, 1>(acc, sM, LD, 0, DK,
                                           [&](int kk, int nn) { return sS[(kb * DK + kk) * LV + nn]; });
            }
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                const int m = TR::row(ii), nn = TR::col(0);
                const float r = sR[m * LV + nn] - acc[ii][0];
                sR[m * LV + nn] = r;
                if (MODE & 2) f.R[ch * BT * D + (size_t)m * D + v0 + nn] = r;
            }
        }
        if (MODE & 2) {
            float* SIN = f.SIN + ch * D * D;
            for (int idx = tid; idx < D * VT; idx += NTHREADS) {
                const int r = idx / VT, cc = idx % VT;
                SIN[(size_t)r * D + v0 + cc] = sS[r * LV + cc];
            }
        }
        __syncthreads();
        if (MODE & 1) {
            const float* QG = f.QG + ch * BT * D;
            const float* AQK = f.AQK + ch * BT * BT;
            tile_copy<BT, BT>([&](int r, int cc) { return ldg(AQK + r * BT + cc); },
                              [&](int r, int cc, float x) { sA[r * LA + cc] = x; });
            float acc[8][1];
            zero(acc);
#pragma unroll 1
            for (int kb = 0; kb < NKB; ++kb) {
                if (kb > 0) __syncthreads();
                stage(QG, kb);
                __syncthreads();
                tile_gemm_ar<BT, VT, 8, 1>(acc, sM, LD, 0, DK,
                                           [&](int kk, int nn) { return sS[(kb * DK + kk) * LV + nn]; });
            }
            tile_gemm_ar<BT, VT, 8, 1>(acc, sA, LA, 0, BT, [&](int kk, int nn) { return sR[kk * LV + nn]; });
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                const int m = TR::row(ii), nn = TR::col(0);
                if (m < len) st(o + ((size_t)(tok0 + m) * H + h) * D + v0 + nn, acc[ii][0]);
            }
            __syncthreads();
        }
        // S <- diag(lambda) S + F^T R, one key block of rows at a time
        {
            const float* KG = f.KG + ch * BT * D;
#pragma unroll 1
            for (int kb = 0; kb < NKB; ++kb) {
                if (kb > 0) __syncthreads();
                stage(KG, kb);
                __syncthreads();
                float acc[DK / 8][1];
                zero(acc);
                tile_gemm_at<DK, VT, DK / 8, 1>(acc, sM, LD, 0, BT, [&](int kk, int nn) { return sR[kk * LV + nn]; });
#pragma unroll
                for (int ii = 0; ii < DK / 8; ++ii) {
                    const int m = kb * DK + TS::row(ii), nn = TS::col(0);
                    sS[m * LV + nn] = sLam[m] * sS[m * LV + nn] + acc[ii][0];
                }
            }
        }
        __syncthreads();
    }
    if (ht) {
        for (int idx = tid; idx < D * VT; idx += NTHREADS) {
            const int r = idx / VT, cc = idx % VT;
            ht[st_off + (size_t)r * D + v0 + cc] = sS[r * LV + cc];
        }
    }
}

template <typename TI, int D>
__global__ void __launch_bounds__(NTHREADS, 2)
    k_bwd_scan(Shape s, const TI* __restrict__ dout, const float* __restrict__ dht, Table t, Fwd f,
               Bwd b, float* __restrict__ dh0) {
    using SD = ScanDims<D>;
    constexpr int DK = SD::DK, NKB = SD::NKB, LD = SD::LD, LV = SD::LV, LA = SD::LA;
    extern __shared__ float smem[];
    float* sSb = smem;             // [D][LV] state adjoint tile
    float* sM = sSb + D * LV;      // [BT][LD] one key block of F, then Q_g, then W
    float* sO = sM + BT * LD;      // [BT][LV] dO tile
    float* sRb = sO + BT * LV;     // [BT][LV] R_bar
    float* sA = sRb + BT * LV;     // [BT][LA] C_q, then A
    float* sLam = sA + BT * LA;    // [D]

    const int H = s.H, tid = threadIdx.x;
    int nseq, h, v0;
    cta_unit(t, H, nseq, h, v0);
    const size_t st_off = ((size_t)nseq * H + h) * D * D;
    tile_copy<D, VT>([&](int r, int cc) { return dht ? ldg(dht + st_off + (size_t)r * D + v0 + cc) : 0.f; },
                     [&](int r, int cc, float x) { sSb[r * LV + cc] = x; });
    const int c0 = t.seq_chunk0[nseq], c1 = t.seq_chunk0[nseq + 1];
    using TR = TileMapB<BT, VT, 8, 1>;
    using TS = TileMapB<DK, VT, DK / 8, 1>;
    auto stage = [&](const float* X, int kb) {
        tile_copy<BT, DK>([&](int r, int cc) { return ldg(X + r * D + kb * DK + cc); },
                          [&](int r, int cc, float x) { sM[r * LD + cc] = x; });
    };
    for (int c = c1 - 1; c >= c0; --c) {
        const size_t ch = (size_t)c * H + h;
        const int len = t.chunk_len[c], tok0 = t.chunk_tok0[c];
        const float* KG = f.KG + ch * BT * D;
        const float* QG = f.QG + ch * BT * D;
        const float* W = f.W + ch * BT * D;
        {
            const float* AQK = f.AQK + ch * BT * BT;
            tile_copy<BT, BT>([&](int r, int cc) { return ldg(AQK + r * BT + cc); },
                              [&](int r, int cc, float x) { sA[r * LA + cc] = x; });
            tile_copy<BT, VT>(
                [&](int r, int cc) { return (r < len) ? ldg(dout + ((size_t)(tok0 + r) * H + h) * D + v0 + cc) : 0.f; },
                [&](int r, int cc, float x) { sO[r * LV + cc] = x; });
            if (tid < D) sLam[tid] = exp2f(ldg(f.GL + ch * D + tid));
        }
        // R_bar = C_q^T dO + F S+bar ; record S+bar for the consumers
        {
            float acc[8][1];
            zero(acc);
#pragma unroll 1
            for (int kb = 0; kb < NKB; ++kb) {
                if (kb > 0) __syncthreads();
                stage(KG, kb);
                __syncthreads();
                if (kb == 0)
                    tile_gemm_at<BT, VT, 8, 1>(acc, sA, LA, 0, BT, [&](int kk, int nn) { return sO[kk * LV + nn]; });
                tile_gemm_ar<BT, VT, 8, 1, true>(acc, sM, LD, 0, DK,
                                                 [&](int kk, int nn) { return sSb[(kb * DK + kk) * LV + nn]; });
            }
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) sRb[TR::row(ii) * LV + TR::col(0)] = acc[ii][0];
            float* SBP = b.SBP + ch * D * D;
            for (int idx = tid; idx < D * VT; idx += NTHREADS) {
                const int r = idx / VT, cc = idx % VT;
                SBP[(size_t)r * D + v0 + cc] = sSb[r * LV + cc];
            }
        }
        __syncthreads();
        {
            const float* AI = f.AINV + ch * BT * BT;
            tile_copy<BT, BT>([&](int r, int cc) { return ldg(AI + r * BT + cc); },
                              [&](int r, int cc, float x) { sA[r * LA + cc] = x; });
        }
        __syncthreads();
        // P = A^T R_bar
        {
            float acc[8][1];
            zero(acc);
            tile_gemm_at<BT, VT, 8, 1>(acc, sA, LA, 0, BT, [&](int kk, int nn) { return sRb[kk * LV + nn]; });
            float* P = b.P + ch * BT * D;
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) P[(size_t)TR::row(ii) * D + v0 + TR::col(0)] = acc[ii][0];
        }
        // S_bar = diag(lambda) S+bar + Q_g^T dO - W^T R_bar, one key block of rows at a time (Q_g
        // and W through the one staging buffer)
#pragma unroll 1
        for (int kb = 0; kb < NKB; ++kb) {
            float acc[DK / 8][1], acc2[DK / 8][1];
            zero(acc);
            zero(acc2);
            __syncthreads();
            stage(QG, kb);
            __syncthreads();
            tile_gemm_at<DK, VT, DK / 8, 1>(acc, sM, LD, 0, BT, [&](int kk, int nn) { return sO[kk * LV + nn]; });
            __syncthreads();
            stage(W, kb);
            __syncthreads();
            tile_gemm_at<DK, VT, DK / 8, 1>(acc2, sM, LD, 0, BT, [&](int kk, int nn) { return sRb[kk * LV + nn]; });
#pragma unroll
            for (int ii = 0; ii < DK / 8; ++ii) {
                const int m = kb * DK + TS::row(ii), nn = TS::col(0);
                sSb[m * LV + nn] = sLam[m] * sSb[m * LV + nn] + acc[ii][0] - acc2[ii][0];
            }
        }
        __syncthreads();
    }
    if (dh0) {
        for (int idx = tid; idx < D * VT; idx += NTHREADS) {
            const int r = idx / VT, cc = idx % VT;
            dh0[st_off + (size_t)r * D + v0 + cc] = sSb[r * LV + cc];
        }
    }
}

template <typename TI, int D, int MODE>
cudaError_t run_fwd(const Shape& s, const float* h0, Table t, Fwd f, void* o, float* ht, cudaStream_t st) {
    using SD = ScanDims<D>;
    constexpr size_t smem = sizeof(float) * (D * SD::LV + BT * SD::LD + BT * SD::LV + BT * SD::LA + D);
    auto kern = k_fwd_scan<TI, D, MODE>;
    cudaError_t e = set_smem_once<k_fwd_scan<TI, D, MODE>>(smem);
    if (e != cudaSuccess) return e;
    dim3 grid(s.N, s.H, D / VT);
    kern<<<grid, NTHREADS, smem, st>>>(s, h0, t, f, (TI*)o, ht);
    return cudaGetLastError();
}

template <typename TI, int D>
cudaError_t run_fwd_mode(int mode, const Shape& s, const float* h0, Table t, Fwd f, void* o,
                         float* ht, cudaStream_t st) {
    switch (mode) {
        case 1: return run_fwd<TI, D, 1>(s, h0, t, f, o, ht, st);
        case 2: return run_fwd<TI, D, 2>(s, h0, t, f, o, ht, st);
        default: return run_fwd<TI, D, 3>(s, h0, t, f, o, ht, st);
    }
}

template <typename TI, int D>
cudaError_t run_bwd(const Shape& s, const void* dout, const float* dht, Table t, Fwd f, Bwd b,
                    float* dh0, cudaStream_t st) {
    using SD = ScanDims<D>;
    constexpr size_t smem = sizeof(float) * (D * SD::LV + BT * SD::LD + 2 * BT * SD::LV + BT * SD::LA + D);
    auto kern = k_bwd_scan<TI, D>;
    cudaError_t e = set_smem_once<k_bwd_scan<TI, D>>(smem);
    if (e != cudaSuccess) return e;
    dim3 grid(s.N, s.H, D / VT);
    kern<<<grid, NTHREADS, smem, st>>>(s, (const TI*)dout, dht, t, f, b, dh0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_scan(const Shape& s, int io_bf16, int mode, const float* h0, Table t,
                            Fwd f, void* o, float* ht, cudaStream_t st) {
    if (s.K == 256)
        return io_bf16 ? run_fwd_mode<__nv_bfloat16, 256>(mode, s, h0, t, f, o, ht, st)
                       : run_fwd_mode<float, 256>(mode, s, h0, t, f, o, ht, st);
    if (s.K == 128)
        return io_bf16 ? run_fwd_mode<__nv_bfloat16, 128>(mode, s, h0, t, f, o, ht, st)
                       : run_fwd_mode<float, 128>(mode, s, h0, t, f, o, ht, st);
    return io_bf16 ? run_fwd_mode<__nv_bfloat16, 64>(mode, s, h0, t, f, o, ht, st)
                   : run_fwd_mode<float, 64>(mode, s, h0, t, f, o, ht, st);
}

cudaError_t launch_bwd_scan(const Shape& s, int io_bf16, const void* dout, const float* dht,
                            Table t, Fwd f, Bwd b, float* dh0, cudaStream_t st) {
    if (s.K == 256)
        return io_bf16 ? run_bwd<__nv_bfloat16, 256>(s, dout, dht, t, f, b, dh0, st)
                       : run_bwd<float, 256>(s, dout, dht, t, f, b, dh0, st);
    if (s.K == 128)
        return io_bf16 ? run_bwd<__nv_bfloat16, 128>(s, dout, dht, t, f, b, dh0, st)
                       : run_bwd<float, 128>(s, dout, dht, t, f, b, dh0, st);
    return io_bf16 ? run_bwd<__nv_bfloat16, 64>(s, dout, dht, t, f, b, dh0, st)
                   : run_bwd<float, 64>(s, dout, dht, t, f, b, dh0, st);
}

}  // namespace kda
