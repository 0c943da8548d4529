// Tensor-core forward path (bf16 I/O, K = V = 128) on tcgen05.
//
// k_prep_tc, one CTA per (chunk slot, head) (a1-a4):
//   G2 = in-chunk cumsum of g / ln 2; one anchor c per feature (the midpoint
//   of the chunk's range) so that
//       [Akk ; Aqk] = [beta K 2^(G2-c) ; s Q 2^(G2-c)] (K 2^(c-G2))^T
//   is a single M = 128, N = 64, K = 128 tf32 MMA ("Kimi Delta Attention"
//   blog, sections 6.3 and 6.5; "ReWY" paper, centered factors); strict /
//   inclusive masks on the TMEM read-back; A = (I + Akk)^-1 in fp32 by
//   forward substitution; W^T = E^T A^T and U^T = Z^T A^T as two M = 128 tf32
//   MMAs. A chunk whose gate range exceeds 2^80 is left to the CUDA-core prep
//   (flag WIDE), which anchors per 16-token sub-chunk instead.
//
// k_fwd_scan_tc, one CTA per (sequence, head), 128 threads, thread v owns
// value column v (TMEM lane v). The transposed state S^T (V x K, fp32) stays
// in TMEM for the whole sequence. Per chunk (a5, a6):
//       R^T  = U^T - S^T W^T            (MMA, bf16 S^T staged in smem)
//       O^T  = S^T Q_g^T + R^T C_q^T    (MMAs, output fused)
//       S^T <- S^T diag(lambda) + R^T F (lambda applied in TMEM, then MMA)
// ("ReWY" paper, "The chunk system and conventional WY backward"; "Kimi Delta
// Attention" blog, section 6.4). Operands of chunk c+1 are prefetched with
// cp.async while chunk c computes.
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
constexpr int PT = 512;
constexpr int LG = D + 1;  // padded row stride of fp32 [64 x 128] tiles
constexpr int LA = BT + 1;
constexpr int LW = D + 8;   // row stride (bf16) of the staged W tile
constexpr int LU = D + 4;   // row stride (fp32) of the staged U tile
constexpr int LQ = BT + 8;  // row stride (bf16) of the staged C_q tile

// Blocked inverse of the unit lower-triangular M = I + L (64 x 64, L strict,
// fp32): the four 16 x 16 diagonal blocks by forward substitution (4 lanes per
// column), then the off-diagonal blocks level by level,
//     A_ij = -A_ii * sum_{m=j}^{i-1} L_im A_mj,
// the 4 x 4 block merge of the GatedDeltaNet-2 spec transcription (section 2.4).
__device__ __forceinline__ void blocked_inverse(const float* sL, float* sA, float* sT, int tid) {
    if (tid < 4 * BT) {  // whole warps: 64 threads per diagonal block, 4 lanes per column
        const int blk = tid >> 6, col = (tid >> 2) & 15, part = tid & 3;
        const int o = blk * BC;
        for (int r = part; r < BT; r += 4) sA[r * LA + o + col] = 0.f;
        for (int r = part; r < BC; r += 4) sA[(o + r) * LA + o + col] = (r == col) ? 1.f : 0.f;
        __syncwarp();
        for (int i = 1; i < BC; ++i) {
            float acc = 0.f;
            if (i > col)
                for (int j = col + part; j < i; j += 4) acc = fmaf(sL[(o + i) * LA + o + j], sA[(o + j) * LA + o + col], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0 && i > col) sA[(o + i) * LA + o + col] = -acc;
            __syncwarp();
        }
    }
    __syncthreads();
    for (int lvl = 1; lvl < BT / BC; ++lvl) {
        const int nb = BT / BC - lvl;  // blocks (i, j = i - lvl) on this level
        // T_ij = sum_{m=j}^{i-1} L_im A_mj
        for (int idx = tid; idx < nb * BC * BC; idx += PT) {
            const int b = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
            const int j = b, i = b + lvl;
            float acc = 0.f;
            for (int m = j; m < i; ++m)
#pragma unroll
                for (int x = 0; x < BC; ++x)
                    acc = fmaf(sL[(i * BC + r) * LA + m * BC + x], sA[(m * BC + x) * LA + j * BC + cc], acc);
            sT[(b * BC + r) * (BC + 1) + cc] = acc;
        }
        __syncthreads();
        // A_ij = -A_ii T_ij
        for (int idx = tid; idx < nb * BC * BC; idx += PT) {
            const int b = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
            const int j = b, i = b + lvl;
            float acc = 0.f;
#pragma unroll
            for (int x = 0; x < BC; ++x) acc = fmaf(sA[(i * BC + r) * LA + i * BC + x], sT[(b * BC + x) * (BC + 1) + cc], acc);
            sA[(i * BC + r) * LA + j * BC + cc] = -acc;
        }
        __syncthreads();
    }
}

template <int GATE, bool BWD>
__global__ void __launch_bounds__(PT, 1)
    k_prep_tc(Shape s, const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
              const bf16* __restrict__ beta, const float* __restrict__ g, Table t, FwdTC f) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    unsigned char* R1 = base;             // 64 KB operand region (1024-aligned)
    unsigned char* R2 = R1 + 65536;       // 32 KB operand region
    float* sA = reinterpret_cast<float*>(R2 + 32768);  // [64][129] G2, then alpha = 2^(G2 - c)
    bf16* sK = reinterpret_cast<bf16*>(sA + BT * LG);  // [64][128] keys
    bf16* sQ = sK + BT * D;                             // [64][128] queries
    float* sAkk = reinterpret_cast<float*>(sQ + BT * D);  // [64][65]
    float* sAi = sAkk + BT * LA;          // [64][65]
    float* sT = sAi + BT * LA;            // [3][16][17] merge temporaries
    float* sBeta = sT + 3 * BC * (BC + 1);  // [64]
    float* sC2 = sBeta + BT;              // [128] 2^c (c = midpoint anchor of the feature)
    float* sAL = sC2 + D;                 // [128] 2^(G2_last - c)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sAL + D);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);

    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = t.chunk_len[c];
    if (n <= 0) return;
    const int tok0 = t.chunk_tok0[c];
    const int H = s.H;
    const size_t ch = (size_t)c * H + h;
    const float scale = s.scale;

    // ---- batched vector loads: k, q, v (bf16, 8 per 16 B), g (fp32, 4 per 16 B)
    constexpr int NU = BT * D / 8 / PT;   // 16-byte bf16 chunks per thread
    constexpr int NG = BT * D / 4 / PT;   // 16-byte fp32 chunks per thread
    uint4 kr4[NU], qr4[NU], vr4[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const int ci = tid + PT * u, r = ci >> 4, c8 = (ci & 15) * 8;
        kr4[u] = qr4[u] = vr4[u] = make_uint4(0, 0, 0, 0);
        if (r < n) {
            const size_t off = ((size_t)(tok0 + r) * H + h) * D + c8;
            kr4[u] = __ldg(reinterpret_cast<const uint4*>(k + off));
            qr4[u] = __ldg(reinterpret_cast<const uint4*>(q + off));
            vr4[u] = __ldg(reinterpret_cast<const uint4*>(v + off));
        }
    }
    float4 gr4[NG];
#pragma unroll
    for (int u = 0; u < NG; ++u) {
        const int ci = tid + PT * u, r = ci >> 5, c4 = (ci & 31) * 4;
        gr4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < n) {
            if (GATE == 2) gr4[u] = __ldg(reinterpret_cast<const float4*>(g + ((size_t)(tok0 + r) * H + h) * D + c4));
            if (GATE == 1) {
                const float x = __ldg(g + (size_t)(tok0 + r) * H + h);
                gr4[u] = make_float4(x, x, x, x);
            }
        }
    }
    if (tid < BT) sBeta[tid] = (tid < n) ? bfx(beta + (size_t)(tok0 + tid) * H + h) : 0.f;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const int ci = tid + PT * u, r = ci >> 4, c8 = (ci & 15) * 8;
        *reinterpret_cast<uint4*>(sK + r * D + c8) = kr4[u];
        *reinterpret_cast<uint4*>(sQ + r * D + c8) = qr4[u];
    }
#pragma unroll
    for (int u = 0; u < NG; ++u) {
        const int ci = tid + PT * u, r = ci >> 5, c4 = (ci & 31) * 4;
        sA[r * LG + c4] = gr4[u].x * LOG2E;
        sA[r * LG + c4 + 1] = gr4[u].y * LOG2E;
        sA[r * LG + c4 + 2] = gr4[u].z * LOG2E;
        sA[r * LG + c4 + 3] = gr4[u].w * LOG2E;
    }
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tslot, 256);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tb = *tslot;

    // a1: cumsum by 4 segments of 16 rows per feature (lanes 4c..4c+3), range, midpoint anchor;
    // then alpha = 2^(G2 - c) replaces G2 (one exp2 per element; every other decay factor of
    // this chunk is alpha times a per-feature constant or its reciprocal)
    int wide_col = 0;
    if (tid < 4 * D) {
        const int col = tid >> 2, seg = tid & 3;
        float x[16];
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            acc += sA[(16 * seg + r) * LG + col];
            x[r] = acc;
        }
        float pre = __shfl_up_sync(0xffffffffu, acc, 1, 4);
        if (seg < 1) pre = 0.f;
        float t2 = __shfl_up_sync(0xffffffffu, acc + pre, 2, 4);
        if (seg < 2) t2 = 0.f;
        const float off = pre + t2;  // exclusive prefix of the segment totals
        float hi = -INFINITY, lo = INFINITY;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            x[r] += off;
            if (16 * seg + r < n) {
                hi = fmaxf(hi, x[r]);
                lo = fminf(lo, x[r]);
            }
        }
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, 1));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, 2));
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, 1));
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, 2));
        const float cc = 0.5f * (hi + lo);
        const float glast = __shfl_sync(0xffffffffu, x[15], (lane & ~3) | 3);  // G2 at row 63 = last token
#pragma unroll
        for (int r = 0; r < 16; ++r) sA[(16 * seg + r) * LG + col] = exp2f(x[r] - cc);
        if (seg == 0) {
            sC2[col] = exp2f(cc);
            sAL[col] = exp2f(glast - cc);
            f.GL[ch * D + col] = glast;
        }
        wide_col = (hi - lo) > PREP_RANGE_LOG2;
    }
    const bool wide = __syncthreads_or(wide_col) != 0;
    if (tid == 0) f.WIDE[ch] = wide ? 1 : 0;
    bool ok = true;
    if (!wide) {
        // a2 operands (tf32): A rows 0..63 beta_i k_i alpha_i, rows 64..127 s q_i alpha_i;
        // B rows j: k_j / alpha_j
        for (int idx = tid; idx < 2 * BT * 32; idx += PT) {
            const int r = idx >> 5, cc = idx & 31, i = r & (BT - 1);
            const bf16* src = (r < BT ? sK : sQ) + i * D + 4 * cc;
            const float mul = (r < BT) ? sBeta[i] : scale;
            const float* al = sA + i * LG + 4 * cc;
            const float4 val = make_float4(mul * __bfloat162float(src[0]) * al[0], mul * __bfloat162float(src[1]) * al[1],
                                           mul * __bfloat162float(src[2]) * al[2], mul * __bfloat162float(src[3]) * al[3]);
            *reinterpret_cast<float4*>(R1 + tc::sw128_off(2 * BT, r, cc * 16)) = val;
        }
        for (int idx = tid; idx < BT * 32; idx += PT) {
            const int j = idx >> 5, cc = idx & 31;
            const bf16* src = sK + j * D + 4 * cc;
            const float* al = sA + j * LG + 4 * cc;
            const float4 val = make_float4(__bfloat162float(src[0]) * __frcp_rn(al[0]), __bfloat162float(src[1]) * __frcp_rn(al[1]),
                                           __bfloat162float(src[2]) * __frcp_rn(al[2]), __bfloat162float(src[3]) * __frcp_rn(al[3]));
            *reinterpret_cast<float4*>(R2 + tc::sw128_off(BT, j, cc * 16)) = val;
        }
        tc::fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t id = tc::idesc_tf32(128, 64);
            const uint32_t a0 = tc::smem_u32(R1), b0 = tc::smem_u32(R2);
#pragma unroll 1
            for (int st = 0; st < 16; ++st)
                tc::mma_tf32(tb, tc::sdesc_k(a0, 2 * BT, st), tc::sdesc_k(b0, BT, st), id, st > 0);
            tc::mma_commit(bar);
        }
        ok = wait_all(bar, 0, t.err);
    }
    if (!wide && ok) {
        tc::fence_after_sync();
        bf16* sAq = reinterpret_cast<bf16*>(R2 + 16384);  // staged C_q [64][72] (transposed copy)
        // read back [Akk ; Aqk]: warps w, w+4, w+8, w+12 share lanes 32(w%4).., split the 64 columns
        {
            const int row = 32 * (warp & 3) + lane, cb = (warp >> 2) * 16;
            float a[16];
            tc::tmem_ld16(tc::taddr(tb, 32 * (warp & 3), cb), a);
            tc::tmem_wait_ld();
            if (row < BT) {
                const int i = row;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = cb + jj;
                    sAkk[i * LA + j] = (j < i && i < n) ? a[jj] : 0.f;
                }
            } else {
                const int i = row - BT;
                uint32_t pw[8];
#pragma unroll
                for (int jj = 0; jj < 16; jj += 2) {
                    const int j = cb + jj;
                    const float x0 = (j <= i && i < n) ? a[jj] : 0.f;
                    const float x1 = (j + 1 <= i && i < n) ? a[jj + 1] : 0.f;
                    pw[jj / 2] = tc::pack_bf16(x0, x1);
                    if (BWD) {
                        sAq[i * LQ + j] = __float2bfloat16_rn(x0);
                        sAq[i * LQ + j + 1] = __float2bfloat16_rn(x1);
                    }
                }
                uint4* dst = reinterpret_cast<uint4*>(f.AQK + ch * BT * BT + (size_t)i * BT + cb);
                dst[0] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                dst[1] = make_uint4(pw[4], pw[5], pw[6], pw[7]);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        // a3: A = (I + Akk)^-1
        blocked_inverse(sAkk, sAi, sT, tid);
        // a4 operands (tf32): R1 <- E^T [128 keys][64 tokens] (beta k 2^G2 = beta k alpha 2^c),
        // R1+32K <- Z^T [128 values][64 tokens], R2 <- A [64 rows i][64 cols j]
        for (int idx = tid; idx < D * 16; idx += PT) {
            const int kr = idx & (D - 1), cc = idx >> 7;
            float4 val;
            float* pv = reinterpret_cast<float*>(&val);
            const float c2 = sC2[kr];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 4 * cc + e;
                pv[e] = sBeta[j] * __bfloat162float(sK[j * D + kr]) * sA[j * LG + kr] * c2;
            }
            *reinterpret_cast<float4*>(R1 + tc::sw128_off(D, kr, cc * 16)) = val;
        }
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int ci = tid + PT * u, j = ci >> 4, c8 = (ci & 15) * 8;
            const bf16* pv = reinterpret_cast<const bf16*>(&vr4[u]);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                *reinterpret_cast<float*>(R1 + 32768 + tc::sw128_off(D, c8 + e, j * 4)) = sBeta[j] * __bfloat162float(pv[e]);
        }
        for (int idx = tid; idx < BT * 16; idx += PT) {
            const int i = idx >> 4, cc = idx & 15;
            const float* ai = sAi + i * LA + 4 * cc;
            *reinterpret_cast<float4*>(R2 + tc::sw128_off(BT, i, cc * 16)) = make_float4(ai[0], ai[1], ai[2], ai[3]);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t id = tc::idesc_tf32(128, 64);
            const uint32_t a0 = tc::smem_u32(R1), a1 = a0 + 32768, b0 = tc::smem_u32(R2);
#pragma unroll 1
            for (int st = 0; st < 8; ++st) tc::mma_tf32(tb + 64, tc::sdesc_k(a0, D, st), tc::sdesc_k(b0, BT, st), id, st > 0);
#pragma unroll 1
            for (int st = 0; st < 8; ++st) tc::mma_tf32(tb + 128, tc::sdesc_k(a1, D, st), tc::sdesc_k(b0, BT, st), id, st > 0);
            tc::mma_commit(bar);
        }
        // element-wise outputs while the MMAs run, as 16-byte stores:
        // Q_g [i][k] (+ Q_g^T), F^T [k][i] (+ F), A^T [j][i], C_q^T
        {
            for (int idx = tid; idx < BT * 16; idx += PT) {           // rows i, 8 keys per store
                const int i = idx >> 4, c8 = (idx & 15) * 8;
                uint32_t pq[4], pk[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const int kk = c8 + e;
                    const float a0 = sA[i * LG + kk], a1 = sA[i * LG + kk + 1];
                    pq[e / 2] = tc::pack_bf16(scale * __bfloat162float(sQ[i * D + kk]) * a0 * sC2[kk],
                                              scale * __bfloat162float(sQ[i * D + kk + 1]) * a1 * sC2[kk + 1]);
                    if (BWD)
                        pk[e / 2] = tc::pack_bf16(__bfloat162float(sK[i * D + kk]) * sAL[kk] * __frcp_rn(a0),
                                                  __bfloat162float(sK[i * D + kk + 1]) * sAL[kk + 1] * __frcp_rn(a1));
                }
                *reinterpret_cast<uint4*>(f.QG + ch * BT * D + (size_t)i * D + c8) = make_uint4(pq[0], pq[1], pq[2], pq[3]);
                if (BWD) *reinterpret_cast<uint4*>(f.KG + ch * BT * D + (size_t)i * D + c8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            for (int idx = tid; idx < D * 8; idx += PT) {             // rows k, 8 tokens per store
                const int kk = idx >> 3, i8 = (idx & 7) * 8;
                uint32_t pk[4], pq[4];
                const float c2 = sC2[kk], al = sAL[kk];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const int i = i8 + e;
                    const float a0 = sA[i * LG + kk], a1 = sA[(i + 1) * LG + kk];
                    pk[e / 2] = tc::pack_bf16(__bfloat162float(sK[i * D + kk]) * al * __frcp_rn(a0),
                                              __bfloat162float(sK[(i + 1) * D + kk]) * al * __frcp_rn(a1));
                    if (BWD)
                        pq[e / 2] = tc::pack_bf16(scale * __bfloat162float(sQ[i * D + kk]) * a0 * c2,
                                                  scale * __bfloat162float(sQ[(i + 1) * D + kk]) * a1 * c2);
                }
                *reinterpret_cast<uint4*>(f.KGT + ch * D * BT + (size_t)kk * BT + i8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                if (BWD) *reinterpret_cast<uint4*>(f.QGT + ch * D * BT + (size_t)kk * BT + i8) = make_uint4(pq[0], pq[1], pq[2], pq[3]);
            }
            if (BWD) {
                for (int idx = tid; idx < BT * 8; idx += PT) {        // rows j of A^T and C_q^T
                    const int j = idx >> 3, i8 = (idx & 7) * 8;
                    uint32_t pa[4], pc[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        pa[e / 2] = tc::pack_bf16(sAi[(i8 + e) * LA + j], sAi[(i8 + e + 1) * LA + j]);
                        pc[e / 2] = (uint32_t)(*reinterpret_cast<const uint16_t*>(&sAq[(i8 + e) * LQ + j])) |
                                    ((uint32_t)(*reinterpret_cast<const uint16_t*>(&sAq[(i8 + e + 1) * LQ + j])) << 16);
                    }
                    *reinterpret_cast<uint4*>(f.AIT + ch * BT * BT + (size_t)j * BT + i8) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
                    *reinterpret_cast<uint4*>(f.AQKT + ch * BT * BT + (size_t)j * BT + i8) = make_uint4(pc[0], pc[1], pc[2], pc[3]);
                }
            }
        }
        ok = wait_all(bar, 1, t.err);
        if (ok) {
            tc::fence_after_sync();
            bf16* sW = reinterpret_cast<bf16*>(R1);                     // staged W [64][136]
            float* sU = reinterpret_cast<float*>(R1 + 2 * BT * LW);     // staged U [64][132]
            const int row = 32 * (warp & 3) + lane, grp = warp >> 2;    // 4 warps per lane quarter
            // W^T (columns 64..127) by groups 0-1, U^T (columns 128..191) by groups 2-3; 32 columns each
            const int cbase = (grp & 1) * 32;
            if (grp < 2) {
#pragma unroll
                for (int cb = cbase; cb < cbase + 32; cb += 16) {
                    float a[16];
                    tc::tmem_ld16(tc::taddr(tb + 64, 32 * (warp & 3), cb), a);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) sW[(cb + jj) * LW + row] = __float2bfloat16_rn(a[jj]);
                    if (BWD) {
                        uint32_t pw[8];
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) pw[jj] = tc::pack_bf16(a[2 * jj], a[2 * jj + 1]);
                        uint4* dst = reinterpret_cast<uint4*>(f.WT + ch * D * BT + (size_t)row * BT + cb);
                        dst[0] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                        dst[1] = make_uint4(pw[4], pw[5], pw[6], pw[7]);
                    }
                }
            } else {
#pragma unroll
                for (int cb = cbase; cb < cbase + 32; cb += 16) {
                    float a[16];
                    tc::tmem_ld16(tc::taddr(tb + 128, 32 * (warp & 3), cb), a);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) sU[(cb + jj) * LU + row] = a[jj];
                }
            }
            __syncthreads();
            for (int idx = tid; idx < BT * 16; idx += PT) {
                const int i = idx >> 4, c8 = (idx & 15) * 8;
                *reinterpret_cast<uint4*>(f.W + ch * BT * D + (size_t)i * D + c8) = *reinterpret_cast<const uint4*>(sW + i * LW + c8);
            }
            for (int idx = tid; idx < BT * 32; idx += PT) {
                const int i = idx >> 5, c4 = (idx & 31) * 4;
                *reinterpret_cast<float4*>(f.U + ch * BT * D + (size_t)i * D + c4) = *reinterpret_cast<const float4*>(sU + i * LU + c4);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 256);
}

// ======================================================= k_fwd_scan_tc
constexpr int ST = 256;  // 8 warps: warps w and w+4 share TMEM lane quarter w%4 and split columns

// Shared-memory map (bytes from the 1024-aligned base).
constexpr int OFF_AS = 0;                    // S^T bf16 [128][128]   32 KB
constexpr int OFF_AR = OFF_AS + 32768;       // R^T bf16 [128][64]    16 KB
constexpr int OFF_STAGE = OFF_AR + 16384;    // two stages
constexpr int STG_W = 0;                     // W   [64][128]  16 KB
constexpr int STG_KG = 16384;                // F^T [128][64]  16 KB
constexpr int STG_QG = 32768;                // Q_g [64][128]  16 KB
constexpr int STG_AQ = 49152;                // C_q [64][64]    8 KB
constexpr int STG_BYTES = 57344;
constexpr int OFF_LAM = OFF_STAGE + 2 * STG_BYTES;   // lambda [128] fp32
constexpr int OFF_TST = OFF_LAM + 512;                 // per-warp transpose staging, 8 x 1280 B
constexpr int OFF_BAR = OFF_TST + 8 * 1280;
constexpr int SCAN_SMEM = OFF_BAR + 64 + 1024;

using tc::cp_async16;
using tc::cp_async_commit;
using tc::cp_async_wait_all;

// Copies a row-major bf16 [R][C] global tile into a K-major SW128 smem tile.
template <int R, int C>
__device__ __forceinline__ void load_tile(uint32_t sbase, const bf16* src, int tid) {
    constexpr int CPR = C * 2 / 16;  // 16-byte chunks per row
    for (int idx = tid; idx < R * CPR; idx += ST) {
        const int r = idx / CPR, cc = idx % CPR;
        cp_async16(sbase + tc::sw128_off(R, r, cc * 16), src + (size_t)r * C + cc * 8);
    }
}

template <int MODE>
__device__ __forceinline__ void fscan_prefetch(uint32_t stg, const FwdTC& f, size_t ch, int tid) {
    load_tile<BT, D>(stg + STG_W, f.W + ch * BT * D, tid);
    load_tile<D, BT>(stg + STG_KG, f.KGT + ch * D * BT, tid);
    if (MODE & 1) {
        load_tile<BT, D>(stg + STG_QG, f.QG + ch * BT * D, tid);
        load_tile<BT, BT>(stg + STG_AQ, f.AQK + ch * BT * BT, tid);
    }
    cp_async_commit();
}

template <int MODE>
__global__ void __launch_bounds__(ST, 1)
    k_fwd_scan_tc(Shape s, const float* __restrict__ h0, Table t, FwdTC f, bf16* __restrict__ o,
                  float* __restrict__ ht) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(base + OFF_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 3);
    float* sLam = reinterpret_cast<float*>(base + OFF_LAM);
    const uint32_t sb = tc::smem_u32(base);
    const int nseq = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    bf16* tst = reinterpret_cast<bf16*>(base + OFF_TST + warp * 1280);
    const int H = s.H;
    const int vcol = 32 * quad + lane;  // TMEM lane and value column of this thread
    const int c0 = t.seq_chunk0[nseq], c1 = t.seq_chunk0[nseq + 1];

    if (tid == 0) {
        tc::mbar_init(&bar[0], 1);
        tc::mbar_init(&bar[1], 1);
        tc::mbar_init(&bar[2], 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tslot, 256);
        tc::tmem_relinquish();
    }
    if (c0 < c1) fscan_prefetch<MODE>(sb + OFF_STAGE, f, (size_t)c0 * H + h, tid);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tb = *tslot;
    const uint32_t tl = tc::taddr(tb, 32 * quad, 0);  // this warp's lane quarter
    const size_t st_off = ((size_t)nseq * H + h) * D * D;
    const int kb = 64 * half;   // this thread's half of the key columns of S^T
    const int ib = 32 * half;   // this thread's half of the chunk rows

    // S^T <- h0^T (thread holds row v: h0[k][v] for its keys)
#pragma unroll 1
    for (int cb = kb; cb < kb + 64; cb += 16) {
        float a[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) a[jj] = h0 ? h0[st_off + (size_t)(cb + jj) * D + vcol] : 0.f;
        tc::tmem_st16(tl + cb, a);
    }
    tc::tmem_wait_st();

    uint32_t ph0 = 0, ph1 = 0, ph2 = 0;
    bool ok = true;
    for (int c = c0; c < c1 && ok; ++c) {
        const int it = c - c0, stage = it & 1;
        const size_t ch = (size_t)c * H + h;
        const int len = t.chunk_len[c], tok0 = t.chunk_tok0[c];
        const uint32_t stg = sb + OFF_STAGE + stage * STG_BYTES;
        // U rows of this thread's value column (consumed after the first MMA)
        float u[32];
        const float* U = f.U + ch * BT * D + (size_t)ib * D + vcol;
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] = U[(size_t)i * D];
        if (tid < D) sLam[tid] = exp2f(f.GL[ch * D + tid]);
        __syncthreads();
        // 1. S^T -> bf16 operand (and the saved state), then S^T <- S^T diag(lambda)
#pragma unroll 1
        for (int cb = kb; cb < kb + 64; cb += 16) {
            float a[16];
            tc::tmem_ld16(tl + cb, a);
            tc::tmem_wait_ld();
            uint32_t pw[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) pw[jj] = tc::pack_bf16(a[2 * jj], a[2 * jj + 1]);
            *reinterpret_cast<uint4*>(base + OFF_AS + tc::sw128_off(D, vcol, cb * 2)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
            *reinterpret_cast<uint4*>(base + OFF_AS + tc::sw128_off(D, vcol, cb * 2 + 16)) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
            if (MODE & 2) tc::warp_store_t16(tst, a, f.HS + ch * D * D + (size_t)cb * D + 32 * quad, D, 16, lane);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) a[jj] *= sLam[cb + jj];
            tc::tmem_st16(tl + cb, a);
        }
        tc::tmem_wait_st();
        cp_async_wait_all();
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        // 2. D1 = S^T W^T ; O^T = S^T Q_g^T
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t id = tc::idesc_bf16(128, 64);
            const uint32_t aS = sb + OFF_AS;
#pragma unroll 1
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16(tb + 128, tc::sdesc_k(aS, D, ks), tc::sdesc_k(stg + STG_W, BT, ks), id, ks > 0);
            tc::mma_commit(&bar[0]);
            if (MODE & 1) {
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16(tb + 192, tc::sdesc_k(aS, D, ks), tc::sdesc_k(stg + STG_QG, BT, ks), id, ks > 0);
            }
        }
        // prefetch chunk c+1 into the other stage (its previous MMAs have completed)
        if (c + 1 < c1) fscan_prefetch<MODE>(sb + OFF_STAGE + (stage ^ 1) * STG_BYTES, f, (size_t)(c + 1) * H + h, tid);
        ok = wait_all(&bar[0], ph0, t.err);
        ph0 ^= 1;
        if (!ok) break;
        tc::fence_after_sync();
        // 3. R^T = U^T - D1 (bf16 operand; saved for the backward)
#pragma unroll
        for (int cq = 0; cq < 32; cq += 16) {
            float a[16];
            tc::tmem_ld16(tl + 128 + ib + cq, a);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) a[jj] = u[cq + jj] - a[jj];
            uint32_t pw[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) pw[jj] = tc::pack_bf16(a[2 * jj], a[2 * jj + 1]);
            *reinterpret_cast<uint4*>(base + OFF_AR + tc::sw128_off(D, vcol, (ib + cq) * 2)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
            *reinterpret_cast<uint4*>(base + OFF_AR + tc::sw128_off(D, vcol, (ib + cq) * 2 + 16)) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
            if (MODE & 2) tc::warp_store_t16(tst, a, f.R + ch * BT * D + (size_t)(ib + cq) * D + 32 * quad, D, 16, lane);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        // 4. O^T += R^T C_q^T (committed first, so its read-back overlaps the state update);
        //    S^T += R^T F
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t aR = sb + OFF_AR;
            if (MODE & 1) {
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tb + 192, tc::sdesc_k(aR, D, ks), tc::sdesc_k(stg + STG_AQ, BT, ks), tc::idesc_bf16(128, 64), 1);
                tc::mma_commit(&bar[2]);
            }
#pragma unroll 1
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16(tb, tc::sdesc_k(aR, D, ks), tc::sdesc_k(stg + STG_KG, D, ks), tc::idesc_bf16(128, 128), 1);
            tc::mma_commit(&bar[1]);
        }
        // 5. output rows of this value column
        if (MODE & 1) {
            ok = wait_all(&bar[2], ph2, t.err);
            ph2 ^= 1;
            if (!ok) break;
            tc::fence_after_sync();
#pragma unroll 1
            for (int cq = 0; cq < 32; cq += 16) {
                const int r0 = ib + cq;
                if (r0 >= len) break;
                float a[16];
                tc::tmem_ld16(tl + 192 + r0, a);
                tc::tmem_wait_ld();
                tc::warp_store_t16(tst, a, o + ((size_t)(tok0 + r0) * H + h) * D + 32 * quad, (size_t)H * D,
                                   len - r0, lane);
            }
            tc::fence_before_sync();
        }
        ok = wait_all(&bar[1], ph1, t.err);
        ph1 ^= 1;
        if (!ok) break;
        tc::fence_after_sync();
    }
    if (ok && ht) {
        tc::fence_after_sync();
#pragma unroll 1
        for (int cb = kb; cb < kb + 64; cb += 16) {
            float a[16];
            tc::tmem_ld16(tl + cb, a);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) ht[st_off + (size_t)(cb + jj) * D + vcol] = a[jj];
        }
    }
    cp_async_wait_all();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 256);
}

constexpr size_t PREP_SMEM = 65536 + 32768 + sizeof(float) * (BT * LG + 2 * BT * LA + 3 * BC * (BC + 1) + BT + 2 * D) +
                             2 * 2 * BT * D + 64 + 1024;

template <int GATE, bool BWD>
cudaError_t run_prep(const Shape& s, const void* q, const void* k, const void* v, const void* beta,
                     const float* g, Table t, FwdTC f, cudaStream_t st) {
    cudaError_t e = set_smem_once<k_prep_tc<GATE, BWD>>(PREP_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(s.NC, s.H);
    k_prep_tc<GATE, BWD><<<grid, PT, PREP_SMEM, st>>>(s, (const bf16*)q, (const bf16*)k, (const bf16*)v,
                                                      (const bf16*)beta, g, t, f);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t run_scan(const Shape& s, const float* h0, Table t, FwdTC f, void* o, float* ht, cudaStream_t st) {
    cudaError_t e = set_smem_once<k_fwd_scan_tc<MODE>>(SCAN_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(s.N, s.H);
    k_fwd_scan_tc<MODE><<<grid, ST, SCAN_SMEM, st>>>(s, h0, t, f, (bf16*)o, ht);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tc(const Shape& s, int gate, int for_bwd, const void* q, const void* k,
                           const void* v, const void* beta, const float* g, Table t, FwdTC f,
                           cudaStream_t st) {
    if (for_bwd) {
        switch (gate) {
            case 0: return run_prep<0, true>(s, q, k, v, beta, g, t, f, st);
            case 1: return run_prep<1, true>(s, q, k, v, beta, g, t, f, st);
            default: return run_prep<2, true>(s, q, k, v, beta, g, t, f, st);
        }
    }
    switch (gate) {
        case 0: return run_prep<0, false>(s, q, k, v, beta, g, t, f, st);
        case 1: return run_prep<1, false>(s, q, k, v, beta, g, t, f, st);
        default: return run_prep<2, false>(s, q, k, v, beta, g, t, f, st);
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
