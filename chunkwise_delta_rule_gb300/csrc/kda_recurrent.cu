// Token-by-token forward of the gated delta rule, for decoding and short
// prompts ("Kimi Delta Attention" derivation blog, §4 boxed KDA update):
//     S~ = diag(exp g_t) S;  r_t = beta_t (v_t - S~^T k_t);  S = S~ + k_t r_t^T;  o_t = S^T (s q_t)
// The update is separable over value columns (column v of S evolves with its
// own entry of r_t), so a CTA owns a 32-column slice of one (sequence, head)
// state and no two CTAs exchange anything. Warp w holds columns 8w..8w+7 of
// the slice, lane l the keys l, l+32, ...; the slice stays in registers for
// the whole call and is read and written once. Each token needs two sums over
// keys (S~^T k and S^T q), formed by a butterfly that leaves every lane one
// column's total. The next token's inputs are loaded while the current one is
// processed. The optional prologue ("GatedDeltaNet-2 (NVlabs) — official spec
// transcription", §3) runs per token on the loaded values: q and k divided by
// sqrt(sum x^2 + eps) (every warp holds all keys, so a warp sum suffices), and
// the decay -exp(A_log) softplus(g + dt_bias) or lower_bound sigmoid(exp(A_log)
// (g + dt_bias)). GatedDeltaNet-2 (same page, §3) erases along b .* k and writes
// w .* v: r_t = w_t .* v_t - S~^T (b_t .* k_t).
#include <string.h>

#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int RT = 128;   // 4 warps x 8 value columns
constexpr int RV = 32;    // value columns per CTA
constexpr unsigned FULL = 0xffffffffu;

struct RecIO {
    const void *q, *k, *v, *beta;
    const float *g, *h0;
    const int32_t* cu;
    void* o;
    float* ht;
    int32_t* err;
    int T;
    const float *A_log, *dt_bias;   // prologue: A_log NULL = g is the decay itself
    float lower_bound, eps;
    int qk_norm;
    const void *erase, *write;      // GatedDeltaNet-2 vectors, or NULL (beta rule)
    int G;                          // value heads per key head (q, k of key head h / G)
};

__device__ __forceinline__ float rwsum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
    return x;
}
__device__ __forceinline__ float ract(float z, float eA, float lb) {
    if (lb == 0.f) return -eA * (z > 20.f ? z : log1pf(expf(z)));
    return lb / (1.f + expf(-eA * z));
}

// Column (of the warp's eight) whose total lane l holds after reduce8.
__device__ __forceinline__ int rcol(int lane) { return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1); }
// A lane holding column c's total.
__device__ __forceinline__ int rsrc(int c) { return ((c >> 2) & 1) * 16 + ((c >> 1) & 1) * 8 + (c & 1) * 4; }

// Sums x[0..7] over the warp's 32 lanes (9 shuffles): each halving step keeps
// half of the columns and adds the partner's copy of them.
__device__ __forceinline__ float reduce8(const float (&x)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float y[4], z[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? x[i] : x[i + 4];
        y[i] = (b4 ? x[i + 4] : x[i]) + __shfl_xor_sync(FULL, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? y[i] : y[i + 2];
        z[i] = (b3 ? y[i + 2] : y[i]) + __shfl_xor_sync(FULL, send, 8);
    }
    const float send = b2 ? z[0] : z[1];
    float w = (b2 ? z[1] : z[0]) + __shfl_xor_sync(FULL, send, 4);
    w += __shfl_xor_sync(FULL, w, 2);
    w += __shfl_xor_sync(FULL, w, 1);
    return w;
}

// Inputs of one token for this thread: its keys' k, q and gate, its column's v,
// beta. load() only issues the reads (the next token's are in flight while the
// current one is processed); finish() applies the scale, the optional
// normalisation and the gate activation, and turns the gate into the decay
// factor exp(g).
template <typename TI, int KJ, int GATE>
struct Tok {
    float k[KJ], q[KJ], a[KJ], eb[KJ], v, b;
    __device__ __forceinline__ void load(const RecIO& io, size_t row, size_t krow, int K, int V, int col, int lane) {
        const TI* kp = static_cast<const TI*>(io.k) + krow * K + lane;
        const TI* qp = static_cast<const TI*>(io.q) + krow * K + lane;
#pragma unroll
        for (int j = 0; j < KJ; ++j) {
            k[j] = ld(kp + 32 * j);
            q[j] = ld(qp + 32 * j);
        }
        if (GATE == 2) {
#pragma unroll
            for (int j = 0; j < KJ; ++j) a[j] = io.g[row * K + lane + 32 * j];
        } else if (GATE == 1) {
            a[0] = io.g[row];
        }
        v = ld(static_cast<const TI*>(io.v) + row * V + col);
        if (io.erase) {
            const TI* ep = static_cast<const TI*>(io.erase) + row * K + lane;
#pragma unroll
            for (int j = 0; j < KJ; ++j) eb[j] = ld(ep + 32 * j);
            b = ld(static_cast<const TI*>(io.write) + row * V + col);   // this column's write weight
        } else {
#pragma unroll
            for (int j = 0; j < KJ; ++j) eb[j] = 1.f;
            b = ld(static_cast<const TI*>(io.beta) + row);
        }
    }
    __device__ __forceinline__ void finish(const RecIO& io, int h, int K, int lane, float scale) {
        float sq = scale, sk = 1.f;
        if (io.qk_norm) {
            float ssq = 0.f, ssk = 0.f;
#pragma unroll
            for (int j = 0; j < KJ; ++j) {
                ssq = fmaf(q[j], q[j], ssq);
                ssk = fmaf(k[j], k[j], ssk);
            }
            sq = scale / sqrtf(rwsum(ssq) + io.eps);
            sk = 1.f / sqrtf(rwsum(ssk) + io.eps);
        }
#pragma unroll
        for (int j = 0; j < KJ; ++j) {
            q[j] *= sq;
            k[j] *= sk;
        }
        if (GATE == 1) {
#pragma unroll
            for (int j = 1; j < KJ; ++j) a[j] = a[0];
        }
        if (GATE != 0) {
            const float eA = io.A_log ? expf(io.A_log[h]) : 0.f;
#pragma unroll
            for (int j = 0; j < KJ; ++j) {
                float x = a[j];
                if (io.A_log) {
                    const float db = io.dt_bias ? (GATE == 2 ? io.dt_bias[h * K + lane + 32 * j] : io.dt_bias[h]) : 0.f;
                    x = ract(x + db, eA, io.lower_bound);
                }
                a[j] = expf(x);
            }
        } else {
#pragma unroll
            for (int j = 0; j < KJ; ++j) a[j] = 1.f;
        }
    }
};

// The state slice moves by TMA when its tensor map could be made (tma bit 0: h0, bit 1: ht): one box
// of 32 keys x 32 columns per 32 keys into a 128-byte-swizzled tile, from which each lane takes its
// key row's two 16-byte chunks (chunk c of row r at c ^ (r mod 8): the eight lanes of a quarter warp
// reach distinct banks); otherwise each lane reads and writes its 32 bytes per key directly.
__device__ __forceinline__ unsigned char* rec_chunk(unsigned char* tile, int j, int lane, int c) {
    return tile + j * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4);
}

template <typename TI, int K, int GATE>
__global__ void __launch_bounds__(RT, K <= 128 ? 6 : 1) k_recurrent(Shape s, RecIO io, const __grid_constant__ CUtensorMap tmh0,
                                                  const __grid_constant__ CUtensorMap tmht, int tma) {
    constexpr int KJ = K / 32;
    extern __shared__ unsigned char rsm_raw[];
    unsigned char* tile = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(rsm_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(tile + K * 128);
    const int VB = s.V / RV;
    const int n = blockIdx.x / VB, vb = blockIdx.x - n * VB, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = s.H, V = s.V;
    const int col0 = vb * RV + 8 * warp;   // first of this warp's eight columns
    const int cme = col0 + rcol(lane);     // the column whose totals this lane holds
    int t0, t1;
    if (io.cu) {
        t0 = io.cu[n];
        t1 = io.cu[n + 1];
        if (t0 < 0 || t1 < t0 || t1 > s.Ttot) {   // inconsistent offsets: an empty sequence
            if (threadIdx.x == 0 && vb == 0 && h == 0 && io.err) atomicOr(io.err, 1);
            t0 = t1 = 0;
        }
    } else {
        t0 = n * io.T;
        t1 = t0 + io.T;
    }
    // the first token's inputs, in flight while the state slice loads
    Tok<TI, KJ, GATE> cur, nxt;
    const int Hk = H / io.G, hk = h / io.G;   // key heads; this value head's key head
    if (t0 < t1) cur.load(io, (size_t)t0 * H + h, (size_t)t0 * Hk + hk, K, V, cme, lane);
    // the state slice: keys lane + 32 j, columns col0 .. col0 + 7
    float S[KJ][8];
    const size_t sb = ((size_t)n * H + h) * K * V;
    if ((tma & 1) && io.h0) {
        if (threadIdx.x == 0) {
            tc::mbar_init(bar, 1);
            tc::fence_mbar_init();
            tc::mbar_arrive_expect_tx(bar, K * 128);
#pragma unroll
            for (int j = 0; j < KJ; ++j) tc::tma_load3(tc::smem_u32(tile + j * 4096), &tmh0, vb * RV, 32 * j, n * H + h, bar);
        }
        __syncthreads();
        if (!__syncthreads_and(tc::mbar_wait(bar, 0))) {   // a lost copy: recorded, and it lands first
            if (threadIdx.x == 0) {
                if (io.err) atomicOr(io.err, 2);
                tc::mbar_wait(bar, 0);
            }
            return;
        }
#pragma unroll
        for (int j = 0; j < KJ; ++j) {
            const float4 x0 = *reinterpret_cast<const float4*>(rec_chunk(tile, j, lane, 2 * warp));
            const float4 x1 = *reinterpret_cast<const float4*>(rec_chunk(tile, j, lane, 2 * warp + 1));
            S[j][0] = x0.x; S[j][1] = x0.y; S[j][2] = x0.z; S[j][3] = x0.w;
            S[j][4] = x1.x; S[j][5] = x1.y; S[j][6] = x1.z; S[j][7] = x1.w;
        }
    } else {
#pragma unroll
    for (int j = 0; j < KJ; ++j) {
        if (io.h0) {
            const float4* src = reinterpret_cast<const float4*>(io.h0 + sb + (size_t)(lane + 32 * j) * V + col0);
            const float4 x0 = src[0], x1 = src[1];
            S[j][0] = x0.x; S[j][1] = x0.y; S[j][2] = x0.z; S[j][3] = x0.w;
            S[j][4] = x1.x; S[j][5] = x1.y; S[j][6] = x1.z; S[j][7] = x1.w;
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) S[j][c] = 0.f;
        }
    }
    }
    for (int t = t0; t < t1; ++t) {
        if (t + 1 < t1) nxt.load(io, (size_t)(t + 1) * H + h, (size_t)(t + 1) * Hk + hk, K, V, cme, lane);
        cur.finish(io, h, K, lane, s.scale);
        // S~ = diag(alpha) S and p = S~^T k (this lane's keys)
        const float (&al)[KJ] = cur.a;
        float p[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < KJ; ++j) {
                S[j][c] *= al[j];
                acc = fmaf(S[j][c], cur.k[j] * cur.eb[j], acc);
            }
            p[c] = acc;
        }
        const float pm = reduce8(p, lane);
        const float rm = io.erase ? cur.b * cur.v - pm : cur.b * (cur.v - pm);   // r_t of column cme
        // S = S~ + k r^T, then o = S^T (s q)
        float oq[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float r = __shfl_sync(FULL, rm, rsrc(c));
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < KJ; ++j) {
                S[j][c] = fmaf(cur.k[j], r, S[j][c]);
                acc = fmaf(S[j][c], cur.q[j], acc);
            }
            oq[c] = acc;
        }
        const float ov = reduce8(oq, lane);
        if ((lane & 3) == 0) st(static_cast<TI*>(io.o) + ((size_t)t * H + h) * V + cme, ov);
        cur = nxt;
    }
    if (io.ht && (tma & 2)) {
        // the slice into the tile (the loads, if any, were all read before the token loop), then one
        // TMA store per 32 keys; the tile must outlive the stores' reads
        __syncthreads();
#pragma unroll
        for (int j = 0; j < KJ; ++j) {
            *reinterpret_cast<float4*>(rec_chunk(tile, j, lane, 2 * warp)) = make_float4(S[j][0], S[j][1], S[j][2], S[j][3]);
            *reinterpret_cast<float4*>(rec_chunk(tile, j, lane, 2 * warp + 1)) = make_float4(S[j][4], S[j][5], S[j][6], S[j][7]);
        }
        tc::fence_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
#pragma unroll
            for (int j = 0; j < KJ; ++j) tc::tma_store3(&tmht, vb * RV, 32 * j, n * H + h, tc::smem_u32(tile + j * 4096));
            tc::bulk_commit();
            tc::bulk_wait_all();
        }
    } else if (io.ht) {
#pragma unroll
        for (int j = 0; j < KJ; ++j) {
            float4* dst = reinterpret_cast<float4*>(io.ht + sb + (size_t)(lane + 32 * j) * V + col0);
            dst[0] = make_float4(S[j][0], S[j][1], S[j][2], S[j][3]);
            dst[1] = make_float4(S[j][4], S[j][5], S[j][6], S[j][7]);
        }
    }
}

template <typename TI, int K>
cudaError_t run_recurrent_k(const Shape& s, int gate, const RecIO& io, cudaStream_t st) {
    const long long blocks = (long long)s.N * (s.V / RV);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)blocks, s.H);
    // the states by TMA where their maps can be made (16-byte aligned; K and V are multiples of 32)
    CUtensorMap mh0, mht;
    memset(&mh0, 0, sizeof(mh0));
    memset(&mht, 0, sizeof(mht));
    const long long nh = (long long)s.N * s.H;
    int tma = 0;
    if (nh <= 0x7fffffffLL) {
        if (io.h0 && tmap_state_f32(&mh0, io.h0, (int)nh, K, s.V)) tma |= 1;
        if (io.ht && tmap_state_f32(&mht, io.ht, (int)nh, K, s.V)) tma |= 2;
    }
    const size_t smem = tma ? (size_t)K * 128 + 1024 + 16 : 0;
    switch (gate) {
        case 0: k_recurrent<TI, K, 0><<<grid, RT, smem, st>>>(s, io, mh0, mht, tma); break;
        case 1: k_recurrent<TI, K, 1><<<grid, RT, smem, st>>>(s, io, mh0, mht, tma); break;
        default: k_recurrent<TI, K, 2><<<grid, RT, smem, st>>>(s, io, mh0, mht, tma); break;
    }
    return cudaGetLastError();
}

template <typename TI>
cudaError_t run_recurrent_t(const Shape& s, int gate, const RecIO& io, cudaStream_t st) {
    switch (s.K) {
        case 64: return run_recurrent_k<TI, 64>(s, gate, io, st);
        case 128: return run_recurrent_k<TI, 128>(s, gate, io, st);
        case 160: return run_recurrent_k<TI, 160>(s, gate, io, st);
        case 192: return run_recurrent_k<TI, 192>(s, gate, io, st);
        case 256: return run_recurrent_k<TI, 256>(s, gate, io, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool recurrent_key_width(int K) { return K == 64 || K == 128 || K == 160 || K == 192 || K == 256; }

cudaError_t launch_recurrent(const Shape& s, int bf16, int gate, int T, const int32_t* cu, const void* q,
                             const void* k, const void* v, const void* beta, const float* g, const float* h0,
                             void* o, float* ht, int32_t* err, const float* A_log, const float* dt_bias,
                             float lower_bound, int qk_norm, float eps, cudaStream_t st, const Gdn2& gd, int group) {
    if (s.V % RV != 0 || !recurrent_key_width(s.K)) return cudaErrorInvalidValue;
    RecIO io{q, k, v, beta, g, h0, cu, o, ht, err, T, A_log, dt_bias, lower_bound, eps, qk_norm, gd.erase, gd.write,
             group};
    return bf16 ? run_recurrent_t<__nv_bfloat16>(s, gate, io, st) : run_recurrent_t<float>(s, gate, io, st);
}

}  // namespace kda
