// The operator's optional input transforms ("GatedDeltaNet-2 (NVlabs) —
// official spec transcription", §2.0, §3 and §4.2): q and k L2-normalised per
// (token, head) with eps inside the square root, and the decay activated from
// the raw gate with the head's A_log and the per-channel dt_bias:
//     softplus form     g = -exp(A_log) softplus(g_raw + dt_bias)
//     lower-bound form  g = lower_bound sigmoid(exp(A_log) (g_raw + dt_bias))
// k_prologue writes the transformed q, k and g for the chunk pipeline;
// k_epilogue carries the pipeline's gradients (with respect to the normalised
// q, k and the activated g) back to the raw inputs,
//     dx = r (dx_hat - x_hat <x_hat, dx_hat>),  r = (sum x^2 + eps)^(-1/2),
//     dg_raw = dg dg/dz  (softplus form: -exp(A) sigmoid(z); lower-bound form:
//              lb s (1 - s) exp(A), s = sigmoid(exp(A) z)),
// and forms per 64-token block the partial sums of dt_bias's gradient (dg_raw)
// and of A_log's (dg dg/dA: g itself, or lb s (1 - s) exp(A) z); k_prologue_sum
// adds the blocks in order, so both reductions are deterministic.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int PW = 8;      // rows (token, head) per CTA of k_prologue: one warp each
constexpr int ETB = 64;    // tokens per CTA of k_epilogue

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
    return x;
}
__device__ __forceinline__ float sigm(float u) { return 1.f / (1.f + expf(-u)); }
__device__ __forceinline__ float softplus(float z) { return z > 20.f ? z : log1pf(expf(z)); }

__device__ __forceinline__ float act(float z, float eA, float lb) {
    return lb == 0.f ? -eA * softplus(z) : lb * sigm(eA * z);
}
// dg/dz and dg/dA of the activation at z
__device__ __forceinline__ void act_grad(float z, float eA, float lb, float& dz, float& dA) {
    if (lb == 0.f) {
        dz = -eA * sigm(z);
        dA = -eA * softplus(z);
    } else {
        const float s = sigm(eA * z);
        dz = lb * s * (1.f - s) * eA;
        dA = dz * z;
    }
}

// A lane's EL consecutive elements of a row (one vector access).
__device__ __forceinline__ void ldv(const float* p, float (&x)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void ldv(const float* p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void ldv(const float* p, float (&x)[2]) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
}
__device__ __forceinline__ void ldv(const __nv_bfloat16* p, float (&x)[4]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}
__device__ __forceinline__ void ldv(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(h[i]);
        x[2 * i] = a.x;
        x[2 * i + 1] = a.y;
    }
}
__device__ __forceinline__ void ldv(const __nv_bfloat16* p, float (&x)[2]) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(p);
    const float2 a = __bfloat1622float2(v);
    x[0] = a.x; x[1] = a.y;
}
__device__ __forceinline__ void stv(float* p, const float (&x)[4]) { *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]); }
__device__ __forceinline__ void stv(float* p, const float (&x)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}
__device__ __forceinline__ void stv(float* p, const float (&x)[2]) { *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]); }
__device__ __forceinline__ void stv(__nv_bfloat16* p, const float (&x)[4]) {
    uint2 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
    h[0] = __floats2bfloat162_rn(x[0], x[1]);
    h[1] = __floats2bfloat162_rn(x[2], x[3]);
    *reinterpret_cast<uint2*>(p) = v;
}
__device__ __forceinline__ void stv(__nv_bfloat16* p, const float (&x)[8]) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = v;
}
__device__ __forceinline__ void stv(__nv_bfloat16* p, const float (&x)[2]) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x[0], x[1]);
}

// r = (sum x^2 + eps)^(-1/2) of one (token, head) row spread over the warp
template <int EL>
__device__ __forceinline__ float row_rnorm(const float (&x)[EL], float eps) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < EL; ++e) ss = fmaf(x[e], x[e], ss);
    return 1.f / sqrtf(warp_sum(ss) + eps);
}

// One warp per (token, head) row; lane l owns elements EL l .. EL l + EL - 1.
template <typename TI, int K, int GATE>
__global__ void __launch_bounds__(32 * PW) k_prologue(int rows, int H, PrologueArgs a) {
    constexpr int EL = K / 32;
    const int row = blockIdx.x * PW + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int h = row % H, c0 = EL * lane;
    float xq[EL], xk[EL], z[EL], db[EL];
    if (a.qk_norm) {
        ldv(static_cast<const TI*>(a.q) + (size_t)row * K + c0, xq);
        ldv(static_cast<const TI*>(a.k) + (size_t)row * K + c0, xk);
    }
    const bool act_on = GATE != 0 && a.A_log;
    if (act_on && GATE == 2) {
        ldv(a.g + (size_t)row * K + c0, z);
        if (a.dt_bias) ldv(a.dt_bias + (size_t)h * K + c0, db);
    }
    if (a.qk_norm) {
        const float rq = row_rnorm<EL>(xq, a.eps), rk = row_rnorm<EL>(xk, a.eps);
#pragma unroll
        for (int e = 0; e < EL; ++e) {
            xq[e] *= rq;
            xk[e] *= rk;
        }
        stv(static_cast<TI*>(a.qh) + (size_t)row * K + c0, xq);
        stv(static_cast<TI*>(a.kh) + (size_t)row * K + c0, xk);
    }
    if (act_on) {
        const float eA = expf(a.A_log[h]);
        if (GATE == 2) {
#pragma unroll
            for (int e = 0; e < EL; ++e) z[e] = act(z[e] + (a.dt_bias ? db[e] : 0.f), eA, a.lower_bound);
            stv(a.ga + (size_t)row * K + c0, z);
        } else if (lane == 0) {
            a.ga[row] = act(a.g[row] + (a.dt_bias ? a.dt_bias[h] : 0.f), eA, a.lower_bound);
        }
    }
}

// One CTA per (64-token block, head); warp w takes tokens w, w + 8, ... of the block, two at a
// time (both tokens' loads in flight before either reduction).
template <typename TI, int K, int GATE>
__global__ void __launch_bounds__(32 * PW) k_epilogue(int Ttot, int H, EpilogueArgs a) {
    constexpr int EL = K / 32;
    __shared__ float sZ[PW][K];
    __shared__ float sAp[PW];
    const int tb = blockIdx.x, h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = EL * lane;
    const bool gated = GATE != 0 && a.A_log;
    const float eA = gated ? expf(a.A_log[h]) : 0.f;
    float db[EL];
#pragma unroll
    for (int e = 0; e < EL; ++e) db[e] = 0.f;
    if (gated && a.dt_bias) {
        if (GATE == 2) ldv(a.dt_bias + (size_t)h * K + c0, db);
        else db[0] = a.dt_bias[h];
    }
    float accz[EL], accA = 0.f;
#pragma unroll
    for (int e = 0; e < EL; ++e) accz[e] = 0.f;
    const int tend = min(Ttot, tb * ETB + ETB);
    for (int t0 = tb * ETB + warp; t0 < tend; t0 += 2 * PW) {
        float xq[2][EL], dq[2][EL], xk[2][EL], dk[2][EL], zg[2][EL], ug[2][EL];
        bool in[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = t0 + u * PW;
            in[u] = t < tend;
            if (!in[u]) continue;
            const size_t row = (size_t)t * H + h;
            if (a.qk_norm) {
                ldv(static_cast<const TI*>(a.q) + row * K + c0, xq[u]);
                ldv(static_cast<const TI*>(a.dq) + row * K + c0, dq[u]);
                ldv(static_cast<const TI*>(a.k) + row * K + c0, xk[u]);
                ldv(static_cast<const TI*>(a.dk) + row * K + c0, dk[u]);
            }
            if (gated) {
                if (GATE == 2) {
                    ldv(a.g + row * K + c0, zg[u]);
                    ldv(a.dg + row * K + c0, ug[u]);
                } else if (lane == 0) {
                    zg[u][0] = a.g[row];
                    ug[u][0] = a.dg[row];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (!in[u]) continue;
            const size_t row = (size_t)(t0 + u * PW) * H + h;
            if (a.qk_norm) {
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    float(&x)[EL] = w ? xk[u] : xq[u];
                    float(&d)[EL] = w ? dk[u] : dq[u];
                    const float r = row_rnorm<EL>(x, a.eps);
                    float dot = 0.f;
#pragma unroll
                    for (int e = 0; e < EL; ++e) dot = fmaf(x[e] * r, d[e], dot);
                    dot = warp_sum(dot);
#pragma unroll
                    for (int e = 0; e < EL; ++e) d[e] = r * (d[e] - x[e] * r * dot);
                    stv(static_cast<TI*>(w ? a.dk : a.dq) + row * K + c0, d);
                }
            }
            if (gated) {
                const int ne = (GATE == 2) ? EL : (lane == 0 ? 1 : 0);
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    if (e >= ne) break;
                    float gz, gA;
                    act_grad(zg[u][e] + db[e], eA, a.lower_bound, gz, gA);
                    const float dz = ug[u][e] * gz;
                    accA = fmaf(ug[u][e], gA, accA);
                    accz[e] += dz;
                    ug[u][e] = dz;
                }
                if (GATE == 2) stv(a.dg + row * K + c0, ug[u]);
                else if (lane == 0) a.dg[row] = ug[u][0];
            }
        }
    }
    if (!gated) return;
    // partial sums of this token block: per channel (dt_bias) and per head (A_log)
    constexpr int NC = (GATE == 2) ? K : 1;
#pragma unroll
    for (int e = 0; e < EL; ++e) sZ[warp][c0 + e] = accz[e];
    accA = warp_sum(accA);
    if (lane == 0) sAp[warp] = accA;
    __syncthreads();
    for (int c = threadIdx.x; c < NC; c += 32 * PW) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < PW; ++w) x += sZ[w][c];
        a.pz[((size_t)tb * H + h) * NC + c] = x;
    }
    if (threadIdx.x == 0) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < PW; ++w) x += sAp[w];
        a.pA[(size_t)tb * H + h] = x;
    }
}

// dt_bias's and A_log's gradients: the token-block partials added in block order.
__global__ void k_prologue_sum(int nTB, int H, int NC, const float* __restrict__ pz, const float* __restrict__ pA,
                               float* __restrict__ ddt, float* __restrict__ dA) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (ddt && i < H * NC) {
        float x = 0.f;
        for (int b = 0; b < nTB; ++b) x += pz[(size_t)b * H * NC + i];
        ddt[i] = x;
    }
    if (dA && i < H) {
        float x = 0.f;
        for (int b = 0; b < nTB; ++b) x += pA[(size_t)b * H + i];
        dA[i] = x;
    }
}

template <typename TI, int K>
cudaError_t run_prologue_k(const Shape& s, int gate, const PrologueArgs& a, cudaStream_t st) {
    const long long rows = (long long)s.Ttot * s.H;
    if (rows <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)((rows + PW - 1) / PW);
    switch (gate) {
        case 0: k_prologue<TI, K, 0><<<grid, 32 * PW, 0, st>>>((int)rows, s.H, a); break;
        case 1: k_prologue<TI, K, 1><<<grid, 32 * PW, 0, st>>>((int)rows, s.H, a); break;
        default: k_prologue<TI, K, 2><<<grid, 32 * PW, 0, st>>>((int)rows, s.H, a); break;
    }
    return cudaGetLastError();
}

template <typename TI, int K>
cudaError_t run_epilogue_k(const Shape& s, int gate, const EpilogueArgs& a, cudaStream_t st) {
    if (s.Ttot <= 0) return cudaSuccess;
    const dim3 grid((s.Ttot + ETB - 1) / ETB, s.H);
    switch (gate) {
        case 0: k_epilogue<TI, K, 0><<<grid, 32 * PW, 0, st>>>(s.Ttot, s.H, a); break;
        case 1: k_epilogue<TI, K, 1><<<grid, 32 * PW, 0, st>>>(s.Ttot, s.H, a); break;
        default: k_epilogue<TI, K, 2><<<grid, 32 * PW, 0, st>>>(s.Ttot, s.H, a); break;
    }
    return cudaGetLastError();
}

}  // namespace

int prologue_blocks(int Ttot) { return (Ttot + ETB - 1) / ETB; }

cudaError_t launch_prologue(const Shape& s, int bf16, int gate, const PrologueArgs& a, cudaStream_t st) {
    switch (s.K) {
        case 64: return bf16 ? run_prologue_k<__nv_bfloat16, 64>(s, gate, a, st) : run_prologue_k<float, 64>(s, gate, a, st);
        case 128: return bf16 ? run_prologue_k<__nv_bfloat16, 128>(s, gate, a, st) : run_prologue_k<float, 128>(s, gate, a, st);
        case 256: return bf16 ? run_prologue_k<__nv_bfloat16, 256>(s, gate, a, st) : run_prologue_k<float, 256>(s, gate, a, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_epilogue(const Shape& s, int bf16, int gate, const EpilogueArgs& a, cudaStream_t st) {
    cudaError_t e;
    switch (s.K) {
        case 64: e = bf16 ? run_epilogue_k<__nv_bfloat16, 64>(s, gate, a, st) : run_epilogue_k<float, 64>(s, gate, a, st); break;
        case 128: e = bf16 ? run_epilogue_k<__nv_bfloat16, 128>(s, gate, a, st) : run_epilogue_k<float, 128>(s, gate, a, st); break;
        case 256: e = bf16 ? run_epilogue_k<__nv_bfloat16, 256>(s, gate, a, st) : run_epilogue_k<float, 256>(s, gate, a, st); break;
        default: return cudaErrorInvalidValue;
    }
    return e;
}

cudaError_t launch_prologue_sum(const Shape& s, int gate, const EpilogueArgs& a, cudaStream_t st) {
    if (gate == 0 || !a.A_log) return cudaSuccess;
    const int NC = gate == 2 ? s.K : 1;
    const int n = s.H * NC;
    k_prologue_sum<<<(n + 255) / 256, 256, 0, st>>>(prologue_blocks(s.Ttot), s.H, NC, a.pz, a.pA, a.ddt_bias,
                                                    a.dA_log);
    return cudaGetLastError();
}

}  // namespace kda
