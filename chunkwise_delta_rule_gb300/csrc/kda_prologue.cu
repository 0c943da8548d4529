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

// x_hat = x r of one (token, head) row, r = (sum x^2 + eps)^(-1/2); lane holds x[lane + 32 j]
template <int KJ>
__device__ __forceinline__ float row_rnorm(const float (&x)[KJ], float eps) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < KJ; ++j) ss = fmaf(x[j], x[j], ss);
    return 1.f / sqrtf(warp_sum(ss) + eps);
}

template <typename TI, int K, int GATE>
__global__ void __launch_bounds__(32 * PW) k_prologue(int rows, int H, PrologueArgs a) {
    constexpr int KJ = K / 32;
    const int row = blockIdx.x * PW + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int h = row % H;
    if (a.qk_norm) {
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const TI* src = static_cast<const TI*>(w ? a.k : a.q) + (size_t)row * K + lane;
            TI* dst = static_cast<TI*>(w ? a.kh : a.qh) + (size_t)row * K + lane;
            float x[KJ];
#pragma unroll
            for (int j = 0; j < KJ; ++j) x[j] = ld(src + 32 * j);
            const float r = row_rnorm<KJ>(x, a.eps);
#pragma unroll
            for (int j = 0; j < KJ; ++j) st(dst + 32 * j, x[j] * r);
        }
    }
    if (GATE != 0 && a.A_log) {
        const float eA = expf(a.A_log[h]);
        if (GATE == 2) {
#pragma unroll
            for (int j = 0; j < KJ; ++j) {
                const int c = lane + 32 * j;
                const float z = a.g[(size_t)row * K + c] + (a.dt_bias ? a.dt_bias[h * K + c] : 0.f);
                a.ga[(size_t)row * K + c] = act(z, eA, a.lower_bound);
            }
        } else if (lane == 0) {
            const float z = a.g[row] + (a.dt_bias ? a.dt_bias[h] : 0.f);
            a.ga[row] = act(z, eA, a.lower_bound);
        }
    }
}

template <typename TI, int K, int GATE>
__global__ void __launch_bounds__(32 * PW) k_epilogue(int Ttot, int H, EpilogueArgs a) {
    constexpr int KJ = K / 32;
    __shared__ float sZ[PW][K];
    __shared__ float sAp[PW];
    const int tb = blockIdx.x, h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool gated = GATE != 0 && a.A_log;
    const float eA = gated ? expf(a.A_log[h]) : 0.f;
    float accz[KJ], accA = 0.f;
#pragma unroll
    for (int j = 0; j < KJ; ++j) accz[j] = 0.f;
    for (int t = tb * ETB + warp; t < min(Ttot, tb * ETB + ETB); t += PW) {
        const size_t row = (size_t)t * H + h;
        if (a.qk_norm) {
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const TI* xs = static_cast<const TI*>(w ? a.k : a.q) + row * K + lane;
                TI* dx = static_cast<TI*>(w ? a.dk : a.dq) + row * K + lane;
                float x[KJ], d[KJ];
#pragma unroll
                for (int j = 0; j < KJ; ++j) {
                    x[j] = ld(xs + 32 * j);
                    d[j] = ld(dx + 32 * j);
                }
                const float r = row_rnorm<KJ>(x, a.eps);
                float dot = 0.f;
#pragma unroll
                for (int j = 0; j < KJ; ++j) dot = fmaf(x[j] * r, d[j], dot);
                dot = warp_sum(dot);
#pragma unroll
                for (int j = 0; j < KJ; ++j) st(dx + 32 * j, r * (d[j] - x[j] * r * dot));
            }
        }
        if (gated) {
            if (GATE == 2) {
#pragma unroll
                for (int j = 0; j < KJ; ++j) {
                    const int c = lane + 32 * j;
                    const float z = a.g[row * K + c] + (a.dt_bias ? a.dt_bias[h * K + c] : 0.f);
                    float gz, gA;
                    act_grad(z, eA, a.lower_bound, gz, gA);
                    const float up = a.dg[row * K + c];
                    const float dz = up * gz;
                    a.dg[row * K + c] = dz;
                    accz[j] += dz;
                    accA = fmaf(up, gA, accA);
                }
            } else if (lane == 0) {
                const float z = a.g[row] + (a.dt_bias ? a.dt_bias[h] : 0.f);
                float gz, gA;
                act_grad(z, eA, a.lower_bound, gz, gA);
                const float up = a.dg[row];
                const float dz = up * gz;
                a.dg[row] = dz;
                accz[0] += dz;
                accA = fmaf(up, gA, accA);
            }
        }
    }
    if (!gated) return;
    // partial sums of this token block: per channel (dt_bias) and per head (A_log)
    constexpr int NC = (GATE == 2) ? K : 1;
#pragma unroll
    for (int j = 0; j < KJ; ++j) sZ[warp][lane + 32 * j] = accz[j];
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
    if (s.K != 64 && s.K != 128) return cudaErrorInvalidValue;
    if (bf16) return s.K == 128 ? run_prologue_k<__nv_bfloat16, 128>(s, gate, a, st)
                                : run_prologue_k<__nv_bfloat16, 64>(s, gate, a, st);
    return s.K == 128 ? run_prologue_k<float, 128>(s, gate, a, st) : run_prologue_k<float, 64>(s, gate, a, st);
}

cudaError_t launch_epilogue(const Shape& s, int bf16, int gate, const EpilogueArgs& a, cudaStream_t st) {
    if (s.K != 64 && s.K != 128) return cudaErrorInvalidValue;
    cudaError_t e = bf16 ? (s.K == 128 ? run_epilogue_k<__nv_bfloat16, 128>(s, gate, a, st)
                                       : run_epilogue_k<__nv_bfloat16, 64>(s, gate, a, st))
                         : (s.K == 128 ? run_epilogue_k<float, 128>(s, gate, a, st)
                                       : run_epilogue_k<float, 64>(s, gate, a, st));
    if (e != cudaSuccess || gate == 0 || !a.A_log) return e;
    const int NC = gate == 2 ? s.K : 1;
    const int n = s.H * NC;
    k_prologue_sum<<<(n + 255) / 256, 256, 0, st>>>(prologue_blocks(s.Ttot), s.H, NC, a.pz, a.pA, a.ddt_bias,
                                                    a.dA_log);
    return cudaGetLastError();
}

}  // namespace kda
