// Grouped value heads: HV = G * H value heads share the H key heads, value
// head j reading q and k of key head j / G ("GatedDeltaNet-2 (NVlabs) —
// official spec transcription", the GVA head map of §3: v-head -> k-head).
// The chunked paths run on q and k expanded to one copy per value head
// (k_gva_expand), and the backward sums each group's dq and dk back onto its
// key head (k_gva_reduce, fp32 accumulation in a fixed order). Value widths
// above 128 reuse the same map with value blocks as value heads (below).
// Every copy moves 16 bytes per thread where the rows allow it.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int GT = 256;

// One thread per 16 bytes of an output row: dst[t][j][:] = src[t][j / G][:] (32-bit indices:
// the launcher checks the 16-byte count).
__global__ void __launch_bounds__(GT) k_gva_expand(unsigned chunks, unsigned HV, unsigned G, unsigned per,
                                                   const uint4* __restrict__ q, const uint4* __restrict__ k,
                                                   uint4* __restrict__ qx, uint4* __restrict__ kx) {
    const unsigned i = blockIdx.x * GT + threadIdx.x;
    if (i >= chunks) return;
    const unsigned row = i / per, off = i - row * per;   // row: (token, value head)
    const unsigned t = row / HV, j = row - t * HV;
    const size_t src = ((size_t)t * (HV / G) + j / G) * per + off;
    qx[i] = q[src];
    kx[i] = k[src];
}

// 16 bytes of TI as floats and back.
template <typename TI> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ static void add(const uint4& u, float* a) {
        a[0] += __uint_as_float(u.x); a[1] += __uint_as_float(u.y);
        a[2] += __uint_as_float(u.z); a[3] += __uint_as_float(u.w);
    }
    __device__ static uint4 pack(const float* a) {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]), __float_as_uint(a[3]));
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void add(const uint4& u, float* a) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            a[2 * e] += __uint_as_float(w[e] << 16);
            a[2 * e + 1] += __uint_as_float(w[e] & 0xffff0000u);
        }
    }
    __device__ static uint4 pack(const float* a) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * e], a[2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// dst[r][:] = sum over g < G of src[r * G + g][:], 16 bytes per thread (per = 16-byte chunks of a
// row), fp32 accumulation in group order.
template <typename TI>
__device__ __forceinline__ void group_sum16(unsigned i, unsigned G, unsigned per, const uint4* __restrict__ src,
                                            uint4* __restrict__ dst) {
    const unsigned r = i / per, c = i - r * per;
    float a[Vec16<TI>::N] = {};
    for (unsigned g = 0; g < G; ++g) Vec16<TI>::add(src[((size_t)r * G + g) * per + c], a);
    dst[i] = Vec16<TI>::pack(a);
}

// dq, dk of each key head: the sums over its group of value heads.
template <typename TI>
__global__ void __launch_bounds__(GT) k_gva_reduce(unsigned n, unsigned G, unsigned per, const uint4* __restrict__ dqx,
                                                   const uint4* __restrict__ dkx, uint4* __restrict__ dq,
                                                   uint4* __restrict__ dk) {
    const unsigned i = blockIdx.x * GT + threadIdx.x;
    if (i >= n) return;
    group_sum16<TI>(i, G, per, dqx, dq);
    group_sum16<TI>(i, G, per, dkx, dk);
}

// Value blocks. A value width V above 128 runs as NB value blocks of width Vb (NB * Vb >= V),
// each block a value head of its own: column j of the state obeys its own recurrence, driven
// by q, k, the gate and beta and by column j of v alone ("ReWY" paper, the delta-rule state
// update, which acts on the state's value columns independently), so the blocks are exact
// sub-problems. Per-head inputs repeat per block; their gradients sum over the blocks.

// dst[m][b][:] = src[m][:] for b < NB (raw copies of 2- or 4-byte elements).
template <typename T>
__global__ void __launch_bounds__(GT) k_vblock_repeat(unsigned n, unsigned NB, unsigned W, const T* __restrict__ src,
                                                      T* __restrict__ dst) {
    const unsigned i = blockIdx.x * GT + threadIdx.x;
    if (i >= n) return;
    const unsigned row = i / W, c = i - row * W;
    dst[i] = src[(size_t)(row / NB) * W + c];
}

// dst[m][:] = sum over b of src[m][b][:], fp32 accumulation in block order.
template <typename T>
__global__ void __launch_bounds__(GT) k_vblock_sum(unsigned n, unsigned NB, unsigned W, const T* __restrict__ src,
                                                   T* __restrict__ dst) {
    const unsigned i = blockIdx.x * GT + threadIdx.x;
    if (i >= n) return;
    const unsigned m = i / W, c = i - m * W;
    float s = 0.f;
    for (unsigned b = 0; b < NB; ++b) s += ld(src + ((size_t)m * NB + b) * W + c);
    st(dst + i, s);
}

// The same over 16-byte chunks (rows whose width is a whole number of them).
__global__ void __launch_bounds__(GT) k_vblock_repeat16(unsigned n, unsigned NB, unsigned per,
                                                        const uint4* __restrict__ src, uint4* __restrict__ dst) {
    const unsigned i = blockIdx.x * GT + threadIdx.x;
    if (i >= n) return;
    const unsigned row = i / per, c = i - row * per;
    dst[i] = src[(size_t)(row / NB) * per + c];
}
template <typename TI>
__global__ void __launch_bounds__(GT) k_vblock_sum16(unsigned n, unsigned NB, unsigned per,
                                                     const uint4* __restrict__ src, uint4* __restrict__ dst) {
    const unsigned i = blockIdx.x * GT + threadIdx.x;
    if (i >= n) return;
    group_sum16<TI>(i, NB, per, src, dst);
}

// States: split [M][K][V] -> [M][NB][K][Vb] (zero past column V); merge the reverse.
__global__ void __launch_bounds__(GT) k_vblock_split(unsigned n, unsigned K, unsigned V, unsigned NB, unsigned Vb,
                                                     const float* __restrict__ src, float* __restrict__ dst) {
    const unsigned i = blockIdx.x * GT + threadIdx.x;
    if (i >= n) return;
    const unsigned c = i % Vb, r = i / Vb, kk = r % K, mb = r / K, b = mb % NB, m = mb / NB;
    const unsigned j = b * Vb + c;
    dst[i] = j < V ? src[((size_t)m * K + kk) * V + j] : 0.f;
}
__global__ void __launch_bounds__(GT) k_vblock_merge(unsigned n, unsigned K, unsigned V, unsigned NB, unsigned Vb,
                                                     const float* __restrict__ src, float* __restrict__ dst) {
    const unsigned i = blockIdx.x * GT + threadIdx.x;
    if (i >= n) return;
    const unsigned j = i % V, r = i / V, kk = r % K, m = r / K, b = j / Vb, c = j - b * Vb;
    dst[i] = src[(((size_t)m * NB + b) * K + kk) * Vb + c];
}

bool aligned16(const void* a, const void* b, const void* c = nullptr, const void* d = nullptr) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(c) |
             reinterpret_cast<uintptr_t>(d)) % 16) == 0;
}

// Element count of one launch; 0 when empty, -1 when it does not fit the 32-bit indices.
long long vblock_count(long long n) { return n <= 0 ? 0 : (n > 0x7fffffffLL ? -1 : n); }

}  // namespace

cudaError_t launch_vblock_repeat(int es, long long M, int NB, int W, const void* src, void* dst, cudaStream_t st) {
    const long long n = vblock_count(M * NB * W);
    if (n == 0) return cudaSuccess;
    if (n < 0) return cudaErrorInvalidValue;
    const bool vec = (W * es) % 16 == 0 && aligned16(src, dst);
    if (vec) {
        const long long n16 = n * es / 16;
        k_vblock_repeat16<<<(unsigned)((n16 + GT - 1) / GT), GT, 0, st>>>((unsigned)n16, NB, W * es / 16,
                                                                          (const uint4*)src, (uint4*)dst);
        return cudaGetLastError();
    }
    const unsigned grid = (unsigned)((n + GT - 1) / GT);
    if (es == 2)
        k_vblock_repeat<uint16_t><<<grid, GT, 0, st>>>((unsigned)n, NB, W, (const uint16_t*)src, (uint16_t*)dst);
    else
        k_vblock_repeat<uint32_t><<<grid, GT, 0, st>>>((unsigned)n, NB, W, (const uint32_t*)src, (uint32_t*)dst);
    return cudaGetLastError();
}

cudaError_t launch_vblock_sum(int es, long long M, int NB, int W, const void* src, void* dst, cudaStream_t st) {
    const long long n = vblock_count(M * W);
    if (n == 0) return cudaSuccess;
    if (n < 0 || n * NB > 0x7fffffffLL) return cudaErrorInvalidValue;
    if ((W * es) % 16 == 0 && aligned16(src, dst)) {
        const long long n16 = n * es / 16;
        const unsigned g16 = (unsigned)((n16 + GT - 1) / GT);
        if (es == 2)
            k_vblock_sum16<__nv_bfloat16><<<g16, GT, 0, st>>>((unsigned)n16, NB, W * es / 16, (const uint4*)src, (uint4*)dst);
        else
            k_vblock_sum16<float><<<g16, GT, 0, st>>>((unsigned)n16, NB, W * es / 16, (const uint4*)src, (uint4*)dst);
        return cudaGetLastError();
    }
    const unsigned grid = (unsigned)((n + GT - 1) / GT);
    if (es == 2)
        k_vblock_sum<__nv_bfloat16><<<grid, GT, 0, st>>>((unsigned)n, NB, W, (const __nv_bfloat16*)src,
                                                         (__nv_bfloat16*)dst);
    else
        k_vblock_sum<float><<<grid, GT, 0, st>>>((unsigned)n, NB, W, (const float*)src, (float*)dst);
    return cudaGetLastError();
}

cudaError_t launch_vblock_state(bool split, long long M, int K, int V, int NB, int Vb, const float* src, float* dst,
                                cudaStream_t st) {
    const long long n = vblock_count(split ? M * NB * K * Vb : M * K * V);
    if (n == 0) return cudaSuccess;
    if (n < 0 || M * NB * K * Vb > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)((n + GT - 1) / GT);
    if (split)
        k_vblock_split<<<grid, GT, 0, st>>>((unsigned)n, K, V, NB, Vb, src, dst);
    else
        k_vblock_merge<<<grid, GT, 0, st>>>((unsigned)n, K, V, NB, Vb, src, dst);
    return cudaGetLastError();
}

cudaError_t launch_gva_expand(int Ttot, int HV, int G, int K, int bf16, const void* q, const void* k, void* qx, void* kx,
                              cudaStream_t st) {
    const int per = K * (bf16 ? 2 : 4) / 16;
    const long long chunks = (long long)Ttot * HV * per;
    if (chunks <= 0) return cudaSuccess;
    if (chunks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (!aligned16(q, k, qx, kx)) return cudaErrorMisalignedAddress;   // 16-byte rows need 16-byte bases
    k_gva_expand<<<(unsigned)((chunks + GT - 1) / GT), GT, 0, st>>>((unsigned)chunks, HV, G, per, (const uint4*)q,
                                                                   (const uint4*)k, (uint4*)qx, (uint4*)kx);
    return cudaGetLastError();
}

cudaError_t launch_gva_reduce(int Ttot, int H, int G, int K, int bf16, const void* dqx, const void* dkx, void* dq, void* dk,
                              cudaStream_t st) {
    const int per = K * (bf16 ? 2 : 4) / 16;
    const long long n = (long long)Ttot * H * per;
    if (n <= 0) return cudaSuccess;
    if (n * G > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (!aligned16(dqx, dkx, dq, dk)) return cudaErrorMisalignedAddress;
    const unsigned grid = (unsigned)((n + GT - 1) / GT);
    if (bf16)
        k_gva_reduce<__nv_bfloat16><<<grid, GT, 0, st>>>((unsigned)n, G, per, (const uint4*)dqx, (const uint4*)dkx,
                                                         (uint4*)dq, (uint4*)dk);
    else
        k_gva_reduce<float><<<grid, GT, 0, st>>>((unsigned)n, G, per, (const uint4*)dqx, (const uint4*)dkx, (uint4*)dq,
                                                 (uint4*)dk);
    return cudaGetLastError();
}

}  // namespace kda
