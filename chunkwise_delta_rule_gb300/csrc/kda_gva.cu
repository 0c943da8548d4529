// Grouped value heads: HV = G * H value heads share the H key heads, value
// head j reading q and k of key head j / G ("GatedDeltaNet-2 (NVlabs) —
// official spec transcription", the GVA head map of §3: v-head -> k-head).
// The chunked paths run on q and k expanded to one copy per value head
// (k_gva_expand), and the backward sums each group's dq and dk back onto its
// key head (k_gva_reduce, fp32 accumulation in a fixed order).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int GT = 256;

// One thread per 16 bytes of an output row: dst[t][j][:] = src[t][j / G][:].
__global__ void __launch_bounds__(GT) k_gva_expand(long long chunks, int HV, int G, int rowb,
                                                   const unsigned char* __restrict__ q, const unsigned char* __restrict__ k,
                                                   unsigned char* __restrict__ qx, unsigned char* __restrict__ kx) {
    const long long i = (long long)blockIdx.x * GT + threadIdx.x;
    if (i >= chunks) return;
    const int per = rowb / 16;
    const long long row = i / per;                 // (token, value head)
    const int off = (int)(i - row * per) * 16;
    const long long t = row / HV;
    const int j = (int)(row - t * HV);
    const long long src = (t * (HV / G) + j / G) * rowb + off;
    *reinterpret_cast<uint4*>(qx + row * rowb + off) = *reinterpret_cast<const uint4*>(q + src);
    *reinterpret_cast<uint4*>(kx + row * rowb + off) = *reinterpret_cast<const uint4*>(k + src);
}

// One thread per (token, key head, 4 consecutive channels): dst = sum over the group.
template <typename TI>
__global__ void __launch_bounds__(GT) k_gva_reduce(long long items, int H, int G, int K, const TI* __restrict__ dqx,
                                                   const TI* __restrict__ dkx, TI* __restrict__ dq, TI* __restrict__ dk) {
    const long long i = (long long)blockIdx.x * GT + threadIdx.x;
    if (i >= items) return;
    const int per = K / 4;
    const long long row = i / per;                 // (token, key head)
    const int c = (int)(i - row * per) * 4;
    const long long t = row / H;
    const int h = (int)(row - t * H);
    float sq[4] = {0.f, 0.f, 0.f, 0.f}, sk[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g = 0; g < G; ++g) {
        const long long src = (t * H * G + (long long)h * G + g) * K + c;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            sq[e] += ld(dqx + src + e);
            sk[e] += ld(dkx + src + e);
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        st(dq + row * K + c + e, sq[e]);
        st(dk + row * K + c + e, sk[e]);
    }
}

}  // namespace

cudaError_t launch_gva_expand(int Ttot, int HV, int G, int K, int bf16, const void* q, const void* k, void* qx, void* kx,
                              cudaStream_t st) {
    const int rowb = K * (bf16 ? 2 : 4);
    const long long chunks = (long long)Ttot * HV * (rowb / 16);
    if (chunks <= 0) return cudaSuccess;
    k_gva_expand<<<(unsigned)((chunks + GT - 1) / GT), GT, 0, st>>>(chunks, HV, G, rowb, (const unsigned char*)q,
                                                                   (const unsigned char*)k, (unsigned char*)qx,
                                                                   (unsigned char*)kx);
    return cudaGetLastError();
}

cudaError_t launch_gva_reduce(int Ttot, int H, int G, int K, int bf16, const void* dqx, const void* dkx, void* dq, void* dk,
                              cudaStream_t st) {
    const long long items = (long long)Ttot * H * (K / 4);
    if (items <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)((items + GT - 1) / GT);
    if (bf16)
        k_gva_reduce<__nv_bfloat16><<<grid, GT, 0, st>>>(items, H, G, K, (const __nv_bfloat16*)dqx,
                                                         (const __nv_bfloat16*)dkx, (__nv_bfloat16*)dq, (__nv_bfloat16*)dk);
    else
        k_gva_reduce<float><<<grid, GT, 0, st>>>(items, H, G, K, (const float*)dqx, (const float*)dkx, (float*)dq,
                                                 (float*)dk);
    return cudaGetLastError();
}

}  // namespace kda
