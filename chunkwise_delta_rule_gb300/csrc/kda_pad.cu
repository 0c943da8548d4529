// Widths the kernels do not take as they are (bf16 widths that are not multiples
// of 8, or that the in-operator prologue does not cover; fp32 widths other than
// 64 or 128; keys above 128): the problem is served
// at one width D (64, 128 or 256) with every key-side tensor zero-padded from K to D channels and
// every value-side one from V to D. Padded key channels have k = q = 0, so they
// neither write nor read the state; padded value columns of the state start at
// zero and stay zero (their write value and prediction are both zero). The
// real channels therefore see exactly the unpadded recurrence; outputs and
// gradients are cropped back. k_pad copies a batch of [R][C] matrices into
// [Rd][Cd] ones with zero fill; k_crop copies the leading [R][C] block back.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int PT2 = 256;

// One thread per destination element (32-bit indices: the callers' tensors stay below 2^31
// elements). Token rows (R = Rd = 1) skip the matrix arithmetic.
template <typename T>
__global__ void __launch_bounds__(PT2) k_pad(int n, int R, int C, int Rd, int Cd, const T* __restrict__ src,
                                             T* __restrict__ dst) {
    const int i = blockIdx.x * PT2 + threadIdx.x;
    if (i >= n) return;
    const int row = i / Cd, c = i - row * Cd;
    if (Rd == 1) {
        dst[i] = c < C ? src[(size_t)row * C + c] : T(0.f);
        return;
    }
    const int m = row / Rd, r = row - m * Rd;
    dst[i] = (r < R && c < C) ? src[((size_t)m * R + r) * C + c] : T(0.f);
}

template <typename T>
__global__ void __launch_bounds__(PT2) k_crop(int n, int R, int C, int Rd, int Cd, const T* __restrict__ src,
                                              T* __restrict__ dst) {
    const int i = blockIdx.x * PT2 + threadIdx.x;
    if (i >= n) return;
    const int row = i / C, c = i - row * C;
    if (R == 1) {
        dst[i] = src[(size_t)row * Cd + c];
        return;
    }
    const int m = row / R, r = row - m * R;
    dst[i] = src[((size_t)m * Rd + r) * Cd + c];
}

// Token rows whose widths are whole 16-byte vectors: one thread per destination vector.
__global__ void __launch_bounds__(PT2) k_pad_rows16(int n, int C16, int Cd16, const uint4* __restrict__ src,
                                                    uint4* __restrict__ dst) {
    const int i = blockIdx.x * PT2 + threadIdx.x;
    if (i >= n) return;
    const int row = i / Cd16, c = i - row * Cd16;
    dst[i] = c < C16 ? src[(size_t)row * C16 + c] : make_uint4(0, 0, 0, 0);
}
__global__ void __launch_bounds__(PT2) k_crop_rows16(int n, int C16, int Cd16, const uint4* __restrict__ src,
                                                     uint4* __restrict__ dst) {
    const int i = blockIdx.x * PT2 + threadIdx.x;
    if (i >= n) return;
    const int row = i / C16, c = i - row * C16;
    dst[i] = src[(size_t)row * Cd16 + c];
}

template <typename T>
cudaError_t run(bool pad, long long M, int R, int C, int Rd, int Cd, const void* src, void* dst, cudaStream_t st) {
    constexpr int VE = 16 / sizeof(T);
    if (R == 1 && Rd == 1 && C % VE == 0 && Cd % VE == 0 &&
        (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 16 == 0) {
        const long long n = M * (pad ? Cd : C) / VE;
        if (n <= 0) return cudaSuccess;
        if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
        const unsigned grid = (unsigned)((n + PT2 - 1) / PT2);
        if (pad)
            k_pad_rows16<<<grid, PT2, 0, st>>>((int)n, C / VE, Cd / VE, (const uint4*)src, (uint4*)dst);
        else
            k_crop_rows16<<<grid, PT2, 0, st>>>((int)n, C / VE, Cd / VE, (const uint4*)src, (uint4*)dst);
        return cudaGetLastError();
    }
    const long long n = M * (pad ? (long long)Rd * Cd : (long long)R * C);
    if (n <= 0) return cudaSuccess;
    if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)((n + PT2 - 1) / PT2);
    if (pad)
        k_pad<T><<<grid, PT2, 0, st>>>((int)n, R, C, Rd, Cd, (const T*)src, (T*)dst);
    else
        k_crop<T><<<grid, PT2, 0, st>>>((int)n, R, C, Rd, Cd, (const T*)src, (T*)dst);
    return cudaGetLastError();
}

}  // namespace

// es: element size in bytes (2: bf16, 4: fp32). pad: [M][R][C] -> [M][Rd][Cd] zero-filled;
// crop: [M][Rd][Cd] -> [M][R][C].
cudaError_t launch_pad(bool pad, int es, long long M, int R, int C, int Rd, int Cd, const void* src, void* dst,
                       cudaStream_t st) {
    return es == 2 ? run<__nv_bfloat16>(pad, M, R, C, Rd, Cd, src, dst, st) : run<float>(pad, M, R, C, Rd, Cd, src, dst, st);
}

}  // namespace kda
