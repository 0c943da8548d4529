// Internal declarations shared by the CUDA translation units of libkda.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int BT = 64;        // chunk length C
constexpr int BC = 16;        // sub-chunk length used by the strong-gate path
constexpr int NTHREADS = 256; // threads per CTA for every kernel

// Gate-range threshold of the centered matrix-intra path, in log2 units: a
// chunk whose per-feature range of cumulative log2-decay exceeds it takes the
// 16-token anchored path instead.
constexpr float CENTER_RANGE_LOG2 = 80.0f;

constexpr float LOG2E = 1.4426950408889634f;

// The bf16 tensor-core intermediates (W, F, Q_g, C_q, A) are stored in HBM as
// images of their shared-memory operand tiles: a [R][C] tile (C = 64 or 128)
// in the K-major 128-byte swizzle layout (64-column atom blocks of R rows of
// 128 bytes; the 16-byte chunk c of row r sits at position c ^ (r % 8)), so a
// single bulk copy stages a whole tile. Element offset of (r, col):
__host__ __device__ __forceinline__ int tile_el(int R, int r, int col) {
    return ((col >> 6) * R + r) * 64 + ((((col >> 3) & 7) ^ (r & 7)) << 3) + (col & 7);
}

// TMA tensor maps of a token-major input [Ttot][H][D] whose boxes are one
// head's 64-token chunk rows: bf16 in 64-column boxes with the 128-byte swizzle
// (each lands as one atom column of a K-major operand tile), fp32 in one
// unswizzled [64][box_x] box (box_x = D when 0). D may be narrower than the
// 128-column tiles (a multiple of 8 for bf16, 4 for fp32): the columns past D
// read as zeros and stores past D are dropped. False if the map cannot be
// encoded.
bool tmap_rows_bf16(CUtensorMap* m, const void* base, int Ttot, int H, int D);
bool tmap_rows_f32(CUtensorMap* m, const void* base, int Ttot, int H, int D, int box_x = 0);
// fp32 states [NH][K][V] in boxes of 32 keys x 32 value columns, 128-byte swizzled (K, V multiples of
// 32; false when the base is not 16-byte aligned).
bool tmap_state_f32(CUtensorMap* m, const float* base, int NH, int K, int V);

// Chunk bookkeeping built on the device from cu_seqlens (or from B, T).
struct Table {
    int32_t* chunk_tok0;  // [NC] first token of the chunk (packed axis)
    int32_t* chunk_len;   // [NC] tokens in the chunk; 0 marks an unused slot
    int32_t* seq_chunk0;  // [N+1] first chunk slot of each sequence
    int32_t* seq_tok0;    // [N] first token of each sequence
    int32_t* seq_len;     // [N] tokens of each sequence
    int32_t* seq_order;   // [N] sequences by chunk count, most chunks first (ties by index; identity
                          //     above ORDER_MAX sequences): the order the scans' CTAs take them in
    int32_t* err;         // [1] device error word
};
// Packed batches of up to this many sequences get their scans dispatched longest first.
constexpr int ORDER_MAX = 256;

// Forward chunk intermediates, fp32, one block per (chunk slot, head).
struct Fwd {
    float* W;     // [NC,H,BT,K]  A E
    float* U;     // [NC,H,BT,V]  A Z
    float* KG;    // [NC,H,BT,K]  F = keys decayed to the chunk end
    float* QG;    // [NC,H,BT,K]  Q_g = scale q decayed from the chunk start
    float* AQK;   // [NC,H,BT,BT] C_q
    float* AINV;  // [NC,H,BT,BT] A = (I + L)^-1
    float* GL;    // [NC,H,K]     cumulative log2-decay at the chunk's last token
    float* R;     // [NC,H,BT,V]  corrections R (filled by the recompute scan)
    float* SIN;   // [NC,H,K,V]   state entering the chunk (recompute scan)
};

// Backward chunk intermediates, fp32.
struct Bwd {
    float* P;     // [NC,H,BT,V]  shared sensitivity A^T R_bar
    float* SBP;   // [NC,H,K,V]   adjoint of the state leaving the chunk
    float* QS;    // [NC,H,BT,K]  dO S^T
    float* PS;    // [NC,H,BT,K]  -P S^T
    float* FB;    // [NC,H,BT,K]  R S+bar^T
    float* DM;    // [NC,H,BT,BT] D = -L_<(P R^T)
    float* HQ;    // [NC,H,BT,BT] H_q = L_<=(dO R^T)
    float* LAMB;  // [NC,H,K]     rowsum(S .* S+bar)
    float* DBW;   // [NC,H,BT]    <v_i, P_i>
};

// Chunk intermediates of the tensor-core (bf16 I/O, K = V = 128) path, each
// stored once in its natural [row][col] layout (the MMAs read them K-major or
// MN-major as needed).
struct FwdTC {
    __nv_bfloat16* W;     // [NC,H,BT,D]  W = A E, rows = chunk tokens
    __nv_bfloat16* KG;    // [NC,H,BT,D]  F (keys decayed to the chunk end)
    __nv_bfloat16* QG;    // [NC,H,BT,D]  Q_g
    __nv_bfloat16* AQK;   // [NC,H,BT,BT] C_q, rows = receiving token i
    __nv_bfloat16* U;     // [NC,H,BT,D]  U = A Z, rows = chunk tokens (bf16, as the other WY factors)
    float* GL;            // [NC,H,D]     cumulative log2-decay at the last token
    int32_t* WIDE;        // [NC,H]       1: gate range too wide for one anchor
    int32_t* WLIST;       // [1 + NC*H]   count, then chunk slot * H + head of every WIDE chunk
    // backward-only (null in the forward)
    __nv_bfloat16* AI;    // [NC,H,BT,BT] A = (I + L)^-1
    float* ALK;           // alpha = 2^(G2 - c) and 2^c, 2^(G2_last - c) for the backward consumer:
                          // per-channel gate [NC,H][ALK_UNIT] (fp32 token rows of 128, then a row of
                          // each per key); scalar gate [NC,H][ALK_SCALAR] (per token, then the two)
    __nv_bfloat16* HS;    // [NC,H,D,D]   state entering the chunk, [key][value]
    __nv_bfloat16* R;     // [NC,H,BT,D]  corrections
};

// Floats per (chunk, head) of FwdTC::ALK: per-channel gate, alpha as [BT][128] token rows and two
// rows of 128; scalar gate, BT alphas and the two constants (padded to 16 bytes).
constexpr int ALK_UNIT = 128 * BT + 2 * 128;
constexpr int ALK_SCALAR = BT + 16;

// Backward intermediates of the tensor-core path (bf16, [row][col] as named).
struct BwdTC {
    __nv_bfloat16* SBP;   // [NC,H,D,D]   adjoint of the state leaving the chunk, [key][value]
    __nv_bfloat16* P;     // [NC,H,BT,D]  shared sensitivity P = A^T R_bar, [token][value]
};

// Single-anchor limit of the tensor-core prep (log2 units of the per-feature
// in-chunk gate range); wider chunks are prepared on CUDA cores.
constexpr float PREP_RANGE_LOG2 = 80.0f;

struct Shape {
    int H, K, V;  // H: value heads (one state each)
    int N;        // sequences
    int NC;       // chunk slots (upper bound)
    int Ttot;     // tokens on the packed axis
    float scale;
    // Value heads per head of q, k (Gq) and per head of g, beta, erase (Gg): value head h reads
    // q, k of head h / Gq and g, beta, erase of head h / Gg, so grouped heads and value blocks
    // read those inputs in place (1 and 1 on every path but the tensor-core one). Hq = H / Gq and
    // Hg = H / Gg are the head counts of those rows, set with them (kernel parameters, so no
    // register holds them).
    int Gq = 1, Gg = 1, Hq = 0, Hg = 0;
};
// Head counts of the q, k and of the g, beta, erase rows.
__host__ __device__ __forceinline__ int heads_q(const Shape& s) { return s.Hq; }
__host__ __device__ __forceinline__ int heads_g(const Shape& s) { return s.Hg; }

// ---------------------------------------------------------------- element I/O
__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
// read-only loads (data no launch writes while it runs)
__device__ __forceinline__ float ldg(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldg(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }

// Fills an [R][C] tile: v = get(r, c), then put(r, c, v), over the CTA's threads (consecutive
// threads take consecutive c, so the loads coalesce). The loads of a batch of B elements per
// thread are all issued before any of their stores, so a tile costs about IT / B memory latencies
// instead of IT (IT = R C / NTHREADS elements per thread).
template <int R, int C, int B = 16, class G, class P>
__device__ __forceinline__ void tile_copy(G get, P put) {
    static_assert((R * C) % NTHREADS == 0, "tile must split evenly over the threads");
    constexpr int IT = R * C / NTHREADS;
    constexpr int BB = IT < B ? IT : B;
    static_assert(IT % BB == 0, "batch must divide the per-thread count");
#pragma unroll 1
    for (int i0 = 0; i0 < IT; i0 += BB) {
        float v[BB];
#pragma unroll
        for (int i = 0; i < BB; ++i) {
            const int idx = (int)threadIdx.x + (i0 + i) * NTHREADS;
            v[i] = get(idx / C, idx % C);
        }
#pragma unroll
        for (int i = 0; i < BB; ++i) {
            const int idx = (int)threadIdx.x + (i0 + i) * NTHREADS;
            put(idx / C, idx % C, v[i]);
        }
    }
}

// ------------------------------------------------------- CUDA-core tile GEMM
// acc[i][j] += sum_{kk < Kdim} A(m_i, kk) * B(kk, n_j) over the calling
// thread's share of an M x N tile: threads are laid out TMX x TNX with
// TNX = N / TN lanes along n (consecutive lanes take consecutive n), and the
// thread's rows / columns are strided: m_i = tm + i*TMX, n_j = tn + j*TNX.
// A and B are callables reading shared memory.
template <int M, int N, int TM, int TN>
struct TileMap {
    static constexpr int TNX = N / TN;
    static constexpr int TMX = M / TM;
    static_assert(TNX * TMX == NTHREADS, "tile shape must use every thread");
    __device__ __forceinline__ static int tn() { return threadIdx.x % TNX; }
    __device__ __forceinline__ static int tm() { return threadIdx.x / TNX; }
    __device__ __forceinline__ static int row(int i) { return tm() + i * TMX; }
    __device__ __forceinline__ static int col(int j) { return tn() + j * TNX; }
};

template <int M, int N, int TM, int TN, class FA, class FB>
__device__ __forceinline__ void tile_gemm(float (&acc)[TM][TN], int k0, int k1, FA A, FB B) {
    using TMp = TileMap<M, N, TM, TN>;
    const int tm = TMp::tm(), tn = TMp::tn();
#pragma unroll 2
    for (int kk = k0; kk < k1; ++kk) {
        float a[TM], b[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) a[i] = A(tm + i * TMp::TMX, kk);
#pragma unroll
        for (int j = 0; j < TN; ++j) b[j] = B(kk, tn + j * TMp::TNX);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
}

// The same product with A row-major in shared memory, A(m, kk) = pa[m * lda + kk], rows of
// 16-byte aligned storage (lda % 4 == 0): four steps of kk per 16-byte load of each of the
// thread's rows (k0, k1 multiples of 4). Rows as TileMap, or with BLK as TileMapB (below);
// columns as TileMap.
template <int M, int N, int TM, int TN, bool BLK = false, class FB>
__device__ __forceinline__ void tile_gemm_ar(float (&acc)[TM][TN], const float* pa, int lda, int k0, int k1, FB B) {
    using TMp = TileMap<M, N, TM, TN>;
    const int tm = TMp::tm(), tn = TMp::tn();
#pragma unroll 1
    for (int kk = k0; kk < k1; kk += 4) {
        float4 a[TM];
        float b[4][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int m = BLK ? tm * TM + i : tm + i * TMp::TMX;
            a[i] = *reinterpret_cast<const float4*>(pa + m * lda + kk);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < TN; ++j) b[q][j] = B(kk + q, tn + j * TMp::TNX);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                acc[i][j] = fmaf(a[i].x, b[0][j], acc[i][j]);
                acc[i][j] = fmaf(a[i].y, b[1][j], acc[i][j]);
                acc[i][j] = fmaf(a[i].z, b[2][j], acc[i][j]);
                acc[i][j] = fmaf(a[i].w, b[3][j], acc[i][j]);
            }
    }
}

// The product with both operands contiguous along the contraction: A(m, kk) = pa[m * lda + kk],
// B(kk, n) = pb[n * ldb + kk], four steps of kk per 16-byte load of each row (lda, ldb % 4 == 0;
// ldb % 32 == 4 puts the loads of eight consecutive columns on distinct banks). Rows and columns
// as TileMap; k0, k1 multiples of 4.
template <int M, int N, int TM, int TN>
__device__ __forceinline__ void tile_gemm_nt(float (&acc)[TM][TN], const float* pa, int lda, const float* pb, int ldb,
                                             int k0, int k1) {
    using TMp = TileMap<M, N, TM, TN>;
    const int tm = TMp::tm(), tn = TMp::tn();
#pragma unroll 1
    for (int kk = k0; kk < k1; kk += 4) {
        float4 a[TM], b[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) a[i] = *reinterpret_cast<const float4*>(pa + (tm + i * TMp::TMX) * lda + kk);
#pragma unroll
        for (int j = 0; j < TN; ++j) b[j] = *reinterpret_cast<const float4*>(pb + (tn + j * TMp::TNX) * ldb + kk);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                acc[i][j] = fmaf(a[i].x, b[j].x, acc[i][j]);
                acc[i][j] = fmaf(a[i].y, b[j].y, acc[i][j]);
                acc[i][j] = fmaf(a[i].z, b[j].z, acc[i][j]);
                acc[i][j] = fmaf(a[i].w, b[j].w, acc[i][j]);
            }
    }
}

// Blocked row map: the thread's TM rows are consecutive, m_i = tm * TM + i (columns as TileMap).
template <int M, int N, int TM, int TN>
struct TileMapB {
    using Base = TileMap<M, N, TM, TN>;
    __device__ __forceinline__ static int row(int i) { return Base::tm() * TM + i; }
    __device__ __forceinline__ static int col(int j) { return Base::col(j); }
};

// The product with A stored transposed in shared memory, A(m, kk) = pa[kk * lda + m] (lda % 4 == 0),
// on the blocked row map: a thread's TM consecutive rows come in TM / 4 16-byte loads per kk.
template <int M, int N, int TM, int TN, class FB>
__device__ __forceinline__ void tile_gemm_at(float (&acc)[TM][TN], const float* pa, int lda, int k0, int k1, FB B) {
    static_assert(TM % 4 == 0, "blocked rows come four at a time");
    using TMp = TileMap<M, N, TM, TN>;
    const int m0 = TMp::tm() * TM, tn = TMp::tn();
#pragma unroll 2
    for (int kk = k0; kk < k1; ++kk) {
        float4 a[TM / 4];
        float b[TN];
#pragma unroll
        for (int i = 0; i < TM / 4; ++i) a[i] = *reinterpret_cast<const float4*>(pa + kk * lda + m0 + 4 * i);
#pragma unroll
        for (int j = 0; j < TN; ++j) b[j] = B(kk, tn + j * TMp::TNX);
#pragma unroll
        for (int i = 0; i < TM / 4; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                acc[4 * i][j] = fmaf(a[i].x, b[j], acc[4 * i][j]);
                acc[4 * i + 1][j] = fmaf(a[i].y, b[j], acc[4 * i + 1][j]);
                acc[4 * i + 2][j] = fmaf(a[i].z, b[j], acc[4 * i + 2][j]);
                acc[4 * i + 3][j] = fmaf(a[i].w, b[j], acc[4 * i + 3][j]);
            }
    }
}

template <int TM, int TN>
__device__ __forceinline__ void zero(float (&acc)[TM][TN]) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
}

// Raises a kernel's dynamic shared-memory limit once per device (so that no
// attribute call is issued again once a stream is being captured).
// Streaming multiprocessors of the current device (cached per device).
inline int sm_count() {
    static int cnt[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cnt[dev]) {
        int v = 0;
        cnt[dev] = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 148;
    }
    return cnt[dev];
}

template <auto Kern>
inline cudaError_t set_smem_once(size_t bytes) {
    static int done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
    return e;
}

// Sets the message kda_last_error() returns on this host thread.
void set_last_error(const char* msg);

// --------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error. Defined in the .cu files.
// Self-test of the device-timeout path (sets bit 1 of t.err after a bounded wait of limit_ns).
cudaError_t launch_wait_selftest(Table t, uint64_t limit_ns, cudaStream_t st);
// Counters the chunk table's launch zeroes as well (the list of wide chunks, the backward's claim
// counters and ready flags), so that they need no launches of their own.
struct TableZeros {
    int32_t* p[3] = {nullptr, nullptr, nullptr};
    int n[3] = {0, 0, 0};
};
cudaError_t launch_table(const Shape& s, int B, int T, const int32_t* cu, Table t, cudaStream_t st,
                         const TableZeros& z = TableZeros{});
// GatedDeltaNet-2 ("GatedDeltaNet-2 (NVlabs) — official spec transcription", §3):
// an erase vector b per key channel and a write vector w per value channel take
// beta's place (E = b .* K exp(G), Z = w .* V); erase NULL: the beta rule. Every
// chunk kernel that reads beta takes it; derase / dwrite receive the gradients.
struct Gdn2 {
    const void* erase = nullptr;   // [tokens, H, K] io dtype
    const void* write = nullptr;   // [tokens, H, V] io dtype
    void* derase = nullptr;
    void* dwrite = nullptr;
};

// the optional input transforms (kda_prologue.cu): q, k normalised, decay activated
struct PrologueArgs {
    const void *q, *k;                      // raw q, k (io dtype)
    const float *g, *A_log, *dt_bias;       // raw gate and its parameters (A_log NULL: no activation)
    float lower_bound, eps;
    int qk_norm;
    void *qh, *kh;                          // normalised q, k (io dtype)
    float* ga;                              // activated decay, shaped like g
};
struct EpilogueArgs {
    const void *q, *k;
    const float *g, *A_log, *dt_bias;
    float lower_bound, eps;
    int qk_norm;
    void *dq, *dk;                          // in: gradients w.r.t. the normalised q, k; out: w.r.t. raw
    float* dg;                              // in: w.r.t. the activated decay; out: w.r.t. the raw gate
    float *pz, *pA;                         // per 64-token block partial sums [blocks][H][K or 1], [blocks][H]
    float *ddt_bias, *dA_log;               // outputs (either may be NULL)
};
int prologue_blocks(int Ttot);
cudaError_t launch_prologue(const Shape& s, int bf16, int gate, const PrologueArgs& a, cudaStream_t st);
cudaError_t launch_epilogue(const Shape& s, int bf16, int gate, const EpilogueArgs& a, cudaStream_t st);
// dt_bias's and A_log's gradients from the epilogue's token-block partial sums (no-op without A_log).
cudaError_t launch_prologue_sum(const Shape& s, int gate, const EpilogueArgs& a, cudaStream_t st);
// unequal or narrower widths (kda_pad.cu): [M][R][C] <-> [M][Rd][Cd], zero fill (es = element bytes)
cudaError_t launch_pad(bool pad, int es, long long M, int R, int C, int Rd, int Cd, const void* src, void* dst,
                       cudaStream_t st);
// grouped value heads (kda_gva.cu): q, k copied per value head; dq, dk summed per group
cudaError_t launch_gva_expand(int Ttot, int HV, int G, int K, int bf16, const void* q, const void* k, void* qx, void* kx,
                              cudaStream_t st);
cudaError_t launch_gva_reduce(int Ttot, int H, int G, int K, int bf16, const void* dqx, const void* dkx, void* dq, void* dk,
                              cudaStream_t st);
// Value blocks (value widths above 128): es is the element size in bytes (2: bf16, 4: fp32).
// repeat: [M][W] -> [M][NB][W]; sum: [M][NB][W] -> [M][W]; state split: [M][K][V] ->
// [M][NB][K][Vb] zero past column V, merge the reverse.
cudaError_t launch_vblock_repeat(int es, long long M, int NB, int W, const void* src, void* dst, cudaStream_t st);
cudaError_t launch_vblock_sum(int es, long long M, int NB, int W, const void* src, void* dst, cudaStream_t st);
cudaError_t launch_vblock_state(bool split, long long M, int K, int V, int NB, int Vb, const float* src, float* dst,
                                cudaStream_t st);
// token-by-token forward (kda_recurrent.cu); T = tokens per sequence when cu is NULL. Key widths it
// is built for (recurrent_key_width); V any multiple of 32.
bool recurrent_key_width(int K);
cudaError_t launch_recurrent(const Shape& s, int bf16, int gate, int T, const int32_t* cu, const void* q,
                             const void* k, const void* v, const void* beta, const float* g, const float* h0,
                             void* o, float* ht, int32_t* err, const float* A_log, const float* dt_bias,
                             float lower_bound, int qk_norm, float eps, cudaStream_t st, const Gdn2& gd = Gdn2{},
                             int group = 1);

cudaError_t launch_prep(const Shape& s, int io_bf16, int gate, const void* q, const void* k,
                        const void* v, const void* beta, const float* g, Table t, Fwd f,
                        cudaStream_t st, const Gdn2& gd = Gdn2{});

// mode bit 0: write o; bit 1: write R and SIN for the backward pass.
cudaError_t launch_fwd_scan(const Shape& s, int io_bf16, int mode, const float* h0, Table t,
                            Fwd f, void* o, float* ht, cudaStream_t st);

// Tensor-core path (bf16 I/O, K = V = 128). The prep appends to the list of wide chunks, whose
// count the caller zeroes first (the chunk table's launch does).
cudaError_t launch_prep_tc(const Shape& s, int gate, int for_bwd, const void* q, const void* k,
                           const void* v, const void* beta, const float* g, Table t, FwdTC f,
                           cudaStream_t st, const Gdn2& gd = Gdn2{});
// CUDA-core prep of the chunks flagged WIDE, written in the tensor-core layouts.
cudaError_t launch_prep_wide(const Shape& s, int gate, const void* q, const void* k, const void* v,
                             const void* beta, const float* g, Table t, FwdTC ft, cudaStream_t st,
                             const Gdn2& gd = Gdn2{});
cudaError_t launch_fwd_scan_tc(const Shape& s, int mode, const float* h0, Table t, FwdTC f, void* o,
                               float* ht, cudaStream_t st);

// A time piece of the backward for a batch of equal-length sequences of `per` chunks each: chunks
// lo .. lo+L-1 of every sequence (L = 0: every chunk of every sequence). The reverse scan runs one
// piece per launch, latest first, handing the state adjoint on through dht / dh0; the consumer of a
// piece claims its units from ctr (zeroed before the launch; NULL: a fixed stride per CTA).
constexpr int MAX_PIECES = 8;       // time pieces of the tensor-core backward, at most
// The joint schedule (flags set): every unit in one launch, latest chunk first, each waiting for the
// ready flag of its (chunk slot, head) that the reverse scan sets; ctr hands out the unit indices.
struct ConsPiece {
    int lo = 0, L = 0, per = 0;
    int* ctr = nullptr;
    int* flags = nullptr;
};
constexpr int SCHEDULE_JOINT = 9;   // kda_problem.schedule value of the joint schedule
cudaError_t launch_bwd_scan_tc(const Shape& s, const void* dout, const float* dht, Table t, FwdTC f,
                               BwdTC b, float* dh0, cudaStream_t st, const ConsPiece& pc = ConsPiece{});
// The joint schedule: reverse scans and consumer in one cooperative launch of one CTA per SM
// (N * H at most the SM count; pc.per, pc.ctr and pc.flags set, ctr and flags zeroed before the launch).
cudaError_t launch_bwd_joint_tc(const Shape& s, int gate, const void* q, const void* k, const void* v,
                                const void* beta, const void* dout, const float* dht, float* dh0,
                                Table t, FwdTC f, BwdTC b, void* dq, void* dk, void* dv, void* dbeta, float* dg,
                                cudaStream_t st, const Gdn2& gd, const ConsPiece& pc);
cudaError_t launch_bwd_consumer_tc(const Shape& s, int gate, const void* q, const void* k, const void* v,
                                   const void* beta, const void* dout, Table t, FwdTC f,
                                   BwdTC b, void* dq, void* dk, void* dv, void* dbeta, float* dg,
                                   cudaStream_t st, const Gdn2& gd = Gdn2{}, const ConsPiece& pc = ConsPiece{});
// CUDA-core consumers for the WIDE chunks of the tensor-core path (reading its
// bf16 intermediates, fp32 scratch in `scratch`).
cudaError_t launch_bwd_wide(const Shape& s, int gate, const void* q, const void* k, const void* v,
                            const void* beta, const float* g, const void* dout, Table t, FwdTC f,
                            BwdTC b, Bwd scratch, void* dq, void* dk, void* dv, void* dbeta, float* dg,
                            cudaStream_t st, const Gdn2& gd = Gdn2{});

cudaError_t launch_bwd_scan(const Shape& s, int io_bf16, const void* dout, const float* dht,
                            Table t, Fwd f, Bwd b, float* dh0, cudaStream_t st);

cudaError_t launch_bwd_dstate(const Shape& s, int io_bf16, const void* dout, const void* v,
                              const void* beta, Table t, Fwd f, Bwd b, void* dv,
                              cudaStream_t st, const Gdn2& gd = Gdn2{});

cudaError_t launch_bwd_intra(const Shape& s, int io_bf16, int gate, const void* q,
                             const void* k, const void* beta, const float* g, Table t, Fwd f,
                             Bwd b, void* dq, void* dk, void* dbeta, float* dg,
                             cudaStream_t st, const Gdn2& gd = Gdn2{});

}  // namespace kda
