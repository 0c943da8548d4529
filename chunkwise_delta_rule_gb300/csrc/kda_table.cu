// Chunk table: maps chunk slots to (first token, length) and sequences to
// their chunk ranges, from cu_seqlens on the device (no host copy needed) or
// from (B, T) for equal-length batches. Chunks restart at every sequence
// start; the last chunk of a sequence holds the remainder (1..64 tokens).
// It also ranks the sequences by chunk count: the state scans are serial over
// a sequence's chunks, one CTA per (sequence, head), so dispatching the longest
// sequences first keeps a packed batch's scans from ending on a long sequence
// that started late (longest-processing-time-first list scheduling).
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int TBL_THREADS = 1024;

__global__ void __launch_bounds__(TBL_THREADS) k_table(Shape s, int B, int T,
                                                       const int32_t* __restrict__ cu, Table t, TableZeros z) {
    __shared__ int32_t s_cnt[TBL_THREADS];
    __shared__ int32_t s_bad;
    const int tid = threadIdx.x;
    const int N = s.N;
#pragma unroll
    for (int i = 0; i < 3; ++i)
        for (int j = tid; j < z.n[i]; j += TBL_THREADS) z.p[i][j] = 0;
    if (!cu) {
        // equal lengths: every entry by arithmetic, one thread per chunk slot and per sequence
        // (sequence n owns slots n per .. n per + per - 1; the ranking is the identity)
        const int per = (T + BT - 1) / BT;
        for (int slot = tid; slot < s.NC; slot += TBL_THREADS) {
            const int n = slot / per, j = slot - n * per;
            t.chunk_tok0[slot] = n * T + j * BT;
            t.chunk_len[slot] = min(BT, T - j * BT);
        }
        for (int n = tid; n < N; n += TBL_THREADS) {
            t.seq_tok0[n] = n * T;
            t.seq_len[n] = T;
            t.seq_chunk0[n] = n * per;
            t.seq_order[n] = n;
        }
        if (tid == 0) {
            t.seq_chunk0[N] = N * per;
            t.err[0] = 0;
        }
        return;
    }
    if (tid == 0) s_bad = 0;
    __syncthreads();
    const int per = (N + TBL_THREADS - 1) / TBL_THREADS;
    const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
    // clamped bounds of this thread's sequences; count their chunks
    int32_t cnt = 0;
    int bad = 0;
    for (int n = n0; n < n1; ++n) {
        int32_t a, b;
        if (cu) {
            int32_t ra = cu[n], rb = cu[n + 1];
            a = min(max(ra, 0), s.Ttot);
            b = min(max(rb, a), s.Ttot);
            if (ra != a || rb != b) bad = 1;
            if (n == 0 && ra != 0) bad = 1;
            if (n == N - 1 && rb != s.Ttot) bad = 1;
        } else {
            a = n * T;
            b = a + T;
        }
        t.seq_tok0[n] = a;
        t.seq_len[n] = b - a;
        cnt += (b - a + BT - 1) / BT;
    }
    if (bad) atomicOr(&s_bad, 1);
    s_cnt[tid] = cnt;
    __syncthreads();
    // inclusive scan of the per-thread counts (Hillis-Steele)
    for (int off = 1; off < TBL_THREADS; off <<= 1) {
        int32_t x = (tid >= off) ? s_cnt[tid - off] : 0;
        __syncthreads();
        s_cnt[tid] += x;
        __syncthreads();
    }
    int32_t c = s_cnt[tid] - cnt;  // exclusive prefix: first chunk slot of n0
    for (int n = n0; n < n1; ++n) {
        const int32_t a = t.seq_tok0[n], L = t.seq_len[n];
        const int32_t nch = (L + BT - 1) / BT;
        const int32_t c0 = min(c, s.NC);
        t.seq_chunk0[n] = c0;
        for (int j = 0; j < nch; ++j) {
            const int32_t slot = c + j;
            if (slot < s.NC) {
                t.chunk_tok0[slot] = a + j * BT;
                t.chunk_len[slot] = min(BT, L - j * BT);
            } else {
                atomicOr(&s_bad, 1);
            }
        }
        c += nch;
    }
    const int32_t total = min(s_cnt[TBL_THREADS - 1], s.NC);
    if (tid == 0) t.seq_chunk0[N] = total;
    // rank = sequences with more chunks, or as many and a lower index (seq_len of every
    // sequence is visible after the scan's barriers)
    for (int n = tid; n < N; n += TBL_THREADS) {
        int rank = n;
        if (N <= ORDER_MAX) {
            const int32_t cn = (t.seq_len[n] + BT - 1) / BT;
            rank = 0;
            for (int m = 0; m < N; ++m) {
                const int32_t cm = (t.seq_len[m] + BT - 1) / BT;
                rank += (cm > cn || (cm == cn && m < n)) ? 1 : 0;
            }
        }
        t.seq_order[rank] = n;
    }
    for (int slot = total + tid; slot < s.NC; slot += TBL_THREADS) {
        t.chunk_tok0[slot] = 0;
        t.chunk_len[slot] = 0;
    }
    __syncthreads();
    if (tid == 0) t.err[0] = s_bad ? 1 : 0;
}

// Self-test of the timeout path: one warp waits, with the library's bounded
// mbarrier wait, on a barrier that nothing arrives at. The wait gives up after
// limit_ns and the kernel sets bit 1 of the error word, exactly as a kernel of
// the pipeline does when one of its waits runs out; no copy or MMA is in
// flight, so the kernel simply returns.
__global__ void __launch_bounds__(32) k_wait_selftest(Table t, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncwarp();
    const bool ok = tc::mbar_wait_for(&bar, 0, limit_ns);
    if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicOr(t.err, 2);
}

}  // namespace

cudaError_t launch_wait_selftest(Table t, uint64_t limit_ns, cudaStream_t st) {
    k_wait_selftest<<<1, 32, 0, st>>>(t, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_table(const Shape& s, int B, int T, const int32_t* cu, Table t, cudaStream_t st,
                         const TableZeros& z) {
    k_table<<<1, TBL_THREADS, 0, st>>>(s, B, T, cu, t, z);
    return cudaGetLastError();
}

}  // namespace kda
