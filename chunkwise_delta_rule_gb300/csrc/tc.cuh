// Thin inline-PTX layer for the 5th-generation tensor cores (tcgen05) of
// sm_103a: TMEM allocation, shared-memory operand descriptors, instruction
// descriptors, MMA issue / commit, TMEM loads and stores, mbarriers with
// bounded waits, and the proxy fences that order them.
//
// Operand convention used by every kernel here: K-major tiles in the 128-byte
// swizzle layout. A tile of R rows (the M or N index) by 128 bytes of K is an
// "atom column": row r lives at byte r*128, its 16-byte chunk c is stored at
// chunk position c ^ (r % 8); 8-row groups are 1024 bytes apart. Wider K uses
// further atom columns of R*128 bytes each. Atom columns start on 1024-byte
// boundaries. The accumulator of an M = 128 MMA keeps row i in TMEM lane i.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_internal.cuh"


namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ swizzled tiles
// Byte offset of (row r, byte b within the K extent) in a K-major SW128 tile
// with R rows.
__device__ __forceinline__ uint32_t sw128_off(int R, int r, int b) {
    const int atom = b >> 7;           // which 128-byte atom column
    const int inrow = b & 127;
    const int chunk = inrow >> 4;
    return (uint32_t)(atom * R * 128 + r * 128 + (((chunk ^ (r & 7)) << 4) | (inrow & 15)));
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle, SBO = 1024 B.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;     // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;   // stride byte offset: 8-row groups
    d |= (uint64_t)1 << 46;              // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// Descriptor of k-step s (K = 16 bf16 or 8 tf32 elements = 32 bytes) of a tile
// with R rows starting at saddr.
__device__ __forceinline__ uint64_t sdesc_k(uint32_t saddr, int R, int s) {
    return sdesc(saddr + (uint32_t)((s >> 2) * R * 128 + (s & 3) * 32));
}

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle
// layout: rows are K indices (128 bytes of MN each, swizzled exactly like a
// K-major tile with R = K rows), 8-row K groups 1024 bytes apart (SBO),
// 64-element MN atoms `atom_stride` bytes apart (LBO). k-step s (16 K rows of
// bf16) starts 2048 bytes further.
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr, uint32_t atom_stride, int s) {
    const uint32_t a = saddr + (uint32_t)s * 2048u;
    uint64_t d = 0;
    d |= (uint64_t)((a & 0x3FFFFu) >> 4);
    d |= (uint64_t)((atom_stride >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptors (dense, fp32 accumulator, K-major A and B).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// bf16, K-major A, MN-major B.
__host__ __device__ constexpr uint32_t idesc_bf16_bmn(int M, int N) { return idesc_bf16(M, N) | (1u << 16); }
// bf16, MN-major A, K-major B.
__host__ __device__ constexpr uint32_t idesc_bf16_amn(int M, int N) { return idesc_bf16(M, N) | (1u << 15); }
// bf16, MN-major A and B.
__host__ __device__ constexpr uint32_t idesc_bf16_abmn(int M, int N) { return idesc_bf16(M, N) | (3u << 15); }
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase with the given parity; gives up once more than limit_ns
// nanoseconds have passed (checked every 256 tries) and returns false.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}
// The wait every kernel uses: gives up after ~1 s and returns false (the
// caller then records a device timeout and unwinds).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, 1000000000ull);
}
// A plain arrival (release at CTA scope) on a barrier of count 1.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Bulk copy (TMA, no tensor map) of `bytes` contiguous bytes global -> shared;
// completion is signalled as transaction bytes on `bar`. Both addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// TMA load of one box of a 3-D tensor map at element coordinates (x, y, z)
// into shared memory (1024-byte aligned for swizzled maps); completion as
// transaction bytes on bar. x times the element size must be a multiple of 16.
__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// TMA store of one box of a 3-D tensor map at (x, y, z) from shared memory
// (laid out as the map's swizzle expects), in this thread's bulk group. The
// box is written whole: use it only where every row of the box is the caller's.
__device__ __forceinline__ void tma_store3(const CUtensorMap* map, int x, int y, int z, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

// Bulk copy shared -> global (no tensor map) in this thread's bulk group; both
// addresses 16-byte aligned, bytes a multiple of 16. commit / wait_read /
// wait_all manage the thread's groups (wait_read: the shared source may be
// reused; wait_all: the writes are complete).
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// All but the most recent group have finished reading their shared source.
__device__ __forceinline__ void bulk_wait_read_prev() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// The writes of all but the most recent group are complete.
__device__ __forceinline__ void bulk_wait_prev() { asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); }

// Cross-SM hand-off of data written to global memory. publish: after the writes are complete
// (bulk copies: waited for; generic stores: this thread's, or the CTA's after a barrier), orders
// them before a release store of 1 to the flag. ready: an acquire load of the flag; once it reads
// nonzero, bulk copies issued afterwards see the published data.
__device__ __forceinline__ void publish_flag(int* flag) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}
__device__ __forceinline__ bool flag_set(const int* flag) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    return v != 0;
}
// Waits (about 1 s at most) for a published flag; false if it never came, or at once if the error
// word err already records a wait that gave up (so that one lost flag costs one second, not one per
// waiting unit). The caller records a failure in err.
__device__ __forceinline__ bool wait_flag(const int* flag, const int32_t* err) {
    if (!flag_set(flag)) {
        const uint64_t t0 = global_ns();
        for (uint32_t i = 1;; ++i) {
            if (flag_set(flag)) break;
            if ((i & 63u) == 0 &&
                (global_ns() - t0 > 1000000000ull || (*reinterpret_cast<const volatile int32_t*>(err) & 2)))
                return false;
            __nanosleep(64);
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// Named CTA barrier (id 1..15; 0 is __syncthreads): waits for `count` threads
// (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Asks for the 128-byte line holding p to be brought into L2 (no register, no completion).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ------------------------------------------------------------------- fences
// Generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// --------------------------------------------------------------------- TMEM
// Whole-warp operations.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// TMEM address of lane `lane`, column `col` relative to base.
__device__ __forceinline__ uint32_t taddr(uint32_t base, int lane, int col) {
    return base + ((uint32_t)lane << 16) + (uint32_t)col;
}

// 32 lanes x 32 bits, 16 consecutive columns per thread (lane = warp quarter
// base + lane id).
__device__ __forceinline__ void tmem_ld16(uint32_t a, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(a));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 32 bits, 8 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld8(uint32_t a, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(a));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16u(uint32_t a, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(a),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t a, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(a),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------- MMA
// D[tmem] (+)= A[smem] * B[smem]^T-in-K-major, single thread.
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], tf32; A is M lanes x K columns of 32-bit values.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Warp-wide forms: every lane of the warp executes them with the same
// (warp-uniform) operands and the elected leader lane issues, so the
// descriptors stay in uniform registers. Commits must come from the same
// warp, which elects the same leader while all lanes are active.
__device__ __forceinline__ void mma_bf16_w(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// A from TMEM: M = 128 lanes (row i in lane i), K along columns with two bf16
// per 32-bit column (lower half = lower k); k-step s starts at column a + 8 s.
__device__ __forceinline__ void mma_bf16_ts_w(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_w(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_ts_w(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}
// Descriptor of k-step s from the descriptor of k-step 0 (the start address
// field holds address / 16; shared-memory addresses stay below 2^18).
__device__ __forceinline__ uint64_t kstep_k(uint64_t d0, int R, int s) {
    return d0 + (uint64_t)(((s >> 2) * R * 128 + (s & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t kstep_mn(uint64_t d0, int s) { return d0 + (uint64_t)(s * 2048 >> 4); }

// Completion of all previously issued MMAs of this thread arrives once on bar.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// cp.async (16 bytes; src_bytes < 16 zero-fills the rest) and its groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes = 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// A warp holds a 32-row x 16-column block of an M = 128 accumulator (lane t:
// row t, a[0..15]). Writes its transpose, dst[c * ld + t] for c < ncols rows
// of the destination, as 16-byte stores through a per-warp staging tile of
// 16 x 40 bf16.
// wcols: columns of the 32 that exist in dst (a multiple of 8; 32 for a full block).
__device__ __forceinline__ void warp_store_t16(__nv_bfloat16* stg, const float (&a)[16], __nv_bfloat16* dst,
                                               size_t ld, int ncols, int lane, int wcols = 32) {
#pragma unroll
    for (int j = 0; j < 16; ++j) stg[j * 40 + lane] = __float2bfloat16_rn(a[j]);
    __syncwarp();
#pragma unroll
    for (int p = lane; p < 64; p += 32) {
        const int r = p >> 2, q = p & 3;
        if (r < ncols && q * 8 < wcols)
            *reinterpret_cast<uint4*>(dst + (size_t)r * ld + q * 8) = *reinterpret_cast<const uint4*>(stg + r * 40 + q * 8);
    }
    __syncwarp();
}
// The same block from packed bf16 pairs (a[2k], a[2k+1] in pw[k]), written into
// a tile image with R rows: rows row0.. and 32 columns from col0.
__device__ __forceinline__ void warp_store_t16_img_packed(__nv_bfloat16* stg, const uint32_t* pw, __nv_bfloat16* tile,
                                                          int R, int row0, int col0, int lane) {
    uint16_t* s16 = reinterpret_cast<uint16_t*>(stg);
#pragma unroll
    for (int j = 0; j < 16; ++j) s16[j * 40 + lane] = (uint16_t)((j & 1) ? (pw[j >> 1] >> 16) : (pw[j >> 1] & 0xffffu));
    __syncwarp();
#pragma unroll
    for (int p = lane; p < 64; p += 32) {
        const int r = p >> 2, q = p & 3;
        *reinterpret_cast<uint4*>(tile + ::kda::tile_el(R, row0 + r, col0 + 8 * q)) =
            *reinterpret_cast<const uint4*>(stg + r * 40 + q * 8);
    }
    __syncwarp();
}
// The same block written into a tile image with R rows (see tile_el): rows
// row0.. and 32 columns from col0 (a multiple of 8).
__device__ __forceinline__ void warp_store_t16_img(__nv_bfloat16* stg, const float (&a)[16], __nv_bfloat16* tile,
                                                   int R, int row0, int col0, int lane) {
#pragma unroll
    for (int j = 0; j < 16; ++j) stg[j * 40 + lane] = __float2bfloat16_rn(a[j]);
    __syncwarp();
#pragma unroll
    for (int p = lane; p < 64; p += 32) {
        const int r = p >> 2, q = p & 3;
        *reinterpret_cast<uint4*>(tile + ::kda::tile_el(R, row0 + r, col0 + 8 * q)) =
            *reinterpret_cast<const uint4*>(stg + r * 40 + q * 8);
    }
    __syncwarp();
}

// A warp holds 8 values per lane (lane t: column t of rows 0..7 of a 8 x 32
// block, e.g. one key per lane and 8 tokens). Writes the block as 8 rows of 32
// bf16, dst[r * ld + t] for r < nrows and t < wcols (a multiple of 8), through a
// dense per-warp staging tile of 8 x 32 bf16 (512 bytes): one 16-byte store per lane.
__device__ __forceinline__ void warp_store_t8(__nv_bfloat16* stg, const float (&a)[8], __nv_bfloat16* dst,
                                              size_t ld, int nrows, int lane, int wcols = 32) {
#pragma unroll
    for (int r = 0; r < 8; ++r) stg[r * 32 + lane] = __float2bfloat16_rn(a[r]);
    __syncwarp();
    const int r = lane >> 2, q = lane & 3;
    if (r < nrows && q * 8 < wcols)
        *reinterpret_cast<uint4*>(dst + (size_t)r * ld + q * 8) = *reinterpret_cast<const uint4*>(stg + r * 32 + q * 8);
    __syncwarp();
}

// Sums 8 per-lane values over the 32 lanes of a warp with 9 shuffles: lane t
// ends with the total of value 4 b4 + 2 b3 + b2 (b_i = bit i of t); the four
// lanes that share bits 4..2 hold the same total.
__device__ __forceinline__ float warp_sum8_spread(const float (&v)[8], int lane) {
    const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
    float a4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? v[i] : v[4 + i], keep = b4 ? v[4 + i] : v[i];
        a4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float a2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? a4[i] : a4[2 + i], keep = b3 ? a4[2 + i] : a4[i];
        a2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? a2[0] : a2[1], keep = b2 ? a2[1] : a2[0];
    float a1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
    a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
    return a1;
}

// Approximate reciprocal (the PTX rcp.approx instruction, about 1 ulp); for
// operands that are rounded to bf16 afterwards.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16 pair packing
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}

}  // namespace tc
}  // namespace kda
