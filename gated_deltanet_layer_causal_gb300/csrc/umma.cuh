// tcgen05 (5th-generation tensor core) helpers for sm_103a: tensor-memory
// allocation, shared-memory matrix descriptors, MMA issue, commit to an
// mbarrier, bounded waits, and tensor-memory loads.
//
// Operands live in shared memory in the no-swizzle K-major layout: an R x Kd
// fp32 (tf32) tile is a grid of core matrices of 8 rows x 16 bytes (4
// elements); core (r/8, k/4) sits at float offset ((r/8)*(Kd/4) + k/4)*32 and
// row r%8 of it at +4*(r%8).  Adjacent cores along K are 128 B apart (the
// descriptor's leading byte offset), adjacent 8-row groups (Kd/4)*128 B apart
// (stride byte offset).  One 16-byte piece of a row-major global row is one
// core-matrix row, so row-major tiles stage with plain 16-byte copies.
//
// Accumulators (fp32) live in tensor memory.  For M = 128, row i of D is lane
// i; for M = 64, row i is lane (i % 16) + 32 * (i / 16).  Warp w reads lanes
// 32*(w%4) .. 32*(w%4)+31.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdn {
namespace umma {

// Shared-memory base rounded up to 1024 bytes (swizzled tiles need it; the
// dynamic allocation reserves the extra kilobyte).
__device__ __forceinline__ float* align1024(float* p) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    return p + (((1024u - (a & 1023u)) & 1023u) >> 2);
}

__device__ __forceinline__ int kidx(int r, int k, int Kd) {
    return (((r >> 3) * (Kd >> 2) + (k >> 2)) << 5) + ((r & 7) << 2) + (k & 3);
}

__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Descriptor of the K = 8 slice starting at column k0 of an R x Kd K-major tile.
__device__ __forceinline__ uint64_t desc(const float* tile, int k0, int Kd) {
    const uint32_t a = saddr(tile) + (uint32_t)(k0 >> 2) * 128u;
    uint64_t d = (uint64_t)((a >> 4) & 0x3FFFu);
    d |= (uint64_t)(128u >> 4) << 16;                          // leading byte offset
    d |= (uint64_t)(((uint32_t)(Kd >> 2) * 128u) >> 4) << 32;  // stride byte offset
    d |= (uint64_t)1 << 46;                                    // descriptor version
    return d;                                                  // no swizzle, base offset 0
}

// 128-byte-swizzled K-major tiles, as the tensor-memory-access unit (TMA)
// writes them: a [rows][128] fp32 tile is four boxes of [rows][32] (128 B per
// row); within a box, 16-byte piece p of row r sits at piece p ^ (r % 8).
// Tile bases are 1024-byte aligned.  Float offset of element (r, c):
__device__ __forceinline__ int swz(int r, int c, int rows) {
    return ((c >> 5) * rows + r) * 32 + ((((c >> 2) & 7) ^ (r & 7)) << 2) + (c & 3);
}

// Descriptor of the K = 8 slice at column k0 of a swizzled tile: start inside
// the 128-byte row, 8-row groups 1024 B apart, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t desc_sw(const float* tile, int rows, int k0) {
    const uint32_t a = saddr(tile) + (uint32_t)((k0 >> 5) * rows * 128 + (k0 & 31) * 4);
    uint64_t d = (uint64_t)((a >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset
    d |= (uint64_t)1 << 46;                    // descriptor version
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// MN-major tile: 64 rows of the contraction dimension (tokens) x 128 columns,
// four boxes of [64][32] in the 128-byte swizzle with 32-byte atoms (32-byte
// chunk c of row r sits at chunk c ^ (r % 4)).  The tensor core reads K = 8 rows
// per step as two 4-row groups 512 B apart, 32-column atoms one box (8 KB)
// apart: layout type 1, start address 1 KB-aligned at every step.
// A tile of `rows` contraction rows (64 or 128) has its atoms rows * 128 B apart.
__device__ __forceinline__ uint64_t desc_mn(const float* tile, int k0, int rows = 64) {
    const uint32_t a = saddr(tile) + (uint32_t)(k0 >> 3) * 1024u;
    uint64_t d = (uint64_t)((a >> 4) & 0x3FFFu);
    d |= (uint64_t)(((uint32_t)rows * 128u) >> 4) << 16;   // leading byte offset: next atom
    d |= (uint64_t)(512u >> 4) << 32;           // stride byte offset: next 4-row group
    d |= (uint64_t)1 << 46;                     // descriptor version
    d |= (uint64_t)1 << 61;                     // 128-byte swizzle, 32-byte atoms
    return d;
}
// Float offset of element (r, c) of an MN-major tile of `rows` rows.
__device__ __forceinline__ int swz_mn(int r, int c, int rows = 64) {
    return ((c >> 5) * rows + r) * 32 + ((((c >> 3) & 3) ^ (r & 3)) << 3) + (c & 7);
}

// An MMA operand in shared memory: a no-swizzle K-major tile (n = its K
// extent), a swizzled K-major tile (n = its row count) or an MN-major tile
// (n = its row count, the contraction extent: 64 or 128).
struct Op {
    const float* p;
    int n;
    int kind;   // 0 no-swizzle K-major, 1 swizzled K-major, 2 MN-major
};
__device__ __forceinline__ Op kmaj(const float* p, int kd) { return Op{p, kd, 0}; }
__device__ __forceinline__ Op swt(const float* p, int rows) { return Op{p, rows, 1}; }
__device__ __forceinline__ Op mnt(const float* p, int rows = 64) { return Op{p, rows, 2}; }
__device__ __forceinline__ uint64_t opdesc(const Op& o, int k0) {
    return o.kind == 2 ? desc_mn(o.p, k0, o.n)
         : o.kind == 1 ? desc_sw(o.p, o.n, k0) : desc(o.p, k0, o.n);
}

// Offset, in the descriptor's 16-byte address units, of the K = 8 slice at
// column k0 from the slice at column 0 (the start-address field is the low 14
// bits and shared-memory tiles never carry out of it).
__device__ __forceinline__ uint64_t koff(const Op& o, int k0) {
    return o.kind == 2 ? (uint64_t)(k0 >> 3) * 64u
         : o.kind == 1 ? (uint64_t)(((k0 >> 5) * o.n * 128 + (k0 & 31) * 4) >> 4)
                       : (uint64_t)(k0 >> 2) * 8u;
}

// Instruction descriptor: D fp32, A and B tf32, both K-major, M x N.
__device__ __forceinline__ uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// D[M x N] (+)= A[M x K] * B[N x K]^T.  Issued by one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, const float* A, int lda_k,
                                         const float* B, int ldb_k, int M, int N, int K,
                                         bool accumulate) {
    const uint32_t id = idesc_tf32(M, N);
    const uint64_t a0 = desc(A, 0, lda_k), b0 = desc(B, 0, ldb_k);
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        const uint64_t ad = a0 + (uint64_t)(k0 >> 2) * 8u, bd = b0 + (uint64_t)(k0 >> 2) * 8u;
        const uint32_t acc = (accumulate || k0 > 0) ? 1u : 0u;
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
            "l"(ad), "l"(bd), "r"(id), "r"(acc));
    }
}

// The same for operands of either layout.  The descriptors are built once and
// advanced by a constant per K step (the loop unrolls at the call sites, where
// K and the layouts are constants).
__device__ __forceinline__ void mma(uint32_t d_tmem, const Op& A, const Op& B, int M, int N, int K,
                                    bool accumulate) {
    const uint32_t id = idesc_tf32(M, N) | (A.kind == 2 ? 1u << 15 : 0u) |
                        (B.kind == 2 ? 1u << 16 : 0u);   // MN-major ("transposed") operands
    const uint64_t a0 = opdesc(A, 0), b0 = opdesc(B, 0);
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        const uint64_t ad = a0 + koff(A, k0), bd = b0 + koff(B, k0);
        const uint32_t acc = (accumulate || k0 > 0) ? 1u : 0u;
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
            "l"(ad), "l"(bd), "r"(id), "r"(acc));
    }
}

// D[M x N] (+)= A[M x K] * B[N x K]^T with A in tensor memory (row m of A in
// lane m, element k in column a_tmem + k; M = 128) and B in shared memory.
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, const Op& B, int M, int N,
                                       int K, bool accumulate) {
    const uint32_t id = idesc_tf32(M, N) | (B.kind == 2 ? 1u << 16 : 0u);
    const uint64_t b0 = opdesc(B, 0);
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        const uint64_t bd = b0 + koff(B, k0);
        const uint32_t acc = (accumulate || k0 > 0) ? 1u : 0u;
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
            "r"(a_tmem + (uint32_t)k0), "l"(bd), "r"(id), "r"(acc));
    }
}

// Named barrier `id` over the first n threads of the CTA (n % 32 == 0; the
// threads of a role that syncs without the rest).
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
// The same with an AND reduction of v over the n threads.
__device__ __forceinline__ bool named_sync_and(int id, int n, bool v) {
    int r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.s32 p, %1, 0;\nbar.red.and.pred q, %2, %3, p;\n"
        "selp.s32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((int)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Plain arrive (count 1) on `mbar`.
__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(saddr(mbar)) : "memory");
}

// Arrive on `mbar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void commit(uint64_t* mbar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
            saddr(mbar)));
}

__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(saddr(mbar)), "r"(count));
    asm volatile("fence.mbarrier_init.release.cluster;\n");
}

// Wait for phase `parity` of `mbar` to complete, at most `limit` polls.
// Returns false (and the caller flags an error) if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, int limit = 1 << 24) {
    uint32_t done = 0;
    for (int it = 0; it < limit && !done; it++) {
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(saddr(mbar)), "r"(parity));
    }
    return done != 0;
}

// Arm `mbar` (count 1) for `bytes` of asynchronous copies; the calling thread
// arrives.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(saddr(mbar)),
                 "r"(bytes)
                 : "memory");
}

// 64 rows (tokens t0..t0+63) x 128 fp32 of one head through a 3-D tensor map
// {128, heads, tokens}: four swizzled 64 x 32 boxes into a tile whose boxes
// are `rows` rows apart (rows = 64, or 128 for the lower half of a stacked
// tile).  Rows past the end of the tensor arrive as zeros.  32 KB on `mbar`.
__device__ __forceinline__ void tma_rows(float* dst, int rows, const CUtensorMap* map, int head,
                                         int t0, uint64_t* mbar) {
#pragma unroll
    for (int b = 0; b < 4; b++)
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(saddr(dst + b * rows * 32)),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(b * 32), "r"(head), "r"(t0),
            "r"(saddr(mbar))
            : "memory");
}

// One swizzled 64 x 32 box (columns x .. x + 31 of rows t0 .. t0 + 63 of one
// head) into dst.  8 KB on `mbar`.
__device__ __forceinline__ void tma_box(float* dst, const CUtensorMap* map, int x, int head,
                                        int t0, uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(saddr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(head), "r"(t0), "r"(saddr(mbar))
        : "memory");
}

// Prefetch into L2 what tma_rows / tma_box would load (no shared memory, no
// barrier): a later load of the same tile then hits L2.
__device__ __forceinline__ void tma_prefetch_rows(const CUtensorMap* map, int head, int t0) {
#pragma unroll
    for (int b = 0; b < 4; b++)
        asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                         reinterpret_cast<uint64_t>(map)),
                     "r"(b * 32), "r"(head), "r"(t0)
                     : "memory");
}
// Prefetch `bytes` (a multiple of 16) of contiguous global memory at p
// (16-byte aligned) into L2.
__device__ __forceinline__ void bulk_prefetch(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(reinterpret_cast<uint64_t>(p)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_box(const CUtensorMap* map, int x, int head, int t0) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(head), "r"(t0)
                 : "memory");
}

// Contiguous copy shared -> global (both 16-byte aligned, bytes % 16 == 0), in
// the calling thread's bulk group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst),
                 "r"(saddr(src)), "r"(bytes)
                 : "memory");
}

// Contiguous copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];\n" ::"r"(saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(mbar))
        : "memory");
}

// Zero rows [r0, 64) of the 64-row block at `row0` of a swizzled tile (a chunk
// shorter than 64 tokens: its tail rows hold the next sequence's tokens).
// A whole 128-byte row is one box row, so the swizzle does not matter.
// NTH: the threads taking part, 0 .. NTH - 1 (0: the whole CTA).
template <int NTH = 0>
__device__ __forceinline__ void zero_tail_rows(float* tile, int rows, int row0, int r0) {
    const int n = (64 - r0) * 32;   // floats per box
    const int step = (NTH ? NTH : (int)blockDim.x) * 4;
    for (int e = threadIdx.x * 4; e < 4 * n; e += step) {
        const int b = e / n, o = e % n;
        *reinterpret_cast<float4*>(tile + (b * rows + row0 + r0) * 32 + o) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Generic-proxy shared-memory writes -> visible to the tensor core.
__device__ __forceinline__ void fence_smem_to_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

// Tensor-memory allocation (whole warp).  The base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     saddr(slot)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
__device__ __forceinline__ void tmem_free(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(base),
                 "r"(ncols));
}

// 16 consecutive fp32 columns of this thread's lane, starting at `taddr`
// (lane field already set to the warp's 32-lane window).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive fp32 columns of this thread's lane (one wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}
// Store 32 consecutive fp32 columns of this thread's lane (no wait: the caller
// waits with tmem_wait_st before the columns are read by anything else).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// Store 16 consecutive fp32 columns of this thread's lane (the inverse of
// tmem_ld16), then wait until the stores have completed.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// Round to the nearest tf32 value (ties away from zero).  The tensor core reads
// only the top 19 bits of an fp32 operand (it truncates), so operands are
// rounded when they are written to shared memory: rounding then happens once,
// to nearest, instead of being a truncation biased towards zero.
__device__ __forceinline__ float tf32r(float x) {
    // nearest, ties away from zero, on the bit pattern (see f2tf32 in common.cuh)
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
__device__ __forceinline__ float4 tf32r(float4 v) {
    return make_float4(tf32r(v.x), tf32r(v.y), tf32r(v.z), tf32r(v.w));
}
// Round n floats (n % 4 == 0, 16-byte aligned) in place; threads 0 .. NTH - 1
// (0: the whole CTA).
template <int NTH = 0>
__device__ __forceinline__ void tf32r_inplace(float* p, int n) {
    const int step = (NTH ? NTH : (int)blockDim.x) * 4;
    for (int i = threadIdx.x * 4; i < n; i += step) {
        float4* q = reinterpret_cast<float4*>(p + i);
        *q = tf32r(*q);
    }
}

// Eight 16x256b loads of an M = 64 accumulator (columns col0 .. col0 + 63 of
// this warp's 16-lane window, one wait): thread t holds, for column block k,
// v[4k + j] = D[row0 + t/4 + 8 (j/2)][col0 + 8k + 2 (t%4) + j%2], where row0 =
// 16 * (warp % 4).  All 32 lanes carry data (the 32x32b shape leaves half of
// them empty for M = 64).
template <int NB>
__device__ __forceinline__ void tmem_ld_m64(uint32_t taddr, float (&v)[4 * NB]) {
    uint32_t r[4 * NB];
#pragma unroll
    for (int k = 0; k < NB; k++)
        asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(r[4 * k]), "=r"(r[4 * k + 1]), "=r"(r[4 * k + 2]), "=r"(r[4 * k + 3])
                     : "r"(taddr + 8 * k));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 4 * NB; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld64_m64(uint32_t taddr, float (&v)[32]) {
    tmem_ld_m64<8>(taddr, v);
}
// The inverse of tmem_ld64_m64 (eight 16x256b stores), then wait until the
// stores have completed.
__device__ __forceinline__ void tmem_st64_m64(uint32_t taddr, const float (&v)[32]) {
#pragma unroll
    for (int k = 0; k < 8; k++)
        asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(taddr + 8 * k),
                     "r"(__float_as_uint(v[4 * k])), "r"(__float_as_uint(v[4 * k + 1])),
                     "r"(__float_as_uint(v[4 * k + 2])), "r"(__float_as_uint(v[4 * k + 3]))
                     : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// Write this thread's part of an M = 64 fragment (tmem_ld64_m64) into columns
// c0 .. c0 + 63 of a swizzled [64][128] tile, rows scaled by s_lo / s_hi (the
// thread's rows r and r + 8).  Two-float stores, no bank conflicts.
__device__ __forceinline__ void frag_to_sw(float* tile, const float (&v)[32], int c0, float s_lo,
                                           float s_hi) {
    const int lane = threadIdx.x & 31, r = 16 * ((threadIdx.x >> 5) & 3) + (lane >> 2);
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const int c = c0 + 8 * k + 2 * (lane & 3);
        *reinterpret_cast<float2*>(tile + swz(r, c, 64)) =
            make_float2(v[4 * k] * s_lo, v[4 * k + 1] * s_lo);
        *reinterpret_cast<float2*>(tile + swz(r + 8, c, 64)) =
            make_float2(v[4 * k + 2] * s_hi, v[4 * k + 3] * s_hi);
    }
}
// Rows of this thread in an M = 64 fragment (the other one is 8 further), and
// the first of its two columns in each 8-column block.
__device__ __forceinline__ int frag_row_lo() {
    return 16 * ((threadIdx.x >> 5) & 3) + ((threadIdx.x & 31) >> 2);
}
__device__ __forceinline__ int frag_col() { return 2 * (threadIdx.x & 3); }
// Sum over the four lanes that share a fragment row.
__device__ __forceinline__ float row_quad_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x + __shfl_xor_sync(0xffffffffu, x, 2);
}
// Sum over the eight lanes that share fragment columns (rows r .. r + 7).
__device__ __forceinline__ float col_oct_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    return x + __shfl_xor_sync(0xffffffffu, x, 16);
}

// Store a 64-row swizzled tile to 64 rows of a 3-D row tensor through its
// tensor map (rows past the tensor's end are dropped).  Shared-memory writes
// must be fenced to the async proxy and synchronised before the call; the
// caller commits and waits (bulk_commit / bulk_wait_read) before the tile's
// space is reused or the CTA exits.
__device__ __forceinline__ void tma_store_rows(const CUtensorMap* map, int head, int t0,
                                               const float* src) {
#pragma unroll
    for (int b = 0; b < 4; b++)
        asm volatile(
            "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
                reinterpret_cast<uint64_t>(map)),
            "r"(b * 32), "r"(head), "r"(t0), "r"(saddr(src + b * 64 * 32))
            : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

// Rows 0 .. L-1 of a 64-row swizzled tile to a row-major global tensor (row r
// at dst + r * stride), one warp per row: the path for a chunk shorter than 64
// tokens, whose remaining rows belong to the next sequence.
__device__ __forceinline__ void store_rows_sw(float* dst, int64_t stride, const float* src, int L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int r = warp; r < L; r += nw)
        *reinterpret_cast<float4*>(dst + r * stride + 4 * lane) =
            *reinterpret_cast<const float4*>(src + swz(r, 4 * lane, 64));
}

// Tensor-memory address of (lane window of this warp, column col).
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, int col) {
    const uint32_t lane0 = (uint32_t)((threadIdx.x >> 5) & 3) * 32u;
    return base + (lane0 << 16) + (uint32_t)col;
}

}  // namespace umma
}  // namespace gdn
