// Blackwell (sm_103a) tensor-core building blocks in inline PTX: tensor
// memory (TMEM) allocation and access, shared-memory matrix descriptors for
// the 128-byte-swizzled K-major layout, tcgen05.mma issue/commit, and
// mbarriers with bounded waits.
//
// Conventions used by every kernel of this library:
//   - one CTA, cta_group::1, M = 128: row i of the accumulator lives in TMEM
//     lane i, column c holds element (i, c) (fp32, one column per element);
//   - operands in shared memory are K-major with the 128-byte swizzle: the
//     tile of R rows (R % 8 == 0) is stored as K/(128 B) "atom columns" of
//     R x 128 B each, 8-row groups 1024 B apart, and the 16-byte chunk c of
//     row r sits at chunk position c ^ (r % 8); every tile base is 1024-byte
//     aligned;
//   - an A operand may instead sit in TMEM (lane = row, one 32-bit column per
//     tf32 element, or two bf16 per column).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gma {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (r, k) inside a K-major SW128 tile of R rows, elements of E bytes.
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t k, uint32_t R, uint32_t E)
{
    const uint32_t kb = k * E;
    const uint32_t atom = kb >> 7, inner = kb & 127u;
    return atom * (R * 128u) + (r >> 3) * 1024u + (r & 7u) * 128u + ((((inner >> 4) ^ (r & 7u))) << 4) +
           (inner & 15u);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 B apart.  `saddr` is the shared address of the first element the MMA
// reads (tile base + atom column offset + k offset inside the atom).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
    d |= (uint64_t)1u << 16;                    // leading byte offset (unused by this layout)
    d |= (uint64_t)(1024u >> 4) << 32;          // stride byte offset: 8-row group pitch
    d |= (uint64_t)1u << 46;                    // descriptor version
    d |= (uint64_t)2u << 61;                    // 128-byte swizzle
    return d;
}

// Shared-memory matrix descriptor: MN-major, 128-byte swizzle.  The operand is
// stored as blocks of 64 MN-elements (16-bit) by K rows of 128 bytes; groups of 8
// rows along K are 1024 bytes apart and the blocks along MN are `lbo` bytes apart.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t lbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16; // leading byte offset: MN block pitch
    d |= (uint64_t)(1024u >> 4) << 32;          // stride byte offset: 8-row group pitch along K
    d |= (uint64_t)1u << 46;                    // descriptor version
    d |= (uint64_t)2u << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor: D fp32, A/B of format `fmt` (0 f16, 1 bf16, 2 tf32), both K-major.
__host__ __device__ constexpr uint32_t idesc(uint32_t M, uint32_t N, uint32_t fmt)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t kFmtBF16 = 1, kFmtTF32 = 2;
// Instruction descriptor bits: A, B read MN-major (transposed) instead of K-major.
constexpr uint32_t kAMajorMN = 1u << 15, kBMajorMN = 1u << 16;

// ---- TMEM allocation (executed by one full warp) ----
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- ordering between tcgen05 operations and thread synchronisation ----
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes -> visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- MMA issue (one thread) ----
__device__ __forceinline__ void mma_ss(uint32_t kind_tf32, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                      uint32_t id, uint32_t accumulate)
{
    if (kind_tf32)
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(id), "r"(accumulate)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(id), "r"(accumulate)
                     : "memory");
}
// A operand in TMEM
__device__ __forceinline__ void mma_ts(uint32_t kind_tf32, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                      uint32_t id, uint32_t accumulate)
{
    if (kind_tf32)
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "r"(a_tmem), "l"(b_desc), "r"(id), "r"(accumulate)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "r"(a_tmem), "l"(b_desc), "r"(id), "r"(accumulate)
                     : "memory");
}
// Arrive (once) on an mbarrier when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

// ---- TMEM <-> registers: 32 lanes x 32 bit, 16 consecutive columns per thread ----
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMEM address of (lane, column): lane in bits 31..16, column in 15..0.
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, uint32_t lane, uint32_t col)
{
    return base + (lane << 16) + col;
}

// ---- mbarriers ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// One arrival on the barrier (release: the caller's earlier memory operations are seen by its waiters).
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Waits for phase `parity` of the barrier for at most ~`limit_cycles` SM cycles.
// Returns false on timeout (the caller records the error and winds down).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit_cycles = 4000000000LL)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit_cycles) return false;
    return true;
}

// Records that a bounded wait of this kernel expired: one word per device in
// host memory mapped into the device (see timeout_flag_dev), read and cleared
// by the host.  Idempotent; any thread may call it.
__device__ __forceinline__ void report_timeout(unsigned int *flag)
{
    if (flag) {
        *reinterpret_cast<volatile unsigned int *>(flag) = 1u;
        __threadfence_system();
    }
}

// ---- TMA (bulk tensor copies) ----
// Arms the barrier's current phase for one arrival plus `bytes` of transactions.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// 2-D tiled load of the tensor map's box at (x = innermost, y) into shared memory;
// completion is counted in bytes on `bar`.  x * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, int x, int y, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

// 3-D tiled load (x innermost, then y, then z); completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, int x, int y, int z, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
                 : "memory");
}
// 3-D tiled store from shared memory (elements outside the tensor are not written),
// tracked by the bulk async-group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const void *map, int x, int y, int z, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the shared-memory sources of every committed bulk store have been read.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Non-tensor bulk copy global -> shared (both addresses and the size multiples of 16 bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// tf32 split of an fp32 value: hi keeps the 10 explicit mantissa bits the
// tensor core reads, lo = x - hi is exact in fp32.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

} // namespace tc
} // namespace gma
