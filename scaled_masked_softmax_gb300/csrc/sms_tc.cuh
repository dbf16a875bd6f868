// Blackwell tensor-core primitives for sm_103a, as inline PTX: tensor-memory
// (TMEM) allocation, tcgen05.mma with operands in shared memory, completion
// through mbarriers (tcgen05.commit), TMEM <-> register moves, the 128-byte
// swizzled shared-memory matrix descriptors the MMA reads, and tiled TMA
// loads (cp.async.bulk.tensor) that write that swizzle.
//
// Layout conventions used by every caller:
//   * a "K-major" tile of R rows x 64 16-bit elements is R rows of 128 bytes,
//     8-row groups 1024 bytes apart, 16-byte chunk c of row r stored at chunk
//     c ^ (r % 8) (the 128-byte swizzle TMA applies); tiles are 1024-byte
//     aligned.  Wider rows are several such tiles ("atoms") side by side.
//   * the MMA accumulator D (M = 128 rows) sits in TMEM with row i in lane i
//     and column n in column base + n, fp32.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sms {
namespace tc {

// ------------------------------------------------------------------ TMEM ---
// Allocate `ncols` TMEM columns (a power of two >= 32) for this CTA; the
// whole warp calls it; the base address is written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(slot));
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(s), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------------- MMA ---
// D[tmem] (+)= A[smem] * B[smem]^T for one K = 16 slice, kind::f16 (fp16 or
// bf16 operands, fp32 accumulate).  Issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// The mbarrier gets one arrival once every MMA this thread issued before the
// call has completed.
__device__ __forceinline__ void commit(uint64_t *bar)
{
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(s) : "memory");
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of format
// `ab` (0 = fp16, 1 = bf16), each K-major (0) or MN-major (1: b_mn for B,
// a_mn for A), M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int ab, int b_mn, int M, int N, int a_mn = 0)
{
    return (1u << 4)                       // D format: fp32
           | ((uint32_t)ab << 7)           // A format
           | ((uint32_t)ab << 10)          // B format
           | ((uint32_t)a_mn << 15)        // A major-ness
           | ((uint32_t)b_mn << 16)        // B major-ness
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle.  `lbo` / `sbo`: byte
// strides (leading dimension: between 64-element atoms along M/N of an
// MN-major tile, unused for K-major; stride dimension: between 8-row groups).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((smem_addr >> 4) & 0x3FFFu)
           | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16)
           | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32)
           | (1ull << 46)    // descriptor version of sm_100 and later
           | (2ull << 61);   // 128-byte swizzle
}

// ---------------------------------------------------- TMEM <-> registers ---
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes: lane t of the
// warp gets lane (taddr.lane + t), columns taddr.col .. +31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
           "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
           "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------- TMA ---
// Tiled 3-D load of one box (x = innermost coordinate, in elements) into
// shared memory, completion counted on `bar` as transaction bytes.  x times
// the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int x, int y, int z, uint64_t *bar)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(d), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(b) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// `bytes` of fp32 in shared memory added element-wise to global memory by the
// TMA unit (both addresses 16-byte aligned, bytes a multiple of 16), in the
// issuing thread's current bulk group.  The shared source stays in use until
// bulk_wait_read() returns.
__device__ __forceinline__ void bulk_reduce_add_f32(float *gdst, uint32_t s_src, uint32_t bytes)
{
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
                 :: "l"(gdst), "r"(s_src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed bulk group of this thread has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed bulk group of this thread but the most recent one has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_but_last() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every committed bulk group of this thread has finished
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Shared-memory writes by ordinary stores become visible to the tensor-core
// and TMA (async proxy) reads that follow a barrier.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Byte offset of (row r, 16-byte chunk c) inside a K-major 128-byte-swizzled
// tile (c in 0..7; one atom of 64 16-bit elements per row).
__host__ __device__ constexpr uint32_t sw128_off(uint32_t r, uint32_t c)
{
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

}  // namespace tc
}  // namespace sms
