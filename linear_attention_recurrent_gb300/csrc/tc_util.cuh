// tc_util.cuh -- sm_100-family tensor-core primitives for the chunked prefill:
// tensor-memory (TMEM) allocation and access, tcgen05.mma (kind::tf32 and
// kind::f16 with bf16 operands) with the A operand in TMEM or shared memory and
// the B operand in shared memory, completion through mbarriers, tensor-map bulk
// copies, and the tf32 split that keeps fp32 accuracy.
//
// Shared-memory operands use the K-major, no-swizzle layout: an operand tile
// of R rows x KD elements (4-byte) is made of "core matrices" of 8 rows x 16
// bytes, each stored as 128 contiguous bytes (row r of the core matrix at
// r * 16).  Core matrices adjacent along K are LBO bytes apart, core matrices
// adjacent along the rows (8-row groups) SBO bytes apart.  LBO = 144 (not 128)
// spreads the 16-byte chunks of one row over all shared-memory banks, so a
// warp writing one row (a chunk per lane) does not serialise.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lar {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 64-bit shared-memory matrix descriptor (start address, LBO, SBO in 16-byte
// units; bit 46 set: the fixed field of the sm_100 descriptor format; no
// swizzle, base offset 0, relative LBO).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}

// 32-bit instruction descriptor of kind::tf32: D fp32, A and B tf32, both
// K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// 32-bit instruction descriptor of kind::f16 with bf16 A and B (both), D fp32,
// both K-major, M x N (16 elements of K per instruction)
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// byte offset of element (r, k) of a K-major no-swizzle tile
__host__ __device__ constexpr uint32_t kmaj(int r, int k, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint32_t>((r & 7) * 16 + (r >> 3) * sbo + (k >> 2) * lbo + (k & 3) * 4);
}

// the same for 16-bit elements (8 per 16-byte core-matrix row).  In tensor
// memory a 16-bit A operand packs elements 2j (low half) and 2j + 1 (high half)
// of a row into 32-bit column j.
__host__ __device__ constexpr uint32_t kmaj16(int r, int k, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint32_t>((r & 7) * 16 + (r >> 3) * sbo + (k >> 3) * lbo + (k & 7) * 2);
}

// ---- 3-pass tf32 split: x = hi + lo with hi = x rounded to tf32 (nearest,
// ties away), lo = x - hi exact in fp32; A B ~ Ah Bh + Ah Bl + Al Bh.
__device__ __forceinline__ float tf32_hi(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// ---- TMEM allocation (one warp, all lanes)
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// generic-proxy shared-memory writes made visible to the tensor cores' reads
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// ---- MMA: D[tmem] (+)= A[tmem] B[smem]^T, issued by one thread
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// ---- MMA: D[tmem] (+)= A[smem] B[smem]^T, issued by one thread
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Tensor-memory lane of row r of an M = 64 product (cta_group::1): rows
// 16 j .. 16 j + 15 sit in lanes 32 j .. 32 j + 15 (lanes 16..31 of each warp's
// quarter are not written).
__host__ __device__ constexpr int m64_lane(int r) { return 32 * (r >> 4) + (r & 15); }

// arrive on `mbar` once every MMA this thread issued so far has completed
__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     smem_addr(mbar))
                 : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(mbar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }

// Bounded wait for phase `parity` of `mbar` to complete: false if it did not
// within the limit (the caller turns that into an error status; no wait here
// can run forever).
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity) {
    const uint32_t a = smem_addr(mbar);
#pragma unroll 1
    for (int i = 0; i < (1 << 22); ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// One arrival on `mbar` by this thread, releasing its prior writes (shared
// memory included) to whoever waits for the phase.
__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(mbar)) : "memory");
}

// One arrival on `mbar` that also raises the phase's expected transaction
// count by `bytes` (the bulk copies that complete on it count them down).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(mbar)), "r"(bytes)
                 : "memory");
}

// One box of a 3-d tiled tensor map (in kernel parameter space) at coordinates
// (x, y, z) into this CTA's shared memory (128-byte aligned), completing on
// `mbar` as transactions of the box's full size (out-of-range elements are
// written as zeros).  x times the element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z, uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(mbar))
        : "memory");
}

// As mbar_wait, but it also gives up as soon as `*abort` is set (checked every
// 256 polls), so that a group of threads whose partner group has stopped does
// not spin out the whole limit.
__device__ __forceinline__ bool mbar_wait_or(uint64_t* mbar, uint32_t parity, const volatile int* abort) {
    const uint32_t a = smem_addr(mbar);
#pragma unroll 1
    for (int i = 0; i < (1 << 22); ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    return false;
}

// Named barrier `id` over the `n` threads (a multiple of 32) that use it,
// returning the OR of `pred` over them.
__device__ __forceinline__ bool bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

// ---- TMEM <-> registers, 32 lanes x 16 columns (one lane per thread of the
// warp; the warp reaches lanes 32 (warp % 4) .. + 31)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

// 32 lanes x 8 columns (the column offset a multiple of 8)
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

}  // namespace tc
}  // namespace lar
