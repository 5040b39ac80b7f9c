// Inline-PTX primitives used by the backward pass on top of sm103_ptx.cuh:
// untiled bulk copies (global -> shared, mbarrier completion), bulk
// reductions (shared -> global, add.f32, bulk-group completion), named
// barriers, and the instruction descriptor with both operand majors.
//
// Written against the public PTX ISA (cp.async.bulk, cp.reduce.async.bulk,
// bar.sync, tcgen05 instruction descriptor).
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

// `bytes` (a multiple of 16) from global `src` to shared `dst`, both 16-byte
// aligned; completion is reported on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// global[dst .. dst + bytes) += shared[src ..) elementwise as float32
// (bytes a multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N committed bulk groups of this thread still read
// their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Barrier `id` (1..15) among `count` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier `id` among `count` threads that also ANDs a predicate over them:
// every thread gets true only if every participating thread passed true.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Instruction descriptor for kind::f16 with both operand majors given
// (0 = K-major, 1 = MN-major); fields as in make_idesc.
__host__ __device__ constexpr uint32_t make_idesc_ab(uint32_t ab_format, uint32_t M, uint32_t N, uint32_t a_mn,
                                                     uint32_t b_mn) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}

}  // namespace attn
