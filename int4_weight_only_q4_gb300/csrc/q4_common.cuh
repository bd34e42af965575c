// Internal helpers shared by the library's CUDA translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "q4.h"

// D += A * B on the tensor cores: 16 x 8 x 16, bf16 operands, fp32 accumulators.
static __device__ __forceinline__ void mma_bf16_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A * B (the accumulator input is zero)
static __device__ __forceinline__ void mma_bf16_m16n8k16_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                            uint32_t a3, uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

// Programmatic dependent launch: wait for the previous kernel's memory, let the next kernel start.
static __device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
static __device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Loads of data written by the previous kernel, issued after grid_dependency_wait: coherent
// loads that the compiler keeps below the wait.  (A non-coherent ld.global.nc is only valid for
// data that is read-only for the whole life of the kernel, and the compiler may move it above
// the wait.)
static __device__ __forceinline__ uint32_t ld_dep_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
    return r;
}
static __device__ __forceinline__ uint2 ld_dep_u2(const void* p) {
    uint2 r;
    asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p) : "memory");
    return r;
}
static __device__ __forceinline__ uint4 ld_dep_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}
static __device__ __forceinline__ float ld_dep_f32(const float* p) {
    float r;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(r) : "l"(p) : "memory");
    return r;
}

static __device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (through L2 only) and its group bookkeeping.
static __device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
static __device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
static __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// mbarriers (shared::cta) and 1-D bulk copies
static __device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

static __device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

static __device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

static __device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Wait for the phase with the given parity to complete, at most `limit` polls.
static __device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
    const uint32_t a = smem_addr(bar);
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes: multiple of 16).
static __device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// bf16 pair times m1 * m2 (powers of two), exact for the supported range (|x| < 2^121 after scaling).
static __device__ __forceinline__ uint32_t bf16x2_scale(uint32_t v, float m1, float m2) {
    const float lo = (__uint_as_float(v << 16) * m1) * m2, hi = (__uint_as_float(v & 0xFFFF0000u) * m1) * m2;
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Host side, defined in q4_gemv.cu.
int q4i_sm_count(int* dev_out);  // SMs of the current device (cached), -1 on error
bool q4i_fault_injected();       // Q4_FAULT_INJECT=launch: every launch reports Q4_ERR_CUDA
// Defined in q4_attn.cu: read and clear the attention kernels' device error word (1 if a bounded
// wait gave up since the last call, 0 if not, -1 if the read failed).
int q4i_attn_take_error();
// Defined in q4_prefill_tc.cu: the tensor-memory prefill GEMM (compute capability 10.x).
bool q4i_prefill_tc_usable(int64_t K, int64_t M);
size_t q4i_prefill_tc_ws(int64_t K, int64_t M);
q4_status q4i_prefill_tc(const q4_matrix* W, const uint16_t* X, int64_t M, float* Y, void* ws, size_t ws_bytes,
                         cudaStream_t stream, bool pdl);
int q4i_prefill_take_error();  // as q4i_attn_take_error, for its error word
