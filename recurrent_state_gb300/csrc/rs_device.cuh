// rs_device.cuh -- small inline-PTX helpers for sm_103a kernels of this
// library: shared-memory mbarriers, 1-D bulk TMA copies (cp.async.bulk),
// named barriers for thread groups inside a CTA, and warp reductions.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace rs {

// Upper bound on polls of one mbarrier wait.  Each try_wait that finds the
// phase incomplete suspends the thread for a hardware-chosen time slice --
// about 3.8 us on GB300 (7,800 cycles, measured by tests/c/wait_timeout.cu)
// -- so this bounds a wait to about a second, while a stage's bulk copy
// lands in microseconds; a wait that runs out reports RS_DEV_PIPE_TIMEOUT and
// the kernel returns instead of spinning forever.
constexpr uint32_t kWaitPollLimit = 1u << 18;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Programmatic dependent launch.  A kernel launched with the
// programmatic-stream-serialization attribute (launch_pdl) may begin while
// the kernel before it in the stream is still finishing; pdl_wait blocks
// until that kernel has completed and its memory writes are visible, so a
// kernel calls it before its first global-memory access.  Without the
// attribute it returns at once.  pdl_launch_next lets the next such kernel
// in the stream start launching (it still waits in its own pdl_wait).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_next() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete: false once
// `limit` polls have found it incomplete.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint32_t limit = kWaitPollLimit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 1-D bulk copy global -> shared; completion is signalled on `bar` as
// transaction bytes.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 1-D bulk copy shared -> global (async proxy), tracked as a bulk group of
// the issuing thread.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_store_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store of this thread has finished reading
// its shared-memory source (the buffer may then be rewritten).
__device__ __forceinline__ void bulk_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_store_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Barrier over `count` threads (a multiple of 32) of this CTA, id 1..15.
__device__ __forceinline__ void group_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool group_sync_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return out != 0;
}

// max over the warp of |x|, NaN if any lane holds a NaN.
__device__ __forceinline__ float warp_max_abs_nan(float x) {
    float r;
    asm("redux.sync.max.abs.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
    return r;
}

template <typename T> __device__ __forceinline__ float load_as_f32(const T *p);
template <> __device__ __forceinline__ float load_as_f32<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float load_as_f32<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <> __device__ __forceinline__ float load_as_f32<__half>(const __half *p) {
    return __half2float(*p);
}

template <typename T> __device__ __forceinline__ void store_from_f32(T *p, float x);
template <> __device__ __forceinline__ void store_from_f32<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void store_from_f32<__nv_bfloat16>(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
}

}  // namespace rs
