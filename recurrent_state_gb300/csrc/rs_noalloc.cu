// rs_noalloc.cu -- checkpoint pack for callers that must not allocate device
// memory.
//
// rs_ckpt_pack reads its index table from device memory that rs_plan_upload
// allocates with cudaMalloc.  Some callers cannot do that: a serving engine
// that reserves a fixed fraction of HBM for its own pools at start-up and
// treats any later allocation as an out-of-memory risk, or a latency-critical
// path where the device-wide synchronisation of cudaFree is not acceptable.
// rs_ckpt_pack_noalloc gives them the same pack with the table held in a
// file-scope __device__ array instead, copied in on the caller's stream at
// each call from the page-locked copy that rs_plan_create made (so the copy
// is asynchronous).  The array is a fixed size (kNoallocTableEntries int32
// entries, 1 MiB), and every GPU that loads the library keeps it until the
// process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/recurrent_state.h"
#include "rs_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Shared by every call on a device; holds the last call's table.
static __device__ __align__(256) int32_t g_pack_table[rs::kNoallocTableEntries];

std::mutex g_mu;
int32_t *g_table_addr[kMaxDevices];  // device address of g_pack_table, per device

// Set-up, once per device with that device current: look up the device
// address of the array (host code must not pass the array's name itself to
// a kernel: on the host it names a stand-in, not device memory).  The
// address is kept for the life of the process, so the call must not be used
// on a device after cudaDeviceReset.
cudaError_t table_address(int dev, int32_t **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_table_addr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_pack_table);
        if (e != cudaSuccess) return e;
        g_table_addr[dev] = static_cast<int32_t *>(ptr);
    }
    *out = g_table_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" rs_status rs_ckpt_pack_noalloc(const rs_plan *p, const void *pool,
                                          int64_t layer_stride_bytes, int64_t n_pool_slots,
                                          const int32_t *src_slots, const int32_t *dst_ckpt_slots,
                                          int32_t n, void *ckpt_pool, int64_t n_ckpt_slots,
                                          int32_t *status, void *stream) {
    if (!p || n < 0 || n_pool_slots < 0 || n_ckpt_slots < 0) return RS_ERR_INVALID_ARG;
    const int64_t n_kept = p->offsets.back();
    if (n_kept > rs::kNoallocTableEntries) return RS_ERR_UNSUPPORTED;  // plan larger than the table
    if (n == 0 || n_kept == 0) return RS_OK;
    if (!pool || !src_slots || !dst_ckpt_slots || !ckpt_pool) return RS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(pool) & 15) || (reinterpret_cast<uintptr_t>(ckpt_pool) & 15) ||
        (layer_stride_bytes & 15))
        return RS_ERR_MISALIGNED;
    const int64_t slot_bytes = (int64_t)p->Hv * (int64_t)p->head_bytes;
    if (p->L > 1 && layer_stride_bytes < slot_bytes * n_pool_slots) return RS_ERR_INVALID_ARG;
    if (!p->h_kept_pinned) return RS_ERR_UNSUPPORTED;  // no CUDA device when the plan was made
    rs::CkptParams P;
    P.src = static_cast<const uint8_t *>(pool);
    P.dst = static_cast<uint8_t *>(ckpt_pool);
    P.layer_stride = layer_stride_bytes;
    P.slot_bytes = slot_bytes;
    P.unit_bytes = p->unit_bytes;
    P.ckpt_slot_bytes = n_kept * p->unit_bytes;
    P.n_pool_slots = n_pool_slots;
    P.n_ckpt_slots = n_ckpt_slots;
    P.n_kept = n_kept;
    P.n_all = (int64_t)p->L * p->nu;
    P.kept_unit = nullptr;  // set below, once the table is in place
    P.all_pidx = nullptr;   // pack does not read it
    P.pool_slots = src_slots;
    P.ckpt_slots = dst_ckpt_slots;
    P.status = status;
    P.n = n;
    P.units_per_layer = p->nu;
    // A shape the kernel refuses must be refused before the shared table is
    // touched: a pack of an earlier call may still be reading it.
    if (rs::check_ckpt_pack(P) != cudaSuccess) return RS_ERR_UNSUPPORTED;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return rs::fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return RS_ERR_UNSUPPORTED;
    int32_t *table = nullptr;
    if ((e = table_address(dev, &table)) != cudaSuccess) return rs::fail_cuda(e);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The whole table is rewritten on every call: nothing is left to clear.
    e = cudaMemcpyAsync(table, p->h_kept_pinned, (size_t)n_kept * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return rs::fail_cuda(e);
    P.kept_unit = table;
    e = rs::launch_ckpt_pack(P, s);
    if (e != cudaSuccess) return rs::fail_launch(e);
    return RS_OK;
}
