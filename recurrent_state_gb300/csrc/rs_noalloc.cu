// rs_noalloc.cu -- checkpoint pack for callers that must not allocate device
// memory.
//
// rs_ckpt_pack reads its index table from device memory that rs_plan_upload
// allocates with cudaMalloc.  Some callers cannot do that: a serving engine
// that reserves a fixed fraction of HBM for its own pools at start-up and
// treats any later allocation as an out-of-memory risk, code that runs while
// a CUDA graph is being captured, or a latency-critical path where the
// device-wide synchronisation of cudaFree is not acceptable.
// rs_ckpt_pack_noalloc gives them the same pack with the table held in a
// file-scope __device__ array instead, copied in on the caller's stream at
// each call.  The array is a fixed size (kTableEntries int32 entries, 1 MiB),
// and every GPU that loads the library keeps it until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/recurrent_state.h"
#include "rs_internal.h"

namespace {

constexpr int64_t kTableEntries = int64_t(1) << 18;  // 262,144 units per checkpoint

// Shared by every call on a device; holds the last call's table.
static __device__ __align__(256) int32_t g_pack_table[kTableEntries];

std::mutex g_mu;
int32_t *g_table_addr[64];  // device address of g_pack_table, per device

// Set-up, once per device with that device current: look up the device
// address of the array (host code must not pass the array's name itself to
// a kernel: on the host it names a stand-in, not device memory).
cudaError_t table_address(int dev, int32_t **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_table_addr[dev & 63]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_pack_table);
        if (e != cudaSuccess) return e;
        g_table_addr[dev & 63] = static_cast<int32_t *>(ptr);
    }
    *out = g_table_addr[dev & 63];
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
    if (n_kept > kTableEntries) return RS_ERR_UNSUPPORTED;  // plan larger than the static table
    if (n == 0 || n_kept == 0) return RS_OK;
    if (!pool || !src_slots || !dst_ckpt_slots || !ckpt_pool) return RS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(pool) & 15) || (reinterpret_cast<uintptr_t>(ckpt_pool) & 15) ||
        (layer_stride_bytes & 15))
        return RS_ERR_MISALIGNED;
    const int64_t slot_bytes = (int64_t)p->Hv * (int64_t)p->head_bytes;
    if (p->L > 1 && layer_stride_bytes < slot_bytes * n_pool_slots) return RS_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return RS_ERR_CUDA;
    int32_t *table = nullptr;
    if ((e = table_address(dev, &table)) != cudaSuccess) return RS_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The whole table is rewritten on every call: nothing is left to clear.
    e = cudaMemcpyAsync(table, p->kept_unit.data(), (size_t)n_kept * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return RS_ERR_CUDA;
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
    P.kept_unit = table;
    P.all_pidx = nullptr;  // pack does not read it
    P.pool_slots = src_slots;
    P.ckpt_slots = dst_ckpt_slots;
    P.status = status;
    P.n = n;
    P.units_per_layer = p->nu;
    e = rs::launch_ckpt_pack(P, s);
    if (e == cudaErrorNotSupported) return RS_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return RS_ERR_CUDA;
    return RS_OK;
}
