// rs_ckpt_int8.h -- launch interface of the INT8 state checkpoint kernels
// (rs_ckpt_int8.cu).  Internal to the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rs {

struct Int8CkptParams {
    const uint8_t *src;
    uint8_t *dst;
    int64_t layer_stride;      // bytes between layers of the FP32 pool
    int64_t slot_bytes;        // bytes of one pool slot of one layer (Hv heads)
    int64_t unit_bytes;        // bytes of one unit in the pool (head or row)
    int64_t ckpt_slot_bytes;   // bytes of one checkpoint slot (codes + scales, padded)
    int64_t codes_bytes;       // bytes of the codes region of a checkpoint slot
    int64_t n_pool_slots, n_ckpt_slots;
    int64_t n_kept;            // o_L
    int64_t n_all;             // L * units per layer
    const int32_t *kept_unit;  // [n_kept]  (layer << 20) | unit, packed order
    const int32_t *all_pidx;   // [n_all]   packed index or -1
    const int32_t *pool_slots; // [n]
    const int32_t *ckpt_slots; // [n]
    int32_t *status;
    int32_t n;
    int32_t units_per_layer;
    int32_t rows_log2;         // log2 of the rows per unit (dk for heads, 1 for rows)
    int32_t dv;                // 64 or 128
};

cudaError_t launch_ckpt_pack_int8(const Int8CkptParams &P, cudaStream_t s);
cudaError_t launch_ckpt_restore_int8(const Int8CkptParams &P, cudaStream_t s);

}  // namespace rs
