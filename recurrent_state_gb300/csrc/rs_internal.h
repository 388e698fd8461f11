// rs_internal.h -- launch parameters and launcher entry points shared by the
// host-side C ABI (rs_api.cu) and the kernel translation units.  Not part of
// the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>
#include <cuda_runtime.h>

// A dasc selection plan (the opaque rs_plan of the C ABI).
struct rs_plan {
    int32_t L, unit, Hv, dk, dv, nu;
    size_t head_bytes;
    int64_t unit_bytes;
    std::vector<int64_t> offsets;     // o_0..o_L
    std::vector<int32_t> kept_unit;   // packed order: (layer << 20) | unit
    std::vector<int32_t> all_pidx;    // [L * nu]: packed index or -1
    int device = -1;
    int32_t *d_kept = nullptr;
    int32_t *d_all = nullptr;
    // Page-locked copy of kept_unit, made when the plan is created (null when
    // no CUDA device could be reached then, or the plan is larger than the
    // fixed table of rs_ckpt_pack_noalloc): the source of that call's
    // asynchronous table copy.
    int32_t *h_kept_pinned = nullptr;
};

namespace rs {

constexpr int kMaxTokens = 8;        // replay window (draft tokens per call)
constexpr int kStepThreads = 384;    // threads per CTA of the step kernel (single token)
// Replay keeps the state live across a runtime token loop: two groups per CTA
// leave it the registers it needs (255 per thread) without spilling.
constexpr int step_threads(int max_tokens) { return max_tokens > 1 ? 256 : kStepThreads; }
constexpr int kMaxRowMap = 8192;     // bytes of row maps carried in the launch params
// Retained units per checkpoint that rs_ckpt_pack_noalloc's fixed device
// table holds (int32 entries: 1 MiB).
constexpr int64_t kNoallocTableEntries = int64_t(1) << 18;

struct StepParams {
    void *pool;
    int64_t n_slots;
    const int32_t *slot_idx;
    const int32_t *n_accept;   // replay only
    const void *q;
    const void *k;
    const void *v;
    const float *alpha;
    const float *beta;
    void *o;
    int32_t *status;
    int32_t B, Hk, Hv, T_max;
    int32_t replay;            // 0: one token per item; 1: n_accept[b] tokens
    int32_t header_bytes;      // shared memory before the per-group regions
    int32_t region_bytes;      // shared memory per group
    int32_t stages;            // stage ring length (kernels that take one)
};

// Mixed layout: the row map pi (physical row -> key channel), [Hv][D] bytes,
// travels with the launch so the library needs no device allocation for it.
struct StepParamsPi : StepParams {
    uint8_t pi[kMaxRowMap];
};

struct StepLaunch {
    int D;          // 64 or 128
    int khi;        // -1 = FP32 layout, else FP16 rows of the mixed layout
    bool kda;
    int in_dt;      // RS_F32 / RS_BF16 / RS_F16
    int out_dt;     // RS_F32 / RS_BF16
    bool fused;     // mixed layouts: RS_QUANT_FUSED arithmetic
};

// Defined in rs_step_*.cu (one translation unit each, compiled in parallel).
// They return cudaErrorNotSupported for a combination that is not built.
cudaError_t launch_step_f32_d64(const StepLaunch &L, StepParams &P, cudaStream_t s);
cudaError_t launch_step_f32_d128(const StepLaunch &L, StepParams &P, cudaStream_t s);
cudaError_t launch_step_mixed_decode(const StepLaunch &L, StepParamsPi &P, cudaStream_t s);
cudaError_t launch_step_mixed_replay(const StepLaunch &L, StepParamsPi &P, cudaStream_t s);

// rs_prefill.cu: prefill chunks (FP32 steps on chip, state read and written once)
struct PrefillParams {
    void *pool;
    int64_t n_slots;
    const int32_t *slot_idx;
    const int32_t *n_tokens;   // [B] tokens of each sequence's chunk, or null: all L
    const void *q;
    const void *k;
    const void *v;
    const float *alpha;
    const float *beta;
    void *o;
    int32_t *status;
    int32_t B, Hk, Hv, L;
    uint8_t pi[kMaxRowMap];    // mixed layout: physical row -> key channel
};
cudaError_t launch_prefill(const StepLaunch &L, PrefillParams &P, cudaStream_t s);
// rs_chunk.cu / rs_chunk_mixed.cu: the chunk-parallel form on the tensor cores (FP32 and mixed layouts)
cudaError_t launch_prefill_chunked(const StepLaunch &L, PrefillParams &P, cudaStream_t s);
cudaError_t launch_prefill_chunked_mixed(const StepLaunch &L, PrefillParams &P, cudaStream_t s);

// rs_convert.cu
struct ConvertParams {
    const void *src;
    void *dst;
    int64_t n_slots;
    const int32_t *slots;
    int32_t *status;
    int32_t n, Hv;
    int32_t to_mixed;          // 1: FP32 -> mixed, 0: mixed -> FP32
    int32_t fused;             // FP32 -> mixed: RS_QUANT_FUSED codes
};
struct ConvertParamsPi : ConvertParams {
    uint8_t pi[kMaxRowMap];
};
cudaError_t launch_convert(int D, int khi, ConvertParamsPi &P, cudaStream_t s);
cudaError_t launch_copy_heads(const void *src, void *dst, int64_t head_bytes, const int32_t *slots,
                              int32_t n, int64_t n_slots, int32_t Hv, int32_t *status,
                              cudaStream_t s);

// rs_ckpt.cu
struct CkptParams {
    const uint8_t *src;
    uint8_t *dst;
    int64_t layer_stride;      // bytes between layers of the pool
    int64_t slot_bytes;        // bytes of one slot of one layer (Hv heads)
    int64_t ckpt_slot_bytes;   // o_L * unit_bytes
    int64_t unit_bytes;
    int64_t n_pool_slots, n_ckpt_slots;
    int64_t n_kept;            // o_L
    int64_t n_all;             // L * n_units
    const int32_t *kept_unit;  // [n_kept]  (layer << 20) | unit, packed order
    const int32_t *all_pidx;   // [n_all]   packed index or -1 (restore)
    const int32_t *pool_slots; // [n]
    const int32_t *ckpt_slots; // [n]
    int32_t *status;
    int32_t n;
    int32_t units_per_layer;
};
cudaError_t launch_ckpt_pack(const CkptParams &P, cudaStream_t s);
// cudaErrorNotSupported when launch_ckpt_pack would refuse P's shape (no launch).
cudaError_t check_ckpt_pack(const CkptParams &P);
cudaError_t launch_ckpt_restore(const CkptParams &P, cudaStream_t s);

// Record e as the library's last CUDA error (rs_last_cuda_error) and return
// RS_ERR_CUDA; fail_launch maps cudaErrorNotSupported (a combination that is
// not built) to RS_ERR_UNSUPPORTED first.  Defined in rs_api.cu.
int32_t fail_cuda(cudaError_t e);
int32_t fail_launch(cudaError_t e);

// Launch kern<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialization: its CTAs may be scheduled while the previous kernel in the
// stream drains (kernels launched this way call pdl_wait before touching
// global memory), which hides the launch gap between back-to-back steps.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Per-device cached attributes.
int device_sm_count();
int device_max_smem_optin();

// Raise kernel `fn`'s dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute call is made only the first time a larger
// size is needed for (fn, device), so steady-state launches -- including
// launches recorded into a CUDA graph -- issue none.
cudaError_t set_dynamic_smem(const void *fn, int bytes);

}  // namespace rs
