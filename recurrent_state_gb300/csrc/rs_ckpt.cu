// rs_ckpt.cu -- dasc checkpoint pack and restore (sm_103a).
//
// dasc §4.1 and Appendix B "Ragged (Scheme 2)": the retained units of each
// layer are flat-packed, layer l at units [o_{l-1}, o_l); a unit is one head
// (GDN) or one (head, key channel) row of dv floats (KDA).  dasc §4.2
// (dasc-nr): restore writes every unit of the destination slot, retained
// units from the checkpoint and omitted units as +0.0.
//
// Both kernels are plain streaming copies.  The work is cut into 512-byte
// chunks (a whole KDA unit at dv = 128, 1/128 of a GDN head, the last chunk
// of a unit possibly shorter: a mixed FP16/INT8 head of 18,880 B is 36
// chunks and 448 B); a warp moves one chunk per step with one 16-byte load
// and one 16-byte store per lane,
// and each warp keeps several chunks in flight so that enough bytes are
// outstanding per SM to cover HBM latency: four for pack, eight for restore,
// whose chunks wait on an index-table lookup before their load (measured at
// batch 64: restore 15% faster with eight, pack slower).  Pack reads ragged source units
// and writes the checkpoint contiguously; restore walks the destination
// contiguously, so its writes (the larger side) are fully sequential.
#include "rs_internal.h"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

constexpr int kChunkBytes = 512;
__host__ __device__ constexpr int chunks_in_flight(bool pack) { return pack ? 4 : 8; }  // per warp

struct Chunk {
    const uint4 *src;  // nullptr: write zeros
    uint4 *dst;
    bool active;
};

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_stream(uint4 *p, uint4 v) {
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Unit and chunk within the unit of a flat chunk index: a shift when the
// chunks per unit are a power of two, else a division.
struct Split {
    uint32_t cpu;  // chunks per unit
    int log2cpu;   // log2(cpu), or -1
};
__device__ __forceinline__ void split(uint32_t cc, Split sp, uint32_t &unit, uint32_t &part) {
    if (sp.log2cpu >= 0) {
        unit = cc >> sp.log2cpu;
        part = cc & ((1u << sp.log2cpu) - 1u);
    } else {
        unit = cc / sp.cpu;
        part = cc - unit * sp.cpu;
    }
}

// Chunk cc (within checkpoint i) of the pack: cc = j * cpu + part.
__device__ __forceinline__ Chunk pack_chunk(const CkptParams &P, int32_t s, int32_t d, uint32_t cc,
                                            Split sp, int lane) {
    Chunk ch;
    uint32_t j, part;
    split(cc, sp, j, part);
    const int32_t ku = __ldg(P.kept_unit + j);
    const int64_t l = ku >> 20, x = ku & 0xfffff;
    const int64_t off = (int64_t)part * kChunkBytes + (int64_t)lane * 16;
    ch.src = reinterpret_cast<const uint4 *>(P.src + l * P.layer_stride + (int64_t)s * P.slot_bytes +
                                             x * P.unit_bytes + off);
    ch.dst = reinterpret_cast<uint4 *>(P.dst + (int64_t)d * P.ckpt_slot_bytes +
                                       (int64_t)j * P.unit_bytes + off);
    ch.active = off < P.unit_bytes;
    return ch;
}

// Chunk cc (within slot i) of the restore: cc = u * cpu + part, u = l * nu + x.
__device__ __forceinline__ Chunk restore_chunk(const CkptParams &P, int32_t s, int32_t d, uint32_t cc,
                                               Split sp, int lane) {
    Chunk ch;
    uint32_t u, part;
    split(cc, sp, u, part);
    const uint32_t l = u / (uint32_t)P.units_per_layer;
    const uint32_t x = u - l * (uint32_t)P.units_per_layer;
    const int32_t pidx = __ldg(P.all_pidx + u);
    const int64_t off = (int64_t)part * kChunkBytes + (int64_t)lane * 16;
    ch.dst = reinterpret_cast<uint4 *>(P.dst + (int64_t)l * P.layer_stride + (int64_t)d * P.slot_bytes +
                                       (int64_t)x * P.unit_bytes + off);
    ch.src = pidx >= 0 ? reinterpret_cast<const uint4 *>(P.src + (int64_t)s * P.ckpt_slot_bytes +
                                                         (int64_t)pidx * P.unit_bytes + off)
                       : nullptr;
    ch.active = off < P.unit_bytes;
    return ch;
}

// grid.y walks the n (slot, checkpoint) pairs; grid.x the chunks of one pair.
template <bool PACK>
__global__ void __launch_bounds__(256) ckpt_kernel(const __grid_constant__ CkptParams P,
                                                   uint32_t chunks_per_pair, Split sp) {
    constexpr int kChunks = chunks_in_flight(PACK);
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.y;
    const int32_t ps = P.pool_slots[i], cs = P.ckpt_slots[i];
    const bool ps_ok = ps >= 0 && (int64_t)ps < P.n_pool_slots;
    const bool cs_ok = cs >= 0 && (int64_t)cs < P.n_ckpt_slots;
    if (!ps_ok || !cs_ok) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && P.status)
            atomicOr(P.status, (ps_ok ? 0 : RS_DEV_BAD_SLOT) | (cs_ok ? 0 : RS_DEV_BAD_CKPT_SLOT));
        return;
    }
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    for (uint32_t base = warp * kChunks; base < chunks_per_pair; base += nwarps * kChunks) {
        Chunk ch[kChunks];
        uint4 v[kChunks];
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
            const uint32_t cc = base + k;
            ch[k] = Chunk{nullptr, nullptr, false};
            if (cc < chunks_per_pair)
                ch[k] = PACK ? pack_chunk(P, ps, cs, cc, sp, lane) : restore_chunk(P, cs, ps, cc, sp, lane);
        }
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
            v[k] = make_uint4(0, 0, 0, 0);
            if (ch[k].active && ch[k].src) v[k] = ld_stream(ch[k].src);
        }
#pragma unroll
        for (int k = 0; k < kChunks; ++k)
            if (ch[k].active) st_stream(ch[k].dst, v[k]);
    }
}

// The shapes the kernel is built for: whole 16-byte lanes per unit, 32-bit
// chunk indices within a (slot, checkpoint) pair, and n in grid.y.
cudaError_t check(const CkptParams &P, bool pack) {
    if (P.unit_bytes <= 0 || (P.unit_bytes & 15)) return cudaErrorNotSupported;
    const int64_t cpu = (P.unit_bytes + kChunkBytes - 1) / kChunkBytes;
    const int64_t units = pack ? P.n_kept : P.n_all;
    if (units * cpu >= (1ll << 31) || P.n > 65535) return cudaErrorNotSupported;
    return cudaSuccess;
}

cudaError_t launch(const CkptParams &P, bool pack, cudaStream_t s) {
    const cudaError_t ce = check(P, pack);
    if (ce != cudaSuccess) return ce;
    const int64_t cpu = (P.unit_bytes + kChunkBytes - 1) / kChunkBytes;
    int log2cpu = 0;
    while ((1ll << log2cpu) < cpu) ++log2cpu;
    if ((1ll << log2cpu) != cpu) log2cpu = -1;
    const int64_t units = pack ? P.n_kept : P.n_all;
    const int64_t per_pair = units * cpu;
    if (per_pair == 0 || P.n == 0) return cudaSuccess;
    const int kChunks = chunks_in_flight(pack);
    const int64_t warps_needed = (per_pair + kChunks - 1) / kChunks;
    int64_t bx = (warps_needed * 32 + 255) / 256;
    // up to 16 CTAs of 8 warps per SM over the whole grid
    int64_t cap = ((int64_t)device_sm_count() * 16 + P.n - 1) / P.n;
    if (cap < 1) cap = 1;
    if (bx > cap) bx = cap;
    dim3 grid((unsigned)bx, (unsigned)P.n);
    const Split sp{(uint32_t)cpu, log2cpu};
    if (pack)
        ckpt_kernel<true><<<grid, 256, 0, s>>>(P, (uint32_t)per_pair, sp);
    else
        ckpt_kernel<false><<<grid, 256, 0, s>>>(P, (uint32_t)per_pair, sp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t check_ckpt_pack(const CkptParams &P) { return check(P, true); }
cudaError_t launch_ckpt_pack(const CkptParams &P, cudaStream_t s) { return launch(P, true, s); }
cudaError_t launch_ckpt_restore(const CkptParams &P, cudaStream_t s) { return launch(P, false, s); }

}  // namespace rs
