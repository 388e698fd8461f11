/*
 * recurrent_state.h -- C ABI of the GB300 recurrent-state library.
 *
 * The library runs the batched decode-step update of gated delta-rule linear
 * attention on one GPU (sm_103a), for GDN (one decay per head) and KDA (one
 * decay per key channel), with FP32 or mixed FP16/INT8 state storage,
 * speculative-token replay, and ragged dasc checkpoint pack/restore.
 *
 * Pages cited (by title and section):
 *   [dasc] "dasc: Decay-Aware State Compression for Hybrid Linear-Attention
 *          Serving" (arXiv 2608.30386).
 *   [DAMP] "DAMP: Decay-Aware Mixed-Precision Recurrent-State Quantization"
 *          (arXiv 2608.27513).
 *   [SRA]  "Serving recurrent attention" (Kimi K3 explainer, section 22).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every call returns an rs_status.  No C++ exception crosses this ABI.
 * - Pointers named "device" must point to memory of the current CUDA device,
 *   16-byte aligned, contiguous in the layout stated; RS_ERR_MISALIGNED
 *   otherwise.  Pointers named "host" are read during the call only.
 * - The caller owns every device buffer, every stream and every event.  The
 *   library owns only the rs_layout and rs_plan objects it creates (host
 *   memory, plus the device tables of an uploaded plan).  Decode, replay,
 *   convert, pack and restore never allocate and never synchronise: they
 *   enqueue kernels on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and return.
 * - Host-side validation failures return before any launch and modify
 *   nothing.
 * - Index errors that can only be seen on the device (a slot index out of
 *   range, an accepted-token count out of range) skip the affected item and
 *   OR a bit into the caller's int32 device status word `status` (may be
 *   NULL).  Nothing traps, nothing hangs; read the word after the stream
 *   completes.  Every on-chip pipeline wait is bounded; a wait that runs out
 *   sets RS_DEV_PIPE_TIMEOUT and the kernel returns.
 * - Slot indices within one call must be distinct (two items that name the
 *   same slot race on it).
 *
 * State layouts (one linear-attention layer; a pool is [slots][Hv][head])
 * ----------------------------------------------------------------------
 * RS_LAYOUT_FP32: head = float32 S[dk][dv], row u = key channel u ([DAMP]
 *   §3.1: S in R^{dk x dv}, row S_{t,u} per key channel), 4*dk*dv bytes.
 * RS_LAYOUT_MIXED_FP16_INT8 ([DAMP] §5.2, Appendix A.4; one FP32 scale per
 *   INT8 row as in [DAMP] §3.2 Eq. 5-6): head = the permuted state T = P_K S
 *   ([DAMP] Appendix A.3 Eq. 17) stored as three contiguous regions
 *     fp16  rows 0..k_hi-1           2*k_hi*dv bytes
 *     int8  rows k_hi..dk-1          (dk-k_hi)*dv bytes
 *     fp32  one scale per INT8 row   4*(dk-k_hi) bytes, row order
 *   (18,880 bytes at dk = dv = 128, k_hi = 16).  Inside the fp16 and int8
 *   regions rows are interleaved by 32-bit word so that one word holds one
 *   column of 2 fp16 rows or of 4 int8 rows: fp16 value (r, c) is half
 *   ((r/2)*dv + c)*2 + r%2; int8 value (r, c) is byte ((q/4)*dv + c)*4 + q%4
 *   with q = r - k_hi (k_hi a multiple of 4).  Physical row r holds key
 *   channel pi[r]: the k_hi selected channels in ascending order, then the
 *   rest in ascending order ([DAMP] Appendix A.2, Algorithm 1, last step).
 *   INT8 rows use a = max_v |x_v| (NaN if any x_v is NaN),
 *   s = max(a, 1e-8)/127, c = clip(round_half_even(x/s), -127, 127), with the
 *   maximum, the division and the rounding in IEEE FP32 ([dasc] Appendix E.1
 *   Eq. 8); dequantised value c*s.  FP16 rows round to nearest even.  A NaN
 *   state value stays a NaN (its payload bits are unspecified); its INT8 code
 *   is -127.
 *
 * Decode step (per sequence b and value head h; [DAMP] §3.1 Eq. 1-2,
 * equivalently [dasc] §3.1 Eq. 1 on the transposed state):
 *     S <- diag(alpha) S
 *     p = S^T k,   e = v - p
 *     S <- S + beta k e^T
 *     o = S^T q                          (o reads the updated state)
 * FP32 evaluation order (fixed so results are reproducible bit for bit):
 * decay = one multiply per element; both sums over key channels run in
 * ascending physical row order from +0.0, one fused multiply-add per term;
 * the write is fmaf(beta*k[u], e[v], S[u][v]) with beta*k[u] rounded first.
 * Value head h reads q and k of key head h / (Hv/Hk): the Hv/Hk adjacent
 * value heads share one key head ([dasc] Appendix B.1).  The kernels take q
 * and k as given (the model L2-normalises them upstream, [DAMP] §3.1).
 * Mixed layout: each step dequantises once, updates and reads out in FP32,
 * requantises once and writes back ([DAMP] Appendix A.4 "Fused decoding");
 * o is read from the FP32 updated state before requantisation.
 */
#ifndef RECURRENT_STATE_H
#define RECURRENT_STATE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) -------------------------------------- */
typedef int32_t rs_status;
#define RS_OK                0
#define RS_ERR_INVALID_ARG  (-1)  /* bad size, NULL pointer, unknown enum   */
#define RS_ERR_UNSUPPORTED  (-2)  /* valid but not built (e.g. dk = 96)     */
#define RS_ERR_MISALIGNED   (-3)  /* a device pointer not 16-byte aligned   */
#define RS_ERR_CUDA         (-4)  /* a CUDA runtime call failed (see below) */

/* ---- device status word bits (OR-ed by kernels into *status) ----------- */
#define RS_DEV_BAD_SLOT       1   /* a pool slot index outside [0, n_slots) */
#define RS_DEV_BAD_ACCEPT     2   /* n_accept[b] outside [0, T_max]         */
#define RS_DEV_BAD_CKPT_SLOT  4   /* a checkpoint slot outside its pool     */
#define RS_DEV_PIPE_TIMEOUT   8   /* an on-chip pipeline wait ran out       */

/* ---- enums ------------------------------------------------------------- */
#define RS_LAYOUT_FP32             0
#define RS_LAYOUT_MIXED_FP16_INT8  1

#define RS_F32   0
#define RS_BF16  1
#define RS_F16   2

#define RS_QUANT_IEEE    0   /* mixed layouts: IEEE quotient (default)     */
#define RS_QUANT_FUSED   1   /* mixed layouts: division-free arithmetic    */

#define RS_UNIT_HEAD     0   /* GDN checkpoint unit: one head state        */
#define RS_UNIT_CHANNEL  1   /* KDA checkpoint unit: one key-channel row   */

/* ---- opaque objects ---------------------------------------------------- */
typedef struct rs_layout rs_layout;
typedef struct rs_plan rs_plan;

typedef struct {
    int32_t kind;          /* RS_LAYOUT_FP32 or RS_LAYOUT_MIXED_FP16_INT8   */
    int32_t dk;            /* key channels per head (64 or 128)            */
    int32_t dv;            /* values per key channel; must equal dk        */
    int32_t num_v_heads;   /* Hv: state heads per layer                    */
    int32_t num_qk_heads;  /* Hk: q/k heads; Hv % Hk == 0                  */
    int32_t k_hi;          /* FP16 rows per head (mixed layout), else 0    */
} rs_layout_params;

/* Human-readable text for a status code (static storage). */
const char *rs_status_string(rs_status s);

/* Text of the last CUDA error seen by this thread in the library ("" if none). */
const char *rs_last_cuda_error(void);

/* Library version, e.g. "0.1.0". */
const char *rs_version(void);

/* ---- layout descriptors (host only; no CUDA call) ---------------------- */

/* Create a state-pool layout.  hi_rows (host, may be NULL for the FP32
 * layout) holds, per value head, the k_hi selected key channels
 * ([DAMP] §5.1 "Budgeted selection": the same count for every head); order
 * within a head does not matter, duplicates are rejected.  *out receives a
 * library-owned object; free it with rs_layout_destroy. */
rs_status rs_layout_create(rs_layout **out, const rs_layout_params *p,
                           const int16_t *hi_rows /* host [Hv][k_hi] */);
/* DAMP-exact storage ([DAMP] Appendix A.1 "Integer formats" and "Value
 * scaling and reordering", A.3 Eq. 17-18, A.4): a mixed layout (kind
 * RS_LAYOUT_MIXED_FP16_INT8, hi_rows as in rs_layout_create) whose INT8 rows
 * are quantised in groups of `group` consecutive values along dv with one
 * FP32 scale per group (the page's 32; only 32 is built), and whose state is
 * stored in value-scaled coordinates T = P_K S D_c^{-1}.  value_scales: host
 * float [Hv][dv], c'_v > 0 and finite, in the value order the model produces
 * (the value reordering P_V is absorbed into the projections, [DAMP] A.3);
 * NULL means all ones.  The library copies them.  Decode computes v' = v / c'
 * (IEEE division), the step of rs_gdn/kda_decode_update on T, and returns
 * o = c' (T^T q') -- the page's o' = D'_c T^T q'.
 * Tile: the FP16 and INT8 regions of the one-scale-per-row layout (same word
 * interleave), then scales [dk - k_hi][dv / group] f32 row-major: 20,224 B at
 * d = 128, k_hi = 16 (9.875 bits per value).  rs_state_convert converts FP32
 * states (S in logical rows) to and from it; checkpoint plans take its heads
 * as units; speculative replay and prefill chunks run on it (one
 * dequantisation and one requantisation per call).  Hv * dv <= 4096. */
rs_status rs_layout_create_damp(rs_layout **out, const rs_layout_params *p, const int16_t *hi_rows,
                                int32_t group, const float *value_scales);
rs_status rs_layout_destroy(rs_layout *l);

/* Requantisation arithmetic of a mixed layout (either kind of
 * rs_layout_create or rs_layout_create_damp).  The pages fix the quantiser
 * (s = max(a, 1e-8)/127, code = round(x/s) clipped to +-127, FP32: [DAMP]
 * §3.2 Eq. 5-6, [dasc] Appendix E.1 Eq. 8) and the fused step ([DAMP]
 * Appendix A.4: dequantise, decay and update in FP32, requantise), not how
 * x/s is evaluated or where the decay's rounding falls.
 *   RS_QUANT_IEEE  (default) code = clip(round_half_even(x/s)) with the IEEE
 *                  FP32 quotient; a step decays the dequantised value,
 *                  RN(RN(c*s) * a).
 *   RS_QUANT_FUSED the code is the integer nearest to the exact product
 *                  x * RN(1/s), ties to even (rows or groups whose absmax is
 *                  inf or NaN keep the IEEE quotient); a step decays an INT8
 *                  row through its scale, c * RN(s * a_u) (diag(a) diag(s) C
 *                  = diag(a s) C).  FP16 rows are as in RS_QUANT_IEEE.
 * The two agree on every scale and every FP16 value given the same FP32
 * state; a code may differ by one where x/s lies within about 2^-23 |x/s|
 * of a half-integer.  The stored format is the same: a pool may be used
 * with either mode.  The mode applies to decode, replay and FP32 -> mixed
 * conversion.  RS_ERR_INVALID_ARG for an unknown mode or RS_QUANT_FUSED on
 * an FP32 layout. */
rs_status rs_layout_set_quant(rs_layout *l, int32_t mode);
rs_status rs_layout_quant(const rs_layout *l, int32_t *mode);

/* Bytes of one head state in this layout (65,536 or 18,880 at d = 128). */
rs_status rs_layout_head_bytes(const rs_layout *l, size_t *bytes);

/* The row map pi (physical row -> key channel) per head, host [Hv][dk]. */
rs_status rs_layout_row_map(const rs_layout *l, int16_t *pi);

/* Storage cost per state value in bits, scales included ([DAMP] Table 1
 * "Avg. bits"): 32 for FP32, (16*k_hi*dv + 8*(dk-k_hi)*dv + 32*(dk-k_hi))
 * / (dk*dv) for the mixed layout. */
rs_status rs_layout_bits_per_value(const rs_layout *l, double *bits);

/* ---- decode-step updates ----------------------------------------------- */

/* GDN decode step, one scalar decay per (sequence, value head)
 * ([DAMP] §3.1: Lambda = alpha I).
 *   pool      device  [n_slots][Hv][head_bytes]   state of one layer, in place
 *   slot_idx  device  int32 [B]                   pool slot of sequence b
 *   q, k      device  in_dtype [B][Hk][dk]
 *   v         device  in_dtype [B][Hv][dv]
 *   alpha     device  float [B][Hv]               decay in (0, 1]
 *   beta      device  float [B][Hv]               write strength
 *   o         device  out_dtype [B][Hv][dv]        readout (may be NULL)
 *   status    device  int32 (may be NULL)
 * in_dtype and out_dtype: built for bf16 -> f32, f16 -> f32, f32 -> f32
 * and, at dk = 128, bf16 -> bf16 (o rounded once from FP32, nearest even);
 * bf16 and f16 inputs widen to FP32 exactly.  Other combinations (f16 -> bf16
 * among them) return RS_ERR_UNSUPPORTED before any launch.
 * B = 0 is a no-op. */
rs_status rs_gdn_decode_update(const rs_layout *l, void *pool, int64_t n_slots,
                               const int32_t *slot_idx, int32_t B,
                               const void *q, const void *k, const void *v,
                               int32_t in_dtype, const float *alpha, const float *beta,
                               void *o, int32_t out_dtype, int32_t *status,
                               void *stream);

/* KDA decode step, one decay per key channel ([DAMP] §3.1:
 * Lambda = diag(exp g); [dasc] §3.1 Eq. 1, alpha in (0,1)^dk).  As above,
 * except alpha is device float [B][Hv][dk], indexed by key channel (not by
 * physical row). */
rs_status rs_kda_decode_update(const rs_layout *l, void *pool, int64_t n_slots,
                               const int32_t *slot_idx, int32_t B,
                               const void *q, const void *k, const void *v,
                               int32_t in_dtype, const float *alpha, const float *beta,
                               void *o, int32_t out_dtype, int32_t *status,
                               void *stream);

/* Speculative-token replay ([SRA] "Speculative decoding without state
 * snapshots"): the projected inputs of T_max draft tokens were logged; for
 * each sequence b the first n_accept[b] of them are replayed on the state,
 * which is read (and dequantised) once, kept on chip across the tokens, and
 * written (and requantised) once.  To add the target model's bonus token,
 * log it as one more token.  With the FP32 layout the result equals
 * n_accept[b] decode steps bit for bit.
 *   per_channel_decay  0 = GDN (alpha [B][T_max][Hv]),
 *                      1 = KDA (alpha [B][T_max][Hv][dk])
 *   T_max     1..8
 *   n_accept  device int32 [B]; 0 leaves the state untouched
 *   q, k      device in_dtype [B][T_max][Hk][dk]; v [B][T_max][Hv][dv]
 *   beta      device float [B][T_max][Hv]
 *   o         device out_dtype [B][T_max][Hv][dv] or NULL; rows t >= n_accept[b]
 *             are not written. */
rs_status rs_spec_replay_update(const rs_layout *l, int32_t per_channel_decay,
                                void *pool, int64_t n_slots, const int32_t *slot_idx,
                                int32_t B, int32_t T_max, const int32_t *n_accept,
                                const void *q, const void *k, const void *v,
                                int32_t in_dtype, const float *alpha, const float *beta,
                                void *o, int32_t out_dtype, int32_t *status,
                                void *stream);

/* Prefill chunk ([DAMP] Appendix A.4 "Prefill path": prefill uses FP32
 * arithmetic within each chunk and writes its final state to the same
 * packed cache, which later chunks and decoding steps read).  For each
 * sequence b, the first n_tokens[b] tokens of its chunk of L tokens are
 * applied to the state in order, each as one decode step (GDN or KDA, as
 * per_channel_decay), with the state read (and dequantised) once, kept in
 * FP32 on chip, and written (and requantised) once.  On the FP32 layout the
 * result equals n_tokens[b] decode calls bit for bit; on a mixed layout it
 * is the multi-token replay of the same tokens (one dequantisation and one
 * requantisation, in the layout's RS_QUANT mode).
 *   L         tokens per chunk (>= 0; 0 is a no-op)
 *   n_tokens  device int32 [B], each in [0, L], or NULL for L tokens each;
 *             an out-of-range count skips the sequence and sets
 *             RS_DEV_BAD_ACCEPT
 *   q, k      device in_dtype [B][L][Hk][dk]; v [B][L][Hv][dv]
 *   alpha     device float [B][L][Hv] (GDN) or [B][L][Hv][dk] (KDA)
 *   beta      device float [B][L][Hv]
 *   o         device out_dtype [B][L][Hv][dv] or NULL; rows t >= n_tokens[b]
 *             are not written.
 * Built for dk = dv = 128: the FP32 layout and the mixed layouts with
 * k_hi = 16 (one scale per row, or DAMP-exact groups of 32 with value
 * scaling); other shapes return RS_ERR_UNSUPPORTED. */
rs_status rs_prefill_update(const rs_layout *l, int32_t per_channel_decay, void *pool,
                            int64_t n_slots, const int32_t *slot_idx, int32_t B, int32_t L,
                            const int32_t *n_tokens, const void *q, const void *k, const void *v,
                            int32_t in_dtype, const float *alpha, const float *beta, void *o,
                            int32_t out_dtype, int32_t *status, void *stream);

/* Prefill chunk in the chunk-parallel form, on the tensor cores.  Same
 * arguments, layouts and status bits as rs_prefill_update, and the same map
 * ([DAMP] Appendix A.4 "Prefill path"; [SRA] "Kernels follow the serving
 * phase": prefill exposes parallel work across a chunk's tokens): the tokens
 * are taken 32 at a time, and each group is applied as dense products on
 * the tensor cores (the written rows W solve (I + diag(beta) A) W =
 * diag(beta)(V - Khat S0), with A the decay-weighted key Gram matrix; the
 * outputs and the new state follow from W).  The products use tf32 operands
 * split into a high part and an exact remainder, with fp32 accumulation, so
 * the result equals the token-by-token recurrence up to rounding (about
 * 1e-6 relative), not bit for bit; the same call on the same state gives
 * the same bits every time.  A mixed tile is dequantised once when
 * its chunk starts and requantised once at its end (its layout's
 * arithmetic), so its INT8 codes can differ by one from those of
 * rs_prefill_update where the FP32 state sits that close to a rounding
 * boundary.  Built for dk = dv = 128 on the FP32 layout and on the mixed
 * layouts with k_hi = 16 (one scale per row, or DAMP-exact groups of 32
 * with value scaling); other layouts return RS_ERR_UNSUPPORTED before any
 * launch, as do in_dtype RS_F16 on a mixed layout and B * L >= 2^31 - 32.
 * Use rs_prefill_update where bit-exactness with single decode steps is
 * needed. */
rs_status rs_prefill_chunked_update(const rs_layout *l, int32_t per_channel_decay, void *pool,
                                    int64_t n_slots, const int32_t *slot_idx, int32_t B,
                                    int32_t L, const int32_t *n_tokens, const void *q,
                                    const void *k, const void *v, int32_t in_dtype,
                                    const float *alpha, const float *beta, void *o,
                                    int32_t out_dtype, int32_t *status, void *stream);

/* Convert n slots between two layouts of the same shape (FP32 -> mixed
 * quantises with the rules above; mixed -> FP32 dequantises and un-permutes
 * rows; same kind copies).  slots: device int32 [n], used as both source and
 * destination slot. */
rs_status rs_state_convert(const rs_layout *src_l, const void *src_pool,
                           const rs_layout *dst_l, void *dst_pool, int64_t n_slots,
                           const int32_t *slots, int32_t n, int32_t *status,
                           void *stream);

/* ---- dasc checkpoint plans and pack / restore --------------------------- */

/* Selection plan ([dasc] §4.1): keep (host uint8 [L][n_units], 0/1) marks
 * the retained units of each of num_layers layers.  unit = RS_UNIT_HEAD
 * (GDN: n_units = Hv, unit = one head of the layout's head bytes) or
 * RS_UNIT_CHANNEL (KDA: n_units = Hv*dk, unit = row (h, u) of dv floats).
 * FP32 layouts take either unit.  A mixed FP16/INT8 layout ([DAMP] §5.2)
 * takes head units only: a head is copied verbatim with its FP16 rows, INT8
 * rows and scales; its rows are interleaved by word, so a key channel is not
 * a unit of its own (RS_ERR_UNSUPPORTED).  Host only: offsets o_0 = 0,
 * o_l = o_{l-1} + r_l ([dasc] Appendix B "Ragged (Scheme 2)") are computed
 * here. */
rs_status rs_plan_create(rs_plan **out, const rs_layout *l, int32_t num_layers,
                         int32_t unit, const uint8_t *keep);
rs_status rs_plan_destroy(rs_plan *p);

/* offsets: host int64 [L+1] (o_0..o_L, in units); unit_bytes: bytes per unit.
 * Checkpoint slot size is o_L * unit_bytes. */
rs_status rs_plan_offsets(const rs_plan *p, int64_t *offsets, int64_t *unit_bytes);

/* Copy the plan's index tables to the current device (allocates them once
 * per plan; [dasc] Appendix B.2: masks and offsets are precomputed once and
 * reused).  Required before pack/restore; synchronous. */
rs_status rs_plan_upload(rs_plan *p);

/* Pack ([dasc] §4.1, Appendix B): for each i < n, copy the retained units of
 * every layer of pool slot src_slots[i] into checkpoint slot
 * dst_ckpt_slots[i], layer l at units [o_{l-1}, o_l), ascending unit order.
 *   pool         device  [L] x (layer_stride_bytes apart) x [n_pool_slots][Hv][head]
 *   ckpt_pool    device  [n_ckpt_slots][o_L * unit_bytes] (may be NULL when o_L = 0)
 *   src_slots, dst_ckpt_slots  device int32 [n]   */
rs_status rs_ckpt_pack(const rs_plan *p, const void *pool, int64_t layer_stride_bytes,
                       int64_t n_pool_slots, const int32_t *src_slots,
                       const int32_t *dst_ckpt_slots, int32_t n, void *ckpt_pool,
                       int64_t n_ckpt_slots, int32_t *status, void *stream);

/* Restore, dasc-nr ([dasc] §4.2; [SRA] "One pool, two cache types": restore
 * the immutable checkpoint into the request's private running state): for
 * each i < n, every unit of every layer of pool slot dst_slots[i] is written,
 * retained units from checkpoint slot src_ckpt_slots[i], omitted units as
 * +0.0 (all bytes zero). */
rs_status rs_ckpt_restore(const rs_plan *p, const void *ckpt_pool, int64_t n_ckpt_slots,
                          const int32_t *src_ckpt_slots, void *pool,
                          int64_t layer_stride_bytes, int64_t n_pool_slots,
                          const int32_t *dst_slots, int32_t n, int32_t *status,
                          void *stream);

/* Pack for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call; it exists for integrations such as a serving
 * engine that reserves a fixed share of HBM for its own pools when it starts
 * and must not allocate afterwards, or a caller on a latency-critical path
 * that cannot afford the device-wide synchronisation of cudaFree.
 * Same arguments, layout and result as rs_ckpt_pack, but the plan needs no
 * rs_plan_upload: the plan's index table is copied (cudaMemcpyAsync on
 * `stream`, from a page-locked host copy that rs_plan_create made, so the
 * call does not synchronise) into a fixed array that the library holds in
 * device memory, and nothing is allocated or freed.  Limits and behaviour:
 *   - the plan may retain at most 262,144 units per checkpoint (o_L); a
 *     larger plan returns RS_ERR_UNSUPPORTED before any work;
 *   - a plan created while no CUDA device was reachable has no page-locked
 *     copy: RS_ERR_UNSUPPORTED;
 *   - a shape rs_ckpt_pack would refuse (n > 65,535, too many 512-byte
 *     chunks per checkpoint) returns RS_ERR_UNSUPPORTED before the array is
 *     touched;
 *   - the array (1 MiB) lives on every GPU that loads the library until the
 *     process exits;
 *   - the first call on a device looks up the array's device address (a
 *     host-side runtime query).  The address is kept for the process: do
 *     not use this call on a device after cudaDeviceReset.  Devices 0..63
 *     only;
 *   - all calls share the one array, which keeps the last call's table:
 *     calls whose work overlaps on the GPU (on different streams) race and
 *     must be ordered by the caller;
 *   - destroy the plan only after the call's copy has run (the copy reads
 *     the plan's page-locked table). */
rs_status rs_ckpt_pack_noalloc(const rs_plan *p, const void *pool, int64_t layer_stride_bytes,
                               int64_t n_pool_slots, const int32_t *src_slots,
                               const int32_t *dst_ckpt_slots, int32_t n, void *ckpt_pool,
                               int64_t n_ckpt_slots, int32_t *status, void *stream);

/* ---- dasc INT8 state checkpoint ------------------------------------------
 * [dasc] Appendix E.1 Eq. 8: an FP32 state is quantised once when the
 * checkpoint is written and dequantised once when it is reused.  Each row of
 * a retained unit (key channel u of head h: the [dasc] scale index (l, h, k)
 * shared over dv) gets a = max_v |S[u][v]|, s = max(a, 1e-8) / 127 and codes
 * clip(round_half_even(S / s), -127, 127) (FP32 maximum, division and
 * rounding; a NaN absmax takes the 1e-8 floor, as in the mixed layout);
 * reuse writes S^ = code * s.  The plan must be on an FP32 layout; units are
 * those of the plan (a head: dk rows; a key channel: 1 row).
 *
 * Checkpoint slot layout:
 *   codes  int8  [o_L][rows_per_unit][dv]   units in packed order
 *   scales f32   [o_L][rows_per_unit]       from byte codes_bytes on
 * and the slot is slot_bytes = codes + scales rounded up to 16 bytes (16,896
 * B per 128 x 128 head, 3.88x smaller than FP32). */
rs_status rs_ckpt_int8_bytes(const rs_plan *p, int64_t *codes_bytes, int64_t *slot_bytes);

/* INT8 pack: as rs_ckpt_pack (same slots, order, status bits and argument
 * rules), quantising each retained row into checkpoint slot
 * dst_ckpt_slots[i] of ckpt_pool (device, [n_ckpt_slots][slot_bytes]).
 * Requires rs_plan_upload and dv = 64 or 128. */
rs_status rs_ckpt_pack_int8(const rs_plan *p, const void *pool, int64_t layer_stride_bytes,
                            int64_t n_pool_slots, const int32_t *src_slots,
                            const int32_t *dst_ckpt_slots, int32_t n, void *ckpt_pool,
                            int64_t n_ckpt_slots, int32_t *status, void *stream);

/* INT8 restore, dasc-nr: every row of every layer of pool slot dst_slots[i]
 * is written, retained rows dequantised from checkpoint slot
 * src_ckpt_slots[i], omitted rows +0.0. */
rs_status rs_ckpt_restore_int8(const rs_plan *p, const void *ckpt_pool, int64_t n_ckpt_slots,
                               const int32_t *src_ckpt_slots, void *pool,
                               int64_t layer_stride_bytes, int64_t n_pool_slots,
                               const int32_t *dst_slots, int32_t n, int32_t *status,
                               void *stream);

/* ---- selection-plan builders (host only, offline) ------------------------
 * These compute the inputs of rs_plan_create (keep masks) and of
 * rs_layout_create (FP16 channel sets) from model weights and calibration
 * trajectories.  Host memory only; no device work; fp64 arithmetic from FP32
 * inputs, except that the quantisation error uses the FP32 storage
 * quantiser itself.  NULL pointers with a zero count are allowed. */

#define RS_GATE_STD 0   /* g = -exp(A_log) * softplus(a_s + d)             */
#define RS_GATE_K3  1   /* g = -5 * sigmoid(exp(A_log) * (a_s + d)) (safe) */

/* [dasc] §3.3 Eq. 2-3: static log-decay g_s of each unit from its learned
 * log-scale A_log[u] and decay bias d_bias[u] (host float [n_units]) with
 * the model-wide representative gate input a_s (the page uses -0.3 for the
 * standard gate, 0.8 for the Kimi-K3 safe gate), and the static retention
 * horizon H[u] = ln(epsilon) / g_s (host double [n_units]; the page uses
 * epsilon = 1e-3).  A unit is a GDN head or a KDA (head, key channel). */
rs_status rs_dasc_horizons(int32_t gate, const float *A_log, const float *d_bias, int64_t n_units,
                           double a_s, double epsilon, double *H);

/* [dasc] §4.1: keep[u] = 1 when H[u] > W_max (retained, global unit), else 0
 * (omitted, local).  The result is one layer's row of rs_plan_create's keep. */
rs_status rs_dasc_keep(const double *H, int64_t n_units, double W_max, uint8_t *keep);

/* [dasc] §4.2 Eq. 7: suffix-refresh window of dasc-wr.  For each omitted
 * unit (keep[u] = 0), W_u = clamp(next_pow2(H[u]), 4, W_max) with
 * next_pow2(x) = 2^ceil(log2 x) (x > 0; 4 for x = 0); *W_replay = min(
 * n_prefix, max W_u), or 0 when no unit is omitted.  W_max >= 4. */
rs_status rs_dasc_refresh_window(const double *H, const uint8_t *keep, int64_t n_units, int64_t W_max,
                                 int64_t n_prefix, int64_t *W_replay);

/* [DAMP] §5.1 Eq. 14-15: accumulated-error risk of each key channel of one
 * (layer, head).  states: host float [n_anchors][dk][dv], calibration
 * states at the scoring anchors (DAMP orientation, row = key channel);
 * decays: host float [n_anchors][horizon][dk], the decay factors a_{t+r,u}
 * of the horizon updates that follow each anchor.  C[u] (host double [dk]) =
 * mean over anchors of e_u * (1 + sum_{j=1..horizon} prod_{r<=j} a_r^2) with
 * e_u = sum_v (Q(S)[u][v] - S[u][v])^2 and Q the storage quantiser (one INT8
 * scale per row, as in rs_layout_create's INT8 rows). */
rs_status rs_damp_risk_scores(const float *states, const float *decays, int32_t n_anchors, int32_t dk,
                              int32_t dv, int32_t horizon, double *C);

/* [DAMP] §5.1 budgeted selection: for each of n_heads heads, the k_hi key
 * channels with the largest C (host double [n_heads][dk]); equal scores
 * rank the lower channel first; each head's channels are written in
 * ascending order to hi_rows (host int16 [n_heads][k_hi]) -- the format
 * rs_layout_create takes.  A NaN score is an error. */
rs_status rs_damp_select_hi_rows(const double *C, int32_t n_heads, int32_t dk, int32_t k_hi,
                                 int16_t *hi_rows);

#ifdef __cplusplus
}
#endif

#endif /* RECURRENT_STATE_H */
