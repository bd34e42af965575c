/*
 * q4.h -- C ABI of libq4.so: group-quantised int4 weight-only GEMV and skinny
 * GEMM (batch 1..8) for small-batch autoregressive decoding on GB300 (sm_103a).
 *
 * Weight format (rumik-oss-1 int4 engine page, rtts.neoandmatrix.me,
 * "Step 3: an int4 file and a first kernel"): each row of a projection is cut
 * into runs of 128 columns; a run has one fp16 scale and one fp16 minimum, and
 * its 4-bit codes are packed in pairs; a weight is
 *     w = code * scale + min.
 *
 * Canonical layout used by every call ("L0"):
 *   W       logical [N, K]: output row n, input column k.  K % 128 == 0.
 *   codes   uint8  [N, K/2] row-major.  Byte n*(K/2) + j holds column 2j in
 *           bits 0-3 (low nibble first) and column 2j+1 in bits 4-7.
 *   scales  fp16 bit patterns (uint16) [N, K/128] row-major, group g = k/128.
 *   mins    fp16 bit patterns (uint16) [N, K/128] row-major.
 *   X       bf16 bit patterns (uint16) [B, K] row-major (batch row b is X + b*K).
 *   Y       fp32 [B, N] row-major (batch row b is the slice Y + b*N).
 *
 * Conventions for every device call below:
 *   - Pointers marked "device" must be device (or managed) memory of the
 *     current CUDA device.  The caller owns every buffer; the library never
 *     allocates, frees or synchronises.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; a Q4_OK return means the
 *     launch was accepted, not that it finished.
 *   - Arguments are validated on the host before anything is enqueued; on an
 *     error nothing is launched.  Launch failures are reported as Q4_ERR_CUDA.
 *   - Every output column b of a call with batch B is bit-identical to the
 *     output of the same call with B = 1 on that activation row alone
 *     ("batch invariance", the pure-C TTS engine page, wpnews.pro, section
 *     on the batched matvec that first accumulated in a different order).
 *   - Calls are stateless apart from the caller's workspace and may be
 *     issued from several host threads on different streams.
 *   - Kernels that need more than 48 KB of shared memory get that limit raised
 *     (a function attribute, not stream work) on their first launch per
 *     device: make each entry point's first call outside stream capture.
 */
#ifndef Q4_H
#define Q4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    Q4_OK = 0,
    Q4_ERR_INVALID_ARG = 1,        /* null pointer, N <= 0, B outside 1..8, non-finite weight, fp16 range */
    Q4_ERR_UNSUPPORTED_SHAPE = 2,  /* K not a positive multiple of 128, or K > 65536, or N >= 2^31 */
    Q4_ERR_MISALIGNED = 3,         /* codes/X/workspace not 16-byte aligned, Y not 4, scales/mins not 2 */
    Q4_ERR_WORKSPACE = 4,          /* workspace missing or smaller than q4_workspace_bytes() */
    Q4_ERR_CUDA = 5,               /* a CUDA runtime call or kernel launch failed */
    Q4_ERR_TIMEOUT = 6             /* a bounded device-side wait gave up (see q4_device_status) */
} q4_status;

/*
 * One quantised matrix, device memory.  Either or both of:
 *   - the canonical layout L0 (codes, scales, mins; all three non-NULL), and
 *   - a tiled copy (`tiled`, built by q4_tile from L0): the layout the default
 *     kernels stream.  For each 16-row tile j (rows 16j..16j+15; rows >= N are
 *     zero) and each 128-column group g, one 1,088-byte record at offset
 *     (j * K/128 + g) * 1088:
 *        bytes    0..511   for l = 0..31: L0 bytes g*64 + 16*(l%4) .. +15 of row 16j + l/4
 *        bytes  512..1023  the same for row 16j + l/4 + 8
 *        bytes 1024..1087  for q = 0..7: (scale | min << 16) of row 16j+q, then of row 16j+q+8
 *     A warp reads one record with two 512-byte loads and one 64-byte load.
 * A call uses the tiled copy when present (and the default kernel is selected),
 * else L0.
 */
typedef struct {
    const uint8_t*  codes;   /* L0 [N, K/2], or NULL */
    const uint16_t* scales;  /* L0 [N, K/128] fp16 bits, or NULL */
    const uint16_t* mins;    /* L0 [N, K/128] fp16 bits, or NULL */
    int64_t N;
    int64_t K;
    const void*     tiled;   /* tiled copy, q4_tiled_bytes(N, K) bytes, 16-byte aligned, or NULL */
} q4_matrix;

/* How a call on an (N, K) matrix is split across the GPU.  Depends on N, K
 * and the device's SM count only -- never on the batch size B. */
typedef struct {
    int32_t row_blocks;      /* CTAs along N */
    int32_t k_splits;        /* CTAs along K (> 1: partial sums through the workspace) */
    int32_t warps_per_cta;
    int32_t prefetch_depth;  /* direct kernel: groups in flight per warp; stream kernel: ring stages */
    int32_t kernel;          /* 0 direct on the tiled copy + tensor-core dot (single matrices),
                                1 direct on L0 + tensor-core dot, 2 direct on L0 + CUDA-core fp32 dot,
                                3 stream (bulk copies into a shared-memory ring) on the tiled copy
                                  + tensor-core dot, 4 direct on the tiled copy + CUDA-core fp32 dot,
                                5 tile kernel: prepared activations + whole 16-row tiles per warp,
                                  persistent over a list (independent lists of several matrices),
                                6 flat kernel: one matrix, its records split evenly over all warps,
                                  partials of cut tiles added in shared memory (single matrices
                                  with fewer than two 16-row tiles per SM) */
    int32_t sm_count;
} q4_plan_info;

/*
 * q4_pack_host -- the offline export job ("Step 3": the int4 file is written
 * once, on the CPU, before the GPU sees the weights).  Host memory only.
 *   w       host fp32 [N, K] row-major, finite.
 *   codes   host out uint8 [N, K/2]; scales, mins host out uint16 [N, K/128].
 *   n_threads  worker threads (<= 0: all hardware threads).
 * Per row and per group of 128 columns: mn = min, mx = max (in double);
 * scale = fp16((mx - mn) / 15) and min = fp16(mn), each rounded once from
 * double to nearest-even; code = clamp(rint((w - min) / scale), 0, 15) in
 * double with the stored fp16 scale/min (code 0 when scale == 0).
 * Returns Q4_ERR_INVALID_ARG for null pointers, N <= 0, a non-finite weight,
 * or a group whose scale or min overflows fp16 (outputs then undefined);
 * Q4_ERR_UNSUPPORTED_SHAPE if K is not a positive multiple of 128.
 */
q4_status q4_pack_host(const float* w, int64_t N, int64_t K,
                       uint8_t* codes, uint16_t* scales, uint16_t* mins,
                       int n_threads);

/* Bytes of the tiled copy of an (N, K) matrix: ceil(N/16) * (K/128) * 1088 (0 if invalid). */
size_t q4_tiled_bytes(int64_t N, int64_t K);

/*
 * q4_tile -- build the tiled copy of W's L0 arrays into `tiled` (device,
 * 16-byte aligned, at least q4_tiled_bytes(N, K) bytes), asynchronously on
 * `stream`.  A pure rearrangement: no value changes.  Q4_ERR_INVALID_ARG if
 * W's L0 arrays or `tiled` are NULL, Q4_ERR_WORKSPACE if tiled_bytes is too
 * small, Q4_ERR_MISALIGNED / Q4_ERR_UNSUPPORTED_SHAPE as for q4_gemv.
 */
q4_status q4_tile(const q4_matrix* W, void* tiled, size_t tiled_bytes, void* stream);

/*
 * q4_workspace_bytes -- device workspace a q4_gemv / q4_gemm_skinny call on
 * (N, K, B) needs on the current device (0 when the call needs none).  The
 * workspace holds fp32 partial sums and arrival counters of a K split, or
 * the prepared activations when they do not fit in shared memory.  It must be
 * zero-filled once before its first use; every call leaves its counters at
 * zero again when it completes, so the same buffer can be reused by later
 * calls on the same stream (and by graph replays) without clearing.
 * Returns 0 for invalid shapes.
 */
size_t q4_workspace_bytes(int64_t N, int64_t K, int B);

/* q4_plan -- fill `out` with the split q4_gemv would use for (N, K) on the
 * current device.  Host only; Q4_ERR_UNSUPPORTED_SHAPE / Q4_ERR_INVALID_ARG
 * as for q4_gemv. */
q4_status q4_plan(int64_t N, int64_t K, q4_plan_info* out);

/*
 * q4_gemv -- y = W x for one activation vector ("Step 3": the GEMV that
 * dominates batch-1 decoding; fp32 accumulation).
 *   W     host pointer to a q4_matrix whose arrays are device memory.
 *   x     device bf16 bits [K], 16-byte aligned.
 *   y     device fp32 [N], 4-byte aligned; fully overwritten.
 *   ws    device workspace of ws_bytes >= q4_workspace_bytes(N, K, 1), or
 *         NULL when that is 0.
 * Same as q4_gemm_skinny with B = 1.
 */
q4_status q4_gemv(const q4_matrix* W, const uint16_t* x, float* y,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * q4_gemm_skinny -- Y[b, :] = W X[b, :] for b < B, 1 <= B <= 8 (the pure-C TTS
 * engine page's continuous batching: every weight row is read once and reused
 * for all B activation rows).  Column b of Y is bit-identical to q4_gemv on
 * X[b, :] alone.
 *   X  device bf16 bits [B, K] (16-byte aligned);  Y  device fp32 [B, N].
 *   ws as for q4_gemv with q4_workspace_bytes(N, K, B).
 */
q4_status q4_gemm_skinny(const q4_matrix* W, const uint16_t* X, int B, float* Y,
                         void* ws, size_t ws_bytes, void* stream);

/* Flag of q4_decode_step: the matrices are independent (no X[j] overlaps any Y[i]). */
#define Q4_STEP_INDEPENDENT 1u

/*
 * q4_decode_step -- the weight-streaming part of one decode step: n_mats skinny
 * GEMMs Y[i] = mats[i] X[i] in list order ("Step 3": 108 projections of 36
 * layers in one CUDA graph; "Step 4": q, k, v, gate and up fused into one
 * 25,088-row matrix, three GEMVs per layer).
 *   mats  host array [n_mats] of q4_matrix (device arrays inside).
 *   X     host array [n_mats] of device bf16 pointers, X[i] is [B, mats[i].K].
 *   Y     host array [n_mats] of device fp32 pointers, Y[i] is [B, mats[i].N].
 *   ws    workspace of at least q4_decode_step_workspace_bytes(...) for the
 *         same shapes, B and flags (zero-filled once before first use).
 *   flags Q4_STEP_INDEPENDENT: the caller guarantees that no X[j] overlaps any
 *         Y[i]; the whole list then runs as ONE persistent launch (at most 128
 *         matrices per launch) in which every SM walks the list in order and
 *         starts streaming the next matrix's weights while finishing the
 *         previous one (the rumik-oss-1 page's H100 lesson: at ~230 launches
 *         per step the fixed cost per kernel, not the bytes, set the speed).
 *         0: one launch per matrix; launch i+1 may start streaming its
 *         weights early but reads X[i+1] and writes Y[i+1] only after launch i
 *         has completed, so Y[i] may feed X[j] for j > i.
 * Kernels: an independent list of more than one matrix whose matrices all carry
 * the tiled copy runs as q4_step_prepare + q4_step_stream (two launches per 128
 * matrices).  Otherwise each matrix runs as q4_gemm_skinny does.  The two add
 * the 128-column groups of a row in different fixed orders (all groups in
 * sequence, versus K split across the warps of a CTA), so their outputs agree
 * to fp32 rounding, not bit for bit; each is bit-identical across batch sizes.
 * The host arrays are consumed before the call returns, so the call can be
 * captured into a CUDA graph and replayed.  Validates every matrix before
 * launching any.
 */
q4_status q4_decode_step(const q4_matrix* mats, int n_mats,
                         const uint16_t* const* X, float* const* Y, int B,
                         void* ws, size_t ws_bytes, unsigned flags, void* stream);

/* Workspace q4_decode_step needs for matrices of shapes (N[i], K[i]), batch B and
 * `flags` on the current device (0 for invalid input). */
size_t q4_decode_step_workspace_bytes(const int64_t* N, const int64_t* K, int n_mats, int B,
                                      unsigned flags);

/*
 * The two phases of q4_decode_step for an independent list whose matrices all
 * carry the tiled copy.
 *
 * q4_step_workspace_bytes -- bytes of device workspace both phases need for
 * matrices of input widths K[i] at batch B: the prepared activations, about
 * (K/128) * (256 * BT + 32) bytes per matrix, BT = B rounded up to 1, 2, 4 or 8.
 * 0 for invalid input.
 *
 * q4_step_prepare -- stage each X[i] (device bf16 [B, K_i], 16-byte aligned)
 * once into ws: in mma B-fragment order, times a power of two per batch column
 * (so that the products of codes and activations are normal fp32 numbers), with
 * the sum of every 128-column group and the per-column factors that undo the
 * scaling.  One launch per 128 matrices, one CTA per matrix.
 *
 * q4_step_stream -- Y[i] = mats[i] X[i] (device fp32 [B, N_i]) from the
 * activations that the last q4_step_prepare on this ws staged for the same
 * list (same order, shapes and B).  One persistent launch per 128 matrices,
 * one CTA per SM: CTA c owns one block of 16-row tiles of every matrix; its
 * warps take whole tiles from a shared counter, matrix after matrix, with no
 * block-wide barrier, and add all groups of a row in order.  Reading ws waits
 * for the previous kernel in the stream (programmatic dependent launch), so
 * the two phases may be enqueued back to back and captured in one graph.
 *
 * Both: Q4_ERR_INVALID_ARG for null pointers, B outside 1..8 or a matrix
 * without the tiled copy, Q4_ERR_WORKSPACE if ws_bytes is too small,
 * Q4_ERR_MISALIGNED / Q4_ERR_UNSUPPORTED_SHAPE as for q4_gemv.
 */
size_t q4_step_workspace_bytes(const int64_t* K, int n_mats, int B);
q4_status q4_step_prepare(const q4_matrix* mats, int n_mats, const uint16_t* const* X, int B,
                          void* ws, size_t ws_bytes, void* stream);
q4_status q4_step_stream(const q4_matrix* mats, int n_mats, float* const* Y, int B,
                         const void* ws, size_t ws_bytes, void* stream);

/*
 * q4_step_stream_readonly -- a measurement aid, not a computation: the read-only
 * twin of q4_step_stream (the rumik-oss-1 write-up, "Step 7: why the GEMV was
 * stuck": a copy of the GEMV that performs the same loads but no arithmetic shows
 * whether memory or the instruction stream sets the speed).  Same arguments,
 * same checks, same launch shape, the same weight records, activation words and
 * group sums read through the same shared-memory ring in the same tile order,
 * and the same Y stores -- but no unpack, no tensor-core product and no scale or
 * minimum arithmetic.  The values written to Y are meaningless.  Its time over
 * q4_step_stream's is the practical ceiling of the access pattern.
 */
q4_status q4_step_stream_readonly(const q4_matrix* mats, int n_mats, float* const* Y, int B,
                                  const void* ws, size_t ws_bytes, void* stream);

/*
 * q4_gemm_skinny_noalloc -- Y = W X exactly as the tile kernel computes it
 * (q4_step_prepare + q4_step_stream on a one-matrix list), for callers that
 * cannot allocate device memory and so cannot supply a workspace: code that
 * runs while a CUDA graph is being captured (cudaMalloc is not allowed there),
 * real-time threads such as an audio callback that must never wait on the
 * allocator (cudaMalloc/cudaFree can synchronise the device and take driver
 * locks), and plugins or embedded hosts whose device memory is budgeted and
 * owned by someone else.  The pages have no counterpart of this call.
 *   W  as for q4_gemm_skinny, and it must carry the tiled copy;
 *   X  device bf16 [B, K];  Y  device fp32 [B, N];  1 <= B <= 8.
 * Scratch: a fixed q4_noalloc_scratch_bytes() = 512 KiB array inside the
 * library, one per GPU that loads it, held until the process exits.  It holds
 * the prepared activations, (K/128) * (256 * BT + 32) + 32 bytes with BT = B
 * rounded up to 1, 2, 4 or 8: every K for B <= 2, K <= 63,488 for B <= 4 and
 * K <= 32,256 for B <= 8.  Larger requests return Q4_ERR_WORKSPACE before
 * anything is launched.  The call allocates nothing and frees nothing.
 * All calls on a device share the one array and each leaves its contents
 * behind (nothing in it needs to start at zero: every call rewrites what it
 * reads).  Calls that overlap on the GPU -- on different streams, or from
 * different host threads -- race on it; serialise them.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Only a successful lookup is kept (a failed one is tried again on the next
 * call); a device reset invalidates it, so do not reset a device this runs on.
 * Other errors as for q4_gemm_skinny; Q4_ERR_CUDA if the lookup fails.
 */
q4_status q4_gemm_skinny_noalloc(const q4_matrix* W, const uint16_t* X, int B, float* Y,
                                 void* stream);

/* Size in bytes of q4_gemm_skinny_noalloc's fixed scratch array. */
size_t q4_noalloc_scratch_bytes(void);

/*
 * q4_argmax_f32 -- per batch row of logits Y [B, N] (device fp32), the index
 * of the largest value, the lowest index among equal maxima (NaN ranks above
 * every number, as numpy's argmax does), written to idx (device int32 [B]).
 * The greedy pick after the output head ("Step 4" of the rumik-oss-1 page
 * samples on the GPU; argmax is its deterministic case).
 * Q4_ERR_INVALID_ARG for null pointers, B outside 1..8 or N outside 1..2^31-1.
 */
q4_status q4_argmax_f32(const float* Y, int B, int64_t N, int32_t* idx, void* stream);

/*
 * Argmax over a row-sharded head (one process per GPU, each holding a range of
 * the head's rows; the full logits never leave their GPUs).  A rank's best
 * logit per batch row is packed into one 64-bit key whose order is the
 * q4_argmax_f32 rule over the whole row: bits 63..32 rank the value (NaN above
 * every number, -0 equal to +0, larger above smaller), bits 31..0 hold the
 * complement of the global row index (lower index above higher among equal
 * values); the top bit is then flipped so that signed int64 order equals it.
 * The largest key over all ranks -- one MAX all-reduce of B int64 values -- is
 * the whole row's argmax.  (The pages run on one GPU; this is the plain
 * reading of splitting a GEMV's output rows across GPUs and merging the
 * per-GPU maxima.)
 *
 * q4_argmax_key_f32 -- keys[b] = the key of the best of Y[b, 0..N-1] (device
 *   fp32 [B, N], 4-byte aligned), whose global row indices are index_base + n.
 *   keys device int64 [B], 8-byte aligned.  1 <= B <= 65535, 1 <= N < 2^31,
 *   0 <= index_base and index_base + N <= 2^32 - 1.
 * q4_argmax_key_index -- idx[b] = the global row index held in keys[b]
 *   (device int64 [B] -> device int32 [B]).
 * Both: Q4_ERR_INVALID_ARG for null pointers or out-of-range sizes,
 * Q4_ERR_MISALIGNED, Q4_ERR_CUDA for a failed launch.  Asynchronous on stream.
 */
q4_status q4_argmax_key_f32(const float* Y, int B, int64_t N, int64_t index_base, int64_t* keys, void* stream);
q4_status q4_argmax_key_index(const int64_t* keys, int B, int32_t* idx, void* stream);

/*
 * q4_gemm_prefill -- Y[m, :] = W X[m, :] for a prompt of M tokens (the rumik-oss-1
 * write-up, "Step 8: a prefill that stays int4": no dequantised copy of the
 * weights; each group is expanded for the tensor cores and its scale and
 * minimum are folded into the fp32 result).  fp32 accumulation; a tensor-core
 * GEMM, not bound by the weight bytes once M is large.  Two kernels:
 *   - on a compute capability 10.x device: tcgen05.mma with TMEM accumulators,
 *     activations by TMA (a prep kernel first writes a scaled, slot-permuted
 *     copy of X into the workspace), 128 x 128 output tiles;
 *   - otherwise (or with the environment variable Q4_PREFILL_TC=0): mma.sync
 *     over token blocks of 8.
 *   Both are deterministic; they agree with each other to fp32 rounding.
 *   W   host pointer; W->tiled (device) is required.
 *   X   device bf16 bits [M, K], 16-byte aligned;  Y device fp32 [M, N].
 *   ws  device workspace of ws_bytes >= q4_prefill_workspace_bytes(K, M) (enough
 *       for either kernel; no initial content needed), 16-byte aligned.
 * Q4_ERR_INVALID_ARG for null pointers, no tiled copy or M outside 1..2^24.
 * A bounded wait of the tcgen05 kernel that gives up is reported by
 * q4_device_status as Q4_ERR_TIMEOUT.
 * q4_prefill_kernel -- which kernel q4_gemm_prefill runs for (K, M) on the
 *   current device: 1 the tcgen05 kernel, 0 the mma.sync kernel, -1 invalid sizes.
 */
size_t q4_prefill_workspace_bytes(int64_t K, int64_t M);
q4_status q4_gemm_prefill(const q4_matrix* W, const uint16_t* X, int64_t M, float* Y, void* ws, size_t ws_bytes,
                          void* stream);
int q4_prefill_kernel(int64_t K, int64_t M);

/*
 * q4_sample_topk -- top-k sampling with the Gumbel-max trick over logits
 * (rumik-oss-1 write-up, "Step 4": the next token drawn on the device, top-k
 * plus Gumbel-max; "Steps 9-10": candidates ranked by 64-bit integer keys
 * built from each logit's bit pattern and its position).  Per batch row b of Y [B, N] (device
 * fp32): rank the logits -- NaN above every number, larger first, the lower
 * index first among equal values (the q4_argmax_f32 order) -- and keep the first
 * k; score rank r as fp32(fp32(Y[b, i_r] * inv_temperature) + noise[b, r]), two
 * rounded binary32 operations (never fused); token[b] = i_r of the best score
 * (NaN first, ties to the lower rank).  The caller supplies the randomness:
 * noise [B, k] (device fp32), Gumbel(0, 1) noise for ranks 0..k-1.
 *   k     1 <= k <= min(N, 1024);  inv_temperature > 0 and finite.
 *   token device int32 [B];  topk device int32 [B, k] (the ranked indices) or NULL.
 * One CTA of 1024 threads per row, no workspace.  Q4_ERR_INVALID_ARG for null
 * pointers or out-of-range k, B (1..65535), N or inv_temperature;
 * Q4_ERR_MISALIGNED unless every pointer is 4-byte aligned.
 */
q4_status q4_sample_topk(const float* Y, int B, int64_t N, int k, float inv_temperature, const float* noise,
                         int32_t* token, int32_t* topk, void* stream);

/* ------------------------------------------------------------------------
 * The int8 output head.  The rumik-oss-1 write-up keeps every projection in
 * int4 except the output head ("Steps 9-10: streaming to the speaker": the
 * audio head got int8 weights and a dedicated CUDA kernel, int4 having cost that
 * matrix clearly more accuracy than the others; "Step 2": int8 weights as
 * torchao quantized tensors).  Format (torchao's int8 weight-only scheme; the pages give no more
 * detail): per output row n an fp16 scale s_n = fp16(max_k |w[n,k]| / 127),
 * codes c = clamp(rint(w / s_n), -127, 127) as int8, w_hat = c * s_n.
 * ------------------------------------------------------------------------ */
typedef struct {
    const int8_t*   codes;   /* [N, K] row-major (device for q8_tile), or NULL once tiled */
    const uint16_t* scales;  /* [N] fp16 bits, device */
    int64_t N;
    int64_t K;               /* K % 128 == 0 */
    const void*     tiled;   /* q8_tiled_bytes(N, K) bytes, 16-byte aligned, or NULL */
} q8_matrix;

/* q8_pack_host -- quantise fp32 w [N, K] (host) into codes int8 [N, K] and
 * scales uint16 [N] (host), as above.  Q4_ERR_INVALID_ARG for null pointers,
 * non-finite weights or a row whose scale overflows fp16. */
q4_status q8_pack_host(const float* w, int64_t N, int64_t K, int8_t* codes, uint16_t* scales, int n_threads);

/* q8_tiled_bytes -- bytes of the tiled copy: one 2,048-byte record per 16-row
 * tile and 128-column group at (tile * K/128 + group) * 2048; lane l's 32 code
 * bytes of row 16 tile + l/4 (columns 32 (l%4) ..) at 32 l, the same of row
 * + 8 at 1024 + 32 l; rows >= N are zero.  0 for invalid shapes. */
size_t q8_tiled_bytes(int64_t N, int64_t K);

/* q8_tile -- build the tiled copy from W->codes on `stream`.  Q4_ERR_INVALID_ARG
 * for null codes/tiled, Q4_ERR_WORKSPACE if tiled_bytes is too small. */
q4_status q8_tile(const q8_matrix* W, void* tiled, size_t tiled_bytes, void* stream);

/* q8_head_workspace_bytes -- device workspace of q8_head on (N, K, B): the
 * per-CTA argmax candidates, and the prepared activations when they do not fit
 * in shared memory.  No initial content needed.  0 for invalid shapes. */
size_t q8_head_workspace_bytes(int64_t N, int64_t K, int B);

/*
 * q8_head -- Y[b, :] = W_hat X[b, :] (fp32 accumulation) for b < B, 1 <= B <= 8,
 * and/or idx[b] = the index of the largest Y[b, n] (lowest index among equal
 * maxima, NaN first), computed in the same launch as the logits: each CTA keeps
 * its best row per column, and a one-CTA pass picks the best of those.
 *   W    host pointer; W->tiled and W->scales device memory.
 *   X    device bf16 bits [B, K], 16-byte aligned.
 *   Y    device fp32 [B, N] (4-byte aligned), or NULL to skip the logits.
 *   idx  device int32 [B], or NULL to skip the argmax (not both NULL).
 *   ws   device workspace of ws_bytes >= q8_head_workspace_bytes(N, K, B).
 * Every batch column is bit-identical to the same call at B = 1 (the split of
 * the work depends on N, K and the SM count only).  Asynchronous on `stream`.
 */
q4_status q8_head(const q8_matrix* W, const uint16_t* X, int B, float* Y, int32_t* idx, void* ws,
                  size_t ws_bytes, void* stream);

/*
 * q4_flash_decode -- one decode step of grouped-query attention over a KV
 * cache, split over chunks of the cache (the rumik-oss-1 write-up, "Step 6:
 * flash-decoding for long clips": each KV head's cache cut into pieces worked
 * on in parallel, the grouped query heads forming the rows of one
 * matrix-multiply tile, a separate small kernel merging the pieces).  For every
 * sequence b and query head h, with g = n_q_heads / n_kv_heads:
 *     O[b,h,:] = sum_{p < len_b} softmax_p(scale * <Q[b,h,:], K[b,h/g,p,:]>) V[b,h/g,p,:]
 * (query head h reads KV head h / g).  fp32 softmax and accumulation; the
 * weights enter the tensor cores as bf16 hi + lo parts (relative error below
 * 2^-18).
 *   Q        device bf16 bits [B, n_q_heads, head_dim], 16-byte aligned.
 *   K_cache, V_cache  device bf16 bits [B, n_kv_heads, max_len, head_dim], 16-byte aligned
 *            (every KV head's positions contiguous).
 *   lengths  device int32 [B]: len_b = lengths[b] clamped to 0..max_len; only
 *            positions 0..len_b-1 are read.  len_b = 0 gives O[b] = 0.
 *   head_dim 64 or 128;  1 <= n_q_heads / n_kv_heads <= 16 (a whole multiple);
 *   B, n_kv_heads 1..65535;  1 <= max_len <= 2^30;  scale finite.
 *   n_chunks chunks per KV head at most, 1..4096, or 0 for the default of
 *            about eight per SM for one sequence (q4_flash_decode_chunks
 *            reports it), but no more than ceil(max_len / 32) (a shorter cache
 *            has no more chunks than that).  The chunk length is ceil(len_b / chunks) rounded up
 *            to 16 and at least 32 positions, so a sequence's result does not
 *            depend on B or on the other sequences.
 *   O        device fp32 [B, n_q_heads, head_dim], 4-byte aligned.
 *   ws       device workspace, 16-byte aligned, of ws_bytes >=
 *            q4_flash_decode_workspace_bytes(...) (no initial content needed).
 * Two kernels on `stream` (chained by programmatic dependent launch); nothing
 * allocated.  Every device-side wait is bounded; one that gives up is reported
 * by q4_device_status (Q4_ERR_TIMEOUT).  The first call per device and head
 * size raises the split kernel's shared-memory limit and queries its
 * occupancy: make it before any stream capture.  Q4_ERR_INVALID_ARG for null pointers or out-of-range B, heads,
 * group, chunks, max_len or scale; Q4_ERR_UNSUPPORTED_SHAPE for another
 * head_dim; Q4_ERR_MISALIGNED; Q4_ERR_WORKSPACE if ws_bytes is too small.
 */
/* Chunks per KV head that q4_flash_decode plans for (n_chunks itself when > 0;
 * the default needs the current device's SM count, and a call with a short
 * max_len uses at most ceil(max_len / 32) of them); the workspace is sized for
 * this count.  0 for invalid arguments or when the device cannot be queried. */
int q4_flash_decode_chunks(int n_kv_heads, int n_chunks);
/* Workspace bytes for these sizes (0 for invalid arguments, as above). */
size_t q4_flash_decode_workspace_bytes(int B, int n_q_heads, int n_kv_heads, int head_dim, int n_chunks);
q4_status q4_flash_decode(const uint16_t* Q, const uint16_t* K_cache, const uint16_t* V_cache,
                          const int32_t* lengths, int B, int n_q_heads, int n_kv_heads, int head_dim,
                          int64_t max_len, float scale, int n_chunks, float* O, void* ws, size_t ws_bytes,
                          void* stream);

/*
 * q4_device_status -- wait for `stream`, then read and clear the device error
 * word.  Every wait inside the kernels is bounded; one that gives up sets the
 * word and the kernel carries on to its end (its outputs are then invalid).
 * Returns Q4_ERR_TIMEOUT if a wait gave up since the last call, Q4_OK if not,
 * Q4_ERR_CUDA if the stream reports an error.
 */
q4_status q4_device_status(void* stream);

/* Static, NUL-terminated description of a status code. */
const char* q4_status_string(q4_status s);

#ifdef __cplusplus
}
#endif
#endif /* Q4_H */
