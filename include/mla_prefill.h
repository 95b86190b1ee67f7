/*
 * libmla_prefill -- MLA (multi-head latent attention) prefill over a ragged
 * batch and a paged K_rope cache, for one sm_103 GPU.
 *
 * Two stages:
 *   mla_prefill_plan    tiles each sequence's K context into buffer rows
 *                       (generic_flare_mla_prefill_ragged_paged_plan).
 *   mla_prefill_ragged  ragged causal attention with a 192-wide Q head, 128
 *                       per-head K_nope dims plus 64 K_rope dims shared by all
 *                       heads, 128-wide V and output (flare_mla_prefill).
 * Chunked execution runs the second stage over the plan's buffer rows: all
 * rows in one call (mla_prefill_ragged_chunked), or one row per call
 * (mla_prefill_ragged_chunk) folded in place or combined by mla_prefill_merge.
 *
 * Conventions shared by every entry point:
 *   - Every pointer marked "device" is caller-owned device memory; the library
 *     never allocates or frees device memory and keeps no per-call state.  The
 *     one exception is mla_prefill_ragged_noalloc: its scheduler workspace is
 *     a fixed 33,024-byte device array inside the library, held on every GPU
 *     that loads it until process exit and shared by all calls of that entry
 *     point.
 *   - Calls are asynchronous on `stream`; none synchronises except
 *     mla_read_device_status, which says so.  Descriptor structs are host
 *     memory read during the call only.
 *   - Argument errors are detected on the host before any launch and return
 *     MLA_ERR_INVALID_ARG; nothing is enqueued in that case.  A device that is
 *     not compute capability 10.3 gives MLA_ERR_UNSUPPORTED (there is no CPU
 *     path).  A failed launch gives MLA_ERR_CUDA.  mla_last_error_string()
 *     describes the last failure of the calling thread.
 *   - `stream` is a cudaStream_t (0 = legacy default stream).
 */
#ifndef MLA_PREFILL_H_
#define MLA_PREFILL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mla_stream_t; /* same type as cudaStream_t */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,
  MLA_ERR_UNSUPPORTED = 2,
  MLA_ERR_CUDA = 3,
} mla_status_t;

typedef enum {
  MLA_DTYPE_BF16 = 0,
  MLA_DTYPE_FP8_E4M3 = 1, /* float8_e4m3fn: no infinities, 0x7F/0xFF are NaN */
  MLA_DTYPE_U32 = 2,
  MLA_DTYPE_F32 = 3,
} mla_dtype_t;

typedef enum {
  MLA_MASK_CAUSAL = 0, /* query i of sequence b sees keys j <= cache_lens[b] + i */
  MLA_MASK_NULL = 1,   /* every key of the sequence's context is visible */
} mla_mask_t;

typedef enum {
  MLA_SCALE_NONE = 0,
  MLA_SCALE_PER_TENSOR = 1, /* `scale` points at one float */
  MLA_SCALE_PER_TOKEN = 2,  /* one float per token: K_rope pool slot (index page * P + slot),
                               contiguous K_rope row, or fp8 K_nope row (index = K row) */
} mla_scale_gran_t;

/* A strided view of device memory.  `data` addresses element [0, 0, ...];
 * strides are in elements and the innermost dimension must have stride 1.
 * fp8 tensors carry a dequantisation scale: real value = code value * scale. */
typedef struct {
  void* data;
  mla_dtype_t dtype;
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];
  const float* scale; /* device; fp8 only, else NULL */
  mla_scale_gran_t scale_gran;
} mla_tensor_t;

/*
 * Prefill plan (generic_flare_mla_prefill_ragged_paged_plan: summary; Args:
 * input_row_offsets, buffer_token_size, buffer_row_offsets, cache_offsets,
 * buffer_lengths).
 *
 * Sequence b has n_b = input_row_offsets[b+1] - input_row_offsets[b] new tokens
 * and cache_lens[b] previously cached tokens; its K context holds
 * L_b = cache_lens[b] + n_b tokens.  The contexts are packed in batch order
 * (G_b = L_0 + ... + L_{b-1}, S = G_batch) and cut into buffer rows of
 * T = buffer_token_size tokens; R = ceil(S / T) rows are used.  For every row
 * r < max_buffer_rows:
 *   buffer_row_offsets[r*(batch+1) + b] = clamp(G_b - r*T, 0, T)   (b = 0..batch)
 *   cache_offsets[r*batch + b]          = clamp(r*T - G_b, 0, L_b)
 *   buffer_lengths[r]                   = min(T, S - r*T) if r < R, else -1
 * so row r holds tokens [cache_offsets[r,b], cache_offsets[r,b] + len) of
 * sequence b at positions [buffer_row_offsets[r,b], buffer_row_offsets[r,b+1]).
 *
 *   input_row_offsets  device uint32 [batch+1], non-decreasing, first entry 0
 *   cache_lens         device uint32 [batch], prior (cached) length per sequence
 *   batch              1 .. 16384
 *   buffer_token_size  T >= 1
 *   max_buffer_rows    rows the three outputs have room for (may be 0)
 *   buffer_row_offsets device uint32 [max_buffer_rows, batch+1] (written)
 *   cache_offsets      device uint32 [max_buffer_rows, batch]   (written)
 *   buffer_lengths     device int32  [max_buffer_rows]          (written)
 *   num_rows           device uint32 [1] or NULL: receives R; rows past
 *                      max_buffer_rows are not written.  It receives
 *                      0xFFFFFFFF, and the outputs are unspecified, when S does
 *                      not fit in 32 bits or input_row_offsets decreases
 *                      somewhere (a negative new-token count).
 * One kernel launch, no host synchronisation.
 */
mla_status_t mla_prefill_plan(const uint32_t* input_row_offsets, const uint32_t* cache_lens,
                              uint32_t batch, uint32_t buffer_token_size,
                              uint32_t max_buffer_rows, uint32_t* buffer_row_offsets,
                              uint32_t* cache_offsets, int32_t* buffer_lengths,
                              uint32_t* num_rows, mla_stream_t stream);

/* Rows needed for a K total of at most `total_k_upper_bound` tokens:
 * ceil(total_k_upper_bound / buffer_token_size); 0 if buffer_token_size is 0. */
uint32_t mla_prefill_plan_max_rows(uint64_t total_k_upper_bound, uint32_t buffer_token_size);

/* Bytes of device workspace mla_prefill_ragged needs for `batch` sequences
 * with bf16 inputs. */
size_t mla_prefill_ragged_workspace_size(uint32_t batch);

/* Bytes of device workspace mla_prefill_ragged needs with fp8 inputs: the bf16
 * size plus 128 bytes per K_rope pool slot (pool_slots = num_pages * P), where
 * each call first writes K_rope converted to bf16 (code * s_r[slot] / s_k).
 * With per-token K_nope scales the converted rows sit at the K rows instead:
 * pass the number of K rows Sk as pool_slots. */
size_t mla_prefill_ragged_workspace_size_fp8(uint32_t batch, uint64_t pool_slots);

/*
 * Ragged MLA prefill attention (flare_mla_prefill: description; Args: output,
 * q, k, v, k_rope, mask_functor, valid_length, scale; the k_rope_scales
 * overload for fp8 K_rope).
 *
 * For sequence b (B = page_table->shape[0]) with n_b new tokens at rows
 * row_offsets[b] .. row_offsets[b+1]-1 of q/out, prior length p_b =
 * cache_lens[b] and context L_b = p_b + n_b whose K/V rows are
 * G_b .. G_b + L_b - 1 of k_nope/v (G_b = L_0 + ... + L_{b-1}), every head h
 * and query i < n_b:
 *   K[j]   = [ k_nope[G_b + j, h, 0:128] , k_rope(b, j)[0:64] ]
 *   k_rope(b, j) = k_rope_pages[page_table[b, j / P], j % P, 0:64]
 *   s_j    = scale * dot(q[row_offsets[b] + i, h, 0:192], K[j])
 *   out[row_offsets[b] + i, h, :] = sum_j softmax(s)_j * v[G_b + j, h, :]
 * over the keys the mask leaves visible (causal: j <= p_b + i; null: j < L_b).
 *
 *   out          device bf16 [Tq, H, 128]                       (written)
 *   q            device [Tq, H, 192], bf16 or fp8 (per-tensor scale);
 *                dims 0..127 pair with k_nope, 128..191 with K_rope
 *   k_nope, v    device [Sk, H, 128], same dtype as q, Sk >= sum of L_b.  fp8:
 *                per-tensor scales, or for k_nope one float per K row
 *                (scale_gran MLA_SCALE_PER_TOKEN, [Sk] floats, > 0): key row t
 *                is then dequantised with k_nope->scale[t]
 *   k_rope_pages device [num_pages, P, 64]; stride[1] (token stride) may exceed
 *                64, e.g. the rope tail of a wider latent row.  bf16 with bf16
 *                q; fp8 (per-token scale) with fp8 q.
 *   page_table   device uint32 [B, max_pages]; entries must be < num_pages for
 *                every page a context touches
 *   row_offsets  device uint32 [B+1], non-decreasing, first entry 0, last = Tq
 *   cache_lens   device uint32 [B]
 *   scale        softmax scale applied to q.k (typically 1/sqrt(192))
 *   workspace    device, >= mla_prefill_ragged_workspace_size(B) bytes for bf16
 *                inputs, >= mla_prefill_ragged_workspace_size_fp8(B, num_pages * P)
 *                for fp8 inputs (with per-token K_nope scales: (B, Sk));
 *                256-byte aligned; overwritten by every call, so concurrent
 *                calls need distinct workspaces.  Its first uint32 is the
 *                device status word (0 = ok; see mla_read_device_status).
 * Shapes, dtypes, strides, alignment and 32-bit index limits are checked on the
 * host.  Offsets and page ids live on the device: an out-of-range page id or
 * page-table column makes the kernel skip that load and set a status bit
 * (MLA_DEVICE_STATUS_*) instead of faulting.
 * Launches: a one-CTA scheduler, for fp8 inputs a K_rope conversion pass
 * (before the scheduler, or after it with per-token K_nope scales, when it
 * converts by K row), then the persistent attention kernel; no host
 * synchronisation.
 */
mla_status_t mla_prefill_ragged(const mla_tensor_t* out, const mla_tensor_t* q,
                                const mla_tensor_t* k_nope, const mla_tensor_t* v,
                                const mla_tensor_t* k_rope_pages, const mla_tensor_t* page_table,
                                const uint32_t* row_offsets, const uint32_t* cache_lens,
                                float scale, mla_mask_t mask, void* workspace,
                                size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_prefill_ragged with an optional lse output and flags
 * (flare_mla_prefill: description; Args as mla_prefill_ragged):
 *   lse    device float32 [Tq, H] (written) or NULL: ln sum_j exp(s_j) over
 *          each query's visible keys (s_j the scaled scores)
 *   flags  0 or MLA_FP8_PRECISE
 * Everything else as mla_prefill_ragged.
 */
mla_status_t mla_prefill_ragged_ex(const mla_tensor_t* out, const mla_tensor_t* lse,
                                   const mla_tensor_t* q, const mla_tensor_t* k_nope,
                                   const mla_tensor_t* v, const mla_tensor_t* k_rope_pages,
                                   const mla_tensor_t* page_table, const uint32_t* row_offsets,
                                   const uint32_t* cache_lens, float scale, mla_mask_t mask,
                                   uint32_t flags, void* workspace, size_t workspace_bytes,
                                   mla_stream_t stream);

/*
 * Ragged MLA prefill attention with a contiguous K_rope (flare_mla_prefill:
 * the overload taking k_rope as a plain tensor, and cache_offsets, which is
 * None "when the cache is contiguous").
 *
 * As mla_prefill_ragged, except that K_rope is not paged: k_rope row
 * G_b + j holds the 64 rope dims of key j of sequence b, the same row as
 * k_nope / v, so K[j] = [ k_nope[G_b + j, h, :] , k_rope[G_b + j, :] ].
 *   k_rope       device [Sk, 64] (rows = k_nope's rows), bf16 with bf16 q;
 *                fp8 with fp8 q, with one float scale per row
 *                (scale_gran MLA_SCALE_PER_TOKEN, index = row).  The row
 *                stride may exceed 64 (the rope tail of a wider latent row)
 *                and must be a multiple of 16 bytes.
 *   batch        B >= 1 (no page table carries it); row_offsets has B+1
 *                entries, cache_lens B.
 *   workspace    >= mla_prefill_ragged_workspace_size(B) for bf16 inputs,
 *                >= mla_prefill_ragged_workspace_size_fp8(B, Sk) for fp8.
 * Each 128-key tile's K_rope arrives as one TMA box (no page lookups).
 */
mla_status_t mla_prefill_ragged_contiguous(const mla_tensor_t* out, const mla_tensor_t* q,
                                           const mla_tensor_t* k_nope, const mla_tensor_t* v,
                                           const mla_tensor_t* k_rope, const uint32_t* row_offsets,
                                           const uint32_t* cache_lens, uint32_t batch, float scale,
                                           mla_mask_t mask, void* workspace, size_t workspace_bytes,
                                           mla_stream_t stream);

/*
 * Ragged MLA prefill attention with Q split into q_nope and q_rope
 * (flare_mla_prefill: the overloads taking q_nope, q_rope, q_scale, k_scales;
 * k_rope as a plain tensor, or from the paged cache).
 *
 * The result is that of mla_prefill_ragged with q = [q_nope | q_rope]:
 *   q_nope   device [Tq, H, 128], bf16 or fp8 e4m3 with a per-tensor scale
 *            (the pages' q_scale; scale_gran MLA_SCALE_PER_TENSOR)
 *   q_rope   device bf16 [Tq, H, 64], real values (not scaled)
 *   k_nope   device [Sk, H, 128], q_nope's dtype; fp8 with a per-tensor scale
 *            or one scale per K row, MLA_SCALE_PER_TOKEN, [Sk] floats > 0 (the
 *            pages' k_scales, whose granularity the pages leave open)
 *   v        device [Sk, H, 128], q_nope's dtype; fp8 v without a scale of
 *            its own is dequantised with k_nope's scale (per-tensor k_nope
 *            only; with per-token k_nope scales v needs its own)
 *   k_rope, page_table  page_table != NULL: k_rope is the paged pool
 *            [num_pages, P, 64] as in mla_prefill_ragged (fp8: per-token
 *            scales); page_table == NULL: k_rope is contiguous [Sk, 64] as in
 *            mla_prefill_ragged_contiguous
 *   batch    B (must match page_table's rows when one is given)
 * Workspace as for the matching fused-Q call (per-token K_nope scales:
 * mla_prefill_ragged_workspace_size_fp8(B, Sk)).
 */
mla_status_t mla_prefill_ragged_split(const mla_tensor_t* out, const mla_tensor_t* q_nope,
                                      const mla_tensor_t* q_rope, const mla_tensor_t* k_nope,
                                      const mla_tensor_t* v, const mla_tensor_t* k_rope,
                                      const mla_tensor_t* page_table, uint32_t batch,
                                      const uint32_t* row_offsets, const uint32_t* cache_lens,
                                      float scale, mla_mask_t mask, void* workspace,
                                      size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_prefill_ragged for callers that cannot allocate device memory.  No
 * counterpart on the reference pages: it exists for callers such as a plug-in
 * whose host framework owns all device memory and offers it no scratch
 * buffer, or a latency-critical path that may not call cudaMalloc (which can
 * synchronise the device).  Arguments and results are those of
 * mla_prefill_ragged without `workspace` / `workspace_bytes`; the caller still
 * passes every input and output.
 *   - The scheduler workspace is a fixed device array inside the library
 *     (33,024 bytes, room for 1024 sequences) that every GPU loading the
 *     library keeps until process exit.  A batch above 1024 returns
 *     MLA_ERR_INVALID_ARG, and so do fp8 inputs (any of q, k_nope, v,
 *     k_rope_pages), whose K_rope conversion needs more room than the array
 *     has.
 *   - The first call on a device looks the array's address up with
 *     cudaGetSymbolAddress (one-time set-up with that device current); make
 *     that first call before any stream capture.  Later calls only launch.
 *     The address is kept together with the id of the device's current
 *     context; after cudaDeviceReset (a new primary context, the array at a
 *     new address) the next call repeats the set-up, so make that call
 *     before any stream capture too.
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 *   - All calls share the one array and each call rewrites what it needs, so
 *     calls whose kernels can overlap on the GPU (different streams without
 *     ordering between them) race and must not be issued.
 *   - The device status word of these calls stays inside the library and is
 *     not readable through mla_read_device_status.
 */
mla_status_t mla_prefill_ragged_noalloc(const mla_tensor_t* out, const mla_tensor_t* q,
                                        const mla_tensor_t* k_nope, const mla_tensor_t* v,
                                        const mla_tensor_t* k_rope_pages,
                                        const mla_tensor_t* page_table,
                                        const uint32_t* row_offsets, const uint32_t* cache_lens,
                                        float scale, mla_mask_t mask, mla_stream_t stream);

/*
 * One buffer row of chunked execution (flare_mla_prefill: Args
 * cache_row_offsets, cache_offsets; generic_flare_mla_prefill_ragged_paged_plan:
 * buffer_row_offsets, cache_offsets, buffer_lengths).
 *
 * The plan cuts the K context into buffer rows; row r holds, for sequence b,
 * W_b = buffer_row_offsets[b+1] - buffer_row_offsets[b] keys, the context
 * positions a = cache_offsets[b] .. cache_offsets[b] + W_b - 1, at rows
 * buffer_row_offsets[b] + (a - cache_offsets[b]) of this call's k_nope / v
 * (the row's contiguous K buffer).  Pass row r of the plan's outputs:
 * buffer_row_offsets + r * (B + 1) and cache_offsets + r * B.  Everything
 * else is as in mla_prefill_ragged, with these differences:
 *   - keys are the row's only; the causal mask and the K_rope page lookup use
 *     the context position a (causal: a <= cache_lens[b] + i);
 *   - out receives the softmax over the row's visible keys, and
 *     lse[t, h] = ln sum_j exp(s_j) over the same keys (natural log, s_j the
 *     scaled scores; fp8 scores include the dequantisation scales);
 *   - a query that sees no key of the row gets out = 0 and lse = -inf;
 *   - rows of sequences with W_b = 0 are not written (neither out nor lse);
 *   - flags = MLA_CHUNK_ACCUMULATE folds the row into out / lse instead of
 *     overwriting them: for a sequence whose window starts after context
 *     position 0 (cache_offsets[b] > 0), out and lse must hold the result
 *     over its earlier positions (the earlier rows' calls, made in row
 *     order with this flag), and the call leaves the combination
 *       lse' = ln(e^lse + e^lse_row),
 *       out' = (e^lse out + e^lse_row out_row) / (e^lse + e^lse_row);
 *     a sequence whose window starts at position 0 is written afresh.  After
 *     the last row, out is the full-context result and lse its log-sum-exp,
 *     with no mla_prefill_merge and no per-row buffers.  flags = 0 writes the
 *     row's own result.  MLA_FP8_PRECISE may be ORed in (fp8 inputs).
 *   lse          device float32 [Tq, H] (written), 4-byte aligned
 *   k_nope, v    device [S_row, H, 128] with S_row >= buffer_row_offsets[B] >= 1
 *                (fp8 per-token K_nope scales: the row's own [S_row] floats, and
 *                the workspace needs mla_prefill_ragged_workspace_size_fp8(B, S_row))
 *   buffer_row_offsets  device uint32 [B+1], non-decreasing
 *   cache_offsets       device uint32 [B]; cache_offsets[b] + W_b <= L_b
 * A window outside a sequence's context sets MLA_DEVICE_STATUS_BAD_OFFSETS
 * and skips that sequence.  Workspace sizes and launches are those of
 * mla_prefill_ragged.
 */
mla_status_t mla_prefill_ragged_chunk(const mla_tensor_t* out, const mla_tensor_t* lse,
                                      const mla_tensor_t* q, const mla_tensor_t* k_nope,
                                      const mla_tensor_t* v, const mla_tensor_t* k_rope_pages,
                                      const mla_tensor_t* page_table, const uint32_t* row_offsets,
                                      const uint32_t* cache_lens, const uint32_t* buffer_row_offsets,
                                      const uint32_t* cache_offsets, float scale, mla_mask_t mask,
                                      uint32_t flags, void* workspace, size_t workspace_bytes,
                                      mla_stream_t stream);

#define MLA_CHUNK_ACCUMULATE 0x1u /* mla_prefill_ragged_chunk*: fold into out / lse */
/* fp8 inputs, a wider error envelope at a cost in speed: two quantities that
 * the fp8 path rounds once are carried as two terms each, a value and the
 * remainder of its rounding, and their products run once per term into the
 * same accumulator: P (the softmax weights, e4m3 for the e4m3 P.V) as
 * e4m3(P) + e4m3(P - e4m3(P)), about 7 significant bits instead of 3, and
 * the bf16 copy of K_rope (code * s_r / s_k) as bf16 + bf16, about 16 bits
 * instead of 8.  Measured on inputs whose values spread 1x / 2x / 3x the fp8
 * workload's: the largest error relative to the 6e-2 + 6e-2|ref| tolerance
 * drops from about 0.56 / 1.6 / 2.6 to 0.04 / 0.05 / 0.07.  Costs: a second
 * e4m3 P.V pass, four more bf16 UMMAs per score tile, a third ring chunk per
 * KV tile (the fp8 workload runs at about 0.59x the speed), and twice the
 * workspace for the converted K_rope
 * (mla_prefill_ragged_workspace_size_fp8 with 2 x pool_slots, or 2 x Sk with
 * per-token K_nope scales).  Accepted by mla_prefill_ragged_ex,
 * mla_prefill_ragged_chunked and the chunk calls; MLA_ERR_INVALID_ARG with
 * bf16 inputs.  No counterpart on the pages, which leave the fp8 kernel's
 * intermediate precisions open. */
#define MLA_FP8_PRECISE 0x2u

/*
 * Chunked execution of every buffer row of the plan in one call and one
 * attention launch (flare_mla_prefill: Args cache_row_offsets, cache_offsets;
 * generic_flare_mla_prefill_ragged_paged_plan: Args buffer_row_offsets,
 * cache_offsets, buffer_lengths; the rows' combination is the log-sum-exp
 * fold of mla_prefill_ragged_chunk with MLA_CHUNK_ACCUMULATE).
 *
 * The rows' K buffers are stacked: row r's buffer is K rows
 * [r * T, (r + 1) * T) of k_nope / v (T = buffer_token_size), laid out as the
 * plan describes (sequence b's keys of row r at row-local positions
 * buffer_row_offsets[r, b] .. [r, b+1]).  Under the plan's global packing a
 * sequence's windows in consecutive rows are then adjacent K rows, so one work
 * item covers a (sequence, head, query block) across all its rows and folds
 * them in its online softmax; the rows share one launch and one tail.  The
 * result is that of mla_prefill_ragged_chunk applied to rows 0..R-1 in order
 * with MLA_CHUNK_ACCUMULATE:
 *   out   the softmax over all the sequence's visible keys (the full-context
 *         result), bf16 [Tq, H, 128] (written)
 *   lse   float32 [Tq, H] (written) or NULL: ln sum_j exp(s_j) over the same
 *         keys
 *   buffer_row_offsets  device uint32 [max_rows, B+1], cache_offsets device
 *         uint32 [max_rows, B]: the plan's outputs for these lengths and T
 *   num_rows            device uint32 [1]: the plan's row count R; rows
 *         r >= min(R, max_rows) are not read
 *   k_nope, v           device [>= R * T, H, 128] (fp8 per-token K_nope
 *         scales: [rows] floats indexed by stacked K row)
 * flags: 0 or MLA_FP8_PRECISE.
 * Per sequence the kernel checks the first and the last row holding its keys
 * against the stacked layout (offset, context position and window end); a
 * sequence whose rows disagree, or that needs a row >= min(R, max_rows), is
 * skipped and sets MLA_DEVICE_STATUS_BAD_OFFSETS.  Everything else (K_rope,
 * page table, scales, workspace sizes, masks, errors) as mla_prefill_ragged;
 * the launches are those of mla_prefill_ragged.
 */
mla_status_t mla_prefill_ragged_chunked(const mla_tensor_t* out, const mla_tensor_t* lse,
                                        const mla_tensor_t* q, const mla_tensor_t* k_nope,
                                        const mla_tensor_t* v, const mla_tensor_t* k_rope_pages,
                                        const mla_tensor_t* page_table, const uint32_t* row_offsets,
                                        const uint32_t* cache_lens, const uint32_t* buffer_row_offsets,
                                        const uint32_t* cache_offsets, const uint32_t* num_rows,
                                        uint32_t max_rows, uint32_t buffer_token_size, float scale,
                                        mla_mask_t mask, uint32_t flags, void* workspace,
                                        size_t workspace_bytes, mla_stream_t stream);

/*
 * Combines the rows of a chunked execution (the pages give only the per-row
 * call; the combination is the standard log-sum-exp weighting).  For each
 * token t of sequence b and head h, over the rows r whose window holds keys of
 * b (buffer_row_offsets[r, b+1] > buffer_row_offsets[r, b]) and whose
 * lse_r = partial_lse[r, t, h] is finite:
 *   out[t, h, :] = sum_r e^(lse_r - m) partial_out[r, t, h, :] / sum_r e^(lse_r - m),
 *   m = max_r lse_r;  0 when no row qualifies.
 *   out                 device bf16 [Tq, H, 128] (written for tokens
 *                       row_offsets[0] .. row_offsets[B]-1 only), 16-byte
 *                       aligned rows
 *   partial_out         device bf16 [R, Tq, H, 128], as written by
 *                       mla_prefill_ragged_chunk for rows 0..R-1
 *   partial_lse         device float32 [R, Tq, H]
 *   row_offsets         device uint32 [B+1] (the attention calls' Q offsets)
 *   buffer_row_offsets  device uint32, row r at buffer_row_offsets + r * (B+1)
 *                       (the plan's output), rows 0..R-1 read
 *   batch               B >= 1
 * One launch, no host synchronisation.
 */
mla_status_t mla_prefill_merge(const mla_tensor_t* out, const mla_tensor_t* partial_out,
                               const mla_tensor_t* partial_lse, const uint32_t* row_offsets,
                               const uint32_t* buffer_row_offsets, uint32_t batch,
                               mla_stream_t stream);

/*
 * mla_prefill_ragged_chunk with a contiguous K_rope for the row (the
 * flare_mla_prefill overload with a plain k_rope tensor): k_rope is
 * [S_row, 64], row t holding the rope dims of the row's K buffer position t
 * (for example the last 64 columns of rows gathered by mla_gather_rows), so no
 * page table is read.  batch gives B; fp8 K_rope takes one scale per row and
 * the workspace then needs mla_prefill_ragged_workspace_size_fp8(B, S_row).
 * Everything else as mla_prefill_ragged_chunk.
 */
mla_status_t mla_prefill_ragged_chunk_contiguous(
    const mla_tensor_t* out, const mla_tensor_t* lse, const mla_tensor_t* q, const mla_tensor_t* k_nope,
    const mla_tensor_t* v, const mla_tensor_t* k_rope, const uint32_t* row_offsets,
    const uint32_t* cache_lens, const uint32_t* buffer_row_offsets, const uint32_t* cache_offsets,
    uint32_t batch, float scale, mla_mask_t mask, uint32_t flags, void* workspace,
    size_t workspace_bytes, mla_stream_t stream);

/*
 * Gather of one buffer row out of a paged cache into a contiguous buffer
 * (generic_flare_mla_prefill_ragged_paged_plan summary: the plan exists so the
 * prefill kernel "can gather K/V entries into a contiguous buffer"; Args:
 * buffer_row_offsets, cache_offsets).  For every sequence b and
 * 0 <= i < buffer_row_offsets[b+1] - buffer_row_offsets[b], with context
 * position a = cache_offsets[b] + i:
 *   dst[buffer_row_offsets[b] + i, :] = cache[page_table[b, a / P], a % P, :]
 *   dst          device [rows, W] (written for positions < min(rows,
 *                buffer_row_offsets[B]) only); same dtype as cache
 *   cache        device [num_pages, P, W], bf16 or fp8 (codes copied as
 *                bytes), W * element size a multiple of 16 bytes; e.g. a
 *                DeepSeek-V3 latent cache row [c_kv 512 | k_rope 64]
 *   page_table   device uint32 [B, max_pages]
 *   buffer_row_offsets, cache_offsets  one row of the plan ([B+1], [B])
 *   status       device uint32 or NULL: an out-of-range page id or
 *                page-table column skips that row chunk and ORs
 *                MLA_DEVICE_STATUS_BAD_PAGE / _BAD_COLUMN into *status
 * One launch, HBM-bound; no host synchronisation.
 */
mla_status_t mla_gather_rows(const mla_tensor_t* dst, const mla_tensor_t* cache,
                             const mla_tensor_t* page_table, const uint32_t* buffer_row_offsets,
                             const uint32_t* cache_offsets, uint32_t* status, mla_stream_t stream);

/*
 * Up-projection of latent rows (the step between the gather and the
 * attention when the cache holds the compressed latent row rather than K_nope
 * and V: mla_prefill_v2_ragged Args: v, "the nope segment of the latent
 * cache"; the weights are the caller's):
 *   out[t, n] = sum_k latent[t, k] * weight[n, k]
 *   out     device bf16 [rows, N] (e.g. K_nope [rows, H, 128] viewed as
 *           [rows, H * 128]), row stride a multiple of 16 bytes
 *   latent  device bf16 [rows, K] (row stride may exceed K: the c_kv
 *           columns of gathered latent rows); 1 <= K <= 512 (the latent
 *           width, kv_lora_rank: a 128-row block of it stays on chip)
 *   weight  device bf16 [N, K] (nn.Linear layout)
 *   status  device uint32 or NULL: MLA_DEVICE_STATUS_TIMEOUT is ORed in if a
 *           pipeline wait of the kernel gives up
 * Rows of every operand must start 16-byte aligned.  One launch of this
 * library's tensor-core GEMM (fp32 accumulation in tensor memory, bf16
 * output, 128 x 128 output tiles); no library GEMM, no workspace.
 */
mla_status_t mla_up_project(const mla_tensor_t* out, const mla_tensor_t* latent,
                            const mla_tensor_t* weight, uint32_t* status, mla_stream_t stream);

/*
 * Gather and up-projection of one buffer row in one launch
 * (generic_flare_mla_prefill_ragged_paged_plan summary: the plan exists so the
 * prefill kernel can gather K/V entries into a contiguous buffer; Args:
 * buffer_row_offsets, cache_offsets; mla_prefill_v2_ragged Args: v, the nope
 * segment of the latent cache).  For every sequence b and buffer position
 * t = buffer_row_offsets[b] + i < buffer_row_offsets[b+1], with context
 * position a = cache_offsets[b] + i and cache row
 * c = cache[page_table[b, a / P], a % P, 0:kv_lora_rank]:
 *   k_out[t, n] = sum_k c[k] * w_uk[n, k]
 *   v_out[t, n] = sum_k c[k] * w_uv[n, k]
 * The cache rows are fetched through the page table straight into the GEMM's
 * operand tiles (TMA row gathers); no contiguous copy of the row is made.
 *   k_out, v_out  device bf16 [rows, N] (e.g. [rows, H, 128] viewed as
 *                 [rows, H * 128]); positions t >= buffer_row_offsets[B]
 *                 (and positions whose page id or page-table column is out of
 *                 range) receive unspecified values.  v_out and w_uv may both
 *                 be NULL for a single projection.
 *   cache         device bf16 [num_pages, P, W], W >= kv_lora_rank, pages
 *                 contiguous (page stride = P x token stride), token stride a
 *                 multiple of 16 bytes; e.g. DeepSeek-V3's latent row
 *                 [c_kv 512 | k_rope 64]
 *   w_uk, w_uv    device bf16 [N, kv_lora_rank] (nn.Linear layout)
 *   page_table    device uint32 [B, max_pages]
 *   buffer_row_offsets, cache_offsets  one row of the plan ([B+1], [B])
 *   kv_lora_rank  K of the projection, a multiple of 8 and at most 512 (512
 *                 for DeepSeek-V3)
 *   status        device uint32 or NULL: an out-of-range page id or page-table
 *                 column ORs MLA_DEVICE_STATUS_BAD_PAGE / _BAD_COLUMN, a
 *                 pipeline wait that gives up MLA_DEVICE_STATUS_TIMEOUT
 * One launch, no host synchronisation.  The row's K_rope needs no copy
 * either: mla_prefill_ragged_chunk reads it from the same cache as a paged
 * K_rope whose token stride is the latent row.
 */
mla_status_t mla_gather_up_project(const mla_tensor_t* k_out, const mla_tensor_t* v_out,
                                   const mla_tensor_t* cache, const mla_tensor_t* w_uk,
                                   const mla_tensor_t* w_uv, const mla_tensor_t* page_table,
                                   const uint32_t* buffer_row_offsets, const uint32_t* cache_offsets,
                                   uint32_t kv_lora_rank, uint32_t* status, mla_stream_t stream);

/* Device status bits written into the workspace's first uint32. */
#define MLA_DEVICE_STATUS_BAD_PAGE 0x1u    /* page id >= num_pages */
#define MLA_DEVICE_STATUS_BAD_COLUMN 0x2u  /* context needs more pages than max_pages */
#define MLA_DEVICE_STATUS_BAD_OFFSETS 0x4u /* row offsets decrease or exceed Tq/Sk */
#define MLA_DEVICE_STATUS_TIMEOUT 0x8u     /* a pipeline wait gave up (kernel bug) */

/* Synchronising helper: waits for `stream`, then copies the status word of
 * `workspace` to *status_out. */
mla_status_t mla_read_device_status(const void* workspace, uint32_t* status_out,
                                    mla_stream_t stream);

/*
 * Test hook for the timeout path (no counterpart on the pages).  While
 * enabled (process-wide), every attention launch leaves the first K group of
 * each CTA's first work item unloaded: the UMMA issuers' bounded wait for it
 * runs out (after a few seconds), the kernel winds down every role, waits for
 * its copies in flight, frees tensor memory and sets
 * MLA_DEVICE_STATUS_TIMEOUT; the output is then incomplete.  The CUDA context
 * stays usable.  Never enable it outside tests.
 */
mla_status_t mla_test_inject_stall(uint32_t enable);

/*
 * Test hook for the pipeline's ordering (no counterpart on the pages).  While
 * nonzero (process-wide), the softmax warps of the second query tile of every
 * attention work item wait `nanoseconds` (at most 100000) before loading each
 * score tile, so that tile runs far behind the first one; results must be
 * bit-identical to an undelayed launch, only slower.  0 turns it off.  Never
 * set it outside tests.
 */
mla_status_t mla_test_delay_softmax(uint32_t nanoseconds);

/* Text for the last error returned to the calling thread (never NULL). */
const char* mla_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PREFILL_H_ */
