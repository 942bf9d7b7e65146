/*
 * lora_sgmv.h -- C ABI of the GB300 (sm_103a) segmented gather matrix-vector
 * (SGMV) LoRA library.
 *
 * The library adds, for every token row t routed to an adapter slot s,
 *     y_t += B_s . (A_s . x_t)
 * to a projection's base output y ("vLLM LoRA 实现深度解析", section 1: the
 * forward pass h = W0 x + (alpha/r) B A x with the scale folded into B;
 * section 6: output += lora_b_stacked[slot] . lora_a_stacked[slot] . x).
 *
 * Routing follows the triple of the "max.pipelines.lora.LoRAManagerV3" API
 * page (get_lora_graph_inputs): lora_ids and grouped_offsets live on the
 * device, end on the host.  Rows at or past `end` (base requests, which the
 * sort puts last) are never read or written.  Within [0, end) every kernel
 * writes only the rows of the group it is working on; the tensor-core
 * kernels for long groups load whole 128-row boxes of x and y, so they may
 * READ rows of neighbouring groups (never rows at or past `end`: their
 * tensor maps end there).
 *
 * Conventions for every entry point:
 *   - Every buffer is owned by the caller.  No entry point allocates or frees
 *     device memory, and none keeps a pointer after it returns.
 *   - Device work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and is asynchronous; host arrays passed in may be reused
 *     as soon as the call returns.
 *   - Arguments are validated on the host before anything is launched; on any
 *     error nothing is launched and the error code is returned.
 *   - The device-side routing arrays are checked by the kernels themselves
 *     (slot range, monotone offsets, first offset 0, last offset == end).  A
 *     violation makes that launch skip ALL of its work, leaves y untouched and
 *     records a flag that lora_get_device_status() returns.
 *   - A CUDA launch failure returns LORA_ERR_CUDA.
 *   - Entry points are thread-safe as far as CUDA itself is; two calls that
 *     write the same y concurrently on different streams race.
 */
#ifndef LORA_SGMV_H
#define LORA_SGMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, without pulling in the CUDA headers. */
typedef struct CUstream_st* lora_stream_t;

typedef enum {
  LORA_OK = 0,
  LORA_ERR_NULL = 1,          /* a required pointer is NULL */
  LORA_ERR_SHAPE = 2,         /* a count, size or stride is out of range */
  LORA_ERR_RANK = 3,          /* adapter rank r > max_lora_rank, or r < 0 */
  LORA_ERR_SLOT_RANGE = 4,    /* a slot id < -1 (requests) or >= max_num_loras */
  LORA_ERR_ROUTING = 5,       /* routing triple inconsistent (num_groups, end) */
  LORA_ERR_DTYPE = 6,         /* unknown storage type */
  LORA_ERR_ALIGN = 7,         /* pointer/stride alignment required by the call */
  LORA_ERR_WORKSPACE = 8,     /* workspace NULL or smaller than lora_workspace_bytes() */
  LORA_ERR_CUDA = 9,          /* a CUDA runtime call or kernel launch failed */
  LORA_ERR_TOO_MANY_GROUPS = 10 /* num_groups > max_num_loras ("No free lora slots") */
} lora_status_t;

/* Storage type of x, y and the A/B stacks of one problem. */
typedef enum { LORA_DTYPE_F32 = 0, LORA_DTYPE_BF16 = 1 } lora_dtype_t;

/* Flags of the device status word (lora_get_device_status). */
#define LORA_DEV_BAD_SLOT 1u     /* lora_ids[g] outside [0, max_num_loras) */
#define LORA_DEV_BAD_OFFSETS 2u  /* grouped_offsets[0] != 0 or a decreasing offset */
#define LORA_DEV_BAD_END 4u      /* grouped_offsets[num_groups] != end */
#define LORA_DEV_TIMEOUT 8u      /* a kernel gave up (after ~1 s) waiting for its own copies */
#define LORA_DEV_BAD_ROW 16u     /* a token_rows entry outside [0, num_tokens) */

#define LORA_MAX_SLICES 3

/*
 * One projection slice of a problem.  A and B are the per-slot stacks of the
 * "vLLM LoRA 实现深度解析" page, section 9 (memory layout):
 *   A: slot s block at A + s*A_slot_stride, shape [max_lora_rank, in_dim],
 *      row-major, row stride in_dim (elements).
 *   B: slot s block at B + s*B_slot_stride, shape [out_dim, max_lora_rank],
 *      row-major, row stride max_lora_rank.
 *   y: row t of this slice's output at y + t*y_row_stride, out_dim elements.
 * Strides are in elements.  Fused q/k/v ("MAX max.pipelines.lora 模块解析",
 * load pipeline, QKV fusion: A concatenated on the rank dimension, B on the
 * output dimension) is pure pointer arithmetic on one fused stack:
 *   slice j: A = A_fused + j*R*in_dim, A_slot_stride = n*R*in_dim,
 *            B = B_fused + off_j*R,   B_slot_stride = O*R,
 *            y = y_fused + off_j,      y_row_stride  = O,
 * so slice j's B multiplies only rank columns [jR, (j+1)R) of the
 * intermediate.  Per-projection (unfused) q/k/v is three slices with their
 * own stacks.
 */
typedef struct {
  const void* A;
  int64_t A_slot_stride;
  const void* B;
  int64_t B_slot_stride;
  int32_t out_dim;
  void* y;
  int64_t y_row_stride;
  /* Optional LoRA bias ("MAX max.pipelines.lora 模块解析", LoRA types: BIAS, the
   * bias attached to B; "vLLM LoRA 实现深度解析" section 8, --enable-lora-bias):
   * slot s's vector of out_dim values at bias + s*bias_slot_stride, storage
   * type, added unscaled to every routed row (inside the one rounding).
   * NULL: no bias. */
  const void* bias;
  int64_t bias_slot_stride;
} lora_slice_t;

/*
 * One LoRA problem: a projection input x[num_tokens, in_dim] (row stride
 * x_row_stride elements, rows in sorted-batch order) and 1..3 slices sharing
 * it.  max_num_loras (S) and max_lora_rank (R) are the stack sizes.
 */
typedef struct {
  lora_dtype_t dtype;
  int32_t num_tokens;
  int32_t in_dim;
  int32_t max_num_loras;
  int32_t max_lora_rank;
  const void* x;
  int64_t x_row_stride;
  int32_t num_slices;
  lora_slice_t slices[LORA_MAX_SLICES];
  /* Optional DEVICE int32 [max_num_loras]: the true rank r_s of each slot
   * (0..max_lora_rank), a hint that lets the kernels skip the zero padding:
   * rank columns from ceil16(r_s) on (A rows, B columns) are then never read
   * and contribute nothing; columns [r_s, ceil16(r_s)) must still be zero, as
   * lora_set_slot writes them.  NULL: every slot uses max_lora_rank. */
  const int32_t* slot_ranks;
} lora_problem_t;

/*
 * The routing triple ("max.pipelines.lora.LoRAManagerV3",
 * get_lora_graph_inputs): lora_ids[num_groups] and
 * grouped_offsets[num_groups + 1] are DEVICE int32 arrays; num_groups and end
 * are host values.  Group g covers sorted-batch rows
 * [grouped_offsets[g], grouped_offsets[g+1]) and uses slot lora_ids[g].
 * num_groups == 0 or end == 0 is a valid no-op.  num_groups > max_num_loras
 * returns LORA_ERR_TOO_MANY_GROUPS (a batch needs a slot per group: "No free
 * lora slots", "vLLM LoRA 实现深度解析" section 5.3); other inconsistent host
 * values (end < 0, end > num_tokens, end > 0 with no group) LORA_ERR_ROUTING.
 * The same slot may appear in two groups (each group uses its slot); the
 * routing builder never produces that.
 */
typedef struct {
  const int32_t* lora_ids;
  const int32_t* grouped_offsets;
  int32_t num_groups;
  int32_t end;
  /* Optional, DEVICE int32 [end]: token_rows[i] is the row of x and y that
   * holds the i-th routed token of the sorted order, for batches that are not
   * physically sorted (the per-token slot mapping of "vLLM LoRA 实现深度解析"
   * section 6, whose kernels walk tokens sorted by adapter).  NULL: row i is
   * row i (the sorted batch of the MAX page).  Entries must be distinct and in
   * [0, num_tokens); an entry outside that range makes the launch skip the
   * tiles containing it and raises LORA_DEV_BAD_ROW.  Long gathered groups
   * run on the tcgen05 kernels too (x rows gathered with 16-byte copies, y
   * rows read and written in place); lora_base_gemm_apply refuses token_rows. */
  const int32_t* token_rows;
  /* Optional HOST int32 [num_groups + 1]: the same values as
   * grouped_offsets, read by the call itself (not by the kernels).  With it
   * lora_sgmv_apply picks the kernels per group: groups of at least
   * LORA_TC_MIN_ROWS routed rows on the tensor-core (tcgen05) kernels, the
   * others on the mma.sync kernels, both in the same call.  NULL: one choice
   * per call, from the average group length (end / num_groups).  When given
   * it is checked on the host (entry 0 is 0, entries non-decreasing, entry
   * num_groups equals end; else LORA_ERR_ROUTING). */
  const int32_t* host_grouped_offsets;
  /* Optional HOST int32 [num_groups]: the same values as lora_ids; used only
   * together with host_grouped_offsets (alone: LORA_ERR_NULL), each entry in
   * [0, max_num_loras) (else LORA_ERR_SLOT_RANGE).  With both host copies,
   * lora_sgmv_apply gives its mma.sync shrink a table of its tiles (up to
   * 128 tiles of 64 rows) as a launch parameter: each CTA knows its slot and
   * rows without reading the device triple.  The expand still reads the
   * device triple and checks it against a 64-bit digest of the host copies
   * (SplitMix64 terms per group, summed): a difference raises
   * LORA_DEV_BAD_OFFSETS and the expand skips its work, leaving y as it was
   * (a difference that leaves the digest unchanged goes unseen; for unequal
   * triples that is a chance of about 2^-64).  A CUDA graph that captures the
   * call replays the captured copies: recapture after changing the triple. */
  const int32_t* host_lora_ids;
} lora_routing_t;

/* Routed rows from which a group counts as long (tcgen05 tiles) when the
 * kernels are picked per group. */
#define LORA_TC_MIN_ROWS 64

/*
 * lora_build_routing -- HOST ONLY.  Sort + group ("max.pipelines.lora.
 * LoRAManagerV3", sort_lora_batch and get_lora_graph_inputs).
 *
 * Input: num_requests requests in arrival order, request i on slot
 * req_slot[i] (-1 = base model, else 0..max_num_loras-1) with
 * req_num_tokens[i] >= 0 token rows.
 * Output (caller-allocated host arrays):
 *   perm[num_requests]               sorted order: perm[i] is the arrival index
 *                                    of the i-th request of the sorted batch.
 *                                    Ascending slot, stable, base last.
 *   lora_ids[max_num_loras]          slot of each group (first *num_groups used)
 *   grouped_offsets[max_num_loras+1] first row of each group; entry
 *                                    [*num_groups] equals *end
 *   *num_groups, *end (LoRA-routed rows), *total_tokens (all rows).
 * Consecutive same-slot requests form one group; the walk stops at the first
 * base request.  A zero-token request still opens its slot's group.
 * Errors: LORA_ERR_SHAPE (num_requests < 0, max_num_loras < 1, a negative
 * token count, total rows > INT32_MAX), LORA_ERR_SLOT_RANGE, LORA_ERR_NULL.
 * Outputs are unspecified on error.
 */
lora_status_t lora_build_routing(int32_t num_requests, const int32_t* req_slot,
                                 const int32_t* req_num_tokens, int32_t max_num_loras,
                                 int32_t* perm, int32_t* lora_ids, int32_t* grouped_offsets,
                                 int32_t* num_groups, int32_t* end, int32_t* total_tokens);

/*
 * lora_build_token_rows -- HOST ONLY.  For a batch whose rows are in ARRIVAL
 * order (request i owns rows [start_i, start_i + req_num_tokens[i]), start
 * the running sum in arrival order), write the row of every routed token in
 * the sorted order produced by lora_build_routing: token_rows[0, end) lists
 * the rows of request perm[0], then perm[1], ..., stopping after `end` rows.
 * Pass it (uploaded) as lora_routing_t.token_rows.
 * Errors: LORA_ERR_NULL, LORA_ERR_SHAPE (negative counts, a perm entry out of
 * range, end larger than the rows of the batch).
 */
lora_status_t lora_build_token_rows(int32_t num_requests, const int32_t* req_num_tokens,
                                    const int32_t* perm, int32_t end, int32_t* token_rows);

/*
 * lora_set_slot -- load-time preparation of one adapter slot for one slice
 * ("MAX max.pipelines.lora 模块解析", load pipeline: scale pre-multiplied into
 * B, rank padding, dtype unification; "vLLM LoRA 实现深度解析" section 1,
 * scale alpha/r or alpha/sqrt(r) with rsLoRA, and section 5.3 set_lora).
 *
 * Writes slot `slot` of slice `slice` of the stacks described by `problem`
 * (the stacks must be writable device memory):
 *   A[slot, k, i] = A_raw[k, i]                        for k < r, else 0
 *   B[slot, o, k] = rne(fp32(B_raw[o, k]) * scale)     for k < r, else 0
 * where scale = fp32(lora_alpha / r), or fp32(lora_alpha / sqrt(r)) when
 * use_rslora != 0, computed in double on the host; the product is formed in
 * fp32 and rounded once (round to nearest even) to problem->dtype.
 * A_raw [r, in_dim] and B_raw [out_dim, r] are contiguous DEVICE arrays of
 * raw_dtype (fp32 or bf16).  r == 0 zeroes the slot (A_raw/B_raw may be NULL).
 * Errors: LORA_ERR_RANK (r < 0 or r > max_lora_rank), LORA_ERR_SLOT_RANGE,
 * LORA_ERR_SHAPE (slice out of range, bad dims), LORA_ERR_NULL, LORA_ERR_DTYPE.
 */
lora_status_t lora_set_slot(const lora_problem_t* problem, int32_t slice, int32_t slot, int32_t r,
                            double lora_alpha, int32_t use_rslora, const void* A_raw,
                            const void* B_raw, lora_dtype_t raw_dtype, lora_stream_t stream);

/*
 * lora_set_slot_bias -- load-time preparation of slot `slot`'s bias for slice
 * `slice`: bias[slot, o] = cast(bias_raw[o]) (round to nearest even), or zero
 * when bias_raw is NULL.  bias_raw is a contiguous DEVICE array of out_dim
 * values of raw_dtype.  The slice's bias pointer must be set.
 * Errors: LORA_ERR_NULL (no bias stack), LORA_ERR_SLOT_RANGE, LORA_ERR_SHAPE,
 * LORA_ERR_DTYPE.
 */
lora_status_t lora_set_slot_bias(const lora_problem_t* problem, int32_t slice, int32_t slot,
                                 const void* bias_raw, lora_dtype_t raw_dtype, lora_stream_t stream);

/*
 * lora_shrink -- u[t, j*R + k] = sum_i A_j[lora_ids[g], k, i] * x[t, i] for
 * every routed row t < end (group g), slice j, k < R.  u is a DEVICE fp32
 * array [end, num_slices*R] (row stride num_slices*R), fully overwritten.
 * Products of the stored values are exact; sums are fp32.
 */
lora_status_t lora_shrink(const lora_problem_t* problem, const lora_routing_t* routing, float* u,
                          lora_stream_t stream);

/*
 * lora_expand -- boundary-aware expand: y_j[t, o] = rn(y_j[t, o] +
 * bias_j[s, o] + sum_k B_j[s, o, k] * u[t, j*R + k]) with s = lora_ids[g]
 * (bias only when the slice has one) for routed rows t < end only,
 * with one rounding to the storage type.  u as produced by lora_shrink.
 * Accumulation is fp32.  On the bf16 tensor-core path u enters the product as
 * two bf16 terms (u = hi + lo, 16 significant bits, the split is exact);
 * elsewhere it enters as fp32.
 */
lora_status_t lora_expand(const lora_problem_t* problem, const lora_routing_t* routing,
                          const float* u, lora_stream_t stream);

/*
 * Bytes of device workspace lora_sgmv_apply needs for `end` routed rows: for
 * max_lora_rank 64 or 128 the packed intermediate of the tensor-core path
 * ((max_num_loras + end / 128) tiles x n*R x 512 bytes), then room for the
 * fp32 intermediate (up to 16 partial planes of end x n*R); both are live
 * when the kernels are picked per group.  Depends on shapes only.
 */
size_t lora_workspace_bytes(const lora_problem_t* problem, int32_t end);

/*
 * lora_sgmv_apply -- shrink then expand in one call; the intermediate lives in
 * `workspace` (DEVICE, >= lora_workspace_bytes(problem, end) bytes, 16-byte
 * aligned, contents on entry ignored): fp32 partial planes, or, on the
 * tensor-core path (bf16, rank 64 or 128, long groups), u already split into
 * bf16 hi + lo terms and laid out as the expand's operand per 128-row tile.
 * The expand is launched as a programmatic dependent of the shrink, so its
 * weight and y loads overlap the shrink.  With the routing's host copy of
 * the offsets (host_grouped_offsets), a batch mixing long and short groups
 * runs both kernel families in the one call, each on its own groups.  Two
 * calls whose kernels may overlap on the GPU need two workspaces.
 */
lora_status_t lora_sgmv_apply(const lora_problem_t* problem, const lora_routing_t* routing,
                              void* workspace, size_t workspace_bytes, lora_stream_t stream);

/*
 * lora_sgmv_apply_noalloc -- lora_sgmv_apply for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point.
 *
 * Some callers cannot call cudaMalloc: plug-ins living inside a host
 * framework that owns every device allocation (and gives them none), or
 * latency-critical loops where an allocation could stall or fail.  This call
 * takes no workspace argument and allocates nothing; the fp32 intermediate
 * lives in a fixed array of LORA_NOALLOC_MAX_WORKSPACE_BYTES compiled into the
 * library (every GPU that loads the library holds it until the process exits).
 *
 * Same problem, routing, results and errors as lora_sgmv_apply, plus:
 *   - LORA_ERR_WORKSPACE if the fp32 intermediate, end x n*R x 4 bytes
 *     rounded up to 256, exceeds LORA_NOALLOC_MAX_WORKSPACE_BYTES (use
 *     lora_sgmv_apply with your own workspace for such batches).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; LORA_ERR_CUDA if the lookup fails.
 *     Make that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its own
 *     intermediate in it.  Nothing has to start at zero (each call writes
 *     every value it later reads), but calls whose GPU work overlaps -- on
 *     different streams, or from different threads -- race on the array.
 *     Serialize them (one stream, or events).
 */
#define LORA_NOALLOC_MAX_WORKSPACE_BYTES (16u * 1024u * 1024u)
lora_status_t lora_sgmv_apply_noalloc(const lora_problem_t* problem, const lora_routing_t* routing,
                                      lora_stream_t stream);

/* Base projection weight of one slice: W0 [out_dim, in_dim] in the
 * problem's storage type, row o at W0 + o * row_stride (elements). */
typedef struct {
  const void* W0;
  int64_t row_stride;
} lora_base_weight_t;

/*
 * lora_base_gemm_apply -- the LoRA delta fused into the base projection
 * ("vLLM LoRA 实现深度解析" section 1: h = W0 x + (alpha/r) B A x, the scale
 * folded into B):
 *   y_j[t, o] = rn( sum_i W0_j[o, i] x[t, i]
 *                   + [t < end] (bias_j[s, o] + sum_k B_j[s, o, k] u[t, j*R + k]) )
 * for EVERY row t < num_tokens and every slice j (s: the slot of t's group;
 * base rows get the base product alone), with one rounding to the storage
 * type.  y is written, never read: the delta joins the base product in the
 * accumulator instead of a read-modify-write of y.  base[num_slices] gives
 * each slice's W0 (DEVICE).  The shrink writes u into `workspace` as for
 * lora_sgmv_apply (same size; NULL allowed when
 * num_groups or end is 0).  Rows must be in sorted order: token_rows is
 * refused (LORA_ERR_SHAPE).
 * Kernels: bf16 fast-path shapes (16-byte aligned W0, row stride a multiple
 * of 8) run a tcgen05 GEMM whose K loop ends with the delta as extra K
 * steps (u = hi + lo as bf16 terms against the slot's B block, per group
 * overlapping a 128-row tile); other shapes a generic kernel.
 * Errors: as lora_sgmv_apply, plus LORA_ERR_NULL (base or a W0 missing),
 * LORA_ERR_SHAPE (a row stride below in_dim, token_rows given).
 */
lora_status_t lora_base_gemm_apply(const lora_problem_t* problem, const lora_routing_t* routing,
                                   const lora_base_weight_t* base, void* workspace, size_t workspace_bytes,
                                   lora_stream_t stream);

/*
 * lora_get_device_status -- reads and clears, in one atomic exchange ordered
 * after the work already on `stream`, the device status word of the current
 * device (an OR of LORA_DEV_* flags from every launch since the last read,
 * on any stream), then synchronizes `stream` and returns the flags.  A flag
 * raised by a kernel on another stream is never lost: it is either returned
 * by this call or kept for the next.  Returns LORA_ERR_CUDA if the exchange,
 * the copy or the synchronization fails.
 */
lora_status_t lora_get_device_status(lora_stream_t stream, uint32_t* flags);

/*
 * Kernel families (bits of lora_last_call_path).  The pages have no
 * counterpart; this is an introspection aid for tests and profiling.
 */
#define LORA_PATH_GENERIC_SHRINK 0x1u  /* one warp per u element (fp32, odd shapes) */
#define LORA_PATH_GENERIC_EXPAND 0x2u  /* one thread per y element */
#define LORA_PATH_MMA_SHRINK 0x4u      /* mma.sync shrink (short groups) */
#define LORA_PATH_MMA_EXPAND 0x8u      /* mma.sync expand (short groups) */
#define LORA_PATH_TC_SHRINK 0x10u      /* tcgen05 + TMA shrink (long groups) */
#define LORA_PATH_TC_EXPAND 0x20u      /* persistent tcgen05 + TMA expand (long groups) */
#define LORA_PATH_PREP 0x80u           /* load-time slot / bias preparation */
#define LORA_PATH_BASE_GEMM 0x100u     /* base projection GEMM with the delta as K tail */

/*
 * lora_last_call_path -- the OR of LORA_PATH_* bits of the kernels launched
 * by the most recent entry-point call made on the calling host thread (0 if
 * it launched nothing: a no-op, or an error before any launch), and, when
 * num_launches is not NULL, how many kernels that call launched.  Host only;
 * reads thread-local state, no CUDA call.
 */
uint32_t lora_last_call_path(uint32_t* num_launches);

/*
 * lora_selftest_wait_timeout -- exercises the failure path of the pipelined
 * kernels without faulting the GPU (no counterpart on the pages).  One thread
 * waits on a fresh shared-memory barrier that nothing completes, gives up
 * after `polls` polls of mbarrier.try_wait (bounded), sets LORA_DEV_TIMEOUT
 * in the device status word and exits; the context stays usable.  Read the
 * flag with lora_get_device_status.  Returns LORA_ERR_CUDA if the launch
 * fails.
 */
lora_status_t lora_selftest_wait_timeout(uint32_t polls, lora_stream_t stream);

/* Static, human-readable name of a status code. */
const char* lora_status_string(lora_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* LORA_SGMV_H */
