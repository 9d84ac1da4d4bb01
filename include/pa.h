/*
 * pa.h -- C ABI of the GB300 paged-KV step library (libpa.so).
 *
 * One continuous-batching engine step, data plane only, as traced on the
 * page "vLLM 推理流程分析" (§5.1.2 _prepare_inputs, §6.1-6.3 attention dispatch,
 * FlashAttention path and KV-cache write):
 *
 *   pa_plan          host: validate the step's metadata and build the work
 *                    decomposition every layer of the step reuses;
 *   pa_slot_mapping  device: slot of every scheduled token;
 *   pa_write_kv      device: scatter the new K/V rows into the paged caches;
 *   pa_attention     device: causal GQA attention of every scheduled query
 *                    token over its request's context, read through the block
 *                    table; decode rows, chunked-prefill/extend rows, prefix
 *                    hits and the shared-prefix (cascade) route;
 *   pa_zero_blocks   device: clear newly allocated cache blocks (§4, §5.1.1);
 *   pa_attention_with_kv_update
 *                    device: the cache write and attention as one call (§6.1,
 *                    fused dispatch).
 *
 * Fixed-shape plans (pa_plan_fixed) make the attention launches of a step a
 * function of capacities only, so that they can be captured once in a CUDA
 * graph and replayed for later steps: pa_upload_metadata then replay (or
 * pa_attention_launch).  pa_graph_create / pa_graph_step do that inside the
 * library: two captured graphs of one fixed shape, one C call per step,
 * optionally with the step's host inputs and output copied inside the graph.
 *
 * Data types: every tensor element is IEEE bfloat16, passed as raw 16-bit
 * patterns; metadata is int32 except slot_mapping (int64).  All layouts are
 * dense row-major:
 *   q, out              [T][Hq][D]
 *   key, value (new)    [T][Hkv][D]
 *   key_cache,
 *   value_cache         [num_blocks][block_size][Hkv][D]     (§6.2 layout)
 *   block_table         [num_reqs][max_blocks_per_req]
 * T is the number of scheduled tokens of the step (query_start_loc[num_reqs]).
 * Query head h reads kv head h / (Hq / Hkv).  Query token i of request r is
 * at absolute position num_computed_tokens[r] + i and attends to keys
 * 0..position (bottom-right causal alignment).
 *
 * Supported: head_dim 64 or 128 (128 only with FP8 caches), block_size 16,
 * Hq % Hkv == 0 with the group size G = Hq/Hkv at most 128 (groups of more
 * than 16 query heads run every row on the tensor-core tiles), num_blocks *
 * 16 < 2^31.  Other shapes return PA_ERR_UNSUPPORTED.
 *
 * Ownership: the caller allocates and owns every device buffer (q, caches,
 * block table, out, slot mapping, workspace), except the workspace, slot
 * buffer, metadata images and streams a pa_graph_t allocates for itself.  A
 * plan is host memory owned by the library from pa_plan until pa_plan_destroy.  Device entry points only
 * enqueue work on the given stream (a cudaStream_t; NULL = the legacy default
 * stream) and never synchronise, except pa_check_device_errors.  Errors come
 * back as a status; nothing aborts, traps or throws across the ABI.
 *
 * Library-owned host resources: (1) pinned staging buffers for the metadata
 * upload of pa_attention / pa_upload_metadata, kept in a pool; a buffer is
 * reused once its last copy has run, and the pool calls cudaMallocHost only
 * when no such buffer is free (the first calls of a process, and whenever more
 * plans' uploads are in flight than the pool holds; it keeps up to 32 free
 * buffers).  The capturable path (pa_plan_copy_metadata +
 * pa_upload_metadata_from, and pa_graph_*) never uses the pool.  (2) A
 * second stream with two events per host thread and device, created the
 * first time that thread prepares a plan whose tensor-core tiles run beside
 * the decode kernel (pa_plan_info.side_by_side) and kept for the thread's
 * lifetime.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARGUMENT = 1,   /* malformed metadata or pointer; nothing enqueued */
    PA_ERR_UNSUPPORTED = 2,        /* well-formed but outside the supported shapes    */
    PA_ERR_CUDA = 3,               /* a CUDA runtime call failed                      */
    PA_ERR_DEVICE_CHECK = 4,       /* a kernel recorded an error in the error word    */
    PA_ERR_WORKSPACE_TOO_SMALL = 5,/* workspace smaller than pa_plan reported         */
    PA_ERR_CAPACITY = 6            /* the step exceeds a fixed-shape plan's capacity  */
} pa_status;

/* Bits a kernel may set in the device error word (see pa_check_device_errors). */
#define PA_DEVERR_SLOT_RANGE   0x1  /* pa_write_kv: slot >= number of cache slots      */
#define PA_DEVERR_BLOCK_RANGE  0x2  /* block id outside [0, num_blocks)                */
#define PA_DEVERR_TIMEOUT      0x4  /* a bounded wait inside a kernel gave up          */

typedef struct pa_plan_s pa_plan_t;

/*
 * The step's metadata, as CommonAttentionMetadata carries it ("vLLM 推理流程分析"
 * §5.1.3) plus the scheduler's common-prefix count (§4.4).  All arrays are
 * HOST memory, read during pa_plan only.
 */
typedef struct {
    int32_t num_reqs;              /* R >= 0                                          */
    int32_t num_heads_q;           /* Hq                                              */
    int32_t num_heads_kv;          /* Hkv                                             */
    int32_t head_dim;              /* D: 64 or 128                                    */
    int32_t block_size;            /* tokens per cache block: 16                      */
    int32_t num_blocks;            /* physical blocks in each cache                   */
    int32_t max_blocks_per_req;    /* block_table row stride                          */
    const int32_t *query_start_loc;      /* [R+1]: 0, then running sums of the
                                            scheduled token counts (§5.1.2)         */
    const int32_t *seq_lens;             /* [R]: context length after this step    */
    const int32_t *num_computed_tokens;  /* [R]: must equal seq_len - q_len          */
    const int32_t *block_table_host;     /* optional [R][max_blocks_per_req] host
                                            copy; enables block-id range checks and
                                            the common-prefix equality check       */
    int32_t num_common_prefix_blocks;    /* n >= 0: the first n blocks of every
                                            request with query tokens are the same
                                            physical blocks and fully computed
                                            (n*16 <= num_computed_tokens[r]); n > 0
                                            selects the cascade route              */
    float softmax_scale;           /* scores are softmax_scale * <q, k>; must be > 0   */
    int32_t num_sms;               /* SMs to plan for; 0 = query the current device    */
    int32_t kv_cache_dtype;        /* PA_KV_BF16 or PA_KV_FP8_E4M3                      */
    float k_scale;                 /* FP8 caches: a key reads code_value * k_scale     */
    float v_scale;                 /* FP8 caches: a value reads code_value * v_scale   */
} pa_batch_desc;

/* Element type of the K/V caches ("vLLM 推理流程分析" §6.3: kv_cache_dtype, FP8
 * conversion with k_scale / v_scale).  FP8 caches hold one E4M3 code per
 * element (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest finite
 * 448, S.1111.111 = NaN) in the same [num_blocks][16][Hkv][D] layout. */
#define PA_KV_BF16 0
#define PA_KV_FP8_E4M3 1

/* Work decomposition of a plan (for tests, benchmarks and launch counts). */
typedef struct {
    int32_t num_tokens;            /* T                                               */
    int32_t num_decode_rows;       /* requests with exactly one query token           */
    int32_t num_extend_rows;       /* requests on the tensor-core tiles (> 1 token)   */
    int32_t num_decode_ctas;       /* persistent CTAs of the split-KV decode kernel   */
    int32_t num_decode_items;      /* (request, key range, head group) segments       */
    int32_t num_extend_tiles;      /* CTA tiles (<= 256 rows) of the tensor-core kernel */
    int32_t num_prefix_tiles;      /* of which: shared-prefix (cascade) tiles         */
    int32_t num_partial_slots;     /* (token, partition) partial results              */
    int32_t num_merge_rows;        /* tokens whose output is merged from partials     */
    int32_t kernels_per_call;      /* kernel launches one pa_attention call makes     */
    int32_t num_dequant_blocks;    /* FP8: cache blocks the tensor-core tiles read,
                                      expanded to bf16 in the workspace each call   */
    int64_t decode_kv_bytes;       /* K+V bytes the decode kernel's rows must read    */
    int64_t prefix_kv_bytes;       /* K+V bytes of the shared prefix (read once)      */
    double  extend_flops;          /* 4*D*Hq * visible (query, key) pairs, extend     */
    double  prefix_flops;          /* the same for the shared-prefix tiles            */
    int32_t num_small_q_rows;      /* rows of 2..8 query tokens (speculative verify)
                                      on the split-KV decode kernel, in units of
                                      16 / G tokens: every row of at most 16 / G
                                      tokens, longer ones only while their tiles
                                      (Hkv per row) would not fill the GPU
                                      (decode_kv_bytes counts each unit's keys)   */
    int32_t num_extend_ctas;       /* CTAs of the tensor-core kernel that get tiles   */
    int32_t side_by_side;          /* 1: the tensor-core tiles run on a second stream,
                                      concurrently with the decode kernel on the
                                      other SMs (num_extend_ctas of them go to the
                                      tiles); 0: one after the other              */
} pa_plan_info;

/*
 * Validate the step's metadata and build its plan.
 *   desc              the step (host arrays, read only during this call)
 *   out               receives the plan on PA_OK (NULL otherwise)
 *   workspace_bytes   receives the device workspace size pa_attention needs
 * Returns PA_ERR_INVALID_ARGUMENT for: a NULL pointer, R < 0, non-positive
 * head counts or num_blocks, Hq % Hkv != 0, query_start_loc[0] != 0 or a
 * decreasing query_start_loc, num_computed + q_len != seq_len, a context
 * needing more than max_blocks_per_req blocks, a non-positive or non-finite
 * softmax_scale, a block id out of range in block_table_host, a violated
 * common-prefix precondition, an unknown kv_cache_dtype, or (FP8) a scale that
 * is not finite and > 0.  PA_ERR_UNSUPPORTED for shapes listed above.
 * Host-only (no CUDA call) unless num_sms == 0.
 */
pa_status pa_plan(const pa_batch_desc *desc, pa_plan_t **out, size_t *workspace_bytes);

/* Release a plan.  Never waits for the device: the plan's pinned staging
 * buffer goes back to a library pool and is reused only after its last
 * host->device copy has completed.  NULL is ignored. */
void pa_plan_destroy(pa_plan_t *plan);

/* Fill *info with the plan's work decomposition. */
pa_status pa_plan_get_info(const pa_plan_t *plan, pa_plan_info *info);

/*
 * slot_mapping[t] for every scheduled token ("vLLM 推理流程分析" §5.1.2,
 * block_table.compute_slot_mapping; "vLLM 源码完全拆解（十六）", third
 * walk-through): token i of request r has position p = num_computed[r] + i
 * and slot = block_table[r][p / block_size] * block_size + p % block_size.
 * All pointers are DEVICE memory: query_start_loc [R+1], num_computed [R],
 * block_table [R][max_blocks_per_req], slot_mapping [T] (written).  The
 * metadata must be the same that pa_plan accepted.  num_tokens may exceed
 * query_start_loc[num_reqs] (read on the device): tokens past it get slot -1,
 * so a launch sized for a fixed token capacity skips the padding rows in
 * pa_write_kv.
 */
pa_status pa_slot_mapping(const int32_t *query_start_loc, const int32_t *num_computed,
                          const int32_t *block_table, int32_t num_reqs, int32_t num_tokens,
                          int32_t max_blocks_per_req, int32_t block_size,
                          int64_t *slot_mapping, void *stream);

/*
 * The KV-cache write ("vLLM 推理流程分析" §6.3, reshape_and_cache_flash):
 * for every t with slot_mapping[t] >= 0, row slot_mapping[t] of key_cache and
 * value_cache (viewed as [num_slots][Hkv*D]) becomes a bit copy of key[t] and
 * value[t].  Negative slots are skipped.  A slot >= num_slots is skipped and
 * sets PA_DEVERR_SLOT_RANGE in *device_error_word when that is non-NULL.
 * Duplicate non-negative slots in one call are invalid input (which copy wins
 * is unspecified).  All buffers are DEVICE memory, 16-byte aligned:
 * key/value [T][Hkv][D], slot_mapping [T], caches [num_slots/16][16][Hkv][D].
 * Must be enqueued before pa_attention of the same step on the same stream
 * (write first, then attend: §6.1).
 */
pa_status pa_write_kv(const void *key, const void *value, const int64_t *slot_mapping,
                      int32_t num_tokens, int32_t num_heads_kv, int32_t head_dim,
                      void *key_cache, void *value_cache, int64_t num_slots,
                      int32_t *device_error_word, void *stream);

/*
 * The KV-cache write into FP8 caches ("vLLM 推理流程分析" §6.3: with an FP8
 * kv_cache_dtype the write converts with k_scale / v_scale): element e of
 * key[t] is stored as the E4M3 code of (float)key[t][e] / k_scale, the
 * quotient formed in IEEE binary32 and rounded to the nearest E4M3 value, ties
 * to even, saturating to +-448 (NaN stays NaN); values likewise with v_scale.
 * Slots, skipping, the error word, ordering and alignment as for pa_write_kv;
 * the caches are uint8 [num_slots/16][16][Hkv][D].  The scales must be finite
 * and > 0 (else PA_ERR_INVALID_ARGUMENT).
 */
pa_status pa_write_kv_fp8(const void *key, const void *value, const int64_t *slot_mapping,
                          int32_t num_tokens, int32_t num_heads_kv, int32_t head_dim,
                          void *key_cache, void *value_cache, int64_t num_slots, float k_scale,
                          float v_scale, int32_t *device_error_word, void *stream);

/*
 * Causal GQA attention of the step ("vLLM 推理流程分析" §6.2,
 * flash_attn_varlen_func(q, key_cache, value_cache, cu_seqlens_q, seqlen_k,
 * block_table, softmax_scale, causal=True)).
 *   plan          from pa_plan for this step (may be reused by every layer)
 *   q             DEVICE bf16 [T][Hq][D]
 *   key_cache,
 *   value_cache   DEVICE [num_blocks][16][Hkv][D] of the plan's kv_cache_dtype
 *                 (bf16, or E4M3 codes read as code_value * k_scale / v_scale),
 *                 already holding this step's new rows (written earlier)
 *   block_table   DEVICE int32 [R][max_blocks_per_req]; entries past a
 *                 request's last needed block are never read
 *   out           DEVICE bf16 [T][Hq][D], written for every scheduled token
 *   workspace     DEVICE scratch of at least the size pa_plan reported, 256-byte
 *                 aligned.  Its first 4 bytes are the device error word: zero it
 *                 once before first use; kernels only ever OR bits into it.
 * The result depends only on the metadata and the logical contents: physical
 * block placement does not change a single bit of it.  Slots past seq_len in a
 * request's last block are never used (their contents may be anything,
 * including NaN).  Returns PA_ERR_WORKSPACE_TOO_SMALL, PA_ERR_INVALID_ARGUMENT
 * (NULL or misaligned pointer) or PA_ERR_CUDA (launch failure).  Equivalent to
 * pa_upload_metadata then pa_attention_launch, plus the optional timing events.
 *
 * Side by side (pa_plan_info.side_by_side): when a step has both
 * tensor-core tiles and decode rows and the planner's step-time model says it
 * pays, the tiles get a share of the SMs (num_extend_ctas CTAs) and run on
 * the calling thread's library stream, which first waits for everything
 * enqueued on `stream` so far; the decode kernel runs on `stream` over the
 * other SMs, and `stream` waits for the tiles before the merge.  Seen from
 * `stream` the call stays one ordered unit of work, and under stream capture
 * the library stream joins and leaves the capture inside the call.
 */
pa_status pa_attention(const pa_plan_t *plan, const void *q, const void *key_cache,
                       const void *value_cache, const int32_t *block_table, void *out,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * Capacities of a fixed-shape plan.  Graph mode captures the execution of a
 * stable shape once, then for each step copies the new data to fixed
 * addresses and replays; request counts are rounded up to a capture size and
 * the spare rows padded ("vLLM 源码完全拆解（十六）", fourth walk-through;
 * "vLLM 推理流程分析" §4: total_num_scheduled_tokens selects the CUDA graph).
 * A replay repeats the same launches with the same arguments, so a
 * fixed-shape plan sizes its workspace
 * layout, its grids and every kernel argument from these capacities, so every
 * fixed-shape plan with equal capacities and equal model fields of
 * pa_batch_desc (head counts, head_dim, block_size, num_blocks,
 * max_blocks_per_req, softmax_scale, num_sms, kv_cache_dtype, k_scale,
 * v_scale) launches identically; the step's own lengths reach the kernels
 * only through the uploaded metadata.
 */
typedef struct {
    int32_t max_tokens;          /* T <= max_tokens; q and out hold max_tokens rows */
    int32_t max_reqs;            /* num_reqs <= max_reqs                            */
    int32_t max_extend_tiles;    /* tensor-core tiles (extend rows and cascade
                                    prefix); 0: steps made of decode rows only     */
    int32_t max_dequant_blocks;  /* FP8 caches: blocks those tiles read; 0 if none  */
    int32_t max_partial_slots;   /* partial results; 0 = room for every decode
                                    split plus one slot per (token, head group)    */
    int32_t decode_prefix_tokens;/* 0, or P > 0: every query row of the decode
                                    stream (one-token decode rows and the small
                                    multi-token rows it also takes) lies in token
                                    rows [0, P), and no row from P on is split
                                    (merged from partials, as cascade steps with
                                    chunk rows are), so rows from P on may arrive
                                    later and are final when the tiles finish
                                    (pa_attention_with_kv_update_launch_staged);
                                    steps that break it are rejected with
                                    PA_ERR_CAPACITY.  The SM split then assumes
                                    those rows' q/key/value cross the host link
                                    (~200 GB/s) before the tiles start and their
                                    output rows cross it back after them       */
} pa_fixed_shape;

/*
 * pa_plan with a fixed shape (see pa_fixed_shape).  As pa_plan, plus
 * PA_ERR_INVALID_ARGUMENT for a NULL shape or a capacity < 0 (max_tokens and
 * max_reqs must be > 0), and PA_ERR_CAPACITY when this step needs more tokens,
 * requests, tiles, FP8 blocks or partial slots than the shape allows, or
 * breaks the shape's decode_prefix_tokens.  The
 * workspace size depends on the shape and model fields only.  The decode
 * kernel always runs on num_sms x (CTAs per SM) CTAs.  With tensor-core tiles
 * (max_extend_tiles > 0, num_sms >= 2) the tiles always run on the library
 * stream beside the decode kernel (side_by_side = 1); each step's work cut is
 * the one pa_plan makes for the same step, so a fixed-shape plan and a plain
 * plan of one step compute bit-identical results.
 */
pa_status pa_plan_fixed(const pa_batch_desc *desc, const pa_fixed_shape *shape, pa_plan_t **out,
                        size_t *workspace_bytes);

/*
 * Copy the plan's metadata into the workspace (stream ordered, from a pinned
 * host buffer the plan owns) and prepare the kernels the plan launches.  Not
 * for stream capture.  Arguments and errors as for pa_attention.
 */
pa_status pa_upload_metadata(const pa_plan_t *plan, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Capturable metadata upload (graph mode with the upload inside the graph).
 * pa_plan_metadata_bytes: size of the plan's metadata image (equal for every
 * fixed-shape plan of one shape; 0 for a NULL plan).
 * pa_plan_copy_metadata: copy that image into caller memory, e.g. the
 * page-locked buffer a captured pa_upload_metadata_from reads (host work
 * only; PA_ERR_INVALID_ARGUMENT for a NULL or too small buffer).
 *   host_dst   HOST, bytes >= pa_plan_metadata_bytes(plan)
 * pa_upload_metadata_from: enqueue the copy of an image from page-locked host
 * memory into a workspace, read by the GPU when the copy runs.  Its
 * arguments are plain addresses, so it may be captured in a CUDA graph: the
 * caller refreshes the image (pa_plan_copy_metadata) before each replay and
 * must not overwrite it while an enqueued copy of it has not run yet (use
 * two images and two graphs, or wait for the previous replay).  As for
 * pa_attention_launch, call pa_upload_metadata (which prepares the kernels)
 * at least once before the first capture.
 *   host_src   HOST, page-locked and device-mapped (cudaHostAlloc /
 *              cudaHostRegister), 16-byte aligned
 *   bytes      the image size (a multiple of 16)
 *   workspace  DEVICE, as for pa_attention; workspace_bytes must cover the
 *              plan the image came from
 * Errors: PA_ERR_INVALID_ARGUMENT (NULL, misaligned, bytes not a multiple of
 * 16 or host_src not page-locked), PA_ERR_WORKSPACE_TOO_SMALL,
 * PA_ERR_CUDA.
 */
size_t pa_plan_metadata_bytes(const pa_plan_t *plan);
pa_status pa_plan_copy_metadata(const pa_plan_t *plan, void *host_dst, size_t bytes);
pa_status pa_upload_metadata_from(const void *host_src, size_t bytes, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * The kernels of pa_attention alone: they read the metadata that the last
 * pa_upload_metadata put into this workspace, which must come from a plan of
 * the same fixed shape (or, for a plan made by pa_plan, from this plan).
 * Records no timing events and makes no host<->device copy, so it may be
 * captured in a CUDA graph.  For a fixed-shape plan the enqueued work is
 * identical for every plan of equal shape (see pa_fixed_shape): a graph
 * captured once replays correctly after pa_upload_metadata of any later
 * plan of that shape.  Call pa_upload_metadata (which prepares the kernels)
 * at least once before the first capture.  Arguments and errors as for
 * pa_attention; q and out must hold max_tokens rows for a fixed-shape plan.
 */
pa_status pa_attention_launch(const pa_plan_t *plan, const void *q, const void *key_cache,
                              const void *value_cache, const int32_t *block_table, void *out,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * The step's cache write and attention in one call: the fused dispatch of
 * "vLLM 推理流程分析" §6.1 (the attention layer's forward includes the KV-cache
 * update instead of a separate unified_kv_cache_update).  The caches end up
 * exactly as pa_slot_mapping + pa_write_kv (bf16) or pa_write_kv_fp8 (E4M3,
 * with the plan's k_scale / v_scale) would leave them, and out is the result
 * pa_attention computes over those caches.  A decode row's new K/V row is
 * stored by the decode kernel itself (before it loads the row's last page); the new
 * rows of extend rows are stored by one kernel before the tensor-core tiles
 * read them.  No separate slot-mapping or write launch is needed.
 *   key, value     DEVICE bf16 [T][Hkv][D] (16-byte aligned): the new rows
 *   key_cache,
 *   value_cache    written (the new slots) and read
 *   slot_mapping   optional DEVICE int64 [T]: receives every token's slot
 * Other arguments, errors and ordering as for pa_attention (a block id out of
 * range sets PA_DEVERR_BLOCK_RANGE and that row is not stored).
 */
pa_status pa_attention_with_kv_update(const pa_plan_t *plan, const void *q, const void *key, const void *value,
                                      void *key_cache, void *value_cache, const int32_t *block_table,
                                      int64_t *slot_mapping, void *out, void *workspace, size_t workspace_bytes,
                                      void *stream);

/* Its kernels alone, after pa_upload_metadata: as pa_attention_launch is to
 * pa_attention (capturable; identical launches for plans of one fixed shape). */
pa_status pa_attention_with_kv_update_launch(const pa_plan_t *plan, const void *q, const void *key,
                                             const void *value, void *key_cache, void *value_cache,
                                             const int32_t *block_table, int64_t *slot_mapping, void *out,
                                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Staged inputs: as pa_attention_with_kv_update_launch, for a fixed-shape
 * plan with decode_prefix_tokens = P > 0, when rows P.. of q, key and value
 * are still being written as the call's work starts on `stream` (a host copy
 * in flight on another stream, say).  Rows [0, P) and everything else the
 * call reads must be complete in stream order as usual; rows P.. must be
 * complete once late_rows (a cudaEvent_t, recorded before this call) has
 * fired.  The decode stream, which reads rows below P only, starts at once;
 * the cache write of the rows from P on and the tensor-core tiles wait for
 * late_rows on the library stream.  Without tiles beside the decode stream
 * (no max_extend_tiles, or num_sms < 2) the whole step waits for late_rows.
 * Results are those of pa_attention_with_kv_update_launch.
 *   late_rows       cudaEvent_t (not NULL)
 *   late_out_ready  optional cudaEvent_t: recorded once rows P.. of out are
 *                   final (after the tiles, on the library stream; after the
 *                   whole step when there is no second stream), so that the
 *                   caller can copy them out while the decode stream runs on.
 *                   Rows [0, P) are final in stream order at the call's end.
 * Errors: as pa_attention_with_kv_update_launch, plus PA_ERR_INVALID_ARGUMENT
 * for a NULL late_rows or a plan that is not fixed-shape with P > 0.
 */
pa_status pa_attention_with_kv_update_launch_staged(const pa_plan_t *plan, const void *q, const void *key,
                                                    const void *value, void *key_cache, void *value_cache,
                                                    const int32_t *block_table, int64_t *slot_mapping, void *out,
                                                    void *workspace, size_t workspace_bytes, void *stream,
                                                    void *late_rows, void *late_out_ready);

/*
 * Zero newly allocated cache blocks ("vLLM 推理流程分析" §4: the scheduler
 * output lists new_block_ids_to_zero, blocks whose old contents must be
 * cleared; §5.1.1: _update_states zeroes them so that cache positions not yet
 * written are never read as stale KV).  Every byte of the K and V entries of
 * each listed block becomes 0 (+0 in bf16, code 0x00 in E4M3).
 *   block_ids        DEVICE int32 [num_ids]; ids < 0 are skipped (padding of a
 *                    fixed-size launch); an id >= num_blocks is skipped and
 *                    sets PA_DEVERR_BLOCK_RANGE in *device_error_word (if
 *                    non-NULL)
 *   key_cache,
 *   value_cache      DEVICE, 16-byte aligned, [num_blocks][16][Hkv][D] of
 *                    kv_cache_dtype (PA_KV_BF16 or PA_KV_FP8_E4M3)
 * Returns PA_ERR_INVALID_ARGUMENT for a negative count or size, a NULL or
 * misaligned pointer, or an unknown kv_cache_dtype; PA_ERR_CUDA on a launch
 * failure.  Enqueue before the step's pa_write_kv.
 */
pa_status pa_zero_blocks(const int32_t *block_ids, int32_t num_ids, int32_t num_blocks, int32_t num_heads_kv,
                         int32_t head_dim, int32_t kv_cache_dtype, void *key_cache, void *value_cache,
                         int32_t *device_error_word, void *stream);

/*
 * Read and clear the device error word (the first 4 bytes of a workspace, or
 * any int32 the caller passed to pa_write_kv).  Synchronises the stream.
 * *bits (optional) receives the PA_DEVERR_* bits seen.  Returns PA_OK when no
 * bit was set, PA_ERR_DEVICE_CHECK otherwise, PA_ERR_CUDA if the read failed.
 */
pa_status pa_check_device_errors(int32_t *device_error_word, int32_t *bits, void *stream);

/*
 * Optional per-kernel timing.  While enabled, every pa_attention call with
 * this plan records CUDA events around each kernel it launches.
 * pa_plan_kernel_times waits for those events and returns, per kernel kind
 * (0 decode, 1 extend/prefix, 2 merge, 3 metadata copy), the summed
 * milliseconds and the launch count since timing was enabled.
 */
pa_status pa_plan_enable_timing(pa_plan_t *plan, int32_t enable);
pa_status pa_plan_kernel_times(pa_plan_t *plan, double ms_total[4], int32_t launches[4]);

/* Size in bytes of the library-owned scratch array pa_attention_no_alloc
 * uses in place of a caller workspace (16 MiB per device). */
#define PA_NO_ALLOC_SCRATCH_BYTES (16u << 20)

/*
 * pa_attention for callers that cannot allocate device memory.  The pages
 * have no counterpart of this call; it exists for users of this library, not
 * for the method.
 *
 * Who can't allocate: an engine that gives nearly all free device memory to
 * its paged KV pool at start-up has no room for a per-step workspace, and a
 * hot path that must not call cudaMalloc/cudaFree (they can synchronise the
 * whole device) cannot create one on demand.  Such a caller passes the same
 * inputs and output as to pa_attention but no workspace: the scratch is a
 * library-owned device array of PA_NO_ALLOC_SCRATCH_BYTES, created on each
 * device that loads the library's module holding it and kept until exit.
 * This call allocates nothing: no cudaMalloc, cudaMallocHost, cudaFree, no
 * pinned staging buffer (the metadata is copied from the plan's pageable host
 * image, so the upload waits for the stream's earlier work), and it records
 * no timing events.
 *
 *   plan, q, key_cache, value_cache, block_table, out   as for pa_attention
 *   device_error_word  optional DEVICE int32: receives (overwritten, not ORed)
 *                      this call's PA_DEVERR_* bits; read it with
 *                      pa_check_device_errors
 *   stream             cudaStream_t
 * Returns PA_ERR_WORKSPACE_TOO_SMALL, before enqueueing anything, when the
 * plan's workspace_bytes exceeds PA_NO_ALLOC_SCRATCH_BYTES; otherwise as
 * pa_attention.
 *
 * The first call on a device (made with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * Every call on a device shares the one array and the array keeps the last
 * call's contents: the error word is cleared by each call, everything else is
 * rewritten before it is read.  Calls whose work can overlap on the GPU (on
 * different streams, or from different host threads without ordering) race
 * on the array and must be serialised by the caller.
 */
pa_status pa_attention_no_alloc(const pa_plan_t *plan, const void *q, const void *key_cache,
                                const void *value_cache, const int32_t *block_table, void *out,
                                int32_t *device_error_word, void *stream);

/*
 * Native graph executor: graph mode of "vLLM 源码完全拆解（十六）" (fourth
 * walk-through: capture a stable shape once; per step copy the new data to
 * fixed addresses and replay) without a framework around it.  A pa_graph_t
 * holds two instantiated CUDA graphs of one fixed shape, each made of
 *   [copy of a page-locked input image to the device]   (optional host I/O)
 *   pa_upload_metadata_from(its own page-locked metadata image)
 *   the step: pa_attention_with_kv_update_launch (fused), or pa_slot_mapping
 *             + pa_write_kv / pa_write_kv_fp8 + pa_attention_launch
 *   [copy of out back to a page-locked output buffer]   (optional host I/O)
 * and alternates between them, so the host prepares one step while the
 * previous one may still run.  It owns its workspace (error word included),
 * its slot buffer, both metadata images, two events and a capture stream; the
 * caller owns every buffer listed in pa_graph_buffers and must keep them (and
 * their addresses) for the graph's lifetime.  pa_graph_step costs one fixed
 * plan (host), one copy of its metadata image (host) and one graph launch.
 * A pa_graph_t is not thread-safe: one host thread at a time may call
 * pa_graph_step / pa_graph_wait on it (different graphs are independent).
 */
typedef struct pa_graph_s pa_graph_t;

typedef struct {
    /* DEVICE buffers sized for the fixed shape (16-byte aligned). */
    void *q;                         /* bf16 [max_tokens][Hq][D]          */
    void *key;                       /* bf16 [max_tokens][Hkv][D]         */
    void *value;                     /* bf16 [max_tokens][Hkv][D]         */
    void *out;                       /* bf16 [max_tokens][Hq][D]          */
    int32_t *query_start_loc;        /* [max_reqs + 1]                     */
    int32_t *num_computed;           /* [max_reqs]                         */
    int32_t *block_table;            /* [max_reqs][max_blocks_per_req]     */
    void *key_cache;                 /* [num_blocks][16][Hkv][D] of the    */
    void *value_cache;               /*   desc's kv_cache_dtype            */
    int32_t fused;                   /* 1: write + attention in one call   */
    /* Optional host I/O (all NULL / 0 for none).  host_in[i] (page-locked
     * HOST, in_bytes) is copied to device_in (DEVICE, in_bytes) at the start
     * of graph i; device_in normally spans the device buffers above, so that
     * one copy brings a whole step's inputs in.  Output: when out_bytes
     * covers the whole out buffer (max_tokens * Hq * D * 2), graph i's
     * kernels store the output rows straight into host_out[i] through its
     * device mapping, during the step (device `out` is then not written);
     * with a smaller out_bytes, out (out_bytes from its start) is copied to
     * host_out[i] (page-locked HOST) at the end of graph i.
     * Staged (fused, shape.decode_prefix_tokens = P with 0 < P < max_tokens,
     * and q, key, value inside device_in): the image is copied in two parts,
     * everything but rows P.. of q, key and value first and those rows after
     * it on a second stream, through pa_attention_with_kv_update_launch_
     * staged, so the decode stream starts after the first part; with a
     * whole-output host buffer, out is written on the device and rows
     * P..max_tokens are copied back as soon as the tiles are done, rows
     * [0, P) after the step (no direct stores). */
    const void *host_in[2];
    void *device_in;
    size_t in_bytes;
    void *host_out[2];
    size_t out_bytes;
} pa_graph_buffers;

/*
 * Capture the two graphs.  desc is any step the shape accepts (its model
 * fields fix the graph's: head counts, head_dim, block_size, num_blocks,
 * max_blocks_per_req, softmax_scale, num_sms, kv_cache_dtype, k_scale,
 * v_scale); it is planned with pa_plan_fixed and its metadata uploaded
 * eagerly on the capture stream, which also prepares the kernels.  The
 * device buffers are not read during this call.
 * Errors: as pa_plan_fixed; PA_ERR_INVALID_ARGUMENT for a NULL or misaligned
 * buffer, host I/O given in part, or a host buffer that is not page-locked;
 * PA_ERR_CUDA when an allocation, the capture or the instantiation fails.
 */
pa_status pa_graph_create(const pa_batch_desc *desc, const pa_fixed_shape *shape, const pa_graph_buffers *bufs,
                          pa_graph_t **out);

/*
 * One step: wait until the graph that next runs (pa_graph_turn) has finished
 * its previous launch, plan desc with the graph's fixed shape, copy the
 * plan's metadata into that graph's image, launch it on stream and flip the
 * turn.  With host I/O, host_in[pa_graph_turn(g)] must hold the step's inputs
 * before the call (write them after pa_graph_wait of that turn), and the
 * output is in host_out[that turn] once pa_graph_wait returns for it.
 * Errors: PA_ERR_INVALID_ARGUMENT (NULL, or desc's model fields differ from
 * the graph's), the errors of pa_plan_fixed (nothing is launched then),
 * PA_ERR_CUDA.
 */
pa_status pa_graph_step(pa_graph_t *g, const pa_batch_desc *desc, void *stream);

/* Index (0 or 1) of the graph the next pa_graph_step launches. */
int32_t pa_graph_turn(const pa_graph_t *g);

/* Block until graph `turn`'s last launch (if any) has completed. */
pa_status pa_graph_wait(pa_graph_t *g, int32_t turn);

/* The graph's workspace: its first 4 bytes are the device error word (read
 * it with pa_check_device_errors). */
void *pa_graph_workspace(const pa_graph_t *g);

/* The graph's DEVICE slot buffer (int64 [max_tokens]): every token's slot
 * after a step (fused or not). */
int64_t *pa_graph_slot_mapping(const pa_graph_t *g);

/* Waits for both graphs, then frees everything the graph owns.  NULL is a no-op. */
void pa_graph_destroy(pa_graph_t *g);

/* Static description of a status code. */
const char *pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
