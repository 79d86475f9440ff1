/*
 * liblora_gb300 -- multi-tenant LoRA delta on one GB300 (sm_103a), C ABI.
 *
 * For a batch whose rows (tokens, or (token, k) pairs after top-k routing)
 * each carry an adapter slot a (-1 = none) the library adds, in place,
 *
 *     y[t][off_j + o] += scale[a] * sum_k ( sum_h x[t][h] * A_j[a][k][h] ) * B_j[a][o][k]
 *
 * for every packed output slice j, k < rank[a].  This is the shrink
 * (x -> rank, fp32) / expand (rank -> out, added into y) pair of the vLLM LoRA
 * layer pages (RowParallelLinearWithShardedLoRA.apply: zeroed fp32 buffer
 * [n_slices][T][rank], add_shrink with scale 1.0, add_expand with
 * add_input=True at the slice offsets), for packed column layers (QKV,
 * gate_up; MergedColumnParallelLinearWithLoRA, MergedQKVParallelLinearWithLoRA),
 * row/replicated layers and lm_head (LogitsProcessorWithLoRA, add_lora_logits),
 * and for the fused-MoE per-(adapter, expert) variant (FusedMoEWithLoRA,
 * add_lora_fused_moe) including the shared-outer layout of the Inkling LoRA
 * PR report.
 *
 * Conventions common to every entry point
 *  - Every call is asynchronous on `stream` (a cudaStream_t, NULL = the legacy
 *    default stream).  Only lora_get_device_status and lora_pool_destroy
 *    synchronise.  Calls that take only device pointers launch kernels and
 *    cudaMemsetAsync/cudaMemcpyAsync only, so they can be captured in a CUDA
 *    graph.
 *  - bf16 tensors are passed as `void *` (2-byte elements, row-major).  All
 *    device tensors given to compute calls must be 16-byte aligned and their
 *    leading dimensions (in elements) multiples of 8.
 *  - Host-checked argument errors return synchronously and launch nothing.
 *    No call throws, traps or asserts on the device.  Bad adapter indices seen
 *    on the device set the pool's status word (LORA_ERR_DEVICE_INDEX) and the
 *    row is treated as idx -1; a cross-CTA wait that runs out of iterations
 *    sets LORA_ERR_TIMEOUT.  Read and clear it with lora_get_device_status.
 *  - A row is *active* when 0 <= idx < max_loras, the slot is enabled and its
 *    rank is > 0 (and, for MoE, its expert id is in range).  Inactive rows of
 *    y / ic1 / ic3 are left bit-identical.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LORA_API __attribute__((visibility("default")))
#else
#define LORA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,   /* null pointer, bad alignment, bad size */
    LORA_ERR_INDEX = 2,         /* slot outside [0, max_loras) */
    LORA_ERR_RANK = 3,          /* rank < 0 or rank > max_rank (SGLang validate_new_adapter) */
    LORA_ERR_SHAPE = 4,         /* dims/expert count do not match the pool; vocab > 257024 */
    LORA_ERR_LAYOUT = 5,        /* shared-outer pool given per-expert A/B or the reverse */
    LORA_ERR_NOMEM = 6,         /* device allocation failed */
    LORA_ERR_CUDA = 7,          /* a CUDA runtime call failed */
    LORA_ERR_DEVICE_INDEX = 8,  /* (device status) idx or expert id out of range was seen */
    LORA_ERR_TIMEOUT = 9,       /* (device status) a bounded cross-CTA wait gave up */
    LORA_ERR_CAPACITY = 10,     /* meta/workspace buffer too small for the call */
    LORA_ERR_UNSUPPORTED = 11   /* call does not apply to this pool kind */
} lora_status_t;

#define LORA_MAX_SLICES 8
#define LORA_MAX_RANK 256
#define LORA_MAX_VOCAB 257024
#define LORA_TILE_ROWS 16
#define LORA_LTILE_ROWS 128
#define LORA_LONG_MIN 64

/* ------------------------------------------------------------------ pool */

/* Shape of one LoRA-wrapped layer (create_lora_weights of the pages).
 * Dense pool (num_experts == 0): n_slices packed output slices of widths
 *   out_dims[j] over one input of width in_dim.  lm_head is n_slices = 1 with
 *   out_dims[0] = vocab and is_lm_head = 1 (vocab <= 257024; the pages' guard
 *   in LogitsProcessorWithLoRA.create_lora_weights, read as "reject only
 *   vocab > 257024").
 * MoE pool (num_experts > 0): w13 has n_w13_slices (2 = gate and up as in
 *   FusedMoEWithLoRA; 1 = non-gated or the FusedMoE3DWithLoRA layout) slices
 *   of width w13_slice_width (d_mlp, or 2*d_mlp for the 3D layout) over input
 *   d_model; w2 maps d_mlp -> d_model.  shared_outer = 1 gives w13-A and w2-B
 *   an expert dimension of 1 (enable_moe_shared_loras of the Inkling report).
 * Every width must be a positive multiple of 8. */
typedef struct {
    int32_t max_loras;                  /* L >= 1 */
    int32_t max_rank;                   /* R in [1, LORA_MAX_RANK] */
    int32_t in_dim;                     /* dense: H */
    int32_t n_slices;                   /* dense: 1..LORA_MAX_SLICES */
    int32_t out_dims[LORA_MAX_SLICES];  /* dense: widths O_j */
    int32_t is_lm_head;                 /* dense: apply the vocab guard */
    int32_t num_experts;                /* 0 = dense; MoE: E >= 1 */
    int32_t d_model;                    /* MoE: D */
    int32_t d_mlp;                      /* MoE: F (w2 input width) */
    int32_t n_w13_slices;               /* MoE: 1 or 2 */
    int32_t w13_slice_width;            /* MoE: width of one w13 slice */
    int32_t shared_outer;               /* MoE: 0 or 1 */
} lora_pool_desc_t;

typedef struct lora_pool lora_pool_t;   /* opaque; owns the stacked weights and tables */

/* Allocate a zeroed pool on the current device (every slot reset: zero
 * weights, rank 0, disabled).  The pool owns its device memory; it keeps its
 * weights in its own layout (A rows [R][in], B compact [out][ceil8(rank)]).
 * With max_rank <= 64 it also holds TMA tensor maps of its B tensors for the
 * tensor-core kernels (built here, with a host synchronisation of `stream`);
 * kernels that would use a map that could not be built take another path.
 * Errors: LORA_ERR_INVALID_ARG, LORA_ERR_SHAPE, LORA_ERR_NOMEM, LORA_ERR_CUDA. */
LORA_API lora_status_t lora_pool_create(const lora_pool_desc_t *desc, void *stream, lora_pool_t **out);

/* Synchronise the device and free the pool. */
LORA_API lora_status_t lora_pool_destroy(lora_pool_t *pool);

/* Copy the descriptor the pool was created with. */
LORA_API lora_status_t lora_pool_get_desc(const lora_pool_t *pool, lora_pool_desc_t *out);

/* set_lora of a dense pool (MergedColumnParallelLinearWithLoRA.set_lora):
 * reset the slot, then copy A[j] ([rank][in_dim] bf16, row-major) and B[j]
 * ([out_dims[j]][rank] bf16) for j < n (n == n_slices); a NULL pair leaves
 * that slice zero.  Sources may be host or device memory (cudaMemcpyDefault);
 * host sources must stay valid until the stream reaches the copy.  Sets
 * rank, scale and enabled = 1.  Errors: LORA_ERR_INDEX (slot), LORA_ERR_RANK
 * (rank > max_rank or < 0), LORA_ERR_SHAPE (n != n_slices),
 * LORA_ERR_UNSUPPORTED (MoE pool). */
LORA_API lora_status_t lora_set(lora_pool_t *pool, int32_t slot, int32_t rank, float scale,
                       const void *const *A, const void *const *B, int32_t n, void *stream);

/* set_lora of MergedColumnParallelLinearVariableSliceWithLoRA (one checkpoint
 * tensor for a layer with packed slices): A ([rank][in_dim]) is duplicated to
 * every slice and B ([sum_j out_dims[j]][rank]) is split along its rows by
 * the slice widths.  Errors as lora_set. */
LORA_API lora_status_t lora_set_packed(lora_pool_t *pool, int32_t slot, int32_t rank, float scale,
                              const void *A, const void *B, void *stream);

/* set_lora of a MoE pool (FusedMoEWithLoRA.set_lora): reset, enable, copy
 *   A[s] = w13 A of slice s: [a_experts[s]][rank][d_model]          (s < n_w13_slices)
 *   B[s] = w13 B of slice s: [b_experts[s]][w13_slice_width][rank]
 *   A[n_w13_slices] = w2 A:  [a_experts[..]][rank][d_mlp]
 *   B[n_w13_slices] = w2 B:  [b_experts[..]][d_model][rank]
 * The expert counts must be E, except w13-A and w2-B which must be 1 in a
 * shared-outer pool (LoRAManager._detect_shared_outer_loras: mixed formats
 * are an error).  n must equal n_w13_slices + 1.
 * Errors: LORA_ERR_INDEX, LORA_ERR_RANK, LORA_ERR_SHAPE (expert count or n),
 * LORA_ERR_LAYOUT (1 where E is expected for w13-A/w2-B or the reverse),
 * LORA_ERR_UNSUPPORTED (dense pool). */
LORA_API lora_status_t lora_set_moe(lora_pool_t *pool, int32_t slot, int32_t rank, float scale,
                           const void *const *A, const int32_t *a_experts,
                           const void *const *B, const int32_t *b_experts, int32_t n,
                           void *stream);

/* reset_lora: zero every tensor of the slot, rank 0, scale 0, enabled 0.
 * Errors: LORA_ERR_INDEX. */
LORA_API lora_status_t lora_reset(lora_pool_t *pool, int32_t slot, void *stream);

/* ------------------------------------------------------------- metadata */

/* Batch metadata in caller-owned device memory (bind it with lora_meta_bind).
 * A "row" is a token (dense) or a pair p = t*top_k + k (MoE); a "key" is the
 * slot a (dense) or a*E + e (MoE).  After lora_build_meta:
 *   sorted[max_rows]      rows stably sorted by key (keys ascending, rows in
 *                         original order within a key); inactive rows last,
 *                         in original order
 *   key_count[max_keys]   active rows per key
 *   key_offset[max_keys+1] exclusive prefix sum of key_count
 *   group_key[max_keys]   the non-empty keys, ascending (one "group" each)
 *   group_start[max_keys+1] first sorted position of each group; [n_groups] = n_active
 *   key_group[max_keys]   group index of each key, -1 if empty
 *   tile_group[max_tiles], tile_row0[max_tiles]: groups cut into tiles of at
 *                         most LORA_TILE_ROWS rows, in group order
 *   tile_keyn[max_tiles]  (key << 5) | rows of each tile
 *   ltile_row0, ltile_keyn ((key << 8) | rows), ltile_tok0 [max_ltiles]: for
 *                         a dense pool, each group of >= LORA_LONG_MIN rows
 *                         whose token ids form one contiguous run, cut into
 *                         tiles of <= 128 rows (tok0 = first token of the tile)
 *   stile_row0, stile_keyn [max_tiles]: 16-row tiles of the other groups
 *   counters[8]           n_active, n_groups, n_bad, n_tiles, n_stiles, n_ltiles
 *   counters[4]           n_active, n_groups, n_bad, n_tiles
 * The host fields T, top_k, n_keys and mode (0 dense, 1 MoE) record the last
 * build.  Buffers stay valid until the next build into the same meta; rebuild
 * after lora_set / lora_reset of a slot the batch uses. */
typedef struct {
    int32_t max_rows;
    int32_t max_keys;
    int32_t max_tiles;
    int32_t max_ltiles;
    int32_t T, top_k, n_keys, mode;
    int32_t *sorted;
    int32_t *key_count;
    int32_t *key_offset;
    int32_t *group_key;
    int32_t *group_start;
    int32_t *key_group;
    int32_t *tile_group;
    int32_t *tile_row0;
    int32_t *tile_keyn;
    int32_t *ltile_row0;
    int32_t *ltile_keyn;
    int32_t *ltile_tok0;
    int32_t *stile_row0;
    int32_t *stile_keyn;
    int32_t *counters;
} lora_meta_t;

/* Device bytes lora_meta_bind needs for the given capacities. */
LORA_API size_t lora_meta_bytes(int32_t max_rows, int32_t max_keys);

/* Carve `d_buf` (device, 16-byte aligned, >= lora_meta_bytes) into the meta
 * arrays.  Errors: LORA_ERR_INVALID_ARG, LORA_ERR_CAPACITY. */
LORA_API lora_status_t lora_meta_bind(lora_meta_t *meta, void *d_buf, size_t bytes, int32_t max_rows,
                             int32_t max_keys);

/* Build the metadata on the device (one kernel, no host synchronisation,
 * graph-capturable).  d_idx: [T] int32 slot per token (-1 = none).  Dense
 * pool: d_topk_ids must be NULL.  MoE pool: d_topk_ids is [T][top_k] int32.
 * Rows are counted against the pool's enabled/rank tables as they are on the
 * stream at launch.  Errors: LORA_ERR_INVALID_ARG, LORA_ERR_CAPACITY
 * (T*top_k > max_rows, keys > max_keys, or more than 6144 keys). */
LORA_API lora_status_t lora_build_meta(const lora_pool_t *pool, const int32_t *d_idx, int32_t T,
                              const int32_t *d_topk_ids, int32_t top_k, lora_meta_t *meta,
                              void *stream);

/* --------------------------------------------------------- dense compute */

/* add_shrink (scale 1.0) of a dense pool into a zeroed buffer: v is
 * [n_slices][T][max_rank] fp32 device and is overwritten; for every active
 * token t with slot a and slice j, v[j][t][k] = sum_h x[t][h] A_j[a][k][h]
 * for k < rank[a]; every other entry is 0.  The sum over h is split into
 * chunks accumulated with fp32 atomics, so the last bit may vary between
 * runs (lora_apply_slices is deterministic).  x: [T][ldx] bf16 device. */
LORA_API lora_status_t lora_shrink(const lora_pool_t *pool, const lora_meta_t *meta, const void *x,
                          int64_t ldx, float *v, void *stream);

/* add_expand (add_input=True): for every active token t with slot a,
 * y[t][off_j + o] += scale[a] * sum_{k<rank[a]} v[j][t][k] * B_j[a][o][k]
 * with off_j the running sum of the slice widths; y: [T][ldy] bf16 device,
 * fp32 accumulation, one rounding to bf16 per element. */
LORA_API lora_status_t lora_expand(const lora_pool_t *pool, const lora_meta_t *meta, const float *v,
                          void *y, int64_t ldy, void *stream);

/* Workspace bytes for lora_apply_slices / lora_moe_apply on up to T tokens
 * (top_k = 1 for a dense pool).  The first eighth of a workspace holds
 * counters that every call leaves zero; the rest is scratch.  One workspace
 * may serve every layer of a pool and any batch of up to T tokens, as long
 * as every call passes the same (workspace, ws_bytes) pair. */
LORA_API size_t lora_workspace_bytes(const lora_pool_t *pool, int32_t T, int32_t top_k);

/* Zero a workspace (a cudaMemsetAsync).  A workspace must be zero before its
 * first use; every apply call leaves its control words zero again. */
LORA_API lora_status_t lora_workspace_init(void *workspace, size_t bytes, void *stream);

/* Shrink and expand of every slice in one persistent kernel (the fused
 * apply of a LoRA linear layer: QKV, gate_up, o_proj/down_proj, lm_head):
 * y += delta as in lora_expand.  The fp32 intermediate never leaves the
 * workspace.  Calls that share a workspace must not overlap on the device.
 * Errors: LORA_ERR_INVALID_ARG, LORA_ERR_CAPACITY (workspace too small),
 * LORA_ERR_UNSUPPORTED (MoE pool). */
LORA_API lora_status_t lora_apply_slices(const lora_pool_t *pool, const lora_meta_t *meta, const void *x,
                                int64_t ldx, void *y, int64_t ldy, void *workspace,
                                size_t ws_bytes, void *stream);

/* The first LoRA layer of a serving step in one call: builds the batch
 * metadata of d_idx ([T] int32 slots, -1 = none) into meta exactly as
 * lora_build_meta(pool, d_idx, T, NULL, 1, meta, stream) does, and adds the
 * delta of this dense layer to y as lora_apply_slices(pool, meta, x, ldx, y,
 * ldy, workspace, ws_bytes, stream) does (the per-batch tables of SGLang's
 * LoRAManager.prepare_lora_batch followed by the layer's add_shrink /
 * add_expand).  Later layers of the step reuse meta with lora_apply_slices.
 * For decode-sized batches of a pool the fused decode kernel serves (see
 * lora_set_kernel_policy) both happen in one launch: every slot's cluster
 * finds its rows in d_idx while one more CTA writes the metadata, so the
 * layer does not wait for the metadata build.  Otherwise the two calls are
 * made in order.  Arguments, errors and the workspace as the two calls;
 * LORA_ERR_UNSUPPORTED for a MoE pool. */
LORA_API lora_status_t lora_build_meta_apply(const lora_pool_t *pool, const int32_t *d_idx, int32_t T,
                                             lora_meta_t *meta, const void *x, int64_t ldx, void *y, int64_t ldy,
                                             void *workspace, size_t ws_bytes, void *stream);

/* Same result as lora_apply_slices, but for callers that cannot provide a
 * workspace: the library allocates nothing and uses one fixed scratch array
 * in its own device image (lora_static_scratch_bytes() bytes, 8 MiB, held on
 * every GPU that loads the library until the process exits).  This is for
 * hosts whose device memory is fully reserved by another allocator (so
 * cudaMalloc would fail), latency-critical paths that may not block on an
 * allocation, and C callers with no allocator to lend.  It has no
 * counterpart in the LoRA layer pages; it is a deployment convenience of
 * this library.
 * The first call on a device (with that device current) looks up the array's
 * device address; make that first call before any stream capture.  All calls
 * share the array, each call clears the control words it needs, and calls
 * that overlap on the GPU race.  Errors as lora_apply_slices, plus
 * LORA_ERR_CAPACITY when the batch needs more scratch than the array holds
 * and LORA_ERR_CUDA if the address lookup fails. */
LORA_API lora_status_t lora_apply_slices_static(const lora_pool_t *pool, const lora_meta_t *meta,
                                                const void *x, int64_t ldx, void *y, int64_t ldy,
                                                void *stream);

/* Size in bytes of the fixed scratch array used by lora_apply_slices_static. */
LORA_API size_t lora_static_scratch_bytes(void);

/* lm_head with LoRA, end to end (LogitsProcessorWithLoRA._get_logits of the
 * vLLM LoRA layer page, with the muP multiplier of the Inkling report's
 * _lora_forward).  For every token t and column i < vocab_size:
 *   out[t][i] = mup * ( in[t][mapping[i]] + delta[t][i] )
 * where in is the gathered base logits [T][ld_in] bf16 (in_cols valid
 * columns, sharded order), mapping is the device int32 gather index
 * (sharded_to_full_mapping applied as logits[:, mapping]; NULL = identity),
 * and delta is the LoRA delta of the pool (a dense pool with one slice whose
 * width is the padded vocab; add_lora_logits uses scale 1.0, so set_lora the
 * lm_head adapters with scale 1 for that behaviour).  mup = 1 when the model
 * has no muP multiplier.  hidden is [T][ld_h] bf16.  logits_out is
 * [T][ld_out] bf16 with ld_out >= the pool's width; columns in
 * [vocab_size, width) are scratch.  A mapping entry outside [0, in_cols) sets
 * LORA_ERR_DEVICE_INDEX and reads column 0.  Workspace as lora_apply_slices.
 * Errors: LORA_ERR_INVALID_ARG, LORA_ERR_SHAPE (vocab_size > width or
 * > 257024, in_cols), LORA_ERR_UNSUPPORTED (not a one-slice dense pool). */
LORA_API lora_status_t lora_logits_apply(const lora_pool_t *pool, const lora_meta_t *meta, const void *hidden,
                                         int64_t ld_h, const void *logits_in, int64_t ld_in, int32_t in_cols,
                                         const int32_t *mapping, void *logits_out, int64_t ld_out,
                                         int32_t vocab_size, float mup, void *workspace, size_t ws_bytes,
                                         void *stream);

/* ------------------------------------------------------------ MoE compute */

#define LORA_MOE_W13 0
#define LORA_MOE_W2 1

/* add_lora_fused_moe of a MoE pool after lora_build_meta with topk ids.
 * W13: in = hidden states x [T][ld_in] (row t of pair p = p / top_k),
 *      out = ic1 [T*top_k][ld_out], slice s written at columns
 *      [s*w13_slice_width, (s+1)*w13_slice_width), before the activation:
 *      ic1[p][s*W + o] += scale[a] * B13_s[a][e] (A13_s[a][e'] x[t]).
 * W2:  in = ic2 [T*top_k][ld_in], out = ic3 [T*top_k][ld_out], before the
 *      top-k sum: ic3[p][o] += topk_w[p] * scale[a] * B2[a][e''] (A2[a][e] ic2[p]);
 *      topk_w is [T*top_k] fp32 device, NULL = 1.
 * e' = 0 for w13-A and e'' = 0 for w2-B in a shared-outer pool, else e.
 * Errors: LORA_ERR_INVALID_ARG, LORA_ERR_CAPACITY, LORA_ERR_UNSUPPORTED. */
LORA_API lora_status_t lora_moe_apply(const lora_pool_t *pool, const lora_meta_t *meta, int32_t which,
                             const void *in, int64_t ld_in, const float *topk_w, void *out,
                             int64_t ld_out, void *workspace, size_t ws_bytes, void *stream);

/* The block-padded form of moe_lora_align_block_size (vLLM
 * FusedMoEWithLoRA: sorted_token_ids_lora and expert_ids_lora viewed as
 * (max_loras, -1), num_tokens_post_padded_lora), derived on the device from a
 * MoE metadata build: for every adapter a, the (token, k) pairs of its keys
 * (a, e) in ascending expert order, each expert's run padded with the
 * sentinel T*top_k to a multiple of block_m.
 *   d_sorted [L][cap]            pair ids and sentinels (unused entries T*top_k)
 *   d_expert [L][cap / block_m]  expert of each block (unused entries -1)
 *   d_npp    [L]                 padded length of each adapter (0 if none)
 * cap must be a multiple of block_m and >= T*top_k + E*(block_m - 1).
 * Errors: LORA_ERR_INVALID_ARG, LORA_ERR_CAPACITY, LORA_ERR_UNSUPPORTED. */
LORA_API lora_status_t lora_moe_align_padded(const lora_pool_t *pool, const lora_meta_t *meta, int32_t block_m,
                                             int32_t cap, int32_t *d_sorted, int32_t *d_expert,
                                             int32_t *d_npp, void *stream);

/* add_lora_fused_moe over a block-padded alignment (the schedule vLLM's
 * FusedMoEWithLoRA runs on sorted_token_ids_lora / expert_ids_lora; with
 * block_m = 1 every routed pair is a block of its own, the naive assignment
 * it takes when num_tokens * top_k * 8 <= num_experts * max_loras).
 * d_sorted, d_expert, d_npp, block_m and cap as written by
 * lora_moe_align_padded from the same meta; which, in, ld_in, topk_w, out
 * and ld_out as lora_moe_apply, with the same result.  No workspace.
 * Entries of d_sorted outside [0, T*top_k) and blocks whose expert is
 * outside [0, num_experts) are skipped.
 * Errors: LORA_ERR_INVALID_ARG (also block_m outside [1, 16] or cap not a
 * multiple of block_m), LORA_ERR_UNSUPPORTED (not a MoE pool; more than two
 * w13 slices, max_rank above 64, or an input width above 4096). */
LORA_API lora_status_t lora_moe_apply_blocks(const lora_pool_t *pool, const lora_meta_t *meta, int32_t which,
                                             const void *in, int64_t ld_in, const float *topk_w, void *out,
                                             int64_t ld_out, const int32_t *d_sorted, const int32_t *d_expert,
                                             const int32_t *d_npp, int32_t block_m, int32_t cap, void *stream);

/* ------------------------------------------------------------ status */

/* Synchronise `stream`, return the pool's device status word (LORA_OK,
 * LORA_ERR_DEVICE_INDEX or LORA_ERR_TIMEOUT) and clear it. */
LORA_API lora_status_t lora_get_device_status(const lora_pool_t *pool, void *stream);

/* Bound on the polls of every cross-CTA wait of lora_apply_slices and
 * lora_moe_apply (default 1 << 20, each poll sleeps up to ~64 ns).  When a wait
 * gives up, the device status becomes LORA_ERR_TIMEOUT and that work item is
 * skipped.  A negative value makes every wait that is not already satisfied
 * give up at once (to exercise the error path).  Process-wide. */
LORA_API void lora_set_spin_limit(int32_t max_polls);

/* The full LoRA linear layer of a dense pool (vLLM LoRA layer pages,
 * BaseLinearLayerWithLoRA / ColumnParallelLinearWithLoRA.apply: base output,
 * then the LoRA delta added in place):
 *   y = x W^T + bias + delta          (delta as in lora_apply_slices)
 * W is the base weight [out_total][ldw] bf16 row-major (the packed slices'
 * weights stacked in slice order), bias [out_total] bf16 or NULL, y is fully
 * written for the meta's T tokens (meta from a dense lora_build_meta).
 * By default the base GEMM is a cuBLASLt call and the delta a second pass
 * over y (lora_apply_slices).  Under lora_set_kernel_policy(6), when
 * max_rank <= 64 and every slice width is a multiple of 128, the delta is
 * accumulated inside a tensor-core GEMM of this library (tcgen05) instead:
 * the shrink writes x A^T into the workspace, and the expand runs as extra K
 * blocks of the base GEMM's accumulator (Vhat . Bhat^T over the distinct
 * adapters of each 128-token tile, v rounded to bf16), so y is written once.
 * The workspace holds lora_workspace_bytes(pool, T, 1) bytes either way.
 * Errors: as lora_apply_slices, plus
 * LORA_ERR_INVALID_ARG for a null or misaligned x/W/y (16 bytes), leading
 * dimensions not multiples of 8 or too small, or a meta not built for this
 * dense pool, LORA_ERR_UNSUPPORTED for a MoE pool or when cuBLASLt offers no
 * algorithm, LORA_ERR_CUDA on a cuBLASLt error. */
LORA_API lora_status_t lora_linear_apply(const lora_pool_t *pool, const lora_meta_t *meta, const void *x,
                                         int64_t ldx, const void *W, int64_t ldw, const void *bias, void *y,
                                         int64_t ldy, void *workspace, size_t ws_bytes, void *stream);

/* Inkling sink experts between their two LoRA-wrapped linear layers (Inkling
 * LoRA PR report, InklingSinkExpertsLinear.forward and _gamma_expand).  With
 * W = n_experts * d_mlp, gate_up is the w13 output [T][ld_gate_up] bf16
 * (base + LoRA delta: gate in columns [0, W), up in [W, 2W)), gammas is
 * [T][ld_gammas] fp32 (one factor per token and expert) and h is the w2 input
 * [T][ld_h] bf16:
 *   h[t][c] = bf16( bf16( bf16(silu(gate[t][c])) * up[t][c] ) * gammas[t][c / d_mlp] )
 * The caller owns every buffer (device memory); asynchronous on the stream.
 * Errors (synchronous): LORA_ERR_INVALID_ARG for a null or misaligned pointer
 * (gate_up and h 16-byte aligned, gammas 4-byte aligned), T < 0,
 * n_experts < 1, d_mlp < 1, W not a multiple of 8, ld_gate_up < 2W or not a
 * multiple of 8, ld_h < W or not a multiple of 8, ld_gammas < n_experts. */
LORA_API lora_status_t lora_sink_experts_act(const void *gate_up, int64_t ld_gate_up, const float *gammas,
                                             int64_t ld_gammas, int32_t T, int32_t n_experts, int32_t d_mlp,
                                             void *h, int64_t ld_h, void *stream);

/* Kernel selection for lora_apply_slices / lora_moe_apply (process-wide):
 * 0 = automatic (tcgen05 for long contiguous runs of a rank-64 dense pool;
 *     the fused decode kernel -- one thread-block cluster per adapter slot,
 *     shrink, on-chip reduction and expand in one launch -- for dense
 *     batches of a few rows per slot; for a MoE batch with
 *     T*top_k*8 <= num_experts*max_loras the kernel of
 *     lora_moe_apply_blocks over the metadata's 16-row tiles (one
 *     thread-block cluster per (adapter, expert) key); otherwise the split
 *     shrink/expand kernels when the workspace holds their region, else the
 *     one-pass cluster kernel, else the persistent split-K kernel),
 * 1 = always the persistent split-K kernel,
 * 2 = like 0 but the one-pass cluster kernel before the split kernels
 *     (and neither the fused decode kernel nor the MoE block kernel),
 * 3 = like 0 without the fused decode kernel and the MoE block kernel
 *     (the split 16-row-tile kernels at every MoE batch size),
 * 4 = like 0, with the per-pair schedule (lora_moe_align_padded with
 *     block_m 1, then lora_moe_apply_blocks) for every MoE batch it supports,
 * 5 = like 0, with the kernel of lora_moe_apply_blocks run over the
 *     metadata's 16-row tiles (one thread-block cluster per tile) for every
 *     MoE batch it supports,
 * 6 = like 0, with lora_linear_apply as this library's tcgen05 GEMM that
 *     takes the delta into its accumulator (see lora_linear_apply),
 * 7 = like 0, with the fused decode kernel for batches of up to 32 rows per
 *     slot on average (0 stops at 16, past which the split kernels measured
 *     faster),
 * 8 = like 0, with the split expand on warp-level MMAs (mma.sync) where 0
 *     runs it on tcgen05 (every slice width a multiple of 128, rank <= 64).
 * For tests and tuning. */
LORA_API void lora_set_kernel_policy(int32_t policy);

/* Number of kernel launches this library has issued since it was loaded
 * (all pools, all devices; host-side counter, launches captured into a CUDA
 * graph count once at capture).  A diagnostic: never fails. */
LORA_API unsigned long long lora_kernel_launch_count(void);

/* The cudaError_t value of the last CUDA runtime call that made a library
 * call return LORA_ERR_CUDA (0 if none yet; process-wide, not cleared).
 * A diagnostic: never fails. */
LORA_API int32_t lora_last_cuda_error(void);

/* Static string naming a status code. */
LORA_API const char *lora_status_string(lora_status_t s);

#ifdef __cplusplus
}
#endif
#endif /* LORA_GB300_H */
