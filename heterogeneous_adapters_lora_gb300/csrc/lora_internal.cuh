// Internal definitions shared by the CUDA translation units of liblora_gb300.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_gb300.h"

// Tensor descriptors: a dense pool has one A/B pair per output slice; a MoE
// pool has one pair per w13 slice followed by the w2 pair.
#define LORA_MAX_TENSORS (LORA_MAX_SLICES + 1)
#define LORA_MAX_KEYS 6144

struct lora_pool {
    lora_pool_desc_t desc;
    int device;
    int num_sms;
    int is_moe;
    int R8;                           // max_rank rounded up to a multiple of 8
    int n_tensors;
    // per tensor: A is [slot][a_experts][R][a_in], B is [slot][b_experts][b_out][rs]
    // with rs = ceil8(rank of the slot) (compact rows, zero-padded to 16 bytes)
    uint16_t *A[LORA_MAX_TENSORS];
    uint16_t *B[LORA_MAX_TENSORS];
    int32_t a_in[LORA_MAX_TENSORS];
    int32_t a_experts[LORA_MAX_TENSORS];
    int32_t b_out[LORA_MAX_TENSORS];
    int32_t b_experts[LORA_MAX_TENSORS];
    int64_t a_slot_elems[LORA_MAX_TENSORS];  // capacity of one slot of A
    int64_t b_slot_elems[LORA_MAX_TENSORS];  // capacity of one slot of B
    int32_t *d_rank;
    float *d_scale;
    int32_t *d_enabled;
    int32_t *d_status;
    void *d_base;
    size_t bytes;
    int32_t *h_rank;                  // host mirror of the rank table
    // dense pools of max_rank <= 64: TMA maps of every slice's B for each
    // compact row length rs = 8, 16, .., 64 ([slice][rs/8 - 1], device
    // memory), 3D over (rank, output row, slot); null when not built
    CUtensorMap *d_bmaps;
    // pools of max_rank <= 64 (dense and MoE): TMA maps of every tensor's B
    // for each compact row length ([tensor][rs/8 - 1]), 3D over (rank, row =
    // expert * out + output, slot), boxes of 8 ranks x 128 rows without
    // swizzle (one column of 8-row x 16-byte core matrices); null when not built
    CUtensorMap *d_kmaps;
};

// ------------------------------------------------------------ device helpers

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Shared-window address of a shared-memory pointer.  Aligning a dynamic
// shared buffer by adding (pad from this address) to the pointer keeps the
// compiler's knowledge that it points to shared memory; a round trip through
// an integer would turn every access through it into a generic one.
__device__ __forceinline__ uint32_t smem_u32_of(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------ host helpers

// Last CUDA runtime error a library call returned LORA_ERR_CUDA for
// (lora_last_cuda_error reads it).
void lora_note_cuda_error(cudaError_t e);

#define LORA_CUDA_TRY(expr)                         \
    do {                                            \
        cudaError_t _e = (expr);                    \
        if (_e != cudaSuccess) {                    \
            lora_note_cuda_error(_e);               \
            return LORA_ERR_CUDA;                   \
        }                                           \
    } while (0)

static inline int lora_ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
static inline int lora_round8(int x) { return (x + 7) & ~7; }
static inline bool lora_aligned16(const void *p) { return (((uintptr_t)p) & 15u) == 0; }

// Launch the metadata kernel (meta.cu).
lora_status_t lora_launch_build_meta(const lora_pool_t *pool, const int32_t *d_idx, int32_t T,
                                     const int32_t *d_topk, int32_t top_k, lora_meta_t *meta,
                                     cudaStream_t stream);

// One grouped LoRA problem (a dense layer, or one MoE projection) as the
// compute kernels see it.  Rows are the sorted entries of the metadata.
struct LoraProblem {
    int n_slices, in_dim, E, row_div, R, T, rows, n_keys;
    int out_w[LORA_MAX_SLICES], out_off[LORA_MAX_SLICES];
    const uint16_t *A[LORA_MAX_SLICES];
    long long A_ss[LORA_MAX_SLICES], A_es[LORA_MAX_SLICES];
    const uint16_t *B[LORA_MAX_SLICES];
    long long B_ss[LORA_MAX_SLICES];
    int B_shared[LORA_MAX_SLICES];
    const int32_t *rank;
    const float *scale;
    const lora_meta_t *meta;
    const int32_t *tile_row0, *tile_keyn;  // tile list the kernel walks
    int count_idx;                          // meta counter holding its length
    const uint16_t *in;
    long long ld_in;
    uint16_t *out;
    long long ld_out;
    const float *row_w;
    int *status;
    int spin_limit;
    float post_scale;
    int shrink_only;                        // split path: launch the shrink alone
    int *nc_out;                            // ... and report its hidden chunk count here
    int tok_dedup;                          // MoE with A of expert dimension 1: shrink once per token
    int kmap_base;                          // first pool tensor of the problem's slices (d_kmaps index / 8)
};

// Cluster kernel (cluster.cu): launches and sets *launched when the shape
// fits its shared-memory plan; otherwise leaves *launched false.
lora_status_t lora_cluster_apply(const lora_pool_t *pool, const LoraProblem &pr, cudaStream_t s,
                                 bool *launched);

// Host-side count of kernel launches made by this library (all devices).
void lora_note_launch();

// Kernel selection policy (0 = automatic: the fused decode kernel, else the
// split shrink/expand kernels when the shapes fit; 1 = persistent split-K
// kernel only; 2 = cluster kernel preferred; 3 = automatic without the fused
// decode kernel).
extern int g_lora_kernel_policy;

// 2D bf16 tensor map over rows x cols (row stride in elements), optional
// 128-byte swizzle (sgmv.cu).
bool lora_make_tmap_2d(CUtensorMap *m, const void *base, long long cols, long long rows, long long stride,
                       int box_cols, int box_rows, bool swizzle128);

// 3D bf16 tensor map over a row-major [rows][cols] matrix (cols % 64 == 0)
// that lands a box of box_rows rows x box_chunks 128-byte column chunks in
// shared memory chunk-major: for each chunk, the rows as 128-byte lines in
// the 128-byte swizzle (sgmv.cu).
// 3D bf16 map over a B tensor stored compactly per slot: dims {rs, rows,
// slots}, slot stride slot_elems elements, box {64, 128, 1}, 128-byte swizzle
// (columns past rs read as zero).
bool lora_make_tmap_b3d(CUtensorMap *m, const void *base, int rs, int rows, int slots, long long slot_elems);
// The same view with boxes of 8 ranks x 128 rows and no swizzle.
bool lora_make_tmap_bk(CUtensorMap *m, const void *base, int rs, long long rows, int slots, long long slot_elems);
bool lora_make_tmap_a_chunks(CUtensorMap *m, const void *base, long long rows, long long cols, int box_rows,
                             int box_chunks);

// Split shrink/expand kernels (bgmv.cu): workspace bytes and launcher.
size_t lora_split_ws_bytes(int n_slices, int in_dim, int R, int rows, int max_tiles);
// tickets: 4 ints of the workspace's zeroed control words (left zero again).
lora_status_t lora_split_apply(const lora_pool_t *pool, const LoraProblem &pr, void *ws, size_t ws_bytes,
                               int *tickets, cudaStream_t s, bool *launched);

// Tensor-core SGMV (sgmv.cu) for long contiguous runs of a dense pool.
bool lora_sgmv_eligible(const lora_pool_t *pool);
size_t lora_sgmv_ws_bytes(const lora_pool_t *pool, int rows);
lora_status_t lora_sgmv_apply(const lora_pool_t *pool, const lora_meta_t *meta, const void *x, int64_t ldx,
                              void *y, int64_t ldy, void *V, int spin_limit, int num_sms, float post_scale,
                              cudaStream_t s);

// Fused decode kernel (fused.cu): one thread-block cluster per adapter slot,
// shrink, DSMEM reduction and expand in one launch, no workspace.  Launches
// and sets *launched when the batch and pool fit its plan.
bool lora_fused_eligible(const lora_pool_t *pool, int T);
// With d_idx (batch mode) the kernel also builds the batch metadata into
// meta (as lora_build_meta would, T rows) in the same launch, and the slot
// clusters find their rows in d_idx; without it they read meta.
lora_status_t lora_fused_apply(const lora_pool_t *pool, const lora_meta_t *meta, const int32_t *d_idx, int32_t T,
                               const void *x, int64_t ldx, void *y, int64_t ldy, float post_scale, int spin_limit,
                               cudaStream_t s, bool *launched);

// Dense apply shared by lora_apply_slices and lora_logits_apply (grouped.cu).
lora_status_t lora_dense_apply(const lora_pool_t *pool, const lora_meta_t *meta, const void *x, int64_t ldx,
                               void *y, int64_t ldy, void *workspace, size_t ws_bytes, float post_scale,
                               cudaStream_t s);

// Block-padded MoE alignment (moe_align.cu), launched with programmatic
// dependent launch after a metadata build; arguments checked by the caller.
lora_status_t lora_moe_align_launch(const lora_pool_t *pool, const lora_meta_t *meta, int32_t block_m, int32_t cap,
                                    int32_t *d_sorted, int32_t *d_expert, int32_t *d_npp, cudaStream_t s);
// Per-block MoE-LoRA over that alignment (moe_block.cu): whether the kernel
// takes projection `which` of the pool, and its launch (arguments checked).
bool lora_moe_block_supported(const lora_pool_t *pool, int which);
lora_status_t lora_moe_block_launch(const lora_pool_t *pool, const lora_meta_t *meta, int32_t which, const void *in,
                                    int64_t ld_in, const float *topk_w, void *out, int64_t ld_out,
                                    const int32_t *d_sorted, const int32_t *d_expert, const int32_t *d_npp,
                                    int32_t block_m, int32_t cap, cudaStream_t s);
// The same kernel over the 16-row tiles of the metadata (one block per tile;
// in the sparse-occupancy regime a tile is an (adapter, expert) key's few pairs).
lora_status_t lora_moe_tile_launch(const lora_pool_t *pool, const lora_meta_t *meta, int32_t which, const void *in,
                                   int64_t ld_in, const float *topk_w, void *out, int64_t ld_out, cudaStream_t s);

// The scratch part of an apply workspace (past its control words); false
// if the workspace is null, misaligned or too small to carve.
bool lora_ws_data(void *workspace, size_t ws_bytes, char **data, size_t *data_bytes);

// The shrink of a dense layer alone, for lora_linear_apply: unscaled fp32
// sums of x A^T over hidden chunks, part[nc][n_slices][T][r8], in the
// workspace's scratch past its first head_bytes (a multiple of 256).  With
// *sorted_rows = 1 (the split shrink), row i of a slice is the metadata's
// sorted row i; otherwise (the atomic shrink, nc = 1, r8 = max_rank) row t
// is token t.
lora_status_t lora_dense_shrink(const lora_pool_t *pool, const lora_meta_t *meta, const void *x, int64_t ldx,
                                void *workspace, size_t ws_bytes, size_t head_bytes, cudaStream_t s, float **part,
                                int *nc, int *r8, int *sorted_rows);
