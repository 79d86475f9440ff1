// Internal definitions shared by the CUDA translation units of liblora_gb300.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_gb300.h"

// Tensor descriptors: a dense pool has one A/B pair per output slice; a MoE
// pool has one pair per w13 slice followed by the w2 pair.
#define LORA_MAX_TENSORS (LORA_MAX_SLICES + 1)
#define LORA_MAX_KEYS 12288

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

#define LORA_CUDA_TRY(expr)                         \
    do {                                            \
        cudaError_t _e = (expr);                    \
        if (_e != cudaSuccess) return LORA_ERR_CUDA; \
    } while (0)

static inline int lora_ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
static inline int lora_round8(int x) { return (x + 7) & ~7; }
static inline bool lora_aligned16(const void *p) { return (((uintptr_t)p) & 15u) == 0; }

// Launch the metadata kernel (meta.cu).
lora_status_t lora_launch_build_meta(const lora_pool_t *pool, const int32_t *d_idx, int32_t T,
                                     const int32_t *d_topk, int32_t top_k, lora_meta_t *meta,
                                     cudaStream_t stream);
