// Block-padded per-adapter MoE alignment (the padded output format of
// vLLM's moe_lora_align_block_size, used by FusedMoEWithLoRA with
// sorted_token_ids_lora / expert_ids_lora viewed as (max_loras, -1) and
// num_tokens_post_padded_lora), derived on the device from the unpadded
// metadata of lora_build_meta: for adapter a, the pairs of each key
// (a, e) in ascending e, each run padded with the sentinel T*K to a
// multiple of block_m.  One CTA per adapter.
#include <string.h>

#include "lora_internal.cuh"

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) moe_align_padded_kernel(const int32_t *sorted, const int32_t *key_count,
                                                                    const int32_t *key_offset, int E, int P,
                                                                    int block_m, int cap, int32_t *out_sorted,
                                                                    int32_t *out_expert, int32_t *npp) {
    __shared__ int s_blocks[kThreads];
    __shared__ int s_warp[kThreads / 32 + 1];
    const int a = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = cap / block_m;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the metadata build is complete
    asm volatile("griddepcontrol.launch_dependents;");
    // this thread's contiguous range of experts
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int mine = 0;
    for (int e = e0; e < e1; ++e) mine += (key_count[a * E + e] + block_m - 1) / block_m;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            const int v = s_warp[w];
            s_warp[w] = run;
            run += v;
        }
        s_warp[kThreads / 32] = run;
    }
    __syncthreads();
    s_blocks[tid] = s_warp[warp] + incl - mine;  // first block of this thread's experts
    const int total = s_warp[kThreads / 32];
    if (tid == 0) npp[a] = total * block_m;
    int32_t *os = out_sorted + (long long)a * cap;
    int32_t *oe = out_expert + (long long)a * nb;
    // sentinels / -1 everywhere, then the experts' runs (disjoint per thread)
    for (int i = total * block_m + tid; i < cap; i += kThreads) os[i] = P;
    for (int b = total + tid; b < nb; b += kThreads) oe[b] = -1;
    int blk = s_blocks[tid];
    for (int e = e0; e < e1; ++e) {
        const int c = key_count[a * E + e];
        const int nbk = (c + block_m - 1) / block_m;
        const int src = key_offset[a * E + e];
        for (int i = 0; i < nbk * block_m; ++i) os[blk * block_m + i] = i < c ? sorted[src + i] : P;
        for (int b = 0; b < nbk; ++b) oe[blk + b] = e;
        blk += nbk;
    }
}

}  // namespace

lora_status_t lora_moe_align_launch(const lora_pool_t *pool, const lora_meta_t *meta, int32_t block_m, int32_t cap,
                                    int32_t *d_sorted, int32_t *d_expert, int32_t *d_npp, cudaStream_t s) {
    const int E = pool->desc.num_experts, L = pool->desc.max_loras;
    const long long P = (long long)meta->T * meta->top_k;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)L, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, moe_align_padded_kernel, (const int32_t *)meta->sorted,
                                     (const int32_t *)meta->key_count, (const int32_t *)meta->key_offset, E, (int)P,
                                     (int)block_m, (int)cap, d_sorted, d_expert, d_npp));
    lora_note_launch();
    return LORA_OK;
}

extern "C" lora_status_t lora_moe_align_padded(const lora_pool_t *pool, const lora_meta_t *meta, int32_t block_m,
                                               int32_t cap, int32_t *d_sorted, int32_t *d_expert,
                                               int32_t *d_npp, void *stream) {
    if (!pool || !meta || !d_sorted || !d_expert || !d_npp) return LORA_ERR_INVALID_ARG;
    if (!pool->is_moe || meta->mode != 1) return LORA_ERR_UNSUPPORTED;
    if (block_m < 1 || cap < block_m || cap % block_m) return LORA_ERR_INVALID_ARG;
    const int E = pool->desc.num_experts;
    const long long P = (long long)meta->T * meta->top_k;
    // worst case for one adapter: every pair plus block_m - 1 padding per expert
    if ((long long)cap < P + (long long)E * (block_m - 1)) return LORA_ERR_CAPACITY;
    return lora_moe_align_launch(pool, meta, block_m, cap, d_sorted, d_expert, d_npp, (cudaStream_t)stream);
}
