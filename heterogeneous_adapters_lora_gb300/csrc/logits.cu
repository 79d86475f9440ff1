// lm_head with LoRA end to end: LogitsProcessorWithLoRA._get_logits of the
// vLLM LoRA layer page (reindex the gathered logits with
// sharded_to_full_mapping, add_lora_logits with scale 1.0, keep the first
// vocab_size columns) and the muP multiplier of the Inkling report's
// _lora_forward (base + LoRA logits, all multiplied by 1/mup_multiplier).
//
//   1. logits_reindex_kernel: out[t][i] = bf16(mup * in[t][map[i]]), i < V
//   2. the dense LoRA apply on out with every delta multiplied by mup
#include <string.h>

#include "lora_internal.cuh"

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) logits_reindex_kernel(const uint16_t *in, long long ld_in, int in_cols,
                                                                  const int32_t *map, uint16_t *out,
                                                                  long long ld_out, int V, float mup,
                                                                  int *status) {
    const int t = blockIdx.y;
    const int i0 = (blockIdx.x * kThreads + threadIdx.x) * 8;
    if (i0 >= V) return;
    const uint16_t *row = in + (long long)t * ld_in;
    float v[8];
    int bad = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[k] = 0.f;
        const int i = i0 + k;
        if (i < V) {
            int src = map ? map[i] : i;
            if (src < 0 || src >= in_cols) {
                bad = 1;
                src = 0;
            }
            v[k] = mup * __uint_as_float((uint32_t)row[src] << 16);
        }
    }
    if (bad) atomicExch(status, (int)LORA_ERR_DEVICE_INDEX);
    uint16_t *orow = out + (long long)t * ld_out + i0;
    if (i0 + 8 <= V) {
        uint4 w;
        __nv_bfloat162 h;
        h = __floats2bfloat162_rn(v[0], v[1]); w.x = *(uint32_t *)&h;
        h = __floats2bfloat162_rn(v[2], v[3]); w.y = *(uint32_t *)&h;
        h = __floats2bfloat162_rn(v[4], v[5]); w.z = *(uint32_t *)&h;
        h = __floats2bfloat162_rn(v[6], v[7]); w.w = *(uint32_t *)&h;
        *(uint4 *)orow = w;
    } else {
        for (int k = 0; i0 + k < V; ++k) {
            const __nv_bfloat16 b = __float2bfloat16_rn(v[k]);
            orow[k] = *(const uint16_t *)&b;
        }
    }
}

}  // namespace

extern "C" lora_status_t lora_logits_apply(const lora_pool_t *pool, const lora_meta_t *meta, const void *hidden,
                                           int64_t ld_h, const void *logits_in, int64_t ld_in, int32_t in_cols,
                                           const int32_t *mapping, void *logits_out, int64_t ld_out,
                                           int32_t vocab_size, float mup, void *workspace, size_t ws_bytes,
                                           void *stream) {
    if (!pool || !meta || !logits_in || !logits_out) return LORA_ERR_INVALID_ARG;
    if (pool->is_moe || pool->desc.n_slices != 1) return LORA_ERR_UNSUPPORTED;
    const int width = pool->desc.out_dims[0];
    if (vocab_size < 1 || vocab_size > width || vocab_size > LORA_MAX_VOCAB) return LORA_ERR_SHAPE;
    if (in_cols < 1 || in_cols > ld_in || (!mapping && in_cols < vocab_size)) return LORA_ERR_SHAPE;
    if (ld_out < width || ld_out % 8 || !lora_aligned16(logits_out)) return LORA_ERR_INVALID_ARG;
    if (meta->mode != 0) return LORA_ERR_INVALID_ARG;
    const int T = meta->T;
    if (T == 0) return LORA_OK;
    cudaStream_t s = (cudaStream_t)stream;
    dim3 grid((unsigned)lora_ceil_div(lora_ceil_div(vocab_size, 8), kThreads), (unsigned)T, 1);
    logits_reindex_kernel<<<grid, kThreads, 0, s>>>((const uint16_t *)logits_in, ld_in, in_cols, mapping,
                                                    (uint16_t *)logits_out, ld_out, vocab_size, mup,
                                                    pool->d_status);
    LORA_CUDA_TRY(cudaGetLastError());
    lora_note_launch();
    return lora_dense_apply(pool, meta, hidden, ld_h, logits_out, ld_out, workspace, ws_bytes, mup, s);
}
