// Inkling sink experts between their two LoRA-wrapped linear layers (Inkling
// LoRA PR report, InklingSinkExpertsLinear.forward and _gamma_expand): the w13
// output gate_up [T][2 * n * d_mlp] (base + LoRA delta, bf16) is split in
// halves, h = SiLU(gate) * up is scaled per column by the gamma of the column's
// expert (column c belongs to expert c / d_mlp) and rounded to bf16, the input
// of the w2 layer.  Rounding follows the page's bf16 tensors: SiLU(gate) and
// SiLU(gate) * up are bf16, the gamma factor is fp32, the result is bf16.
//
// HBM-bound elementwise work: 8 columns per thread (16-byte loads and
// stores), grid-stride over T x n*d_mlp / 8.  Launched with programmatic
// stream serialization between the two layers' LoRA kernels: it starts while
// the w13 expand drains and lets the w2 shrink fetch its weights meanwhile.
#include <string.h>

#include <atomic>

#include "lora_internal.cuh"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_round(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

__global__ void __launch_bounds__(kThreads) sink_act_kernel(const uint16_t *__restrict__ gu, long long ld_gu,
                                                           const float *__restrict__ gammas, long long ld_g,
                                                           int T, int n_experts, int d_mlp,
                                                           uint16_t *__restrict__ h, long long ld_h) {
    const long long W = (long long)n_experts * d_mlp;
    const long long V = W / 8;
    const long long total = (long long)T * V;
    // the next kernel may start its prologue; it waits for this grid's
    // completion before it reads h
    asm volatile("griddepcontrol.launch_dependents;");
    // gate_up is complete once the kernel before this one has finished
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < total;
         i += (long long)gridDim.x * kThreads) {
        const long long t = i / V;
        const long long c0 = (i - t * V) * 8;
        // written by the previous kernel: L2 loads, no L1 lines
        const uint4 gv = __ldcg((const uint4 *)(gu + t * ld_gu + c0));
        const uint4 uv = __ldcg((const uint4 *)(gu + t * ld_gu + W + c0));
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
        uint32_t ow[4];
        const float *grow = gammas + t * ld_g;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float r[2];
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const float g = e2 ? bf16hi(gw[q]) : bf16lo(gw[q]);
                const float u = e2 ? bf16hi(uw[q]) : bf16lo(uw[q]);
                const float s = bf16_round(g / (1.0f + expf(-g)));
                const float p = bf16_round(s * u);  // exact product of two bf16 values, then bf16
                const int col = (int)(c0 + 2 * q + e2);
                r[e2] = p * __ldg(grow + col / d_mlp);
            }
            const __nv_bfloat162 b = __floats2bfloat162_rn(r[0], r[1]);
            ow[q] = *(const uint32_t *)&b;
        }
        *(uint4 *)(h + t * ld_h + c0) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
}

std::atomic<int> g_sink_sms[64];  // SM count per device, looked up once

}  // namespace

extern "C" lora_status_t lora_sink_experts_act(const void *gate_up, int64_t ld_gate_up, const float *gammas,
                                               int64_t ld_gammas, int32_t T, int32_t n_experts, int32_t d_mlp,
                                               void *h, int64_t ld_h, void *stream) {
    if (T < 0 || n_experts < 1 || d_mlp < 1) return LORA_ERR_INVALID_ARG;
    const long long W = (long long)n_experts * d_mlp;
    if (W % 8 || ld_gate_up < 2 * W || ld_gate_up % 8 || ld_h < W || ld_h % 8 || ld_gammas < n_experts)
        return LORA_ERR_INVALID_ARG;
    if (T == 0) return LORA_OK;
    if (!gate_up || !gammas || !h || !lora_aligned16(gate_up) || !lora_aligned16(h) || ((uintptr_t)gammas & 3))
        return LORA_ERR_INVALID_ARG;
    int dev = 0;
    LORA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return LORA_ERR_INVALID_ARG;
    int n_sms = g_sink_sms[dev].load(std::memory_order_relaxed);
    if (!n_sms) {
        LORA_CUDA_TRY(cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev));
        n_sms = n_sms > 0 ? n_sms : 1;
        g_sink_sms[dev].store(n_sms, std::memory_order_relaxed);
    }
    const long long vecs = (long long)T * (W / 8);
    long long grid = (vecs + kThreads - 1) / kThreads;
    const long long cap = (long long)n_sms * 8;
    if (grid > cap) grid = cap;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = (cudaStream_t)stream;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, sink_act_kernel, (const uint16_t *)gate_up, (long long)ld_gate_up,
                                     gammas, (long long)ld_gammas, (int)T, (int)n_experts, (int)d_mlp,
                                     (uint16_t *)h, (long long)ld_h));
    lora_note_launch();
    return LORA_OK;
}
