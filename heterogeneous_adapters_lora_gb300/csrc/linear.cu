// The full LoRA linear layer (vLLM LoRA layer pages, BaseLinearLayerWithLoRA:
// the base layer's output, then the LoRA delta added in place):
//   y = x W^T + bias + delta
// The base GEMM is a plain library GEMM (cuBLASLt, bf16 in, fp32 accumulate,
// bias epilogue, no workspace); the delta is the library's own apply.  The
// delta is a second pass over y (read + write), not fused into the GEMM
// epilogue.
#include <cublasLt.h>
#include <string.h>

#include "lora_internal.cuh"

namespace {

cublasLtHandle_t g_lt[64];

#define LT_TRY(x)                                        \
    do {                                                 \
        if ((x) != CUBLAS_STATUS_SUCCESS) return LORA_ERR_CUDA; \
    } while (0)

struct LtDesc {
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    ~LtDesc() {
        if (pref) cublasLtMatmulPreferenceDestroy(pref);
        if (c) cublasLtMatrixLayoutDestroy(c);
        if (b) cublasLtMatrixLayoutDestroy(b);
        if (a) cublasLtMatrixLayoutDestroy(a);
        if (op) cublasLtMatmulDescDestroy(op);
    }
};

// y[T][ldy] (row-major, bf16) = x[T][ldx] W[O][ldw]^T + bias[O]; in column-major
// terms Y (O x T) = op(W) (O x H) X (H x T) with op = transpose.
lora_status_t base_gemm(int dev, const void *x, int64_t ldx, const void *W, int64_t ldw, const void *bias,
                        void *y, int64_t ldy, int T, int H, int O, cudaStream_t s) {
    if (!g_lt[dev]) LT_TRY(cublasLtCreate(&g_lt[dev]));
    LtDesc d;
    LT_TRY(cublasLtMatmulDescCreate(&d.op, CUBLAS_COMPUTE_32F, CUDA_R_32F));
    const cublasOperation_t tA = CUBLAS_OP_T, tB = CUBLAS_OP_N;
    LT_TRY(cublasLtMatmulDescSetAttribute(d.op, CUBLASLT_MATMUL_DESC_TRANSA, &tA, sizeof(tA)));
    LT_TRY(cublasLtMatmulDescSetAttribute(d.op, CUBLASLT_MATMUL_DESC_TRANSB, &tB, sizeof(tB)));
    if (bias) {
        const cublasLtEpilogue_t ep = CUBLASLT_EPILOGUE_BIAS;
        const cudaDataType_t bt = CUDA_R_16BF;
        LT_TRY(cublasLtMatmulDescSetAttribute(d.op, CUBLASLT_MATMUL_DESC_EPILOGUE, &ep, sizeof(ep)));
        LT_TRY(cublasLtMatmulDescSetAttribute(d.op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof(bias)));
        LT_TRY(cublasLtMatmulDescSetAttribute(d.op, CUBLASLT_MATMUL_DESC_BIAS_DATA_TYPE, &bt, sizeof(bt)));
    }
    LT_TRY(cublasLtMatrixLayoutCreate(&d.a, CUDA_R_16BF, H, O, ldw));
    LT_TRY(cublasLtMatrixLayoutCreate(&d.b, CUDA_R_16BF, H, T, ldx));
    LT_TRY(cublasLtMatrixLayoutCreate(&d.c, CUDA_R_16BF, O, T, ldy));
    LT_TRY(cublasLtMatmulPreferenceCreate(&d.pref));
    const size_t ws = 0;
    LT_TRY(cublasLtMatmulPreferenceSetAttribute(d.pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws, sizeof(ws)));
    cublasLtMatmulHeuristicResult_t heur;
    int n = 0;
    LT_TRY(cublasLtMatmulAlgoGetHeuristic(g_lt[dev], d.op, d.a, d.b, d.c, d.c, d.pref, 1, &heur, &n));
    if (n < 1) return LORA_ERR_UNSUPPORTED;
    const float alpha = 1.0f, beta = 0.0f;
    LT_TRY(cublasLtMatmul(g_lt[dev], d.op, &alpha, W, d.a, x, d.b, &beta, y, d.c, y, d.c, &heur.algo, nullptr, 0,
                          s));
    return LORA_OK;
}

}  // namespace

extern "C" lora_status_t lora_linear_apply(const lora_pool_t *pool, const lora_meta_t *meta, const void *x,
                                           int64_t ldx, const void *W, int64_t ldw, const void *bias, void *y,
                                           int64_t ldy, void *workspace, size_t ws_bytes, void *stream) {
    if (!pool || !meta) return LORA_ERR_INVALID_ARG;
    if (pool->is_moe) return LORA_ERR_UNSUPPORTED;
    const lora_pool_desc_t &d = pool->desc;
    int O = 0;
    for (int j = 0; j < d.n_slices; ++j) O += d.out_dims[j];
    if (!x || !W || !y || !lora_aligned16(x) || !lora_aligned16(W) || !lora_aligned16(y) || ldx % 8 || ldw % 8 ||
        ldy % 8 || ldx < d.in_dim || ldw < d.in_dim || ldy < O || (bias && ((uintptr_t)bias & 1)))
        return LORA_ERR_INVALID_ARG;
    if (meta->T == 0) return LORA_OK;
    int dev = -1;
    LORA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != pool->device || dev < 0 || dev >= 64) return LORA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    lora_status_t st = base_gemm(dev, x, ldx, W, ldw, bias, y, ldy, meta->T, d.in_dim, O, s);
    if (st != LORA_OK) return st;
    return lora_apply_slices(pool, meta, x, ldx, y, ldy, workspace, ws_bytes, stream);
}
