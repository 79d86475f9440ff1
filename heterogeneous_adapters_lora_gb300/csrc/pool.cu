// Stacked adapter pool: create / set / reset (create_lora_weights, set_lora
// and reset_lora of the vLLM LoRA layer pages), status word and metadata
// buffer binding.
//
// Device layout (one allocation).  Per tensor i (a dense slice, a w13 slice
// or w2):
//   A_i: [L][a_experts][R][a_in]        rows k >= rank are zero
//   B_i: [L][b_experts][b_out][R8]      capacity; a slot of rank r stores
//        its B compactly as [b_experts][b_out][rs], rs = ceil8(r), so the
//        kernels read exactly rows of rs elements (16-byte multiples)
//   then rank[L] int32, scale[L] fp32, enabled[L] int32, status int32.
#include <stdlib.h>
#include <string.h>

#include "lora_internal.cuh"

__global__ void lora_set_tables_kernel(int32_t *rank, float *scale, int32_t *enabled, int slot,
                                       int r, float s, int en) {
    rank[slot] = r;
    scale[slot] = s;
    enabled[slot] = en;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static lora_status_t validate_desc(const lora_pool_desc_t *d) {
    if (d->max_loras < 1 || d->max_rank < 1 || d->max_rank > LORA_MAX_RANK)
        return LORA_ERR_INVALID_ARG;
    if (d->num_experts == 0) {
        if (d->n_slices < 1 || d->n_slices > LORA_MAX_SLICES) return LORA_ERR_SHAPE;
        if (d->in_dim < 8 || d->in_dim % 8) return LORA_ERR_SHAPE;
        for (int j = 0; j < d->n_slices; ++j)
            if (d->out_dims[j] < 8 || d->out_dims[j] % 8) return LORA_ERR_SHAPE;
        if (d->is_lm_head && (d->n_slices != 1 || d->out_dims[0] > LORA_MAX_VOCAB))
            return LORA_ERR_SHAPE;
    } else if (d->num_experts > 0) {
        if (d->n_w13_slices < 1 || d->n_w13_slices > 2) return LORA_ERR_SHAPE;
        if (d->d_model < 8 || d->d_model % 8 || d->d_mlp < 8 || d->d_mlp % 8) return LORA_ERR_SHAPE;
        if (d->w13_slice_width < 8 || d->w13_slice_width % 8) return LORA_ERR_SHAPE;
        if (d->shared_outer != 0 && d->shared_outer != 1) return LORA_ERR_INVALID_ARG;
        if ((int64_t)d->max_loras * d->num_experts > LORA_MAX_KEYS) return LORA_ERR_CAPACITY;
    } else {
        return LORA_ERR_INVALID_ARG;
    }
    return LORA_OK;
}

extern "C" lora_status_t lora_pool_create(const lora_pool_desc_t *desc, void *stream,
                                          lora_pool_t **out) {
    if (!desc || !out) return LORA_ERR_INVALID_ARG;
    *out = nullptr;
    lora_status_t st = validate_desc(desc);
    if (st != LORA_OK) return st;
    lora_pool_t *p = (lora_pool_t *)calloc(1, sizeof(lora_pool_t));
    if (!p) return LORA_ERR_NOMEM;
    p->desc = *desc;
    const int L = desc->max_loras, R = desc->max_rank;
    p->R8 = lora_round8(R);
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
        free(p);
        return LORA_ERR_CUDA;
    }
    if (desc->num_experts == 0) {
        p->is_moe = 0;
        p->n_tensors = desc->n_slices;
        for (int j = 0; j < desc->n_slices; ++j) {
            p->a_in[j] = desc->in_dim;
            p->a_experts[j] = 1;
            p->b_out[j] = desc->out_dims[j];
            p->b_experts[j] = 1;
        }
    } else {
        const int E = desc->num_experts, n13 = desc->n_w13_slices;
        const int Eo = desc->shared_outer ? 1 : E;
        p->is_moe = 1;
        p->n_tensors = n13 + 1;
        for (int s = 0; s < n13; ++s) {
            p->a_in[s] = desc->d_model;
            p->a_experts[s] = Eo;
            p->b_out[s] = desc->w13_slice_width;
            p->b_experts[s] = E;
        }
        p->a_in[n13] = desc->d_mlp;
        p->a_experts[n13] = E;
        p->b_out[n13] = desc->d_model;
        p->b_experts[n13] = Eo;
    }
    size_t bytes = 0;
    size_t offA[LORA_MAX_TENSORS], offB[LORA_MAX_TENSORS];
    for (int i = 0; i < p->n_tensors; ++i) {
        p->a_slot_elems[i] = (int64_t)p->a_experts[i] * R * p->a_in[i];
        p->b_slot_elems[i] = (int64_t)p->b_experts[i] * p->b_out[i] * p->R8;
        offA[i] = bytes;
        bytes = align256(bytes + (size_t)L * p->a_slot_elems[i] * 2);
        offB[i] = bytes;
        bytes = align256(bytes + (size_t)L * p->b_slot_elems[i] * 2);
    }
    size_t offRank = bytes;
    bytes = align256(bytes + (size_t)L * 4);
    size_t offScale = bytes;
    bytes = align256(bytes + (size_t)L * 4);
    size_t offEn = bytes;
    bytes = align256(bytes + (size_t)L * 4);
    size_t offStatus = bytes;
    bytes = align256(bytes + 4);
    // TMA maps of B for the tensor-core prefill path (dense, max_rank <= 64)
    const bool maps = !p->is_moe && desc->max_rank <= 64;
    const size_t offMaps = bytes;
    if (maps) bytes = align256(bytes + (size_t)desc->n_slices * 8 * sizeof(CUtensorMap));
    // K-chunk maps of every tensor's B for the tensor-core split expand
    const bool kmaps = desc->max_rank <= 64;
    const size_t offKmaps = bytes;
    if (kmaps) bytes = align256(bytes + (size_t)p->n_tensors * 8 * sizeof(CUtensorMap));
    if (cudaMalloc(&p->d_base, bytes) != cudaSuccess) {
        free(p);
        return LORA_ERR_NOMEM;
    }
    p->bytes = bytes;
    char *base = (char *)p->d_base;
    for (int i = 0; i < p->n_tensors; ++i) {
        p->A[i] = (uint16_t *)(base + offA[i]);
        p->B[i] = (uint16_t *)(base + offB[i]);
    }
    p->d_rank = (int32_t *)(base + offRank);
    p->d_scale = (float *)(base + offScale);
    p->d_enabled = (int32_t *)(base + offEn);
    p->d_status = (int32_t *)(base + offStatus);
    p->h_rank = (int32_t *)calloc((size_t)L, sizeof(int32_t));
    if (!p->h_rank || cudaMemsetAsync(p->d_base, 0, bytes, (cudaStream_t)stream) != cudaSuccess) {
        cudaFree(p->d_base);
        free(p->h_rank);
        free(p);
        return LORA_ERR_CUDA;
    }
    p->d_bmaps = nullptr;
    if (maps) {
        const int ns = desc->n_slices;
        CUtensorMap *h = (CUtensorMap *)calloc((size_t)ns * 8, sizeof(CUtensorMap));
        bool ok = h != nullptr;
        for (int j = 0; ok && j < ns; ++j)
            for (int q = 0; ok && q < 8; ++q)
                ok = lora_make_tmap_b3d(&h[j * 8 + q], p->B[j], 8 * (q + 1), desc->out_dims[j], L, p->b_slot_elems[j]);
        if (ok && cudaStreamSynchronize((cudaStream_t)stream) == cudaSuccess &&
            cudaMemcpy(base + offMaps, h, (size_t)ns * 8 * sizeof(CUtensorMap), cudaMemcpyHostToDevice) == cudaSuccess)
            p->d_bmaps = (CUtensorMap *)(base + offMaps);
        free(h);
    }
    p->d_kmaps = nullptr;
    if (kmaps) {
        const int nt = p->n_tensors;
        CUtensorMap *h = (CUtensorMap *)calloc((size_t)nt * 8, sizeof(CUtensorMap));
        bool ok = h != nullptr;
        for (int i = 0; ok && i < nt; ++i)
            for (int q = 0; ok && q < 8; ++q)
                ok = lora_make_tmap_bk(&h[i * 8 + q], p->B[i], 8 * (q + 1), (long long)p->b_experts[i] * p->b_out[i], L,
                                       p->b_slot_elems[i]);
        if (ok && cudaStreamSynchronize((cudaStream_t)stream) == cudaSuccess &&
            cudaMemcpy(base + offKmaps, h, (size_t)nt * 8 * sizeof(CUtensorMap), cudaMemcpyHostToDevice) == cudaSuccess)
            p->d_kmaps = (CUtensorMap *)(base + offKmaps);
        free(h);
    }
    *out = p;
    return LORA_OK;
}

extern "C" lora_status_t lora_pool_destroy(lora_pool_t *pool) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    cudaError_t f = cudaFree(pool->d_base);
    free(pool->h_rank);
    free(pool);
    return (e == cudaSuccess && f == cudaSuccess) ? LORA_OK : LORA_ERR_CUDA;
}

extern "C" lora_status_t lora_pool_get_desc(const lora_pool_t *pool, lora_pool_desc_t *out) {
    if (!pool || !out) return LORA_ERR_INVALID_ARG;
    *out = pool->desc;
    return LORA_OK;
}

static lora_status_t reset_slot(lora_pool_t *p, int slot, cudaStream_t s) {
    for (int i = 0; i < p->n_tensors; ++i) {
        LORA_CUDA_TRY(cudaMemsetAsync(p->A[i] + (size_t)slot * p->a_slot_elems[i], 0,
                                      (size_t)p->a_slot_elems[i] * 2, s));
        LORA_CUDA_TRY(cudaMemsetAsync(p->B[i] + (size_t)slot * p->b_slot_elems[i], 0,
                                      (size_t)p->b_slot_elems[i] * 2, s));
    }
    lora_set_tables_kernel<<<1, 1, 0, s>>>(p->d_rank, p->d_scale, p->d_enabled, slot, 0, 0.0f, 0);
    LORA_CUDA_TRY(cudaGetLastError());
    lora_note_launch();
    p->h_rank[slot] = 0;
    return LORA_OK;
}

extern "C" lora_status_t lora_reset(lora_pool_t *pool, int32_t slot, void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->desc.max_loras) return LORA_ERR_INDEX;
    return reset_slot(pool, slot, (cudaStream_t)stream);
}

// Copy one adapter tensor pair (per expert) into tensor i of the slot.
//   A src: [experts][rank][a_in]; B src: [experts][b_out][rank]
static lora_status_t copy_pair(lora_pool_t *p, int i, int slot, int rank, int experts,
                               const void *A, const void *B, cudaStream_t s) {
    const int R = p->desc.max_rank;
    const int rs = lora_round8(rank);
    if (A && rank > 0) {
        uint16_t *dst = p->A[i] + (size_t)slot * p->a_slot_elems[i];
        // expert e: rows [0, rank) of [R][a_in]
        LORA_CUDA_TRY(cudaMemcpy2DAsync(dst, (size_t)R * p->a_in[i] * 2, A,
                                        (size_t)rank * p->a_in[i] * 2, (size_t)rank * p->a_in[i] * 2,
                                        (size_t)experts, cudaMemcpyDefault, s));
    }
    if (B && rank > 0) {
        uint16_t *dst = p->B[i] + (size_t)slot * p->b_slot_elems[i];
        // compact rows of rs elements; each of experts*b_out rows copies rank values
        LORA_CUDA_TRY(cudaMemcpy2DAsync(dst, (size_t)rs * 2, B, (size_t)rank * 2, (size_t)rank * 2,
                                        (size_t)experts * p->b_out[i], cudaMemcpyDefault, s));
    }
    return LORA_OK;
}

static lora_status_t finish_set(lora_pool_t *p, int slot, int rank, float scale, cudaStream_t s) {
    lora_set_tables_kernel<<<1, 1, 0, s>>>(p->d_rank, p->d_scale, p->d_enabled, slot, rank, scale, 1);
    LORA_CUDA_TRY(cudaGetLastError());
    lora_note_launch();
    p->h_rank[slot] = rank;
    return LORA_OK;
}

extern "C" lora_status_t lora_set(lora_pool_t *pool, int32_t slot, int32_t rank, float scale,
                                  const void *const *A, const void *const *B, int32_t n,
                                  void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (pool->is_moe) return LORA_ERR_UNSUPPORTED;
    if (slot < 0 || slot >= pool->desc.max_loras) return LORA_ERR_INDEX;
    if (rank < 0 || rank > pool->desc.max_rank) return LORA_ERR_RANK;
    if (n != pool->n_tensors || !A || !B) return LORA_ERR_SHAPE;
    cudaStream_t s = (cudaStream_t)stream;
    lora_status_t st = reset_slot(pool, slot, s);
    if (st != LORA_OK) return st;
    for (int j = 0; j < n; ++j) {
        st = copy_pair(pool, j, slot, rank, 1, A[j], B[j], s);
        if (st != LORA_OK) return st;
    }
    return finish_set(pool, slot, rank, scale, s);
}

extern "C" lora_status_t lora_set_packed(lora_pool_t *pool, int32_t slot, int32_t rank,
                                         float scale, const void *A, const void *B, void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (pool->is_moe) return LORA_ERR_UNSUPPORTED;
    if (slot < 0 || slot >= pool->desc.max_loras) return LORA_ERR_INDEX;
    if (rank < 0 || rank > pool->desc.max_rank) return LORA_ERR_RANK;
    if (!A || !B) return LORA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    lora_status_t st = reset_slot(pool, slot, s);
    if (st != LORA_OK) return st;
    size_t row_off = 0;
    for (int j = 0; j < pool->n_tensors; ++j) {
        const void *Bj = (const char *)B + row_off * (size_t)rank * 2;
        st = copy_pair(pool, j, slot, rank, 1, A, Bj, s);
        if (st != LORA_OK) return st;
        row_off += (size_t)pool->b_out[j];
    }
    return finish_set(pool, slot, rank, scale, s);
}

extern "C" lora_status_t lora_set_moe(lora_pool_t *pool, int32_t slot, int32_t rank, float scale,
                                      const void *const *A, const int32_t *a_experts,
                                      const void *const *B, const int32_t *b_experts, int32_t n,
                                      void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (!pool->is_moe) return LORA_ERR_UNSUPPORTED;
    if (slot < 0 || slot >= pool->desc.max_loras) return LORA_ERR_INDEX;
    if (rank < 0 || rank > pool->desc.max_rank) return LORA_ERR_RANK;
    if (n != pool->n_tensors || !A || !B || !a_experts || !b_experts) return LORA_ERR_SHAPE;
    const int E = pool->desc.num_experts;
    for (int i = 0; i < n; ++i) {
        for (int which = 0; which < 2; ++which) {
            const int got = which ? b_experts[i] : a_experts[i];
            const int want = which ? pool->b_experts[i] : pool->a_experts[i];
            if (got == want) continue;
            // a 1-vs-E confusion on a tensor whose expert dim depends on the
            // shared-outer flag is a layout mismatch; anything else a shape error
            const bool outer = (which == 0 && i < n - 1) || (which == 1 && i == n - 1);
            if (outer && E > 1 && ((got == 1 && want == E) || (got == E && want == 1)))
                return LORA_ERR_LAYOUT;
            return LORA_ERR_SHAPE;
        }
    }
    cudaStream_t s = (cudaStream_t)stream;
    lora_status_t st = reset_slot(pool, slot, s);
    if (st != LORA_OK) return st;
    for (int i = 0; i < n; ++i) {
        // expert dims of A and B may differ (shared-outer): copy them separately
        st = copy_pair(pool, i, slot, rank, pool->a_experts[i], A[i], nullptr, s);
        if (st != LORA_OK) return st;
        st = copy_pair(pool, i, slot, rank, pool->b_experts[i], nullptr, B[i], s);
        if (st != LORA_OK) return st;
    }
    return finish_set(pool, slot, rank, scale, s);
}

extern "C" lora_status_t lora_get_device_status(const lora_pool_t *pool, void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t v = 0;
    LORA_CUDA_TRY(cudaStreamSynchronize(s));
    LORA_CUDA_TRY(cudaMemcpy(&v, pool->d_status, 4, cudaMemcpyDeviceToHost));
    LORA_CUDA_TRY(cudaMemset(pool->d_status, 0, 4));
    return (lora_status_t)v;
}

extern "C" const char *lora_status_string(lora_status_t s) {
    switch (s) {
        case LORA_OK: return "LORA_OK";
        case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG";
        case LORA_ERR_INDEX: return "LORA_ERR_INDEX";
        case LORA_ERR_RANK: return "LORA_ERR_RANK";
        case LORA_ERR_SHAPE: return "LORA_ERR_SHAPE";
        case LORA_ERR_LAYOUT: return "LORA_ERR_LAYOUT";
        case LORA_ERR_NOMEM: return "LORA_ERR_NOMEM";
        case LORA_ERR_CUDA: return "LORA_ERR_CUDA";
        case LORA_ERR_DEVICE_INDEX: return "LORA_ERR_DEVICE_INDEX";
        case LORA_ERR_TIMEOUT: return "LORA_ERR_TIMEOUT";
        case LORA_ERR_CAPACITY: return "LORA_ERR_CAPACITY";
        case LORA_ERR_UNSUPPORTED: return "LORA_ERR_UNSUPPORTED";
    }
    return "LORA_ERR_UNKNOWN";
}

// ------------------------------------------------------------ meta buffers

static size_t meta_layout(int32_t max_rows, int32_t max_keys, size_t off[16]) {
    const int32_t max_tiles = max_rows / LORA_TILE_ROWS + max_keys + 1;
    const int32_t max_ltiles = max_rows / LORA_LTILE_ROWS + max_keys + 1;
    const size_t n[15] = {(size_t)max_rows,   (size_t)max_keys,   (size_t)max_keys + 1,
                          (size_t)max_keys,   (size_t)max_keys + 1, (size_t)max_keys,
                          (size_t)max_tiles,  (size_t)max_tiles,  (size_t)max_tiles,
                          (size_t)max_ltiles, (size_t)max_ltiles, (size_t)max_ltiles,
                          (size_t)max_tiles,  (size_t)max_tiles,  8};
    size_t b = 0;
    for (int i = 0; i < 15; ++i) {
        off[i] = b;
        b = align256(b + n[i] * 4);
    }
    off[15] = b;
    return b;
}

extern "C" size_t lora_meta_bytes(int32_t max_rows, int32_t max_keys) {
    if (max_rows < 0 || max_keys < 1) return 0;
    size_t off[16];
    return meta_layout(max_rows, max_keys, off);
}

extern "C" lora_status_t lora_meta_bind(lora_meta_t *m, void *d_buf, size_t bytes,
                                        int32_t max_rows, int32_t max_keys) {
    if (!m || !d_buf || max_rows < 0 || max_keys < 1 || !lora_aligned16(d_buf))
        return LORA_ERR_INVALID_ARG;
    size_t off[16];
    if (meta_layout(max_rows, max_keys, off) > bytes) return LORA_ERR_CAPACITY;
    char *b = (char *)d_buf;
    memset(m, 0, sizeof(*m));
    m->max_rows = max_rows;
    m->max_keys = max_keys;
    m->max_tiles = max_rows / LORA_TILE_ROWS + max_keys + 1;
    m->max_ltiles = max_rows / LORA_LTILE_ROWS + max_keys + 1;
    m->sorted = (int32_t *)(b + off[0]);
    m->key_count = (int32_t *)(b + off[1]);
    m->key_offset = (int32_t *)(b + off[2]);
    m->group_key = (int32_t *)(b + off[3]);
    m->group_start = (int32_t *)(b + off[4]);
    m->key_group = (int32_t *)(b + off[5]);
    m->tile_group = (int32_t *)(b + off[6]);
    m->tile_row0 = (int32_t *)(b + off[7]);
    m->tile_keyn = (int32_t *)(b + off[8]);
    m->ltile_row0 = (int32_t *)(b + off[9]);
    m->ltile_keyn = (int32_t *)(b + off[10]);
    m->ltile_tok0 = (int32_t *)(b + off[11]);
    m->stile_row0 = (int32_t *)(b + off[12]);
    m->stile_keyn = (int32_t *)(b + off[13]);
    m->counters = (int32_t *)(b + off[14]);
    m->mode = -1;
    return LORA_OK;
}

extern "C" lora_status_t lora_build_meta(const lora_pool_t *pool, const int32_t *d_idx, int32_t T,
                                         const int32_t *d_topk_ids, int32_t top_k,
                                         lora_meta_t *meta, void *stream) {
    if (!pool || !meta || T < 0 || (T > 0 && !d_idx)) return LORA_ERR_INVALID_ARG;
    if (pool->is_moe) {
        if (!d_topk_ids || top_k < 1) return LORA_ERR_INVALID_ARG;
    } else {
        if (d_topk_ids) return LORA_ERR_INVALID_ARG;
        top_k = 1;
    }
    return lora_launch_build_meta(pool, d_idx, T, d_topk_ids, top_k, meta, (cudaStream_t)stream);
}
