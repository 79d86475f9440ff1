// Tensor-core SGMV for long contiguous token runs (prefill): the shrink and
// expand of the multi-tenant LoRA delta on tcgen05 with operands staged by
// TMA and accumulators in tensor memory.
//
// The vLLM LoRA layer pages compute add_shrink (x -> fp32 rank buffer, scale
// 1.0) and add_expand (rank -> out, added into y at the slice offsets).  For a
// group (adapter slot) whose tokens form one contiguous run of >= 64 tokens
// the metadata cuts the run into tiles of up to 128 tokens; per tile:
//
//   shrink:  D[t][k] = sum_h x[t][h] * A_j[a][k][h]   one CTA per (tile, slice j):
//            M = 128 tokens, N = R, K = hidden in blocks of 64, 4-stage TMA ring.
//            Epilogue: v = scale[a] * D, split into bf16 hi + lo (v - hi), so
//            that the expand keeps the fp32 intermediate to ~16 bits.
//   expand:  y[t][off_j + o] += v_hi[t] . B_j[a][o] + v_lo[t] . B_j[a][o]
//            M = 128 tokens, N = 128 outputs, K = R (x2 for hi/lo); the y
//            tile is read by TMA, updated in shared memory and written back
//            by TMA (or row by row for a partial last tile of a run).
//
// Warp roles: warp 0 issues TMA, warp 1 allocates tensor memory and issues
// the MMAs, the other warps run the epilogue (warp w reads the accumulator
// lanes 32*(w%4) .. +31; 4 epilogue warps in the shrink, 8 in the expand,
// where two warps share a lane quarter and split the columns).  Every wait is
// a bounded poll that records LORA_ERR_TIMEOUT in the status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>

#include "lora_internal.cuh"
#include "tc_common.cuh"

namespace {

constexpr int kRows = LORA_LTILE_ROWS;  // 128 tokens per tile (MMA M)
constexpr int kBK = 64;                 // hidden elements per K block (one 128-byte swizzle row)
constexpr int kStages = 8;                 // shrink TMA ring: 8 x (16 KB x + R x 128 B A)
constexpr int kThreads = 192;          // shrink: TMA warp, MMA warp, 4 epilogue warps
constexpr int kEThreads = 320;         // expand: TMA warp, MMA warp, 8 epilogue warps
constexpr int kNY = 3;                 // y tiles in flight in the expand
constexpr int kOT = 128;                // outputs per expand tile (MMA N)
constexpr int kOG = 8;                  // expand tiles per work unit
constexpr uint32_t kTileBytes = kRows * kBK * 2;  // 16 KB: 128 rows x 128 B
constexpr int kVRow = 2 * kBK;          // V row: 64 hi columns, then 64 lo columns

struct alignas(64) ShrinkArgs {
    CUtensorMap tm_x;                    // x [T][H]: box {64, 128}
    CUtensorMap tm_a[LORA_MAX_SLICES];   // A_j [L*R][H]: box {64, R}
    int n_slices, in_dim, R;
    const int32_t *ltile_row0, *ltile_keyn, *ltile_tok0, *counters;
    const float *scale;
    uint16_t *V;                         // [n_slices][rows][2R] bf16: hi | lo
    long long v_slice;                   // elements per slice of V
    int *status;
    int spin_limit;
    float post_scale;
};

struct alignas(64) ExpandArgs {
    CUtensorMap tm_v[LORA_MAX_SLICES];   // V_j [rows][128]: box {64, 128}
    CUtensorMap tm_y;                    // y [T][out]: box {64, 128}
    const CUtensorMap *bmaps;            // the pool's B maps [slice][rs / 8 - 1]: box {64, 128, 1}
    const int32_t *rank;
    int n_slices, R;
    int out_w[LORA_MAX_SLICES], out_off[LORA_MAX_SLICES];
    int grp_start[LORA_MAX_SLICES + 1];  // prefix over slices of ceil(otiles_j / kOG)
    const int32_t *ltile_row0, *ltile_keyn, *ltile_tok0, *counters;
    uint16_t *y;
    long long ld_y;
    int *status;
    int spin_limit;
};

__device__ __forceinline__ void wait_or_flag(uint64_t *bar, uint32_t parity, int limit, int *status) {
    if (!tc::mbar_wait(bar, parity, limit)) atomicExch(status, (int)LORA_ERR_TIMEOUT);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *(const uint32_t *)&v;
}

// ------------------------------------------------------------------ shrink

__global__ void __launch_bounds__(kThreads, 1) sgmv_shrink_kernel(const __grid_constant__ ShrinkArgs p) {
    extern __shared__ __align__(1024) char smem_raw[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], acc_full;
    __shared__ uint32_t s_tmem;
    char *smem = smem_raw + ((1024u - (smem_u32_of(smem_raw) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / p.n_slices, js = blockIdx.x - tile * p.n_slices;  // one slice per CTA
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tile >= p.counters[5]) return;

    const int N = (p.R + 15) & ~15;  // accumulator columns: the ranks of slice js (MMA N: a multiple of 16)
    const uint32_t a_bytes = (uint32_t)p.R * 128;  // the A box: R rows of 64 hidden elements
    const uint32_t stage_bytes = kTileBytes + (((uint32_t)N * 128 + 1023) & ~1023u);
    const int keyn = p.ltile_keyn[tile];
    const int key = keyn >> 8, n = keyn & 255;
    const int row0 = p.ltile_row0[tile], tok0 = p.ltile_tok0[tile];
    const int nkb = p.in_dim / kBK;
    uint32_t ncols = 32;
    while ((int)ncols < N) ncols <<= 1;

    if (warp == 1) {
        tc::tmem_alloc(&s_tmem, ncols);
        tc::tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(&acc_full, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&p.tm_x);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % kStages;
            if (kb >= kStages) wait_or_flag(&empty[s], (uint32_t)((kb / kStages - 1) & 1), p.spin_limit, p.status);
            char *st = smem + (size_t)s * stage_bytes;
            tc::mbar_expect_tx(&full[s], kTileBytes + a_bytes);
            tc::tma_load_2d(st, &p.tm_x, kb * kBK, tok0, &full[s]);
            tc::tma_load_2d(st + kTileBytes, &p.tm_a[js], kb * kBK, key * p.R, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = tc::idesc_bf16(kRows, N);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % kStages;
            wait_or_flag(&full[s], (uint32_t)((kb / kStages) & 1), p.spin_limit, p.status);
            tc::tc_fence_after();
            const uint32_t xa = tc::smem_u32(smem + (size_t)s * stage_bytes);
            const uint32_t aa = xa + kTileBytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
                tc::mma_bf16(tmem, tc::desc_sw128(xa + k * 32), tc::desc_sw128(aa + k * 32), idesc,
                             (kb | k) != 0);
            tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(&acc_full);
    } else if (warp >= 2) {
        const int q = warp & 3;
        const int t = q * 32 + lane;
        wait_or_flag(&acc_full, 0, p.spin_limit, p.status);
        tc::tc_fence_after();
        const float sc = p.scale[key] * p.post_scale;
        // the 64 hi and 64 lo columns of the row, zero past the rank
        for (int c = 0; c < 2; ++c) {
            uint32_t r[32];
            if (c * 32 < (int)ncols) {
                tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), r);
                tc::tmem_wait_ld();
            }
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c * 32 + i >= p.R) r[i] = 0u;
            if (t < n) {
                const int j = js, k0 = c * 32;
                uint16_t *vrow = p.V + (long long)j * p.v_slice + (long long)(row0 + t) * kVRow;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const float v0 = __uint_as_float(r[i * 8 + 2 * e2]) * sc;
                        const float v1 = __uint_as_float(r[i * 8 + 2 * e2 + 1]) * sc;
                        hw[e2] = pack2(v0, v1);
                        const float h0 = bf16lo(hw[e2]), h1 = bf16hi(hw[e2]);
                        lw[e2] = pack2(v0 - h0, v1 - h1);
                    }
                    *(uint4 *)(vrow + k0 + i * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *(uint4 *)(vrow + kBK + k0 + i * 8) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, ncols);
}

// ------------------------------------------------------------------ expand

__global__ void __launch_bounds__(kEThreads, 1) sgmv_expand_kernel(const __grid_constant__ ExpandArgs p) {
    extern __shared__ __align__(1024) char smem_raw[];
    __shared__ __align__(8) uint64_t v_full, v_empty, b_full[2], b_empty[2], y_full[kNY], y_empty[kNY],
        acc_full[2], acc_empty[2];
    __shared__ uint32_t s_tmem;
    char *smem = smem_raw + ((1024u - (smem_u32_of(smem_raw) & 1023u)) & 1023u);
    char *vt = smem;                           // V hi tile (16 KB) then lo tile (16 KB)
    char *bt = smem + 2 * kTileBytes;          // 2 x B tile (16 KB)
    char *yt = smem + 4 * kTileBytes;          // kNY x y tile (2 boxes of 16 KB each)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_lt = p.counters[5];
    const int n_grp = p.grp_start[p.n_slices];
    const int n_units = n_lt * n_grp;
    if ((int)blockIdx.x >= n_units) return;

    if (warp == 1) {
        tc::tmem_alloc(&s_tmem, 256);
        tc::tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        tc::mbar_init(&v_full, 1);
        tc::mbar_init(&v_empty, 1);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&b_full[b], 1);
            tc::mbar_init(&b_empty[b], 1);
            tc::mbar_init(&acc_full[b], 1);
            tc::mbar_init(&acc_empty[b], 8);
        }
        for (int b = 0; b < kNY; ++b) {
            tc::mbar_init(&y_full[b], 1);
            tc::mbar_init(&y_empty[b], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;

    // unit u -> (long tile, slice j, first o-tile, o-tile count)
    auto decode = [&](int u, int &lt, int &j, int &ot0, int &n_ot) {
        lt = u / n_grp;
        const int gq = u - lt * n_grp;
        j = 0;
        while (gq >= p.grp_start[j + 1]) ++j;
        ot0 = (gq - p.grp_start[j]) * kOG;
        n_ot = min(kOG, p.out_w[j] / kOT - ot0);
    };

    if (warp == 0 && lane == 0) {
        int it = 0, uc = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
            int lt, j, ot0, n_ot;
            decode(u, lt, j, ot0, n_ot);
            const int key = p.ltile_keyn[lt] >> 8;
            const int row0 = p.ltile_row0[lt], tok0 = p.ltile_tok0[lt];
            // the slot's compact B rows (rs = ceil8(rank) columns, the rest read as zero)
            const CUtensorMap *bm = p.bmaps + j * 8 + (((p.rank[key] + 7) >> 3) - 1);
            if (uc > 0) wait_or_flag(&v_empty, (uint32_t)((uc - 1) & 1), p.spin_limit, p.status);
            tc::mbar_expect_tx(&v_full, 2 * kTileBytes);
            tc::tma_load_2d(vt, &p.tm_v[j], 0, row0, &v_full);
            tc::tma_load_2d(vt + kTileBytes, &p.tm_v[j], kBK, row0, &v_full);
            for (int i = 0; i < n_ot; ++i, ++it) {
                const int b = it & 1, yb = it % kNY;
                const int o_local = (ot0 + i) * kOT;
                if (it >= 2) wait_or_flag(&b_empty[b], (uint32_t)(((it >> 1) - 1) & 1), p.spin_limit, p.status);
                tc::mbar_expect_tx(&b_full[b], kTileBytes);
                tc::tma_load_3d(bt + b * kTileBytes, bm, 0, o_local, key, &b_full[b]);
                if (it >= kNY)
                    wait_or_flag(&y_empty[yb], (uint32_t)((it / kNY - 1) & 1), p.spin_limit, p.status);
                char *yb_ptr = yt + (size_t)yb * 2 * kTileBytes;
                tc::mbar_expect_tx(&y_full[yb], 2 * kTileBytes);
                tc::tma_load_2d(yb_ptr, &p.tm_y, p.out_off[j] + o_local, tok0, &y_full[yb]);
                tc::tma_load_2d(yb_ptr + kTileBytes, &p.tm_y, p.out_off[j] + o_local + kBK, tok0, &y_full[yb]);
            }
        }
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = tc::idesc_bf16(kRows, kOT);
        const uint32_t vh = tc::smem_u32(vt), vl = vh + kTileBytes;
        int it = 0, uc = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
            int lt, j, ot0, n_ot;
            decode(u, lt, j, ot0, n_ot);
            wait_or_flag(&v_full, (uint32_t)(uc & 1), p.spin_limit, p.status);
            tc::tc_fence_after();
            for (int i = 0; i < n_ot; ++i, ++it) {
                const int b = it & 1;
                wait_or_flag(&b_full[b], (uint32_t)((it >> 1) & 1), p.spin_limit, p.status);
                if (it >= 2) wait_or_flag(&acc_empty[b], (uint32_t)(((it >> 1) - 1) & 1), p.spin_limit, p.status);
                tc::tc_fence_after();
                const uint32_t ba = tc::smem_u32(bt + b * kTileBytes);
                const uint32_t d = tmem + (uint32_t)(b * kOT);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                    tc::mma_bf16(d, tc::desc_sw128(vh + k * 32), tc::desc_sw128(ba + k * 32), idesc, k != 0);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                    tc::mma_bf16(d, tc::desc_sw128(vl + k * 32), tc::desc_sw128(ba + k * 32), idesc, 1);
                tc::mma_commit(&b_empty[b]);
                tc::mma_commit(&acc_full[b]);
            }
            tc::mma_commit(&v_empty);
        }
    } else if (warp >= 2) {
        // 8 epilogue warps: warp w reads accumulator lanes 32*(w%4).. (token
        // rows) and half (w-2)/4 of the 128 columns of each tile
        const int q = warp & 3, half = (warp - 2) >> 2;
        const int t = q * 32 + lane;
        const bool leader = (warp == 2 && lane == 0);
        int it = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
            int lt, j, ot0, n_ot;
            decode(u, lt, j, ot0, n_ot);
            const int n = p.ltile_keyn[lt] & 255;
            const int tok0 = p.ltile_tok0[lt];
            for (int i = 0; i < n_ot; ++i, ++it) {
                const int b = it & 1, yb = it % kNY;
                const int col0 = p.out_off[j] + (ot0 + i) * kOT;
                char *ybuf = yt + (size_t)yb * 2 * kTileBytes;
                wait_or_flag(&acc_full[b], (uint32_t)((it >> 1) & 1), p.spin_limit, p.status);
                wait_or_flag(&y_full[yb], (uint32_t)((it / kNY) & 1), p.spin_limit, p.status);
                tc::tc_fence_after();
                // this warp's columns half*64 .. +63 are box `half`, 16-byte units 0..7
                char *row = ybuf + (size_t)half * kTileBytes + (size_t)t * 128;
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    uint32_t r[32];
                    tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kOT + half * 64 + c * 32), r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i4 = 0; i4 < 4; ++i4) {
                        const int unit = (c * 4 + i4) ^ (t & 7);
                        uint4 *ptr = (uint4 *)(row + unit * 16);
                        uint4 yv = *ptr;
                        uint32_t w[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2)
                            w[e2] = pack2(bf16lo(w[e2]) + __uint_as_float(r[i4 * 8 + 2 * e2]),
                                          bf16hi(w[e2]) + __uint_as_float(r[i4 * 8 + 2 * e2 + 1]));
                        *ptr = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&acc_empty[b]);
                if (n == kRows) {
                    tc::fence_proxy_async();
                    asm volatile("bar.sync 1, 256;" ::: "memory");
                    if (leader) {
                        tc::tma_store_2d(&p.tm_y, col0, tok0, ybuf);
                        tc::tma_store_2d(&p.tm_y, col0 + kBK, tok0, ybuf + kTileBytes);
                        tc::bulk_commit();
                        tc::bulk_wait_read0();
                        tc::mbar_arrive(&y_empty[yb]);
                    }
                } else {
                    // partial last tile of a run: write back only its own rows
                    if (t < n) {
                        uint16_t *dst = p.y + (long long)(tok0 + t) * p.ld_y + col0 + half * 64;
#pragma unroll
                        for (int u16 = 0; u16 < 8; ++u16) {
                            const int unit = u16 ^ (t & 7);
                            *(uint4 *)(dst + u16 * 8) = *(const uint4 *)(row + unit * 16);
                        }
                    }
                    tc::fence_proxy_async();  // generic reads before the next TMA write
                    asm volatile("bar.sync 1, 256;" ::: "memory");
                    if (leader) tc::mbar_arrive(&y_empty[yb]);
                }
            }
        }
        if (leader) tc::bulk_wait0();
    }
    asm volatile("griddepcontrol.launch_dependents;");
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    // looked up once (thread-safe initialisation of a function-local static)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000)ptr;
        return nullptr;
    }();
    return fn;
}

// 2D bf16 tensor map, rows x cols (row stride in elements), 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, long long cols, long long rows, long long stride,
              int box_cols, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::atomic<int> g_sgmv_configured[64];

}  // namespace

bool lora_make_tmap_2d(CUtensorMap *m, const void *base, long long cols, long long rows, long long stride,
                       int box_cols, int box_rows, bool swizzle128) {
    PFN_cuTensorMapEncodeTiled_v12000 f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool lora_make_tmap_b3d(CUtensorMap *m, const void *base, int rs, int rows, int slots, long long slot_elems) {
    PFN_cuTensorMapEncodeTiled_v12000 f = encode_fn();
    if (!f || rs % 8 || slot_elems % 8) return false;
    cuuint64_t dims[3] = {(cuuint64_t)rs, (cuuint64_t)rows, (cuuint64_t)slots};
    cuuint64_t strides[2] = {(cuuint64_t)rs * 2, (cuuint64_t)slot_elems * 2};
    cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)kOT, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool lora_make_tmap_bk(CUtensorMap *m, const void *base, int rs, long long rows, int slots, long long slot_elems) {
    PFN_cuTensorMapEncodeTiled_v12000 f = encode_fn();
    if (!f || rs % 8 || slot_elems % 8 || rows < kOT) return false;
    cuuint64_t dims[3] = {(cuuint64_t)rs, (cuuint64_t)rows, (cuuint64_t)slots};
    cuuint64_t strides[2] = {(cuuint64_t)rs * 2, (cuuint64_t)slot_elems * 2};
    cuuint32_t box[3] = {8, (cuuint32_t)kOT, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool lora_make_tmap_a_chunks(CUtensorMap *m, const void *base, long long rows, long long cols, int box_rows,
                             int box_chunks) {
    PFN_cuTensorMapEncodeTiled_v12000 f = encode_fn();
    if (!f || cols % 64) return false;
    // dims: 64 elements of a 128-byte chunk, the rows, the chunks of a row
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks};
    cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool lora_sgmv_eligible(const lora_pool_t *pool) {
    const lora_pool_desc_t &d = pool->desc;
    if (pool->is_moe || !pool->d_bmaps || d.max_rank > 64) return false;
    if (d.n_slices * d.max_rank > 256 || d.in_dim % kBK) return false;
    for (int j = 0; j < d.n_slices; ++j)
        if (d.out_dims[j] % kOT) return false;
    return encode_fn() != nullptr;
}

size_t lora_sgmv_ws_bytes(const lora_pool_t *pool, int rows) {
    return (size_t)pool->desc.n_slices * rows * kVRow * 2;
}

lora_status_t lora_sgmv_apply(const lora_pool_t *pool, const lora_meta_t *meta, const void *x, int64_t ldx,
                              void *y, int64_t ldy, void *V, int spin_limit, int num_sms, float post_scale,
                              cudaStream_t s) {
    const lora_pool_desc_t &d = pool->desc;
    const int T = meta->T, R = d.max_rank, ns = d.n_slices;
    int out_total = 0;
    for (int j = 0; j < ns; ++j) out_total += d.out_dims[j];
    const int dev = pool->device < 64 ? pool->device : 63;
    if (!g_sgmv_configured[dev].load(std::memory_order_acquire)) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(sgmv_shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           200 * 1024));
        LORA_CUDA_TRY(cudaFuncSetAttribute(sgmv_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           200 * 1024));
        g_sgmv_configured[dev].store(1, std::memory_order_release);
    }
    // long tiles: a run of >= LORA_LONG_MIN tokens of one slot gives at most
    // ceil(run / 128) of them, so at most T / LORA_LONG_MIN in all (a decode
    // batch in a large pool launches a few CTAs that find no tile, not one
    // per slot)
    int max_lt = T / kRows + d.max_loras + 1;
    if (max_lt > T / LORA_LONG_MIN + 1) max_lt = T / LORA_LONG_MIN + 1;
    if (spin_limit > (1 << 18)) spin_limit = 1 << 18;  // each poll may suspend the thread for a while

    ShrinkArgs sa;
    memset(&sa, 0, sizeof(sa));
    if (!make_map(&sa.tm_x, x, d.in_dim, T, ldx, kBK, kRows)) return LORA_ERR_CUDA;
    for (int j = 0; j < ns; ++j)
        if (!make_map(&sa.tm_a[j], pool->A[j], d.in_dim, (long long)d.max_loras * R, d.in_dim, kBK, R))
            return LORA_ERR_CUDA;
    sa.n_slices = ns;
    sa.in_dim = d.in_dim;
    sa.R = R;
    sa.ltile_row0 = meta->ltile_row0;
    sa.ltile_keyn = meta->ltile_keyn;
    sa.ltile_tok0 = meta->ltile_tok0;
    sa.counters = meta->counters;
    sa.scale = pool->d_scale;
    sa.V = (uint16_t *)V;
    sa.v_slice = (long long)T * kVRow;
    sa.status = pool->d_status;
    sa.spin_limit = spin_limit;
    sa.post_scale = post_scale;
    const size_t a_bytes = (size_t)((R + 15) & ~15) * 128;  // the MMA reads N = ceil16(R) rows of A
    const size_t stage = kTileBytes + ((a_bytes + 1023) & ~(size_t)1023);
    const size_t smem_s = kStages * stage + 1024;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(max_lt * ns), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_s;
    cfg.stream = s;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, sgmv_shrink_kernel, sa));
    lora_note_launch();

    ExpandArgs ea;
    memset(&ea, 0, sizeof(ea));
    for (int j = 0; j < ns; ++j)
        if (!make_map(&ea.tm_v[j], (const uint16_t *)V + (long long)j * T * kVRow, kVRow, T, kVRow, kBK, kRows))
            return LORA_ERR_CUDA;
    ea.bmaps = pool->d_bmaps;
    ea.rank = pool->d_rank;
    if (!make_map(&ea.tm_y, y, out_total, T, ldy, kBK, kRows)) return LORA_ERR_CUDA;
    ea.n_slices = ns;
    ea.R = R;
    int g = 0, off = 0;
    for (int j = 0; j < ns; ++j) {
        ea.out_w[j] = d.out_dims[j];
        ea.out_off[j] = off;
        off += d.out_dims[j];
        ea.grp_start[j] = g;
        g += lora_ceil_div(d.out_dims[j] / kOT, kOG);
    }
    ea.grp_start[ns] = g;
    ea.ltile_row0 = meta->ltile_row0;
    ea.ltile_keyn = meta->ltile_keyn;
    ea.ltile_tok0 = meta->ltile_tok0;
    ea.counters = meta->counters;
    ea.y = (uint16_t *)y;
    ea.ld_y = ldy;
    ea.status = pool->d_status;
    ea.spin_limit = spin_limit;
    const size_t smem_e = (4 + 2 * kNY) * (size_t)kTileBytes + 1024;
    long long units = (long long)max_lt * g;
    cfg.gridDim = dim3((unsigned)(units < num_sms ? units : num_sms), 1, 1);
    cfg.blockDim = dim3(kEThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_e;
    cfg.numAttrs = 0;  // the expand reads the shrink's V: plain stream order
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, sgmv_expand_kernel, ea));
    lora_note_launch();
    return LORA_OK;
}
