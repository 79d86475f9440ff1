// Grouped shrink/expand on CUDA cores (BGMV-style decode path, and the
// fallback for every group size): the multi-tenant LoRA delta of the vLLM
// LoRA layer pages (add_shrink into an fp32 buffer, then add_expand with
// add_input=True at the slice offsets; add_lora_fused_moe per (adapter,
// expert) group after top-k routing).
//
// Work is cut into items over the tile list built by lora_build_meta (tiles
// of up to 16 rows of one group, i.e. one slot or one (slot, expert)):
//   shrink item (tile, slice j, hidden chunk c):
//       partial[c][j][k][row] = sum_{h in chunk c} x[row][h] * A_j[a][k][h]
//       (x tile staged in shared memory with cp.async, A rows streamed with
//       16-byte non-allocating loads, 4 ranks x 16 rows of fp32 accumulators
//       per lane, one butterfly reduce-scatter across the warp)
//   expand item (tile, slice j, 512-column chunk):
//       v[row][k] = scale[a] * w[row] * sum_c partial[c][j][k][row]
//       y[row][off_j + o] += sum_k v[row][k] * B_j[a][o][k]   (bf16x2 RMW)
// In the fused kernel one persistent grid takes items from a ticket counter
// (all shrink items precede all expand items), and an expand item waits with
// a bounded spin for its tile's shrink chunks.  Waits only ever point to
// lower tickets, which are held by running CTAs, so the schedule cannot
// deadlock whatever the residency.  The last CTA to finish zeroes the
// control words so the workspace is ready for the next call.
#include <algorithm>
#include <atomic>
#include <stdlib.h>
#include <string.h>

#include "lora_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kTile = LORA_TILE_ROWS;  // 16 rows per tile
constexpr int kOC = 2 * kThreads;      // output columns per expand item
constexpr int kMaxHC = 1024;           // hidden chunk cap (shared-memory x tile)
constexpr int kXPad = 8;               // bf16 padding per staged x row
constexpr int kRedUnits = 16;
// vLLM's FusedMoEWithLoRA gives every routed pair a block of its own when
// num_tokens * top_k * SPARSITY_FACTOR <= num_experts * max_loras
constexpr long long kSparsityFactor = 8;

enum Mode { kFused = 0, kShrinkAtomic = 1, kExpandOnly = 2 };

struct GArgs {
    int n_slices, in_dim, E, row_div, R, T, NC, HC;
    int out_w[LORA_MAX_SLICES], out_off[LORA_MAX_SLICES], och_start[LORA_MAX_SLICES + 1];
    const uint16_t *A[LORA_MAX_SLICES];
    long long A_ss[LORA_MAX_SLICES], A_es[LORA_MAX_SLICES];
    const uint16_t *B[LORA_MAX_SLICES];
    long long B_ss[LORA_MAX_SLICES];
    int B_shared[LORA_MAX_SLICES];
    const int32_t *rank;
    const float *scale;
    const int32_t *sorted, *tile_row0, *tile_keyn, *counters;
    int count_idx;  // counters[count_idx] = number of tiles in the list
    const uint16_t *in;
    long long ld_in;
    uint16_t *out;
    long long ld_out;
    const float *row_w;
    float *part;  // fused: [NC][n_slices][R][rows]; shrink: v [n_slices][T][R]; expand: v
    int rows;     // row capacity of the partial buffer (T * top_k)
    int *ctrl;    // [0] ticket, [1] finished CTAs
    int *tile_cnt;
    int *status;
    int spin_limit;
    float post_scale;
};

struct TileInfo {
    int row0, n, a, e, r;
};

__device__ __forceinline__ TileInfo tile_info(const GArgs &p, int tile) {
    TileInfo ti;
    ti.row0 = p.tile_row0[tile];
    const int keyn = p.tile_keyn[tile];
    ti.n = keyn & 31;
    const int key = keyn >> 5;
    ti.a = key / p.E;
    ti.e = key - ti.a * p.E;
    ti.r = p.rank[ti.a];
    return ti;
}

__device__ __forceinline__ void cvt8(const uint4 &u, float f[8]) {
    f[0] = bf16lo(u.x); f[1] = bf16hi(u.x);
    f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
    f[4] = bf16lo(u.z); f[5] = bf16hi(u.z);
    f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}

// Reduce-scatter of 64 per-lane values across the warp: afterwards lane l
// holds the warp sums of entries 2l and 2l+1 in v[0], v[1].
__device__ __forceinline__ void warp_reduce_scatter64(float v[64], int lane) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const bool up = lane & 16;
        const float send = up ? v[i] : v[i + 32];
        const float keep = up ? v[i + 32] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const bool up = lane & 8;
        const float send = up ? v[i] : v[i + 16];
        const float keep = up ? v[i + 16] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = lane & 4;
        const float send = up ? v[i] : v[i + 8];
        const float keep = up ? v[i + 8] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = lane & 2;
        const float send = up ? v[i] : v[i + 4];
        const float keep = up ? v[i + 4] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = lane & 1;
        const float send = up ? v[i] : v[i + 2];
        const float keep = up ? v[i + 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
}

template <int MODE>
__device__ __forceinline__ void store_partial(const GArgs &p, const TileInfo &ti, int j, int c,
                                              int k, int t, float s) {
    if (MODE == kFused) {
        p.part[(((long long)c * p.n_slices + j) * p.R + k) * p.rows + ti.row0 + t] = s;
    } else {
        const int tok = p.sorted[ti.row0 + t];
        atomicAdd(p.part + ((long long)j * p.T + tok) * p.R + k, s);
    }
}

template <int MODE>
__device__ void shrink_item(const GArgs &p, int tile, int j, int c, char *smem) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const TileInfo ti = tile_info(p, tile);
    const int XS = p.HC + kXPad;
    uint16_t *xs = (uint16_t *)smem;
    float *red = (float *)(smem + (size_t)kTile * XS * 2);
    const int h0 = c * p.HC;
    const int hc = min(p.in_dim - h0, p.HC);
    const int nvec = hc >> 3;
    const uint16_t *Ab = p.A[j] + (long long)ti.a * p.A_ss[j] + (long long)ti.e * p.A_es[j] + h0;

    for (int i = tid; i < ti.n * nvec; i += kThreads) {
        const int t = i / nvec, q = i - t * nvec;
        const int row = p.sorted[ti.row0 + t];
        cp_async16(xs + t * XS + q * 8, p.in + (long long)(row / p.row_div) * p.ld_in + h0 + q * 8);
    }
    cp_async_wait_all();
    __syncthreads();

    const int nkg = (ti.r + 3) >> 2;
    const int nhs = nkg >= 8 ? 1 : nkg >= 4 ? 2 : nkg >= 2 ? 4 : 8;
    const int units = nkg * nhs;
    const int hs_len = ((nvec + nhs - 1) / nhs) * 8;
    for (int u = warp; u < units; u += kThreads / 32) {
        const int kg = u / nhs, hs = u - kg * nhs;
        const int hb = hs * hs_len, he = min(hc, hb + hs_len);
        float v[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = 0.f;
        for (int hh = hb + lane * 8; hh < he; hh += 256) {
            float af[4][8];
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                const int k = kg * 4 + kb;
                uint4 q = make_uint4(0, 0, 0, 0);
                if (k < ti.r) q = ldg_stream(Ab + (long long)k * p.in_dim + hh);
                cvt8(q, af[kb]);
            }
#pragma unroll
            for (int t = 0; t < kTile; ++t) {
                if (t < ti.n) {
                    float xf[8];
                    cvt8(*(const uint4 *)(xs + t * XS + hh), xf);
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
                        float s = v[kb * kTile + t];
#pragma unroll
                        for (int i = 0; i < 8; ++i) s = fmaf(af[kb][i], xf[i], s);
                        v[kb * kTile + t] = s;
                    }
                }
            }
        }
        warp_reduce_scatter64(v, lane);
        // lane holds f = 2*lane + m: rank kg*4 + (f >> 4), row f & 15
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int f = 2 * lane + m;
            const int k = kg * 4 + (f >> 4), t = f & 15;
            if (nhs == 1) {
                if (k < ti.r && t < ti.n) store_partial<MODE>(p, ti, j, c, k, t, v[m]);
            } else {
                red[u * 64 + f] = v[m];
            }
        }
    }
    if (nhs > 1) {
        __syncthreads();
        for (int i = tid; i < nkg * 64; i += kThreads) {
            const int kg = i >> 6, f = i & 63;
            const int k = kg * 4 + (f >> 4), t = f & 15;
            if (k < ti.r && t < ti.n) {
                float s = 0.f;
                for (int hs = 0; hs < nhs; ++hs) s += red[(kg * nhs + hs) * 64 + f];
                store_partial<MODE>(p, ti, j, c, k, t, s);
            }
        }
    }
}

template <int MODE>
__device__ void expand_item(const GArgs &p, int tile, int j, int oc, char *smem, int *s_flag) {
    const int tid = threadIdx.x;
    const TileInfo ti = tile_info(p, tile);
    if (MODE == kFused) {
        if (tid == 0) {
            const int *cnt = p.tile_cnt + tile * p.n_slices + j;
            int ok = 1, polls = 0;
            while (ld_acquire_gpu(cnt) < p.NC) {
                if (p.spin_limit < 0 || ++polls > p.spin_limit) {
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
            if (!ok) atomicExch(p.status, (int)LORA_ERR_TIMEOUT);
            *s_flag = ok;
        }
        __syncthreads();
        if (!*s_flag) return;
    }
    const int rs = (ti.r + 7) & ~7;
    const int VS = ((p.R + 7) & ~7) + 4;  // row stride of v in shared memory (multiple of 4)
    float *vs = (float *)smem;
    const float sc = p.scale[ti.a] * p.post_scale;
    for (int i = tid; i < ti.n * rs; i += kThreads) {
        const int t = i / rs, k = i - t * rs;
        float s = 0.f;
        if (k < ti.r) {
            if (MODE == kFused) {
                const float *src = p.part + ((long long)j * p.R + k) * p.rows + ti.row0 + t;
                const long long cstride = (long long)p.n_slices * p.R * p.rows;
                for (int c = 0; c < p.NC; ++c) s += __ldcg(src + c * cstride);
            } else {
                const int tok = p.sorted[ti.row0 + t];
                s = p.part[((long long)j * p.T + tok) * p.R + k];
            }
            float w = sc;
            if (p.row_w) w *= p.row_w[p.sorted[ti.row0 + t]];
            s *= w;
        }
        vs[t * VS + k] = s;
    }
    __syncthreads();
    const int Ow = p.out_w[j];
    const int o = oc * kOC + tid * 2;
    if (o < Ow) {
        const uint16_t *Bb = p.B[j] + (long long)ti.a * p.B_ss[j] +
                             (p.B_shared[j] ? 0ll : (long long)ti.e * Ow * rs);
        const uint16_t *b0p = Bb + (long long)o * rs;
        const uint16_t *b1p = b0p + rs;
        float acc0[kTile], acc1[kTile];
#pragma unroll
        for (int t = 0; t < kTile; ++t) acc0[t] = acc1[t] = 0.f;
        for (int kk = 0; kk < rs; kk += 8) {
            float f0[8], f1[8];
            cvt8(ldg_stream(b0p + kk), f0);
            cvt8(ldg_stream(b1p + kk), f1);
#pragma unroll
            for (int t = 0; t < kTile; ++t) {
                if (t < ti.n) {
                    const float4 va = *(const float4 *)(vs + t * VS + kk);
                    const float4 vb = *(const float4 *)(vs + t * VS + kk + 4);
                    const float vv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
                    float s0 = acc0[t], s1 = acc1[t];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        s0 = fmaf(vv[i], f0[i], s0);
                        s1 = fmaf(vv[i], f1[i], s1);
                    }
                    acc0[t] = s0;
                    acc1[t] = s1;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kTile; ++t) {
            if (t < ti.n) {
                const int row = p.sorted[ti.row0 + t];
                uint32_t *yp = (uint32_t *)(p.out + (long long)row * p.ld_out + p.out_off[j] + o);
                const uint32_t u = *yp;
                const __nv_bfloat162 r2 = __floats2bfloat162_rn(bf16lo(u) + acc0[t], bf16hi(u) + acc1[t]);
                *yp = *(const uint32_t *)&r2;
            }
        }
    }
}

template <int MODE>
__device__ __forceinline__ void run_item(const GArgs &p, int item, int n_sh, char *smem, int *s_flag) {
    if (item < n_sh) {
        const int per_tile = p.n_slices * p.NC;
        const int tile = item / per_tile;
        const int rem = item - tile * per_tile;
        const int j = rem / p.NC, c = rem - j * p.NC;
        shrink_item<MODE>(p, tile, j, c, smem);
        if (MODE == kFused) {
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                atomicAdd(p.tile_cnt + tile * p.n_slices + j, 1);
            }
        }
    } else {
        const int it = item - n_sh;
        const int och = p.och_start[p.n_slices];
        const int tile = it / och;
        const int q = it - tile * och;
        int j = 0;
        while (q >= p.och_start[j + 1]) ++j;
        expand_item<MODE>(p, tile, j, q - p.och_start[j], smem, s_flag);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) grouped_lora_kernel(const __grid_constant__ GArgs p) {
    extern __shared__ __align__(16) char smem[];
    __shared__ int s_item, s_flag, s_last;
    const int n_tiles = p.counters[p.count_idx];
    const int n_sh = (MODE == kExpandOnly) ? 0 : n_tiles * p.n_slices * p.NC;
    const int n_ex = (MODE == kShrinkAtomic) ? 0 : n_tiles * p.och_start[p.n_slices];
    const int total = n_sh + n_ex;
    if (MODE == kFused) {
        int nxt = 0;
        if (threadIdx.x == 0) nxt = atomicAdd(p.ctrl, 1);
        for (;;) {
            if (threadIdx.x == 0) {
                s_item = nxt;
                nxt = atomicAdd(p.ctrl, 1);
            }
            __syncthreads();
            const int item = s_item;
            if (item >= total) break;
            run_item<MODE>(p, item, n_sh, smem, &s_flag);
            __syncthreads();
        }
        asm volatile("griddepcontrol.launch_dependents;");
        if (threadIdx.x == 0) {
            __threadfence();
            s_last = (atomicAdd(p.ctrl + 1, 1) == (int)gridDim.x - 1);
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            for (int i = threadIdx.x; i < n_tiles * p.n_slices; i += kThreads) p.tile_cnt[i] = 0;
            if (threadIdx.x == 0) {
                p.ctrl[0] = 0;
                p.ctrl[1] = 0;
            }
        }
    } else {
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            run_item<MODE>(p, item, n_sh, smem, &s_flag);
            __syncthreads();
        }
    }
}

int g_spin_limit = 1 << 20;

struct Plan {
    int NC, HC;
    size_t part_floats, cnt_ints;
};

// Split the hidden dimension so that every shrink item stays small
// (<= ~0.5M FMAs) and the grid has several items per SM.
Plan make_plan(int num_sms, int in_dim, int n_slices, int R, int rows, int n_keys) {
    Plan pl;
    const long long tiles_est = (rows + kTile - 1) / kTile + (rows < n_keys ? rows : n_keys);
    const long long units = tiles_est * n_slices > 0 ? tiles_est * n_slices : 1;
    int nc_par = (int)((6LL * num_sms + units - 1) / units);
    int nc_work = (int)(((long long)in_dim * kTile * R + (1 << 19) - 1) >> 19);
    int nc = nc_par > nc_work ? nc_par : nc_work;
    if (nc < 1) nc = 1;
    int hc = lora_round8(lora_ceil_div(in_dim, nc));
    if (hc > kMaxHC) hc = kMaxHC;
    if (hc < 8) hc = 8;
    pl.HC = hc;
    pl.NC = lora_ceil_div(in_dim, hc);
    pl.part_floats = (size_t)pl.NC * n_slices * R * (size_t)rows;
    const size_t max_tiles = (size_t)rows / kTile + n_keys + 1;
    pl.cnt_ints = max_tiles * n_slices;
    return pl;
}

constexpr size_t kCtrlBytes = 256;

size_t ws_bytes_for(const Plan &pl) {
    size_t b = kCtrlBytes + ((pl.cnt_ints * 4 + 255) & ~(size_t)255);
    return b + pl.part_floats * 4;
}

size_t smem_bytes(const GArgs &g) {
    const size_t shrink = (size_t)kTile * (g.HC + kXPad) * 2 + (size_t)kRedUnits * 64 * 4;
    const size_t expand = (size_t)kTile * (((g.R + 7) & ~7) + 4) * 4;
    return shrink > expand ? shrink : expand;
}

constexpr size_t kMaxSmem = (size_t)kTile * (kMaxHC + kXPad) * 2 + (size_t)kRedUnits * 64 * 4;
static_assert(kMaxSmem <= 48 * 1024, "grouped kernel must fit the default shared-memory limit");
static_assert((size_t)kTile * (((LORA_MAX_RANK + 7) & ~7) + 4) * 4 <= kMaxSmem, "v tile");

// Occupancy per (device, mode), queried once outside any stream capture.
std::atomic<int> g_occ[64][3];

template <int MODE>
lora_status_t launch(const lora_pool_t *pool, GArgs &g, long long est_items, cudaStream_t s) {
    const size_t smem = smem_bytes(g);
    int dev = pool->device < 64 ? pool->device : 63;
    int occ = g_occ[dev][MODE].load(std::memory_order_relaxed);
    if (occ == 0) {
        int o = 0;
        LORA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, grouped_lora_kernel<MODE>,
                                                                    kThreads, kMaxSmem));
        occ = o < 1 ? 1 : o;
        g_occ[dev][MODE].store(occ, std::memory_order_relaxed);  // every thread computes the same value
    }
    long long grid = (long long)pool->num_sms * occ;
    if (est_items < grid) grid = est_items;
    if (grid < 1) grid = 1;
    g.spin_limit = g_spin_limit;
    grouped_lora_kernel<MODE><<<(unsigned)grid, kThreads, smem, s>>>(g);
    LORA_CUDA_TRY(cudaGetLastError());
    lora_note_launch();
    return LORA_OK;
}

// Fill the fields shared by every mode for a dense pool.
lora_status_t dense_args(const lora_pool_t *pool, const lora_meta_t *meta, GArgs &g) {
    if (pool->is_moe) return LORA_ERR_UNSUPPORTED;
    if (!meta || meta->mode != 0 || meta->n_keys != pool->desc.max_loras) return LORA_ERR_INVALID_ARG;
    memset(&g, 0, sizeof(g));
    const lora_pool_desc_t &d = pool->desc;
    g.n_slices = d.n_slices;
    g.in_dim = d.in_dim;
    g.E = 1;
    g.row_div = 1;
    g.R = d.max_rank;
    g.T = meta->T;
    int off = 0, och = 0;
    for (int j = 0; j < d.n_slices; ++j) {
        g.out_w[j] = d.out_dims[j];
        g.out_off[j] = off;
        off += d.out_dims[j];
        g.och_start[j] = och;
        och += lora_ceil_div(d.out_dims[j], kOC);
        g.A[j] = pool->A[j];
        g.A_ss[j] = pool->a_slot_elems[j];
        g.A_es[j] = 0;
        g.B[j] = pool->B[j];
        g.B_ss[j] = pool->b_slot_elems[j];
        g.B_shared[j] = 1;
    }
    g.och_start[d.n_slices] = och;
    g.rank = pool->d_rank;
    g.scale = pool->d_scale;
    g.sorted = meta->sorted;
    g.tile_row0 = meta->tile_row0;
    g.tile_keyn = meta->tile_keyn;
    g.count_idx = 3;
    g.counters = meta->counters;
    g.status = pool->d_status;
    g.rows = meta->T;
    g.post_scale = 1.0f;
    return LORA_OK;
}

int out_total(const lora_pool_t *pool) {
    int s = 0;
    for (int j = 0; j < pool->desc.n_slices; ++j) s += pool->desc.out_dims[j];
    return s;
}

// A workspace sized for T tokens always fits a smaller batch once the hidden
// chunks are widened (fewer chunks, fewer partials).
Plan fit_plan(Plan pl, int in_dim, int n_slices, int R, int rows, size_t part_cap_bytes) {
    while (pl.part_floats * 4 > part_cap_bytes && pl.HC < kMaxHC) {
        pl.HC = pl.HC * 2 > kMaxHC ? kMaxHC : pl.HC * 2;
        pl.NC = lora_ceil_div(in_dim, pl.HC);
        pl.part_floats = (size_t)pl.NC * n_slices * R * (size_t)rows;
    }
    return pl;
}

void bind_splitk(GArgs &g, const Plan &pl, int *ctrl, int *cnt, float *part) {
    g.ctrl = ctrl;
    g.tile_cnt = cnt;
    g.part = part;
    g.NC = pl.NC;
    g.HC = pl.HC;
}

size_t align1k(size_t x) { return (x + 1023) & ~(size_t)1023; }
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
int max_tiles(int rows, int keys) { return rows / kTile + (rows < keys ? rows : keys) + 1; }

// Workspace of an apply call.  Its first part holds the words that must be
// zero when a call starts (the split-K kernel's ticket, finish count and
// per-tile counters; every call leaves them zero again).  The size of that
// part depends only on the workspace size, so calls with different token
// counts or layer types that share one workspace agree on where it is.  The
// rest is scratch with no state between calls: [bf16 hi/lo rank buffer of
// the tensor-core path][split-K partials, or the split kernels' chunk
// partials].
struct Carve {
    int *ctrl, *cnt;
    size_t cnt_cap;  // ints
    char *data;
    size_t data_bytes;
};

size_t counter_reserve(size_t ws_bytes) {
    const size_t r = align256(ws_bytes / 8);
    return r < 512 ? 512 : r;
}

bool carve(void *ws, size_t ws_bytes, Carve &c) {
    const size_t res = counter_reserve(ws_bytes);
    if (!ws || ws_bytes < res) return false;
    c.ctrl = (int *)ws;
    c.cnt = (int *)((char *)ws + kCtrlBytes);
    c.cnt_cap = (res - kCtrlBytes) / 4;
    c.data = (char *)ws + res;
    c.data_bytes = ws_bytes - res;
    return true;
}

// Smallest workspace whose carve holds data_bytes of scratch and cnt_ints counters.
size_t ws_total(size_t data_bytes, size_t cnt_ints) {
    const size_t need = kCtrlBytes + cnt_ints * 4;
    size_t w = data_bytes + align256(need) + 512;
    while (counter_reserve(w) < need || w - counter_reserve(w) < data_bytes) w += align256(w / 16 + 256);
    return w;
}

size_t sgmv_region_bytes(const lora_pool_t *pool, int T) {
    if (pool->is_moe || pool->desc.max_rank > 64) return 0;
    return (lora_sgmv_ws_bytes(pool, T) + 1023) & ~(size_t)1023;
}

long long est_items(const GArgs &g, int rows, int n_keys, int mode) {
    const long long tiles = (rows + kTile - 1) / kTile + (rows < n_keys ? rows : n_keys);
    long long n = 0;
    if (mode != kExpandOnly) n += tiles * g.n_slices * g.NC;
    if (mode != kShrinkAtomic) n += tiles * g.och_start[g.n_slices];
    return n;
}

LoraProblem to_problem(const GArgs &g, const lora_meta_t *meta, int n_keys) {
    LoraProblem pr;
    memset(&pr, 0, sizeof(pr));
    pr.n_slices = g.n_slices;
    pr.in_dim = g.in_dim;
    pr.E = g.E;
    pr.row_div = g.row_div;
    pr.R = g.R;
    pr.T = g.T;
    pr.rows = g.rows;
    pr.n_keys = n_keys;
    for (int j = 0; j < g.n_slices; ++j) {
        pr.out_w[j] = g.out_w[j];
        pr.out_off[j] = g.out_off[j];
        pr.A[j] = g.A[j];
        pr.A_ss[j] = g.A_ss[j];
        pr.A_es[j] = g.A_es[j];
        pr.B[j] = g.B[j];
        pr.B_ss[j] = g.B_ss[j];
        pr.B_shared[j] = g.B_shared[j];
    }
    pr.rank = g.rank;
    pr.scale = g.scale;
    pr.meta = meta;
    pr.tile_row0 = g.tile_row0;
    pr.tile_keyn = g.tile_keyn;
    pr.count_idx = g.count_idx;
    pr.in = g.in;
    pr.ld_in = g.ld_in;
    pr.out = g.out;
    pr.ld_out = g.ld_out;
    pr.row_w = g.row_w;
    pr.status = g.status;
    pr.spin_limit = g_spin_limit;
    pr.post_scale = g.post_scale;
    return pr;
}

}  // namespace

int g_lora_kernel_policy = 0;

// Kernel policies (lora_set_kernel_policy) under which the fused decode
// kernel and the split kernels may run: 0 automatic, 3 without the fused
// kernel, 4-8 automatic apart from their own choice.
static bool pol_fused(int p) { return p == 0 || p >= 4; }
static bool pol_split(int p) { return p == 0 || p >= 3; }
static std::atomic<unsigned long long> g_lora_launches{0};
void lora_note_launch() { g_lora_launches.fetch_add(1, std::memory_order_relaxed); }
extern "C" unsigned long long lora_kernel_launch_count(void) { return g_lora_launches.load(); }

static std::atomic<int> g_last_cuda_error{0};
void lora_note_cuda_error(cudaError_t e) { g_last_cuda_error.store((int)e, std::memory_order_relaxed); }
extern "C" int32_t lora_last_cuda_error(void) { return g_last_cuda_error.load(std::memory_order_relaxed); }

extern "C" void lora_set_kernel_policy(int32_t policy) { g_lora_kernel_policy = policy; }

extern "C" void lora_set_spin_limit(int32_t max_polls) { g_spin_limit = max_polls; }

bool lora_ws_data(void *workspace, size_t ws_bytes, char **data, size_t *data_bytes) {
    Carve cv;
    if (!workspace || !lora_aligned16(workspace) || !carve(workspace, ws_bytes, cv)) return false;
    *data = cv.data;
    *data_bytes = cv.data_bytes;
    return true;
}

extern "C" size_t lora_workspace_bytes(const lora_pool_t *pool, int32_t T, int32_t top_k) {
    if (!pool || T < 0) return 0;
    const lora_pool_desc_t &d = pool->desc;
    if (!pool->is_moe) {
        const Plan pl = make_plan(pool->num_sms, d.in_dim, d.n_slices, d.max_rank, T, d.max_loras);
        const size_t sp = lora_split_ws_bytes(d.n_slices, d.in_dim, d.max_rank, T, max_tiles(T, d.max_loras));
        const size_t pk = align256(pl.part_floats * 4);
        // lora_linear_apply: the shrink's sums and a slot and a sorted position per token
        const size_t lin = std::max(align256(sp), align256((size_t)d.n_slices * T * d.max_rank * 4)) +
                           2 * align256((size_t)T * 4);
        size_t data = sgmv_region_bytes(pool, T) + (pk > sp ? pk : sp);
        if (lin > data) data = lin;
        return ws_total(data, pl.cnt_ints);
    }
    if (top_k < 1) return 0;
    const int rows = T * top_k, keys = d.max_loras * d.num_experts;
    const Plan p13 = make_plan(pool->num_sms, d.d_model, d.n_w13_slices, d.max_rank, rows, keys);
    const Plan p2 = make_plan(pool->num_sms, d.d_mlp, 1, d.max_rank, rows, keys);
    size_t data = align256(p13.part_floats * 4);
    data = std::max(data, align256(p2.part_floats * 4));
    data = std::max(data, lora_split_ws_bytes(d.n_w13_slices, d.d_model, d.max_rank, rows, max_tiles(rows, keys)));
    data = std::max(data, lora_split_ws_bytes(1, d.d_mlp, d.max_rank, rows, max_tiles(rows, keys)));
    return ws_total(data, std::max(p13.cnt_ints, p2.cnt_ints));
}

extern "C" lora_status_t lora_workspace_init(void *workspace, size_t bytes, void *stream) {
    if (!workspace) return LORA_ERR_INVALID_ARG;
    LORA_CUDA_TRY(cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream));
    return LORA_OK;
}

lora_status_t lora_dense_apply(const lora_pool_t *pool, const lora_meta_t *meta, const void *x, int64_t ldx,
                               void *y, int64_t ldy, void *workspace, size_t ws_bytes, float post_scale,
                               cudaStream_t s) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    GArgs g;
    lora_status_t st = dense_args(pool, meta, g);
    if (st != LORA_OK) return st;
    if (meta->T == 0) return LORA_OK;
    if (!x || !y || !lora_aligned16(x) || !lora_aligned16(y) || ldx % 8 || ldy % 8 ||
        ldx < pool->desc.in_dim || ldy < out_total(pool))
        return LORA_ERR_INVALID_ARG;
    g.post_scale = post_scale;
    if (!workspace || !lora_aligned16(workspace)) return LORA_ERR_INVALID_ARG;
    Carve cv;
    if (!carve(workspace, ws_bytes, cv)) return LORA_ERR_CAPACITY;
    const size_t sg_bytes = sgmv_region_bytes(pool, meta->T);
    // decode-sized batches (the fused decode kernel takes them) do not look
    // for long runs: a batch of a few rows per slot has none worth a tile
    const bool decode_sized = pol_fused(g_lora_kernel_policy) && lora_fused_eligible(pool, meta->T);
    const bool use_sgmv = g_lora_kernel_policy != 1 && !decode_sized && sg_bytes > 0 && meta->T >= LORA_LONG_MIN &&
                          cv.data_bytes >= sg_bytes && lora_sgmv_eligible(pool);
    char *scratch = cv.data + (use_sgmv ? sg_bytes : 0);
    const size_t scratch_bytes = cv.data_bytes - (use_sgmv ? sg_bytes : 0);
    const Plan pl = fit_plan(make_plan(pool->num_sms, g.in_dim, g.n_slices, g.R, meta->T, pool->desc.max_loras),
                             g.in_dim, g.n_slices, g.R, meta->T, scratch_bytes);
    // the split-K kernel is the fallback for every shape: its plan must fit
    if (pl.cnt_ints > cv.cnt_cap || pl.part_floats * 4 > scratch_bytes) return LORA_ERR_CAPACITY;
    bind_splitk(g, pl, cv.ctrl, cv.cnt, (float *)scratch);
    const size_t sp_bytes = lora_split_ws_bytes(g.n_slices, g.in_dim, g.R, meta->T,
                                                max_tiles(meta->T, pool->desc.max_loras));
    const bool have_split_region = sp_bytes <= scratch_bytes;
    g.in = (const uint16_t *)x;
    g.ld_in = ldx;
    g.out = (uint16_t *)y;
    g.ld_out = ldy;
    if (use_sgmv) {
        // long contiguous runs on tcgen05; the remaining groups' 16-row tiles below
        st = lora_sgmv_apply(pool, meta, x, ldx, y, ldy, cv.data, g_spin_limit, pool->num_sms, post_scale, s);
        if (st != LORA_OK) return st;
        g.tile_row0 = meta->stile_row0;
        g.tile_keyn = meta->stile_keyn;
        g.count_idx = 4;
    }
    const int pol = g_lora_kernel_policy;
    if (pol_fused(pol) && !use_sgmv) {
        // decode-sized batches: shrink, reduction and expand in one launch
        bool launched = false;
        st = lora_fused_apply(pool, meta, nullptr, meta->T, x, ldx, y, ldy, post_scale, g_spin_limit, s, &launched);
        if (st != LORA_OK || launched) return st;
    }
    if (pol != 1) {
        bool launched = false;
        const LoraProblem pr = to_problem(g, meta, pool->desc.max_loras);
        if (pol_split(pol) && have_split_region) {
            st = lora_split_apply(pool, pr, scratch, scratch_bytes, cv.ctrl + 2, s, &launched);
            if (st != LORA_OK || launched) return st;
        }
        st = lora_cluster_apply(pool, pr, s, &launched);
        if (st != LORA_OK || launched) return st;
    }
    return launch<kFused>(pool, g, est_items(g, meta->T, pool->desc.max_loras, kFused), s);
}

extern "C" lora_status_t lora_apply_slices(const lora_pool_t *pool, const lora_meta_t *meta,
                                           const void *x, int64_t ldx, void *y, int64_t ldy,
                                           void *workspace, size_t ws_bytes, void *stream) {
    return lora_dense_apply(pool, meta, x, ldx, y, ldy, workspace, ws_bytes, 1.0f, (cudaStream_t)stream);
}

lora_status_t lora_dense_shrink(const lora_pool_t *pool, const lora_meta_t *meta, const void *x, int64_t ldx,
                                void *workspace, size_t ws_bytes, size_t head_bytes, cudaStream_t s, float **part,
                                int *nc, int *r8, int *sorted_rows) {
    GArgs g;
    lora_status_t st = dense_args(pool, meta, g);
    if (st != LORA_OK) return st;
    Carve cv;
    if (!workspace || !lora_aligned16(workspace) || !carve(workspace, ws_bytes, cv) || head_bytes % 256)
        return LORA_ERR_CAPACITY;
    const int T = meta->T;
    g.in = (const uint16_t *)x;
    g.ld_in = ldx;
    char *data = cv.data + head_bytes;
    const size_t sp = align256(lora_split_ws_bytes(g.n_slices, g.in_dim, g.R, T, max_tiles(T, pool->desc.max_loras)));
    if (g_lora_kernel_policy != 1 && head_bytes + sp <= cv.data_bytes) {
        LoraProblem pr = to_problem(g, meta, pool->desc.max_loras);
        int NC = 0;
        pr.shrink_only = 1;
        pr.nc_out = &NC;
        bool launched = false;
        st = lora_split_apply(pool, pr, data, sp, cv.ctrl + 2, s, &launched);
        if (st != LORA_OK) return st;
        if (launched) {
            *part = (float *)data;
            *nc = NC;
            *r8 = lora_round8(g.R);
            *sorted_rows = 1;
            return LORA_OK;
        }
    }
    // the atomic shrink: v [n_slices][T][max_rank] in token order
    if (head_bytes + align256((size_t)g.n_slices * T * g.R * 4) > cv.data_bytes) return LORA_ERR_CAPACITY;
    st = lora_shrink(pool, meta, x, ldx, (float *)data, s);
    if (st != LORA_OK) return st;
    *part = (float *)data;
    *nc = 1;
    *r8 = g.R;
    *sorted_rows = 0;
    return LORA_OK;
}

extern "C" lora_status_t lora_build_meta_apply(const lora_pool_t *pool, const int32_t *d_idx, int32_t T,
                                               lora_meta_t *meta, const void *x, int64_t ldx, void *y, int64_t ldy,
                                               void *workspace, size_t ws_bytes, void *stream) {
    if (!pool || !meta || T < 0 || (T > 0 && !d_idx)) return LORA_ERR_INVALID_ARG;
    if (pool->is_moe) return LORA_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    const lora_pool_desc_t &d = pool->desc;
    if (pol_fused(g_lora_kernel_policy) && T > 0 && T <= meta->max_rows && d.max_loras <= meta->max_keys &&
        meta->sorted && meta->counters && meta->tile_keyn && meta->ltile_keyn && meta->stile_keyn && x && y &&
        lora_aligned16(x) && lora_aligned16(y) && ldx % 8 == 0 && ldy % 8 == 0 && ldx >= d.in_dim &&
        ldy >= out_total(pool)) {
        // one launch: the metadata build and the delta of this layer together
        bool launched = false;
        const lora_status_t st =
            lora_fused_apply(pool, meta, d_idx, T, x, ldx, y, ldy, 1.0f, g_spin_limit, s, &launched);
        if (st != LORA_OK) return st;
        if (launched) {
            meta->T = T;
            meta->top_k = 1;
            meta->n_keys = d.max_loras;
            meta->mode = 0;
            return LORA_OK;
        }
    }
    lora_status_t st = lora_launch_build_meta(pool, d_idx, T, nullptr, 1, meta, s);
    if (st != LORA_OK) return st;
    return lora_dense_apply(pool, meta, x, ldx, y, ldy, workspace, ws_bytes, 1.0f, s);
}

extern "C" lora_status_t lora_shrink(const lora_pool_t *pool, const lora_meta_t *meta,
                                     const void *x, int64_t ldx, float *v, void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    GArgs g;
    lora_status_t st = dense_args(pool, meta, g);
    if (st != LORA_OK) return st;
    if (meta->T == 0) return LORA_OK;
    if (!x || !v || !lora_aligned16(x) || ldx % 8 || ldx < pool->desc.in_dim)
        return LORA_ERR_INVALID_ARG;
    const Plan pl = make_plan(pool->num_sms, g.in_dim, g.n_slices, g.R, meta->T, pool->desc.max_loras);
    g.NC = pl.NC;
    g.HC = pl.HC;
    g.in = (const uint16_t *)x;
    g.ld_in = ldx;
    g.part = v;
    cudaStream_t s = (cudaStream_t)stream;
    LORA_CUDA_TRY(cudaMemsetAsync(v, 0, (size_t)g.n_slices * meta->T * g.R * 4, s));
    return launch<kShrinkAtomic>(pool, g, est_items(g, meta->T, pool->desc.max_loras, kShrinkAtomic), s);
}

extern "C" lora_status_t lora_expand(const lora_pool_t *pool, const lora_meta_t *meta,
                                     const float *v, void *y, int64_t ldy, void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    GArgs g;
    lora_status_t st = dense_args(pool, meta, g);
    if (st != LORA_OK) return st;
    if (meta->T == 0) return LORA_OK;
    if (!v || !y || !lora_aligned16(y) || ldy % 8 || ldy < out_total(pool)) return LORA_ERR_INVALID_ARG;
    g.NC = 1;
    g.HC = 8;
    g.part = (float *)v;
    g.out = (uint16_t *)y;
    g.ld_out = ldy;
    return launch<kExpandOnly>(pool, g, est_items(g, meta->T, pool->desc.max_loras, kExpandOnly),
                               (cudaStream_t)stream);
}

extern "C" lora_status_t lora_moe_apply(const lora_pool_t *pool, const lora_meta_t *meta,
                                        int32_t which, const void *in, int64_t ld_in,
                                        const float *topk_w, void *out, int64_t ld_out,
                                        void *workspace, size_t ws_bytes, void *stream) {
    if (!pool || !meta) return LORA_ERR_INVALID_ARG;
    if (!pool->is_moe) return LORA_ERR_UNSUPPORTED;
    const lora_pool_desc_t &d = pool->desc;
    const int E = d.num_experts;
    if (meta->mode != 1 || meta->n_keys != d.max_loras * E) return LORA_ERR_INVALID_ARG;
    if (which != LORA_MOE_W13 && which != LORA_MOE_W2) return LORA_ERR_INVALID_ARG;
    if (meta->T == 0) return LORA_OK;
    GArgs g;
    memset(&g, 0, sizeof(g));
    const int rows = meta->T * meta->top_k;
    const int n13 = d.n_w13_slices;
    g.E = E;
    g.R = d.max_rank;
    g.T = meta->T;
    g.rows = rows;
    g.post_scale = 1.0f;
    int och = 0;
    if (which == LORA_MOE_W13) {
        g.n_slices = n13;
        g.in_dim = d.d_model;
        g.row_div = meta->top_k;
        for (int s = 0; s < n13; ++s) {
            g.out_w[s] = d.w13_slice_width;
            g.out_off[s] = s * d.w13_slice_width;
            g.och_start[s] = och;
            och += lora_ceil_div(d.w13_slice_width, kOC);
            g.A[s] = pool->A[s];
            g.A_ss[s] = pool->a_slot_elems[s];
            g.A_es[s] = pool->a_experts[s] == 1 ? 0 : (long long)d.max_rank * d.d_model;
            g.B[s] = pool->B[s];
            g.B_ss[s] = pool->b_slot_elems[s];
            g.B_shared[s] = pool->b_experts[s] == 1;
        }
        if (topk_w) return LORA_ERR_INVALID_ARG;
        if (ld_out < (long long)n13 * d.w13_slice_width || ld_in < d.d_model) return LORA_ERR_INVALID_ARG;
    } else {
        g.n_slices = 1;
        g.in_dim = d.d_mlp;
        g.row_div = 1;
        g.out_w[0] = d.d_model;
        g.out_off[0] = 0;
        g.och_start[0] = 0;
        och = lora_ceil_div(d.d_model, kOC);
        g.A[0] = pool->A[n13];
        g.A_ss[0] = pool->a_slot_elems[n13];
        g.A_es[0] = pool->a_experts[n13] == 1 ? 0 : (long long)d.max_rank * d.d_mlp;
        g.B[0] = pool->B[n13];
        g.B_ss[0] = pool->b_slot_elems[n13];
        g.B_shared[0] = pool->b_experts[n13] == 1;
        g.row_w = topk_w;
        if (ld_out < d.d_model || ld_in < d.d_mlp) return LORA_ERR_INVALID_ARG;
    }
    g.och_start[g.n_slices] = och;
    if (!in || !out || !lora_aligned16(in) || !lora_aligned16(out) || ld_in % 8 || ld_out % 8)
        return LORA_ERR_INVALID_ARG;
    g.rank = pool->d_rank;
    g.scale = pool->d_scale;
    g.sorted = meta->sorted;
    g.tile_row0 = meta->tile_row0;
    g.tile_keyn = meta->tile_keyn;
    g.count_idx = 3;
    g.counters = meta->counters;
    g.status = pool->d_status;
    g.in = (const uint16_t *)in;
    g.ld_in = ld_in;
    g.out = (uint16_t *)out;
    g.ld_out = ld_out;
    const int keys = d.max_loras * E;
    if (!workspace || !lora_aligned16(workspace)) return LORA_ERR_INVALID_ARG;
    Carve cv;
    if (!carve(workspace, ws_bytes, cv)) return LORA_ERR_CAPACITY;
    const Plan pl = fit_plan(make_plan(pool->num_sms, g.in_dim, g.n_slices, g.R, rows, keys), g.in_dim,
                             g.n_slices, g.R, rows, cv.data_bytes);
    if (pl.cnt_ints > cv.cnt_cap || pl.part_floats * 4 > cv.data_bytes) return LORA_ERR_CAPACITY;
    bind_splitk(g, pl, cv.ctrl, cv.cnt, (float *)cv.data);
    const size_t sp_bytes = lora_split_ws_bytes(g.n_slices, g.in_dim, g.R, rows, max_tiles(rows, keys));
    const bool have_split_region = sp_bytes <= cv.data_bytes;
    lora_status_t st = LORA_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const int pol = g_lora_kernel_policy;
    const bool sparse = (long long)rows * kSparsityFactor <= keys;
    if ((pol == 5 || ((pol == 0 || pol >= 6) && sparse)) && lora_moe_block_supported(pool, which)) {
        // sparse occupancy: one thread-block cluster per (adapter, expert) key's tile
        return lora_moe_tile_launch(pool, meta, which, in, ld_in, topk_w, out, ld_out, s);
    }
    if (pol == 4 && lora_moe_block_supported(pool, which)) {
        // sparse occupancy: every routed pair a block of its own (block_m 1),
        // aligned into the workspace, then one cluster per block
        const size_t L = d.max_loras;
        const size_t b_sorted = align256(L * rows * 4), b_expert = align256(L * rows * 4);
        if (b_sorted + b_expert + align256(L * 4) <= cv.data_bytes) {
            int32_t *ds = (int32_t *)cv.data;
            int32_t *de = (int32_t *)(cv.data + b_sorted);
            int32_t *dn = (int32_t *)(cv.data + b_sorted + b_expert);
            st = lora_moe_align_launch(pool, meta, 1, rows, ds, de, dn, s);
            if (st != LORA_OK) return st;
            return lora_moe_block_launch(pool, meta, which, in, ld_in, topk_w, out, ld_out, ds, de, dn, 1, rows, s);
        }
    }
    if (pol != 1) {
        bool launched = false;
        LoraProblem pr = to_problem(g, meta, keys);
        // shared-outer w13 (every A_j with expert dimension 1): the shrink of a
        // routed pair is that of its token, computed once per token
        bool shared_a = which == LORA_MOE_W13 && E > 1 && meta->top_k > 1;
        for (int j = 0; j < g.n_slices; ++j) shared_a = shared_a && g.A_es[j] == 0;
        pr.tok_dedup = shared_a ? 1 : 0;
        pr.kmap_base = which == LORA_MOE_W13 ? 0 : n13;  // the pool's tensors: w13 slices, then w2
        if (pol_split(pol) && have_split_region) {
            st = lora_split_apply(pool, pr, cv.data, cv.data_bytes, cv.ctrl + 2, s, &launched);
            if (st != LORA_OK || launched) return st;
        }
        st = lora_cluster_apply(pool, pr, s, &launched);
        if (st != LORA_OK || launched) return st;
    }
    return launch<kFused>(pool, g, est_items(g, rows, keys, kFused), s);
}

// ------------------------------------------------------------------------
// Allocation-free variant of lora_apply_slices.
//
// Some callers cannot hand the library a workspace: a serving engine that
// has already reserved every free byte of HBM for its own pools (KV cache,
// activations) so a further cudaMalloc would fail, a latency-critical path
// that may not block on an allocation, or a plain C host with no allocator
// to lend.  For them the fused kernel can run on a fixed scratch array that
// lives in the library's device image instead.
//
// The array is a file-scope __device__ object of kStaticScratchBytes; every
// GPU that loads this library holds it until the process exits.  Host code
// must not pass the symbol itself to a kernel (on the host it only names a
// shadow copy): the first call on each device, with that device current,
// looks up its device address with cudaGetSymbolAddress and caches it.
// That first call should therefore come before any stream capture.
// All calls share the one array and it keeps the previous call's contents,
// so each call clears the control words it needs at zero; calls that
// overlap on the GPU (two streams, or two host threads) race on it.
namespace {
constexpr size_t kStaticScratchBytes = (size_t)8 << 20;  // 8 MiB
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
std::atomic<void *> g_static_scratch_addr[64];  // looked up once per device
}  // namespace

extern "C" lora_status_t lora_apply_slices_static(const lora_pool_t *pool, const lora_meta_t *meta,
                                                  const void *x, int64_t ldx, void *y, int64_t ldy,
                                                  void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    GArgs g;
    lora_status_t st = dense_args(pool, meta, g);
    if (st != LORA_OK) return st;
    if (meta->T == 0) return LORA_OK;
    if (!x || !y || !lora_aligned16(x) || !lora_aligned16(y) || ldx % 8 || ldy % 8 ||
        ldx < pool->desc.in_dim || ldy < out_total(pool))
        return LORA_ERR_INVALID_ARG;
    int dev = -1;
    LORA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != pool->device || dev < 0 || dev >= 64) return LORA_ERR_INVALID_ARG;
    void *scratch = g_static_scratch_addr[dev].load(std::memory_order_acquire);
    if (!scratch) {
        // two host threads making their first call on this device at once
        // both look the address up and store the same value
        if (cudaGetSymbolAddress(&scratch, g_static_scratch) != cudaSuccess || !scratch) return LORA_ERR_CUDA;
        g_static_scratch_addr[dev].store(scratch, std::memory_order_release);
    }
    const Plan pl0 = make_plan(pool->num_sms, g.in_dim, g.n_slices, g.R, meta->T, pool->desc.max_loras);
    const size_t cnt_bytes = align256(pl0.cnt_ints * 4);
    if (kCtrlBytes + cnt_bytes >= kStaticScratchBytes) return LORA_ERR_CAPACITY;
    const Plan pl = fit_plan(pl0, g.in_dim, g.n_slices, g.R, meta->T, kStaticScratchBytes - kCtrlBytes - cnt_bytes);
    if (ws_bytes_for(pl) > kStaticScratchBytes) return LORA_ERR_CAPACITY;
    bind_splitk(g, pl, (int *)scratch, (int *)((char *)scratch + kCtrlBytes),
                (float *)((char *)scratch + kCtrlBytes + cnt_bytes));
    // ticket, finish count and per-tile counters must start at zero
    LORA_CUDA_TRY(cudaMemsetAsync(scratch, 0, kCtrlBytes + pl.cnt_ints * 4, (cudaStream_t)stream));
    g.in = (const uint16_t *)x;
    g.ld_in = ldx;
    g.out = (uint16_t *)y;
    g.ld_out = ldy;
    return launch<kFused>(pool, g, est_items(g, meta->T, pool->desc.max_loras, kFused),
                          (cudaStream_t)stream);
}

extern "C" size_t lora_static_scratch_bytes(void) { return kStaticScratchBytes; }
