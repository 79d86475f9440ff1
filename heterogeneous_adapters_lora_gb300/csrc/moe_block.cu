// MoE-LoRA over the block-padded alignment: the sparse-occupancy schedule of
// vLLM's FusedMoEWithLoRA.  When num_tokens * top_k * SPARSITY_FACTOR (8) <=
// num_experts * max_loras, most (adapter, expert) keys hold one routed pair or
// none, and the pages give every pair a block of its own instead of padding
// each key's run to BLOCK_M rows.  Here the blocks come from
// lora_moe_align_padded: for adapter a, block b holds block_m pair ids (the
// sentinel T*K pads a run) of expert expert[a][b], and npp[a] / block_m of
// adapter a's blocks are in use.  With block_m = 1 every routed pair is one
// block, which is the naive assignment.
//
// One thread-block cluster of CL CTAs takes one used block at a time:
//   shrink  CTA c sums its 1/CL of the input columns for every
//           (row, slice, rank) of the block:
//             P_c[i][s*r + k] = sum_{h in cols(c)} in[row_i][h] * A_s[a][e'][k][h]
//           warp w takes the (s, k) rows w, w+8, ...; a lane holds its 16-byte
//           chunks of the input row in registers; the warp sums by shuffles
//   reduce  cluster barrier; every CTA adds the CL partials of every value
//           in CTA order through distributed shared memory
//   expand  CTA c takes 1/CL of the output columns, a thread per column:
//             out[row_i][s*W + o] += w_i * scale[a] * sum_{k<r} v[i][s*r + k] * B_s[a][e''][o][k]
//           with the B row in registers for all rows of the block; fp32
//           accumulation, one bf16 rounding
// e' = 0 for a shared-outer A, e'' = 0 for a shared-outer B.  W13: the input
// row of pair p is x[p / K] and w_i = 1; W2: the input row is ic2[p] and w_i
// is the routed weight of p.
#include <string.h>

#include <atomic>

#include "lora_internal.cuh"
#include "mma_common.cuh"

namespace {

using namespace bgmv;

constexpr int kBThreads = 256;
constexpr int kBWarps = kBThreads / 32;
constexpr int kChunksLane = 16;  // at most 16-byte input chunks per lane and row: 4096 columns per CTA
// (slice, rank) rows a warp sums at once: their A chunks stay in registers
__host__ __device__ constexpr int qb_of(int ncl) { return ncl >= 8 ? 1 : ncl >= 4 ? 2 : 4; }
constexpr int kMaxBlockM = 16;   // rows of one block
constexpr int kMaxVR = 128;      // slices x ranks of one row
constexpr int kTabSlots = 256;   // pools of up to this many slots keep rank and scale in shared memory

struct BArgs {
    int n_slices, in_dim, W, E, L, nb;  // W: width of one output slice; nb: blocks per adapter (cap / block_m)
    int block_m, P;                     // P = T * K, the sentinel
    const uint16_t *A[2];
    long long A_ss[2], A_es[2];         // slot and expert strides of A (expert stride 0: shared)
    const uint16_t *B[2];
    long long B_ss[2];
    int B_shared[2];
    const int32_t *rank;
    const float *scale;
    const int32_t *sorted, *expert, *npp;
    const uint16_t *in;
    long long ld_in;
    int row_div;                        // input row of pair p: p / row_div
    uint16_t *out;
    long long ld_out;
    const float *row_w;
    int tiles;                          // 1: the blocks are the metadata's 16-row tiles
    int max_tiles;
    const int32_t *tile_keyn, *tile_row0, *counters;
};

__device__ __forceinline__ float ld_dsmem_f32(const float *local, uint32_t peer) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(peer));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

__device__ __forceinline__ float dot8(const uint4 &a, const uint4 &x) {
    return bf16lo(a.x) * bf16lo(x.x) + bf16hi(a.x) * bf16hi(x.x) + bf16lo(a.y) * bf16lo(x.y) +
           bf16hi(a.y) * bf16hi(x.y) + bf16lo(a.z) * bf16lo(x.z) + bf16hi(a.z) * bf16hi(x.z) +
           bf16lo(a.w) * bf16lo(x.w) + bf16hi(a.w) * bf16hi(x.w);
}

// CL: CTAs per cluster; NCL: 16-byte input chunks per lane (32 * NCL * CL * 8
// input columns at most).
template <int CL, int NCL>
__global__ void __launch_bounds__(kBThreads, 2) moe_block_kernel(const __grid_constant__ BArgs p) {
    __shared__ float s_part[kMaxBlockM * kMaxVR];  // this CTA's partial sums
    __shared__ float s_v[kMaxBlockM * kMaxVR];     // the reduced shrink output
    __shared__ int s_rows[kMaxBlockM];
    __shared__ float s_w[kMaxBlockM];
    __shared__ int s_blk[4];  // adapter (-1: no block left), expert, first entry, entries
    __shared__ int s_rk[kTabSlots];
    __shared__ float s_sc[kTabSlots];
    constexpr int kQB = qb_of(NCL);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int crank = CL > 1 ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    const int nch = p.in_dim >> 3;  // 16-byte chunks of an input row
    const int c0 = crank * nch / CL, c1 = (crank + 1) * nch / CL;
    const int tot = p.n_slices * p.W;  // output columns; this CTA expands [o0, o1)
    const int o0 = crank * tot / CL, o1 = (crank + 1) * tot / CL;
    // the pool's rank and scale tables (written only by lora_set / lora_reset,
    // which the caller orders before the step) before the wait
    if (p.L <= kTabSlots && tid < p.L) {
        s_rk[tid] = __ldg(p.rank + tid);
        s_sc[tid] = __ldg(p.scale + tid);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int j = cid;; j += ncl) {
        // ---- block j: adapter, expert and its entries
        if (warp == 0) {
            int fa = -1, fe = 0, f0 = 0, fn = 0;
            if (p.tiles) {
                // the metadata's 16-row tiles; the count and the tile's words in flight together
                if (lane == 0) {
                    const int nt = p.counters[3];
                    const int keyn = j < p.max_tiles ? p.tile_keyn[j] : 0;
                    const int row0 = j < p.max_tiles ? p.tile_row0[j] : 0;
                    if (j < nt && j < p.max_tiles) {
                        const int key = keyn >> 5;
                        fa = key / p.E;
                        fe = key - fa * p.E;
                        f0 = row0;
                        fn = min(keyn & 31, kMaxBlockM);
                    }
                }
            } else {
                // used block j of all adapters, in adapter order
                int base = 0, fb = 0;
                for (int a0 = 0; a0 < p.L && fa < 0; a0 += 32) {
                    const int a = a0 + lane;
                    const int nblk = a < p.L ? min(p.npp[a] / p.block_m, p.nb) : 0;
                    int incl = nblk;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int v = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += v;
                    }
                    const int excl = base + incl - nblk;
                    const unsigned hit = __ballot_sync(0xffffffffu, j >= excl && j < excl + nblk);
                    if (hit) {
                        const int src = __ffs(hit) - 1;
                        fa = a0 + src;
                        fb = j - __shfl_sync(0xffffffffu, excl, src);
                    }
                    base += __shfl_sync(0xffffffffu, incl, 31);
                }
                if (lane == 0 && fa >= 0) {
                    fe = p.expert[(long long)fa * p.nb + fb];
                    f0 = fa * p.nb * p.block_m + fb * p.block_m;
                    fn = p.block_m;
                }
            }
            if (lane == 0) {
                s_blk[0] = fa;
                s_blk[1] = fe;
                s_blk[2] = f0;
                s_blk[3] = fn;
            }
        }
        __syncthreads();
        const int a = s_blk[0], e = s_blk[1], f0 = s_blk[2], nrow = s_blk[3];
        if (a < 0) break;  // no block left: the same in every CTA of the cluster
        const int r = p.L <= kTabSlots ? s_rk[a] : __ldg(p.rank + a);
        if (e < 0 || e >= p.E || a >= p.L || r <= 0) {
            __syncthreads();  // s_blk is rewritten by the next iteration
            continue;
        }
        const int rs = (r + 7) & ~7;
        const int nv = p.n_slices * r;
        if (tid < nrow) {
            const int row = p.sorted[f0 + tid];
            const bool ok = row >= 0 && row < p.P;
            s_rows[tid] = ok ? row : -1;
            s_w[tid] = ok ? (p.L <= kTabSlots ? s_sc[a] : __ldg(p.scale + a)) * (p.row_w ? p.row_w[row] : 1.f) : 0.f;
        }
        // the B rows of this CTA's output columns into L2 while the shrink runs
        for (int s = 0; s < p.n_slices; ++s) {
            const int lo = max(o0, s * p.W) - s * p.W, hi = min(o1, (s + 1) * p.W) - s * p.W;
            if (lo >= hi) continue;
            const char *base = (const char *)((s == 0 ? p.B[0] + a * p.B_ss[0] + (p.B_shared[0] ? 0ll : (long long)e * p.W * rs)
                                                      : p.B[1] + a * p.B_ss[1] + (p.B_shared[1] ? 0ll : (long long)e * p.W * rs)) +
                                             (long long)lo * rs);
            const int lines = (int)(((long long)(hi - lo) * rs * 2 + 127) >> 7);
            for (int l = tid; l < lines; l += kBThreads) asm volatile("prefetch.global.L2 [%0];" ::"l"(base + l * 128));
        }
        // the first (slice, rank) rows of this warp: A chunks in flight before the rows are known
        uint4 av[kQB][NCL];
        const uint16_t *Ar[kQB];
        auto a_rows = [&](int q0) {
#pragma unroll
            for (int u = 0; u < kQB; ++u) {
                const int q = min(q0 + u * kBWarps, nv - 1);  // duplicates of the last row are not stored
                const int s = q / r, k = q - s * r;
                Ar[u] = (s == 0 ? p.A[0] + a * p.A_ss[0] + e * p.A_es[0] : p.A[1] + a * p.A_ss[1] + e * p.A_es[1]) +
                        (long long)k * p.in_dim;
#pragma unroll
                for (int jj = 0; jj < NCL; ++jj) {
                    const int ch = c0 + lane + 32 * jj;
                    av[u][jj] = ch < c1 ? __ldg((const uint4 *)(Ar[u] + ch * 8)) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
        };
        if (warp < nv) a_rows(warp);
        __syncthreads();  // s_rows, s_w
        // the old output values of this CTA's columns into L2
        {
            const int lines_row = ((o1 - o0) * 2 + 127) >> 7;
            for (int l = tid; l < nrow * lines_row; l += kBThreads) {
                const int i = l / lines_row, row = s_rows[i];
                if (row >= 0)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"((const char *)(p.out + (long long)row * p.ld_out + o0) +
                                                                  (l - i * lines_row) * 128));
            }
        }
        // ---- shrink: partial sums over this CTA's input columns
        for (int q0 = warp; q0 < nv; q0 += kBWarps * kQB) {
            if (q0 != warp) a_rows(q0);
            for (int i = 0; i < nrow; ++i) {
                const int row = s_rows[i];
                if (row < 0) continue;
                const uint16_t *xr = p.in + (long long)(row / p.row_div) * p.ld_in;
                float acc[kQB];
#pragma unroll
                for (int u = 0; u < kQB; ++u) acc[u] = 0.f;
#pragma unroll
                for (int jj = 0; jj < NCL; ++jj) {
                    const int ch = c0 + lane + 32 * jj;
                    const uint4 xv = ch < c1 ? __ldg((const uint4 *)(xr + ch * 8)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int u = 0; u < kQB; ++u) acc[u] += dot8(av[u][jj], xv);
                }
#pragma unroll
                for (int u = 0; u < kQB; ++u) {
#pragma unroll
                    for (int o = 16; o; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
                    const int q = q0 + u * kBWarps;
                    if (lane == 0 && q < nv) (CL > 1 ? s_part : s_v)[i * kMaxVR + q] = acc[u];
                }
            }
        }
        // ---- reduce across the cluster (fixed order)
        if (CL > 1) {
            cluster_arrive();
            cluster_wait();  // every CTA's partials are complete and visible
            for (int t = tid; t < nrow * nv; t += kBThreads) {
                const int i = t / nv, q = t - i * nv;
                if (s_rows[i] < 0) continue;
                float v = 0.f;
#pragma unroll
                for (int c = 0; c < CL; ++c) v += ld_dsmem_f32(s_part + i * kMaxVR + q, (uint32_t)c);
                s_v[i * kMaxVR + q] = v;
            }
            cluster_arrive();  // this CTA has read its peers' partials
        }
        __syncthreads();
        // ---- expand: a thread per output column of this CTA's share
        for (int oc = o0 + tid; oc < o1; oc += kBThreads) {
            const int s = oc / p.W, o = oc - s * p.W;
            const uint16_t *Brow =
                (s == 0 ? p.B[0] + a * p.B_ss[0] + (p.B_shared[0] ? 0ll : (long long)e * p.W * rs)
                        : p.B[1] + a * p.B_ss[1] + (p.B_shared[1] ? 0ll : (long long)e * p.W * rs)) +
                (long long)o * rs;
            uint4 bv[8];
#pragma unroll
            for (int kc = 0; kc < 8; ++kc)
                bv[kc] = kc * 8 < rs ? __ldg((const uint4 *)(Brow + kc * 8)) : make_uint4(0u, 0u, 0u, 0u);
            for (int i = 0; i < nrow; ++i) {
                const int row = s_rows[i];
                if (row < 0) continue;
                const float *v = s_v + i * kMaxVR + s * r;
                float acc = 0.f;
#pragma unroll
                for (int kc = 0; kc < 8; ++kc) {
                    if (kc * 8 < rs) {
                        float vk[8];
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) vk[kk] = kc * 8 + kk < r ? v[kc * 8 + kk] : 0.f;
                        acc += vk[0] * bf16lo(bv[kc].x) + vk[1] * bf16hi(bv[kc].x) + vk[2] * bf16lo(bv[kc].y) +
                               vk[3] * bf16hi(bv[kc].y) + vk[4] * bf16lo(bv[kc].z) + vk[5] * bf16hi(bv[kc].z) +
                               vk[6] * bf16lo(bv[kc].w) + vk[7] * bf16hi(bv[kc].w);
                    }
                }
                __nv_bfloat16 *op = (__nv_bfloat16 *)(p.out + (long long)row * p.ld_out + oc);
                *op = __float2bfloat16_rn(__bfloat162float(*op) + s_w[i] * acc);
            }
        }
        if (CL > 1) cluster_wait();  // the peers have read this CTA's partials
        __syncthreads();             // s_blk, s_rows, s_w and s_v are rewritten by the next block
    }
    asm volatile("griddepcontrol.launch_dependents;");
}

std::atomic<int> g_block_sms[64];

template <int CL, int NCL>
lora_status_t launch_cl(const BArgs &a, int ncl, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(ncl * CL), 1, 1);
    cfg.blockDim = dim3(kBThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = CL;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, moe_block_kernel<CL, NCL>, a));
    lora_note_launch();
    return LORA_OK;
}

template <int CL>
lora_status_t launch_nc_cl(int nc, const BArgs &a, int ncl, cudaStream_t s) {
    switch (nc) {
        case 1: return launch_cl<CL, 1>(a, ncl, s);
        case 2: return launch_cl<CL, 2>(a, ncl, s);
        case 4: return launch_cl<CL, 4>(a, ncl, s);
        case 8: return launch_cl<CL, 8>(a, ncl, s);
        default: return launch_cl<CL, kChunksLane>(a, ncl, s);
    }
}

lora_status_t launch_nc(int cl, int nc, const BArgs &a, int ncl, cudaStream_t s) {
    switch (cl) {
        case 8: return launch_nc_cl<8>(nc, a, ncl, s);
        case 4: return launch_nc_cl<4>(nc, a, ncl, s);
        case 2: return launch_nc_cl<2>(nc, a, ncl, s);
        default: return launch_nc_cl<1>(nc, a, ncl, s);
    }
}

}  // namespace

// Whether the block kernel can take a projection of this pool.
bool lora_moe_block_supported(const lora_pool_t *pool, int which) {
    const lora_pool_desc_t &d = pool->desc;
    const int in_dim = which == LORA_MOE_W13 ? d.d_model : d.d_mlp;
    const int ns = which == LORA_MOE_W13 ? d.n_w13_slices : 1;
    return pool->is_moe && ns <= 2 && in_dim % 8 == 0 && in_dim <= kChunksLane * 32 * 8 && d.max_rank <= 64 &&
           d.max_rank * ns <= kMaxVR;
}

namespace {

BArgs layer_args(const lora_pool_t *pool, const lora_meta_t *meta, int32_t which, const void *in, int64_t ld_in,
                 const float *topk_w, void *out, int64_t ld_out) {
    const lora_pool_desc_t &d = pool->desc;
    const int n13 = d.n_w13_slices;
    BArgs a;
    memset(&a, 0, sizeof(a));
    a.E = d.num_experts;
    a.L = d.max_loras;
    a.P = meta->T * meta->top_k;
    if (which == LORA_MOE_W13) {
        a.n_slices = n13;
        a.in_dim = d.d_model;
        a.W = d.w13_slice_width;
        a.row_div = meta->top_k;
        for (int t = 0; t < n13; ++t) {
            a.A[t] = pool->A[t];
            a.A_ss[t] = pool->a_slot_elems[t];
            a.A_es[t] = pool->a_experts[t] == 1 ? 0 : (long long)d.max_rank * d.d_model;
            a.B[t] = pool->B[t];
            a.B_ss[t] = pool->b_slot_elems[t];
            a.B_shared[t] = pool->b_experts[t] == 1;
        }
    } else {
        a.n_slices = 1;
        a.in_dim = d.d_mlp;
        a.W = d.d_model;
        a.row_div = 1;
        a.A[0] = pool->A[n13];
        a.A_ss[0] = pool->a_slot_elems[n13];
        a.A_es[0] = pool->a_experts[n13] == 1 ? 0 : (long long)d.max_rank * d.d_mlp;
        a.B[0] = pool->B[n13];
        a.B_ss[0] = pool->b_slot_elems[n13];
        a.B_shared[0] = pool->b_experts[n13] == 1;
        a.row_w = topk_w;
    }
    a.rank = pool->d_rank;
    a.scale = pool->d_scale;
    a.in = (const uint16_t *)in;
    a.ld_in = ld_in;
    a.out = (uint16_t *)out;
    a.ld_out = ld_out;
    return a;
}

// `blocks`: an upper bound on the blocks of the launch
lora_status_t launch_blocks(const lora_pool_t *pool, const BArgs &a, long long blocks, cudaStream_t s) {
    const int dev = pool->device < 64 ? pool->device : 63;
    int sms = g_block_sms[dev].load(std::memory_order_relaxed);
    if (!sms) {
        LORA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, pool->device));
        g_block_sms[dev].store(sms, std::memory_order_relaxed);
    }
    if (blocks < 1) blocks = 1;
    // the widest cluster with which every block's cluster is resident at once
    // (two CTAs per SM), one block per cluster; larger batches loop
    const long long slots = 2ll * sms;
    int cl = 1;
    while (cl < 8 && blocks * cl * 2 <= slots) cl *= 2;
    long long ncl = blocks;
    if (ncl > slots / cl) ncl = slots / cl;
    const int per_cta = (a.in_dim / 8 + cl - 1) / cl;  // input chunks of one CTA
    int nc = 1;
    while (nc * 32 < per_cta) nc *= 2;
    return launch_nc(cl, nc, a, (int)ncl, s);
}

}  // namespace

lora_status_t lora_moe_block_launch(const lora_pool_t *pool, const lora_meta_t *meta, int32_t which, const void *in,
                                    int64_t ld_in, const float *topk_w, void *out, int64_t ld_out,
                                    const int32_t *d_sorted, const int32_t *d_expert, const int32_t *d_npp,
                                    int32_t block_m, int32_t cap, cudaStream_t s) {
    BArgs a = layer_args(pool, meta, which, in, ld_in, topk_w, out, ld_out);
    a.nb = cap / block_m;
    a.block_m = block_m;
    a.sorted = d_sorted;
    a.expert = d_expert;
    a.npp = d_npp;
    // every used block holds at least one routed pair: at most P of them
    long long used = (long long)a.L * a.nb;
    if (used > a.P) used = a.P;
    return launch_blocks(pool, a, used, s);
}

lora_status_t lora_moe_tile_launch(const lora_pool_t *pool, const lora_meta_t *meta, int32_t which, const void *in,
                                   int64_t ld_in, const float *topk_w, void *out, int64_t ld_out, cudaStream_t s) {
    BArgs a = layer_args(pool, meta, which, in, ld_in, topk_w, out, ld_out);
    a.tiles = 1;
    a.max_tiles = meta->max_tiles;
    a.sorted = meta->sorted;
    a.tile_keyn = meta->tile_keyn;
    a.tile_row0 = meta->tile_row0;
    a.counters = meta->counters;
    // 16-row tiles of the non-empty keys: at most rows / 16 + min(rows, keys) + 1
    const long long rows = a.P, keys = (long long)a.L * a.E;
    long long bound = rows / LORA_TILE_ROWS + (rows < keys ? rows : keys) + 1;
    if (bound > meta->max_tiles) bound = meta->max_tiles;
    return launch_blocks(pool, a, bound, s);
}

extern "C" lora_status_t lora_moe_apply_blocks(const lora_pool_t *pool, const lora_meta_t *meta, int32_t which,
                                               const void *in, int64_t ld_in, const float *topk_w, void *out,
                                               int64_t ld_out, const int32_t *d_sorted, const int32_t *d_expert,
                                               const int32_t *d_npp, int32_t block_m, int32_t cap, void *stream) {
    if (!pool || !meta) return LORA_ERR_INVALID_ARG;
    if (!pool->is_moe) return LORA_ERR_UNSUPPORTED;
    const lora_pool_desc_t &d = pool->desc;
    if (meta->mode != 1 || meta->n_keys != d.max_loras * d.num_experts) return LORA_ERR_INVALID_ARG;
    if (which != LORA_MOE_W13 && which != LORA_MOE_W2) return LORA_ERR_INVALID_ARG;
    if (block_m < 1 || block_m > kMaxBlockM || cap < block_m || cap % block_m) return LORA_ERR_INVALID_ARG;
    if (!d_sorted || !d_expert || !d_npp) return LORA_ERR_INVALID_ARG;
    const int width = which == LORA_MOE_W13 ? d.n_w13_slices * d.w13_slice_width : d.d_model;
    const int in_w = which == LORA_MOE_W13 ? d.d_model : d.d_mlp;
    if (which == LORA_MOE_W13 && topk_w) return LORA_ERR_INVALID_ARG;
    if (!in || !out || !lora_aligned16(in) || !lora_aligned16(out) || ld_in % 8 || ld_out % 8 || ld_in < in_w ||
        ld_out < width)
        return LORA_ERR_INVALID_ARG;
    if (!lora_moe_block_supported(pool, which)) return LORA_ERR_UNSUPPORTED;
    if (meta->T == 0) return LORA_OK;
    return lora_moe_block_launch(pool, meta, which, in, ld_in, topk_w, out, ld_out, d_sorted, d_expert, d_npp, block_m,
                                 cap, (cudaStream_t)stream);
}
