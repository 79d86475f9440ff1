// Split BGMV: the multi-tenant LoRA delta for small row groups (decode
// tokens, MoE (adapter, expert) groups) as two kernels chained by
// programmatic dependent launch, so that the expand's weight and output
// traffic overlaps the shrink.
//
// The vLLM LoRA layer pages compute add_shrink into a zeroed fp32 buffer
// [n_slices][T][rank] (scale 1.0) and add_expand with add_input=True at the
// slice offsets; add_lora_fused_moe does the same per (adapter, expert).
//
//   bgmv_shrink_kernel: items (16-row tile, slice j, hidden chunk c).  Bulk
//     copies (cp.async.bulk + mbarrier) bring the tile's x rows and the
//     slot's A_j rows of chunk c, 16 ranks at a time; m16n8k16 bf16 MMAs
//     (fp32 accumulate) give the partial v of chunk c, stored unscaled in fp32.
//   bgmv_shrink_tile_kernel: the same items when they fit the grid (one per
//     CTA), all ranks of the slot per stage.
//   bgmv_shrink_slot_kernel: the same partials from one CTA per (key, slice,
//     chunk) that multiplies every tile of the key against its A rows.
//   bgmv_expand_kernel: items (tile, 256 or 512 output columns).  Before it waits
//     for the shrink it bulk-copies its first item's B rows and y rows; it sums
//     the chunk partials of the slices it touches in chunk order, scales them
//     by scale[a] (and the routed weight for MoE w2), splits v into bf16 hi +
//     lo (the expand keeps the fp32 intermediate to ~16 bits), runs the MMAs,
//     updates y in shared memory and writes the rows back with bulk copies.
//   The partials are plain stores (no atomics), so results do not depend on
//   CTA timing; the only state between calls is the item counters, which the
//   last CTA of each grid puts back to zero.
#include <string.h>

#include <algorithm>
#include <atomic>

#include "lora_internal.cuh"
#include "mma_common.cuh"
#include "tc_common.cuh"

namespace {

using namespace bgmv;

constexpr int kSThreads = 128;            // shrink: 4 warps
constexpr int kSWarps = kSThreads / 32;
constexpr int kThreads = 128;             // expand: 4 warps
constexpr int kWarps = kThreads / 32;
constexpr int kTileRows = LORA_TILE_ROWS;
constexpr int kOC = 256;                  // output columns per expand CTA

struct SArgs {
    int n_slices, in_dim, E, row_div, R, R8;
    const uint16_t *A[LORA_MAX_SLICES];
    long long A_ss[LORA_MAX_SLICES], A_es[LORA_MAX_SLICES];
    const int32_t *rank;
    const int32_t *sorted, *tile_row0, *tile_keyn, *counters;
    int count_idx;
    const uint16_t *in;
    long long ld_in;
    int NC, HC, SC;          // hidden chunks, chunk length, stage length (elements)
    int nst;                 // per-tile shrink: bulk-copy ring depth (2..4)
    int xs_stride, as_stride;
    int off_x, off_a, x_stage_bytes, a_stage_bytes, off_red;
    float *part;             // [NC][n_slices][rows][R8], unscaled
    int rows;
    int *status;
    int spin_limit;
    // slot-major variant
    const int32_t *enabled, *key_count, *key_offset;
    int n_slots, x_stages;
    int *ticket;             // [0] next item, [1] finished CTAs; zero between calls
    // token mode of the key-major shrink (an MoE projection whose A has
    // expert dimension 1): keys are slots, each slot's tokens are gathered
    // from its pair range in the MoE order, and partials land at row = token
    int tok_K, tok_E, tok_G, tok_T, off_tok;
};

struct EArgs {
    int n_slices, R, R8, E, out_total, NC;
    int out_w[LORA_MAX_SLICES], out_off[LORA_MAX_SLICES];
    const uint16_t *B[LORA_MAX_SLICES];
    long long B_ss[LORA_MAX_SLICES];
    int B_shared[LORA_MAX_SLICES];
    const int32_t *rank;
    const float *scale;
    const float *row_w;
    float post_scale;
    const int32_t *sorted, *tile_row0, *tile_keyn, *counters;
    int count_idx;
    uint16_t *out;
    long long ld_out;
    const float *part;
    int rows;
    int n_oc, oc_w;          // output column chunks per tile and their width
    int ys_stride, vr_stride;
    int off_b, off_ys, off_vh, off_vl;
    int *ticket;             // [0] next item, [1] finished CTAs; zero between calls
    int *status;
    int spin_limit;
    int v_div, v_rows;       // v_div > 0: partials of row r at row sorted[r] / v_div of v_rows
    const CUtensorMap *kmaps;  // tensor-core expand: B maps of the slices ([slice][rs/8 - 1])
};

// Dynamic work distribution: the CTAs of a one-wave grid take items from a
// counter in the workspace; the last CTA to finish puts the counter back to
// zero for the next call (calls that share a workspace do not overlap).
__device__ __forceinline__ int take_item(int *ticket, int *s_item) {
    if (threadIdx.x == 0) *s_item = atomicAdd(ticket, 1);
    __syncthreads();
    return *s_item;
}
__device__ __forceinline__ void finish_items(int *ticket) {
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(ticket + 1, 1) == (int)gridDim.x - 1) {
            ticket[0] = 0;
            ticket[1] = 0;
            __threadfence();
        }
    }
}

// MMA part of a shrink stage: warp w takes the k steps i = w (mod 4) of the
// stage for every 8-rank block of the slot, so each x fragment is loaded once
// and feeds every block.  NBMAX is the pool's most 8-rank blocks (1, 2, 4, 8);
// consecutive k steps go to SETS separate accumulators, so SETS * nnb MMA
// chains are in flight instead of nnb (a warp-level MMA has a latency of
// hundreds of cycles here, so independent chains are what keeps it busy).
// A rows of (slot a, expert e) for slice j, read from the parameters with
// constant indices (a run-time index into a parameter array is slow).
__device__ __forceinline__ const uint16_t *a_rows(const SArgs &p, int j, int a, int e) {
    const uint16_t *r = p.A[0] + (long long)a * p.A_ss[0] + (long long)e * p.A_es[0];
#pragma unroll
    for (int q = 1; q < LORA_MAX_SLICES; ++q)
        if (q == j) r = p.A[q] + (long long)a * p.A_ss[q] + (long long)e * p.A_es[q];
    return r;
}

template <int NBMAX>
struct ShrinkAcc {
    static constexpr int SETS = NBMAX >= 8 ? 2 : (NBMAX >= 4 ? 4 : 8);  // 8-16 chains per warp
    float v[SETS * NBMAX][4];
};

template <int NBMAX>
__device__ __forceinline__ void shrink_acc_zero(ShrinkAcc<NBMAX> &acc) {
#pragma unroll
    for (int u = 0; u < ShrinkAcc<NBMAX>::SETS * NBMAX; ++u)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc.v[u][q] = 0.f;
}

template <int NBMAX>
__device__ __forceinline__ void shrink_stage_mma(const uint16_t *xs, int xs_stride, const uint16_t *as,
                                                 int as_stride, int len, int nnb, int warp, int lane,
                                                 ShrinkAcc<NBMAX> &acc) {
    constexpr int SETS = ShrinkAcc<NBMAX>::SETS;
    const int steps = (len + 15) >> 4;
    const uint16_t *xq = xs + ((lane & 7) + ((lane >> 3) & 1) * 8) * xs_stride + (lane >> 4) * 8;
    const uint16_t *aq = as + (lane & 7) * as_stride + ((lane >> 3) & 1) * 8;
    for (int i0 = warp; i0 < steps; i0 += kSWarps * SETS) {
#pragma unroll
        for (int q = 0; q < SETS; ++q) {
            const int i = i0 + q * kSWarps;
            if (i < steps) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(xq + i * 16, a0, a1, a2, a3);
                const bool tail = i * 16 + 8 >= len;
                if (tail) a2 = a3 = 0u;
#pragma unroll
                for (int nb = 0; nb < NBMAX; ++nb) {
                    if (nb < nnb) {
                        uint32_t b0, b1;
                        ldsm_x2(aq + nb * 8 * as_stride + i * 16, b0, b1);
                        if (tail) b1 = 0u;
                        mma16816(acc.v[q * NBMAX + nb], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
        }
    }
}

// Writes a warp's accumulators (rows < n, ranks < r) into its [16][R8] slice of red.
template <int NBMAX>
__device__ __forceinline__ void shrink_store_red(float *red, int R8, int nnb, int r, int n, int warp, int lane,
                                                 const ShrinkAcc<NBMAX> &acc) {
    constexpr int SETS = ShrinkAcc<NBMAX>::SETS;
    const int g = lane >> 2, c4 = lane & 3;
    float *base = red + warp * kTileRows * R8;
#pragma unroll
    for (int nb = 0; nb < NBMAX; ++nb) {
        if (nb < nnb) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k = nb * 8 + 2 * c4 + h;
                float lo = 0.f, hi = 0.f;
#pragma unroll
                for (int q = 0; q < SETS; ++q) {
                    lo += acc.v[q * NBMAX + nb][h];
                    hi += acc.v[q * NBMAX + nb][2 + h];
                }
                if (k < r) {
                    if (g < n) base[g * R8 + k] = lo;
                    if (g + 8 < n) base[(g + 8) * R8 + k] = hi;
                }
            }
        }
    }
}

// ---------------------------------------------------------------- shrink, one item per CTA
//
// For batches whose per-tile items fit the grid (one item per CTA): items
// (16-row tile, slice j, hidden chunk c), two stages of [16 x rows][r A rows]
// x SC columns, rows padded by 16 bytes so ldmatrix reads are free of bank
// conflicts; the MMAs as in shrink_stage_mma, the four warps' partial sums
// added in shared memory (reusing the stages).  With one item per CTA there
// is nothing to run ahead to, and this shorter chain starts sooner than the
// copy-warp kernel below.

template <int NBMAX>
__global__ void __launch_bounds__(kSThreads) bgmv_shrink_tile_kernel(const __grid_constant__ SArgs p) {
    extern __shared__ __align__(128) char smem[];
    __shared__ __align__(8) uint64_t full[4];
    __shared__ int s_rows[kTileRows];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int per_tile = p.n_slices * p.NC;

    __shared__ int s_item;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_tiles = p.counters[p.count_idx];
    const int total = n_tiles * per_tile;
    // the expand may launch and prefetch its weights and outputs now
    asm volatile("griddepcontrol.launch_dependents;");
    if (tid < p.nst) mbar_init(&full[tid], 1);
    if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    float *red = (float *)(smem + p.off_red);
    int gs = 0;  // sub-stages consumed by this CTA so far (ring slot and phase)

    // more items than CTAs: take them from the counter; else one item per CTA
    const bool dyn = total > (int)gridDim.x;
    for (int item = dyn ? take_item(p.ticket, &s_item) : (int)blockIdx.x; item < total;
         item = dyn ? take_item(p.ticket, &s_item) : total) {
        const int tile = item / per_tile, rem = item - tile * per_tile;
        const int j = rem / p.NC, c = rem - j * p.NC;
        const int row0 = p.tile_row0[tile];
        const int keyn = p.tile_keyn[tile];
        const int n = keyn & 31, key = keyn >> 5;
        const int a = key / p.E, e = key - a * p.E;
        const int r = p.rank[a];
        const uint16_t *Ab = a_rows(p, j, a, e);
        const int hb = c * p.HC, he = min(p.in_dim, hb + p.HC);
        const int n_sub = (he - hb + p.SC - 1) / p.SC;
        __syncthreads();  // the previous item is done with s_rows, the stages and red
        if (tid < n) s_rows[tid] = p.sorted[row0 + tid];
        __syncthreads();

        auto issue = [&](int s) {
            const int h0 = hb + s * p.SC, len = min(p.SC, he - h0), st = (gs + s) % p.nst;
            uint16_t *xs = (uint16_t *)(smem + p.off_x + st * p.x_stage_bytes);
            uint16_t *as = (uint16_t *)(smem + p.off_a + st * p.a_stage_bytes);
            const uint32_t rowb = (uint32_t)len * 2;
            if (lane == 0) mbar_expect_tx(&full[st], rowb * (uint32_t)(n + r));
            __syncwarp();
            for (int i = lane; i < n + r; i += 32) {
                if (i < n)
                    bulk_g2s(xs + i * p.xs_stride, p.in + (long long)(s_rows[i] / p.row_div) * p.ld_in + h0, rowb,
                             &full[st]);
                else
                    bulk_g2s(as + (i - n) * p.as_stride, Ab + (long long)(i - n) * p.in_dim + h0, rowb, &full[st]);
            }
        };
        if (warp == 0) {
            // the stages were last read through the generic proxy
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            for (int s = 0; s < min(n_sub, p.nst); ++s) issue(s);
        }

        const int nnb = (r + 7) >> 3;
        ShrinkAcc<NBMAX> acc;
        shrink_acc_zero(acc);
        for (int s = 0; s < n_sub; ++s) {
            const int st = (gs + s) % p.nst;
            mbar_wait(&full[st], (uint32_t)(((gs + s) / p.nst) & 1), p.spin_limit, p.status);
            const int len = min(p.SC, he - hb - s * p.SC);
            const uint16_t *xs = (const uint16_t *)(smem + p.off_x + st * p.x_stage_bytes);
            const uint16_t *as = (const uint16_t *)(smem + p.off_a + st * p.a_stage_bytes);
            shrink_stage_mma(xs, p.xs_stride, as, p.as_stride, len, nnb, warp, lane, acc);
            __syncthreads();
            if (warp == 0 && s + p.nst < n_sub) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(s + p.nst);
            }
        }
        gs += n_sub;

        // partials of this chunk: [4 warps][16][R8] in shared memory, summed
        // over the warps, then one row of R8 floats per token to global memory
        for (int i = tid; i < kSWarps * kTileRows * p.R8; i += kSThreads) red[i] = 0.f;
        __syncthreads();
        shrink_store_red(red, p.R8, nnb, r, n, warp, lane, acc);
        __syncthreads();
        // this chunk's partial: part[c][j][row0 + t][k]
        float *dst = p.part + ((long long)c * p.n_slices + j) * p.rows * p.R8 + (long long)row0 * p.R8;
        for (int i = tid; i < n * p.R8; i += kSThreads) {
            const int t = i / p.R8, k = i - t * p.R8;
            float sum = 0.f;
            for (int w = 0; w < kSWarps; ++w) sum += red[(w * kTileRows + t) * p.R8 + k];
            dst[i] = sum;
        }
    }
    if (dyn) finish_items(p.ticket);
}

// ---------------------------------------------------------------- shrink
//
// Items (16-row tile, slice j, hidden chunk c), spread over a grid of at
// most a few waves.  The slot's ranks are taken kRG at a time: for each rank
// group the chunk streams through a ring of stages holding the tile's x rows
// and the group's A rows, SC columns each (rows padded by 16 bytes so
// ldmatrix reads are free of bank conflicts).  Few rows per stage keep the
// stages wide, so every row copy is long whatever the rank; the x rows are
// fetched again for each group (from L2).
//
// Warp-specialized: a copy warp takes the items (from the counter), hands
// each to the MMA warps through a two-entry descriptor ring and issues its
// stages as ring slots come free, running ahead across items; the four MMA
// warps wait for full stages, multiply (as in shrink_stage_mma), release the
// slot, and at the end of a rank group add their sums in shared memory and
// store the group's ranks of the unscaled chunk partial.  No CTA-wide barrier
// sits between stages or items.

constexpr int kRG = 16;                      // ranks per group (two 8-rank MMA blocks)
constexpr int kPThreads = kSThreads + 32;    // per-tile shrink: 4 MMA warps + 1 copy warp

struct ShrinkItem {
    int valid, row0, n, r, j, c;
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int NBMAX>  // 1 or 2: 8-rank blocks of a group
__global__ void __launch_bounds__(kPThreads) bgmv_shrink_kernel(const __grid_constant__ SArgs p) {
    extern __shared__ __align__(128) char smem[];
    __shared__ __align__(8) uint64_t full[4], empty[4], ifull[2], iempty[2];
    __shared__ ShrinkItem s_info[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per_tile = p.n_slices * p.NC;
    const int nst = p.nst;
    if (tid == 0) {
        for (int q = 0; q < nst; ++q) {
            mbar_init(&full[q], 1);
            mbar_init(&empty[q], kSWarps);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&ifull[q], 1);
            mbar_init(&iempty[q], kSWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_tiles = p.counters[p.count_idx];
    const int total = n_tiles * per_tile;
    // the expand may launch and prefetch its weights and outputs now
    asm volatile("griddepcontrol.launch_dependents;");
    // more items than CTAs: take them from the counter; else one item per CTA
    const bool dyn = total > (int)gridDim.x;

    if (warp == kSWarps) {
        // ---------------- copy warp
        int gs = 0;  // stages issued by this CTA (ring slot and phase)
        int item = (int)blockIdx.x;
        if (dyn) {
            int t = 0;
            if (lane == 0) t = atomicAdd(p.ticket, 1);
            item = __shfl_sync(~0u, t, 0);
        }
        for (int ii = 0;; ++ii) {
            const int k = ii & 1;
            mbar_wait(&iempty[k], ((ii >> 1) & 1) ^ 1, p.spin_limit, p.status);
            if (item >= total) {
                if (lane == 0) {
                    s_info[k].valid = 0;
                    mbar_arrive(&ifull[k]);
                }
                break;
            }
            const int tile = item / per_tile, rem = item - tile * per_tile;
            const int j = rem / p.NC, c = rem - j * p.NC;
            const int row0 = p.tile_row0[tile];
            const int keyn = p.tile_keyn[tile];
            const int n = keyn & 31, key = keyn >> 5;
            const int a = key / p.E, e = key - a * p.E;
            const int r = p.rank[a];
            if (lane == 0) {
                s_info[k].valid = 1;
                s_info[k].row0 = row0;
                s_info[k].n = n;
                s_info[k].r = r;
                s_info[k].j = j;
                s_info[k].c = c;
                mbar_arrive(&ifull[k]);  // release: the MMA warps read the descriptor after their wait
            }
            // lane i < n copies x row i of the tile
            const long long xrow = lane < n ? (long long)(p.sorted[row0 + lane] / p.row_div) * p.ld_in : 0ll;
            const uint16_t *Ab = a_rows(p, j, a, e);
            const int hb = c * p.HC, he = min(p.in_dim, hb + p.HC);
            const int n_sub = (he - hb + p.SC - 1) / p.SC;
            const int n_stage = n_sub * ((r + kRG - 1) / kRG);  // groups x column stages
            for (int s = 0; s < n_stage; ++s, ++gs) {
                const int st = gs % nst;
                mbar_wait(&empty[st], ((gs / nst) & 1) ^ 1, p.spin_limit, p.status);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                const int g = s / n_sub, sub = s - g * n_sub;
                const int h0 = hb + sub * p.SC, len = min(p.SC, he - h0);
                const int rg = min(kRG, r - g * kRG);
                uint16_t *xs = (uint16_t *)(smem + p.off_x + st * p.x_stage_bytes);
                uint16_t *as = (uint16_t *)(smem + p.off_a + st * p.a_stage_bytes);
                const uint16_t *Ag = Ab + (long long)g * kRG * p.in_dim + h0;
                const uint32_t rowb = (uint32_t)len * 2;
                if (lane == 0) mbar_expect_tx(&full[st], rowb * (uint32_t)(n + rg));
                __syncwarp();
                for (int i = lane; i < n + rg; i += 32) {
                    if (i < n)
                        bulk_g2s(xs + i * p.xs_stride, p.in + xrow + h0, rowb, &full[st]);
                    else
                        bulk_g2s(as + (i - n) * p.as_stride, Ag + (long long)(i - n) * p.in_dim, rowb, &full[st]);
                }
            }
            if (dyn) {
                int t = 0;
                if (lane == 0) t = atomicAdd(p.ticket, 1);
                item = __shfl_sync(~0u, t, 0);
            } else {
                item = total;
            }
        }
        return;  // the MMA warps synchronise among themselves from here on
    }

    // ---------------- MMA warps
    float *red = (float *)(smem + p.off_red);  // [2][4 warps][16][kRG], apart from the stages
    int gs = 0, gg = 0;                        // stages and rank groups consumed
    for (int ii = 0;; ++ii) {
        const int k = ii & 1;
        mbar_wait(&ifull[k], (ii >> 1) & 1, p.spin_limit, p.status);
        const ShrinkItem it = s_info[k];
        __syncwarp();
        if (lane == 0) mbar_arrive(&iempty[k]);
        if (!it.valid) break;
        const int n = it.n, r = it.r, j = it.j, c = it.c, row0 = it.row0;
        const int hb = c * p.HC, he = min(p.in_dim, hb + p.HC);
        const int n_sub = (he - hb + p.SC - 1) / p.SC;
        const int n_stage = n_sub * ((r + kRG - 1) / kRG);
        ShrinkAcc<NBMAX> acc;
        shrink_acc_zero(acc);
        for (int s = 0; s < n_stage; ++s, ++gs) {
            const int st = gs % nst;
            const int g = s / n_sub, sub = s - g * n_sub;
            const int rg = min(kRG, r - g * kRG), nnb = (rg + 7) >> 3;
            mbar_wait(&full[st], (uint32_t)((gs / nst) & 1), p.spin_limit, p.status);
            const int len = min(p.SC, he - hb - sub * p.SC);
            const uint16_t *xs = (const uint16_t *)(smem + p.off_x + st * p.x_stage_bytes);
            const uint16_t *as = (const uint16_t *)(smem + p.off_a + st * p.a_stage_bytes);
            shrink_stage_mma(xs, p.xs_stride, as, p.as_stride, len, nnb, warp, lane, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the slot
            if (sub == n_sub - 1) {
                // group g of this chunk: the warps' sums (double-buffered: the
                // barrier of the next group orders this group's reads before
                // the buffer is written again), then ranks g*kRG.. of each row
                // to part[c][j][row0 + t][g*kRG + k]
                float *rb = red + (gg & 1) * (kSWarps * kTileRows * kRG);
                shrink_store_red(rb, kRG, nnb, rg, n, warp, lane, acc);
                asm volatile("bar.sync 1, %0;" ::"n"(kSThreads) : "memory");
                const int gw = min(kRG, p.R8 - g * kRG);
                float *dst = p.part + ((long long)c * p.n_slices + j) * p.rows * p.R8 + (long long)row0 * p.R8 +
                             g * kRG;
                for (int i = tid; i < n * gw; i += kSThreads) {
                    const int t = i / gw, kk = i - t * gw;
                    float sum = 0.f;
                    if (kk < rg)
                        for (int w = 0; w < kSWarps; ++w) sum += rb[(w * kTileRows + t) * kRG + kk];
                    dst[(long long)t * p.R8 + kk] = sum;
                }
                shrink_acc_zero(acc);
                ++gg;
            }
        }
    }
    if (dyn) finish_items(p.ticket);
}

// ---------------------------------------------------------------- shrink, key-major
//
// For pools whose keys (slot, or slot x expert for MoE) are mostly busy in
// the batch: one CTA per (key, slice j, hidden chunk c).  The key's A rows of
// the chunk do not depend on this batch's metadata, so they are requested
// before the kernel waits for the metadata build; then every 16-row tile of
// the key's rows is multiplied against them (A read once per key, not once
// per tile).  The partials land where the per-tile shrink would put them.

// Token mode (tok_K > 0): an MoE projection whose A_j has expert dimension 1
// (the shared-outer layout) has a shrink that depends on the token and its
// slot only, so it is computed once per token instead of once per routed
// pair.  Keys are then the slots; a slot's tokens are the distinct pair / K
// over its pair range of the MoE order (every expert key of the slot), in
// ascending token order; tok_G CTAs share a (slot, slice, chunk) and take its
// tiles round robin; the partials land at row = token of [tok_T] rows.

// This slot's tokens, ascending, into tok[] (a bitmap over the tokens after
// it); returns their count.  Every thread calls it.
__device__ int gather_slot_tokens(const SArgs &p, int a, int *tok, int *s_ws) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = p.tok_T, nw = (T + 31) >> 5;
    unsigned *bm = (unsigned *)(tok + T);
    for (int i = tid; i < nw; i += kSThreads) bm[i] = 0u;
    __syncthreads();
    const int s0 = p.key_offset[a * p.tok_E], s1 = p.key_offset[(a + 1) * p.tok_E];
    for (int q = s0 + tid; q < s1; q += kSThreads) {
        const int t = p.sorted[q] / p.tok_K;
        atomicOr(bm + (t >> 5), 1u << (t & 31));
    }
    __syncthreads();
    // each thread a run of words; an exclusive scan of the runs' counts
    const int wpt = (nw + kSThreads - 1) / kSThreads;
    const int w0 = min(nw, tid * wpt), w1 = min(nw, w0 + wpt);
    int mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(bm[w]);
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) s_ws[warp] = incl;
    __syncthreads();
    int base = incl - mine, total = 0;
#pragma unroll
    for (int w = 0; w < kSWarps; ++w) {
        if (w < warp) base += s_ws[w];
        total += s_ws[w];
    }
    for (int w = w0; w < w1; ++w) {
        unsigned m = bm[w];
        while (m) {
            tok[base++] = w * 32 + __ffs(m) - 1;
            m &= m - 1u;
        }
    }
    __syncthreads();
    return total;
}

template <int NBMAX>
__global__ void __launch_bounds__(kSThreads) bgmv_shrink_slot_kernel(const __grid_constant__ SArgs p) {
    extern __shared__ __align__(128) char smem[];
    __shared__ __align__(8) uint64_t abar, xbar[2];
    __shared__ int s_rows[2][kTileRows];
    __shared__ int s_ws[kSWarps];
    const int XS = p.x_stages;  // 1 or 2
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool tmode = p.tok_K > 0;
    const int G = tmode ? p.tok_G : 1;
    const int gi = blockIdx.x % G, bid = blockIdx.x / G;

    const int c = bid % p.NC, j = (bid / p.NC) % p.n_slices, key = bid / (p.NC * p.n_slices);
    const int a = key / p.E, e = key - a * p.E;
    const int hb = c * p.HC, he = min(p.in_dim, hb + p.HC), len = he - hb;
    const uint16_t *Ab = a_rows(p, j, a, e);
    uint16_t *as = (uint16_t *)(smem + p.off_a);
    // tables written before the metadata build started (never by it): read through L2
    const int r = (__ldcg(p.enabled + a) != 0) ? __ldcg(p.rank + a) : 0;
    if (r <= 0) {
        // Even with nothing to do, trigger the expand only once the metadata
        // build is complete: the expand reads the tile lists and rewrites y
        // rows before its own wait, which is safe only because every CTA of
        // this grid has waited before it triggers.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
        return;
    }
    if (tid == 0) {
        mbar_init(&abar, 1);
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint32_t rowb = (uint32_t)len * 2;
    if (warp == 0) {
        if (lane == 0) mbar_expect_tx(&abar, rowb * (uint32_t)r);
        __syncwarp();
        for (int k = lane; k < r; k += 32)
            bulk_g2s(as + k * p.as_stride, Ab + (long long)k * p.in_dim + hb, rowb, &abar);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    int *tok = (int *)(smem + p.off_tok);  // token mode: the slot's tokens
    int cnt, off = 0;
    if (tmode) {
        cnt = gather_slot_tokens(p, a, tok, s_ws);
    } else {
        cnt = p.key_count[key];
        off = p.key_offset[key];
    }
    const int n_t = (cnt + kTileRows - 1) / kTileRows;
    const int n_my = n_t > gi ? (n_t - gi + G - 1) / G : 0;  // tiles gi, gi + G, ... of the key

    auto load_x = [&](int i) {  // x rows of this CTA's i-th tile into stage i % XS (warp 0)
        const int st = i % XS, tile = gi + i * G, n = min(kTileRows, cnt - tile * kTileRows);
        uint16_t *xs = (uint16_t *)(smem + p.off_x + st * p.x_stage_bytes);
        if (lane < n) s_rows[st][lane] = tmode ? tok[tile * kTileRows + lane] : p.sorted[off + tile * kTileRows + lane];
        __syncwarp();
        if (lane == 0) mbar_expect_tx(&xbar[st], rowb * (uint32_t)n);
        __syncwarp();
        if (lane < n)
            bulk_g2s(xs + lane * p.xs_stride, p.in + (long long)(s_rows[st][lane] / p.row_div) * p.ld_in + hb, rowb,
                     &xbar[st]);
    };
    if (warp == 0) {
        if (n_my > 0) load_x(0);
        if (n_my > 1 && XS > 1) load_x(1);
    }
    mbar_wait(&abar, 0, p.spin_limit, p.status);  // also before any exit: no copy may be in flight

    const int nnb = (r + 7) >> 3;
    float *red = (float *)(smem + p.off_red);
    for (int i = 0; i < n_my; ++i) {
        const int st = i % XS, tile = gi + i * G;
        const int row0 = off + tile * kTileRows, n = min(kTileRows, cnt - tile * kTileRows);
        mbar_wait(&xbar[st], (uint32_t)((i / XS) & 1), p.spin_limit, p.status);
        const uint16_t *xs = (const uint16_t *)(smem + p.off_x + st * p.x_stage_bytes);
        ShrinkAcc<NBMAX> acc;
        shrink_acc_zero(acc);
        shrink_stage_mma(xs, p.xs_stride, as, p.as_stride, len, nnb, warp, lane, acc);
        __syncthreads();  // every warp is done with x stage st and with red of the previous tile
        if (warp == 0 && i + XS < n_my) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            load_x(i + XS);
        }
        for (int q = tid; q < kSWarps * kTileRows * p.R8; q += kSThreads) red[q] = 0.f;
        __syncthreads();
        shrink_store_red(red, p.R8, nnb, r, n, warp, lane, acc);
        __syncthreads();
        float *dst = p.part + ((long long)c * p.n_slices + j) * p.rows * p.R8;
        for (int q = tid; q < n * p.R8; q += kSThreads) {
            const int t2 = q / p.R8, k = q - t2 * p.R8;
            float sum = 0.f;
            for (int w = 0; w < kSWarps; ++w) sum += red[(w * kTileRows + t2) * p.R8 + k];
            const long long prow = tmode ? tok[tile * kTileRows + t2] : row0 + t2;
            dst[prow * p.R8 + k] = sum;
        }
    }
}

// ---------------------------------------------------------------- expand

// Slice of output column o (slices are contiguous and ascending).  The loop has
// constant indices into the parameter array: an indexed parameter load with a
// run-time index costs hundreds of cycles.
__device__ __forceinline__ int slice_of(const EArgs &p, int o) {
    int j = 0;
#pragma unroll
    for (int q = 1; q < LORA_MAX_SLICES; ++q)
        if (q < p.n_slices && o >= p.out_off[q]) j = q;
    return j;
}

__device__ __forceinline__ uint32_t lds32(const void *a) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(a)));
    return v;
}
__device__ __forceinline__ void sts32(void *a, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(smem_u32(a)), "r"(v) : "memory");
}

//
// Items (tile, 256 output columns), tile-major, strided over the grid.  The
// first item's B rows and y rows are requested before the shrink is waited
// for; the metadata was complete before the shrink started.

// KS: the most 16-rank k steps of any slot (ceil(R8 / 16), 1..4).
// Narrow passes keep 5 CTAs per SM, except for ranks above 32, whose larger v
// fragments would spill there: 4 (the many-adapter batch measured 6% faster).
template <int KS, int PW>
__global__ void __launch_bounds__(kThreads, PW == 8 ? 3 : (KS >= 3 ? 4 : 5))
    bgmv_expand_kernel(const __grid_constant__ EArgs p) {
    extern __shared__ __align__(128) char smem[];
    __shared__ __align__(8) uint64_t bbar, ybar;
    __shared__ int s_rows[2][kTileRows];  // this item's rows and the next one's
    __shared__ float s_w[kTileRows];
    __shared__ int s_next, s_ninfo[3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c4 = lane & 3;
    const int ns = p.n_slices;
    __shared__ int s_item;
    const int n_tiles = p.counters[p.count_idx];
    const int total = n_tiles * p.n_oc;
    if (tid == 0) {
        mbar_init(&bbar, 1);
        mbar_init(&ybar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    uint16_t *bs = (uint16_t *)(smem + p.off_b);
    uint16_t *ys = (uint16_t *)(smem + p.off_ys);
    uint16_t *vh = (uint16_t *)(smem + p.off_vh);
    uint16_t *vl = (uint16_t *)(smem + p.off_vl);
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
    bool waited = false;
    const int nc = p.NC;
    uint32_t phase = 0;

    // more items than CTAs: take them from the counter; else one item per CTA.
    // The next item's ticket, tile words, rank and rows are fetched while this
    // item converts its partials, runs its MMAs and stores its rows, so an
    // item starts with its bulk copies instead of a chain of dependent loads.
    const bool dyn = total > (int)gridDim.x;
    int item = dyn ? take_item(p.ticket, &s_item) : (int)blockIdx.x;
    int row0 = 0, keyn = 0, r = 0, buf = 0;
    if (item < total) {
        const int tile = item / p.n_oc;
        row0 = p.tile_row0[tile];
        keyn = p.tile_keyn[tile];
        r = p.rank[(keyn >> 5) / p.E];
        if (tid < (keyn & 31)) s_rows[0][tid] = p.sorted[row0 + tid];
    }
    __syncthreads();
    for (; item < total; phase ^= 1u, buf ^= 1) {
        const int tile = item / p.n_oc, oc = item - tile * p.n_oc;
        const int n = keyn & 31, key = keyn >> 5;
        const int a = key / p.E, e = key - a * p.E;
        const int rs = (r + 7) & ~7;
        const int ob = oc * p.oc_w, oe = min(p.out_total, ob + p.oc_w);
        const int *rows = s_rows[buf];
        int nxt_t = total;
        if (dyn && tid == 0) nxt_t = atomicAdd(p.ticket, 1);  // lands while this item runs
        // weights and outputs do not depend on the shrink: fetch them first
        if (warp == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint32_t rowb = (uint32_t)(oe - ob) * 2;
            if (lane == 0) mbar_expect_tx(&ybar, rowb * (uint32_t)n);
            __syncwarp();
            if (lane < n)
                bulk_g2s(ys + lane * p.ys_stride, p.out + (long long)rows[lane] * p.ld_out + ob, rowb, &ybar);
        } else if (warp == 1) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (lane == 0) mbar_expect_tx(&bbar, (uint32_t)(oe - ob) * rs * 2);
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < LORA_MAX_SLICES; ++jj) {  // constant parameter indices
                if (jj < ns && lane == jj) {
                    const int s0 = max(ob, p.out_off[jj]), s1 = min(oe, p.out_off[jj] + p.out_w[jj]);
                    if (s1 > s0) {
                        const uint16_t *Bj = p.B[jj] + (long long)a * p.B_ss[jj] +
                                             (p.B_shared[jj] ? 0ll : (long long)e * p.out_w[jj] * rs);
                        bulk_g2s(bs + (long long)(s0 - ob) * rs, Bj + (long long)(s0 - p.out_off[jj]) * rs,
                                 (uint32_t)(s1 - s0) * rs * 2, &bbar);
                    }
                }
            }
        }
        if (tid < kTileRows)
            s_w[tid] = tid < n ? p.scale[a] * p.post_scale * (p.row_w ? p.row_w[rows[tid]] : 1.f) : 0.f;
        if (!waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // the shrink's partials are complete
            waited = true;
        }
        __syncthreads();
        // v of the slices this item touches (chunk partials summed in order,
        // scaled) -> bf16 hi / lo, [16][vr_stride] at j * R8 + k
        const int j0 = slice_of(p, ob), j1 = slice_of(p, oe - 1);
        // 16 rows x 8 threads, 4 ranks per thread and step: no divisions
        const int tq = tid >> 3, lq = tid & 7;
        const int vrows = p.v_div > 0 ? p.v_rows : p.rows;
        const long long cstride = (long long)ns * vrows * p.R8 / 4;
        const int prow = tq < n ? (p.v_div > 0 ? rows[tq] / p.v_div : row0 + tq) : 0;
        for (int jj = j0; jj <= j1; ++jj) {
            for (int k = lq * 4; k < p.R8; k += 32) {
                float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tq < n) {
                    const float4 *src =
                        (const float4 *)(p.part + ((long long)jj * vrows + prow) * p.R8 + k);
                    for (int cc = 0; cc < nc; ++cc) {
                        const float4 v = __ldcg(src + cc * cstride);
                        s4.x += v.x;
                        s4.y += v.y;
                        s4.z += v.z;
                        s4.w += v.w;
                    }
                    const float w = s_w[tq];
                    s4.x *= w;
                    s4.y *= w;
                    s4.z *= w;
                    s4.w *= w;
                }
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(s4.x, s4.y);
                const __nv_bfloat162 h23 = __floats2bfloat162_rn(s4.z, s4.w);
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                uint2 hv, lv;
                hv.x = *(const uint32_t *)&h01;
                hv.y = *(const uint32_t *)&h23;
                lv.x = pack_bf16x2(s4.x - f01.x, s4.y - f01.y);
                lv.y = pack_bf16x2(s4.z - f23.x, s4.w - f23.y);
                *(uint2 *)(vh + tq * p.vr_stride + jj * p.R8 + k) = hv;
                *(uint2 *)(vl + tq * p.vr_stride + jj * p.R8 + k) = lv;
            }
        }
        if (tid == 0) s_next = nxt_t;
        __syncthreads();
        // the next item's tile words, in flight during the MMAs
        const int nitem = s_next;
        int nrow0 = 0, nkeyn = 0;
        if (nitem < total && tid < kTileRows) {
            const int nt = nitem / p.n_oc;
            nrow0 = p.tile_row0[nt];
            nkeyn = p.tile_keyn[nt];
        }
        mbar_wait(&bbar, phase, p.spin_limit, p.status);
        mbar_wait(&ybar, phase, p.spin_limit, p.status);

        const int nob = (oe - ob) >> 3;
        const int ksteps = (rs + 15) >> 4;  // <= KS
        // The v fragments (hi, lo) depend only on the slice and the k step: kept in
        // registers while a warp's blocks stay in one slice.  A warp-level MMA has
        // a latency of hundreds of cycles here, so each pass issues the MMAs of up
        // to PW of the warp's 8-column blocks before it reads any result, and then
        // does all their y updates (loads first, then stores).  PW = 8 for batches
        // that fit two waves, 4 (fewer registers, more resident CTAs) otherwise.
        uint32_t hf[KS][4], lf[KS][4];
        int cur = -1;
        auto load_v = [&](int jj) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if (ks < ksteps) {
                    const int col = jj * p.R8 + ks * 16 + (lane >> 4) * 8;
                    ldsm_x4(vh + arow * p.vr_stride + col, hf[ks][0], hf[ks][1], hf[ks][2], hf[ks][3]);
                    ldsm_x4(vl + arow * p.vr_stride + col, lf[ks][0], lf[ks][1], lf[ks][2], lf[ks][3]);
                    if (ks * 16 + 8 >= rs) hf[ks][2] = hf[ks][3] = lf[ks][2] = lf[ks][3] = 0u;
                }
            }
        };
        const uint16_t *bq = bs + (lane & 7) * rs + ((lane >> 3) & 1) * 8;
#pragma unroll 1
        for (int p0 = warp; p0 < nob; p0 += PW * kWarps) {
            int jq[PW];
            bool same = true;
            const int jfirst = slice_of(p, ob + p0 * 8);
#pragma unroll
            for (int q = 0; q < PW; ++q) {
                const int o8 = p0 + q * kWarps;
                jq[q] = jfirst;
                if (j1 > j0 && o8 < nob) {
                    jq[q] = slice_of(p, ob + o8 * 8);
                    same = same && jq[q] == jfirst;
                }
            }
            float acc[PW][4];
#pragma unroll
            for (int q = 0; q < PW; ++q)
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) acc[q][e2] = 0.f;
            if (same) {
                if (jq[0] != cur) {
                    load_v(jq[0]);
                    cur = jq[0];
                }
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    if (ks < ksteps) {
                        const bool tail = ks * 16 + 8 >= rs;
                        uint32_t b[PW][2];
#pragma unroll
                        for (int q = 0; q < PW; ++q) {
                            if (p0 + q * kWarps < nob) {
                                ldsm_x2(bq + (p0 + q * kWarps) * 8 * rs + ks * 16, b[q][0], b[q][1]);
                                if (tail) b[q][1] = 0u;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < PW; ++q)
                            if (p0 + q * kWarps < nob)
                                mma16816(acc[q], hf[ks][0], hf[ks][1], hf[ks][2], hf[ks][3], b[q][0], b[q][1]);
#pragma unroll
                        for (int q = 0; q < PW; ++q)
                            if (p0 + q * kWarps < nob)
                                mma16816(acc[q], lf[ks][0], lf[ks][1], lf[ks][2], lf[ks][3], b[q][0], b[q][1]);
                    }
                }
            } else {  // the pass crosses a slice boundary: block by block
#pragma unroll
                for (int q = 0; q < PW; ++q) {
                    if (p0 + q * kWarps < nob) {
                        if (jq[q] != cur) {
                            load_v(jq[q]);
                            cur = jq[q];
                        }
#pragma unroll
                        for (int ks = 0; ks < KS; ++ks) {
                            if (ks < ksteps) {
                                uint32_t b0, b1;
                                ldsm_x2(bq + (p0 + q * kWarps) * 8 * rs + ks * 16, b0, b1);
                                if (ks * 16 + 8 >= rs) b1 = 0u;
                                mma16816(acc[q], hf[ks][0], hf[ks][1], hf[ks][2], hf[ks][3], b0, b1);
                                mma16816(acc[q], lf[ks][0], lf[ks][1], lf[ks][2], lf[ks][3], b0, b1);
                            }
                        }
                    }
                }
            }
            uint32_t u0[PW], u1[PW];
#pragma unroll
            for (int q = 0; q < PW; ++q) {
                const int ocol = (p0 + q * kWarps) * 8 + 2 * c4;
                u0[q] = u1[q] = 0u;
                if (p0 + q * kWarps < nob) {
                    if (g < n) u0[q] = lds32(ys + g * p.ys_stride + ocol);
                    if (g + 8 < n) u1[q] = lds32(ys + (g + 8) * p.ys_stride + ocol);
                }
            }
#pragma unroll
            for (int q = 0; q < PW; ++q) {
                const int ocol = (p0 + q * kWarps) * 8 + 2 * c4;
                if (p0 + q * kWarps < nob) {
                    if (g < n)
                        sts32(ys + g * p.ys_stride + ocol, pack_bf16x2(bf16lo(u0[q]) + acc[q][0], bf16hi(u0[q]) + acc[q][1]));
                    if (g + 8 < n)
                        sts32(ys + (g + 8) * p.ys_stride + ocol,
                              pack_bf16x2(bf16lo(u1[q]) + acc[q][2], bf16hi(u1[q]) + acc[q][3]));
                }
            }
        }
        // the next item's rows and rank, in flight during the stores
        int nrank = 0, nrow = 0;
        if (nitem < total && tid < kTileRows) {
            nrank = p.rank[(nkeyn >> 5) / p.E];
            if (tid < (nkeyn & 31)) nrow = p.sorted[nrow0 + tid];
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (warp == 0 && lane < n) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             p.out + (long long)rows[lane] * p.ld_out + ob),
                         "r"(smem_u32(ys + lane * p.ys_stride)), "r"((uint32_t)(oe - ob) * 2)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            // the rows may be reused once the copy has read them; the writes
            // are complete when the grid is
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
        if (nitem < total && tid < kTileRows) {
            if (tid < (nkeyn & 31)) s_rows[buf ^ 1][tid] = nrow;
            if (tid == 0) {
                s_ninfo[0] = nrow0;
                s_ninfo[1] = nkeyn;
                s_ninfo[2] = nrank;
            }
        }
        __syncthreads();  // this item's buffers are read and the next item's words are in place
        item = nitem;
        if (item < total) {
            row0 = s_ninfo[0];
            keyn = s_ninfo[1];
            r = s_ninfo[2];
        }
    }
    if (dyn) finish_items(p.ticket);
    asm volatile("griddepcontrol.launch_dependents;");
}

// ---------------------------------------------------------------- expand on tcgen05
//
// The same items as bgmv_expand_kernel (a tile of up to 16 rows of one key,
// oc_w output columns), with the products on the tensor cores: for every
// 128-output block m of the item
//
//   D_m[o][t] = sum_k B_j[a][o][k] * v_hi[t][j][k] + sum_k B_j[a][o][k] * v_lo[t][j][k]
//
// is one tcgen05 MMA pair with M = 128 outputs, N = 16 rows and K = the
// slot's ranks (16 per instruction), accumulated in tensor memory (16 fp32
// columns per block).  Both operands are K-major without swizzle: 8-row x
// 16-byte core matrices, the K-adjacent ones LBO apart and the M/N-adjacent
// ones SBO = 128 bytes apart.  B_j rows arrive by TMA, one box of 8 ranks x
// 128 rows per chunk (chunk kc of row i at kc * 2048 + i * 16 of its block;
// boxes past the slot's rank lie outside the tensor and are zero-filled), v is
// written by the threads that sum the partials (chunk kc of row t at
// kc * 256 + t * 16).
// One thread issues the MMAs; each warp then reads its lane quarter of every
// block (32 outputs x 16 rows) and adds it to the y rows staged in shared
// memory, which are stored back with bulk copies as in bgmv_expand_kernel.
// Every slice width is a multiple of 128, so a block lies in one slice.

constexpr int kTcM = 128;  // outputs per MMA block
static_assert(kThreads == kTcM, "the tensor-core expand copies one B row per thread");

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);        // start address
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;   // K-adjacent core matrices
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;   // M/N-adjacent core matrices
    d |= (uint64_t)1 << 46;                        // descriptor version for tcgen05; no swizzle
    return d;
}
// 32 lanes x 16 consecutive fp32 columns (this warp's lane quarter).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// MT: 128-output blocks per item (oc_w / 128).  Shared memory: B blocks
// [MT][kcb][128][8], y rows [16][ys_stride], v hi and lo [n_slices][kcb][16][8]
// with kcb = the pool's 8-rank chunks rounded up to a 16-rank step.
template <int MT>
__global__ void __launch_bounds__(kThreads) bgmv_expand_tc_kernel(const __grid_constant__ EArgs p) {
    extern __shared__ __align__(128) char smem[];
    __shared__ __align__(8) uint64_t ybar, mbar, bbar;
    __shared__ int s_rows[2][kTileRows];
    __shared__ int s_next, s_ninfo[3];
    __shared__ int s_item;
    __shared__ uint32_t s_tmem;
    __shared__ int s_by[MT];  // this item's block m: row of its first output in its tensor map
    __shared__ int s_mj[MT];  // ... and its slice
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ns = p.n_slices;
    const int n_tiles = p.counters[p.count_idx];
    const int total = n_tiles * p.n_oc;
    constexpr uint32_t kCols = MT * 16 < 32 ? 32 : MT * 16;  // tensor-memory columns: 16 per block
    const int kcb = ((p.R8 + 15) >> 4) * 2;                  // 8-rank chunks per block (16-rank steps)
    const uint32_t blk_bytes = (uint32_t)kcb * kTcM * 16;    // one B block
    const uint32_t vsl_bytes = (uint32_t)kcb * kTileRows * 16;  // v of one slice
    if (warp == 0) {
        tc::tmem_alloc(&s_tmem, kCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&ybar, 1);
        mbar_init(&mbar, 1);
        mbar_init(&bbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    char *bs = smem + p.off_b;
    uint16_t *ys = (uint16_t *)(smem + p.off_ys);
    char *vh = smem + p.off_vh;
    char *vl = smem + p.off_vl;
    bool waited = false;
    const int nc = p.NC;
    uint32_t phase = 0;

    const bool dyn = total > (int)gridDim.x;
    int item = dyn ? take_item(p.ticket, &s_item) : (int)blockIdx.x;  // its barrier also publishes s_tmem
    int row0 = 0, keyn = 0, r = 0, buf = 0;
    if (item < total) {
        const int tile = item / p.n_oc;
        row0 = p.tile_row0[tile];
        keyn = p.tile_keyn[tile];
        r = p.rank[(keyn >> 5) / p.E];
        if (tid < (keyn & 31)) s_rows[0][tid] = p.sorted[row0 + tid];
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;
    for (; item < total; phase ^= 1u, buf ^= 1) {
        const int tile = item / p.n_oc, oc = item - tile * p.n_oc;
        const int n = keyn & 31, key = keyn >> 5;
        const int a = key / p.E, e = key - a * p.E;
        const int rs = (r + 7) & ~7;
        const int ob = oc * p.oc_w, oe = min(p.out_total, ob + p.oc_w);
        const int mta = (oe - ob) / kTcM;         // blocks of this item
        const int kcr = rs >> 3, kcs = ((rs + 15) >> 4) * 2;  // real and stepped 8-rank chunks
        const int *rows = s_rows[buf];
        int nxt_t = total;
        if (dyn && tid == 0) nxt_t = atomicAdd(p.ticket, 1);  // lands while this item runs
        // after the first item: this thread's first partial sums (the slice
        // of the item's first output, ranks 4 lq ..) are requested first, so
        // their latency overlaps the item's set-up, copies and barrier
        const int tq = tid >> 3, lq = tid & 7;
        const int j0 = slice_of(p, ob);
        const int vrows = p.v_div > 0 ? p.v_rows : p.rows;
        const long long cstride = (long long)ns * vrows * p.R8 / 4;
        const int prow = tq < n ? (p.v_div > 0 ? rows[tq] / p.v_div : row0 + tq) : 0;
        float4 pre[4];
        const bool pre_ok = waited && tq < n && lq * 4 < rs;
        if (pre_ok) {
            const float4 *src = (const float4 *)(p.part + ((long long)j0 * vrows + prow) * p.R8 + lq * 4);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                if (cc < nc) pre[cc] = __ldcg(src + cc * cstride);
        }
        // y rows: bulk copies (they do not depend on the shrink).  The y
        // tile's last generic writes were ordered before the async proxy by
        // the fence ahead of the previous item's stores.
        if (warp == 0) {
            const uint32_t rowb = (uint32_t)(oe - ob) * 2;
            if (lane == 0) mbar_expect_tx(&ybar, rowb * (uint32_t)n);
            __syncwarp();
            if (lane < n)
                bulk_g2s(ys + lane * p.ys_stride, p.out + (long long)rows[lane] * p.ld_out + ob, rowb, &ybar);
        } else if (warp == 1 && lane < MT) {
            // each block's slice and row in the slice's maps (constant
            // parameter indices)
            const int o0 = ob + lane * kTcM;
            int jm = 0, by = 0;
#pragma unroll
            for (int jj = 0; jj < LORA_MAX_SLICES; ++jj) {
                if (jj < ns && o0 >= p.out_off[jj] && o0 < p.out_off[jj] + p.out_w[jj]) {
                    jm = jj;
                    by = (p.B_shared[jj] ? 0 : e * p.out_w[jj]) + (o0 - p.out_off[jj]);
                }
            }
            s_mj[lane] = jm;
            s_by[lane] = by;
        }
        // the weight factors of the v row this thread converts (loads in
        // flight across the barrier and the copies; multiplied only in the
        // sum below)
        const float w_sc = tq < n ? __ldg(p.scale + a) : 0.f;
        const float w_rw = (tq < n && p.row_w) ? __ldg(p.row_w + rows[tq]) : 1.f;
        __syncthreads();
        const int j1 = s_mj[mta - 1];  // j0 = s_mj[0]
        // B blocks: a TMA box of 8 ranks x 128 rows per chunk of the rank,
        // issued by one thread; the chunk past an odd 8-rank step (up to the
        // 16-rank step) is zeroed by the threads, one row each
        if (tid == 32) {
            mbar_expect_tx(&bbar, (uint32_t)(mta * kcr) * (kTcM * 16));
            for (int m = 0; m < mta; ++m) {
                const CUtensorMap *bm = p.kmaps + s_mj[m] * 8 + (rs >> 3) - 1;
                for (int kc = 0; kc < kcr; ++kc)
                    tc::tma_load_3d(bs + m * blk_bytes + kc * (kTcM * 16), bm, kc * 8, s_by[m], a, &bbar);
            }
        }
        if (kcs > kcr)
            for (int m = 0; m < mta; ++m) *(uint4 *)(bs + m * blk_bytes + kcr * (kTcM * 16) + tid * 16) = make_uint4(0u, 0u, 0u, 0u);
        if (!waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // the shrink's partials are complete
            waited = true;
        }
        // v of every slice a block uses (chunk partials summed in order,
        // scaled) -> bf16 hi / lo in the core-matrix layout; zero past the rank
        const float w_row = w_sc * p.post_scale * w_rw;
        for (int jj = j0; jj <= j1; ++jj) {
            for (int k = lq * 4; k < kcs * 8; k += 32) {
                float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tq < n && k < rs) {
                    const float4 *src = (const float4 *)(p.part + ((long long)jj * vrows + prow) * p.R8 + k);
                    const bool use_pre = pre_ok && jj == j0 && k == lq * 4;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {  // at most 4 hidden chunks
                        if (cc >= nc) break;
                        const float4 v = use_pre ? pre[cc] : __ldcg(src + cc * cstride);
                        s4.x += v.x;
                        s4.y += v.y;
                        s4.z += v.z;
                        s4.w += v.w;
                    }
                    s4.x *= w_row;
                    s4.y *= w_row;
                    s4.z *= w_row;
                    s4.w *= w_row;
                }
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(s4.x, s4.y);
                const __nv_bfloat162 h23 = __floats2bfloat162_rn(s4.z, s4.w);
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                uint2 hv, lv;
                hv.x = *(const uint32_t *)&h01;
                hv.y = *(const uint32_t *)&h23;
                lv.x = pack_bf16x2(s4.x - f01.x, s4.y - f01.y);
                lv.y = pack_bf16x2(s4.z - f23.x, s4.w - f23.y);
                const int off = jj * (int)vsl_bytes + (k >> 3) * (kTileRows * 16) + tq * 16 + (k & 7) * 2;
                *(uint2 *)(vh + off) = hv;
                *(uint2 *)(vl + off) = lv;
            }
        }
        if (tid == 0) s_next = nxt_t;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // v (generic writes) -> tensor core reads
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
        // the next item's tile words, in flight during the MMAs
        const int nitem = s_next;
        int nrow0 = 0, nkeyn = 0;
        if (nitem < total && tid < kTileRows) {
            const int nt = nitem / p.n_oc;
            nrow0 = p.tile_row0[nt];
            nkeyn = p.tile_keyn[nt];
        }
        if (tid == 0) {
            mbar_wait(&bbar, phase, p.spin_limit, p.status);  // the B boxes are in
            tc::tc_fence_after();
            const uint32_t idesc = tc::idesc_bf16(kTcM, kTileRows);
            const uint32_t b_addr = smem_u32(bs), vh_addr = smem_u32(vh), vl_addr = smem_u32(vl);
            const int ksteps = kcs >> 1;
            for (int m = 0; m < mta; ++m) {
                const uint32_t ab = b_addr + m * blk_bytes, vo = (uint32_t)s_mj[m] * vsl_bytes;
                for (int ks = 0; ks < ksteps; ++ks) {
                    const uint64_t ad = desc_kmajor(ab + ks * 2 * (kTcM * 16), kTcM * 16, 128);
                    tc::mma_bf16(tmem + m * 16, ad, desc_kmajor(vh_addr + vo + ks * 2 * (kTileRows * 16), kTileRows * 16, 128),
                                 idesc, ks != 0);
                    tc::mma_bf16(tmem + m * 16, ad, desc_kmajor(vl_addr + vo + ks * 2 * (kTileRows * 16), kTileRows * 16, 128),
                                 idesc, 1u);
                }
            }
            tc::mma_commit(&mbar);
        }
        mbar_wait(&ybar, phase, p.spin_limit, p.status);
        mbar_wait(&mbar, phase, p.spin_limit, p.status);
        tc::tc_fence_after();
        // this warp's 32 outputs of every block, 16 rows each, added to y
        for (int m = 0; m < mta; ++m) {
            uint32_t d[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(m * 16), d);
            uint16_t *yc = ys + m * kTcM + warp * 32 + lane;
            uint16_t yv[kTileRows];  // every load before the stores (a run-time row stride hides that they differ)
#pragma unroll
            for (int t = 0; t < kTileRows; ++t) yv[t] = t < n ? yc[t * p.ys_stride] : (uint16_t)0;
            tc::tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < kTileRows; t += 2) {  // two rows per conversion
                const __nv_bfloat162 o2 = __floats2bfloat162_rn(
                    __bfloat162float(__ushort_as_bfloat16(yv[t])) + __uint_as_float(d[t]),
                    __bfloat162float(__ushort_as_bfloat16(yv[t + 1])) + __uint_as_float(d[t + 1]));
                if (t < n) yc[t * p.ys_stride] = __bfloat16_as_ushort(o2.x);
                if (t + 1 < n) yc[(t + 1) * p.ys_stride] = __bfloat16_as_ushort(o2.y);
            }
        }
        // the next item's rows and rank, in flight during the stores
        int nrank = 0, nrow = 0;
        if (nitem < total && tid < kTileRows) {
            nrank = p.rank[(nkeyn >> 5) / p.E];
            if (tid < (nkeyn & 31)) nrow = p.sorted[nrow0 + tid];
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::tc_fence_before();
        __syncthreads();
        if (warp == 0 && lane < n) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             p.out + (long long)rows[lane] * p.ld_out + ob),
                         "r"(smem_u32(ys + lane * p.ys_stride)), "r"((uint32_t)(oe - ob) * 2)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
        if (nitem < total && tid < kTileRows) {
            if (tid < (nkeyn & 31)) s_rows[buf ^ 1][tid] = nrow;
            if (tid == 0) {
                s_ninfo[0] = nrow0;
                s_ninfo[1] = nkeyn;
                s_ninfo[2] = nrank;
            }
        }
        __syncthreads();  // this item's buffers are read and the next item's words are in place
        tc::tc_fence_after();
        item = nitem;
        if (item < total) {
            row0 = s_ninfo[0];
            keyn = s_ninfo[1];
            r = s_ninfo[2];
        }
    }
    if (dyn) finish_items(p.ticket);
    asm volatile("griddepcontrol.launch_dependents;");
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

size_t a128(size_t x) { return (x + 127) & ~(size_t)127; }

// per device: shared-memory limits raised (first calls from several host threads may race)
std::atomic<int> g_split_configured[64];
int g_key_major_waves = 8;  // most waves of the key-major shrink grid

// Hidden chunks of a shrink item: ~32 KB of A rows at full rank, >= 256
// columns, at most 4 (the many-adapter down projection measured 3% faster
// with 4 than with 8; 2, 3, 5 and 6 were slower).
void chunking(int in_dim, int R8, int *NC, int *HC) {
    int hc = (16384 / R8 + 63) / 64 * 64;
    if (hc < 256) hc = 256;
    int nc = lora_ceil_div(in_dim, hc);
    if (nc > 4) nc = 4;
    hc = ((lora_ceil_div(in_dim, nc) + 15) / 16) * 16;
    *NC = lora_ceil_div(in_dim, hc);
    *HC = hc;
}

}  // namespace

size_t lora_split_ws_bytes(int n_slices, int in_dim, int R, int rows, int max_tiles) {
    (void)max_tiles;
    int NC, HC;
    chunking(in_dim, lora_round8(R), &NC, &HC);
    return a128((size_t)NC * n_slices * rows * lora_round8(R) * 4);
}

lora_status_t lora_split_apply(const lora_pool_t *pool, const LoraProblem &pr, void *ws, size_t ws_bytes,
                               int *tickets, cudaStream_t s, bool *launched) {
    *launched = false;
    const int ns = pr.n_slices, R = pr.R, R8 = lora_round8(R);
    int out_total = 0;
    for (int j = 0; j < ns; ++j) out_total = max(out_total, pr.out_off[j] + pr.out_w[j]);
    const long long max_tiles = pr.rows / kTileRows + (pr.rows < pr.n_keys ? pr.rows : pr.n_keys);
    // the shrink holds at most two 8-rank MMA column blocks per warp
    if (R8 > 2 * kSWarps * 8 || max_tiles <= 0) return LORA_OK;
    int NC, HC;
    chunking(pr.in_dim, R8, &NC, &HC);
    if (!ws || ws_bytes < lora_split_ws_bytes(ns, pr.in_dim, R, pr.rows, 0) || !lora_aligned16(ws) || !tickets)
        return LORA_OK;
    // kernel instances for the pool's most 8-rank blocks (rounded up to 1, 2, 4, 8)
    const int nbr = R8 / 8;
    const int NBM = nbr <= 1 ? 1 : nbr <= 2 ? 2 : nbr <= 4 ? 4 : 8;
    // the per-tile shrink takes the ranks in groups of kRG
    void (*shrink_fn)(SArgs) = R8 <= 8 ? bgmv_shrink_kernel<1> : bgmv_shrink_kernel<2>;
    const int RG8 = std::min(R8, kRG);
    void (*slot_fn)(SArgs) = NBM == 1 ? bgmv_shrink_slot_kernel<1> : NBM == 2 ? bgmv_shrink_slot_kernel<2>
                           : NBM == 4 ? bgmv_shrink_slot_kernel<4> : bgmv_shrink_slot_kernel<8>;
    const int dev = pool->device < 64 ? pool->device : 63;
    if (!g_split_configured[dev].load(std::memory_order_acquire)) {
        void (*const fns[])(SArgs) = {bgmv_shrink_kernel<1>,      bgmv_shrink_kernel<2>,
                                      bgmv_shrink_tile_kernel<1>, bgmv_shrink_tile_kernel<2>,
                                      bgmv_shrink_tile_kernel<4>, bgmv_shrink_tile_kernel<8>,
                                      bgmv_shrink_slot_kernel<1>, bgmv_shrink_slot_kernel<2>,
                                      bgmv_shrink_slot_kernel<4>, bgmv_shrink_slot_kernel<8>};
        for (auto f : fns)
            LORA_CUDA_TRY(cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        void (*const efns[])(EArgs) = {bgmv_expand_kernel<1, 8>, bgmv_expand_kernel<2, 8>, bgmv_expand_kernel<3, 8>,
                                       bgmv_expand_kernel<4, 8>, bgmv_expand_kernel<1, 4>, bgmv_expand_kernel<2, 4>,
                                       bgmv_expand_kernel<3, 4>, bgmv_expand_kernel<4, 4>};
        for (auto f : efns)
            LORA_CUDA_TRY(cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        for (auto f : {bgmv_expand_tc_kernel<2>, bgmv_expand_tc_kernel<4>})
            LORA_CUDA_TRY(cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        g_split_configured[dev].store(1, std::memory_order_release);
    }
    // per-tile shrink shared memory: 2 stages of (16 + min(R8, kRG)) rows x SC
    // columns (rows padded by 16 bytes) and the group sums.  SC: the widest
    // stage (up to the chunk, <= 75 KB, three CTAs per SM) whose occupancy
    // still runs every item in one wave, else the widest that fits
    const int red_bytes = 4 * kTileRows * R8 * 4;  // key-major shrink: [4 warps][16][R8] sums
    const size_t red_g = a128((size_t)2 * 4 * kTileRows * kRG * 4);  // two group-sum buffers
    // 2 wide stages: a 3-stage ring of narrower stages measured slower on the
    // many-adapter batch
    const int nst = 2;
    const size_t s_budget = 75 * 1024;
    auto smem_for = [&](int sc) {
        return nst * (a128((size_t)kTileRows * (sc + 8) * 2) + a128((size_t)RG8 * (sc + 8) * 2)) + red_g;
    };
    const long long s_items = max_tiles * ns * NC;
    int SC = 0, occ = 0, first = 0, first_occ = 0;
    for (int sc = (HC < 1024 ? HC : 1024); sc >= 64; sc -= 64) {
        if (smem_for(sc) > s_budget) continue;
        int o = 0;
        LORA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, shrink_fn, kPThreads, smem_for(sc)));
        if (!first) {
            first = sc;
            first_occ = o;
        }
        if (sc < 256) break;  // narrower stages only when nothing wider fits
        if ((long long)o * pool->num_sms >= s_items) {
            SC = sc;
            occ = o;
            break;
        }
    }
    if (!SC) {
        SC = first;
        occ = first_occ;
    }
    if (!SC) return LORA_OK;
    size_t s_smem = smem_for(SC);
    // every per-tile item fits two waves: one item per CTA, the CTA-synchronous
    // kernel with full-rank stages (the partial sums reuse them)
    void (*tile_fn)(SArgs) = NBM == 1 ? bgmv_shrink_tile_kernel<1> : NBM == 2 ? bgmv_shrink_tile_kernel<2>
                           : NBM == 4 ? bgmv_shrink_tile_kernel<4> : bgmv_shrink_tile_kernel<8>;
    const int red_t = 4 * kTileRows * R8 * 4;
    auto smem_t = [&](int sc) {
        return std::max((size_t)red_t, 2 * (a128((size_t)kTileRows * (sc + 8) * 2) + a128((size_t)R8 * (sc + 8) * 2)));
    };
    int SC_t = 0, occ_t = 0;
    {
        int first_t = 0, first_occ_t = 0;
        for (int sc = (HC < 1024 ? HC : 1024); sc >= 64; sc -= 64) {
            if (smem_t(sc) > 75 * 1024) continue;
            int o = 0;
            LORA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, tile_fn, kSThreads, smem_t(sc)));
            if (!first_t) {
                first_t = sc;
                first_occ_t = o;
            }
            if (sc < 256) break;  // narrower stages only when nothing wider fits
            if ((long long)o * pool->num_sms >= s_items) {
                SC_t = sc;
                occ_t = o;
                break;
            }
        }
        if (!SC_t) {
            SC_t = first_t;
            occ_t = first_occ_t;
        }
    }
    const bool tile_static = SC_t > 0 && occ_t > 0 && s_items <= 2LL * pool->num_sms * occ_t;
    // expand shared memory: B rows, y rows, v hi/lo
    const int vr_stride = ns * R8 + 8;
    // 512 output columns per expand item for small ranks (fewer items, less fixed work per column)
    int oc_w = R8 <= 32 ? 512 : kOC;
    size_t e_b = a128((size_t)oc_w * R8 * 2 + 32), e_y = a128((size_t)kTileRows * (oc_w + 8) * 2);
    const size_t e_v = a128((size_t)kTileRows * vr_stride * 2);
    size_t e_smem = e_b + e_y + 2 * e_v;

    const long long s_slots = (long long)pool->num_sms * (occ < 1 ? 1 : occ);
    int occ_e = 0;
    const int KS = (R8 + 15) / 16;
    // wide passes when the expand items fit two waves of the wide kernel
    void (*expand_fn)(EArgs) = KS == 1 ? bgmv_expand_kernel<1, 8> : KS == 2 ? bgmv_expand_kernel<2, 8>
                             : KS == 3 ? bgmv_expand_kernel<3, 8> : bgmv_expand_kernel<4, 8>;
    LORA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_e, expand_fn, kThreads, e_smem));
    // 256-column items when 512-column ones would leave over 40% of one wave
    // idle (the sink-expert layers measured 9% faster; decode batches, which
    // fill the wave, are faster with 512)
    if (oc_w == 512 && 10 * max_tiles * lora_ceil_div(out_total, 512) < 6LL * pool->num_sms * (occ_e < 1 ? 1 : occ_e)) {
        oc_w = kOC;
        e_b = a128((size_t)oc_w * R8 * 2 + 32);
        e_y = a128((size_t)kTileRows * (oc_w + 8) * 2);
        e_smem = e_b + e_y + 2 * e_v;
        LORA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_e, expand_fn, kThreads, e_smem));
    }
    if (max_tiles * lora_ceil_div(out_total, oc_w) > 2LL * pool->num_sms * (occ_e < 1 ? 1 : occ_e)) {
        expand_fn = KS == 1 ? bgmv_expand_kernel<1, 4> : KS == 2 ? bgmv_expand_kernel<2, 4>
                  : KS == 3 ? bgmv_expand_kernel<3, 4> : bgmv_expand_kernel<4, 4>;
        LORA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_e, expand_fn, kThreads, e_smem));
    }
    // the tensor-core expand: every slice a whole number of 128-output
    // blocks (a block then lies in one slice) and ranks up to 64
    bool tc_expand = g_lora_kernel_policy != 8 && R8 <= 64 && oc_w % kTcM == 0 && pool->d_kmaps != nullptr;
    for (int j = 0; j < ns; ++j) tc_expand = tc_expand && pr.out_w[j] % kTcM == 0 && pr.out_off[j] % kTcM == 0;
    const int kcb = ((R8 + 15) / 16) * 2;
    if (tc_expand) {
        expand_fn = oc_w == 4 * kTcM ? bgmv_expand_tc_kernel<4> : bgmv_expand_tc_kernel<2>;
        e_b = a128((size_t)(oc_w / kTcM) * kcb * kTcM * 16);
        const size_t e_vt = a128((size_t)ns * kcb * kTileRows * 16);
        e_smem = e_b + e_y + 2 * e_vt;
        // The occupancy query answers 1 for any kernel that allocates tensor
        // memory; the CTAs an SM holds are set by shared memory, registers
        // and threads, and by the 512 tensor-memory columns (a CTA that
        // finds them taken waits in tcgen05.alloc for one that finishes).
        cudaFuncAttributes fa;
        LORA_CUDA_TRY(cudaFuncGetAttributes(&fa, expand_fn));
        int smem_sm = 0, resv = 0;
        LORA_CUDA_TRY(cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, pool->device));
        LORA_CUDA_TRY(cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, pool->device));
        const int by_smem = (int)(smem_sm / (e_smem + fa.sharedSizeBytes + resv));
        const int by_regs = 65536 / (std::max(fa.numRegs, 1) * kThreads);
        const int by_tmem = 512 / std::max(32, (oc_w / kTcM) * 16);
        occ_e = std::min(std::min(by_smem, by_regs), std::min(by_tmem, 2048 / kThreads));
    }
    const long long e_slots = (long long)pool->num_sms * (occ_e < 1 ? 1 : occ_e);

    // key-major shrink when the batch keeps most keys busy and the grid is a
    // few waves at most: the key's A chunk is fetched while the metadata is
    // still being built, and read once per key
    const int L = pr.n_keys;
    const size_t x_stage = a128((size_t)kTileRows * (HC + 8) * 2);
    // a second x stage only when keys average more than one and a half tiles
    const int x_stages = pr.rows > 24LL * L && a128((size_t)R8 * (HC + 8) * 2) + 2 * x_stage + red_bytes <= 100 * 1024 ? 2 : 1;
    const size_t slot_smem = a128((size_t)R8 * (HC + 8) * 2) + x_stages * x_stage + red_bytes;
    bool slot_major = pr.count_idx == 3 && pr.rows >= 4 * L && slot_smem <= 100 * 1024;
    // a key-major CTA walks its key's tiles one after another: with fewer of
    // them than SMs and more than one tile per key on average, the per-tile
    // items spread the work wider (the sink-expert layers: 9% faster)
    if ((long long)L * ns * NC < pool->num_sms && pr.rows > kTileRows * L) slot_major = false;
    if (slot_major) {
        int o = 0;
        LORA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, slot_fn, kSThreads, slot_smem));
        slot_major = (long long)L * ns * NC <= (long long)g_key_major_waves * o * pool->num_sms;
    }
    // token mode (shared-outer MoE A): the key-major kernel over slots, with
    // the slot's token list and a bitmap over the batch's tokens after the
    // reduction buffer
    const size_t tok_bytes = a128((size_t)4 * (pr.T + (pr.T + 31) / 32));
    const bool tmode = pr.tok_dedup && pr.T > 0 && pr.E > 0 && pr.n_keys % pr.E == 0 &&
                       slot_smem + tok_bytes <= 160 * 1024;
    if (tmode) slot_major = true;

    SArgs sa;
    memset(&sa, 0, sizeof(sa));
    sa.n_slices = ns;
    sa.in_dim = pr.in_dim;
    sa.E = pr.E;
    sa.row_div = pr.row_div;
    sa.R = R;
    sa.R8 = R8;
    for (int j = 0; j < ns; ++j) {
        sa.A[j] = pr.A[j];
        sa.A_ss[j] = pr.A_ss[j];
        sa.A_es[j] = pr.A_es[j];
    }
    sa.rank = pr.rank;
    sa.sorted = pr.meta->sorted;
    sa.tile_row0 = pr.tile_row0;
    sa.tile_keyn = pr.tile_keyn;
    sa.counters = pr.meta->counters;
    sa.count_idx = pr.count_idx;
    sa.in = pr.in;
    sa.ld_in = pr.ld_in;
    sa.NC = NC;
    sa.HC = HC;
    sa.SC = SC;
    sa.xs_stride = SC + 8;
    sa.as_stride = SC + 8;
    sa.x_stage_bytes = (int)a128((size_t)kTileRows * (SC + 8) * 2);
    sa.a_stage_bytes = (int)a128((size_t)RG8 * (SC + 8) * 2);
    sa.off_x = 0;
    sa.nst = nst;
    sa.off_a = nst * sa.x_stage_bytes;
    sa.off_red = sa.off_a + nst * sa.a_stage_bytes;  // group sums apart from the stages (the next group's copies are in flight)
    sa.part = (float *)ws;
    sa.ticket = tickets;
    sa.rows = pr.rows;
    sa.status = pr.status;
    sa.spin_limit = pr.spin_limit;

    EArgs ea;
    memset(&ea, 0, sizeof(ea));
    ea.n_slices = ns;
    ea.R = R;
    ea.R8 = R8;
    ea.E = pr.E;
    ea.out_total = out_total;
    for (int j = 0; j < ns; ++j) {
        ea.out_w[j] = pr.out_w[j];
        ea.out_off[j] = pr.out_off[j];
        ea.B[j] = pr.B[j];
        ea.B_ss[j] = pr.B_ss[j];
        ea.B_shared[j] = pr.B_shared[j];
    }
    ea.rank = pr.rank;
    ea.scale = pr.scale;
    ea.row_w = pr.row_w;
    ea.post_scale = pr.post_scale;
    ea.NC = NC;
    ea.sorted = pr.meta->sorted;
    ea.tile_row0 = pr.tile_row0;
    ea.tile_keyn = pr.tile_keyn;
    ea.counters = pr.meta->counters;
    ea.count_idx = pr.count_idx;
    ea.out = pr.out;
    ea.ld_out = pr.ld_out;
    ea.part = sa.part;
    ea.ticket = tickets + 2;
    ea.rows = pr.rows;
    ea.oc_w = oc_w;
    ea.n_oc = lora_ceil_div(out_total, oc_w);
    ea.ys_stride = oc_w + 8;
    ea.vr_stride = vr_stride;
    ea.off_b = 0;
    ea.off_ys = (int)e_b;
    ea.off_vh = (int)(e_b + e_y);
    ea.off_vl = (int)(e_b + e_y + e_v);
    if (tc_expand) {
        const size_t e_vt = a128((size_t)ns * kcb * kTileRows * 16);
        ea.off_vl = (int)(e_b + e_y + e_vt);
        if ((size_t)ea.off_vl + e_vt > e_smem) return LORA_ERR_INVALID_ARG;  // layout check
    }
    ea.status = pr.status;
    ea.spin_limit = pr.spin_limit;
    ea.kmaps = pool->d_kmaps ? pool->d_kmaps + (long long)pr.kmap_base * 8 : nullptr;

    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kSThreads, 1, 1);
    cfg.stream = s;
    // grids of at most one wave; the kernels stride over their items
    // grids of at most two waves (the key-major shrink: one CTA per item); CTAs take items from counters
    const long long e_items = max_tiles * ea.n_oc;
    if (slot_major) {
        sa.enabled = pool->d_enabled;
        sa.key_count = pr.meta->key_count;
        sa.key_offset = pr.meta->key_offset;
        sa.n_slots = L;
        sa.x_stages = x_stages;
        sa.xs_stride = HC + 8;
        sa.as_stride = HC + 8;
        sa.x_stage_bytes = (int)a128((size_t)kTileRows * (HC + 8) * 2);
        sa.off_a = 0;
        sa.off_x = (int)a128((size_t)R8 * (HC + 8) * 2);
        sa.off_red = sa.off_x + x_stages * sa.x_stage_bytes;
        if ((size_t)sa.off_red + red_bytes > slot_smem) return LORA_ERR_INVALID_ARG;  // layout check
        long long grid = (long long)L * ns * NC;
        size_t smem_k = slot_smem;
        if (tmode) {
            // keys are the slots; tok_G CTAs per (slot, slice, chunk) share
            // a slot's tiles: about one tile each on an even batch, and at
            // most two waves in all
            const int Ls = L / pr.E;
            smem_k = slot_smem + tok_bytes;
            int o = 0;
            LORA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, slot_fn, kSThreads, smem_k));
            const long long per_slot = ((long long)pr.T / kTileRows + Ls + Ls - 1) / Ls;
            const long long cap = 2LL * (o < 1 ? 1 : o) * pool->num_sms / ((long long)Ls * ns * NC);
            const int G = (int)std::max(1LL, std::min(per_slot, cap));
            sa.E = 1;
            sa.row_div = 1;
            sa.rows = pr.T;
            sa.n_slots = Ls;
            sa.tok_K = pr.row_div;
            sa.tok_E = pr.E;
            sa.tok_T = pr.T;
            sa.tok_G = G;
            sa.off_tok = (int)slot_smem;
            ea.v_div = pr.row_div;
            ea.v_rows = pr.T;
            grid = (long long)Ls * ns * NC * G;
        }
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.dynamicSmemBytes = smem_k;
        LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, slot_fn, sa));
    } else {
        if (tile_static) {
            sa.SC = SC_t;
            sa.xs_stride = SC_t + 8;
            sa.as_stride = SC_t + 8;
            sa.x_stage_bytes = (int)a128((size_t)kTileRows * (SC_t + 8) * 2);
            sa.a_stage_bytes = (int)a128((size_t)R8 * (SC_t + 8) * 2);
            sa.off_x = 0;
            sa.off_a = nst * sa.x_stage_bytes;
            sa.off_red = 0;  // the partial sums reuse the stages: an item's copies are all consumed by then
            if ((size_t)sa.off_a + nst * sa.a_stage_bytes > smem_t(SC_t) || (size_t)red_t > smem_t(SC_t))
                return LORA_ERR_INVALID_ARG;  // layout check
            cfg.gridDim = dim3((unsigned)s_items, 1, 1);
            cfg.dynamicSmemBytes = smem_t(SC_t);
            LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, tile_fn, sa));
        } else {
            if ((size_t)sa.off_red + red_g > s_smem) return LORA_ERR_INVALID_ARG;  // layout check
            cfg.gridDim = dim3((unsigned)(s_items < 2 * s_slots ? s_items : 2 * s_slots), 1, 1);
            cfg.blockDim = dim3(kPThreads, 1, 1);
            cfg.dynamicSmemBytes = s_smem;
            LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, shrink_fn, sa));
        }
    }
    lora_note_launch();
    if (pr.shrink_only) {
        if (pr.nc_out) *pr.nc_out = NC;
        *launched = true;
        return LORA_OK;
    }
    cfg.blockDim = dim3(kThreads, 1, 1);
    // up to two waves: CTAs of a second wave start as first-wave CTAs finish
    // and find the counter exhausted or take the remaining items
    cfg.gridDim = dim3((unsigned)(e_items < 2 * e_slots ? e_items : 2 * e_slots), 1, 1);
    cfg.dynamicSmemBytes = e_smem;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, expand_fn, ea));
    lora_note_launch();
    *launched = true;
    return LORA_OK;
}
