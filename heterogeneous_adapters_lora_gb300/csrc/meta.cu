// Adapter-batch metadata on the device: a stable counting sort of rows by
// key in one CTA (the grouping the Punica/S-LoRA kernels consume; SGLang's
// LoRAManager.prepare_lora_batch builds the per-row slot table on the host,
// vLLM's moe_lora_align_block_size the per-(adapter, expert) grouping).
//
// Rows are tokens (dense) or pairs p = t*K + k (MoE).  key(row) = a
// (dense) or a*E + e (MoE) for active rows, n_keys for inactive ones, so the
// inactive rows land last in original order.  The rows are cut into up to 32
// contiguous chunks, one per warp; each warp keeps its own histogram in
// shared memory, which makes the scatter stable without atomics:
//   1. per-warp histograms (warp match-any: one leader per key per step)
//   2. per-key prefix over the chunks, block scan over keys -> key offsets
//   3. scatter: position = key offset + earlier chunks + earlier lanes
//   4. groups = non-empty keys, tiles of LORA_TILE_ROWS rows per group
#include <string.h>

#include <algorithm>
#include <atomic>

#include "lora_internal.cuh"
#include "meta_block.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int kSmemBudgetInts = 56 * 1024;  // 224 KB



// Key of one row given the slot-activity table in shared memory.
__device__ __forceinline__ int row_key(const MetaArgs &a, const unsigned char *act, int row, int s,
                                       int *bad) {
    const bool valid = s >= 0 && s < a.L;
    int b = (s != -1 && !valid && (row % a.K) == 0) ? 1 : 0;
    const bool on = valid && act[s];
    int key = a.n_keys;
    if (a.topk) {
        const int e = a.topk[row];
        const bool ev = e >= 0 && e < a.E;
        b += ev ? 0 : 1;
        if (on && ev) key = s * a.E + e;
    } else if (on) {
        key = s;
    }
    *bad += b;
    return key;
}

// The same key from an already loaded slot s and expert e (e unused when dense).
__device__ __forceinline__ int row_key_e(const MetaArgs &a, const unsigned char *act, int row, int s, int e,
                                         int *bad) {
    const bool valid = s >= 0 && s < a.L;
    int b = (s != -1 && !valid && (row % a.K) == 0) ? 1 : 0;
    const bool on = valid && act[s];
    int key = a.n_keys;
    if (a.topk) {
        const bool ev = e >= 0 && e < a.E;
        b += ev ? 0 : 1;
        if (on && ev) key = s * a.E + e;
    } else if (on) {
        key = s;
    }
    *bad += b;
    return key;
}

// Lanes of the warp holding the same key (one warp match instruction).
__device__ __forceinline__ unsigned key_peers(int key, int bits) {
    (void)bits;
    return __match_any_sync(0xffffffffu, key);
}

__global__ void __launch_bounds__(kThreads, 1) build_meta_kernel(MetaArgs a) {
    extern __shared__ int sm[];
    const int NK = a.n_keys, NK1 = NK + 1, W = a.n_chunks;
    int *hist = sm;                  // [W][NK1] per-chunk histograms, then 4 scratch rows
    int *cnt = hist + (W + 4) * NK1; // [NK1]
    int *off = cnt + NK1;            // [NK1]
    int *tmin = off + NK1;           // [NK1] smallest token of each key (dense)
    int *nrun = tmin + NK1;          // [NK1] runs of consecutive tokens of each key (dense)
    int *misc = nrun + NK1;          // [200]: totals at [32..35], n_bad at [36], warp scan totals at [40..199]
    unsigned char *act = (unsigned char *)(misc + 200);  // [L] slot enabled and rank > 0
    int *kc = misc + 200 + (a.L + 3) / 4;                // [rows] keys of pass 1 when cached
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x;
    const int rows = a.T * a.K;
    // let the apply kernel that follows start its prologue; it waits for
    // this grid's completion before reading any metadata
    asm volatile("griddepcontrol.launch_dependents;");
    // launched with programmatic stream serialization: everything above
    // overlaps the previous kernel; nothing is read before it has finished
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // slot (and expert) of this warp's first 8 row steps, issued before the tables
    const int chunk = (rows + W - 1) / W;
    const int r0 = warp * chunk, r1 = min(rows, r0 + chunk);
    int sv[8], ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int row = r0 + u * 32 + lane;
        const bool ok = warp < W && row < r1;
        sv[u] = ok ? a.idx[row / a.K] : -1;
        ev[u] = (ok && a.topk) ? a.topk[row] : 0;
    }
    // dense: the slot of the row before this warp's chunk (run starts at the boundary)
    const int s_prev = (a.K == 1 && warp < W && r0 > 0 && r0 < r1) ? a.idx[r0 - 1] : -1;
    for (int i = tid; i < a.L; i += nthreads) {
        const int en = a.enabled[i], rk = a.rank[i];  // both loads in flight at once
        act[i] = (en != 0 && rk > 0) ? 1 : 0;
    }
    for (int i = tid; i < (W * NK1) / 4; i += nthreads) ((int4 *)hist)[i] = make_int4(0, 0, 0, 0);
    for (int i = (W * NK1) / 4 * 4 + tid; i < W * NK1; i += nthreads) hist[i] = 0;
    for (int i = tid; i < NK1; i += nthreads) {
        tmin[i] = 0x7fffffff;
        nrun[i] = 0;
    }
    if (tid == 0) misc[36] = 0;
    __syncthreads();

    // pass 1: keys (kept for the scatter when they fit) and per-chunk counts
    int bad = 0;
    // dense: key of the row before the current step (-2: none), for run starts
    int carry = -2;
    if (a.K == 1 && warp < W && r0 > 0 && r0 < r1) {
        int dummy = 0;
        carry = row_key_e(a, act, r0 - 1, s_prev, 0, &dummy);
    }
    auto count_step = [&](int base, int s, int e) {
        const int row = base + lane;
        const bool v = row < r1;
        const int key = v ? row_key_e(a, act, row, s, e, &bad) : -1;
        if (v && a.cache_keys) kc[row] = key;
        if (a.K == 1) {
            const unsigned peers = key_peers(key, a.key_bits);
            const int leader = __ffs(peers) - 1;
            if (v && lane == leader) hist[warp * NK1 + key] += __popc(peers);
            // a row starts a run of its key when the previous row has another key:
            // the key's rows are one contiguous run when it has exactly one start
            int prev = __shfl_up_sync(0xffffffffu, key, 1);
            if (lane == 0) prev = carry;
            if (v && key < NK && key != prev) {
                atomicAdd(&nrun[key], 1);
                atomicMin(&tmin[key], row);
            }
            carry = __shfl_sync(0xffffffffu, key, 31);
        } else if (v) {
            atomicAdd(&hist[warp * NK1 + key], 1);  // counts only: order does not matter here
        }
        __syncwarp();
    };
    if (warp < W) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (r0 + u * 32 < r1) count_step(r0 + u * 32, sv[u], ev[u]);
        for (int base = r0 + 256; base < r1; base += 32) {
            const int row = base + lane;
            const bool v = row < r1;
            count_step(base, v ? a.idx[row / a.K] : -1, (v && a.topk) ? a.topk[row] : 0);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&misc[36], bad);
    __syncthreads();

    // one pass over the keys, thread t owning a contiguous block: per key the
    // exclusive prefix over the chunks (in place) and the count, then every
    // key-space prefix sum in one block-wide scan: row offsets, group index,
    // 16-row tiles, long-run tiles and short tiles
    int *gidx = hist + W * NK1;  // the four scratch rows after the chunk histograms
    int *tiles = gidx + NK1;
    int *lt_cnt = tiles + NK1;
    int *st_cnt = lt_cnt + NK1;
    int *wt = misc + 40;         // [5][32] per-warp totals
    {
        const int per = (NK1 + nthreads - 1) / nthreads;
        const int b0 = min(NK1, tid * per), b1 = min(NK1, b0 + per);
        int sv5[5] = {0, 0, 0, 0, 0};
        for (int b = b0; b < b1; ++b) {
            int run_rows = 0;
            for (int w = 0; w < W; ++w) {
                const int cw = hist[w * NK1 + b];
                hist[w * NK1 + b] = run_rows;
                run_rows += cw;
            }
            cnt[b] = run_rows;
            const int c = b < NK ? run_rows : 0;
            const bool run = c > 0 && a.K == 1 && c >= LORA_LONG_MIN && nrun[b] == 1;
            sv5[0] += run_rows;
            sv5[1] += c > 0 ? 1 : 0;
            sv5[2] += (c + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS;
            sv5[3] += run ? (c + LORA_LTILE_ROWS - 1) / LORA_LTILE_ROWS : 0;
            sv5[4] += (c > 0 && !run) ? (c + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS : 0;
        }
        int inc[5];
#pragma unroll
        for (int q = 0; q < 5; ++q) inc[q] = sv5[q];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int q = 0; q < 5; ++q) {
                const int v = __shfl_up_sync(0xffffffffu, inc[q], o);
                if (lane >= o) inc[q] += v;
            }
        }
        if (lane == 31) {
#pragma unroll
            for (int q = 0; q < 5; ++q) wt[q * 32 + warp] = inc[q];
        }
        __syncthreads();
        // every warp sums the totals of the warps before it (no single-warp phase)
        const int nw = nthreads / 32;
        int ex[5];
#pragma unroll
        for (int q = 0; q < 5; ++q) {
            int before = lane < warp ? wt[q * 32 + lane] : 0;
            int all = lane < nw ? wt[q * 32 + lane] : 0;
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                before += __shfl_xor_sync(0xffffffffu, before, o);
                all += __shfl_xor_sync(0xffffffffu, all, o);
            }
            ex[q] = before + inc[q] - sv5[q];
            if (tid == 0 && q > 0) misc[31 + q] = all;  // groups, tiles, long tiles, short tiles
        }
        for (int b = b0; b < b1; ++b) {
            const int c = b < NK ? cnt[b] : 0;
            const bool run = c > 0 && a.K == 1 && c >= LORA_LONG_MIN && nrun[b] == 1;
            off[b] = ex[0];
            gidx[b] = ex[1];
            tiles[b] = ex[2];
            lt_cnt[b] = ex[3];
            st_cnt[b] = ex[4];
            if (b < NK) a.m.key_count[b] = cnt[b];
            a.m.key_offset[b] = ex[0];
            ex[0] += cnt[b];
            ex[1] += c > 0 ? 1 : 0;
            ex[2] += (c + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS;
            ex[3] += run ? (c + LORA_LTILE_ROWS - 1) / LORA_LTILE_ROWS : 0;
            ex[4] += (c > 0 && !run) ? (c + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS : 0;
        }
    }
    __syncthreads();

    // stable scatter: position = key offset + rows of earlier chunks + earlier lanes
    if (warp < W) {
        const unsigned lt = (1u << lane) - 1u;
        for (int base = r0; base < r1; base += 32) {
            const int row = base + lane;
            const bool v = row < r1;
            int key = -1;
            if (v) {
                if (a.cache_keys) {
                    key = kc[row];
                } else {
                    int dummy = 0;
                    key = row_key(a, act, row, a.idx[row / a.K], &dummy);
                }
            }
            const unsigned peers = key_peers(key, a.key_bits);
            int pos = 0;
            if (v) pos = off[key] + hist[warp * NK1 + key] + __popc(peers & lt);
            __syncwarp();
            if (v) {
                a.m.sorted[pos] = row;
                if (lane == __ffs(peers) - 1) hist[warp * NK1 + key] += __popc(peers);
            }
            __syncwarp();
        }
    }

    // groups (non-empty keys, ascending), 16-row tiles, long-run and short tiles
    const int G = misc[32], NT = misc[33], NL = misc[34], NS = misc[35];
    for (int b = tid; b < NK; b += nthreads) {
        const int c = cnt[b];
        if (c > 0) {
            const int g = gidx[b];
            a.m.key_group[b] = g;
            a.m.group_key[g] = b;
            a.m.group_start[g] = off[b];
            const int nt = (c + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS;
            for (int i = 0; i < nt; ++i) {
                const int rows_i = min(LORA_TILE_ROWS, c - i * LORA_TILE_ROWS);
                a.m.tile_group[tiles[b] + i] = g;
                a.m.tile_row0[tiles[b] + i] = off[b] + i * LORA_TILE_ROWS;
                a.m.tile_keyn[tiles[b] + i] = (b << 5) | rows_i;
            }
            for (int i = 0; lt_cnt[b] + i < lt_cnt[b + 1]; ++i) {
                const int rows_i = min(LORA_LTILE_ROWS, c - i * LORA_LTILE_ROWS);
                a.m.ltile_row0[lt_cnt[b] + i] = off[b] + i * LORA_LTILE_ROWS;
                a.m.ltile_keyn[lt_cnt[b] + i] = (b << 8) | rows_i;
                a.m.ltile_tok0[lt_cnt[b] + i] = tmin[b] + i * LORA_LTILE_ROWS;
            }
            for (int i = 0; st_cnt[b] + i < st_cnt[b + 1]; ++i) {
                const int rows_i = min(LORA_TILE_ROWS, c - i * LORA_TILE_ROWS);
                a.m.stile_row0[st_cnt[b] + i] = off[b] + i * LORA_TILE_ROWS;
                a.m.stile_keyn[st_cnt[b] + i] = (b << 5) | rows_i;
            }
        } else {
            a.m.key_group[b] = -1;
        }
    }
    if (tid == 0) {
        const int n_active = off[NK];
        const int n_bad = misc[36];
        a.m.group_start[G] = n_active;
        a.m.counters[0] = n_active;
        a.m.counters[1] = G;
        a.m.counters[2] = n_bad;
        a.m.counters[3] = NT;
        a.m.counters[4] = NS;
        a.m.counters[5] = NL;
        if (n_bad) atomicExch(a.status, (int)LORA_ERR_DEVICE_INDEX);
    }
}

__global__ void __launch_bounds__(kSmallRows, 1) build_meta_small_kernel(MetaArgs a) {
    extern __shared__ int sm[];
    // let the apply kernel that follows start its prologue; it waits for
    // this grid's completion before reading any metadata
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    dense_meta_block(a, sm, 1);
}

// ---------------------------------------------------------------- cluster build
//
// The same metadata from one thread-block cluster of kMetaCL CTAs, for batches
// of thousands of rows (one CTA's issue rate bounds the single-CTA build
// there).  CTA c takes rows [c*rows/CL, (c+1)*rows/CL) and owns keys
// [c*NK1/CL, (c+1)*NK1/CL):
//   1. its rows' keys and per-warp histograms (as the single-CTA build), then
//      per key the prefix over its warps and its total tot_c[key]
//   2. cluster barrier; each owner reads tot_c'[key] (and, dense, the run
//      starts and first rows) of every CTA through distributed shared memory,
//      and scans the key-space sums (row offsets, groups, tiles, long and
//      short tiles) over its keys
//   3. cluster barrier; each owner adds the totals of the owners before it,
//      writes its keys' outputs and, into every CTA c', base_c'[key] = row
//      offset of the key + the rows of the key in CTAs before c'
//   4. cluster barrier; each CTA scatters its rows: base + earlier warps +
//      earlier lanes
// The order is the single-CTA build's: keys ascending, rows in original order
// within a key, inactive rows last.
constexpr int kMetaCL = 8;
constexpr long long kMetaClusterRows = 2048;  // batches of at least this many rows take the cluster build

__device__ __forceinline__ uint32_t meta_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void meta_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t meta_peer_addr(const void *p, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
    return ra;
}
// Volatile (kept after the cluster barrier) but without a memory clobber, so
// that the loads of all peers are issued back to back.
__device__ __forceinline__ int meta_ld_peer(const int *p, uint32_t rank) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(meta_peer_addr(p, rank)));
    return v;
}
__device__ __forceinline__ void meta_st_peer(int *p, uint32_t rank, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(meta_peer_addr(p, rank)), "r"(v) : "memory");
}

// Shared-memory ints of one CTA of the cluster build.
static inline long long meta_cluster_ints(int W, int NK1, int L, int rows_cta) {
    const int own = (NK1 + kMetaCL - 1) / kMetaCL;
    return (long long)(W + 4) * NK1 + (8LL + kMetaCL) * own + 200 + (L + 3) / 4 + rows_cta;
}

__global__ void __launch_bounds__(kThreads, 1) build_meta_cluster_kernel(MetaArgs a) {
    extern __shared__ int sm[];
    const int NK = a.n_keys, NK1 = NK + 1, W = a.n_chunks;
    const int CL = kMetaCL;
    const uint32_t c = meta_cluster_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x;
    const int rows = a.T * a.K;
    const int R0 = (int)((long long)rows * c / CL), R1 = (int)((long long)rows * (c + 1) / CL);
    const int K0 = (int)((long long)NK1 * c / CL), K1 = (int)((long long)NK1 * (c + 1) / CL);
    const int OWN = (NK1 + CL - 1) / CL;
    int *hist = sm;                   // [W][NK1] per-warp counts -> prefix over this CTA's warps
    int *tot = hist + W * NK1;        // [NK1] rows of each key in this CTA
    int *base = tot + NK1;            // [NK1] sorted position of this CTA's first row of each key
    int *tmn = base + NK1;            // [NK1] dense: first row of a run of each key in this CTA
    int *nrn = tmn + NK1;             // [NK1] dense: run starts of each key in this CTA
    int *o_cnt = nrn + NK1;           // [OWN] owned keys: rows
    int *o_nrun = o_cnt + OWN;        //       run starts (dense)
    int *o_tmin = o_nrun + OWN;       //       first row (dense)
    int *o_off = o_tmin + OWN;        //       row offset
    int *o_g = o_off + OWN;           //       group
    int *o_t = o_g + OWN;             //       first 16-row tile
    int *o_lt = o_t + OWN;            //       first long tile (-1: not a long run)
    int *o_st = o_lt + OWN;           //       first short tile (-1: a long run)
    int *o_vt = o_st + OWN;           // [OWN][CL] owned keys: rows in each CTA
    int *misc = o_vt + kMetaCL * OWN; // [200]: this owner's 5 totals at [0..4], the earlier owners' at [8..12], n_bad at [36], warp totals at [40..199]
    unsigned char *act = (unsigned char *)(misc + 200);
    int *kc = misc + 200 + (a.L + 3) / 4;  // [R1 - R0] keys of this CTA's rows
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // this warp's contiguous rows within the CTA's range
    const int crow = R1 - R0;
    const int chunk = (crow + W - 1) / W;
    const int r0 = R0 + warp * chunk, r1 = min(R1, r0 + chunk);
    int sv[8], ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int row = r0 + u * 32 + lane;
        const bool ok = warp < W && row < r1;
        sv[u] = ok ? a.idx[row / a.K] : -1;
        ev[u] = (ok && a.topk) ? a.topk[row] : 0;
    }
    const int s_prev = (a.K == 1 && warp < W && r0 > 0 && r0 < r1) ? a.idx[r0 - 1] : -1;
    for (int i = tid; i < a.L; i += nthreads) {
        const int en = a.enabled[i], rk = a.rank[i];
        act[i] = (en != 0 && rk > 0) ? 1 : 0;
    }
    for (int i = tid; i < W * NK1; i += nthreads) hist[i] = 0;
    for (int i = tid; i < NK1; i += nthreads) {
        tmn[i] = 0x7fffffff;
        nrn[i] = 0;
    }
    if (tid == 0) misc[36] = 0;
    __syncthreads();

    // 1. keys, per-warp counts, dense run starts
    int bad = 0;
    int carry = -2;
    if (a.K == 1 && warp < W && r0 > 0 && r0 < r1) {
        int dummy = 0;
        carry = row_key_e(a, act, r0 - 1, s_prev, 0, &dummy);
    }
    auto count_step = [&](int base_row, int s, int e) {
        const int row = base_row + lane;
        const bool v = row < r1;
        const int key = v ? row_key_e(a, act, row, s, e, &bad) : -1;
        if (v) kc[row - R0] = key;
        if (a.K == 1) {
            const unsigned peers = key_peers(key, a.key_bits);
            const int leader = __ffs(peers) - 1;
            if (v && lane == leader) hist[warp * NK1 + key] += __popc(peers);
            int prev = __shfl_up_sync(0xffffffffu, key, 1);
            if (lane == 0) prev = carry;
            if (v && key < NK && key != prev) {
                atomicAdd(&nrn[key], 1);
                atomicMin(&tmn[key], row);
            }
            carry = __shfl_sync(0xffffffffu, key, 31);
        } else if (v) {
            atomicAdd(&hist[warp * NK1 + key], 1);
        }
        __syncwarp();
    };
    if (warp < W) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (r0 + u * 32 < r1) count_step(r0 + u * 32, sv[u], ev[u]);
        for (int b = r0 + 256; b < r1; b += 32) {
            const int row = b + lane;
            const bool v = row < r1;
            count_step(b, v ? a.idx[row / a.K] : -1, (v && a.topk) ? a.topk[row] : 0);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&misc[36], bad);
    __syncthreads();
    // per key: prefix over this CTA's warps (in place) and the CTA's total
    for (int b = tid; b < NK1; b += nthreads) {
        int run_rows = 0;
        for (int w = 0; w < W; ++w) {
            const int cw = hist[w * NK1 + b];
            hist[w * NK1 + b] = run_rows;
            run_rows += cw;
        }
        tot[b] = run_rows;
    }
    meta_cluster_sync();  // B1: every CTA's tot, tmn, nrn, n_bad

    // 2. owned keys: totals over the CTAs, then the key-space sums over them
    const int NO = K1 - K0;
    const int per = (NO + nthreads - 1) / nthreads;
    const int b0 = K0 + min(NO, tid * per), b1 = K0 + min(NO, tid * per + per);
    int *wt = misc + 40;  // [5][32] per-warp totals
    int sv5[5] = {0, 0, 0, 0, 0};
    for (int b = b0; b < b1; ++b) {
        // every CTA's words of key b: all loads issued before any is used
        int vt[kMetaCL], vn[kMetaCL], vm[kMetaCL];
#pragma unroll
        for (int q = 0; q < kMetaCL; ++q) vt[q] = meta_ld_peer(tot + b, (uint32_t)q);
        if (a.K == 1) {
#pragma unroll
            for (int q = 0; q < kMetaCL; ++q) {
                vn[q] = meta_ld_peer(nrn + b, (uint32_t)q);
                vm[q] = meta_ld_peer(tmn + b, (uint32_t)q);
            }
        }
        int cnt = 0, nr = 0, tm = 0x7fffffff;
#pragma unroll
        for (int q = 0; q < kMetaCL; ++q) {
            o_vt[(b - K0) * kMetaCL + q] = vt[q];
            cnt += vt[q];
            if (a.K == 1) {
                nr += vn[q];
                tm = min(tm, vm[q]);
            }
        }
        o_cnt[b - K0] = cnt;
        o_nrun[b - K0] = nr;
        o_tmin[b - K0] = tm;
        const int cc = b < NK ? cnt : 0;
        const bool run = cc > 0 && a.K == 1 && cc >= LORA_LONG_MIN && nr == 1;
        sv5[0] += cnt;
        sv5[1] += cc > 0 ? 1 : 0;
        sv5[2] += (cc + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS;
        sv5[3] += run ? (cc + LORA_LTILE_ROWS - 1) / LORA_LTILE_ROWS : 0;
        sv5[4] += (cc > 0 && !run) ? (cc + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS : 0;
    }
    int inc[5];
#pragma unroll
    for (int q = 0; q < 5; ++q) inc[q] = sv5[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int q = 0; q < 5; ++q) {
            const int v = __shfl_up_sync(0xffffffffu, inc[q], o);
            if (lane >= o) inc[q] += v;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int q = 0; q < 5; ++q) wt[q * 32 + warp] = inc[q];
    }
    __syncthreads();
    const int nw = nthreads / 32;
    int ex[5];
#pragma unroll
    for (int q = 0; q < 5; ++q) {
        int before = lane < warp ? wt[q * 32 + lane] : 0;
        int all = lane < nw ? wt[q * 32 + lane] : 0;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, o);
            all += __shfl_xor_sync(0xffffffffu, all, o);
        }
        ex[q] = before + inc[q] - sv5[q];
        if (tid == 0) misc[q] = all;  // this owner's totals
    }
    meta_cluster_sync();  // B2: every owner's totals

    // 3. the owners before this one (lane q of warp 0 reads owner q's five
    // totals, summed over the lanes), then this owner's keys' outputs and the
    // sorted position of every CTA's first row of each key
    if (warp == 0) {
        int pre[5];
#pragma unroll
        for (int k = 0; k < 5; ++k) pre[k] = lane < (int)c ? meta_ld_peer(misc + k, (uint32_t)lane) : 0;
#pragma unroll
        for (int k = 0; k < 5; ++k) {
#pragma unroll
            for (int o = 16; o; o >>= 1) pre[k] += __shfl_xor_sync(0xffffffffu, pre[k], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < 5; ++k) misc[8 + k] = pre[k];
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 5; ++k) ex[k] += misc[8 + k];
    for (int b = b0; b < b1; ++b) {
        const int cnt = o_cnt[b - K0];
        const int cc = b < NK ? cnt : 0;
        const bool run = cc > 0 && a.K == 1 && cc >= LORA_LONG_MIN && o_nrun[b - K0] == 1;
        const int off = ex[0];
        if (b < NK) a.m.key_count[b] = cnt;
        a.m.key_offset[b] = off;
        if (b < NK) {
            if (cc > 0) {
                a.m.key_group[b] = ex[1];
                a.m.group_key[ex[1]] = b;
                a.m.group_start[ex[1]] = off;
            } else {
                a.m.key_group[b] = -1;
            }
        }
        o_off[b - K0] = off;
        o_g[b - K0] = ex[1];
        o_t[b - K0] = ex[2];
        o_lt[b - K0] = run ? ex[3] : -1;
        o_st[b - K0] = run ? -1 : ex[4];
        int run_pos = off;
#pragma unroll
        for (int q = 0; q < kMetaCL; ++q) {
            meta_st_peer(base + b, (uint32_t)q, run_pos);
            run_pos += o_vt[(b - K0) * kMetaCL + q];
        }
        ex[0] += cnt;
        ex[1] += cc > 0 ? 1 : 0;
        ex[2] += (cc + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS;
        ex[3] += run ? (cc + LORA_LTILE_ROWS - 1) / LORA_LTILE_ROWS : 0;
        ex[4] += (cc > 0 && !run) ? (cc + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS : 0;
    }
    __syncthreads();
    // the owned keys' tiles: a warp per key, its lanes over the key's tiles
    for (int k = warp; k < NO; k += nw) {
        const int b = K0 + k;
        const int cc = b < NK ? o_cnt[k] : 0;
        if (cc == 0) continue;
        const int g = o_g[b - K0], off = o_off[b - K0];
        const int nt = (cc + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS;
        for (int i = lane; i < nt; i += 32) {
            const int rows_i = min(LORA_TILE_ROWS, cc - i * LORA_TILE_ROWS);
            a.m.tile_group[o_t[b - K0] + i] = g;
            a.m.tile_row0[o_t[b - K0] + i] = off + i * LORA_TILE_ROWS;
            a.m.tile_keyn[o_t[b - K0] + i] = (b << 5) | rows_i;
            if (o_st[b - K0] >= 0) {
                a.m.stile_row0[o_st[b - K0] + i] = off + i * LORA_TILE_ROWS;
                a.m.stile_keyn[o_st[b - K0] + i] = (b << 5) | rows_i;
            }
        }
        if (o_lt[b - K0] >= 0) {
            const int nl = (cc + LORA_LTILE_ROWS - 1) / LORA_LTILE_ROWS;
            for (int i = lane; i < nl; i += 32) {
                const int rows_i = min(LORA_LTILE_ROWS, cc - i * LORA_LTILE_ROWS);
                a.m.ltile_row0[o_lt[b - K0] + i] = off + i * LORA_LTILE_ROWS;
                a.m.ltile_keyn[o_lt[b - K0] + i] = (b << 8) | rows_i;
                a.m.ltile_tok0[o_lt[b - K0] + i] = o_tmin[b - K0] + i * LORA_LTILE_ROWS;
            }
        }
    }
    if ((int)c == CL - 1 && tid == 0) {
        // key NK (the inactive rows) is this owner's last key: its offset is
        // the number of active rows
        int G = 0, NT = 0, NL = 0, NS = 0, n_bad = 0;
#pragma unroll
        for (int q = 0; q < kMetaCL; ++q) {
            G += meta_ld_peer(misc + 1, (uint32_t)q);
            NT += meta_ld_peer(misc + 2, (uint32_t)q);
            NL += meta_ld_peer(misc + 3, (uint32_t)q);
            NS += meta_ld_peer(misc + 4, (uint32_t)q);
            n_bad += meta_ld_peer(misc + 36, (uint32_t)q);
        }
        const int n_active = rows - o_cnt[NK - K0];
        a.m.group_start[G] = n_active;
        a.m.counters[0] = n_active;
        a.m.counters[1] = G;
        a.m.counters[2] = n_bad;
        a.m.counters[3] = NT;
        a.m.counters[4] = NS;
        a.m.counters[5] = NL;
        if (n_bad) atomicExch(a.status, (int)LORA_ERR_DEVICE_INDEX);
    }
    meta_cluster_sync();  // B3: every base written; no shared-memory access across CTAs after this

    // 4. stable scatter: base + rows of earlier warps + earlier lanes
    if (warp < W) {
        const unsigned lt = (1u << lane) - 1u;
        for (int b = r0; b < r1; b += 32) {
            const int row = b + lane;
            const bool v = row < r1;
            const int key = v ? kc[row - R0] : -1;
            const unsigned peers = key_peers(key, a.key_bits);
            int pos = 0;
            if (v) pos = base[key] + hist[warp * NK1 + key] + __popc(peers & lt);
            __syncwarp();
            if (v) {
                a.m.sorted[pos] = row;
                if (lane == __ffs(peers) - 1) hist[warp * NK1 + key] += __popc(peers);
            }
            __syncwarp();
        }
    }
}

}  // namespace

lora_status_t lora_launch_build_meta(const lora_pool_t *pool, const int32_t *d_idx, int32_t T,
                                     const int32_t *d_topk, int32_t top_k, lora_meta_t *meta,
                                     cudaStream_t stream) {
    const int L = pool->desc.max_loras;
    const int E = pool->is_moe ? pool->desc.num_experts : 1;
    const int64_t rows = (int64_t)T * top_k;
    const int n_keys = L * E;
    if (rows > meta->max_rows || n_keys > meta->max_keys || n_keys > LORA_MAX_KEYS)
        return LORA_ERR_CAPACITY;
    if (!meta->sorted || !meta->counters || !meta->tile_keyn || !meta->ltile_keyn || !meta->stile_keyn)
        return LORA_ERR_INVALID_ARG;
    const int NK1 = n_keys + 1;
    if (!d_topk && top_k == 1 && rows <= kSmallRows && NK1 <= kSmallRows) {
        // small dense batch: one row and one key per thread
        int nthreads = (int)(std::max<int64_t>(rows, NK1) + 31) / 32 * 32;
        if (nthreads < 64) nthreads = 64;
        const size_t smem = dense_meta_smem_bytes(nthreads, 1, L);
        static std::atomic<int> configured_small[64];
        const int dev = pool->device < 64 ? pool->device : 63;
        if (!configured_small[dev].load(std::memory_order_acquire)) {
            LORA_CUDA_TRY(cudaFuncSetAttribute(build_meta_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSmemBudgetInts * 4));
            configured_small[dev].store(1, std::memory_order_release);
        }
        if (smem > (size_t)kSmemBudgetInts * 4) return LORA_ERR_CAPACITY;
        MetaArgs a;
        memset(&a, 0, sizeof(a));
        a.idx = d_idx;
        a.rank = pool->d_rank;
        a.enabled = pool->d_enabled;
        a.status = pool->d_status;
        a.T = T;
        a.K = 1;
        a.E = 1;
        a.L = L;
        a.n_keys = n_keys;
        a.m = *meta;
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(1, 1, 1);
        cfg.blockDim = dim3((unsigned)nthreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, build_meta_small_kernel, a));
        lora_note_launch();
        meta->T = T;
        meta->top_k = top_k;
        meta->n_keys = n_keys;
        meta->mode = 0;
        return LORA_OK;
    }
    if (rows >= kMetaClusterRows) {
        // thousands of rows: the cluster build (8 CTAs)
        const int rows_cta = (int)((rows + kMetaCL - 1) / kMetaCL);
        int nt = (rows_cta + 31) / 32 * 32;
        if (nt < 128) nt = 128;
        if (nt > kThreads) nt = kThreads;
        const long long rest = meta_cluster_ints(0, NK1, L, rows_cta);
        int Wc = (int)((kSmemBudgetInts - rest) / NK1);
        if (Wc > nt / 32) Wc = nt / 32;
        if (Wc >= 1) {
            MetaArgs a;
            memset(&a, 0, sizeof(a));
            a.idx = d_idx;
            a.topk = d_topk;
            a.rank = pool->d_rank;
            a.enabled = pool->d_enabled;
            a.status = pool->d_status;
            a.T = T;
            a.K = top_k;
            a.E = E;
            a.L = L;
            a.n_keys = n_keys;
            a.n_chunks = Wc;
            a.cache_keys = 1;
            a.key_bits = 1;
            while ((1LL << a.key_bits) <= (long long)NK1) ++a.key_bits;
            a.m = *meta;
            const size_t smem = (size_t)meta_cluster_ints(Wc, NK1, L, rows_cta) * 4;
            static std::atomic<int> configured_cl[64];
            const int dev = pool->device < 64 ? pool->device : 63;
            if (!configured_cl[dev].load(std::memory_order_acquire)) {
                LORA_CUDA_TRY(cudaFuncSetAttribute(build_meta_cluster_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudgetInts * 4));
                configured_cl[dev].store(1, std::memory_order_release);
            }
            cudaLaunchConfig_t cfg;
            memset(&cfg, 0, sizeof(cfg));
            cfg.gridDim = dim3(kMetaCL, 1, 1);
            cfg.blockDim = dim3((unsigned)nt, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = stream;
            cudaLaunchAttribute at[2];
            at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            at[0].val.programmaticStreamSerializationAllowed = 1;
            at[1].id = cudaLaunchAttributeClusterDimension;
            at[1].val.clusterDim.x = kMetaCL;
            at[1].val.clusterDim.y = 1;
            at[1].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 2;
            LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, build_meta_cluster_kernel, a));
            lora_note_launch();
            meta->T = T;
            meta->top_k = top_k;
            meta->n_keys = n_keys;
            meta->mode = pool->is_moe ? 1 : 0;
            return LORA_OK;
        }
    }
    // threads scale with the rows (one warp per 32 rows, 4..32 warps)
    int nthreads = (int)((rows + 31) / 32) * 32;
    if (nthreads < 128) nthreads = 128;
    if (nthreads > kThreads) nthreads = kThreads;
    const int nwarps = nthreads / 32;
    // chunk histograms [W][NK1] + 4 scratch rows + cnt, off, tmin, nrun + misc + slot table
    const long long fixed = 8LL * NK1 + 200 + (L + 3) / 4;
    int W = (int)((kSmemBudgetInts - fixed) / NK1);
    if (W > nwarps) W = nwarps;
    if (W < 1) return LORA_ERR_CAPACITY;
    const long long used = (long long)W * NK1 + fixed;
    const int cache = used + rows <= kSmemBudgetInts ? 1 : 0;
    MetaArgs a;
    a.idx = d_idx;
    a.topk = d_topk;
    a.rank = pool->d_rank;
    a.enabled = pool->d_enabled;
    a.status = pool->d_status;
    a.T = T;
    a.K = top_k;
    a.E = E;
    a.L = L;
    a.n_keys = n_keys;
    a.n_chunks = W;
    a.cache_keys = cache;
    a.key_bits = 1;
    while ((1LL << a.key_bits) <= (long long)NK1) ++a.key_bits;
    a.m = *meta;
    const size_t smem = (size_t)(used + (cache ? rows : 0)) * 4;
    // raise the kernel's shared-memory limit once per device (outside any capture)
    static std::atomic<int> configured[64];
    const int dev = pool->device < 64 ? pool->device : 63;
    if (!configured[dev].load(std::memory_order_acquire)) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(build_meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBudgetInts * 4));
        configured[dev].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3((unsigned)nthreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, build_meta_kernel, a));
    lora_note_launch();
    meta->T = T;
    meta->top_k = top_k;
    meta->n_keys = n_keys;
    meta->mode = pool->is_moe ? 1 : 0;
    return LORA_OK;
}
