// Block-level metadata build for small dense batches, shared by the
// metadata kernels (meta.cu) and the combined metadata + apply launch of the
// fused decode kernel (fused.cu).
#pragma once

#include "lora_internal.cuh"

// Arguments of the metadata builders: rows are tokens (dense, K = 1) or
// (token, k) pairs (MoE); key(row) = slot (dense) or slot*E + expert (MoE).
struct MetaArgs {
    const int32_t *idx;
    const int32_t *topk;
    const int32_t *rank;
    const int32_t *enabled;
    int32_t *status;
    int T, K, E, L, n_keys, n_chunks, cache_keys;
    int key_bits;  // smallest b with 2^b > n_keys + 1: the pattern of key -1 matches no key
    lora_meta_t m;
};

// Dense batches of at most kSmallRows rows and one key per thread: the
// same metadata as build_meta_kernel, with every warp's path kept short:
//   1. rows in steps of one row per thread (row step*nthreads + tid, so that
//      (step, warp, lane) is row order); each thread loads its rows' slots,
//      the slot tables load alongside
//   2. per (step, warp) segment: the lanes sharing a key (one match
//      instruction) -> the segment's count of each key, each row's rank among
//      them, and the first and last row of the key (a key's rows form one
//      contiguous run when last - first + 1 equals its count)
//   3. key k = thread k: its count and the exclusive prefix over the
//      segments, then one block-wide scan of the row offsets, group index and
//      tile counts, and the key's groups and tiles
//   4. stable scatter: key offset + earlier segments + earlier lanes
// Shared memory: dense_meta_smem_bytes(); the caller has waited for the
// grid dependency before the call.
constexpr int kSmallRows = 1024;  // most rows (one step) and keys of the small build
constexpr int kMaxSteps = 4;      // most row steps of one block

static __host__ __device__ inline size_t dense_meta_smem_bytes(int nthreads, int steps, int L) {
    const int NK1 = L + 1;
    return ((size_t)steps * (nthreads / 32) * NK1 + NK1 + 2 * (size_t)L + 160 + 8) * 4 + (size_t)(L + 3) / 4 * 4;
}

static __device__ void dense_meta_block(const MetaArgs &a, int *sm, int steps) {
    const int L = a.L, NK = a.n_keys, NK1 = NK + 1, T = a.T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, W = nthreads >> 5, NS = steps * W;
    int *hist = sm;                   // [NS][NK1] per-segment counts -> exclusive prefix over the segments
    int *off = hist + NS * NK1;       // [NK1] row offset of each key
    int *tmin = off + NK1;            // [NK] first row of each key
    int *tmax = tmin + NK;            // [NK] last row of each key
    int *wt = tmax + NK;              // [5][32] warp totals of the key scan
    int *misc = wt + 160;             // [8]: n_bad
    unsigned char *act = (unsigned char *)(misc + 8);  // [L] slot enabled with rank > 0

    // 1. this thread's rows' slots and the slot tables (one round trip)
    int sv[kMaxSteps];
#pragma unroll
    for (int st = 0; st < kMaxSteps; ++st) {
        const int t = st * nthreads + tid;
        sv[st] = (st < steps && t < T) ? a.idx[t] : -1;
    }
    for (int i = tid; i < L; i += nthreads) {
        const int en = a.enabled[i], rk = a.rank[i];
        act[i] = (en != 0 && rk > 0) ? 1 : 0;
    }
    for (int i = tid; i < NS * NK1; i += nthreads) hist[i] = 0;
    for (int i = tid; i < NK; i += nthreads) {
        tmin[i] = 0x7fffffff;
        tmax[i] = -1;
    }
    if (tid == 0) misc[0] = 0;
    __syncthreads();

    // 2. keys (inactive rows: NK, so they sort last; no row: -1)
    int keys[kMaxSteps], wranks[kMaxSteps], nbad = 0;
#pragma unroll
    for (int st = 0; st < kMaxSteps; ++st) {
        keys[st] = -1;
        wranks[st] = 0;
        if (st < steps) {
            const int t = st * nthreads + tid;
            const int s = sv[st];
            const bool valid = s >= 0 && s < L;
            const int key = t < T ? ((valid && act[s]) ? s : NK) : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const int wrank = __popc(peers & ((1u << lane) - 1u));
            const int seg = st * W + warp;
            if (key >= 0 && wrank == 0) {
                hist[seg * NK1 + key] = __popc(peers);
                if (key < NK) {
                    atomicMin(&tmin[key], (t - lane) + __ffs(peers) - 1);
                    atomicMax(&tmax[key], (t - lane) + 31 - __clz(peers));
                }
            }
            nbad += (t < T && s != -1 && !valid) ? 1 : 0;
            keys[st] = key;
            wranks[st] = wrank;
        }
    }
    nbad = __reduce_add_sync(0xffffffffu, nbad);
    if (lane == 0 && nbad) atomicAdd(&misc[0], nbad);
    __syncthreads();

    // 3. key k = tid: count and prefix over the segments, then the key-space scan
    const int k = tid;
    int c = 0;
    if (k < NK1)
        for (int sg = 0; sg < NS; ++sg) {
            const int v = hist[sg * NK1 + k];
            hist[sg * NK1 + k] = c;
            c += v;
        }
    const bool real = k < NK, nonempty = real && c > 0;
    const bool run = nonempty && c >= LORA_LONG_MIN && tmax[k] - tmin[k] + 1 == c;
    int v5[5];
    v5[0] = k < NK1 ? c : 0;
    v5[1] = nonempty ? 1 : 0;
    v5[2] = real ? (c + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS : 0;
    v5[3] = run ? (c + LORA_LTILE_ROWS - 1) / LORA_LTILE_ROWS : 0;
    v5[4] = (nonempty && !run) ? (c + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS : 0;
    int inc[5];
#pragma unroll
    for (int q = 0; q < 5; ++q) inc[q] = v5[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int q = 0; q < 5; ++q) {
            const int v = __shfl_up_sync(0xffffffffu, inc[q], o);
            if (lane >= o) inc[q] += v;
        }
    }
    if (lane == 31)
#pragma unroll
        for (int q = 0; q < 5; ++q) wt[q * 32 + warp] = inc[q];
    __syncthreads();
    int ex[5], tot[5];
#pragma unroll
    for (int q = 0; q < 5; ++q) {
        int before = lane < warp ? wt[q * 32 + lane] : 0;
        int all = lane < W ? wt[q * 32 + lane] : 0;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, o);
            all += __shfl_xor_sync(0xffffffffu, all, o);
        }
        ex[q] = before + inc[q] - v5[q];
        tot[q] = all;
    }
    if (k < NK1) {
        off[k] = ex[0];
        a.m.key_offset[k] = ex[0];
    }
    if (real) {
        a.m.key_count[k] = c;
        a.m.key_group[k] = nonempty ? ex[1] : -1;
        if (nonempty) {
            const int g = ex[1];
            a.m.group_key[g] = k;
            a.m.group_start[g] = ex[0];
            for (int i = 0; i < v5[2]; ++i) {
                a.m.tile_group[ex[2] + i] = g;
                a.m.tile_row0[ex[2] + i] = ex[0] + i * LORA_TILE_ROWS;
                a.m.tile_keyn[ex[2] + i] = (k << 5) | min(LORA_TILE_ROWS, c - i * LORA_TILE_ROWS);
            }
            for (int i = 0; i < v5[3]; ++i) {
                a.m.ltile_row0[ex[3] + i] = ex[0] + i * LORA_LTILE_ROWS;
                a.m.ltile_keyn[ex[3] + i] = (k << 8) | min(LORA_LTILE_ROWS, c - i * LORA_LTILE_ROWS);
                a.m.ltile_tok0[ex[3] + i] = tmin[k] + i * LORA_LTILE_ROWS;
            }
            for (int i = 0; i < v5[4]; ++i) {
                a.m.stile_row0[ex[4] + i] = ex[0] + i * LORA_TILE_ROWS;
                a.m.stile_keyn[ex[4] + i] = (k << 5) | min(LORA_TILE_ROWS, c - i * LORA_TILE_ROWS);
            }
        }
    }
    __syncthreads();

    // 4. stable scatter
#pragma unroll
    for (int st = 0; st < kMaxSteps; ++st) {
        const int key = keys[st];
        if (st < steps && key >= 0)
            a.m.sorted[off[key] + hist[(st * W + warp) * NK1 + key] + wranks[st]] = st * nthreads + tid;
    }
    if (tid == 0) {
        const int n_active = off[NK];
        const int n_bad = misc[0];
        a.m.group_start[tot[1]] = n_active;
        a.m.counters[0] = n_active;
        a.m.counters[1] = tot[1];
        a.m.counters[2] = n_bad;
        a.m.counters[3] = tot[2];
        a.m.counters[4] = tot[4];
        a.m.counters[5] = tot[3];
        if (n_bad) atomicExch(a.status, (int)LORA_ERR_DEVICE_INDEX);
    }
}

