// Fused decode apply: the multi-tenant LoRA delta of a small batch (decode
// tokens spread over the pool's slots) in one kernel launch, with the fp32
// rank-space intermediate kept on chip.
//
// The vLLM LoRA layer pages compute add_shrink into a zeroed fp32 buffer
// [n_slices][T][rank] (scale 1.0) and add_expand with add_input=True at the
// slice offsets (RowParallelLinearWithShardedLoRA.apply; SGLang's per-slot
// scalings).  Here one thread-block cluster of CS CTAs serves one adapter
// slot a; CTA c of the cluster owns hidden chunk c (shrink) and output block
// c (expand):
//
//   prologue, before the grid dependency wait (pool weights only: lora_set /
//     lora_reset write them through copies and plain launches, which are
//     complete before this grid starts):
//       the slot's A_j rows of chunk c, one TMA box per slice and 16 ranks
//       (rows as 128-byte lines of each 64-column chunk, 128-byte swizzle),
//       and the B_j fragments of output block c that this thread's expand
//       MMAs use, loaded into registers;
//   after the wait (the metadata build is complete): the batch's sorted
//     rows, this slot's count and offset (one round trip), then for every
//     tile of up to 16 of the slot's rows:
//       x rows of chunk c and y rows of block c into shared memory
//       (16-byte cp.async by every thread; x in the same swizzled layout);
//       shrink  P_c[t][j*KG + k] = sum_{h in chunk c} x[t][h] * A_j[a][k][h]
//               (m16n8k16 bf16 MMAs, fp32 accumulate; one warp per pair of a
//               16-rank M block and an 8-row N block, two accumulators over
//               alternate k steps);
//       cluster barrier; v[t][j][k] = scale[a] * sum_{c'} P_c'[t][j*KG + k]
//               read from the peers' shared memory (DSMEM) in rank order, as
//               bf16 hi + lo (v - hi), which carries the fp32 value to ~16
//               bits through the bf16 MMAs;
//       expand  y[t][o] += v_hi[t] . B[o] + v_lo[t] . B[o] over block c
//               (rows on M, 8 outputs per N block, ranks on K), added to the
//               y tile in shared memory, which is then stored with 16-byte
//               writes.
// Nothing but y is written to global memory, the launch needs no workspace,
// and every sum has a fixed order, so results do not depend on timing.
// Clusters are independent of one another; the only waits are on this CTA's
// own copies (bounded, LORA_ERR_TIMEOUT on give-up) and the cluster's
// hardware barrier, which every CTA of a cluster reaches on the same path.
#include <string.h>

#include <algorithm>
#include <atomic>

#include "lora_internal.cuh"
#include "meta_block.cuh"
#include "mma_common.cuh"

namespace {

using namespace bgmv;

constexpr int kFThreads = 256;
constexpr int kFWarps = kFThreads / 32;
constexpr int kNT = LORA_TILE_ROWS;  // rows per tile: two 8-row N blocks of the shrink, M of the expand
constexpr int kMaxT = 1024;          // batch rows whose sorted list a CTA stages
constexpr int kSmem1 = 212 * 1024;   // dynamic shared memory at one CTA per SM (static + dynamic <= 227 KB)
constexpr int kPW = 6;               // expand blocks per pass
constexpr int kSmem2 = 100 * 1024;   // ... at two (with the static shared memory and the 1 KB per CTA the SM keeps)

struct alignas(64) FArgs {
    CUtensorMap tm_a[LORA_MAX_SLICES];  // A_j as [L*R rows][H]: boxes of BR rows x NCH chunks
    int n_slices, H, out_total, CS, HC, NCH, OB, T, L, R, BR, kgb;
    int out_off[LORA_MAX_SLICES];
    const uint16_t *B[LORA_MAX_SLICES];
    long long B_ss[LORA_MAX_SLICES];
    const int32_t *rank, *enabled;
    const float *scale;
    const int32_t *key_count, *key_offset, *sorted;
    const uint16_t *x;
    long long ldx;
    uint16_t *y;
    long long ldy;
    float post_scale;
    int box_bytes;                      // one A box in shared memory
    int off_x, off_p, off_v;            // byte offsets (A at 0)
    int pp;                             // floats per row of P (multiple of 4)
    int vp, v_bytes;                    // v tile row pitch (elements), bytes of one v tile
    int *status;
    int spin_limit;
    // batch mode: the slot clusters find their rows in idx, and the CTA of
    // one more cluster builds the batch metadata (ma) at the same time
    const int32_t *idx;
    int idx_mode, meta_steps;
    MetaArgs ma;
};

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ uint32_t ldg_nc_u32(const uint16_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float4 ld_dsmem_v4(const float *local, uint32_t peer) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(peer));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(ra)
                 : "memory");
    return v;
}

// KSX: most 16-rank k steps of the expand (1, 2, 4); GMAX: most 32-output
// groups per warp; MINB: CTAs per SM the launch is sized for.
//
// The rank index k is only summed over, so the expand may take the ranks of
// a 16-rank k step in any order that B and v share.  It takes them so that
// each lane's B fragment is one 8-byte load: lane (g, c4) holds ranks 4c4 ..
// 4c4+3 of output row g, which the MMA reads as its k = 2c4, 2c4+1 (first
// half) and 2c4+8, 2c4+9 (second half); the v tile stores rank k at MMA
// column kcol(k) accordingly.
__device__ __forceinline__ int kcol(int k) {  // k within a 16-rank step -> MMA k column
    const int c = k >> 2, e = k & 3;
    return e < 2 ? 2 * c + e : 2 * c + 6 + e;
}

template <int KSX, int GMAX, int MINB>
__global__ void __launch_bounds__(kFThreads, MINB) bgmv_fused_kernel(const __grid_constant__ FArgs p) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = smem_raw + ((1024u - (smem_u32_of(smem_raw) & 1023u)) & 1023u);  // the swizzled boxes want 1 KB
    __shared__ __align__(8) uint64_t abar;
    __shared__ int s_sorted[kMaxT];  // the batch's sorted rows, or its slots in batch mode
    __shared__ int s_list[kMaxT];    // batch mode: this slot's rows
    __shared__ int s_cnt[32];
    __shared__ int s_oo[LORA_MAX_SLICES + 1];
    __shared__ const uint16_t *s_B[LORA_MAX_SLICES];
    __shared__ int s_nb[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c4 = lane & 3;
    const int c = (int)cluster_rank();
    const int a = blockIdx.x / p.CS;
    // batch mode: the batch's slot ids into L2 before the wait (a prefetch
    // cannot return stale data: later loads read L2, which every write
    // reaches first), one 128-byte line per thread of each cluster's first CTA
    if (p.idx_mode && c == 0 && tid < (p.T * 4 + 127) / 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.idx + tid * 32));
    if (a == p.L) {
        // batch mode's last cluster: its first CTA builds the metadata
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
        if (c == 0) dense_meta_block(p.ma, (int *)smem, p.meta_steps);
        return;
    }
    const int ns = p.n_slices;
    const int h0 = c * p.HC, hlen = max(0, min(p.H - h0, p.HC));
    const int ob0 = min(p.out_total, c * p.OB), olen = min(p.out_total - ob0, p.OB);
    // the slot's tables: requested now, first used by the rank-dependent
    // copies below
    const int en = __ldcg(p.enabled + a), rk = __ldcg(p.rank + a);
    const float sc_slot = __ldcg(p.scale + a);
    if (tid == 0) {
        // per-slice tables, read with constant parameter indices (a run-time
        // index into the parameter space is slow); indexed freely from here
#pragma unroll
        for (int j = 0; j < LORA_MAX_SLICES; ++j) {
            s_oo[j] = j < ns ? p.out_off[j] : 0x7fffffff;
            s_B[j] = j < ns ? p.B[j] + (long long)a * p.B_ss[j] : nullptr;
        }
        s_oo[LORA_MAX_SLICES] = 0x7fffffff;
        mbar_init(&abar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ---------------- prologue: the first A box of every slice (ranks 0 ..
    // BR-1, which every active slot needs), before the slot's rank is known
    if (tid == 0 && hlen > 0) {
        asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&abar)),
                     "r"((uint32_t)(ns * p.box_bytes))
                     : "memory");
        for (int j = 0; j < ns; ++j) tma_load_3d(smem + (long long)j * p.kgb * p.box_bytes, &p.tm_a[j], 0, a * p.R, h0 >> 6, &abar);
    }
    // L2 prefetch of this cluster's share of the batch rows (T / L of them):
    // x columns of chunk c and y columns of block c, one 128-byte line per
    // thread.  A prefetch cannot return stale data (later loads read L2,
    // which every write reaches first), so it may run before the wait.
    {
        const int t0 = (int)((long long)a * p.T / p.L), t1 = (int)((long long)(a + 1) * p.T / p.L);
        const int xl = (hlen + 63) >> 6, yl = (olen + 63) >> 6;  // 128-byte lines per row
        const int per = xl + yl;
        for (int i = tid; i < (t1 - t0) * per; i += kFThreads) {
            const int t = t0 + i / per, l = i - (i / per) * per;
            const uint16_t *ptr = l < xl ? p.x + (long long)t * p.ldx + h0 + l * 64
                                         : p.y + (long long)t * p.ldy + ob0 + (l - xl) * 64;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
        }
    }

    const int r = en != 0 ? rk : 0;
    const bool act = r > 0;
    const int rs = (r + 7) & ~7;
    const int nbox = act ? (r + p.BR - 1) / p.BR : 0;  // A boxes per slice for this slot's rank
    if (tid == 0) {
        const int more = (act && hlen > 0) ? nbox - 1 : 0;
        mbar_expect_tx(&abar, (uint32_t)(ns * more * p.box_bytes));  // the arrival that completes the phase
        for (int j = 0; j < ns; ++j)
            for (int b = 1; b <= more; ++b)
                tma_load_3d(smem + (long long)(j * p.kgb + b) * p.box_bytes, &p.tm_a[j], 0, a * p.R + b * p.BR,
                            h0 >> 6, &abar);
    }
    // L2 prefetch of this CTA's B rows (slot a, outputs of block c): the
    // expand's fragments are loaded from L2 after the shrink.  The rank-
    // dependent copies and prefetches read only the pool (rank and enabled
    // change only through lora_set / lora_reset, complete before this grid),
    // so they overlap the previous kernel too.
    if (act) {
        int nl[LORA_MAX_SLICES], tot = 0;
        for (int j = 0; j < ns; ++j) {
            const int s0 = max(ob0, s_oo[j]), s1 = min(ob0 + olen, s_oo[j] + (j + 1 < ns ? s_oo[j + 1] - s_oo[j] : p.out_total - s_oo[j]));
            nl[j] = s1 > s0 ? ((s1 - s0) * rs * 2 + 127) >> 7 : 0;
            tot += nl[j];
        }
        for (int i = tid; i < tot; i += kFThreads) {
            int j = 0, l = i;
            while (l >= nl[j]) l -= nl[j++];
            const int s0 = max(ob0, s_oo[j]);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(s_B[j] + (long long)(s0 - s_oo[j]) * rs + l * 64));
        }
    }
    // ---------------- the metadata (and everything before it) is complete
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    // batch mode: the slots of rows j*256 + tid, kept in registers (stored to
    // shared memory once the work below no longer waits behind them)
    int iv[kMaxT / kFThreads];
#pragma unroll
    for (int j = 0; j < kMaxT / kFThreads; ++j) {
        const int t = j * kFThreads + tid;
        iv[j] = (p.idx_mode && t < p.T) ? __ldcg(p.idx + t) : -1;
    }
    if (!p.idx_mode) {
        for (int i = tid; i < p.T; i += kFThreads) s_sorted[i] = __ldcg(p.sorted + i);
        if (tid == 0) {
            s_nb[0] = __ldcg(p.key_count + a);
            s_nb[1] = __ldcg(p.key_offset + a);
        }
    }
    // this warp's expand groups of 32 outputs G = warp + 8 i.  Within a group
    // MMA block q (q < 4) computes outputs o0 + 4n + q of its N columns n, so
    // lane (g, c4) ends up with the 8 consecutive outputs o0 + 8c4 .. +7 of
    // rows g and g+8, read and written with one 16-byte access each.
    const int ngr = act ? (olen >> 5) : 0;
    const int ngw = ngr > warp ? (ngr - warp + kFWarps - 1) / kFWarps : 0;
    __syncthreads();
    if (p.idx_mode) {
        // this slot's rows in batch order: rows t = j*256 + tid, so (j, warp,
        // lane) is row order; a ballot per warp and row step, a scan over
        // the (step, warp) counts, then each row's place
        const int nj = (p.T + kFThreads - 1) / kFThreads;
        unsigned m4[kMaxT / kFThreads];
#pragma unroll
        for (int j = 0; j < kMaxT / kFThreads; ++j) {
            const int t = j * kFThreads + tid;
            m4[j] = __ballot_sync(0xffffffffu, j < nj && t < p.T && iv[j] == a);
            if (j < nj && lane == 0) s_cnt[j * kFWarps + warp] = __popc(m4[j]);
        }
        __syncthreads();
        const int ncnt = nj * kFWarps;
        const int v = lane < ncnt ? s_cnt[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
        for (int j = 0; j < kMaxT / kFThreads; ++j) {
            // exclusive prefix of this (step, warp) segment, from its lane of the scan
            const int before = __shfl_sync(0xffffffffu, incl - v, (j * kFWarps + warp) & 31);
            if (j < nj && ((m4[j] >> lane) & 1u))
                s_list[before + __popc(m4[j] & ((1u << lane) - 1u))] = j * kFThreads + tid;
        }
        if (tid == 0) {
            s_nb[0] = total;
            s_nb[1] = 0;
        }
        __syncthreads();
    }
    const int n = act ? s_nb[0] : 0, off = s_nb[1];
    const int *rows = p.idx_mode ? s_list : s_sorted;
    if (n <= 0) {  // the same for every CTA of the cluster
        if (hlen > 0) mbar_wait(&abar, 0, p.spin_limit, p.status);  // no copy may be in flight at exit
        return;
    }

    const int KG = p.kgb * 16;          // P columns per slice
    const int MB = ns * nbox;           // shrink M blocks (one per A box)
    const int ksteps = hlen >> 4;       // hlen is a multiple of 64
    const int R16 = (r + 15) & ~15;
    const int ksx = (rs + 15) >> 4;
    int j0 = 0, j1 = 0;
    for (int j = 1; j < ns; ++j) {
        if (ob0 >= s_oo[j]) j0 = j;
        if (ob0 + olen - 1 >= s_oo[j]) j1 = j;
    }
    const int nj = j1 - j0 + 1;
    const float sc = sc_slot * p.post_scale;
    char *Xs = smem + p.off_x;  // [NCH][16 rows][128 B], 128-byte swizzle
    float *P = (float *)(smem + p.off_p);  // [16][pp]
    uint16_t *Vh = (uint16_t *)(smem + p.off_v);
    uint16_t *Vl = (uint16_t *)(smem + p.off_v + p.v_bytes);
    const int xu = hlen >> 3;  // 16-byte units per x row
    const int n_tiles = (n + kNT - 1) / kNT;
    // shrink lane constants: A row of this lane in its box, x row of this lane
    const int rho = ((lane & 7) + ((lane >> 3) & 1) * 8) & (p.BR - 1);  // BR = 8: rows 8-15 repeat 0-7
    const int a_lane = rho * 128, a_sw = rho & 7, a_half = lane >> 4;
    const int x_sw = lane & 7, x_half = (lane >> 3) & 1;
    const int cstride = p.BR * 128;

    for (int tile = 0; tile < n_tiles; ++tile) {
        const int nt = min(kNT, n - tile * kNT);
        if (tile > 0) __syncthreads();  // the previous tile is done with the x tile
        const int *s_tok = rows + off + tile * kNT;
        // x rows of chunk c (swizzled like the A boxes): a warp per row, the
        // lanes over its 16-byte units
        for (int t = warp; t < nt; t += kFWarps) {
            const uint16_t *xr = p.x + (long long)s_tok[t] * p.ldx + h0;
            char *xd = Xs + t * 128;
            for (int u = lane; u < xu; u += 32) cp_async16(xd + (u >> 3) * 2048 + (((u & 7) ^ (t & 7)) << 4), xr + u * 8);
        }
        if (tile == 0) mbar_wait(&abar, 0, p.spin_limit, p.status);
        cp_async_wait_all();
        __syncthreads();

        // ---------------- shrink of chunk c: pairs (M block, k half) pi = warp,
        // warp + 8 (at most 16 pairs: M blocks <= 8), so a warp's pairs share
        // the k half kh = warp & 1.  Each pair runs four accumulator chains
        // (two N blocks x even / odd k steps) with the fragments of two k steps
        // loaded before their MMAs.  First halves are stored to P, then, after
        // a barrier, second halves are added to them.
        const int NB = (nt + 7) >> 3;
        const int khs = (((ksteps + 1) >> 1) + 1) & ~1;  // k steps per half, even
        const int kh = warp & 1;
        float dd[2][2][4];  // [pair of this warp][N block][4]
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
            const int pi = warp + w2 * kFWarps;
#pragma unroll
            for (int u = 0; u < 4; ++u) dd[w2][0][u] = dd[w2][1][u] = 0.f;
            if (pi < 2 * MB) {
                const int mb = pi >> 1;
                const int j = mb / nbox, b = mb - j * nbox;
                const char *abox = smem + (long long)(j * p.kgb + b) * p.box_bytes + a_lane;
                float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};  // N block 0: even, odd k
                float f0[4] = {0.f, 0.f, 0.f, 0.f}, f1[4] = {0.f, 0.f, 0.f, 0.f};  // N block 1: even, odd k
                const int k0 = kh * khs, k1 = min(ksteps, k0 + khs);
                for (int k = k0; k < k1; k += 2) {
                    const int q = k >> 2, e = (k & 3) * 2;  // 64-column chunk, first 16-byte unit of step k
                    const char *aq = abox + q * cstride;
                    const char *xq = Xs + q * 2048 + (lane & 7) * 128;
                    const bool two = k + 1 < k1;
                    uint32_t a0, a1, a2, a3, c0 = 0u, c1 = 0u, c2 = 0u, c3 = 0u;
                    uint32_t b0, b1, b2 = 0u, b3 = 0u, g0 = 0u, g1 = 0u, g2 = 0u, g3 = 0u;
                    ldsm_x4(aq + (((e + a_half) ^ a_sw) << 4), a0, a1, a2, a3);
                    ldsm_x2(xq + (((e + x_half) ^ x_sw) << 4), b0, b1);
                    if (NB > 1) ldsm_x2(xq + 1024 + (((e + x_half) ^ x_sw) << 4), b2, b3);
                    if (two) {
                        ldsm_x4(aq + (((e + 2 + a_half) ^ a_sw) << 4), c0, c1, c2, c3);
                        ldsm_x2(xq + (((e + 2 + x_half) ^ x_sw) << 4), g0, g1);
                        if (NB > 1) ldsm_x2(xq + 1024 + (((e + 2 + x_half) ^ x_sw) << 4), g2, g3);
                    }
                    mma16816(e0, a0, a1, a2, a3, b0, b1);
                    if (NB > 1) mma16816(f0, a0, a1, a2, a3, b2, b3);
                    if (two) {
                        mma16816(e1, c0, c1, c2, c3, g0, g1);
                        if (NB > 1) mma16816(f1, c0, c1, c2, c3, g2, g3);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    dd[w2][0][u] = e0[u] + e1[u];
                    dd[w2][1][u] = f0[u] + f1[u];
                }
            }
        }
        // D[m][t] of a pair -> P[t][j*KG + b*BR + m]: rows m = g (and g+8 when
        // BR = 16), columns t = 2c4, 2c4+1 (N block 0) and +8 (N block 1)
        auto store_pairs = [&](bool add) {
#pragma unroll
            for (int w2 = 0; w2 < 2; ++w2) {
                const int pi = warp + w2 * kFWarps;
                if (pi < 2 * MB) {
                    const int mb = pi >> 1;
                    const int j = mb / nbox, b = mb - j * nbox;
                    float *pk = P + j * KG + b * p.BR + g + 2 * c4 * p.pp;
                    const int nrow = p.BR == 16 ? 2 : 1;
                    for (int h = 0; h < nrow; ++h) {
                        float *q = pk + h * 8;
#pragma unroll
                        for (int nb = 0; nb < 2; ++nb) {
                            float *q2 = q + nb * 8 * p.pp;
                            const float v0 = dd[w2][nb][2 * h], v1 = dd[w2][nb][2 * h + 1];
                            if (add) {
                                q2[0] += v0;
                                q2[p.pp] += v1;
                            } else {
                                q2[0] = v0;
                                q2[p.pp] = v1;
                            }
                        }
                    }
                }
            }
        };
        if (kh == 0) store_pairs(false);
        __syncthreads();
        if (kh == 1) store_pairs(true);
        __syncthreads();
        // the expand's operands, requested before the cluster barrier so their
        // latency hides behind it and the gather: B rows o0 + 4g + q (ranks
        // ks*16 + 4c4 .. +3) of each group and the y values of rows g and g+8,
        // outputs o0 + 8c4 .. +7
        const bool r0ok = g < nt, r1ok = g + 8 < nt;
        const long long yrow0 = r0ok ? (long long)s_tok[g] * p.ldy : 0, yrow1 = r1ok ? (long long)s_tok[g + 8] * p.ldy : 0;
        uint2 bq[GMAX][4][KSX];
        uint4 yv[GMAX][2];
        int gj[GMAX];  // slice of each group
#pragma unroll
        for (int i = 0; i < GMAX; ++i) {
            gj[i] = 0;
            yv[i][0] = yv[i][1] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int ks = 0; ks < KSX; ++ks) bq[i][q][ks] = make_uint2(0u, 0u);
            if (i < ngw) {
                const int o0 = ob0 + (warp + kFWarps * i) * 32;
                int jj = 0;
                for (int j = 1; j < ns; ++j)
                    if (o0 >= s_oo[j]) jj = j;
                gj[i] = jj;
                const uint16_t *bb = s_B[jj] + (long long)(o0 - s_oo[jj] + 4 * g) * rs + 4 * c4;
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int ks = 0; ks < KSX; ++ks)
                        if (ks * 16 + 4 * c4 < rs) bq[i][q][ks] = __ldg((const uint2 *)(bb + (long long)q * rs + ks * 16));
                if (r0ok) yv[i][0] = __ldcg((const uint4 *)(p.y + yrow0 + o0 + 8 * c4));
                if (r1ok) yv[i][1] = __ldcg((const uint4 *)(p.y + yrow1 + o0 + 8 * c4));
            }
        }
        cluster_arrive();
        cluster_wait();  // every CTA's P of this tile is complete and visible

        // ---------------- v of the slices of this CTA's output block
        if (olen > 0) {
            const int per_t = nj * (R16 >> 2);
            for (int i = tid; i < nt * per_t; i += kFThreads) {
                const int t = i / per_t, rem = i - t * per_t;
                const int jq = rem / (R16 >> 2), k4 = (rem - jq * (R16 >> 2)) * 4;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (k4 < r) {
                    const float *src = P + t * p.pp + (j0 + jq) * KG + k4;
#pragma unroll
                    for (int q0 = 0; q0 < 8; q0 += 4) {
                        float4 part[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (q0 + q < p.CS) part[q] = ld_dsmem_v4(src, (uint32_t)(q0 + q));
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (q0 + q < p.CS) {
                                v.x += part[q].x;
                                v.y += part[q].y;
                                v.z += part[q].z;
                                v.w += part[q].w;
                            }
                        }
                    }
                    v.x = k4 + 0 < r ? v.x * sc : 0.f;
                    v.y = k4 + 1 < r ? v.y * sc : 0.f;
                    v.z = k4 + 2 < r ? v.z * sc : 0.f;
                    v.w = k4 + 3 < r ? v.w * sc : 0.f;
                }
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y), h23 = __floats2bfloat162_rn(v.z, v.w);
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                // ranks k4, k4+1 -> MMA columns kcol(k4), +1; k4+2, k4+3 -> kcol(k4+2), +1
                const int base = t * p.vp + jq * R16 + (k4 & ~15);
                const int c0 = base + kcol(k4 & 15), c1 = base + kcol((k4 & 15) + 2);
                *(uint32_t *)(Vh + c0) = *(const uint32_t *)&h01;
                *(uint32_t *)(Vh + c1) = *(const uint32_t *)&h23;
                *(uint32_t *)(Vl + c0) = pack_bf16x2(v.x - f01.x, v.y - f01.y);
                *(uint32_t *)(Vl + c1) = pack_bf16x2(v.z - f23.x, v.w - f23.y);
            }
            // rows of the v tiles past the tile's rows: zero
            for (int i = tid; i < (kNT - nt) * nj * R16 / 2; i += kFThreads) {
                const int t = nt + i / (nj * R16 / 2), cc = (i - (t - nt) * (nj * R16 / 2)) * 2;
                *(uint32_t *)(Vh + t * p.vp + cc) = 0u;
                *(uint32_t *)(Vl + t * p.vp + cc) = 0u;
            }
        }
        cluster_arrive();  // this CTA has read its peers' P
        __syncthreads();   // v tiles written

        // ---------------- expand of output block c: this warp's groups
        if (ngw > 0) {
            const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
            uint32_t hf[KSX][4], lf[KSX][4];
            int cur = -1;
#pragma unroll
            for (int i = 0; i < GMAX; ++i) {
                if (i < ngw) {
                    const int jj = gj[i];
                    if (jj != cur) {
                        cur = jj;
                        const uint16_t *vh = Vh + arow * p.vp + (jj - j0) * R16 + (lane >> 4) * 8;
                        const uint16_t *vl = Vl + arow * p.vp + (jj - j0) * R16 + (lane >> 4) * 8;
#pragma unroll
                        for (int ks = 0; ks < KSX; ++ks) {
                            if (ks < ksx) {
                                ldsm_x4(vh + ks * 16, hf[ks][0], hf[ks][1], hf[ks][2], hf[ks][3]);
                                ldsm_x4(vl + ks * 16, lf[ks][0], lf[ks][1], lf[ks][2], lf[ks][3]);
                            }
                        }
                    }
                    float acc[4][4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
#pragma unroll
                        for (int ks = 0; ks < KSX; ++ks) {
                            if (ks < ksx) {
                                mma16816(acc[q], hf[ks][0], hf[ks][1], hf[ks][2], hf[ks][3], bq[i][q][ks].x, bq[i][q][ks].y);
                                mma16816(acc[q], lf[ks][0], lf[ks][1], lf[ks][2], lf[ks][3], bq[i][q][ks].x, bq[i][q][ks].y);
                            }
                        }
                    }
                    // row g: outputs o0 + 8c4 + q (acc[q][0]) and + 4 + q (acc[q][1]); row g+8: [2], [3]
                    const int o = ob0 + (warp + kFWarps * i) * 32 + 8 * c4;
                    if (r0ok) {
                        const uint4 u = yv[i][0];
                        uint4 w;
                        w.x = pack_bf16x2(bf16lo(u.x) + acc[0][0], bf16hi(u.x) + acc[1][0]);
                        w.y = pack_bf16x2(bf16lo(u.y) + acc[2][0], bf16hi(u.y) + acc[3][0]);
                        w.z = pack_bf16x2(bf16lo(u.z) + acc[0][1], bf16hi(u.z) + acc[1][1]);
                        w.w = pack_bf16x2(bf16lo(u.w) + acc[2][1], bf16hi(u.w) + acc[3][1]);
                        *(uint4 *)(p.y + yrow0 + o) = w;
                    }
                    if (r1ok) {
                        const uint4 u = yv[i][1];
                        uint4 w;
                        w.x = pack_bf16x2(bf16lo(u.x) + acc[0][2], bf16hi(u.x) + acc[1][2]);
                        w.y = pack_bf16x2(bf16lo(u.y) + acc[2][2], bf16hi(u.y) + acc[3][2]);
                        w.z = pack_bf16x2(bf16lo(u.z) + acc[0][3], bf16hi(u.z) + acc[1][3]);
                        w.w = pack_bf16x2(bf16lo(u.w) + acc[2][3], bf16hi(u.w) + acc[3][3]);
                        *(uint4 *)(p.y + yrow1 + o) = w;
                    }
                }
            }
        }
        cluster_wait();  // the peers have read this CTA's P: it may be overwritten, or the CTA may exit
    }
}

struct FPlan {
    int CS = 0, MINB = 1, KSX = 1, GMAX = 3, HC = 0, NCH = 0, OB = 0, BR = 16, kgb = 1;
    size_t box_bytes = 0, off_x = 0, off_p = 0, off_v = 0, v_bytes = 0, smem = 0;
    int pp = 0, vp = 0;
};

size_t f128(size_t x) { return (x + 127) & ~(size_t)127; }
size_t f1k(size_t x) { return (x + 1023) & ~(size_t)1023; }

bool fused_layout(const lora_pool_t *pool, int CS, int MINB, FPlan *pl) {
    const lora_pool_desc_t &d = pool->desc;
    const int ns = d.n_slices, R = d.max_rank, R8 = lora_round8(R);
    int out_total = 0;
    for (int j = 0; j < ns; ++j) out_total += d.out_dims[j];
    FPlan f;
    f.CS = CS;
    f.MINB = MINB;
    f.KSX = R8 <= 16 ? 1 : R8 <= 32 ? 2 : 4;
    f.GMAX = std::max(1, (MINB == 2 ? 3 : 6) / f.KSX);
    f.BR = R8 < 16 ? R8 : 16;
    f.kgb = (R + f.BR - 1) / f.BR;
    // hidden chunks and output blocks in multiples of 64 columns
    f.HC = (int)(((lora_ceil_div(d.in_dim, CS) + 63) / 64) * 64);
    f.NCH = f.HC / 64;
    f.OB = (int)(((lora_ceil_div(out_total, CS) + 63) / 64) * 64);
    if (f.NCH > 256 || lora_ceil_div(f.OB / 32, kFWarps) > f.GMAX) return false;
    f.box_bytes = (size_t)f.BR * f.NCH * 128;
    f.off_x = f1k((size_t)ns * f.kgb * f.box_bytes);
    f.off_p = f.off_x + f1k((size_t)f.NCH * kNT * 128);
    f.pp = ns * f.kgb * 16 + 4;
    f.off_v = f.off_p + f128((size_t)kNT * f.pp * 4);
    f.vp = ns * ((R + 15) & ~15) + 8;
    f.v_bytes = f128((size_t)kNT * f.vp * 2);
    f.smem = f.off_v + 2 * f.v_bytes + 1024;  // + alignment slack of the dynamic base
    if (f.smem > (size_t)(MINB == 2 ? kSmem2 : kSmem1)) return false;
    *pl = f;
    return true;
}

typedef void (*FusedFn)(FArgs);

FusedFn fused_fn(int KSX, int MINB) {
    // GMAX = max(1, (MINB == 2 ? 3 : 6) / KSX), as fused_layout sizes the plan
    if (MINB == 2) return KSX == 1 ? bgmv_fused_kernel<1, 3, 2> : KSX == 2 ? bgmv_fused_kernel<2, 1, 2>
                                                                            : bgmv_fused_kernel<4, 1, 2>;
    return KSX == 1 ? bgmv_fused_kernel<1, 6, 1> : KSX == 2 ? bgmv_fused_kernel<2, 3, 1>
                                                           : bgmv_fused_kernel<4, 1, 1>;
}

std::atomic<int> g_fused_configured[64];

}  // namespace

// Whether the fused decode kernel takes this batch, and its cluster size.
// It needs a dense pool of modest rank with a hidden size in 64-column
// chunks, one wave of clusters (one per slot), and a batch that keeps most
// slots busy (the prologue fetches every enabled slot's weights before the
// batch is known).
static bool fused_plan(const lora_pool_t *pool, int T, FPlan *pl) {
    const lora_pool_desc_t &d = pool->desc;
    if (pool->is_moe || d.max_rank > 64 || d.in_dim % 64) return false;
    // the expand works in groups of 32 outputs that stay inside one slice
    for (int j = 0; j < d.n_slices; ++j)
        if (d.out_dims[j] % 32) return false;
    if (d.n_slices * ((d.max_rank + 15) & ~15) > 8 * 16) return false;
    const int L = d.max_loras;
    // a few rows per slot: past 16 on average a slot's cluster runs its chain
    // of dependent steps once per 16-row tile, and the split kernels, which
    // spread the tiles over the whole GPU, are faster (the Inkling sink-expert
    // layers, 32 rows per slot: 40.9 against 33.0 us per step)
    // (kernel policy 7 keeps the kernel up to 32 rows per slot, for tests)
    const int per_slot = g_lora_kernel_policy == 7 ? 32 : 16;
    if (T <= 0 || T > kMaxT || T < 4 * L || T > per_slot * L) return false;
    // the widest cluster whose CTAs all fit one wave, two per SM first
    for (int CS = 8; CS >= 1; CS >>= 1)
        for (int MINB = 2; MINB >= 1; --MINB) {
            if ((long long)L * CS > (long long)MINB * pool->num_sms) continue;
            if (fused_layout(pool, CS, MINB, pl)) return true;
        }
    return false;
}

bool lora_fused_eligible(const lora_pool_t *pool, int T) {
    FPlan pl;
    return fused_plan(pool, T, &pl);
}

lora_status_t lora_fused_apply(const lora_pool_t *pool, const lora_meta_t *meta, const int32_t *d_idx, int32_t T,
                               const void *x, int64_t ldx, void *y, int64_t ldy, float post_scale, int spin_limit,
                               cudaStream_t s, bool *launched) {
    *launched = false;
    FPlan pl;
    if (!fused_plan(pool, T, &pl)) return LORA_OK;
    const lora_pool_desc_t &d = pool->desc;
    const int meta_steps = (T + kFThreads - 1) / kFThreads;
    if (d_idx) {
        // batch mode: the metadata is built by one CTA (a key per thread)
        if (d.max_loras + 1 > kFThreads || meta_steps > kMaxSteps ||
            dense_meta_smem_bytes(kFThreads, meta_steps, d.max_loras) + 1024 > pl.smem)
            return LORA_OK;
    }
    FArgs a;
    memset(&a, 0, sizeof(a));
    a.n_slices = d.n_slices;
    a.H = d.in_dim;
    a.R = d.max_rank;
    int off = 0;
    for (int j = 0; j < d.n_slices; ++j) {
        // A_j of every slot as one [L*R][H] matrix (a dense pool has one expert)
        if (!lora_make_tmap_a_chunks(&a.tm_a[j], pool->A[j], (long long)d.max_loras * d.max_rank, d.in_dim, pl.BR,
                                     pl.NCH))
            return LORA_OK;  // no tensor maps here: the other kernels take the batch
        a.out_off[j] = off;
        off += d.out_dims[j];
        a.B[j] = pool->B[j];
        a.B_ss[j] = pool->b_slot_elems[j];
    }
    FusedFn fn = fused_fn(pl.KSX, pl.MINB);
    const int dev = pool->device < 64 ? pool->device : 63;
    if (!g_fused_configured[dev].load(std::memory_order_acquire)) {
        const FusedFn all[] = {bgmv_fused_kernel<1, 3, 2>, bgmv_fused_kernel<2, 1, 2>, bgmv_fused_kernel<4, 1, 2>,
                               bgmv_fused_kernel<1, 6, 1>, bgmv_fused_kernel<2, 3, 1>, bgmv_fused_kernel<4, 1, 1>};
        int optin = 0;
        LORA_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, pool->device));
        for (FusedFn f : all) {
            // the static shared memory counts against the opt-in limit too
            cudaFuncAttributes fa;
            LORA_CUDA_TRY(cudaFuncGetAttributes(&fa, f));
            const int dyn = std::min(kSmem1, optin - (int)fa.sharedSizeBytes);
            LORA_CUDA_TRY(cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn));
        }
        g_fused_configured[dev].store(1, std::memory_order_release);
    }
    a.out_total = off;
    a.CS = pl.CS;
    a.HC = pl.HC;
    a.NCH = pl.NCH;
    a.OB = pl.OB;
    a.T = T;
    a.L = d.max_loras;
    a.BR = pl.BR;
    a.kgb = pl.kgb;
    a.rank = pool->d_rank;
    a.enabled = pool->d_enabled;
    a.scale = pool->d_scale;
    a.key_count = meta->key_count;
    a.key_offset = meta->key_offset;
    a.sorted = meta->sorted;
    if (d_idx) {
        a.idx = d_idx;
        a.idx_mode = 1;
        a.meta_steps = meta_steps;
        a.ma.idx = d_idx;
        a.ma.rank = pool->d_rank;
        a.ma.enabled = pool->d_enabled;
        a.ma.status = pool->d_status;
        a.ma.T = T;
        a.ma.K = 1;
        a.ma.E = 1;
        a.ma.L = d.max_loras;
        a.ma.n_keys = d.max_loras;
        a.ma.m = *meta;
    }
    a.x = (const uint16_t *)x;
    a.ldx = ldx;
    a.y = (uint16_t *)y;
    a.ldy = ldy;
    a.post_scale = post_scale;
    a.box_bytes = (int)pl.box_bytes;
    a.off_x = (int)pl.off_x;
    a.off_p = (int)pl.off_p;
    a.off_v = (int)pl.off_v;
    a.pp = pl.pp;
    a.vp = pl.vp;
    a.v_bytes = (int)pl.v_bytes;
    a.status = pool->d_status;
    a.spin_limit = spin_limit;

    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)((d.max_loras + (d_idx ? 1 : 0)) * pl.CS), 1, 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = pl.CS;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, fn, a));
    lora_note_launch();
    *launched = true;
    return LORA_OK;
}
