// Cluster BGMV: the multi-tenant LoRA delta for small row groups (decode
// tokens, MoE (adapter, expert) groups) in one pass, one thread-block
// cluster of 1, 2, 4 or 8 CTAs per tile of <= 16 rows of one group.
//
// The vLLM LoRA layer pages compute it as add_shrink into a zeroed fp32
// buffer [n_slices][T][rank] and add_expand with add_input=True at the slice
// offsets; add_lora_fused_moe does the same per (adapter, expert) group.
// Here the fp32 intermediate never leaves the chip:
//   CTA c of the cluster owns hidden range c and output range c.
//   1. bulk copies (cp.async.bulk, mbarrier transaction counts) bring the
//      tile's x rows and the slot's A rows for hidden range c into shared
//      memory (<= 2 stages in flight), and the slot's B rows for output range c
//   2. partial v[t][j][k] over hidden range c: m16n8k16 bf16 tensor-core
//      MMAs (tokens x rank rows x hidden), fragments from ldmatrix, fp32
//      accumulation; meanwhile the tile's y rows of output range c are
//      bulk-copied into the freed stage buffers
//   3. cluster barrier; every CTA sums the partials of its peers through
//      distributed shared memory, scales by scale[a] (and the routed weight
//      for MoE w2), and splits v into bf16 hi + lo parts so the expand keeps
//      the fp32 intermediate to ~16 bits
//   4. y[t][o] += v_hi[t] . B[o] + v_lo[t] . B[o] for o in output range c
//      (MMAs) in shared memory, then bulk copies write the rows back
// The cluster size is picked per layer so that each CTA moves ~96 KB.
// Launched with programmatic stream serialization so it starts while the
// metadata kernel finishes; griddepcontrol.wait orders its metadata reads.
#include <string.h>

#include <atomic>

#include "lora_internal.cuh"
#include "mma_common.cuh"

namespace {

using namespace bgmv;

constexpr int kMaxCS = 8;  // CTAs per tile (cluster size) is 1, 2, 4 or 8
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileRows = LORA_TILE_ROWS;
constexpr int kMaxHSplit = 4;  // hidden-range split of the shrink across warps

struct CArgs {
    int n_slices, in_dim, E, row_div, R, R8, out_total;
    int out_w[LORA_MAX_SLICES], out_off[LORA_MAX_SLICES];
    const uint16_t *A[LORA_MAX_SLICES];
    long long A_ss[LORA_MAX_SLICES], A_es[LORA_MAX_SLICES];
    const uint16_t *B[LORA_MAX_SLICES];
    long long B_ss[LORA_MAX_SLICES];
    int B_shared[LORA_MAX_SLICES];
    const int32_t *rank;
    const float *scale;
    const int32_t *sorted, *tile_row0, *tile_keyn, *counters;
    int count_idx;
    const uint16_t *in;
    long long ld_in;
    uint16_t *out;
    long long ld_out;
    const float *row_w;
    int CS, HCc, OCc, SC;
    int xs_stride, as_stride, vr_stride, ys_stride;  // elements
    int off_x, off_a, off_b, off_vp, off_ys, off_vsum, off_vh, off_vl, x_stage_bytes, a_stage_bytes;
    int *status;
    int spin_limit;
    float post_scale;  // extra factor on every delta (lm_head muP); 1 otherwise
};

// Issue the copies of hidden sub-chunk s into stage buffer (s & 1) by warp 0.
__device__ __forceinline__ void issue_stage(const CArgs &p, char *smem, uint64_t *full, int s, int hb,
                                            int he, int n, int r, const int *rows, const uint16_t *const *Ab,
                                            int lane) {
    const int h0 = hb + s * p.SC;
    const int len = min(p.SC, he - h0);
    const int st = s & 1;
    uint16_t *xs = (uint16_t *)(smem + p.off_x + st * p.x_stage_bytes);
    uint16_t *as = (uint16_t *)(smem + p.off_a + st * p.a_stage_bytes);
    const uint32_t rowb = (uint32_t)len * 2;
    const int nA = p.n_slices * r;
    if (lane == 0) mbar_expect_tx(&full[st], rowb * (uint32_t)(n + nA));
    __syncwarp();
    for (int i = lane; i < n + nA; i += 32) {
        if (i < n) {
            const uint16_t *src = p.in + (long long)(rows[i] / p.row_div) * p.ld_in + h0;
            bulk_g2s(xs + i * p.xs_stride, src, rowb, &full[st]);
        } else {
            const int q = i - n, j = q / r, k = q - j * r;
            bulk_g2s(as + q * p.as_stride, Ab[j] + (long long)k * p.in_dim + h0, rowb, &full[st]);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) cluster_lora_kernel(const __grid_constant__ CArgs p) {
    extern __shared__ __align__(128) char smem[];
    __shared__ __align__(8) uint64_t full[2];
    __shared__ __align__(8) uint64_t bbar, ybar;
    __shared__ int s_rows[kTileRows];
    __shared__ const uint16_t *s_Ab[LORA_MAX_SLICES];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c4 = lane & 3;
    const int tile = blockIdx.x / p.CS;
    const uint32_t crank = cluster_rank();

    asm volatile("griddepcontrol.wait;" ::: "memory");
    // one round trip: the tile entries are read before the count check (the
    // list has max_tiles entries, so the reads stay inside the buffer)
    const int n_tiles = p.counters[p.count_idx];
    const int row0 = p.tile_row0[tile];
    const int keyn = p.tile_keyn[tile];
    if (tile >= n_tiles) return;  // the whole cluster leaves together

    const int n = keyn & 31, key = keyn >> 5;
    const int a = key / p.E, e = key - a * p.E;
    const int r = p.rank[a];
    const float sc = p.scale[a];
    const int rs = (r + 7) & ~7;
    const int ns = p.n_slices;
    const int nrows = ns * r;  // rank rows of the tile, packed (j, k) -> j * r + k
    const int JK = ns * p.R8;  // width of the v rows, (j, k) -> j * R8 + k

    const int hb = min(p.in_dim, (int)crank * p.HCc);
    const int he = min(p.in_dim, hb + p.HCc);
    const int ob = min(p.out_total, (int)crank * p.OCc);
    const int oe = min(p.out_total, ob + p.OCc);
    const int n_sub = (he - hb + p.SC - 1) / p.SC;

    if (tid < n) s_rows[tid] = p.sorted[row0 + tid];
    if (tid < ns) s_Ab[tid] = p.A[tid] + (long long)a * p.A_ss[tid] + (long long)e * p.A_es[tid];
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&bbar, 1);
        mbar_init(&ybar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ---- issue every copy that does not wait for a stage to drain
    if (warp == 0) {
        for (int s = 0; s < min(n_sub, 2); ++s) issue_stage(p, smem, full, s, hb, he, n, r, s_rows, s_Ab, lane);
    }

    const int nob = (oe - ob) >> 3;  // output blocks of 8 columns

    // ---- partial shrink over this CTA's hidden range (tensor-core MMAs)
    // units: (n-block of 8 rank rows, hidden split); every warp owns <= 2 units
    const int nnb = (nrows + 7) >> 3;
    int hsplit = 1;
    while (nnb * hsplit * 2 <= 2 * kWarps && hsplit < kMaxHSplit) hsplit *= 2;
    const int units = nnb * hsplit;
    float acc[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[u][i] = 0.f;
    // after the shrink the stage buffers hold the y tile and the partials
    uint16_t *ys = (uint16_t *)(smem + p.off_ys);  // [16][ys_stride] y rows of [ob, oe)
    float *vp = (float *)(smem + p.off_vp);        // [hsplit][16][JK]

    for (int s = 0; s < n_sub; ++s) {
        const int st = s & 1;
        mbar_wait(&full[st], (uint32_t)((s >> 1) & 1), p.spin_limit, p.status);
        const int len = min(p.SC, he - hb - s * p.SC);
        const int steps = (len + 15) >> 4;
        const uint16_t *xs = (const uint16_t *)(smem + p.off_x + st * p.x_stage_bytes);
        const uint16_t *as = (const uint16_t *)(smem + p.off_a + st * p.a_stage_bytes);
#pragma unroll
        for (int ui = 0; ui < 2; ++ui) {
            const int u = warp + ui * kWarps;
            if (u < units) {
                const int nb = u / hsplit, hs = u - nb * hsplit;
                for (int i = hs; i < steps; i += hsplit) {
                    const int k0 = i * 16;
                    uint32_t a0, a1, a2, a3, b0, b1;
                    ldsm_x4(xs + ((lane & 7) + ((lane >> 3) & 1) * 8) * p.xs_stride + k0 + (lane >> 4) * 8,
                            a0, a1, a2, a3);
                    ldsm_x2(as + (nb * 8 + (lane & 7)) * p.as_stride + k0 + ((lane >> 3) & 1) * 8, b0, b1);
                    if (k0 + 8 >= len) a2 = a3 = b1 = 0u;  // half step: only k0..k0+7 exist
                    mma16816(acc[ui], a0, a1, a2, a3, b0, b1);
                }
            }
        }
        __syncthreads();  // every thread is done with stage buffer st
        if (warp == 0 && s + 2 < n_sub) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_stage(p, smem, full, s + 2, hb, he, n, r, s_rows, s_Ab, lane);
        }
    }
    // stage buffers are free: bring the y rows of this CTA's output range in
    if (warp == 0) {
        const uint32_t rowb = oe > ob ? (uint32_t)(oe - ob) * 2 : 0;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) mbar_expect_tx(&ybar, rowb * (uint32_t)n);
        __syncwarp();
        if (lane < n && rowb)
            bulk_g2s(ys + lane * p.ys_stride, p.out + (long long)s_rows[lane] * p.ld_out + ob, rowb, &ybar);
    } else if (warp == 1) {
        // B rows of output range [ob, oe), slice by slice, compact rows of rs
        uint16_t *bsw = (uint16_t *)(smem + p.off_b);
        const uint32_t total = oe > ob ? (uint32_t)(oe - ob) * rs * 2 : 0;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) mbar_expect_tx(&bbar, total);
        __syncwarp();
        if (lane < ns) {
            const int j = lane;
            const int s0 = max(ob, p.out_off[j]), s1 = min(oe, p.out_off[j] + p.out_w[j]);
            if (s1 > s0) {
                const uint16_t *Bj = p.B[j] + (long long)a * p.B_ss[j] +
                                     (p.B_shared[j] ? 0ll : (long long)e * p.out_w[j] * rs);
                bulk_g2s(bsw + (long long)(s0 - ob) * rs, Bj + (long long)(s0 - p.out_off[j]) * rs,
                         (uint32_t)(s1 - s0) * rs * 2, &bbar);
            }
        }
    }
    for (int i = tid; i < hsplit * kTileRows * JK; i += kThreads) vp[i] = 0.f;
    __syncthreads();
    // fragment (row t, rank row q): d0 (g, 2c4), d1 (g, 2c4+1), d2 (g+8, 2c4), d3 (g+8, 2c4+1)
#pragma unroll
    for (int ui = 0; ui < 2; ++ui) {
        const int u = warp + ui * kWarps;
        if (u < units) {
            const int nb = u / hsplit, hs = u - nb * hsplit;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int q = nb * 8 + 2 * c4 + h;
                if (q < nrows) {
                    const int j = q / r, k = q - j * r;
                    float *dst = vp + (hs * kTileRows) * JK + j * p.R8 + k;
                    if (g < n) dst[g * JK] = acc[ui][h];
                    if (g + 8 < n) dst[(g + 8) * JK] = acc[ui][2 + h];
                }
            }
        }
    }
    __syncthreads();
    float *vsum = (float *)(smem + p.off_vsum);  // [16][JK]: this CTA's partial, read by its peers
    for (int i = tid; i < kTileRows * JK; i += kThreads) {
        float s = 0.f;
        for (int hs = 0; hs < hsplit; ++hs) s += vp[hs * kTileRows * JK + i];
        vsum[i] = s;
    }

    // ---- cluster reduction through distributed shared memory
    cluster_arrive();
    cluster_wait();
    uint16_t *vh = (uint16_t *)(smem + p.off_vh);  // [16][vr_stride] bf16 hi part
    uint16_t *vl = (uint16_t *)(smem + p.off_vl);  // [16][vr_stride] bf16 lo part
    {
        const int per_t = JK / 4;
        for (int i = tid; i < kTileRows * per_t; i += kThreads) {
            const int t = i / per_t, q = i - t * per_t;
            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < n) {
                const float *src = vsum + t * JK + q * 4;
                float4 v[kMaxCS];
#pragma unroll
                for (int cc = 0; cc < kMaxCS; ++cc)
                    v[cc] = cc < p.CS ? ld_dsmem_f32x4(src, (uint32_t)cc) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int cc = 0; cc < kMaxCS; ++cc) {
                    s4.x += v[cc].x;
                    s4.y += v[cc].y;
                    s4.z += v[cc].z;
                    s4.w += v[cc].w;
                }
                float w = sc * p.post_scale;
                if (p.row_w) w *= p.row_w[s_rows[t]];
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
            *(uint2 *)(vh + t * p.vr_stride + q * 4) = hv;
            *(uint2 *)(vl + t * p.vr_stride + q * 4) = lv;
        }
    }
    cluster_arrive();  // done reading peers; the matching wait comes before exit
    __syncthreads();

    // ---- expand over this CTA's output range (tensor-core MMAs)
    mbar_wait(&bbar, 0, p.spin_limit, p.status);
    const uint16_t *bs = (const uint16_t *)(smem + p.off_b);
    const int ksteps = (rs + 15) >> 4;
    mbar_wait(&ybar, 0, p.spin_limit, p.status);
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll 1
    for (int ob8 = warp; ob8 < nob; ob8 += kWarps) {
        const int o0 = ob + ob8 * 8;
        int j = 0;
        while (j + 1 < ns && o0 >= p.out_off[j + 1]) ++j;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        for (int ks = 0; ks < ksteps; ++ks) {
            const int k0 = ks * 16;
            uint32_t h0, h1, h2, h3, l0, l1, l2, l3, b0, b1;
            const int acol = j * p.R8 + k0 + (lane >> 4) * 8;
            ldsm_x4(vh + arow * p.vr_stride + acol, h0, h1, h2, h3);
            ldsm_x4(vl + arow * p.vr_stride + acol, l0, l1, l2, l3);
            ldsm_x2(bs + (ob8 * 8 + (lane & 7)) * rs + k0 + ((lane >> 3) & 1) * 8, b0, b1);
            if (k0 + 8 >= rs) h2 = h3 = l2 = l3 = b1 = 0u;
            mma16816(d, h0, h1, h2, h3, b0, b1);
            mma16816(d, l0, l1, l2, l3, b0, b1);
        }
        const int oc = ob8 * 8 + 2 * c4;  // column inside the y tile
        if (g < n) {
            uint32_t *yp = (uint32_t *)(ys + g * p.ys_stride + oc);
            const uint32_t u = *yp;
            *yp = pack_bf16x2(bf16lo(u) + d[0], bf16hi(u) + d[1]);
        }
        if (g + 8 < n) {
            uint32_t *yp = (uint32_t *)(ys + (g + 8) * p.ys_stride + oc);
            const uint32_t u = *yp;
            *yp = pack_bf16x2(bf16lo(u) + d[2], bf16hi(u) + d[3]);
        }
    }
    // write the updated rows back with bulk copies
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        const uint32_t rowb = oe > ob ? (uint32_t)(oe - ob) * 2 : 0;
        if (lane < n && rowb) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             p.out + (long long)s_rows[lane] * p.ld_out + ob),
                         "r"(smem_u32(ys + lane * p.ys_stride)), "r"(rowb)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
    }
    // the next kernel in the stream may start its prologue; it still waits
    // for this grid to finish before touching memory
    asm volatile("griddepcontrol.launch_dependents;");
    cluster_wait();  // peers may still read this CTA's partials until here
}

}  // namespace

namespace {

size_t align128(size_t x) { return (x + 127) & ~(size_t)127; }

struct CPlan {
    bool ok;
    int CS, HCc, OCc, SC, n_stage, hsplit_max, xs_stride, as_stride, vr_stride, ys_stride;
    int off_x, off_a, off_b, off_vp, off_ys, off_vsum, off_vh, off_vl, x_stage_bytes, a_stage_bytes;
    size_t smem;
};

constexpr size_t kBudget2 = 110 * 1024;  // two CTAs per SM
constexpr size_t kBudget1 = 220 * 1024;  // one CTA per SM

CPlan make_cplan(int ns, int in_dim, int out_total, int R, int CS) {
    CPlan c;
    memset(&c, 0, sizeof(c));
    const int R8 = lora_round8(R);
    const int JK = ns * R8;
    if (ns * R > 128) return c;  // <= 16 n-blocks of rank rows: two per warp
    c.CS = CS;
    c.HCc = ((lora_ceil_div(in_dim, CS) + 15) / 16) * 16;
    c.OCc = lora_round8(lora_ceil_div(out_total, CS));
    c.hsplit_max = kMaxHSplit;  // a tile of lower rank has fewer n-blocks and may split more
    c.vr_stride = JK + 8;
    c.ys_stride = c.OCc + 8;
    const size_t b_bytes = align128((size_t)c.OCc * R8 * 2 + 32);
    const size_t vp_bytes = align128((size_t)c.hsplit_max * kTileRows * JK * 4);
    const size_t ys_bytes = align128((size_t)kTileRows * c.ys_stride * 2);
    const size_t vsum_bytes = align128((size_t)kTileRows * JK * 4);
    const size_t vh_bytes = align128((size_t)kTileRows * c.vr_stride * 2);
    const size_t fixed = vsum_bytes + 2 * vh_bytes;
    const int arows = lora_round8(ns * R);
    const size_t per_elem = (size_t)(kTileRows + arows) * 2;  // x rows + A rows, one stage
    const size_t budgets[2] = {kBudget2, kBudget1};
    const int min_sc[2] = {c.HCc < 256 ? c.HCc : 256, c.HCc < 64 ? c.HCc : 64};
    for (int bi = 0; bi < 2; ++bi) {
        if (budgets[bi] <= fixed + 2 * 16 * per_elem) continue;
        long long sc = (long long)((budgets[bi] - fixed) / (2 * per_elem)) - 8;
        sc = sc >= 64 ? (sc / 64) * 64 : (sc / 16) * 16;
        if (sc > c.HCc) sc = c.HCc;
        if (sc < min_sc[bi] || sc < 16) continue;
        c.SC = (int)sc;
        const int n_sub = lora_ceil_div(c.HCc, c.SC);
        c.n_stage = n_sub < 2 ? 1 : 2;
        c.xs_stride = c.SC + 8;
        c.as_stride = c.SC + 8;
        c.x_stage_bytes = (int)align128((size_t)kTileRows * c.xs_stride * 2);
        c.a_stage_bytes = (int)align128((size_t)arows * c.as_stride * 2);
        // the y tile, the partials and the slot's B rows reuse the stage
        // buffers after the shrink
        size_t stage_region = (size_t)c.n_stage * (c.x_stage_bytes + c.a_stage_bytes);
        if (stage_region < ys_bytes + vp_bytes + b_bytes) stage_region = ys_bytes + vp_bytes + b_bytes;
        c.off_x = 0;
        c.off_a = c.n_stage * c.x_stage_bytes;
        c.off_ys = 0;
        c.off_vp = (int)ys_bytes;
        c.off_b = (int)(ys_bytes + vp_bytes);
        c.off_vsum = (int)stage_region;
        c.off_vh = c.off_vsum + (int)vsum_bytes;
        c.off_vl = c.off_vh + (int)vh_bytes;
        c.smem = (size_t)c.off_vl + vh_bytes;
        c.ok = c.smem <= budgets[bi];
        if (c.ok) return c;
    }
    c.ok = false;
    return c;
}

std::atomic<int> g_cluster_configured[64];

}  // namespace

lora_status_t lora_cluster_apply(const lora_pool_t *pool, const LoraProblem &pr, cudaStream_t s,
                                 bool *launched) {
    *launched = false;
    int out_total = 0;
    for (int j = 0; j < pr.n_slices; ++j) out_total = max(out_total, pr.out_off[j] + pr.out_w[j]);
    // CTAs per tile: enough that each moves ~96 KB of a full-rank tile (weights,
    // x rows and y rows), and the smallest such cluster whose plan fits
    const double tile_bytes = 2.0 * ((double)pr.n_slices * pr.R * pr.in_dim + kTileRows * (double)pr.in_dim +
                                     (double)out_total * pr.R + 2.0 * kTileRows * out_total);
    int CS = 1;
    while (CS < kMaxCS && tile_bytes / CS > 96.0 * 1024) CS *= 2;
    CPlan cp = make_cplan(pr.n_slices, pr.in_dim, out_total, pr.R, CS);
    while (!cp.ok && CS < kMaxCS) {
        CS *= 2;
        cp = make_cplan(pr.n_slices, pr.in_dim, out_total, pr.R, CS);
    }
    if (!cp.ok) return LORA_OK;
    CArgs a;
    memset(&a, 0, sizeof(a));
    a.n_slices = pr.n_slices;
    a.in_dim = pr.in_dim;
    a.E = pr.E;
    a.row_div = pr.row_div;
    a.R = pr.R;
    a.R8 = lora_round8(pr.R);
    a.out_total = out_total;
    for (int j = 0; j < pr.n_slices; ++j) {
        a.out_w[j] = pr.out_w[j];
        a.out_off[j] = pr.out_off[j];
        a.A[j] = pr.A[j];
        a.A_ss[j] = pr.A_ss[j];
        a.A_es[j] = pr.A_es[j];
        a.B[j] = pr.B[j];
        a.B_ss[j] = pr.B_ss[j];
        a.B_shared[j] = pr.B_shared[j];
    }
    a.rank = pr.rank;
    a.scale = pr.scale;
    a.sorted = pr.meta->sorted;
    a.tile_row0 = pr.tile_row0;
    a.tile_keyn = pr.tile_keyn;
    a.count_idx = pr.count_idx;
    a.counters = pr.meta->counters;
    a.in = pr.in;
    a.ld_in = pr.ld_in;
    a.out = pr.out;
    a.ld_out = pr.ld_out;
    a.row_w = pr.row_w;
    a.CS = cp.CS;
    a.HCc = cp.HCc;
    a.OCc = cp.OCc;
    a.SC = cp.SC;
    a.xs_stride = cp.xs_stride;
    a.as_stride = cp.as_stride;
    a.vr_stride = cp.vr_stride;
    a.ys_stride = cp.ys_stride;
    a.off_ys = cp.off_ys;
    a.off_x = cp.off_x;
    a.off_a = cp.off_a;
    a.off_b = cp.off_b;
    a.off_vp = cp.off_vp;
    a.off_vsum = cp.off_vsum;
    a.off_vh = cp.off_vh;
    a.off_vl = cp.off_vl;
    a.x_stage_bytes = cp.x_stage_bytes;
    a.a_stage_bytes = cp.a_stage_bytes;
    a.status = pr.status;
    a.spin_limit = pr.spin_limit;
    a.post_scale = pr.post_scale;

    const int dev = pool->device < 64 ? pool->device : 63;
    if (!g_cluster_configured[dev].load(std::memory_order_acquire)) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(cluster_lora_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kBudget1));
        g_cluster_configured[dev].store(1, std::memory_order_release);
    }
    const long long max_tiles = pr.rows / kTileRows + (pr.rows < pr.n_keys ? pr.rows : pr.n_keys);
    if (max_tiles <= 0) {
        *launched = true;
        return LORA_OK;
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(max_tiles * cp.CS), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = cp.smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cp.CS;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, cluster_lora_kernel, a));
    lora_note_launch();
    *launched = true;
    return LORA_OK;
}
