// The full LoRA linear layer (vLLM LoRA layer pages, BaseLinearLayerWithLoRA
// and ColumnParallelLinearWithLoRA.apply: the base layer's output, then the
// LoRA delta added in place with add_shrink / add_expand):
//   y[t][o] = sum_h x[t][h] W[o][h] + bias[o] + scale[a_t] * sum_k v[t][k] B_j[a_t][o][k]
//   v[t][k] = sum_h x[t][h] A_j[a_t][k][h]        (slice j holds output o)
//
// Here the delta is part of the base GEMM's accumulation, so y is written
// once.  The contraction over the rank is run on the tensor cores as extra
// K blocks of the same accumulator: for a tile of 128 tokens, the distinct
// adapter slots of its tokens are packed pg = 64 / Rw to a "delta block"
// (Rw = max_rank rounded up to 8, 16, 32 or 64).  Delta block g holds
//   Vhat[t][p*Rw + k] = scale[a_t] * v[t][k]   if a_t is slot p of group g, else 0
//   Bhat[o][p*Rw + k] = B_j[slot p of group g][o][k]   (0 past the slot's rank)
// so that Vhat . Bhat^T adds exactly the delta of the group's tokens.  The
// delta blocks are spread through the K-block sequence (see kb_kind), so
// that building them overlaps the base GEMM.
//
// Kernels: linear_slot_kernel writes each token's slot and sorted position
// from the batch metadata; the split shrink (or, when it does not take the
// pool, the atomic one) writes x A^T in fp32, unscaled; linear_lora_kernel is a
// persistent tcgen05 GEMM over (128-token, BN-output) tiles with a TMA ring
// for x and W, a second ring producer that writes the delta blocks, two
// TMEM accumulators (the epilogue of one tile runs under the next tile's
// MMAs), and an epilogue that adds the bias and stores bf16 y.
//
// Warp roles of linear_lora_kernel (320 threads):
//   warp 0     TMA producer of the base K blocks (x tile 128 x 64, W tile BN x 64)
//   warp 1     TMEM allocation and the MMA issue (one thread)
//   warps 2-5  epilogue: TMEM -> registers, + bias, bf16, stores to y
//   warps 6-9  delta blocks: the tile's distinct slots, Vhat and Bhat written
//              into the ring stage in the 128-byte swizzled layout
// Every wait is a bounded poll that records LORA_ERR_TIMEOUT in the status word.
//
// This kernel runs under kernel policy 6 for pools whose shape it takes
// (max_rank <= 64, every slice width a multiple of 128).  Otherwise the base
// GEMM is a cuBLASLt call and the delta a second pass over y (the
// library's apply), which measured faster on GB300 for both the decode
// (T=256, 4096 -> 6144) and the prefill (8K tokens, 4096 -> 28672) layers:
// with one 128 x 128 or 128 x 256 tile per CTA this kernel is bound by the
// latency of its operand stream (decode) and by L2 bandwidth (prefill), where
// the library GEMM pairs two SMs on each tile.
#include <cublasLt.h>
#include <string.h>

#include <atomic>

#include "lora_internal.cuh"
#include "tc_common.cuh"

namespace {

constexpr int kLM = 128;                        // tokens per tile: MMA M, TMEM lanes
constexpr int kLBK = 64;                        // K elements per block: one 128-byte swizzle row
constexpr int kLThreads = 320;
constexpr int kFill0 = 6;                       // first delta-block warp
constexpr uint32_t kXBytes = kLM * kLBK * 2;    // 16 KB x tile (or Vhat)
constexpr int kRingBytes = 192 * 1024;
constexpr int kSlotThreads = 128;

struct LinArgs {
    CUtensorMap tm_x, tm_w;
    int T, O, KB, G, n_mt, n_tiles;
    int n_slices;
    int out_off[LORA_MAX_SLICES + 1];
    const uint16_t *B[LORA_MAX_SLICES];
    long long B_ss[LORA_MAX_SLICES];
    int R, Rw, pg;                // max_rank; slot segment width; slots per delta block
    const float *part;            // shrink sums [nc][n_slices][T][r8] fp32, unscaled
    int nc, r8, sorted_rows;      // sorted_rows: row i of part is the metadata's sorted row i
    const int32_t *slot_of;       // [T], -1 for a token without an active adapter
    const int32_t *pos_of;        // [T], sorted position of each token
    const int32_t *rank;
    const float *scale;
    const uint16_t *bias;         // [O] or null
    int bias_vec;                 // bias 16-byte aligned
    uint16_t *y;
    long long ldy;
    int *status;
    int spin_limit;
};

// Position kb of a tile's K-block sequence: a base block (>= 0) or delta
// group -(g + 1).  The first delta group comes after F = min(KB, 12) base
// blocks (time for the delta warps to find the tile's slots), the next ones
// after every sp more base blocks while base blocks remain, the rest at the end.
__host__ __device__ __forceinline__ int kb_kind(int kb, int KB, int G) {
    const int F = KB < 12 ? KB : 12;
    if (kb < F) return kb;
    const int sp = G > 0 && (KB - F) / G > 1 ? (KB - F) / G : 1;
    const int gi = G < (KB - F) / sp ? G : (KB - F) / sp;  // interleaved groups
    const int t = kb - F;
    if (t < gi * (sp + 1)) {
        const int q = t / (sp + 1), r = t - q * (sp + 1);
        return r == 0 ? -(q + 1) : F + q * sp + (r - 1);
    }
    const int rest = t - gi * (sp + 1), nb = KB - F - gi * sp;
    return rest < nb ? F + gi * sp + rest : -(gi + (rest - nb) + 1);
}

__device__ __forceinline__ void lwait(uint64_t *bar, uint32_t parity, const LinArgs &p) {
    if (!tc::mbar_wait(bar, parity, p.spin_limit)) atomicExch(p.status, (int)LORA_ERR_TIMEOUT);
}

// byte offset of 16-byte chunk c of row r in a 128-byte swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void fill_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *(const uint32_t *)&v;
}

// Each token's slot and sorted position from the metadata: group g's sorted
// rows get group_key[g], the inactive tail gets -1.
__global__ void __launch_bounds__(kSlotThreads) linear_slot_kernel(const int32_t *sorted, const int32_t *group_key,
                                                                   const int32_t *group_start,
                                                                   const int32_t *counters, int T, int max_groups,
                                                                   int32_t *slot_of, int32_t *pos_of) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_active = counters[0], n_groups = counters[1];
    for (int g = blockIdx.x; g <= max_groups; g += gridDim.x) {
        int i0, i1, val;
        if (g < max_groups) {
            if (g >= n_groups) continue;
            i0 = group_start[g];
            i1 = group_start[g + 1];
            val = group_key[g];
        } else {
            i0 = n_active;
            i1 = T;
            val = -1;
        }
        for (int i = i0 + (int)threadIdx.x; i < i1; i += kSlotThreads) {
            const int t = sorted[i];
            slot_of[t] = val;
            pos_of[t] = i;
        }
    }
    asm volatile("griddepcontrol.launch_dependents;");
}

template <int BN>
__global__ void __launch_bounds__(kLThreads, 1) linear_lora_kernel(const __grid_constant__ LinArgs p) {
    constexpr uint32_t kWBytes = BN * kLBK * 2;
    constexpr uint32_t kStage = kXBytes + kWBytes;
    // two rings: the base blocks (filled by TMA) and the delta blocks (written
    // by the delta warps), each with its own barriers, so that every producer
    // waits only for the consumption of its own previous fills
    constexpr int SD = 1;
    constexpr int SB = kRingBytes / kStage - SD;
    extern __shared__ __align__(1024) char smem_raw[];
    __shared__ __align__(8) uint64_t fullb[SB], emptyb[SB], fulld[SD], emptyd[SD], accf[2], acce[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_skip[SD];
    __shared__ int s_rowslot[kLM], s_uidx[kLM], s_uslot[kLM], s_urs[kLM], s_wcnt[4];
    char *smem = smem_raw + ((1024u - (smem_u32_of(smem_raw) & 1023u)) & 1023u);
    char *dring = smem + (size_t)SB * kStage;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 1) {
        tc::tmem_alloc(&s_tmem, 2 * BN);
        tc::tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < SB; ++s) {
            tc::mbar_init(&fullb[s], 1);
            tc::mbar_init(&emptyb[s], 1);
        }
        for (int s = 0; s < SD; ++s) {
            tc::mbar_init(&fulld[s], 1);
            tc::mbar_init(&emptyd[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&accf[b], 1);
            tc::mbar_init(&acce[b], 4);  // lane 0 of each epilogue warp
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int NKB = p.KB + p.G;

    if (warp == 0) {
        // ---- TMA producer: x and W are not written by the kernels before
        // this one in a step, so the loads start before the dependency wait
        if (lane == 0) {
            tc::prefetch_tmap(&p.tm_x);
            tc::prefetch_tmap(&p.tm_w);
            int gb = 0;
            for (int it = blockIdx.x; it < p.n_tiles; it += gridDim.x) {
                const int mt = it % p.n_mt, nt = it / p.n_mt;
                for (int kb = 0; kb < NKB; ++kb) {
                    const int kind = kb_kind(kb, p.KB, p.G);
                    if (kind < 0) continue;
                    const int s = gb % SB;
                    if (gb >= SB) lwait(&emptyb[s], (uint32_t)((gb / SB - 1) & 1), p);
                    char *st = smem + (size_t)s * kStage;
                    tc::mbar_expect_tx(&fullb[s], kStage);
                    tc::tma_load_2d(st, &p.tm_x, kind * kLBK, mt * kLM, &fullb[s]);
                    tc::tma_load_2d(st + kXBytes, &p.tm_w, kind * kLBK, nt * BN, &fullb[s]);
                    ++gb;
                }
            }
            // every load has landed before the CTA exits: the last fill of each
            // stage (the MMA thread waited for all of them in order)
            for (int s = 0; s < SB && s < gb; ++s) {
                const int last = gb - 1 - ((gb - 1 - s) % SB);  // last fill of stage s
                lwait(&fullb[s], (uint32_t)((last / SB) & 1), p);
            }
        }
    } else if (warp == 1) {
        // ---- MMA issue
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kLM, BN);
            int gb = 0, gd = 0, i = 0;
            for (int it = blockIdx.x; it < p.n_tiles; it += gridDim.x, ++i) {
                const int buf = i & 1;
                if (i >= 2) lwait(&acce[buf], (uint32_t)(((i >> 1) - 1) & 1), p);
                tc::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * BN);
                for (int kb = 0; kb < NKB; ++kb) {
                    const bool base = kb_kind(kb, p.KB, p.G) >= 0;
                    uint64_t *fb = base ? &fullb[gb % SB] : &fulld[gd % SD];
                    uint64_t *eb = base ? &emptyb[gb % SB] : &emptyd[gd % SD];
                    const uint32_t par = base ? (uint32_t)((gb / SB) & 1) : (uint32_t)((gd / SD) & 1);
                    char *st = base ? smem + (size_t)(gb % SB) * kStage : dring + (size_t)(gd % SD) * kStage;
                    lwait(fb, par, p);
                    tc::tc_fence_after();
                    if (base || !s_skip[gd % SD]) {
                        const uint32_t xa = tc::smem_u32(st), wa = xa + kXBytes;
#pragma unroll
                        for (int k = 0; k < kLBK / 16; ++k)
                            tc::mma_bf16(d, tc::desc_sw128(xa + k * 32), tc::desc_sw128(wa + k * 32), idesc,
                                         (kb | k) != 0);
                    }
                    tc::mma_commit(eb);
                    if (base) ++gb; else ++gd;
                }
                tc::mma_commit(&accf[buf]);
            }
            // the last tile's MMAs are complete before the accumulators are freed
            if (i > 0) lwait(&accf[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1), p);
        }
    } else if (warp < kFill0) {
        // ---- epilogue: y = accumulator + bias, bf16
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int q = warp & 3;  // TMEM lane quarter of this warp
        int i = 0;
        for (int it = blockIdx.x; it < p.n_tiles; it += gridDim.x, ++i) {
            const int buf = i & 1;
            const int mt = it % p.n_mt, nt = it / p.n_mt;
            const int row = mt * kLM + q * 32 + lane;
            lwait(&accf[buf], (uint32_t)((i >> 1) & 1), p);
            tc::tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c * 32), r);
                tc::tmem_wait_ld();
                const int col0 = nt * BN + c * 32;
                if (row < p.T && col0 < p.O) {
                    uint16_t *yr = p.y + (long long)row * p.ldy + col0;
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8) {
                        float bsum[8];
                        if (p.bias && p.bias_vec) {
                            const uint4 bb = __ldg((const uint4 *)(p.bias + col0 + g8 * 8));
                            bsum[0] = bf16lo(bb.x); bsum[1] = bf16hi(bb.x); bsum[2] = bf16lo(bb.y); bsum[3] = bf16hi(bb.y);
                            bsum[4] = bf16lo(bb.z); bsum[5] = bf16hi(bb.z); bsum[6] = bf16lo(bb.w); bsum[7] = bf16hi(bb.w);
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                bsum[e] = p.bias ? __uint_as_float((uint32_t)__ldg(p.bias + col0 + g8 * 8 + e) << 16) : 0.f;
                        }
                        uint4 o;
                        o.x = pack_bf2(__uint_as_float(r[g8 * 8 + 0]) + bsum[0], __uint_as_float(r[g8 * 8 + 1]) + bsum[1]);
                        o.y = pack_bf2(__uint_as_float(r[g8 * 8 + 2]) + bsum[2], __uint_as_float(r[g8 * 8 + 3]) + bsum[3]);
                        o.z = pack_bf2(__uint_as_float(r[g8 * 8 + 4]) + bsum[4], __uint_as_float(r[g8 * 8 + 5]) + bsum[5]);
                        o.w = pack_bf2(__uint_as_float(r[g8 * 8 + 6]) + bsum[6], __uint_as_float(r[g8 * 8 + 7]) + bsum[7]);
                        *(uint4 *)(yr + g8 * 8) = o;
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acce[buf]);
        }
    } else {
        // ---- delta blocks
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int f = (int)threadIdx.x - kFill0 * 32, fw = f >> 5;
        const int cpw = p.Rw >> 3;  // 16-byte chunks of one slot's segment
        int gd = 0;
        for (int it = blockIdx.x; it < p.n_tiles; it += gridDim.x) {
            const int mt = it % p.n_mt, nt = it / p.n_mt;
            const int n0 = nt * BN;
            int j = 0;
            while (j + 1 < p.n_slices && n0 >= p.out_off[j + 1]) ++j;
            const int ob = n0 - p.out_off[j];  // first B row of the tile in slice j
            // distinct slots of the tile's tokens, in order of first occurrence
            const int row = mt * kLM + f;
            const int a = row < p.T ? p.slot_of[row] : -1;
            s_rowslot[f] = a;
            const unsigned peers = __match_any_sync(0xffffffffu, a);
            const int leader = __ffs(peers) - 1;
            fill_sync();
            int first = fw * 32 + leader;
            if (lane == leader && a >= 0) {
                for (int r2 = 0; r2 < fw * 32; ++r2)
                    if (s_rowslot[r2] == a) {
                        first = r2;
                        break;
                    }
            }
            first = __shfl_sync(0xffffffffu, first, leader);
            const bool uniq = a >= 0 && first == f;
            const unsigned ub = __ballot_sync(0xffffffffu, uniq);
            if (lane == 0) s_wcnt[fw] = __popc(ub);
            fill_sync();
            int base = 0;
            for (int w = 0; w < fw; ++w) base += s_wcnt[w];
            const int nu = s_wcnt[0] + s_wcnt[1] + s_wcnt[2] + s_wcnt[3];
            if (uniq) {
                const int u = base + __popc(ub & ((1u << lane) - 1u));
                s_uidx[f] = u;
                s_uslot[u] = a;
            }
            fill_sync();
            const int u = a >= 0 ? s_uidx[first] : -1;
            const int my_g = u >= 0 ? u / p.pg : -1;
            const int my_c0 = u >= 0 ? (u - my_g * p.pg) * cpw : 0;  // first chunk of this token's segment
            // this token's scale[a] * v row of slice j, as bf16 chunks of 8 ranks
            uint4 vq[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) vq[c] = make_uint4(0u, 0u, 0u, 0u);
            if (a >= 0) {
                const float sc = p.scale[a];
                const int srow = p.sorted_rows ? p.pos_of[row] : row;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float e[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) e[k] = 0.f;
                    if (c * 8 < p.R) {
#pragma unroll
                        for (int h = 0; h < 4; ++h) {  // the hidden chunks' sums (at most 4), in chunk order
                            if (h < p.nc) {
                                const float *vr =
                                    p.part + (((long long)h * p.n_slices + j) * p.T + srow) * p.r8 + c * 8;
#pragma unroll
                                for (int k = 0; k < 8; ++k)
                                    if (c * 8 + k < p.R) e[k] += vr[k];
                            }
                        }
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k) e[k] *= sc;
                    vq[c] = make_uint4(pack_bf2(e[0], e[1]), pack_bf2(e[2], e[3]), pack_bf2(e[4], e[5]),
                                       pack_bf2(e[6], e[7]));
                }
            }
            // the tile's B rows of every distinct slot into L2, ahead of the delta blocks
            if (f < nu) s_urs[f] = (p.rank[s_uslot[f]] + 7) & ~7;
            fill_sync();
            for (int uu = 0; uu < nu; ++uu) {
                const int sl = s_uslot[uu];
                const int rs = s_urs[uu];
                const char *b0 = (const char *)(p.B[j] + (long long)sl * p.B_ss[j] + (long long)ob * rs);
                const int lines = (BN * rs * 2 + 127) >> 7;
                for (int l = f; l < lines; l += kLM) asm volatile("prefetch.global.L2 [%0];" ::"l"(b0 + l * 128));
            }
            for (int kb = 0; kb < NKB; ++kb) {
                const int kind = kb_kind(kb, p.KB, p.G);
                if (kind >= 0) continue;
                const int s = gd % SD;
                const int g = -kind - 1;
                const bool skip = g * p.pg >= nu;
                // this thread's Bhat rows (tile rows f and f + 128), loaded before the stage is free
                uint4 bw[BN / 128][8];
#pragma unroll
                for (int rr = 0; rr < BN / 128; ++rr)
#pragma unroll
                    for (int c = 0; c < 8; ++c) bw[rr][c] = make_uint4(0u, 0u, 0u, 0u);
                if (!skip) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int pp = c / cpw, kc = c - pp * cpw;  // slot of the group, rank chunk
                        const int uu = g * p.pg + pp;
                        if (uu < nu) {
                            const int sl = s_uslot[uu];
                            const int rs = s_urs[uu];
                            if (kc * 8 < rs) {
                                const uint16_t *bs = p.B[j] + (long long)sl * p.B_ss[j] + kc * 8;
#pragma unroll
                                for (int rr = 0; rr < BN / 128; ++rr)
                                    bw[rr][c] = __ldg((const uint4 *)(bs + (long long)(ob + f + rr * 128) * rs));
                            }
                        }
                    }
                }
                if (gd >= SD) {
                    if (lane == 0) lwait(&emptyd[s], (uint32_t)((gd / SD - 1) & 1), p);
                    __syncwarp();
                }
                if (!skip) {
                    const uint32_t st = tc::smem_u32(dring + (size_t)s * kStage);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 val = make_uint4(0u, 0u, 0u, 0u);
                        if (my_g == g) {
                            const int rc = c - my_c0;
#pragma unroll
                            for (int t = 0; t < 8; ++t)
                                if (t == rc && t < cpw) val = vq[t];
                        }
                        sts128(st + sw128(f, c), val);
                    }
#pragma unroll
                    for (int rr = 0; rr < BN / 128; ++rr)
#pragma unroll
                        for (int c = 0; c < 8; ++c) sts128(st + kXBytes + sw128(f + rr * 128, c), bw[rr][c]);
                    tc::fence_proxy_async();
                }
                fill_sync();
                if (f == 0) {
                    s_skip[s] = skip ? 1 : 0;
                    tc::mbar_arrive(&fulld[s]);
                }
                ++gd;
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, 2 * BN);
}

std::atomic<int> g_lin_configured[64];

// ------------------------------------------------------------------ cuBLASLt fallback

cublasLtHandle_t g_lt[64];

#define LT_TRY(x)                                               \
    do {                                                        \
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

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Whether the fused kernel takes this pool, and its output tile width.
int fused_bn(const lora_pool_t *pool, int T, int num_sms) {
    const lora_pool_desc_t &d = pool->desc;
    if (d.max_rank > 64 || d.n_slices > LORA_MAX_SLICES) return 0;
    bool by128 = true, by256 = true;
    int O = 0;
    for (int j = 0; j < d.n_slices; ++j) {
        by128 = by128 && d.out_dims[j] % 128 == 0;
        by256 = by256 && d.out_dims[j] % 256 == 0;
        O += d.out_dims[j];
    }
    if (!by128) return 0;
    const long long n_mt = (T + kLM - 1) / kLM;
    // 256-wide tiles when they still give every SM two tiles
    return by256 && n_mt * (O / 256) >= 2ll * num_sms ? 256 : 128;
}

template <int BN>
lora_status_t launch_linear(const LinArgs &a, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kLThreads, 1, 1);
    cfg.dynamicSmemBytes = kRingBytes + 1024;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    LORA_CUDA_TRY(cudaLaunchKernelEx(&cfg, linear_lora_kernel<BN>, a));
    lora_note_launch();
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
    if (meta->mode != 0 || meta->n_keys != d.max_loras) return LORA_ERR_INVALID_ARG;
    if (meta->T == 0) return LORA_OK;
    int dev = -1;
    LORA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != pool->device || dev < 0 || dev >= 64) return LORA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const int T = meta->T, R = d.max_rank, ns = d.n_slices;
    const int BN = fused_bn(pool, T, pool->num_sms);
    const size_t slot_bytes = align256((size_t)T * 4);
    LinArgs a;
    memset(&a, 0, sizeof(a));
    bool maps = false;
    if (BN && g_lora_kernel_policy == 6) {
        maps = lora_make_tmap_2d(&a.tm_x, x, d.in_dim, T, ldx, kLBK, kLM, true) &&
               lora_make_tmap_2d(&a.tm_w, W, d.in_dim, O, ldw, kLBK, BN, true);
    }
    if (!maps) {
        // the base GEMM as a library call, then the delta as a second pass
        lora_status_t st = base_gemm(dev, x, ldx, W, ldw, bias, y, ldy, T, d.in_dim, O, s);
        if (st != LORA_OK) return st;
        return lora_apply_slices(pool, meta, x, ldx, y, ldy, workspace, ws_bytes, stream);
    }
    if (!g_lin_configured[dev].load(std::memory_order_acquire)) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(linear_lora_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kRingBytes + 1024));
        LORA_CUDA_TRY(cudaFuncSetAttribute(linear_lora_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kRingBytes + 1024));
        g_lin_configured[dev].store(1, std::memory_order_release);
    }
    // each token's slot and sorted position at the head of the workspace's
    // scratch, then x A^T (fp32, unscaled) past them
    char *head = nullptr;
    size_t data_bytes = 0;
    if (!lora_ws_data(workspace, ws_bytes, &head, &data_bytes) || 2 * slot_bytes > data_bytes)
        return LORA_ERR_CAPACITY;
    int32_t *slot_of = (int32_t *)head;
    int32_t *pos_of = (int32_t *)(head + slot_bytes);
    int sgrid = d.max_loras + 1;
    if (sgrid > 1024) sgrid = 1024;
    linear_slot_kernel<<<sgrid, kSlotThreads, 0, s>>>(meta->sorted, meta->group_key, meta->group_start,
                                                      meta->counters, T, d.max_loras, slot_of, pos_of);
    LORA_CUDA_TRY(cudaGetLastError());
    lora_note_launch();
    float *part = nullptr;
    int nc = 0, r8 = 0, sorted_rows = 0;
    lora_status_t st = lora_dense_shrink(pool, meta, x, ldx, workspace, ws_bytes, 2 * slot_bytes, s, &part, &nc,
                                         &r8, &sorted_rows);
    if (st != LORA_OK) return st;

    a.T = T;
    a.O = O;
    a.KB = (d.in_dim + kLBK - 1) / kLBK;
    a.R = R;
    a.Rw = R <= 8 ? 8 : R <= 16 ? 16 : R <= 32 ? 32 : 64;
    a.pg = 64 / a.Rw;
    const int most = d.max_loras < kLM ? d.max_loras : kLM;  // distinct slots of a tile
    a.G = (most + a.pg - 1) / a.pg;
    a.n_mt = (T + kLM - 1) / kLM;
    a.n_tiles = a.n_mt * (O / BN);
    a.n_slices = ns;
    int off = 0;
    for (int j = 0; j < ns; ++j) {
        a.out_off[j] = off;
        off += d.out_dims[j];
        a.B[j] = pool->B[j];
        a.B_ss[j] = pool->b_slot_elems[j];
    }
    a.out_off[ns] = off;
    a.part = part;
    a.nc = nc;
    a.r8 = r8;
    a.sorted_rows = sorted_rows;
    a.slot_of = slot_of;
    a.pos_of = pos_of;
    a.rank = pool->d_rank;
    a.scale = pool->d_scale;
    a.bias = (const uint16_t *)bias;
    a.bias_vec = bias && lora_aligned16(bias);
    a.y = (uint16_t *)y;
    a.ldy = ldy;
    a.status = pool->d_status;
    // the waits of this kernel are within one CTA's pipeline (no other CTA
    // must make progress first): a fixed bound that only a fault reaches
    a.spin_limit = 1 << 20;
    const int grid = a.n_tiles < pool->num_sms ? a.n_tiles : pool->num_sms;
    return BN == 256 ? launch_linear<256>(a, grid, s) : launch_linear<128>(a, grid, s);
}
