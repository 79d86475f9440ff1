/*
 * CPU oracle for the multi-tenant LoRA delta -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this file's library.  The product path (the CUDA library) never
 * calls it, and this file shares no code, header, table or helper with it.
 *
 * What it computes (plain definitions, written out with per-token loops):
 *
 *  - lo_dense_meta: stable sort of token ids by adapter slot with inactive
 *    tokens last; per-slot counts; one segment per non-empty slot in
 *    ascending slot order.  (SGLang LoRAManager.prepare_lora_batch builds the
 *    per-request weight_indices / lora_ranks / scalings tables; the sort into
 *    segments is the Punica/S-LoRA grouping the pages name.)
 *
 *  - lo_dense_delta: for every active token t with slot a and every packed
 *    output slice j,
 *        v[k]        = sum_h x[t][h] * A_j[a][k][h]            (k < rank[a])
 *        y[t][off_j+o] += scale[a] * sum_k v[k] * B_j[a][o][k]
 *    (vLLM lora layers page, RowParallelLinearWithShardedLoRA.apply: a zeroed
 *    fp32 buffer [n_slices][T][rank], add_shrink with scale 1.0, then
 *    add_expand with add_input=True at the slice offsets; slice offsets and
 *    widths from MergedColumnParallelLinearWithLoRA.output_slices and
 *    MergedQKVParallelLinearWithLoRA; per-slot scaling from
 *    LoRAManager.prepare_lora_batch).  v is fp32 because the pages' shrink
 *    buffer is fp32; accumulation is fp32 in ascending index order.
 *
 *  - lo_moe_meta: stable sort of (token, k) pairs p = t*K + k by the key
 *    (slot, expert), slot-major, dropping pairs whose token has no enabled
 *    adapter; counts, exclusive offsets and the list of non-empty keys
 *    (vLLM FusedMoEWithLoRA: moe_lora_align_block_size, unpadded form).
 *
 *  - lo_sink_act: the Inkling sink-expert activation between the w13 and w2
 *    LoRA layers (InklingSinkExpertsLinear.forward: gate_up split in halves,
 *    SiLU(gate) * up, times the per-expert gamma of column c, expert c / d_mlp
 *    by _gamma_expand), rounded to bf16 where the page's tensors are bf16.
 *
 *  - lo_moe_w13 / lo_moe_w2: the fused-MoE LoRA deltas (vLLM
 *    FusedMoEWithLoRA._inject_lora_into_fused_moe: add_lora_fused_moe into
 *    the pre-activation cache for w13, into the per-(token, k) w2 output
 *    with the routed weight before the top-k sum), with the shared-outer
 *    layout of the Inkling LoRA PR report (expert index 0 for w13-A and
 *    w2-B when the pool's expert dimension is 1).
 *
 * A token is active when 0 <= idx[t] < L, enabled[idx[t]] != 0 and
 * rank[idx[t]] > 0.  idx = -1 is "no adapter"; any other out-of-range value
 * is counted in *n_bad and treated as -1.  Rows of inactive tokens/pairs are
 * copied through unchanged.
 *
 * Numerics: bf16 inputs are widened exactly to fp32; all sums are fp32 in
 * ascending index order with no fused multiply-add (built with
 * -ffp-contract=off), so results are identical on every host and for every
 * thread count (OpenMP only splits independent tokens/pairs).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static float bf(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static int is_active(int32_t a, int32_t L, const int32_t *enabled, const int32_t *rank) {
    return a >= 0 && a < L && enabled[a] != 0 && rank[a] > 0;
}

static void set_threads(int threads) {
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

int lo_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- dense meta */

int32_t lo_dense_meta(int32_t T, const int32_t *idx, int32_t L, const int32_t *enabled,
                      const int32_t *rank,
                      int32_t *sorted_tok,   /* [T] */
                      int32_t *slot_count,   /* [L] */
                      int32_t *seg_slot,     /* [L] (first n_seg used) */
                      int32_t *seg_start,    /* [L+1] (first n_seg+1 used) */
                      int32_t *slot_seg,     /* [L], -1 if the slot has no token */
                      int32_t *n_active, int32_t *n_seg, int32_t *n_bad) {
    int32_t pos = 0, bad = 0, nseg = 0;
    for (int32_t t = 0; t < T; ++t)
        if (idx[t] != -1 && (idx[t] < 0 || idx[t] >= L)) ++bad;
    for (int32_t a = 0; a < L; ++a) {
        slot_count[a] = 0;
        slot_seg[a] = -1;
    }
    /* slots in ascending order; within a slot, tokens in their original order */
    for (int32_t a = 0; a < L; ++a) {
        if (!is_active(a, L, enabled, rank)) continue;
        int32_t start = pos;
        for (int32_t t = 0; t < T; ++t)
            if (idx[t] == a) sorted_tok[pos++] = t;
        slot_count[a] = pos - start;
        if (pos > start) {
            seg_slot[nseg] = a;
            seg_start[nseg] = start;
            slot_seg[a] = nseg;
            ++nseg;
        }
    }
    seg_start[nseg] = pos;
    *n_active = pos;
    /* inactive tokens last, original order */
    for (int32_t t = 0; t < T; ++t)
        if (!is_active(idx[t], L, enabled, rank)) sorted_tok[pos++] = t;
    *n_seg = nseg;
    *n_bad = bad;
    return pos == T ? 0 : -1;
}

/* --------------------------------------------------------------- dense delta */

void lo_dense_delta(int32_t T, int32_t H, int32_t n_slices, const int32_t *out_dims,
                    int32_t L, int32_t R, const int32_t *idx, const int32_t *enabled,
                    const int32_t *rank, const float *scale,
                    const uint16_t *x, int64_t ldx,
                    const uint16_t *const *A,  /* per slice [L][R][H] */
                    const uint16_t *const *B,  /* per slice [L][O_j][R] */
                    const uint16_t *y_in, int64_t ldy,
                    float *y_ref,              /* [T][ldy] */
                    float *delta_ref,          /* [T][ldy] */
                    int threads) {
    int64_t out_total = 0;
    for (int32_t j = 0; j < n_slices; ++j) out_total += out_dims[j];
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t t = 0; t < T; ++t) {
        float *v = (float *)malloc(sizeof(float) * (R > 0 ? R : 1));
        const int32_t a = idx[t];
        const int act = is_active(a, L, enabled, rank);
        int64_t off = 0;
        for (int64_t o = 0; o < out_total; ++o) {
            y_ref[t * ldy + o] = bf(y_in[t * ldy + o]);
            delta_ref[t * ldy + o] = 0.0f;
        }
        for (int32_t j = 0; act && j < n_slices; ++j) {
            const int32_t O = out_dims[j];
            const int32_t r = rank[a];
            const uint16_t *Aa = A[j] + (int64_t)a * R * H;
            const uint16_t *Ba = B[j] + (int64_t)a * O * R;
            /* shrink: fp32 buffer, scale 1.0 */
            for (int32_t k = 0; k < r; ++k) {
                float s = 0.0f;
                for (int32_t h = 0; h < H; ++h) s += bf(x[t * ldx + h]) * bf(Aa[(int64_t)k * H + h]);
                v[k] = s;
            }
            /* expand, added in place at the slice offset */
            for (int32_t o = 0; o < O; ++o) {
                float s = 0.0f;
                for (int32_t k = 0; k < r; ++k) s += v[k] * bf(Ba[(int64_t)o * R + k]);
                const float d = scale[a] * s;
                delta_ref[t * ldy + off + o] = d;
                y_ref[t * ldy + off + o] = bf(y_in[t * ldy + off + o]) + d;
            }
            off += O;
        }
        free(v);
    }
}

/* ------------------------------------------------------------------ MoE meta */

int32_t lo_moe_meta(int32_t T, int32_t K, int32_t E, int32_t L, const int32_t *topk_ids,
                    const int32_t *idx, const int32_t *enabled, const int32_t *rank,
                    int32_t *sorted_pair,  /* [T*K] */
                    int32_t *key_count,    /* [L*E] */
                    int32_t *key_offset,   /* [L*E+1] exclusive prefix of key_count */
                    int32_t *group_key,    /* [L*E] non-empty keys, ascending */
                    int32_t *group_start,  /* [L*E+1] */
                    int32_t *n_active, int32_t *n_groups, int32_t *n_bad) {
    const int64_t P = (int64_t)T * K;
    const int32_t NK = L * E;
    int32_t pos = 0, ng = 0, bad = 0;
    for (int32_t t = 0; t < T; ++t) {
        if (idx[t] != -1 && (idx[t] < 0 || idx[t] >= L)) ++bad;
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = topk_ids[(int64_t)t * K + k];
            if (e < 0 || e >= E) ++bad;
        }
    }
    for (int32_t key = 0; key < NK; ++key) {
        const int32_t a = key / E, e = key % E;
        key_offset[key] = pos;
        int32_t start = pos;
        if (is_active(a, L, enabled, rank)) {
            for (int64_t p = 0; p < P; ++p) {
                const int32_t t = (int32_t)(p / K);
                if (idx[t] == a && topk_ids[p] == e) sorted_pair[pos++] = (int32_t)p;
            }
        }
        key_count[key] = pos - start;
        if (pos > start) {
            group_key[ng] = key;
            group_start[ng] = start;
            ++ng;
        }
    }
    key_offset[NK] = pos;
    group_start[ng] = pos;
    *n_active = pos;
    *n_groups = ng;
    *n_bad = bad;
    /* pairs without an active (slot, expert) key, original order */
    for (int64_t p = 0; p < P; ++p) {
        const int32_t t = (int32_t)(p / K);
        const int32_t e = topk_ids[p];
        if (!(is_active(idx[t], L, enabled, rank) && e >= 0 && e < E)) sorted_pair[pos++] = (int32_t)p;
    }
    return pos == P ? 0 : -1;
}

/* ------------------------------------------------------------------ MoE w13 */

void lo_moe_w13(int32_t T, int32_t K, int32_t D, int32_t F13, int32_t E, int32_t L, int32_t R,
                int32_t n_slices, int32_t shared_outer,
                const int32_t *idx, const int32_t *topk_ids,
                const int32_t *enabled, const int32_t *rank, const float *scale,
                const uint16_t *x, int64_t ldx,
                const uint16_t *const *A13,   /* per slice [L][E or 1][R][D] */
                const uint16_t *const *B13,   /* per slice [L][E][F13][R] */
                const uint16_t *ic1_in, int64_t ld1,
                float *ic1_ref, float *delta_ref,  /* [T*K][ld1] */
                int threads) {
    const int64_t P = (int64_t)T * K;
    const int32_t EA = shared_outer ? 1 : E;
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t p = 0; p < P; ++p) {
        float *v = (float *)malloc(sizeof(float) * (R > 0 ? R : 1));
        const int32_t t = (int32_t)(p / K);
        const int32_t a = idx[t];
        const int32_t e = topk_ids[p];
        const int act = is_active(a, L, enabled, rank) && e >= 0 && e < E;
        for (int64_t c = 0; c < (int64_t)n_slices * F13; ++c) {
            ic1_ref[p * ld1 + c] = bf(ic1_in[p * ld1 + c]);
            delta_ref[p * ld1 + c] = 0.0f;
        }
        for (int32_t s = 0; act && s < n_slices; ++s) {
            const int32_t r = rank[a];
            const int32_t ea = shared_outer ? 0 : e;
            const uint16_t *Aa = A13[s] + ((int64_t)a * EA + ea) * R * D;
            const uint16_t *Ba = B13[s] + ((int64_t)a * E + e) * F13 * R;
            for (int32_t k = 0; k < r; ++k) {
                float acc = 0.0f;
                for (int32_t h = 0; h < D; ++h) acc += bf(x[(int64_t)t * ldx + h]) * bf(Aa[(int64_t)k * D + h]);
                v[k] = acc;
            }
            for (int32_t o = 0; o < F13; ++o) {
                float acc = 0.0f;
                for (int32_t k = 0; k < r; ++k) acc += v[k] * bf(Ba[(int64_t)o * R + k]);
                const float d = scale[a] * acc;
                const int64_t c = (int64_t)s * F13 + o;
                delta_ref[p * ld1 + c] = d;
                ic1_ref[p * ld1 + c] = bf(ic1_in[p * ld1 + c]) + d;
            }
        }
        free(v);
    }
}

/* ------------------------------------------------------------------- MoE w2 */

void lo_moe_w2(int32_t T, int32_t K, int32_t D, int32_t F, int32_t E, int32_t L, int32_t R,
               int32_t shared_outer,
               const int32_t *idx, const int32_t *topk_ids, const float *topk_w,
               const int32_t *enabled, const int32_t *rank, const float *scale,
               const uint16_t *ic2, int64_t ld2,
               const uint16_t *A2,   /* [L][E][R][F] */
               const uint16_t *B2,   /* [L][E or 1][D][R] */
               const uint16_t *ic3_in, int64_t ld3,
               float *ic3_ref, float *delta_ref,  /* [T*K][ld3] */
               int threads) {
    const int64_t P = (int64_t)T * K;
    const int32_t EB = shared_outer ? 1 : E;
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t p = 0; p < P; ++p) {
        float *v = (float *)malloc(sizeof(float) * (R > 0 ? R : 1));
        const int32_t t = (int32_t)(p / K);
        const int32_t a = idx[t];
        const int32_t e = topk_ids[p];
        const int act = is_active(a, L, enabled, rank) && e >= 0 && e < E;
        for (int32_t o = 0; o < D; ++o) {
            ic3_ref[p * ld3 + o] = bf(ic3_in[p * ld3 + o]);
            delta_ref[p * ld3 + o] = 0.0f;
        }
        if (act) {
            const int32_t r = rank[a];
            const int32_t eb = shared_outer ? 0 : e;
            const uint16_t *Aa = A2 + ((int64_t)a * E + e) * R * F;
            const uint16_t *Ba = B2 + ((int64_t)a * EB + eb) * D * R;
            for (int32_t k = 0; k < r; ++k) {
                float acc = 0.0f;
                for (int32_t f = 0; f < F; ++f) acc += bf(ic2[p * ld2 + f]) * bf(Aa[(int64_t)k * F + f]);
                v[k] = acc;
            }
            for (int32_t o = 0; o < D; ++o) {
                float acc = 0.0f;
                for (int32_t k = 0; k < r; ++k) acc += v[k] * bf(Ba[(int64_t)o * R + k]);
                /* routed weight multiplies the w2 delta (the positional True of
                   the w2 add_lora_fused_moe call) */
                const float d = topk_w[p] * (scale[a] * acc);
                delta_ref[p * ld3 + o] = d;
                ic3_ref[p * ld3 + o] = bf(ic3_in[p * ld3 + o]) + d;
            }
        }
        free(v);
    }
}

/* ---------------------------------------------------------------- lm_head */

/* LoRA logits of LogitsProcessorWithLoRA._get_logits (vLLM LoRA layer page),
 * with the muP multiplier of the Inkling report's _lora_forward:
 *   full[t][i] = logits_in[t][map[i]]          (sharded_to_full_mapping; map
 *                                               NULL = identity)
 *   full[t][i] += delta[t][i]                  (add_lora_logits, scale 1.0:
 *                                               the delta of lo_dense_delta)
 *   out[t][i]  = mup * full[t][i]  for i < vocab_size   (slice, then x 1/mup)
 * delta is the fp32 [T][ld_delta] output of lo_dense_delta on the same tokens. */
void lo_logits(int32_t T, int32_t vocab_size, const int32_t *map, const uint16_t *logits_in,
               int64_t ld_in, const float *delta, int64_t ld_delta, float mup, float *out,
               int64_t ld_out) {
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t i = 0; i < vocab_size; ++i) {
            const int32_t src = map ? map[i] : i;
            const float full = bf(logits_in[(int64_t)t * ld_in + src]) + delta[(int64_t)t * ld_delta + i];
            out[(int64_t)t * ld_out + i] = mup * full;
        }
    }
}

/* -------------------------------------------------- MoE block-padded align */

/* The padded per-adapter form of moe_lora_align_block_size (vLLM
 * FusedMoEWithLoRA._inject_lora_into_fused_moe views sorted_token_ids_lora and
 * expert_ids_lora as (max_loras, -1) and passes num_tokens_post_padded_lora):
 * for every enabled adapter a (rank > 0), its pairs p = t*K + k in ascending
 * expert order (pair order kept within an expert); each expert's run is
 * padded with the sentinel T*K to a multiple of block_m.
 *   sorted[a][cap]           pair ids and sentinels; unused entries = T*K
 *   expert[a][cap / block_m] expert id of each block; unused = -1
 *   npp[a]                   padded length of adapter a (0 if none)
 * cap must be a multiple of block_m; returns -1 if an adapter overflows it. */
int32_t lo_moe_align_padded(int32_t T, int32_t K, int32_t E, int32_t L, const int32_t *topk_ids,
                            const int32_t *idx, const int32_t *enabled, const int32_t *rank,
                            int32_t block_m, int32_t cap, int32_t *sorted, int32_t *expert, int32_t *npp) {
    const int64_t P = (int64_t)T * K;
    const int32_t nb = cap / block_m;
    int32_t rc = 0;
    for (int32_t a = 0; a < L; ++a) {
        int32_t pos = 0;
        for (int32_t i = 0; i < cap; ++i) sorted[(int64_t)a * cap + i] = (int32_t)P;
        for (int32_t b = 0; b < nb; ++b) expert[(int64_t)a * nb + b] = -1;
        if (is_active(a, L, enabled, rank)) {
            for (int32_t e = 0; e < E; ++e) {
                const int32_t start = pos;
                for (int64_t p = 0; p < P; ++p) {
                    if (idx[p / K] == a && topk_ids[p] == e) {
                        if (pos >= cap) return -1;
                        sorted[(int64_t)a * cap + pos++] = (int32_t)p;
                    }
                }
                if (pos > start) {
                    const int32_t padded = ((pos - start + block_m - 1) / block_m) * block_m;
                    if (start + padded > cap) return -1;
                    for (int32_t b = start / block_m; b < (start + padded) / block_m; ++b)
                        expert[(int64_t)a * nb + b] = e;
                    pos = start + padded;
                }
            }
        }
        npp[a] = pos;
    }
    return rc;
}

/* -------------------------------------------------- Inkling sink experts */

/* Round to the nearest bf16 value, ties to even (8 significant bits), from an
 * exact double; the result is returned as a double. */
static double round_bf16(double v) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    frexp(v, &e);    /* v = f * 2^e with 0.5 <= |f| < 1 */
    int q = e - 8;   /* spacing of bf16 values in this binade */
    if (q < -133) q = -133;
    return ldexp(rint(ldexp(v, -q)), q); /* rint rounds half to even */
}

/* InklingSinkExpertsLinear.forward between its two linear layers, with
 * n = n_experts and W = n * d_mlp columns per half:
 *   gate = gate_up[t][c], up = gate_up[t][W + c]          (chunk(2, dim=-1))
 *   s    = bf16(silu(gate))      silu(g) = g / (1 + exp(-g)), exact in double
 *   p    = bf16(s * up)
 *   h[t][c] = bf16(p * gammas[t][c / d_mlp])              (_gamma_expand, .to(bf16))
 * Outputs are bf16 bits. */
void lo_sink_act(int32_t T, int32_t n_experts, int32_t d_mlp, const uint16_t *gate_up, int64_t ld_gu,
                 const float *gammas, int64_t ld_gamma, uint16_t *h, int64_t ld_h) {
    const int64_t W = (int64_t)n_experts * d_mlp;
    for (int32_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < W; ++c) {
            const double g = (double)bf(gate_up[(int64_t)t * ld_gu + c]);
            const double u = (double)bf(gate_up[(int64_t)t * ld_gu + W + c]);
            const double sg = round_bf16(g / (1.0 + exp(-g)));
            const double pr = round_bf16(sg * u);
            const double v = round_bf16(pr * (double)gammas[(int64_t)t * ld_gamma + c / d_mlp]);
            /* v is a bf16 value: its float has zero low 16 bits */
            const float f = (float)v;
            uint32_t bits;
            memcpy(&bits, &f, 4);
            h[(int64_t)t * ld_h + c] = (uint16_t)(bits >> 16);
        }
    }
}
