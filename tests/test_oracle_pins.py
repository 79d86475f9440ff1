"""Pins for the CPU oracle: each check ties the oracle to something other than
itself (hand-derived golden values, fp64 brute force, the merged-weight
identity, the invariants the LoRA layer pages fix, numpy's stable argsort).
The last test plants mistakes in copies of the oracle source and checks that
these pins catch every one of them."""
import os

import numpy as np
import pytest

import oracle
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits
from oracle_pins_util import (dense_from_golden, exact_dense, exact_moe, load_golden,
                              moe_from_golden)

# ----------------------------------------------------------------- golden


def test_golden_dense_by_hand():
    g = load_golden("dense_by_hand.json")
    c = dense_from_golden(g)
    _, d = oracle.dense_delta(c)
    np.testing.assert_array_equal(d, np.asarray(g["delta"], np.float32))
    y_in = f32_to_bf16_bits(np.asarray(g["y_in"], np.float32))
    y, _ = oracle.dense_delta(c, y_in=y_in)
    np.testing.assert_array_equal(y, np.asarray(g["y_out"], np.float32))


def test_golden_moe_by_hand():
    g = load_golden("moe_by_hand.json")
    c = moe_from_golden(g)
    _, d13 = oracle.moe_w13(c)
    np.testing.assert_array_equal(d13, np.asarray(g["delta13"], np.float32))
    _, d2 = oracle.moe_w2(c)
    np.testing.assert_array_equal(d2, np.asarray(g["delta2"], np.float32))


def test_golden_meta_by_hand():
    g = load_golden("meta_by_hand.json")
    m = oracle.dense_meta(np.asarray(g["idx"], np.int32), g["L"], np.asarray(g["enabled"], np.int32),
                          np.asarray(g["rank"], np.int32))
    assert m.sorted_tok.tolist() == g["sorted_tok"]
    assert m.n_active == g["n_active"]
    assert m.seg_slot.tolist() == g["seg_slot"]
    assert m.seg_start.tolist() == g["seg_start"]
    assert m.slot_count.tolist() == g["slot_count"]
    assert m.slot_seg.tolist() == g["slot_seg"]
    assert m.n_bad == g["n_bad"]


def test_golden_moe_meta_bad_ids_by_hand():
    g = load_golden("moe_meta_bad_ids_by_hand.json")
    m = oracle.moe_meta(np.asarray(g["topk_ids"], np.int32), np.asarray(g["idx"], np.int32), g["L"], g["E"],
                        np.asarray(g["enabled"], np.int32), np.asarray(g["rank"], np.int32))
    assert m.sorted_pair.tolist() == g["sorted_pair"]
    assert m.key_count.tolist() == g["key_count"]
    assert m.key_offset.tolist() == g["key_offset"]
    assert m.group_key.tolist() == g["group_key"]
    assert m.group_start.tolist() == g["group_start"]
    assert (m.n_active, m.n_groups, m.n_bad) == (g["n_active"], g["n_groups"], g["n_bad"])


# ----------------------------------------------------------------- fp64 brute force

def _tiny_dense(seed, T=7, H=48, out_dims=(16, 8, 8), L=3, R=4, ranks=(4, 2, 3), p_none=0.2):
    rng = np.random.default_rng(seed)
    scales = rng.uniform(0.5, 3.0, size=L).astype(np.float32)
    return gen.dense_case(T=T, H=H, out_dims=out_dims, L=L, R=R, seed=seed, ranks=ranks,
                          scales=scales, p_none=p_none, std=0.5)


@pytest.mark.parametrize("seed", range(6))
def test_dense_bruteforce_fp64(seed):
    c = _tiny_dense(seed)
    _, d = oracle.dense_delta(c)
    exact, bound = exact_dense(c)
    assert np.all(np.abs(d - exact) <= bound), np.max(np.abs(d - exact) / bound)


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("seed", range(3))
def test_moe_bruteforce_fp64(seed, shared):
    c = gen.moe_case(T=5, K=3, E=4, D=40, F=24, L=3, R=4, seed=seed, shared_outer=shared,
                     ranks=(4, 3, 2), scales=(1.5, 0.5, 2.0), p_none=0.2, std=0.5)
    for which, fn in (("w13", oracle.moe_w13), ("w2", oracle.moe_w2)):
        _, d = fn(c)
        exact, bound = exact_moe(c, which)
        assert np.all(np.abs(d - exact) <= bound), (which, np.max(np.abs(d - exact) / bound))


# ----------------------------------------------------------------- merged-weight identity

def test_merged_weight_identity_tiny_preset():
    """x (W + s B A)^T - x W^T equals the delta: checked in fp64 against the
    oracle on the 512 -> 512 preset (T=64, 4 slots of rank 8, scale 2)."""
    c = gen.tiny()
    _, d = oracle.dense_delta(c)
    x = bf16_bits_to_f32(c.x).astype(np.float64)
    W = bf16_bits_to_f32(c.W).astype(np.float64)
    _, bound = exact_dense(c)
    for t in range(c.T):
        a = int(c.idx[t])
        if a < 0:
            assert np.all(d[t] == 0)
            continue
        r = int(c.ranks[a])
        Aa = bf16_bits_to_f32(c.A[0][a, :r]).astype(np.float64)
        Ba = bf16_bits_to_f32(c.B[0][a, :, :r]).astype(np.float64)
        merged = W + c.scales[a] * (Ba @ Aa)
        diff = x[t] @ merged.T - x[t] @ W.T
        # fp64 cancellation error of the subtraction is far below the fp32 bound
        assert np.all(np.abs(d[t] - diff) <= bound[t] + 1e-12), t


# ----------------------------------------------------------------- special cases

def test_none_reset_disabled_rank0_leave_y_bit_identical():
    c = _tiny_dense(11, p_none=0.3)
    c.y0 = f32_to_bf16_bits(np.random.default_rng(0).normal(0, 1, c.y0.shape).astype(np.float32))
    c.y0[0, :4] = 0x8000  # negative zeros must survive too
    base = bf16_bits_to_f32(c.y0)
    # idx -1 rows
    y, d = oracle.dense_delta(c)
    none = c.idx < 0
    assert none.any()
    assert np.array_equal(y[none].view(np.uint32), base[none].view(np.uint32))
    assert np.all(d[none] == 0)
    # reset slot 0 (weights zero, enabled 0) and rank-0 slot 1
    A = [a.copy() for a in c.A]
    B = [b.copy() for b in c.B]
    for j in range(c.n_slices):
        A[j][0] = 0
        B[j][0] = 0
    en = c.enabled.copy()
    en[0] = 0
    rk = c.ranks.copy()
    rk[1] = 0
    y, d = oracle.dense_delta(c, A=A, B=B, enabled=en, ranks=rk)
    sel = np.isin(c.idx, [0, 1])
    assert sel.any()
    assert np.array_equal(y[sel].view(np.uint32), base[sel].view(np.uint32))
    # enabled but all-zero weights: the delta is exactly zero
    y, d = oracle.dense_delta(c, A=A, B=B)
    sel = c.idx == 0
    assert np.all(d[sel] == 0)


def test_rank_padding_is_invisible():
    """set_lora copies into [:r, :in] of a zeroed stack: the same adapters in a
    compact (R = r) and a padded (R = 64) pool give bit-identical results."""
    c = _tiny_dense(5, ranks=(4, 4, 4), R=4)
    _, d_compact = oracle.dense_delta(c)
    A = [np.zeros((c.L, 64, c.H), np.uint16) for _ in c.A]
    B = [np.zeros((c.L, o, 64), np.uint16) for o in c.out_dims]
    for j in range(c.n_slices):
        A[j][:, :4] = c.A[j]
        B[j][:, :, :4] = c.B[j]
    _, d_pad = oracle.dense_delta(c, A=A, B=B)
    assert np.array_equal(d_compact.view(np.uint32), d_pad.view(np.uint32))


def test_packed_slices_equal_separate_application():
    c = _tiny_dense(7)
    _, d = oracle.dense_delta(c)
    off = 0
    for j, o in enumerate(c.out_dims):
        _, dj = oracle.dense_delta(c, A=[c.A[j]], B=[c.B[j]], out_dims=(o,),
                                   y_in=np.zeros((c.T, o), np.uint16))
        assert np.array_equal(d[:, off:off + o].view(np.uint32), dj.view(np.uint32))
        off += o


def test_variable_slice_dup_a_split_b_equals_single_projection():
    """MergedColumnParallelLinearVariableSliceWithLoRA.set_lora: one A duplicated
    to every slice and one B split along its rows by output_sizes gives the same
    delta as that A, B on the whole packed output."""
    c = _tiny_dense(9, out_dims=(8, 16, 8))
    Bw = np.concatenate(c.B, axis=1)            # [L][sum O][R]
    _, d_single = oracle.dense_delta(c, A=[c.A[0]], B=[Bw], out_dims=(sum(c.out_dims),))
    offs = np.cumsum((0,) + c.out_dims)
    Bs = [np.ascontiguousarray(Bw[:, offs[j]:offs[j + 1]]) for j in range(3)]
    _, d_packed = oracle.dense_delta(c, A=[c.A[0]] * 3, B=Bs)
    assert np.array_equal(d_single.view(np.uint32), d_packed.view(np.uint32))


def test_moe_reduces_to_dense_with_one_expert_top1():
    c = gen.moe_case(T=9, K=1, E=1, D=32, F=16, L=3, R=4, seed=3, n13=1, ranks=(4, 2, 3),
                     scales=(1.0, 2.0, 0.5), p_none=0.2, std=0.5)
    c.topk_w[:] = 1.0
    _, d13 = oracle.moe_w13(c)
    _, dd = oracle.dense_delta(x=c.x, idx=c.idx, A=[c.A13[0][:, 0]], B=[c.B13[0][:, 0]],
                               y_in=np.zeros((c.T, c.F13), np.uint16), ranks=c.ranks,
                               scales=c.scales, enabled=c.enabled, out_dims=(c.F13,))
    assert np.array_equal(d13.view(np.uint32), dd.view(np.uint32))
    _, d2 = oracle.moe_w2(c)
    _, dd2 = oracle.dense_delta(x=c.ic2, idx=c.idx, A=[c.A2[:, 0]], B=[c.B2[:, 0]],
                                y_in=np.zeros((c.T, c.D), np.uint16), ranks=c.ranks,
                                scales=c.scales, enabled=c.enabled, out_dims=(c.D,))
    assert np.array_equal(d2.view(np.uint32), dd2.view(np.uint32))


def test_moe_shared_outer_equals_broadcast_per_expert():
    c = gen.moe_case(T=6, K=2, E=3, D=24, F=16, L=2, R=4, seed=4, shared_outer=True, std=0.5)
    _, s13 = oracle.moe_w13(c)
    _, s2 = oracle.moe_w2(c)
    c.A13 = [np.ascontiguousarray(np.repeat(a, c.E, axis=1)) for a in c.A13]
    c.B2 = np.ascontiguousarray(np.repeat(c.B2, c.E, axis=1))
    c.shared_outer = False
    _, p13 = oracle.moe_w13(c)
    _, p2 = oracle.moe_w2(c)
    assert np.array_equal(s13.view(np.uint32), p13.view(np.uint32))
    assert np.array_equal(s2.view(np.uint32), p2.view(np.uint32))


def test_moe_disabled_adapter_gives_no_delta():
    c = gen.moe_case(T=6, K=2, E=3, D=24, F=16, L=2, R=4, seed=6, std=0.5)
    c.ic1_0 = f32_to_bf16_bits(np.ones(c.ic1_0.shape, np.float32))
    en = c.enabled.copy()
    en[1] = 0
    y, d = oracle.moe_w13(c, ic1_in=c.ic1_0, enabled=en)
    rows = np.repeat(c.idx == 1, c.K)
    assert rows.any()
    assert np.all(d[rows] == 0) and np.all(y[rows] == 1.0)
    assert np.any(d[~rows] != 0)


# ----------------------------------------------------------------- metadata vs numpy

@pytest.mark.parametrize("seed", range(5))
def test_dense_meta_matches_numpy_stable_argsort(seed):
    rng = np.random.default_rng(seed)
    T, L = int(rng.integers(1, 300)), int(rng.integers(1, 40))
    idx = rng.integers(-2, L + 2, size=T).astype(np.int32)
    enabled = (rng.random(L) < 0.8).astype(np.int32)
    rank = rng.choice([0, 8, 16], size=L).astype(np.int32)
    m = oracle.dense_meta(idx, L, enabled, rank)
    act = np.array([bool(0 <= a < L and enabled[a] and rank[a] > 0) for a in idx], dtype=bool)
    key = np.where(act, idx, L)
    order = np.argsort(key, kind="stable")
    assert np.array_equal(m.sorted_tok, order)
    assert m.n_active == int(act.sum())
    cnt = np.bincount(idx[act], minlength=L)
    assert np.array_equal(m.slot_count, cnt)
    nz = np.nonzero(cnt)[0]
    assert np.array_equal(m.seg_slot, nz)
    assert np.array_equal(m.seg_start, np.concatenate([[0], np.cumsum(cnt[nz])]))
    assert m.n_bad == int(np.sum((idx != -1) & ((idx < 0) | (idx >= L))))


@pytest.mark.parametrize("seed,bad_ids", [(s, b) for s in range(4) for b in (False, True)])
def test_moe_meta_matches_numpy_lexsort(seed, bad_ids):
    rng = np.random.default_rng(100 + seed)
    T, K, E, L = int(rng.integers(1, 64)), int(rng.integers(1, 5)), int(rng.integers(1, 9)), 4
    # with bad_ids, expert ids run from -2 to E + 1 and slot ids from -2 to L + 1
    lo, hi = (-2, 2) if bad_ids else (0, 0)
    topk = rng.integers(lo, E + hi, size=(T, K)).astype(np.int32)
    idx = rng.integers(-1 + lo, L + hi, size=T).astype(np.int32)
    enabled = np.array([1, 0, 1, 1], np.int32)
    rank = np.array([4, 4, 0, 4], np.int32)
    m = oracle.moe_meta(topk, idx, L, E, enabled, rank)
    pt = np.repeat(np.arange(T), K)
    a = idx[pt]
    e = topk.reshape(-1)
    act = (a >= 0) & np.isin(a, np.nonzero(enabled & (rank > 0))[0]) & (e >= 0) & (e < E)
    key = np.where(act, a * E + e, L * E)
    assert np.array_equal(m.sorted_pair, np.argsort(key, kind="stable"))
    cnt = np.bincount(key[act], minlength=L * E)
    assert np.array_equal(m.key_count, cnt)
    assert np.array_equal(m.key_offset, np.concatenate([[0], np.cumsum(cnt)]))
    assert np.array_equal(m.group_key, np.nonzero(cnt)[0])
    assert m.n_active == int(act.sum())
    n_bad = int(np.sum((idx != -1) & ((idx < 0) | (idx >= L)))) + int(np.sum((e < 0) | (e >= E)))
    assert m.n_bad == n_bad


# ----------------------------------------------------------------- planted mistakes

MUTANTS = {
    "dense_drop_scale": ("const float d = scale[a] * s;", "const float d = s;"),
    "dense_transposed_B": ("s += v[k] * bf(Ba[(int64_t)o * R + k]);",
                           "s += v[k] * bf(Ba[(int64_t)k * O + o]);"),
    "dense_no_slice_offset": ("off += O;", "off += 0;"),
    "dense_sign": ("y_ref[t * ldy + off + o] = bf(y_in[t * ldy + off + o]) + d;",
                   "y_ref[t * ldy + off + o] = bf(y_in[t * ldy + off + o]) - d;"),
    "dense_rank_minus_one": ("for (int32_t k = 0; k < r; ++k) {\n                float s = 0.0f;",
                             "for (int32_t k = 0; k + 1 < r; ++k) {\n                float s = 0.0f;"),
    "meta_unstable": ("for (int32_t t = 0; t < T; ++t)\n            if (idx[t] == a) sorted_tok[pos++] = t;",
                      "for (int32_t t = T - 1; t >= 0; --t)\n            if (idx[t] == a) sorted_tok[pos++] = t;"),
    "moe_w2_no_routed_weight": ("const float d = topk_w[p] * (scale[a] * acc);",
                                "const float d = (scale[a] * acc);"),
    "moe_w13_expert_ignored": ("const int32_t ea = shared_outer ? 0 : e;", "const int32_t ea = 0;"),
    "moe_w13_wrong_token": ("acc += bf(x[(int64_t)t * ldx + h])", "acc += bf(x[(int64_t)(p % T) * ldx + h])"),
    "moe_w2_shared_b_per_expert": ("const int32_t eb = shared_outer ? 0 : e;",
                                   "const int32_t eb = shared_outer ? (e % EB) : (E - 1 - e);"),
    "logits_reindex_inverted": ("const int32_t src = map ? map[i] : i;",
                                "const int32_t src = map ? (map[i] ^ 1) : i;"),
    "sink_gate_up_swapped": ("const double g = (double)bf(gate_up[(int64_t)t * ld_gu + c]);\n            const double u = (double)bf(gate_up[(int64_t)t * ld_gu + W + c]);",
                             "const double u = (double)bf(gate_up[(int64_t)t * ld_gu + c]);\n            const double g = (double)bf(gate_up[(int64_t)t * ld_gu + W + c]);"),
    "sink_gamma_by_column_mod": ("gammas[(int64_t)t * ld_gamma + c / d_mlp]", "gammas[(int64_t)t * ld_gamma + c % n_experts]"),
    "sink_sigmoid_only": ("round_bf16(g / (1.0 + exp(-g)))", "round_bf16(1.0 / (1.0 + exp(-g)))"),
    "moe_meta_high_expert_not_bad": ("if (e < 0 || e >= E) ++bad;", "if (e < 0) ++bad;"),
    "moe_meta_bad_expert_kept_active": ("if (!(is_active(idx[t], L, enabled, rank) && e >= 0 && e < E)) sorted_pair[pos++] = (int32_t)p;",
                                        "if (!is_active(idx[t], L, enabled, rank)) sorted_pair[pos++] = (int32_t)p;"),
    "logits_mup_on_base_only": ("out[(int64_t)t * ld_out + i] = mup * full;",
                                "out[(int64_t)t * ld_out + i] = full + (mup - 1.0f) * bf(logits_in[(int64_t)t * ld_in + src]);"),
}


def _pin_suite_passes():
    checks = [test_golden_dense_by_hand, test_golden_moe_by_hand, test_golden_meta_by_hand,
              test_golden_moe_meta_bad_ids_by_hand, lambda: test_moe_meta_matches_numpy_lexsort(0, True),
              lambda: test_dense_bruteforce_fp64(0), lambda: test_moe_bruteforce_fp64(0, False),
              lambda: test_moe_bruteforce_fp64(1, True), test_merged_weight_identity_tiny_preset,
              test_packed_slices_equal_separate_application,
              lambda: test_dense_meta_matches_numpy_stable_argsort(0),
              test_golden_logits_reindex_example, test_logits_adds_delta_then_scales_everything_by_mup,
              test_golden_sink_act_by_hand, test_sink_act_expert_of_each_column]
    for chk in checks:
        try:
            chk()
        except AssertionError:
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = oracle.source_text()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    with oracle.use_library(lib):
        assert not _pin_suite_passes(), f"pins did not catch mutant {name}"


# ----------------------------------------------------------------- lm_head

def test_golden_logits_reindex_example():
    g = load_golden("logits_reindex.json")
    sharded = np.asarray(g["sharded_token_ids"])
    full = np.asarray(g["full_token_ids"])
    # the two printed mappings: a gather reproduces the printed orders with the
    # derived mapping, and a scatter with the printed one
    assert np.array_equal(sharded[np.asarray(g["gather_mapping"])], full)
    scat = np.empty_like(sharded)
    scat[np.asarray(g["printed_mapping"])] = sharded
    assert np.array_equal(scat, full)
    row = np.where(sharded < 0, 100.0, sharded).astype(np.float32)
    lin = f32_to_bf16_bits(np.stack([row, row * 2]))
    out = oracle.logits(lin, np.zeros((2, 8), np.float32), g["vocab_size"], mapping=g["gather_mapping"])
    np.testing.assert_array_equal(out[0], np.asarray(g["expected_row"], np.float32))
    np.testing.assert_array_equal(out[1], 2 * np.asarray(g["expected_row"], np.float32))


def test_logits_adds_delta_then_scales_everything_by_mup():
    """The Inkling report's _lora_forward multiplies base + LoRA logits by
    1/mup_multiplier, so the delta is scaled too."""
    rng = np.random.default_rng(3)
    base = f32_to_bf16_bits(rng.normal(0, 1, (3, 16)).astype(np.float32))
    delta = rng.normal(0, 0.1, (3, 16)).astype(np.float32)
    out = oracle.logits(base, delta, 12, mup=0.25)
    exp = 0.25 * (bf16_bits_to_f32(base)[:, :12].astype(np.float64) + delta[:, :12])
    assert np.allclose(out, exp, rtol=1e-6, atol=1e-7)
    out1 = oracle.logits(base, np.zeros_like(delta), 12, mup=1.0)
    assert np.array_equal(out1, bf16_bits_to_f32(base)[:, :12])


# ----------------------------------------------------------------- MoE block-padded alignment

def test_golden_moe_align_padded_by_hand():
    g = load_golden("moe_align_padded_by_hand.json")
    m = oracle.moe_align_padded(np.asarray(g["topk_ids"], np.int32), np.asarray(g["idx"], np.int32), g["L"], g["E"],
                                np.asarray(g["enabled"], np.int32), np.asarray(g["rank"], np.int32), g["block_m"],
                                g["cap"])
    assert m.sorted.tolist() == g["sorted"]
    assert m.expert.tolist() == g["expert"]
    assert m.npp.tolist() == g["npp"]


@pytest.mark.parametrize("seed", range(3))
def test_moe_align_padded_consistent_with_unpadded_meta(seed):
    """Dropping the sentinels of adapter a's padded list gives exactly the
    unpadded sorted pairs of a's keys; block counts follow ceil(count / BM)."""
    rng = np.random.default_rng(200 + seed)
    T, K, E, L, BM = 37, 3, 6, 4, 8
    topk = rng.integers(0, E, size=(T, K)).astype(np.int32)
    idx = rng.integers(-1, L, size=T).astype(np.int32)
    en, rk = np.array([1, 1, 0, 1], np.int32), np.array([8, 0, 8, 8], np.int32)
    cap = ((T * K + E * (BM - 1) + BM - 1) // BM) * BM
    pad = oracle.moe_align_padded(topk, idx, L, E, en, rk, BM, cap)
    un = oracle.moe_meta(topk, idx, L, E, en, rk)
    for a in range(L):
        got = pad.sorted[a][pad.sorted[a] != T * K]
        lo, hi = un.key_offset[a * E], un.key_offset[(a + 1) * E]
        assert np.array_equal(got, un.sorted_pair[lo:hi])
        blocks = sum(-(-int(c) // BM) for c in un.key_count[a * E:(a + 1) * E])
        assert pad.npp[a] == blocks * BM
        assert np.sum(pad.expert[a] >= 0) == blocks


# ----------------------------------------------------------------- Inkling sink experts

def test_golden_sink_act_by_hand():
    g = load_golden("sink_act_by_hand.json")
    gu = f32_to_bf16_bits(np.asarray(g["gate_up"], np.float32))
    h = oracle.sink_act(gu, np.asarray(g["gammas"], np.float32), g["n_experts"], g["d_mlp"])
    np.testing.assert_array_equal(bf16_bits_to_f32(h), np.asarray(g["expected_h"], np.float32))


def test_sink_act_expert_of_each_column():
    """gate large (silu(g) = g to bf16 precision), up = 1, one power of two per
    expert: h[t][c] = g * gamma[c // d_mlp] exactly, for d_mlp not a power of two."""
    n, d = 3, 5
    T = 2
    gate = np.full((T, n * d), 20.0, np.float32)
    up = np.ones((T, n * d), np.float32)
    gam = np.array([[0.5, 4.0, 0.125], [2.0, 1.0, 8.0]], np.float32)
    h = bf16_bits_to_f32(oracle.sink_act(f32_to_bf16_bits(np.concatenate([gate, up], 1)), gam, n, d))
    want = 20.0 * gam[:, np.arange(n * d) // d]
    np.testing.assert_array_equal(h, want)


def test_sink_act_reduces_to_logistic_silu():
    """up = 1 and gamma = 1: h = bf16(g * logistic(g)), within half a bf16 ulp
    of the library logistic function."""
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    n, d, T = 2, 8, 3
    gate_bits = f32_to_bf16_bits(rng.normal(0, 3, (T, n * d)).astype(np.float32))
    g = bf16_bits_to_f32(gate_bits).astype(np.float64)
    gu = np.concatenate([gate_bits, f32_to_bf16_bits(np.ones((T, n * d), np.float32))], 1)
    h = bf16_bits_to_f32(oracle.sink_act(gu, np.ones((T, n), np.float32), n, d)).astype(np.float64)
    exact = g * scipy_special.expit(g)
    assert np.all(np.abs(h - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-30)


# ----------------------------------------------------------------- full LoRA linear

def test_linear_equals_merged_weight_form_with_bias():
    """y = x W^T + bias + delta equals x (W + s B A)^T + bias per token (the
    merged-weight form), within the fp32 bound of the delta."""
    c = gen.tiny()
    rng = np.random.default_rng(3)
    bias = f32_to_bf16_bits(rng.normal(0, 0.5, c.out_total).astype(np.float32))
    y = oracle.linear(c, c.W, bias)
    x = bf16_bits_to_f32(c.x).astype(np.float64)
    W = bf16_bits_to_f32(c.W).astype(np.float64)
    b = bf16_bits_to_f32(bias).astype(np.float64)
    _, bound = exact_dense(c)
    for t in range(c.T):
        a = int(c.idx[t])
        merged = W
        if 0 <= a < c.L and c.enabled[a] and c.ranks[a] > 0:
            r = int(c.ranks[a])
            merged = W + c.scales[a] * (bf16_bits_to_f32(c.B[0][a, :, :r]).astype(np.float64)
                                        @ bf16_bits_to_f32(c.A[0][a, :r]).astype(np.float64))
        want = x[t] @ merged.T + b
        assert np.all(np.abs(y[t] - want) <= bound[t] + 1e-9), t
