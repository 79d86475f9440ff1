"""Fused-MoE LoRA on the GPU (lora_moe_apply W13 and W2) against the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
from gpu_util import assert_base_plus_delta, assert_delta, assert_rows_untouched

pytestmark = pytest.mark.gpu


def pair_active(c, enabled=None):
    en = c.enabled if enabled is None else enabled
    t = np.repeat(np.arange(c.T), c.K)
    a = c.idx[t]
    ok = (a >= 0) & (a < c.L)
    act = np.zeros(c.T * c.K, bool)
    act[ok] = (en[a[ok]] != 0) & (c.ranks[a[ok]] > 0)
    e = c.topk_ids.reshape(-1)
    return act & (e >= 0) & (e < c.E)


def run_and_check(c, base_random=False):
    run = H.MoERun(c)
    try:
        run.step()
        ic1 = H.from_dev_u16(run.ic1)
        ic3 = H.from_dev_u16(run.ic3)
        assert run.status() == 0
    finally:
        run.close()
    act = pair_active(c)
    _, d13 = oracle.moe_w13(c)
    _, d2 = oracle.moe_w2(c)
    assert_rows_untouched(ic1, c.ic1_0, ~act)
    assert_rows_untouched(ic3, c.ic3_0, ~act)
    if base_random:
        assert_base_plus_delta(ic1, c.ic1_0, d13, act)
        assert_base_plus_delta(ic3, c.ic3_0, d2, act)
        return
    assert_delta(bf16_bits_to_f32(ic1)[act], d13[act], c.name + " w13")
    assert_delta(bf16_bits_to_f32(ic3)[act], d2[act], c.name + " w2")


@pytest.mark.parametrize("shared", [False, True])
def test_preset_moe(shared):
    run_and_check(gen.moe(shared_outer=shared))


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_small_moe(seed, shared):
    c = gen.moe_case(name=f"moe_small{seed}", T=90, K=3, E=6, D=1040, F=272, L=4, R=24, seed=seed,
                     shared_outer=shared, ranks=(24, 9, 16, 0), scales=(1.5, 0.5, 2.0, 1.0), p_none=0.1)
    run_and_check(c)


def test_moe_random_base():
    c = gen.moe_case(name="moe_base", T=40, K=2, E=4, D=512, F=256, L=3, R=16, seed=4, base="random")
    run_and_check(c, base_random=True)


def test_moe_3d_single_slice_layout():
    """FusedMoE3DWithLoRA: one w13 slice whose B stacks gate and up (2F rows)."""
    c = gen.moe_case(name="moe3d", T=64, K=4, E=8, D=512, F=128, L=3, R=16, seed=5, n13=1, f13=256)
    run_and_check(c)


def test_moe_non_gated():
    c = gen.moe_case(name="moe_ng", T=64, K=2, E=8, D=512, F=128, L=3, R=16, seed=6, n13=1)
    run_and_check(c)


def test_moe_one_expert_top1():
    c = gen.moe_case(name="moe_e1", T=33, K=1, E=1, D=256, F=128, L=3, R=8, seed=7, p_none=0.3)
    run_and_check(c)


def test_moe_disabled_adapter():
    c = gen.moe_case(name="moe_dis", T=50, K=2, E=4, D=256, F=128, L=3, R=8, seed=8, base="random")
    run = H.MoERun(c)
    try:
        from heterogeneous_adapters_lora_gb300 import lora as L
        L.lora_reset(run.pool, 1)
        run.step()
        ic1 = H.from_dev_u16(run.ic1)
        ic3 = H.from_dev_u16(run.ic3)
    finally:
        run.close()
    en = c.enabled.copy()
    en[1] = 0
    act = pair_active(c, en)
    _, d13 = oracle.moe_w13(c, enabled=en)
    _, d2 = oracle.moe_w2(c, enabled=en)
    assert_rows_untouched(ic1, c.ic1_0, ~act)
    assert_rows_untouched(ic3, c.ic3_0, ~act)
    assert_base_plus_delta(ic1, c.ic1_0, d13, act)
    assert_base_plus_delta(ic3, c.ic3_0, d2, act)


@pytest.mark.parametrize("T", [1, 16])
def test_moe_decode_sparse_keys(T):
    """Decode-size MoE batches: T*K pairs over 512 (adapter, expert) keys, most
    keys empty or with one pair (the sparse-occupancy regime)."""
    run_and_check(gen.moe(T=T))


@pytest.mark.parametrize("shared", [False, True])
def test_out_of_range_ids_are_skipped_and_reported(shared):
    # expert ids -1 and E, and slot ids L and -5, on some rows: those pairs get
    # no delta (their rows stay bit-identical), the rest match the oracle, and
    # the device status reports the bad ids
    c = gen.moe_case(name="moe_bad_ids", T=70, K=3, E=6, D=1040, F=272, L=4, R=16, seed=41, shared_outer=shared,
                     scales=(1.5, 0.5, 2.0, 1.0), p_none=0.1)
    c.topk_ids[3, 0] = -1
    c.topk_ids[10, 2] = c.E
    c.topk_ids[11, 1] = c.E + 7
    c.idx[20] = c.L
    c.idx[21] = -5
    run = H.MoERun(c)
    try:
        run.step()
        ic1 = H.from_dev_u16(run.ic1)
        ic3 = H.from_dev_u16(run.ic3)
        st = run.status()
    finally:
        run.close()
    assert st == H.L.CODE["LORA_ERR_DEVICE_INDEX"]
    act = pair_active(c)
    assert not act[3 * c.K] and not act[10 * c.K + 2] and not act[20 * c.K]
    _, d13 = oracle.moe_w13(c)
    _, d2 = oracle.moe_w2(c)
    assert_rows_untouched(ic1, c.ic1_0, ~act)
    assert_rows_untouched(ic3, c.ic3_0, ~act)
    assert_delta(bf16_bits_to_f32(ic1)[act], d13[act], "bad ids w13")
    assert_delta(bf16_bits_to_f32(ic3)[act], d2[act], "bad ids w2")


@pytest.mark.parametrize("policy", [0, 2])
@pytest.mark.parametrize("T", [613, 2500])
def test_shared_outer_shrink_once_per_token(T, policy):
    """Shared-outer w13 (A with expert dimension 1): the shrink runs once per
    token, on slots as keys, with each slot's tokens gathered from its pair
    range.  Skewed slots (several CTAs share a slot's tiles), a ragged tail, a
    token whose first routed pair is dropped, a token with every pair dropped
    and one outside any slot; w2 is the per-expert path on the same batch.
    Policy 2 runs the same batch on the one-pass cluster kernel."""
    from heterogeneous_adapters_lora_gb300 import lora as L
    c = gen.moe_case(name="moe_tok", T=T, K=4, E=8, D=1040, F=272, L=3, R=16, seed=61 + T, shared_outer=True,
                     ranks=(16, 8, 12), scales=(1.0, 0.5, 2.0), p_none=0.05)
    rng = np.random.default_rng(T)
    c.idx[:] = np.where(rng.random(c.T) < 0.7, 0, c.idx)  # most tokens on slot 0
    c.idx[7] = -1
    c.idx[5] = 0
    c.idx[9] = 1
    c.topk_ids[5, 0] = -1
    c.topk_ids[9, :] = c.E
    L.lora_set_kernel_policy(policy)
    run = H.MoERun(c)
    try:
        run.step()
        ic1 = H.from_dev_u16(run.ic1)
        ic3 = H.from_dev_u16(run.ic3)
        st = run.status()
    finally:
        run.close()
        L.lora_set_kernel_policy(0)
    assert st == H.L.CODE["LORA_ERR_DEVICE_INDEX"]
    act = pair_active(c)
    assert not act[5 * c.K] and act[5 * c.K + 1] and not act[9 * c.K:10 * c.K].any()
    _, d13 = oracle.moe_w13(c)
    _, d2 = oracle.moe_w2(c)
    assert_rows_untouched(ic1, c.ic1_0, ~act)
    assert_rows_untouched(ic3, c.ic3_0, ~act)
    assert_delta(bf16_bits_to_f32(ic1)[act], d13[act], "token shrink w13")
    assert_delta(bf16_bits_to_f32(ic3)[act], d2[act], "token shrink w2")
