"""The tensor-core (tcgen05) path for long contiguous token runs, checked
against the oracle: full 128-token tiles, a partial last tile of a run, and
groups that stay on the short-tile path (two runs in one slot, a run shorter
than 64 tokens) in the same call."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
from gpu_util import active_mask, assert_base_plus_delta, assert_delta, assert_rows_untouched

pytestmark = pytest.mark.gpu


def mixed_idx():
    idx = np.full(760, -1, np.int32)
    idx[0:300] = 0            # 128 + 128 + 44: two full tiles and a partial one
    idx[300:500] = 1          # 128 + 72
    idx[520:570] = 2          # two runs of slot 2: short tiles
    idx[600:650] = 2
    idx[700:740] = 3          # 40 tokens: below the long-run threshold
    return idx


def _run(c):
    run = H.DenseRun(c)
    try:
        run.step()
        y = run.y_host()
        meta = run.mb.read()
        assert run.status() == 0
    finally:
        run.close()
    return y, meta


@pytest.mark.parametrize("base", ["zero", "random"])
def test_long_runs_and_short_groups_together(base):
    c = gen.dense_case(name="sgmv_mixed", T=760, H=512, out_dims=(256, 384), L=4, R=64, seed=51,
                       idx=mixed_idx(), scales=(1.0, 2.0, 0.5, 1.5), base_y=base)
    y, meta = _run(c)
    assert meta["n_ltiles"] == 5 and meta["n_stiles"] > 0
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    if base == "zero":
        assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "mixed")
    else:
        assert_base_plus_delta(y, c.y0, d_ref, act)


def test_prefill_preset_matches_split_k_kernel():
    c = gen.prefill_gate_up()
    y_tc, meta = _run(c)
    assert meta["n_ltiles"] > 0 and meta["n_stiles"] == 0
    L.lora_set_kernel_policy(1)
    try:
        y_sk, _ = _run(c)
    finally:
        L.lora_set_kernel_policy(0)
    _, d_ref = oracle.dense_delta(c)
    assert_delta(bf16_bits_to_f32(y_tc), d_ref, "tcgen05")
    assert_delta(bf16_bits_to_f32(y_sk), d_ref, "split-K")


@pytest.mark.parametrize("ranks", [(64, 32, 64, 16), (8, 40, 24, 56)], ids=["64-32-64-16", "8-40-24-56"])
def test_mixed_ranks_on_the_tensor_core_path(ranks):
    """A max_rank-64 pool whose slots have other ranks: the long runs stay on
    tcgen05 (each slot's compact B rows are read through the map of its row
    length; the ranks past a slot's rank read as zero)."""
    c = gen.dense_case(name="sgmv_ranks", T=760, H=512, out_dims=(256, 384), L=4, R=64, seed=52,
                       idx=mixed_idx(), ranks=ranks, scales=(1.0, 2.0, 0.5, 1.5))
    y, meta = _run(c)
    assert meta["n_ltiles"] == 5
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "mixed ranks")


@pytest.mark.parametrize("R", [16, 24, 48])
def test_pools_below_rank_64_on_the_tensor_core_path(R):
    """max_rank 16, 24 and 48: the shrink's MMA N is ceil16(R) and v is laid
    out as 64 hi + 64 lo columns, zero past the rank."""
    c = gen.dense_case(name=f"sgmv_r{R}", T=760, H=1024, out_dims=(384, 128), L=4, R=R, seed=53 + R,
                       idx=mixed_idx(), ranks=(R, R, max(1, R // 2), R), scales=(1.0, 2.0, 0.5, 1.5))
    y, meta = _run(c)
    assert meta["n_ltiles"] == 5
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], f"max_rank {R}")
