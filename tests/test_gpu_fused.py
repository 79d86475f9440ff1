"""The fused decode kernel (one thread-block cluster per adapter slot:
shrink, on-chip reduction over the cluster and expand in one launch)
against the oracle, and against the split kernels on the same inputs.

Each case checks that the automatic path really launched one kernel for the
apply (the fused kernel), and covers a shape feature of its plan: slots with
several 16-row tiles, ranks that end inside an MMA block, output blocks that
straddle slice boundaries, CTAs whose hidden chunk or output block is empty,
disabled and reset slots, a random base, and repeated calls."""
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


def _apply_launches(run):
    run.build_meta()
    torch.cuda.synchronize()
    n0 = L.lora_kernel_launch_count()
    run.apply()
    torch.cuda.synchronize()
    return L.lora_kernel_launch_count() - n0


def _run(c, base_random=False, expect_fused=True, **kw):
    run = H.DenseRun(c, **kw)
    try:
        n = _apply_launches(run)
        y = run.y_host()
        assert run.status() == 0
    finally:
        run.close()
    if expect_fused:
        assert n == 1, f"expected the fused kernel (one launch), got {n}"
    y_ref, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    if base_random:
        assert_base_plus_delta(y, c.y0, d_ref, act)
    else:
        assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], c.name)
    return y


def test_decode_qkv_is_fused():
    _run(gen.decode_qkv())


def test_decode_qkv_random_base():
    _run(gen.decode_qkv(base_y="random"), base_random=True)


@pytest.mark.parametrize("seed", [0, 1])
def test_several_tiles_per_slot(seed):
    # 120 rows over 4 slots, half of them on slot 0: slots of 2 to 5 tiles,
    # the last tile of each partial
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, 4, 120).astype(np.int32)
    idx[rng.random(120) < 0.5] = 0
    idx[rng.random(120) < 0.05] = -1
    c = gen.dense_case(name=f"tiles{seed}", T=120, H=1024, out_dims=(512, 256), L=4, R=16, seed=60 + seed,
                       idx=idx, scales=(1.0, 2.0, 0.5, 1.5))
    L.lora_set_kernel_policy(7)  # 30 rows per slot: past the automatic choice's 16
    try:
        _run(c)
    finally:
        L.lora_set_kernel_policy(0)
    _run(c, expect_fused=False)


def test_mixed_ranks_straddling_blocks():
    # ranks 1..64 (ends inside 8- and 16-rank blocks), slices whose
    # boundaries fall inside the CTAs' output blocks
    ranks = (64, 1, 13, 24, 40, 8, 57, 16)
    c = gen.dense_case(name="mixed_ranks", T=128, H=1024, out_dims=(136, 264, 72), L=8, R=64, seed=62,
                       ranks=ranks, scales=np.linspace(0.5, 2.0, 8).astype(np.float32), p_none=0.1)
    # 3 slices x 64 ranks exceed the fused plan's 8 MMA row blocks: it must fall back
    _run(c, expect_fused=False)
    c2 = gen.dense_case(name="mixed_ranks2", T=128, H=1024, out_dims=(160, 288), L=8, R=64, seed=63,
                        ranks=ranks, scales=np.linspace(0.5, 2.0, 8).astype(np.float32), p_none=0.1)
    _run(c2)


@pytest.mark.parametrize("R,ranks", [(32, (32, 24, 17, 9)), (8, (8, 3, 1, 5)), (12, (12, 7, 0, 11))])
def test_rank_classes(R, ranks):
    # rank <= 8 (8-row A boxes), 12 (16-row boxes that reach into the next
    # slot's rows) and 32 (two boxes per slice, two 16-rank expand k steps)
    c = gen.dense_case(name=f"rank{R}", T=64, H=2048, out_dims=(192, 320), L=4, R=R, seed=67 + R, ranks=ranks,
                       scales=(1.0, 2.0, 0.5, 1.5), p_none=0.1)
    _run(c)


def test_hidden_not_in_64_column_chunks_falls_back():
    c = gen.dense_case(name="h1032", T=64, H=1032, out_dims=(128,), L=4, R=16, seed=70, p_none=0.1)
    _run(c, expect_fused=False)


def test_slices_not_in_32_column_groups_fall_back():
    c = gen.dense_case(name="o136", T=64, H=1024, out_dims=(136, 264), L=4, R=16, seed=71, p_none=0.1)
    _run(c, expect_fused=False)


def test_tiny_preset_is_fused():
    _run(gen.tiny())


def test_empty_chunks_and_blocks():
    # H = 64 and 64 outputs over clusters of 8 CTAs: most CTAs have no hidden
    # chunk and no output block
    c = gen.dense_case(name="tiny_dims", T=40, H=64, out_dims=(32, 32), L=4, R=8, seed=64, ranks=(8, 5, 0, 3),
                       scales=(1.0, 2.0, 1.0, 0.5), p_none=0.1)
    _run(c)


def test_disabled_and_reset_slots():
    c = gen.dense_case(name="disabled", T=96, H=2048, out_dims=(256, 128, 128), L=8, R=16, seed=65,
                       scales=np.full(8, 1.5, np.float32), p_none=0.1)
    c.enabled[3] = 0
    run = H.DenseRun(c)
    try:
        L.lora_reset(run.pool, 5)
        n = _apply_launches(run)
        y = run.y_host()
        assert run.status() == 0
    finally:
        run.close()
    assert n == 1
    en = c.enabled.copy()
    en[5] = 0
    _, d_ref = oracle.dense_delta(c, enabled=en)
    act = active_mask(c.idx, c.L, en, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "disabled/reset")


def test_fused_matches_split_kernels_and_is_deterministic():
    c = gen.decode_qkv(base_y="random")
    outs = []
    for pol in (0, 0, 3):
        L.lora_set_kernel_policy(pol)
        try:
            run = H.DenseRun(c)
            try:
                run.step()
                outs.append(run.y_host())
            finally:
                run.close()
        finally:
            L.lora_set_kernel_policy(0)
    assert np.array_equal(outs[0], outs[1]), "fused kernel not deterministic"
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    base = bf16_bits_to_f32(c.y0)[act].astype(np.float64)
    assert_delta(bf16_bits_to_f32(outs[0])[act] - base, bf16_bits_to_f32(outs[2])[act] - base, "fused vs split")


def test_repeated_calls_accumulate():
    c = gen.dense_case(name="rep", T=64, H=1024, out_dims=(256,), L=8, R=16, seed=66, p_none=0.0,
                       scales=np.ones(8, np.float32))
    run = H.DenseRun(c)
    try:
        run.build_meta()
        for _ in range(4):
            run.apply()
        y = run.y_host()
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    assert_delta(bf16_bits_to_f32(y), 4 * d_ref, "4 calls")
