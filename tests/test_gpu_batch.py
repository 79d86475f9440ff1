"""lora_build_meta_apply: the metadata build and one dense layer's delta in
one call (one launch when the fused decode kernel takes the batch).  The
metadata must equal the oracle's bit for bit, the delta must match the
oracle, and y must equal the two-call path (lora_build_meta, then
lora_apply_slices) bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
from gpu_util import (active_mask, assert_base_plus_delta, assert_delta, assert_rows_untouched, long_short_tiles,
                      tile_keyn, tiles_from_groups)

pytestmark = pytest.mark.gpu


def _check_meta(got, c, en):
    ref = oracle.dense_meta(c.idx, c.L, en, c.ranks)
    assert np.array_equal(got["sorted"], ref.sorted_tok)
    assert (got["n_active"], got["n_groups"], got["n_bad"]) == (ref.n_active, ref.n_seg, ref.n_bad)
    assert np.array_equal(got["key_count"], ref.slot_count)
    assert np.array_equal(got["key_offset"], np.concatenate([[0], np.cumsum(ref.slot_count)]))
    assert np.array_equal(got["group_key"], ref.seg_slot)
    assert np.array_equal(got["group_start"], ref.seg_start)
    assert np.array_equal(got["key_group"], ref.slot_seg)
    tg, tr = tiles_from_groups(ref.seg_start)
    assert got["n_tiles"] == len(tg)
    assert np.array_equal(got["tile_group"], tg) and np.array_equal(got["tile_row0"], tr)
    assert np.array_equal(got["tile_keyn"], tile_keyn(tg, tr, ref.seg_slot, ref.seg_start))
    lt, st = long_short_tiles(ref.seg_slot, ref.seg_start, ref.sorted_tok)
    assert got["n_ltiles"] == len(lt) and got["n_stiles"] == len(st)
    if lt:
        assert np.array_equal(got["ltile_row0"], [x[0] for x in lt])
        assert np.array_equal(got["ltile_keyn"], [x[1] for x in lt])
        assert np.array_equal(got["ltile_tok0"], [x[2] for x in lt])
    if st:
        assert np.array_equal(got["stile_row0"], [x[0] for x in st])
        assert np.array_equal(got["stile_keyn"], [x[1] for x in st])
    return ref


def _run(c, expect_one_launch, base_random=False, reset_slot=None):
    en = c.enabled.copy()
    if reset_slot is not None:
        en[reset_slot] = 0
    out = {}
    for mode in ("batch", "two_calls"):
        run = H.DenseRun(c)
        try:
            if reset_slot is not None:
                L.lora_reset(run.pool, reset_slot)
            torch.cuda.synchronize()
            n0 = L.lora_kernel_launch_count()
            if mode == "batch":
                run.step_batch()
            else:
                run.step()
            torch.cuda.synchronize()
            out[mode] = (run.y_host(), run.mb.read(), run.status(), L.lora_kernel_launch_count() - n0)
        finally:
            run.close()
    y, meta, st, n = out["batch"]
    if expect_one_launch:
        assert n == 1, f"expected one launch, got {n}"
    ref = _check_meta(meta, c, en)
    assert st == (L.CODE["LORA_ERR_DEVICE_INDEX"] if ref.n_bad else 0)
    assert np.array_equal(y, out["two_calls"][0]), "batch call and two calls differ"
    _, d_ref = oracle.dense_delta(c, enabled=en)
    act = active_mask(c.idx, c.L, en, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    if base_random:
        assert_base_plus_delta(y, c.y0, d_ref, act)
    else:
        assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], c.name)


def test_decode_qkv_one_launch():
    _run(gen.decode_qkv(), True)


def test_decode_qkv_random_base():
    _run(gen.decode_qkv(base_y="random"), True, base_random=True)


def test_tiny_one_launch():
    _run(gen.tiny(), True)


@pytest.mark.parametrize("T", [120, 1024])
def test_several_row_steps_and_tiles(T):
    # up to 1024 rows: four row steps of the 256-thread metadata CTA, slots
    # with many 16-row tiles
    rng = np.random.default_rng(T)
    Lk = 32 if T == 1024 else 4
    idx = rng.integers(0, Lk, T).astype(np.int32)
    idx[rng.random(T) < 0.3] = 0
    idx[rng.random(T) < 0.05] = -1
    c = gen.dense_case(name=f"batch{T}", T=T, H=1024, out_dims=(512, 256), L=Lk, R=16, seed=80, idx=idx,
                       scales=np.linspace(0.5, 2.0, Lk).astype(np.float32))
    # 30 and 32 rows per slot: past the automatic choice's 16, kept on the
    # fused kernel by policy 7
    L.lora_set_kernel_policy(7)
    try:
        _run(c, True)
    finally:
        L.lora_set_kernel_policy(0)


def test_bad_indices_and_reset_slot():
    c = gen.dense_case(name="batch_bad", T=96, H=2048, out_dims=(256, 128, 128), L=8, R=16, seed=81,
                       scales=np.full(8, 1.5, np.float32), p_none=0.1)
    c.idx[5] = 8
    c.idx[17] = -3
    _run(c, True, reset_slot=2)


def test_falls_back_to_two_launches():
    # a batch the fused kernel does not take (hidden size not in 64-column chunks)
    c = gen.dense_case(name="batch_fallback", T=100, H=1032, out_dims=(136, 264), L=5, R=24, seed=82,
                       ranks=(24, 13, 1, 8, 0), scales=(1.0, 2.0, 0.5, 1.5, 1.0), p_none=0.15)
    _run(c, False)


def test_long_run_slots_in_batch_mode():
    # a slot whose 64+ rows form one contiguous run: the long-tile lists of
    # the metadata come from the same block build
    idx = np.full(256, -1, np.int32)
    idx[0:100] = 1
    idx[100:180] = 2
    idx[180:200] = 0
    idx[200:256:3] = 3
    c = gen.dense_case(name="batch_runs", T=256, H=1024, out_dims=(256,), L=8, R=16, seed=83, idx=idx,
                       scales=np.ones(8, np.float32))
    L.lora_set_kernel_policy(7)  # 32 rows per slot: past the automatic choice's 16
    try:
        _run(c, True)
    finally:
        L.lora_set_kernel_policy(0)
    _run(c, False)  # the automatic choice: metadata build, then the split kernels
