"""Host-checked argument errors, the device status word, and the bounded-wait
error path of the fused kernels (no GPU fault is ever provoked: every failure
is either rejected on the host or reported through the status word)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
from gpu_util import active_mask, assert_delta

pytestmark = pytest.mark.gpu


def code(name):
    return L.CODE[name]


def small():
    return gen.dense_case(name="err", T=40, H=256, out_dims=(64, 64), L=4, R=16, seed=1, p_none=0.1)


def test_set_rejects_bad_slot_and_rank():
    c = small()
    run = H.DenseRun(c)
    try:
        A = [np.zeros((8, 256), np.uint16)] * 2
        B = [np.zeros((64, 8), np.uint16)] * 2
        for slot in (-1, 4):
            with pytest.raises(L.LoraError) as e:
                L.lora_set(run.pool, slot, 8, 1.0, A, B)
            assert e.value.code == code("LORA_ERR_INDEX")
        with pytest.raises(L.LoraError) as e:
            L.lora_set(run.pool, 0, 17, 1.0, A, B)
        assert e.value.code == code("LORA_ERR_RANK")
        with pytest.raises(L.LoraError) as e:
            L.lora_set(run.pool, 0, 8, 1.0, A[:1], B[:1])
        assert e.value.code == code("LORA_ERR_SHAPE")
        with pytest.raises(L.LoraError) as e:
            L.lora_reset(run.pool, 9)
        assert e.value.code == code("LORA_ERR_INDEX")
    finally:
        run.close()


def test_lm_head_vocab_guard():
    d = L.PoolDesc()
    d.max_loras, d.max_rank, d.in_dim, d.n_slices, d.is_lm_head = 2, 8, 64, 1, 1
    d.out_dims[0] = 257024 + 8
    with pytest.raises(L.LoraError) as e:
        L.lora_pool_create(d)
    assert e.value.code == code("LORA_ERR_SHAPE")
    d.out_dims[0] = 257024
    L.lora_pool_destroy(L.lora_pool_create(d))


def test_moe_layout_mismatch():
    c = gen.moe_case(T=8, K=2, E=4, D=64, F=32, L=2, R=8, seed=2, shared_outer=True)
    run = H.MoERun(c)
    try:
        r = 8
        A = [np.zeros((4, r, 64), np.uint16), np.zeros((1, r, 64), np.uint16), np.zeros((4, r, 32), np.uint16)]
        B = [np.zeros((4, 32, r), np.uint16), np.zeros((4, 32, r), np.uint16), np.zeros((1, 64, r), np.uint16)]
        with pytest.raises(L.LoraError) as e:   # per-expert w13-A into a shared-outer pool
            L.lora_set_moe(run.pool, 0, r, 1.0, A, [4, 1, 4], B, [4, 4, 1])
        assert e.value.code == code("LORA_ERR_LAYOUT")
        with pytest.raises(L.LoraError) as e:   # wrong expert count
            L.lora_set_moe(run.pool, 0, r, 1.0, A, [1, 1, 3], B, [4, 4, 1])
        assert e.value.code == code("LORA_ERR_SHAPE")
    finally:
        run.close()


def test_alignment_and_capacity_errors():
    c = small()
    run = H.DenseRun(c)
    try:
        run.build_meta()
        with pytest.raises(L.LoraError) as e:   # x not 16-byte aligned
            L.lora_apply_slices(run.pool, run.mb.meta, run.x.data_ptr() + 2, c.H, run.y, c.out_total,
                                run.ws, run.ws_bytes)
        assert e.value.code == code("LORA_ERR_INVALID_ARG")
        with pytest.raises(L.LoraError) as e:   # workspace too small
            L.lora_apply_slices(run.pool, run.mb.meta, run.x, c.H, run.y, c.out_total, run.ws, 64)
        assert e.value.code == code("LORA_ERR_CAPACITY")
        small_meta = H.MetaBuffer(8, c.L)
        with pytest.raises(L.LoraError) as e:   # more tokens than the meta holds
            L.lora_build_meta(run.pool, run.idx, c.T, None, 1, small_meta.meta)
        assert e.value.code == code("LORA_ERR_CAPACITY")
    finally:
        run.close()


def test_bad_index_sets_device_status_and_row_is_skipped():
    c = small()
    c.idx[3] = 99
    c.idx[5] = -7
    run = H.DenseRun(c)
    try:
        run.step()
        assert run.status() == code("LORA_ERR_DEVICE_INDEX")
        assert run.status() == 0           # cleared by the read
        y = run.y_host()
    finally:
        run.close()
    assert np.array_equal(y[[3, 5]], c.y0[[3, 5]])
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "bad idx")


def test_wait_that_gives_up_reports_timeout_and_leaves_workspace_clean():
    """Every cross-CTA wait made to give up at once: the call returns, the
    status says LORA_ERR_TIMEOUT or OK (if every wait was already satisfied),
    and the next normal call is exact again."""
    c = gen.decode_qkv()
    run = H.DenseRun(c)
    try:
        run.build_meta()
        L.lora_set_spin_limit(-1)
        try:
            run.apply()
            st = run.status()
        finally:
            L.lora_set_spin_limit(1 << 20)
        assert st in (0, code("LORA_ERR_TIMEOUT"))
        run.y.zero_()
        run.apply()
        assert run.status() == 0
        y = run.y_host()
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "after timeout")
