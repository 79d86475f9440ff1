"""Leading dimensions wider than the layer (a serving stack's x and y are
often column views into wider fused buffers): every compute path must read
only the layer's columns of x / ic2 and write only the layer's columns of
y / ic1 / ic3.  Padding columns hold a NaN pattern, so a kernel that read
them into a product would show NaNs; written padding would differ from it."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
from gpu_util import active_mask, assert_delta, assert_rows_untouched

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[0, 1, 2, 3], ids=["auto", "splitk", "cluster", "split"])
def policy(request):
    L.lora_set_kernel_policy(request.param)
    yield request.param
    L.lora_set_kernel_policy(0)


def _dense(c, x_pad, y_pad, expect_ltiles=None):
    run = H.DenseRun(c, x_pad=x_pad, y_pad=y_pad)
    try:
        run.step()
        yf = run.y_full_host()
        meta = run.mb.read()
        assert run.status() == 0
    finally:
        run.close()
    if expect_ltiles is not None:
        assert (meta["n_ltiles"] > 0) == expect_ltiles
    assert np.all(yf[:, c.out_total:] == H.PAD_BITS), "padding columns of y were written"
    y = np.ascontiguousarray(yf[:, :c.out_total])
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], f"{c.name} ldx+{x_pad} ldy+{y_pad}")


def test_decode_qkv_padded(policy):
    _dense(gen.decode_qkv(), x_pad=72, y_pad=24)


def test_multi_tile_padded(policy):
    c = gen.dense_case(name="smt_pad", T=150, H=2056, out_dims=(264, 136, 80), L=4, R=24, seed=43,
                       ranks=(24, 13, 1, 8), scales=(1.0, 0.5, 2.0, 1.5), p_none=0.1)
    _dense(c, x_pad=8, y_pad=64)


def test_per_tile_items_padded():
    # many slots, few rows each: the per-tile shrink (copy warp, ranks taken
    # 16 at a time) and the expand over 16-row tiles
    ranks = tuple((64, 40, 57, 1, 24, 33, 16, 0)[i % 8] for i in range(1024))
    c = gen.dense_case(name="per_tile_pad", T=512, H=1024, out_dims=(264,), L=1024, R=64, seed=33,
                       ranks=ranks, scales=np.ones(1024, np.float32), p_none=0.1)
    _dense(c, x_pad=24, y_pad=8)


def test_one_item_per_cta_padded():
    c = gen.dense_case(name="tile_static_pad", T=8, H=3000, out_dims=(264,), L=8, R=64, seed=23,
                       ranks=(64, 40, 57, 1, 24, 33, 16, 0), scales=np.ones(8, np.float32), p_none=0.1)
    _dense(c, x_pad=16, y_pad=16)


def test_tensor_core_runs_padded():
    # long contiguous runs of a rank-64 pool: tcgen05 shrink/expand (TMA
    # tensor maps over the padded row strides), short tiles on the other kernels
    idx = np.full(760, -1, np.int32)
    idx[0:300] = 0
    idx[300:500] = 1
    idx[520:570] = 2
    idx[600:650] = 2
    idx[700:740] = 3
    c = gen.dense_case(name="sgmv_pad", T=760, H=512, out_dims=(256, 384), L=4, R=64, seed=53, idx=idx,
                       scales=(1.0, 2.0, 0.5, 1.5))
    _dense(c, x_pad=64, y_pad=128, expect_ltiles=True)


def test_standalone_shrink_expand_padded():
    c = gen.dense_case(name="shrink_pad", T=90, H=1032, out_dims=(136, 72), L=4, R=16, seed=44,
                       ranks=(16, 5, 0, 9), scales=(1.0, 2.0, 1.0, 0.5), p_none=0.1)
    run = H.DenseRun(c, x_pad=40, y_pad=56)
    try:
        run.build_meta()
        v = torch.empty((c.n_slices, c.T, c.R), dtype=torch.float32, device="cuda")
        L.lora_shrink(run.pool, run.mb.meta, run.x, run.ldx, v)
        L.lora_expand(run.pool, run.mb.meta, v, run.y, run.ldy)
        yf = run.y_full_host()
    finally:
        run.close()
    assert np.all(yf[:, c.out_total:] == H.PAD_BITS)
    y = np.ascontiguousarray(yf[:, :c.out_total])
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "shrink+expand padded")


@pytest.mark.parametrize("shared", [False, True])
def test_moe_padded(shared, policy):
    c = gen.moe_case(name="moe_pad", T=90, K=3, E=6, D=1040, F=272, L=4, R=24, seed=7, shared_outer=shared,
                     ranks=(24, 9, 16, 0), scales=(1.5, 0.5, 2.0, 1.0), p_none=0.1)
    run = H.MoERun(c, in_pad=24, out_pad=40)
    try:
        run.step()
        ic1f = H.from_dev_u16(run.ic1)
        ic3f = H.from_dev_u16(run.ic3)
        assert run.status() == 0
    finally:
        run.close()
    W13 = c.n13 * c.F13
    assert np.all(ic1f[:, W13:] == H.PAD_BITS) and np.all(ic3f[:, c.D:] == H.PAD_BITS)
    ic1 = np.ascontiguousarray(ic1f[:, :W13])
    ic3 = np.ascontiguousarray(ic3f[:, :c.D])
    t = np.repeat(np.arange(c.T), c.K)
    a = c.idx[t]
    act = (a >= 0) & (a < c.L)
    act[act] &= (c.enabled[a[act]] != 0) & (c.ranks[a[act]] > 0)
    _, d13 = oracle.moe_w13(c)
    _, d2 = oracle.moe_w2(c)
    assert_rows_untouched(ic1, c.ic1_0, ~act)
    assert_rows_untouched(ic3, c.ic3_0, ~act)
    assert_delta(bf16_bits_to_f32(ic1)[act], d13[act], "w13 padded")
    assert_delta(bf16_bits_to_f32(ic3)[act], d2[act], "w2 padded")
