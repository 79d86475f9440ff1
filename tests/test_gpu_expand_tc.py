"""The split expand on tcgen05 (bgmv_expand_tc_kernel: 128-output MMA blocks,
16 rows per tile, ranks on K) against the oracle, and against the expand on
warp-level MMAs (kernel policy 8) on the same inputs.  The tensor-core expand
runs when every slice width is a multiple of 128: mixed ranks (a rank step of
8 past a multiple of 16 takes a zeroed chunk), 4 and 2 blocks per item, dense
and MoE pools (per expert and shared-outer), padded leading dimensions."""
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


@pytest.fixture(params=[3, 8], ids=["tensor_core", "warp_mma"])
def policy(request):
    L.lora_set_kernel_policy(request.param)
    yield request.param
    L.lora_set_kernel_policy(0)


def _dense(c, x_pad=0, y_pad=0, base_random=False):
    run = H.DenseRun(c, x_pad=x_pad, y_pad=y_pad)
    try:
        run.step()
        yf = run.y_full_host()
        assert run.status() == 0
    finally:
        run.close()
    if y_pad:
        assert np.all(yf[:, c.out_total:] == H.PAD_BITS), "padding columns of y were written"
    y = np.ascontiguousarray(yf[:, :c.out_total])
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    if base_random:
        assert_base_plus_delta(y, c.y0, d_ref, act)
    else:
        assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], c.name)


def test_dense_mixed_ranks_four_blocks(policy):
    # ranks <= 32: items of 512 outputs (4 blocks), slices 512 / 128 / 128
    c = gen.dense_case(name="tc_qkv", T=300, H=1024, out_dims=(512, 128, 128), L=6, R=32, seed=71,
                       ranks=(32, 24, 16, 8, 1, 0), scales=(1.0, 0.5, 2.0, 1.5, 3.0, 1.0), p_none=0.1)
    _dense(c)


def test_dense_mixed_ranks_two_blocks_padded(policy):
    # ranks up to 64: items of 256 outputs (2 blocks), four 16-rank steps
    c = gen.dense_case(name="tc_r64", T=260, H=1536, out_dims=(384, 256), L=7, R=64, seed=72,
                       ranks=(64, 56, 40, 24, 17, 9, 0), scales=(1.0, 0.5, 2.0, 1.5, 1.0, 2.5, 1.0), p_none=0.05)
    _dense(c, x_pad=24, y_pad=40)


def test_dense_random_base(policy):
    c = gen.dense_case(name="tc_base", T=200, H=512, out_dims=(256, 256), L=4, R=16, seed=73,
                       ranks=(16, 8, 12, 16), base_y="random")
    _dense(c, base_random=True)


@pytest.mark.parametrize("shared", [False, True])
def test_moe_widths_of_128(shared, policy):
    c = gen.moe_case(name="tc_moe", T=150, K=4, E=8, D=512, F=384, L=3, R=24, seed=74, shared_outer=shared,
                     ranks=(24, 16, 8), scales=(1.0, 0.5, 2.0), p_none=0.05, base="random")
    run = H.MoERun(c, in_pad=8, out_pad=24)
    try:
        run.step()
        ic1 = np.ascontiguousarray(H.from_dev_u16(run.ic1)[:, :c.n13 * c.F13])
        ic3 = np.ascontiguousarray(H.from_dev_u16(run.ic3)[:, :c.D])
        assert run.status() == 0
    finally:
        run.close()
    t = np.repeat(np.arange(c.T), c.K)
    a = c.idx[t]
    act = (a >= 0) & (a < c.L)
    act[act] &= (c.enabled[a[act]] != 0) & (c.ranks[a[act]] > 0)
    _, d13 = oracle.moe_w13(c)
    _, d2 = oracle.moe_w2(c)
    assert_rows_untouched(ic1, c.ic1_0, ~act)
    assert_rows_untouched(ic3, c.ic3_0, ~act)
    assert_base_plus_delta(ic1, c.ic1_0, d13, act)
    assert_base_plus_delta(ic3, c.ic3_0, d2, act)


def test_tensor_core_and_warp_mma_agree():
    """Both expands on the same batch: each within the oracle tolerance, and
    within a few bf16 steps of one another."""
    c = gen.dense_case(name="tc_ab", T=400, H=1024, out_dims=(256, 384), L=5, R=32, seed=75,
                       ranks=(32, 8, 24, 16, 32), scales=(1.0, 0.5, 2.0, 1.5, 1.0))
    outs = []
    for pol in (3, 8):
        L.lora_set_kernel_policy(pol)
        try:
            run = H.DenseRun(c)
            try:
                run.step()
                outs.append(bf16_bits_to_f32(run.y_host()).astype(np.float64))
                assert run.status() == 0
            finally:
                run.close()
        finally:
            L.lora_set_kernel_policy(0)
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    for o in outs:
        assert_delta(o[act], d_ref[act], "tc/mma")
    scale = np.abs(d_ref[act]).max()
    assert np.abs(outs[0] - outs[1]).max() <= 2 ** -6 * scale
