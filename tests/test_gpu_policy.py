"""Every compute path of lora_apply_slices / lora_moe_apply against the
oracle: the automatic choice (split shrink/expand kernels for these shapes,
tcgen05 for long runs), the persistent split-K kernel (kernel policy 1), the
one-pass cluster kernel (kernel policy 2), the MoE schedules (3-5) and the
split expand on warp-level MMAs instead of tcgen05 (8)."""
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


@pytest.fixture(params=[0, 1, 2, 3, 4, 5, 8],
                ids=["auto", "splitk", "cluster", "split", "perpair", "tilecluster", "warpmma"])
def policy(request):
    L.lora_set_kernel_policy(request.param)
    yield request.param
    L.lora_set_kernel_policy(0)


def _dense(c):
    run = H.DenseRun(c)
    try:
        run.step()
        y = run.y_host()
        assert run.status() == 0
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], c.name)


@pytest.mark.parametrize("name", ["decode_qkv", "many_adapter_down", "small_multi_tile", "prefill_gate_up"])
def test_dense_paths(name, policy):
    if name == "decode_qkv":
        c = gen.decode_qkv()
    elif name == "many_adapter_down":
        c = gen.many_adapter_down()
    elif name == "prefill_gate_up":
        c = gen.prefill_gate_up(permuted=True)
    else:
        c = gen.dense_case(name="smt", T=150, H=2056, out_dims=(264, 136, 80), L=4, R=24, seed=41,
                           ranks=(24, 13, 1, 8), scales=(1.0, 0.5, 2.0, 1.5), p_none=0.1)
    _dense(c)


@pytest.mark.parametrize("shared", [False, True])
def test_moe_paths(shared, policy):
    c = gen.moe(shared_outer=shared)
    run = H.MoERun(c)
    try:
        run.step()
        ic1 = H.from_dev_u16(run.ic1)
        ic3 = H.from_dev_u16(run.ic3)
        assert run.status() == 0
    finally:
        run.close()
    _, d13 = oracle.moe_w13(c)
    _, d2 = oracle.moe_w2(c)
    assert_delta(bf16_bits_to_f32(ic1), d13, "w13")
    assert_delta(bf16_bits_to_f32(ic3), d2, "w2")


@pytest.mark.parametrize("pol", [0, 2], ids=["split", "cluster"])
def test_apply_in_a_graph_replayed(pol):
    """Metadata + apply captured together (programmatic dependent launch
    edges inside the graph) and replayed three times: the split kernels'
    arrival counters and the split-K control words clean up after
    themselves."""
    L.lora_set_kernel_policy(pol)
    c = gen.decode_qkv()
    run = H.DenseRun(c)
    try:
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                run.step()
        run.y.zero_()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        y = run.y_host()
    finally:
        run.close()
        L.lora_set_kernel_policy(0)
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y)[act], 3 * d_ref[act], "3 replays")


def test_moe_repeated_steps_share_workspace(policy):
    """w13 and w2 calls alternate on one workspace for three steps: every call
    type and path leaves the workspace ready for the next call."""
    c = gen.moe(shared_outer=False)
    run = H.MoERun(c)
    try:
        for _ in range(3):
            run.step()
        ic1 = H.from_dev_u16(run.ic1)
        ic3 = H.from_dev_u16(run.ic3)
        assert run.status() == 0
    finally:
        run.close()
    _, d13 = oracle.moe_w13(c)
    _, d2 = oracle.moe_w2(c)
    assert_delta(bf16_bits_to_f32(ic1), 3 * d13, "w13 x3")
    assert_delta(bf16_bits_to_f32(ic3), 3 * d2, "w2 x3")


def test_dense_token_counts_share_workspace(policy):
    """Batches of 256, 100 and 256 tokens on one workspace sized for 256."""
    c = gen.decode_qkv()
    run = H.DenseRun(c)
    try:
        run.build_meta(c.T)
        run.apply()
        run.build_meta(100)
        run.apply()
        run.build_meta(c.T)
        run.apply()
        y = run.y_host()
        assert run.status() == 0
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    w = np.full(c.T, 2.0)
    w[:100] = 3.0
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y)[act] - bf16_bits_to_f32(c.y0)[act], (w[:, None] * d_ref)[act], "256+100+256")


def test_dense_idle_and_disabled_slots(policy):
    """Enabled slots with no tokens, a disabled slot and a rank-0 slot next to
    busy slots with several 16-row tiles each (the slot-major shrink reads A
    of every enabled slot before it knows the batch)."""
    rng = np.random.default_rng(77)
    T, L = 160, 8
    idx = rng.choice(np.array([0, 3, 5, -1], np.int32), size=T, p=[0.4, 0.3, 0.2, 0.1]).astype(np.int32)
    idx[7] = 6   # disabled slot: no delta
    idx[9] = 7   # rank-0 slot: no delta
    c = gen.dense_case(name="idle_slots", T=T, H=1032, out_dims=(264, 520), L=L, R=16, seed=78,
                       ranks=(16, 8, 16, 13, 16, 16, 16, 0), scales=(1.0, 2.0, 0.5, 1.5, 1.0, 0.25, 1.0, 1.0),
                       enabled=(1, 1, 1, 1, 1, 1, 0, 1), idx=idx)
    _dense(c)
