"""MoE-LoRA over the block-padded alignment (lora_moe_apply_blocks), the
per-pair schedule (block_m 1) and the block kernel lora_moe_apply runs at
sparse occupancy, against the oracle (vLLM FusedMoEWithLoRA: naive block
assignment when num_tokens * top_k * 8 <= num_experts * max_loras)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
from gpu_util import assert_delta, assert_rows_untouched
from test_gpu_moe import pair_active, run_and_check

pytestmark = pytest.mark.gpu


def _cap(c, bm):
    P = c.T * c.K
    return max(bm, ((P + c.E * (bm - 1) + bm - 1) // bm) * bm)


def _align(run, c, bm):
    cap = _cap(c, bm)
    ds = torch.empty((c.L, cap), dtype=torch.int32, device="cuda")
    de = torch.empty((c.L, cap // bm), dtype=torch.int32, device="cuda")
    dn = torch.empty(c.L, dtype=torch.int32, device="cuda")
    L.lora_moe_align_padded(run.pool, run.mb.meta, bm, cap, ds, de, dn)
    return ds, de, dn, cap


def _apply_blocks(run, c, bm, ds, de, dn, cap):
    L.lora_moe_apply_blocks(run.pool, run.mb.meta, L.MOE_W13, run.x, c.D + run.in_pad, None, run.ic1,
                            c.n13 * c.F13 + run.out_pad, ds, de, dn, bm, cap)
    L.lora_moe_apply_blocks(run.pool, run.mb.meta, L.MOE_W2, run.ic2, c.F + run.in_pad, run.topk_w, run.ic3,
                            c.D + run.out_pad, ds, de, dn, bm, cap)


def _check(c, ic1, ic3, act):
    _, d13 = oracle.moe_w13(c)
    _, d2 = oracle.moe_w2(c)
    assert_rows_untouched(ic1, c.ic1_0, ~act)
    assert_rows_untouched(ic3, c.ic3_0, ~act)
    assert_delta(bf16_bits_to_f32(ic1)[act], d13[act], c.name + " w13")
    assert_delta(bf16_bits_to_f32(ic3)[act], d2[act], c.name + " w2")


def _small(shared, seed=0, **kw):
    args = dict(name=f"moe_blocks{seed}", T=57, K=3, E=7, D=1040, F=272, L=4, R=24, seed=seed,
                shared_outer=shared, ranks=(24, 9, 16, 0), scales=(1.5, 0.5, 2.0, 1.0), p_none=0.1)
    args.update(kw)
    return gen.moe_case(**args)


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("bm", [1, 4, 16])
def test_blocks_match_oracle(bm, shared):
    c = _small(shared, seed=bm)
    run = H.MoERun(c, in_pad=8, out_pad=16)
    try:
        run.build_meta()
        ds, de, dn, cap = _align(run, c, bm)
        _apply_blocks(run, c, bm, ds, de, dn, cap)
        ic1, ic3 = run.ic1_host(), run.ic3_host()
        assert run.status() == 0
    finally:
        run.close()
    _check(c, ic1, ic3, pair_active(c))


@pytest.mark.parametrize("kind", ["3d", "non_gated", "e1_top1"])
def test_blocks_layouts(kind):
    if kind == "3d":
        c = gen.moe_case(name="moe3d_b", T=24, K=4, E=8, D=512, F=128, L=3, R=16, seed=15, n13=1, f13=256)
    elif kind == "non_gated":
        c = gen.moe_case(name="moe_ng_b", T=24, K=2, E=8, D=512, F=128, L=3, R=16, seed=16, n13=1)
    else:
        c = gen.moe_case(name="moe_e1_b", T=9, K=1, E=1, D=256, F=128, L=3, R=8, seed=17, p_none=0.3)
    run = H.MoERun(c)
    try:
        run.build_meta()
        ds, de, dn, cap = _align(run, c, 1)
        _apply_blocks(run, c, 1, ds, de, dn, cap)
        ic1, ic3 = run.ic1_host(), run.ic3_host()
    finally:
        run.close()
    _check(c, ic1, ic3, pair_active(c))


def test_blocks_skip_dropped_blocks_and_sentinels():
    """Blocks whose expert is -1 or num_experts and entries outside [0, T*K)
    add nothing; every other pair gets its delta."""
    c = _small(False, seed=21)
    run = H.MoERun(c)
    try:
        run.build_meta()
        ds, de, dn, cap = _align(run, c, 1)
        s, e, n = ds.cpu().numpy(), de.cpu().numpy(), dn.cpu().numpy()
        dropped = []
        a_used = [a for a in range(c.L) if n[a] >= 3]
        a = a_used[0]
        dropped.append(s[a][0])
        e[a][0] = -1
        dropped.append(s[a][1])
        e[a][1] = c.E
        dropped.append(s[a][2])
        s[a][2] = -5
        de.copy_(torch.from_numpy(e))
        ds.copy_(torch.from_numpy(s))
        _apply_blocks(run, c, 1, ds, de, dn, cap)
        ic1, ic3 = run.ic1_host(), run.ic3_host()
    finally:
        run.close()
    act = pair_active(c)
    act[np.asarray(dropped)] = False
    _check(c, ic1, ic3, act)


@pytest.mark.parametrize("T", [1, 4, 8])
@pytest.mark.parametrize("shared", [False, True])
def test_block_kernel_at_sparse_occupancy(T, shared):
    """T * 8 * 8 <= 64 * 8: lora_moe_apply runs the block kernel over the
    metadata's tiles."""
    run_and_check(gen.moe(shared_outer=shared, T=T))


@pytest.mark.parametrize("T", [16, 64])
@pytest.mark.parametrize("pol", [4, 5], ids=["perpair", "tilecluster"])
def test_block_kernel_forced(T, pol):
    """Policy 4: the per-pair schedule at any batch size; policy 5: the same
    kernel over the metadata's 16-row tiles."""
    L.lora_set_kernel_policy(pol)
    try:
        run_and_check(gen.moe(T=T))
        run_and_check(_small(True, seed=T))
    finally:
        L.lora_set_kernel_policy(0)


def test_blocks_errors():
    c = _small(False, seed=3)
    run = H.MoERun(c)
    try:
        run.build_meta()
        ds, de, dn, cap = _align(run, c, 4)
        for bm, cp in ((0, cap), (17, 17 * 4), (4, cap + 2)):
            with pytest.raises(L.LoraError) as ei:
                L.lora_moe_apply_blocks(run.pool, run.mb.meta, L.MOE_W13, run.x, c.D, None, run.ic1,
                                        c.n13 * c.F13, ds, de, dn, bm, cp)
            assert ei.value.code == L.CODE["LORA_ERR_INVALID_ARG"]
        with pytest.raises(L.LoraError) as ei:
            L.lora_moe_apply_blocks(run.pool, run.mb.meta, L.MOE_W13, run.x, c.D, run.topk_w, run.ic1,
                                    c.n13 * c.F13, ds, de, dn, 4, cap)
        assert ei.value.code == L.CODE["LORA_ERR_INVALID_ARG"]
        with pytest.raises(L.LoraError) as ei:
            L.lora_moe_apply_blocks(run.pool, run.mb.meta, L.MOE_W2, run.ic2, c.F, run.topk_w, run.ic3,
                                    c.D - 8, ds, de, dn, 4, cap)
        assert ei.value.code == L.CODE["LORA_ERR_INVALID_ARG"]
    finally:
        run.close()
